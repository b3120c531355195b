/*
 * kvq.h - sub-byte KV-cache quantization and packed-cache decode attention for GB300 (sm_103a).
 *
 * A stateless C library. The caller owns every buffer (device memory for the cache, inputs,
 * outputs and workspace); the library validates arguments on the host, then enqueues CUDA
 * kernels on the caller's stream and returns. It allocates nothing. Two kinds of entry point
 * depart from the rest:
 *   - the host-buffer calls (kvq_append_decode_attend_host, kvq_paged_append_decode_attend_host)
 *     wait for their stream before returning, since they return with the host output filled;
 *   - kvq_decode_attend_static keeps its partials in one device array built into the library,
 *     so two of its calls that overlap on the GPU race (see there).
 * Every other entry point is re-entrant and never synchronises.
 *
 * Pages this follows (cited by title and section):
 *   [FT]  FreeToken PR #268 "feat(kvcache): sub-byte Q4_0 and Q6_0 KV cache quantization",
 *         "Storage layouts" and the q4_0 max_magnitude paragraph; packed buffer plus separate
 *         scale buffer per spec ("Changes": mha_pool).
 *   [TR]  tract discussion #2402 "Heads-up / RFC: int4 + Hadamard KV-cache quantization
 *         (CPU + Metal)", "What's done", "Architecture: Data flow (decode)", "Why this quant
 *         scheme", "Causality & mixed precision", "NNEF surface" (axis, scale, causal, n_recent).
 *   [OTQ] "Open-TQ-Metal: Fused Compressed-Domain Attention for Long-Context LLM Inference on
 *         Apple Silicon", per-group asymmetric int4 background; Section 3 (fused kernel, GQA
 *         mapping kv_head = head / gqa, split-K into ceil(S/512) chunks, partial + reduce phases).
 *
 * Conventions
 *   - All device pointers must be 16-byte aligned; the workspace 256-byte aligned.
 *   - Element order is row-major C order in the shapes given below.
 *   - Errors are returned as kvq_status; nothing is printed, nothing aborts. A failed call
 *     enqueues nothing. kvq_last_error() gives a one-line reason for the calling thread's
 *     last failure. KVQ_ECUDA reports a launch error seen right after enqueueing.
 *   - Inputs must be finite; NaN/Inf inputs give unspecified codes and outputs.
 *   - head_dim must be 128 or 256.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. NULL means the legacy default stream. */
typedef struct CUstream_st *kvq_stream_t;

typedef enum {
  KVQ_OK = 0,
  KVQ_EINVAL = 1,        /* null pointer, negative size, bad enum value, kv_len == 0 */
  KVQ_ESHAPE = 2,        /* head_dim not 128/256, H_q not a multiple of H_kv, bad chunk */
  KVQ_ECAPACITY = 3,     /* pos0 + n_new > capacity, kv_len > capacity */
  KVQ_EUNSUPPORTED = 4,  /* layout/dtype combination not provided */
  KVQ_EALIGN = 5,        /* a pointer is not 16-byte aligned (workspace: 256) */
  KVQ_ECUDA = 6,         /* a CUDA launch failed */
  KVQ_EWORKSPACE = 7     /* workspace_bytes smaller than kvq_attend_workspace_bytes() */
} kvq_status;

typedef enum {
  /* [FT] q4_0: per 32 values along head_dim, 16 payload bytes (byte j = value 2j in the low
   * nibble, value 2j+1 in the high nibble; the nibble is read back as (v ^ 0x8) - 0x8) and one
   * fp16 scale = amax / 8; codes clamped to [-8, 7]. */
  KVQ_Q4_0 = 0,
  /* [FT] q6_0: per 32 values a 16-byte low plane (low four bits, q4_0 nibble order) followed by
   * an 8-byte high plane (top two bits, value 4k+i at bits 2i of byte k), one fp16 scale =
   * amax / 32; read back as (v ^ 0x20) - 0x20 with v = low | high << 4; codes in [-32, 31]. */
  KVQ_Q6_0 = 1,
  /* [TR] per-token symmetric int4 in a fixed Hadamard basis: y = FWHT(x) * fp32(1/sqrt(D))
   * (radix-2 butterflies, half-span 1, 2, ..., D/2), one f32 scale s = amax(|y|) / 7 per token,
   * codes rint(y / s) in [-7, 7] packed in q4_0 nibble order (D/2 bytes per token). Scores
   * are the exact integer dot int8(q_rot) . int4(k_rot) times the scales. An optional ring
   * of the newest n_recent rotated rows is kept in exact f32. */
  KVQ_HAD_INT4 = 2,
  /* [OTQ] per-group asymmetric int4, g = 32: fp16 scale = (max - min) / 15 and fp16
   * zero-point = min per group; codes rint((x - zero) / scale) in [0, 15], unsigned, q4_0
   * nibble order; value = code * scale + zero. */
  KVQ_ASYM4_G32 = 3,
  /* [FT] q8_0 (only its density is printed, 1.0625 bytes/element): per 32 values 32 int8 code
   * bytes (byte i = value i, two's complement) and one fp16 scale; by the family rule of q4_0 /
   * q6_0 (magnitude 2^(bits-1)) scale = amax / 128 and codes clamped to [-128, 127]. */
  KVQ_Q8_0 = 4,
  /* [TR] the Hadamard layout with a 2-bit body ("Why this quant scheme": int2 is usable only
   * with the mixed-precision window; "Causality & mixed precision": n_recent is the lever for
   * pushing the body below 4 bits): per-token symmetric int2 in the same rotated basis, one f32
   * scale s = amax(|y|) per token, codes rint(y / s) in [-1, 1], four per byte (value 4j+i at
   * bits 2i of byte j, read back as (v ^ 2) - 2; D/4 bytes per token), the same optional ring
   * of the newest n_recent rotated rows in exact f32. Meant for a wide window. */
  KVQ_HAD_INT2 = 5
} kvq_layout;

/* Mixed K/V precision ([OTQ] Section 5: value quantisation costs more output quality than key
 * quantisation, so V may deserve more bits than K): a cache whose K plane uses layout `k` and
 * whose V plane uses layout `v`, e.g. KVQ_MIXED(KVQ_Q4_0, KVQ_Q8_0). Both must be block layouts
 * (Q4_0, Q6_0, Q8_0, ASYM4_G32) or both Hadamard layouts (HAD_INT4, HAD_INT2: one rotated basis,
 * one window ring per plane). A plain layout value means the same layout for K and V. Mixed caches
 * are stored with kvq_store and attended by every attention entry point. */
#define KVQ_MIXED(k, v) ((int32_t)(k) | (((int32_t)(v) + 1) << 8))

typedef enum { KVQ_F32 = 0, KVQ_BF16 = 1, KVQ_F16 = 2 } kvq_dtype;

/*
 * A caller-owned packed cache for one attention layer. Planes (K and V each):
 *   payload  u8  [batch][n_kv_heads][capacity][kvq_row_bytes(layout, head_dim)]
 *   scale    f16 [batch][n_kv_heads][capacity][head_dim/32]      (Q4_0, Q6_0, Q8_0, ASYM4_G32)
 *            f32 [batch][n_kv_heads][capacity]                   (HAD_INT4, HAD_INT2)
 *   zero     f16 [batch][n_kv_heads][capacity][head_dim/32]      (ASYM4_G32 only, else NULL)
 *   recent   f32 [batch][n_kv_heads][n_recent][head_dim]         (HAD_INT4 / HAD_INT2 with
 *                                                                 n_recent > 0, else NULL)
 * Payload and scales sit in separate buffers ([FT] "packed buffer + separate scale buffer").
 * The cache is preallocated at `capacity` tokens and appended in place ([OTQ]: per-step
 * concatenation instead of preallocated slices cost 18%).
 */
typedef struct kvq_cache {
  int32_t layout;      /* kvq_layout, or KVQ_MIXED(k layout, v layout): each plane's byte layout,
                          scale and zero planes are then those of its own layout */
  int32_t batch;
  int32_t n_kv_heads;
  int32_t head_dim;    /* 128 or 256 */
  int32_t capacity;    /* tokens per (batch, kv head) */
  int32_t n_recent;    /* HAD_INT4 / HAD_INT2: size of the exact-f32 ring (0 = none); others: 0 */
  void *k_payload, *v_payload;
  void *k_scale, *v_scale;
  void *k_zero, *v_zero;
  float *k_recent, *v_recent;
} kvq_cache;

/* Payload bytes of one token row of one head; 0 for an unknown layout or head_dim. */
size_t kvq_row_bytes(int32_t layout, int32_t head_dim);

/* Bytes of each plane of one of K or V: out_sizes = {payload, scale, zero, recent}.
 * Unused planes report 0. `layout` is a plain layout: for a KVQ_MIXED cache ask once with the K
 * layout (for the K planes) and once with the V layout. */
kvq_status kvq_cache_bytes(int32_t layout, int32_t batch, int32_t n_kv_heads, int32_t head_dim,
                           int32_t capacity, int32_t n_recent, size_t out_sizes[4]);

/*
 * Store (append) n_new tokens per (batch, kv head) at positions [pos0, pos0 + n_new).
 *   k_new, v_new: device [batch][n_kv_heads][n_new][head_dim] in `dtype` (f32, bf16 or f16).
 * Quantisation is exact and deterministic: re-storing a token writes identical bytes.
 * HAD_INT4 / HAD_INT2 with n_recent > 0 also write the rotated f32 rows of the last
 * min(n_new, n_recent) tokens to ring slot (position mod n_recent); attention with the window
 * therefore expects kv_len equal to the end of the latest store.
 * One kernel launch covers K and V. n_new == 0 is a no-op.
 */
kvq_status kvq_store_q4_0(const kvq_cache *cache, const void *k_new, const void *v_new,
                          int32_t dtype, int32_t n_new, int32_t pos0, kvq_stream_t stream);
kvq_status kvq_store_q6_0(const kvq_cache *cache, const void *k_new, const void *v_new,
                          int32_t dtype, int32_t n_new, int32_t pos0, kvq_stream_t stream);
kvq_status kvq_store_hadamard_int4(const kvq_cache *cache, const void *k_new, const void *v_new,
                                   int32_t dtype, int32_t n_new, int32_t pos0,
                                   kvq_stream_t stream);
kvq_status kvq_store_asym4_g32(const kvq_cache *cache, const void *k_new, const void *v_new,
                               int32_t dtype, int32_t n_new, int32_t pos0, kvq_stream_t stream);
kvq_status kvq_store_q8_0(const kvq_cache *cache, const void *k_new, const void *v_new,
                          int32_t dtype, int32_t n_new, int32_t pos0, kvq_stream_t stream);
/* The same append for a cache of any layout, KVQ_MIXED ones included (each plane quantised by
 * its own layout; a mixed cache takes one launch per plane). */
kvq_status kvq_store(const kvq_cache *cache, const void *k_new, const void *v_new, int32_t dtype,
                     int32_t n_new, int32_t pos0, kvq_stream_t stream);
kvq_status kvq_store_hadamard_int2(const kvq_cache *cache, const void *k_new, const void *v_new,
                                   int32_t dtype, int32_t n_new, int32_t pos0,
                                   kvq_stream_t stream);

/* Workspace bytes kvq_decode_attend needs for these arguments on the current device (0 on
 * invalid arguments). chunk 0 means the automatic chunk described at kvq_decode_attend. */
size_t kvq_attend_workspace_bytes(const kvq_cache *cache, int32_t n_q_heads, int32_t n_q,
                                  int32_t kv_len, int32_t chunk);

/* The chunk length kvq_decode_attend uses for these arguments on the current device (`chunk`
 * itself when non-zero and valid, the automatic choice for 0); 0 on invalid arguments. The
 * automatic choice depends on the layout, head_dim and query rows per kv head
 * (n_q_heads / n_kv_heads * n_q), which select the phase-1 kernel. */
int32_t kvq_attend_chunk(const kvq_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t kv_len, int32_t chunk);

/*
 * Fused split-K decode attention over the packed cache; the dequantised K/V matrix is never
 * written anywhere ([OTQ] Section 3: fused compressed-domain attention).
 *   q    device [batch][n_q_heads][n_q][head_dim] in q_dtype
 *   out  device f32 [batch][n_q_heads][n_q][head_dim]
 * Query head h reads kv head h / (n_q_heads / n_kv_heads) ([OTQ] GQA mapping). Row i of each
 * head attends tokens t < kv_len and, when causal != 0, t <= q_pos0 + i ([TR] causal
 * masking); a causal call needs 0 <= q_pos0 and q_pos0 + n_q <= kv_len.
 * score = attn_scale * q . k_hat. Phase 1 splits the tokens into chunks of `chunk` tokens
 * (a multiple of 64 in [64, 8192], e.g. 512 as in [OTQ]; 0 = automatic, sized for the phase-1
 * kernel that runs and the current device's SM count -- one wave of resident warps or CTAs for
 * decode shapes, about four waves of 64-row CTAs for many query rows; kvq_attend_chunk returns
 * it) and writes per (row, chunk) the
 * running max, the sum of exponentials and the unnormalised output to the workspace; phase 2
 * combines them with the online-softmax correction ([OTQ] Section 3.2). HAD_INT4 / HAD_INT2: the query
 * is rotated and quantised to int8 (one f32 scale per row, amax / 127), body tokens are
 * scored by the exact integer dot, the newest min(n_recent, kv_len) tokens by exact f32
 * from the ring, and phase 2 un-rotates the output ([TR] data flow).
 * The two phases are separate launches on `stream`; the workspace must not be shared with
 * another call in flight.
 */
kvq_status kvq_decode_attend(const kvq_cache *cache, const void *q, int32_t q_dtype,
                             int32_t n_q_heads, int32_t n_q, int32_t kv_len, int32_t causal,
                             int32_t q_pos0, float attn_scale, int32_t chunk, float *out,
                             void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * One decode (or prefill-chunk) step in one call: the append of n_new tokens at positions
 * [pos0, pos0 + n_new) exactly as the cache layout's kvq_store_* (k_new/v_new and kv_dtype as
 * there), then kvq_decode_attend with the remaining arguments, on the same stream. The result
 * and the stored bytes are identical to those two calls. Because this call knows which token
 * rows the append writes, the phase-1 work that does not read them starts while the append is
 * still running. All arguments of both parts are validated before anything is launched; on an
 * error status nothing has been launched. n_new == 0 is a plain kvq_decode_attend.
 */
kvq_status kvq_append_decode_attend(const kvq_cache *cache, const void *k_new, const void *v_new,
                                    int32_t kv_dtype, int32_t n_new, int32_t pos0, const void *q,
                                    int32_t q_dtype, int32_t n_q_heads, int32_t n_q, int32_t kv_len,
                                    int32_t causal, int32_t q_pos0, float attn_scale, int32_t chunk,
                                    float *out, void *workspace, size_t workspace_bytes,
                                    kvq_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Paged cache ([FT] "Scope": only the paged full-attention KV pool is quantized; "Changes":
 * mha_pool allocates a packed buffer plus a separate scale buffer per spec). Token rows live in
 * a pool of fixed-size pages shared by all sequences of a batch; a block table gives the pool
 * page of each logical page of each sequence, and every sequence has its own length.
 *   payload  u8  [n_pages][n_kv_heads][page_size][kvq_row_bytes(layout, head_dim)]
 *   scale    f16 [n_pages][n_kv_heads][page_size][head_dim/32]   (Q4_0, Q6_0, ASYM4_G32)
 *            f32 [n_pages][n_kv_heads][page_size]                (HAD_INT4, HAD_INT2)
 *   zero     f16 [n_pages][n_kv_heads][page_size][head_dim/32]   (ASYM4_G32 only, else NULL)
 *   recent   f32 [batch][n_kv_heads][n_recent][head_dim]         (HAD_INT4 / HAD_INT2 with
 *                                                                 n_recent > 0: one ring per
 *                                                                 sequence)
 *   block_table  device i32 [batch][max_pages_per_seq]
 * Token t of sequence b is row t % page_size of pool page block_table[b][t / page_size]. Byte
 * layouts and quantisation are those of the contiguous cache (one token row is bit-identical).
 * page_size is a power of two in [64, 2^20]: every 64-token stage the kernels stream is then a
 * run of consecutive rows. The caller owns the pool and the table and keeps every entry that a
 * call reads inside [0, n_pages); an entry outside is clamped into the pool (no access leaves
 * it, the result is then unspecified). A sequence's logical capacity is
 * max_pages_per_seq * page_size tokens.
 */
typedef struct kvq_paged_cache {
  int32_t layout;             /* kvq_layout or KVQ_MIXED(k, v) */
  int32_t batch;              /* sequences (rows of the block table) */
  int32_t n_kv_heads;
  int32_t head_dim;           /* 128 or 256 */
  int32_t page_size;          /* tokens per page: a power of two in [64, 2^20] */
  int32_t n_pages;            /* pages in the pool */
  int32_t max_pages_per_seq;  /* row length of the block table */
  int32_t n_recent;           /* HAD_INT4 / HAD_INT2: exact-f32 ring per sequence (0 = none); others: 0 */
  void *k_payload, *v_payload;
  void *k_scale, *v_scale;
  void *k_zero, *v_zero;
  float *k_recent, *v_recent;
  const int32_t *block_table;
} kvq_paged_cache;

/* Bytes of each pool plane of one of K or V: out_sizes = {payload, scale, zero, recent}. */
kvq_status kvq_paged_cache_bytes(int32_t layout, int32_t n_pages, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t page_size, int32_t batch, int32_t n_recent, size_t out_sizes[4]);

/*
 * Append n_new tokens to every sequence: sequence b's rows go to positions
 * [positions[b], positions[b] + n_new), through the block table.
 *   k_new, v_new: device [batch][n_kv_heads][n_new][head_dim] in `dtype`.
 *   positions:    device i32 [batch].
 * Quantisation as kvq_store_* for the cache's layout (any layout; bit-identical rows). The
 * positions are read on the device: a row whose position falls outside [0, max_pages_per_seq *
 * page_size) is not written. HAD_INT4 / HAD_INT2 with n_recent > 0 also write the rotated f32 rows of the
 * last min(n_new, n_recent) tokens to the sequence's ring slot (position mod n_recent).
 * One kernel launch covers K and V. n_new == 0 is a no-op.
 */
kvq_status kvq_paged_store(const kvq_paged_cache *cache, const void *k_new, const void *v_new, int32_t dtype,
                           int32_t n_new, const int32_t *positions, kvq_stream_t stream);

/* Workspace bytes of kvq_paged_decode_attend for these arguments (0 on invalid arguments).
 * max_kv_len as there. */
size_t kvq_paged_attend_workspace_bytes(const kvq_paged_cache *cache, int32_t n_q_heads, int32_t n_q,
                                        int32_t max_kv_len, int32_t chunk);
/* The chunk kvq_paged_decode_attend uses: `chunk` itself when non-zero and valid; for chunk 0, the
 * automatic choice. total_kv_len = the sum of the batch's sequence lengths, known to the caller's
 * scheduler on the host; 0 means "every sequence at max_kv_len". A ragged batch gets a better
 * balanced chunk from its true total: pass the returned value as `chunk` to the attend call (and
 * to kvq_paged_attend_workspace_bytes). 0 on invalid arguments. */
int32_t kvq_paged_attend_chunk(const kvq_paged_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t max_kv_len,
                               int64_t total_kv_len, int32_t chunk);
/* A balanced chunk for a ragged batch from the host copy of its sequence lengths (host i32
 * [batch], the lengths the attend call will see): every sequence's body is split into
 * ceil(body / chunk) equal chunks, and the returned chunk is the shortest (multiple of 64) whose
 * chunks of all sequences and kv heads fit one wave of the phase-1 kernel these shapes select on
 * the current device (else the fewest waves x chunk). Pass it as `chunk` to the attend call and
 * to kvq_paged_attend_workspace_bytes. 0 on invalid arguments. Host only: reads no device memory. */
int32_t kvq_paged_attend_plan_chunk(const kvq_paged_cache *cache, int32_t n_q_heads, int32_t n_q, int32_t q_dtype,
                                    const int32_t *host_seq_lens);

/*
 * kvq_decode_attend over a paged cache with per-sequence lengths. Each sequence's body is split
 * into ceil(body / chunk) chunks of equal length (multiples of 64 tokens, none longer than chunk).
 *   q    device [batch][n_q_heads][n_q][head_dim] in q_dtype
 *   out  device f32 [batch][n_q_heads][n_q][head_dim]
 *   seq_lens  device i32 [batch]: the number of cached tokens of each sequence, read on the
 *             device and clamped into [0, max_kv_len].
 *   max_kv_len  host: an upper bound of every seq_lens[b] (1 <= max_kv_len <= capacity); the
 *             grid and the workspace are sized for it.
 * Row i of each query head of sequence b attends t < seq_lens[b] and, when causal != 0,
 * t <= seq_lens[b] - n_q + i (the n_q query rows are the sequence's newest tokens). A row that
 * sees no token (an empty sequence, or a causal row before the sequence's start) gets zeros.
 * HAD_INT4 / HAD_INT2: the newest min(n_recent, seq_lens[b]) tokens of each sequence are read from its
 * ring. Everything else (GQA mapping, chunking, the two phases, the workspace rule) is as
 * kvq_decode_attend.
 */
kvq_status kvq_paged_decode_attend(const kvq_paged_cache *cache, const void *q, int32_t q_dtype, int32_t n_q_heads,
                                   int32_t n_q, const int32_t *seq_lens, int32_t max_kv_len, int32_t causal,
                                   float attn_scale, int32_t chunk, float *out, void *workspace,
                                   size_t workspace_bytes, kvq_stream_t stream);

/*
 * One paged decode (or prefill-chunk) step: append n_new tokens to the end of every sequence,
 * at positions [seq_lens[b] - n_new, seq_lens[b]) (seq_lens = the lengths after the append),
 * then kvq_paged_decode_attend with the remaining arguments. Result and stored bytes are those
 * of kvq_paged_store + kvq_paged_decode_attend; as for kvq_append_decode_attend, phase-1 work
 * that does not read the appended rows starts while the append runs. All arguments are
 * validated before anything is launched. n_new == 0 is a plain kvq_paged_decode_attend.
 */
kvq_status kvq_paged_append_decode_attend(const kvq_paged_cache *cache, const void *k_new, const void *v_new,
                                          int32_t kv_dtype, int32_t n_new, const void *q, int32_t q_dtype,
                                          int32_t n_q_heads, int32_t n_q, const int32_t *seq_lens,
                                          int32_t max_kv_len, int32_t causal, float attn_scale, int32_t chunk,
                                          float *out, void *workspace, size_t workspace_bytes,
                                          kvq_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Host-buffer forms of the two append + attend calls, for callers whose new rows and queries are
 * in host memory and who want the result there (no counterpart on the pages: the steps are
 * those of the device-buffer calls above, with the copies around them).
 *   k_new, v_new  host [batch][n_kv_heads][n_new][head_dim] in kv_dtype (unused when n_new == 0)
 *   q             host [batch][n_q_heads][n_q][head_dim] in q_dtype
 *   out           host f32 [batch][n_q_heads][n_q][head_dim]
 *   seq_lens      (paged) host i32 [batch], the lengths after the append, as in
 *                 kvq_paged_append_decode_attend
 *   workspace     device, 256-byte aligned, at least the matching *_host_workspace_bytes: the
 *                 attention partials followed by device staging for k_new, v_new, q, out
 *                 (and seq_lens; the staging of buffers used in place stays unused); the caller
 *                 owns it, the call must not share it with another call in flight.
 * Page-locked (pinned) host buffers that are 16-byte aligned are used in place where that saves
 * a copy: under unified addressing the GPU reaches them directly, so the store kernel reads k_new
 * and v_new from them and the reduce writes `out` into them. q is always copied host -> device on
 * `stream` (cudaMemcpyAsync) into the staging area, because every phase-1 CTA of a kv head reads it.
 * Pageable buffers (or unaligned ones) are staged with copies both ways (the driver stages
 * pageable memory itself; when k_new, v_new and q lie back to back in that order in host memory,
 * one copy moves all three). The call enqueues the same launches as the device-buffer call
 * (identical results and stored bytes) and returns after cudaStreamSynchronize(stream), with
 * `out` filled. Every argument
 * is validated before anything is enqueued; a CUDA error from a copy, a launch or the
 * synchronisation returns KVQ_ECUDA (then nothing can be assumed about `out` or the cache rows
 * of the append). The host buffers may be reused as soon as the call returns.
 */
size_t kvq_append_decode_attend_host_workspace_bytes(const kvq_cache *cache, int32_t kv_dtype, int32_t n_new,
                                                     int32_t q_dtype, int32_t n_q_heads, int32_t n_q,
                                                     int32_t kv_len, int32_t chunk);
kvq_status kvq_append_decode_attend_host(const kvq_cache *cache, const void *k_new, const void *v_new,
                                         int32_t kv_dtype, int32_t n_new, int32_t pos0, const void *q,
                                         int32_t q_dtype, int32_t n_q_heads, int32_t n_q, int32_t kv_len,
                                         int32_t causal, int32_t q_pos0, float attn_scale, int32_t chunk,
                                         float *out, void *workspace, size_t workspace_bytes,
                                         kvq_stream_t stream);
size_t kvq_paged_append_decode_attend_host_workspace_bytes(const kvq_paged_cache *cache, int32_t kv_dtype,
                                                           int32_t n_new, int32_t q_dtype, int32_t n_q_heads,
                                                           int32_t n_q, int32_t max_kv_len, int32_t chunk);
kvq_status kvq_paged_append_decode_attend_host(const kvq_paged_cache *cache, const void *k_new, const void *v_new,
                                               int32_t kv_dtype, int32_t n_new, const void *q, int32_t q_dtype,
                                               int32_t n_q_heads, int32_t n_q, const int32_t *seq_lens,
                                               int32_t max_kv_len, int32_t causal, float attn_scale, int32_t chunk,
                                               float *out, void *workspace, size_t workspace_bytes,
                                               kvq_stream_t stream);

/*
 * HAD_INT4 / HAD_INT2 test hook: the exact integer-domain body scores int8(q_rot) . code(k_rot)
 * ([TR] "What's done": the int8 x int4 -> i32 score dot), from a plain scalar kernel of its own
 * (a cross-check: the attention calls score the body on the tensor cores, see
 * kvq_debug_attend_scores_i32).
 *   scores_out device i32 [batch][n_q_heads][n_q][kv_len - min(n_recent, kv_len)]
 *   s_q_out    device f32 [batch][n_q_heads][n_q]   (the per-row int8 scale of q_rot)
 */
kvq_status kvq_debug_scores_i32(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                int32_t n_q_heads, int32_t n_q, int32_t kv_len,
                                int32_t *scores_out, float *s_q_out, kvq_stream_t stream);

/*
 * HAD_INT4 / HAD_INT2 test hook on the production path: kvq_decode_attend (same arguments, same
 * kernels, chunking and output `out`), with the phase-1 tensor-core kernel that scores the body
 * also writing every exact integer score int8(q_rot) . code(k_rot) it computes ([TR] "What's
 * done": the i32 score dot; exact integers, so any summation order agrees) and each row's int8
 * query scale, read from the values that kernel uses for the softmax.
 *   scores_out device i32 [batch][n_q_heads][n_q][kv_len - min(n_recent, kv_len)]; the entry of
 *              (row, body token t) is written when some row of that row's tile sees t (every
 *              t <= the row's causal limit at least); the caller pre-fills it to tell the rest
 *   s_q_out    device f32 [batch][n_q_heads][n_q]
 * Returns KVQ_EUNSUPPORTED unless the cache is contiguous, one Hadamard layout in both planes,
 * and the call's body runs on a tensor-core kernel (head_dim 128).
 */
kvq_status kvq_debug_attend_scores_i32(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                       int32_t n_q_heads, int32_t n_q, int32_t kv_len, int32_t causal,
                                       int32_t q_pos0, float attn_scale, int32_t chunk, float *out,
                                       void *workspace, size_t workspace_bytes, int32_t *scores_out,
                                       float *s_q_out, kvq_stream_t stream);

/*
 * Measurement hook (no counterpart on the pages): while both events are non-NULL, every
 * kvq_decode_attend call made by this thread records `phase1_begin` on its stream right before
 * the phase-1 launch and `phase1_end` right after it, so a caller can time the streaming kernel
 * alone with cudaEventElapsedTime. The records are external event records, so under stream
 * capture they become event-record nodes of the graph and time every replay. The events are
 * cudaEvent_t handles created by the caller (with timing enabled);
 * passing NULL for either disables recording. Thread-local; returns KVQ_OK.
 */
kvq_status kvq_profile_phase1_events(void *phase1_begin, void *phase1_end);

/* Bytes of the device scratch array built into the library for kvq_decode_attend_static. */
#define KVQ_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * kvq_decode_attend with no workspace argument, for callers that cannot allocate device memory
 * themselves: for instance a plugin running inside a host engine that owns the whole device
 * memory pool and hands out nothing beyond a layer's inputs and outputs, or code on a
 * latency-critical thread that must not enter the CUDA allocator. This entry point has no
 * counterpart in the paper; it exists only for such callers.
 *   Arguments, layouts and results are those of kvq_decode_attend. The split-K partials live in
 *   one device array of KVQ_STATIC_SCRATCH_BYTES that is part of the library: every device that
 *   loads the library holds it until the process exits. A call whose partials would not fit
 *   (see kvq_attend_workspace_bytes) returns KVQ_EWORKSPACE and enqueues nothing.
 *   Nothing is allocated or freed: no cudaMalloc/cudaFree or allocating library routine runs.
 *   The first call made with a given device current looks up the array's device address on that
 *   device (cudaGetSymbolAddress) and keeps it for the life of the process; make that first call
 *   before any stream capture. The kept address belongs to the device's primary context: calls
 *   made after cudaDeviceReset on that device, or from another context, are not supported.
 *   Every call, on every stream, shares the one array, and it keeps the last call's contents
 *   (the kernels write every partial before reading it, so nothing needs clearing). Calls whose
 *   work overlaps on the GPU (other streams, or concurrent host threads) race on the array and
 *   give undefined results: serialise them.
 */
kvq_status kvq_decode_attend_static(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                    int32_t n_q_heads, int32_t n_q, int32_t kv_len, int32_t causal,
                                    int32_t q_pos0, float attn_scale, int32_t chunk, float *out,
                                    kvq_stream_t stream);

/* Static description of a status code. */
const char *kvq_status_string(int32_t status);

/* One-line reason for the calling thread's most recent failed call ("" if none). */
const char *kvq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
