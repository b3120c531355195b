"""Seeded synthetic K/V/Q generators.

Every workload is described by a `Workload` record (shapes, dtype, value recipe, seed) and
turned into host arrays by `make_inputs`. The arrays come in two forms: the raw element bits
of the declared dtype (what a device buffer holds) and the exact float32 value of each element
(what the CPU oracle consumes). The float32 form is derived from the bits, so both sides see
the same numbers.

Value recipes follow the pages' synthetic workloads:
  * "normal": N(0, 1) (the tiny Q4_0 case);
  * "student_t(df)": heavy-tailed K/V ("kurtotic K/V", FreeToken PR #268, Validation table);
  * planted outlier channels: per (kv head, tensor) a seeded set of distinct channels is
    multiplied by a factor for every token ("planted-outlier data", tract discussion #2402,
    Appendix 7);
  * RMS-normalised Q and K rows for the attention-scale-1.0 case (Open-TQ-Metal, Section 4:
    Gemma normalises Q and K by RMS norm and uses scale 1.0).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_paged_inputs", "ragged_lengths", "bf16_bits_from_f32",
           "f32_from_bf16_bits", "f16_bits_from_f32", "f32_from_f16_bits"]


# ----------------------------------------------------------------------------- dtype helpers
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-half-to-even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact float32 value of bfloat16 bits."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32_from_f16_bits(b: np.ndarray) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


# ----------------------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layout: str            # "q4_0" | "q6_0" | "had_int4" | "asym4_g32"
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    kv_len: int            # final cache length attended over
    n_q: int = 1           # query rows per head
    fill: int = -1         # tokens stored by the first (bulk) store call; rest appended after
    causal: bool = False
    q_pos0: int = 0        # absolute position of query row 0 (causal limit of row i = q_pos0 + i)
    attn_scale: float = 0.0  # 0 -> 1/sqrt(head_dim)
    n_recent: int = 0
    dtype: str = "bf16"    # dtype of K/V/Q inputs: "f32" | "bf16"
    values: str = "student_t"
    df: float = 4.0
    n_outlier: int = 0
    outlier_factor: float = 1.0
    outlier_on_v: bool = True
    rms_norm_qk: bool = False
    chunk: int = 512
    seed: int = 0
    page_size: int = 0     # > 0: a paged pool of page_size-token pages, one length per sequence
    seq_lens: tuple = ()   # per-sequence lengths of a paged workload (kv_len = their maximum)

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def alpha(self) -> float:
        return self.attn_scale if self.attn_scale else 1.0 / math.sqrt(self.head_dim)

    @property
    def n_fill(self) -> int:
        return self.kv_len if self.fill < 0 else self.fill

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def ragged_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    """n seeded sequence lengths drawn uniformly from [lo, hi] (a serving batch of mixed lengths)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


_RAGGED = ragged_lengths(1006, 16, 1024, 16384)

WORKLOADS = {
    # Q4_0 tiny: B1, 8 q heads / 2 kv heads, d128, S512 decode; fp32 N(0,1), 2 K outlier channels x8.
    "c1_q4_0_tiny": Workload("c1_q4_0_tiny", "q4_0", 1, 8, 2, 128, 512, dtype="f32", values="normal",
                             n_outlier=2, outlier_factor=8.0, outlier_on_v=False, seed=1001),
    # Llama-3-8B layer: B4, 32/8 heads, d128, S8192; bf16 Student-t(4), 4 outlier ch x10; fill 8191 + append 1.
    "c2_q4_0_llama3_8b": Workload("c2_q4_0_llama3_8b", "q4_0", 4, 32, 8, 128, 8192, fill=8191,
                                  n_outlier=4, outlier_factor=10.0, seed=1002),
    # Hadamard per-token int4, Qwen3-1.7B shape: B8, 16/8 heads, d128, S4096, n_recent 64.
    "c3_had_int4_decode": Workload("c3_had_int4_decode", "had_int4", 8, 16, 8, 128, 4096, fill=4095,
                                   n_recent=64, n_outlier=4, outlier_factor=10.0, seed=1003),
    # same cache, causal prefill chunk of 256 rows appended at 3840.
    "c3_had_int4_prefill": Workload("c3_had_int4_prefill", "had_int4", 8, 16, 8, 128, 4096, n_q=256,
                                    fill=3840, causal=True, q_pos0=3840, n_recent=64, n_outlier=4,
                                    outlier_factor=10.0, seed=1003),
    # Q6_0 Gemma-like: B2, 16/8 heads, d256, S32768, scale 1.0, unit-RMS Q/K rows, Student-t(3).
    "c4_q6_0_gemma": Workload("c4_q6_0_gemma", "q6_0", 2, 16, 8, 256, 32768, fill=32767, attn_scale=1.0,
                              df=3.0, rms_norm_qk=True, seed=1004),
    # Llama-3.1-70B layer at 128K: B1, 64/8 heads, d128, S131072, Q4_0, chunk 512.
    "c5_q4_0_llama70b_128k": Workload("c5_q4_0_llama70b_128k", "q4_0", 1, 64, 8, 128, 131072, fill=131071,
                                      n_outlier=4, outlier_factor=10.0, seed=1005),
    # same shape, per-group asymmetric int4 (g=32, fp16 scale + zero-point).
    "c5_asym4_g32_llama70b_128k": Workload("c5_asym4_g32_llama70b_128k", "asym4_g32", 1, 64, 8, 128, 131072,
                                           fill=131071, n_outlier=4, outlier_factor=10.0, seed=1005),
    # the 128K layer in Q8_0 (8-bit codes, fp16 scale per 32 values) and with mixed precision
    # (4-bit Q4_0 keys, 8-bit Q8_0 values: V errors reach the output directly)
    "c5_q8_0_llama70b_128k": Workload("c5_q8_0_llama70b_128k", "q8_0", 1, 64, 8, 128, 131072, fill=131071,
                                      n_outlier=4, outlier_factor=10.0, seed=1005),
    "c5_q4_0_k_q8_0_v_llama70b_128k": Workload("c5_q4_0_k_q8_0_v_llama70b_128k", "q4_0+q8_0", 1, 64, 8, 128, 131072,
                                               fill=131071, n_outlier=4, outlier_factor=10.0, seed=1005),
    # the Hadamard decode cache with a 2-bit body and a 256-token exact-f32 window
    "c3_had_int2_decode_w256": Workload("c3_had_int2_decode_w256", "had_int2", 8, 16, 8, 128, 4096, fill=4095,
                                        n_recent=256, n_outlier=4, outlier_factor=10.0, seed=1003),
    # serving-style paged batch of a Llama-3-8B layer (32/8 heads, d128), Q4_0: 16 sequences with
    # seeded lengths in [1024, 16384], 64-token pages in a shuffled pool; decode: one new token per
    # sequence, then attention over each sequence's own length.
    "paged_q4_0_llama3_8b_ragged": Workload("paged_q4_0_llama3_8b_ragged", "q4_0", 16, 32, 8, 128, max(_RAGGED),
                                            n_outlier=4, outlier_factor=10.0, seed=1006, page_size=64,
                                            seq_lens=_RAGGED),
}


def _draw(rng: np.random.Generator, w: Workload, shape) -> np.ndarray:
    if w.values == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if w.values == "student_t":
        return rng.standard_t(w.df, size=shape).astype(np.float32)
    raise ValueError(w.values)


def _rms_normalise(x: np.ndarray) -> np.ndarray:
    x64 = x.astype(np.float64)
    r = np.sqrt(np.mean(x64 * x64, axis=-1, keepdims=True))
    r[r == 0] = 1.0
    return (x64 / r).astype(np.float32)


def _plant_outliers(x: np.ndarray, rng: np.random.Generator, n_out: int, factor: float) -> None:
    """x: [B][H_kv][S][D]; scale n_out seeded distinct channels of each kv head by `factor`."""
    if n_out <= 0:
        return
    H, D = x.shape[1], x.shape[3]
    for h in range(H):
        ch = rng.choice(D, size=n_out, replace=False)
        x[:, h, :, ch] *= np.float32(factor)  # advanced index: axis order (ch, B, S)


def make_inputs(w: Workload, kv_len: int | None = None, n_q: int | None = None, seed_offset: int = 0) -> dict:
    """Return the seeded inputs of workload `w`.

    Keys: k_bits, v_bits, q_bits (element bits in w.dtype: uint32 view for f32, uint16 for
    bf16), k, v, q (exact float32 values), plus `dtype`. K/V: [B][H_kv][S][D]; Q: [B][H_q][n_q][D].
    `kv_len`/`n_q` override the sizes (smaller parity cases keep the value recipe).
    """
    S = w.kv_len if kv_len is None else kv_len
    nq = w.n_q if n_q is None else n_q
    rng = np.random.Generator(np.random.PCG64(w.seed + seed_offset))
    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    q = rng.standard_normal((B, Hq, nq, D), dtype=np.float32)
    k = _draw(rng, w, (B, Hkv, S, D))
    v = _draw(rng, w, (B, Hkv, S, D))
    _plant_outliers(k, rng, w.n_outlier, w.outlier_factor)
    if w.outlier_on_v:
        _plant_outliers(v, rng, w.n_outlier, w.outlier_factor)
    if w.rms_norm_qk:
        q = _rms_normalise(q)
        k = _rms_normalise(k)
    out = {"dtype": w.dtype}
    for name, x in (("q", q), ("k", k), ("v", v)):
        if w.dtype == "bf16":
            bits = bf16_bits_from_f32(x)
            out[name + "_bits"] = bits
            out[name] = f32_from_bf16_bits(bits)
        elif w.dtype == "f32":
            x = np.ascontiguousarray(x, dtype=np.float32)
            out[name + "_bits"] = x.view(np.uint32)
            out[name] = x
        else:
            raise ValueError(w.dtype)
    return out


def make_paged_inputs(w: Workload) -> dict:
    """Seeded inputs of a paged workload, drawn by the same recipe as `make_inputs` but only for
    the tokens that exist: K/V of all sequences back to back, [H_kv][T][D] with T = sum(seq_lens)
    (sequence b = tokens offsets[b] .. offsets[b] + seq_lens[b] - 1), and Q [B][H_q][n_q][D].
    Keys as make_inputs (k, v, q and their *_bits) plus seq_lens and offsets (int64 arrays)."""
    lens = np.asarray(w.seq_lens, np.int64)
    T = int(lens.sum())
    flat = make_inputs(w.scaled(batch=1, kv_len=T, n_q=w.n_q * w.batch))
    out = {"dtype": flat["dtype"], "seq_lens": lens, "offsets": np.concatenate([[0], np.cumsum(lens)[:-1]])}
    for name in ("k", "v"):
        out[name] = flat[name][0]
        out[name + "_bits"] = flat[name + "_bits"][0]
    for name in ("q", "q_bits"):
        x = flat[name][0]                                  # [H_q][B * n_q][D]
        out[name] = np.ascontiguousarray(x.reshape(x.shape[0], w.batch, w.n_q, x.shape[-1]).transpose(1, 0, 2, 3))
    return out
