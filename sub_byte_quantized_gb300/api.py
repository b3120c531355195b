"""Thin torch-facing wrappers over the C ABI: they check tensor placement/shape, pass raw
pointers and the current CUDA stream, and nothing else. Every computation runs in libkvq.so.

torch is used for device memory (cache planes, workspace) and streams only.
"""
from __future__ import annotations

import ctypes as C
import math

import torch

from . import _lib as L

_DTYPES = {torch.float32: L.KVQ_F32, torch.bfloat16: L.KVQ_BF16, torch.float16: L.KVQ_F16}
_STORE_FN = {L.KVQ_Q4_0: "kvq_store_q4_0", L.KVQ_Q6_0: "kvq_store_q6_0",
             L.KVQ_HAD_INT4: "kvq_store_hadamard_int4", L.KVQ_ASYM4_G32: "kvq_store_asym4_g32",
             L.KVQ_Q8_0: "kvq_store_q8_0", L.KVQ_HAD_INT2: "kvq_store_hadamard_int2"}


def _layout_id(layout) -> int:
    """Layout value of a name ("q4_0", or "k+v" such as "q4_0+q8_0" for mixed K/V precision) or id."""
    if isinstance(layout, str):
        k, _, v = layout.partition("+")
        return L.mixed(L.LAYOUT_IDS[k], L.LAYOUT_IDS[v]) if v and v != k else L.LAYOUT_IDS[k]
    return int(layout)


def _plane_tensors(layout: int, lead: tuple, head_dim: int, dev, n_recent: int, ring_lead: tuple) -> dict:
    """Zeroed device planes of one of K or V in a plain layout: payload, scale [, zero] [, recent]."""
    rb = row_bytes(layout, head_dim)
    nb = head_dim // 32
    pl = {"payload": torch.zeros(lead + (rb,), dtype=torch.uint8, device=dev)}
    if layout in L.HADAMARD_IDS:
        pl["scale"] = torch.zeros(lead, dtype=torch.float32, device=dev)
        if n_recent:
            pl["recent"] = torch.zeros(ring_lead + (n_recent, head_dim), dtype=torch.float32, device=dev)
    else:
        pl["scale"] = torch.zeros(lead + (nb,), dtype=torch.float16, device=dev)
        if layout == L.KVQ_ASYM4_G32:
            pl["zero"] = torch.zeros(lead + (nb,), dtype=torch.float16, device=dev)
    return pl


def _plane_read_bytes(layout: int, head_dim: int, n_tokens: int, n_recent: int) -> int:
    """Packed bytes one plane of one (batch, kv head) reads over n_tokens tokens."""
    per_tok = row_bytes(layout, head_dim)
    if layout in L.HADAMARD_IDS:
        n_w = min(n_recent, n_tokens)
        return (n_tokens - n_w) * (per_tok + 4) + n_w * head_dim * 4
    return n_tokens * (per_tok + 2 * (head_dim // 32) * (2 if layout == L.KVQ_ASYM4_G32 else 1))


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if isinstance(s, torch.cuda.Stream) else int(s)


def _need_cuda(name: str, t: torch.Tensor) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def row_bytes(layout, head_dim: int) -> int:
    return int(L.lib().kvq_row_bytes(_layout_id(layout), head_dim))


def cache_plane_bytes(layout, batch, n_kv_heads, head_dim, capacity, n_recent=0) -> dict:
    out = (C.c_size_t * 4)()
    L.check(L.lib().kvq_cache_bytes(_layout_id(layout), batch, n_kv_heads, head_dim, capacity, n_recent, out),
            "kvq_cache_bytes")
    return {"payload": out[0], "scale": out[1], "zero": out[2], "recent": out[3]}


class KVCache:
    """Device planes of one layer's packed cache plus the C struct describing them.

    Planes (K and V each): payload u8 [B][H_kv][cap][row_bytes]; scale f16 [B][H_kv][cap][D/32]
    (f32 [B][H_kv][cap] for had_int4 / had_int2); zero f16 (asym4_g32); recent f32 [B][H_kv][n_recent][D]
    (the Hadamard layouts with n_recent > 0).
    """

    def __init__(self, layout, batch: int, n_kv_heads: int, head_dim: int, capacity: int, n_recent: int = 0,
                 device="cuda"):
        self.layout = _layout_id(layout)
        self.plane_layouts = dict(zip(("k", "v"), L.plane_ids(self.layout)))
        self.batch, self.n_kv_heads, self.head_dim, self.capacity = batch, n_kv_heads, head_dim, capacity
        self.n_recent = n_recent if self.plane_layouts["k"] in L.HADAMARD_IDS else 0
        dev = torch.device(device)
        shp = (batch, n_kv_heads, capacity)
        self.planes = {}
        for t in ("k", "v"):
            lt = self.plane_layouts[t]
            sizes = cache_plane_bytes(lt, batch, n_kv_heads, head_dim, capacity, self.n_recent)
            pl = _plane_tensors(lt, shp, head_dim, dev, self.n_recent, (batch, n_kv_heads))
            assert pl["payload"].numel() == sizes["payload"]
            self.planes[t] = pl
        self.struct = L.KvqCache(
            self.layout, batch, n_kv_heads, head_dim, capacity, self.n_recent,
            _ptr(self.planes["k"]["payload"]), _ptr(self.planes["v"]["payload"]),
            _ptr(self.planes["k"]["scale"]), _ptr(self.planes["v"]["scale"]),
            _ptr(self.planes["k"].get("zero")), _ptr(self.planes["v"].get("zero")),
            _ptr(self.planes["k"].get("recent")), _ptr(self.planes["v"].get("recent")))

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for pl in self.planes.values() for t in pl.values())

    def read_bytes(self, kv_len: int) -> int:
        """Packed bytes (payload + scales [+ zeros] [+ window]) one attention call reads."""
        return self.batch * self.n_kv_heads * sum(
            _plane_read_bytes(self.plane_layouts[t], self.head_dim, kv_len, self.n_recent) for t in ("k", "v"))


def store(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, pos0: int, stream=None) -> None:
    """Append k_new/v_new [B][H_kv][n_new][D] at positions [pos0, pos0 + n_new)."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new)
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same shape and dtype")
    B, H, n_new, D = k_new.shape
    if (B, H, D) != (cache.batch, cache.n_kv_heads, cache.head_dim):
        raise ValueError("k_new shape does not match the cache")
    name = _STORE_FN.get(cache.layout, "kvq_store")       # mixed K/V layouts: the generic store
    fn = getattr(L.lib(), name)
    L.check(fn(C.byref(cache.struct), k_new.data_ptr(), v_new.data_ptr(), _DTYPES[k_new.dtype], n_new, pos0,
               _stream(stream)), name)


def attend_workspace_bytes(cache: KVCache, n_q_heads: int, n_q: int, kv_len: int, chunk: int = 0) -> int:
    return int(L.lib().kvq_attend_workspace_bytes(C.byref(cache.struct), n_q_heads, n_q, kv_len, chunk))


def attend_chunk(cache: KVCache, n_q_heads: int, n_q: int, kv_len: int, chunk: int = 0) -> int:
    """The split-K chunk length a decode_attend call with these arguments uses (0 -> automatic)."""
    return int(L.lib().kvq_attend_chunk(C.byref(cache.struct), n_q_heads, n_q, kv_len, chunk))


def decode_attend(cache: KVCache, q: torch.Tensor, kv_len: int, causal: bool = False, q_pos0: int = 0,
                  attn_scale: float | None = None, chunk: int = 0, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Split-K attention of q [B][H_q][n_q][D] over the first kv_len cached tokens -> f32 out."""
    _need_cuda("q", q)
    B, Hq, n_q, D = q.shape
    if B != cache.batch or D != cache.head_dim:
        raise ValueError("q shape does not match the cache")
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    _need_cuda("out", out)
    need = attend_workspace_bytes(cache, Hq, n_q, kv_len, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_cuda("workspace", workspace)
    L.check(L.lib().kvq_decode_attend(C.byref(cache.struct), q.data_ptr(), _DTYPES[q.dtype], Hq, n_q, kv_len,
                                      int(bool(causal)), q_pos0, float(attn_scale), chunk, out.data_ptr(),
                                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "kvq_decode_attend")
    return out


def append_decode_attend(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, pos0: int, q: torch.Tensor,
                         kv_len: int, causal: bool = False, q_pos0: int = 0, attn_scale: float | None = None,
                         chunk: int = 0, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """store(cache, k_new, v_new, pos0) then decode_attend(cache, q, kv_len, ...) in one library
    call (same results; the attention work that does not read the appended rows overlaps the
    append)."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new)
    _need_cuda("q", q)
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same shape and dtype")
    Bk, H, n_new, Dk = k_new.shape
    B, Hq, n_q, D = q.shape
    if (Bk, H, Dk) != (cache.batch, cache.n_kv_heads, cache.head_dim) or B != cache.batch or D != cache.head_dim:
        raise ValueError("k_new/q shape does not match the cache")
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    _need_cuda("out", out)
    need = attend_workspace_bytes(cache, Hq, n_q, kv_len, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_cuda("workspace", workspace)
    L.check(L.lib().kvq_append_decode_attend(
        C.byref(cache.struct), k_new.data_ptr(), v_new.data_ptr(), _DTYPES[k_new.dtype], n_new, pos0, q.data_ptr(),
        _DTYPES[q.dtype], Hq, n_q, kv_len, int(bool(causal)), q_pos0, float(attn_scale), chunk, out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)),
        "kvq_append_decode_attend")
    return out


def decode_attend_static(cache: KVCache, q: torch.Tensor, kv_len: int, causal: bool = False, q_pos0: int = 0,
                         attn_scale: float | None = None, chunk: int = 0, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """decode_attend without a workspace: the library's built-in device scratch holds the partials.

    For callers that cannot allocate device memory of their own. Calls share that scratch, so
    calls that overlap on the GPU race; the first call on a device must precede stream capture.
    """
    _need_cuda("q", q)
    B, Hq, n_q, D = q.shape
    if B != cache.batch or D != cache.head_dim:
        raise ValueError("q shape does not match the cache")
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    _need_cuda("out", out)
    L.check(L.lib().kvq_decode_attend_static(C.byref(cache.struct), q.data_ptr(), _DTYPES[q.dtype], Hq, n_q,
                                             kv_len, int(bool(causal)), q_pos0, float(attn_scale), chunk,
                                             out.data_ptr(), _stream(stream)), "kvq_decode_attend_static")
    return out


def debug_scores_i32(cache: KVCache, q: torch.Tensor, kv_len: int, stream=None):
    """Hadamard-int4 exact integer body scores [B][H_q][n_q][kv_len - n_window] and the int8 row scales."""
    _need_cuda("q", q)
    B, Hq, n_q, D = q.shape
    n_body = kv_len - min(cache.n_recent, kv_len)
    buf = torch.empty(B * Hq * n_q * max(n_body, 1), dtype=torch.int32, device=q.device)
    s_q = torch.empty((B, Hq, n_q), dtype=torch.float32, device=q.device)
    L.check(L.lib().kvq_debug_scores_i32(C.byref(cache.struct), q.data_ptr(), _DTYPES[q.dtype], Hq, n_q, kv_len,
                                         buf.data_ptr(), s_q.data_ptr(), _stream(stream)),
            "kvq_debug_scores_i32")
    return buf[:B * Hq * n_q * n_body].view(B, Hq, n_q, n_body), s_q


def debug_attend_scores_i32(cache: KVCache, q: torch.Tensor, kv_len: int, causal: bool = False, q_pos0: int = 0,
                            attn_scale: float | None = None, chunk: int = 0, fill: int = -(2 ** 31), stream=None):
    """decode_attend on the production kernels, with the tensor-core kernel that scores the body also
    writing its exact integer scores: returns (out, scores [B][H_q][n_q][n_body] int32, s_q [B][H_q][n_q]).
    Score entries the kernels did not compute keep `fill`."""
    _need_cuda("q", q)
    B, Hq, n_q, D = q.shape
    if B != cache.batch or D != cache.head_dim:
        raise ValueError("q shape does not match the cache")
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    n_body = kv_len - min(cache.n_recent, kv_len)
    out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    scores = torch.full((B * Hq * n_q * max(n_body, 1),), fill, dtype=torch.int32, device=q.device)
    s_q = torch.zeros((B, Hq, n_q), dtype=torch.float32, device=q.device)
    need = attend_workspace_bytes(cache, Hq, n_q, kv_len, chunk)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    L.check(L.lib().kvq_debug_attend_scores_i32(
        C.byref(cache.struct), q.data_ptr(), _DTYPES[q.dtype], Hq, n_q, kv_len, int(bool(causal)), q_pos0,
        float(attn_scale), chunk, out.data_ptr(), workspace.data_ptr(), workspace.numel(), scores.data_ptr(),
        s_q.data_ptr(), _stream(stream)), "kvq_debug_attend_scores_i32")
    return out, scores[:B * Hq * n_q * n_body].view(B, Hq, n_q, n_body), s_q


# ------------------------------------------------------------------ paged pool
class PagedKVCache:
    """Device planes of one layer's paged pool, its block table and the C struct describing them.

    Planes (K and V each): payload u8 [n_pages][H_kv][page_size][row_bytes]; scale f16
    [n_pages][H_kv][page_size][D/32] (f32 [n_pages][H_kv][page_size] for had_int4); zero f16
    (asym4_g32); recent f32 [batch][H_kv][n_recent][D] (had_int4 with n_recent > 0, one ring per
    sequence). block_table: int32 [batch][max_pages_per_seq] (pool page of each logical page),
    owned by this object; the caller fills it (set_block_table) before storing.
    """

    def __init__(self, layout, batch: int, n_kv_heads: int, head_dim: int, page_size: int, n_pages: int,
                 max_pages_per_seq: int, n_recent: int = 0, device="cuda"):
        self.layout = _layout_id(layout)
        self.batch, self.n_kv_heads, self.head_dim = batch, n_kv_heads, head_dim
        self.page_size, self.n_pages, self.max_pages_per_seq = page_size, n_pages, max_pages_per_seq
        self.capacity = page_size * max_pages_per_seq
        self.plane_layouts = dict(zip(("k", "v"), L.plane_ids(self.layout)))
        self.n_recent = n_recent if self.plane_layouts["k"] in L.HADAMARD_IDS else 0
        dev = torch.device(device)
        shp = (n_pages, n_kv_heads, page_size)
        self.planes = {}
        for t in ("k", "v"):
            lt = self.plane_layouts[t]
            out = (C.c_size_t * 4)()
            L.check(L.lib().kvq_paged_cache_bytes(lt, n_pages, n_kv_heads, head_dim, page_size, batch,
                                                  self.n_recent, out), "kvq_paged_cache_bytes")
            pl = _plane_tensors(lt, shp, head_dim, dev, self.n_recent, (batch, n_kv_heads))
            assert pl["payload"].numel() == out[0]
            self.planes[t] = pl
        self.block_table = torch.zeros((batch, max_pages_per_seq), dtype=torch.int32, device=dev)
        self.struct = L.KvqPagedCache(
            self.layout, batch, n_kv_heads, head_dim, page_size, n_pages, max_pages_per_seq, self.n_recent,
            _ptr(self.planes["k"]["payload"]), _ptr(self.planes["v"]["payload"]),
            _ptr(self.planes["k"]["scale"]), _ptr(self.planes["v"]["scale"]),
            _ptr(self.planes["k"].get("zero")), _ptr(self.planes["v"].get("zero")),
            _ptr(self.planes["k"].get("recent")), _ptr(self.planes["v"].get("recent")),
            _ptr(self.block_table))

    def set_block_table(self, table) -> None:
        """Copy an int [batch][max_pages_per_seq] table (pool page of each logical page)."""
        t = torch.as_tensor(table, dtype=torch.int32)
        if tuple(t.shape) != (self.batch, self.max_pages_per_seq):
            raise ValueError("block table shape does not match the cache")
        self.block_table.copy_(t)

    def read_bytes(self, seq_lens) -> int:
        """Packed bytes (payload + scales [+ zeros] [+ window]) one attention call reads."""
        return self.n_kv_heads * sum(_plane_read_bytes(self.plane_layouts[t], self.head_dim, int(n), self.n_recent)
                                     for n in seq_lens for t in ("k", "v"))


def _i32_vec(name: str, t: torch.Tensor, n: int) -> None:
    _need_cuda(name, t)
    if t.dtype != torch.int32 or t.numel() != n:
        raise ValueError(f"{name} must be a CUDA int32 tensor of {n} entries")


def paged_store(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor, positions: torch.Tensor,
                stream=None) -> None:
    """Append k_new/v_new [B][H_kv][n_new][D]: sequence b's rows at [positions[b], positions[b] + n_new)."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new)
    _i32_vec("positions", positions, cache.batch)
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same shape and dtype")
    B, H, n_new, D = k_new.shape
    if (B, H, D) != (cache.batch, cache.n_kv_heads, cache.head_dim):
        raise ValueError("k_new shape does not match the cache")
    L.check(L.lib().kvq_paged_store(C.byref(cache.struct), k_new.data_ptr(), v_new.data_ptr(), _DTYPES[k_new.dtype],
                                    n_new, positions.data_ptr(), _stream(stream)), "kvq_paged_store")


def paged_attend_workspace_bytes(cache: PagedKVCache, n_q_heads: int, n_q: int, max_kv_len: int,
                                 chunk: int = 0) -> int:
    return int(L.lib().kvq_paged_attend_workspace_bytes(C.byref(cache.struct), n_q_heads, n_q, max_kv_len, chunk))


def paged_attend_chunk(cache: PagedKVCache, n_q_heads: int, n_q: int, max_kv_len: int, total_kv_len: int = 0,
                       chunk: int = 0) -> int:
    """The split-K chunk of a paged call (0 -> automatic); total_kv_len = the sum of the sequence
    lengths (0: every sequence at max_kv_len) balances a ragged batch."""
    return int(L.lib().kvq_paged_attend_chunk(C.byref(cache.struct), n_q_heads, n_q, max_kv_len, total_kv_len,
                                              chunk))


def paged_attend_plan_chunk(cache: PagedKVCache, n_q_heads: int, n_q: int, seq_lens, q_dtype=torch.bfloat16) -> int:
    """A balanced split-K chunk for this batch from the host copy of its sequence lengths."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if lens.size != cache.batch:
        raise ValueError("seq_lens must have one entry per sequence")
    return int(L.lib().kvq_paged_attend_plan_chunk(C.byref(cache.struct), n_q_heads, n_q, _DTYPES[q_dtype],
                                                   lens.ctypes.data))


def _paged_out_ws(cache, q, max_kv_len, chunk, out, workspace):
    B, Hq, n_q, D = q.shape
    if B != cache.batch or D != cache.head_dim:
        raise ValueError("q shape does not match the cache")
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    _need_cuda("out", out)
    need = paged_attend_workspace_bytes(cache, Hq, n_q, max_kv_len, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_cuda("workspace", workspace)
    return out, workspace


def paged_decode_attend(cache: PagedKVCache, q: torch.Tensor, seq_lens: torch.Tensor, max_kv_len: int,
                        causal: bool = False, attn_scale: float | None = None, chunk: int = 0,
                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Split-K attention of q [B][H_q][n_q][D] over each sequence's seq_lens[b] tokens -> f32 out
    (causal rows are each sequence's newest n_q tokens)."""
    _need_cuda("q", q)
    _i32_vec("seq_lens", seq_lens, cache.batch)
    Hq, n_q, D = q.shape[1], q.shape[2], q.shape[3]
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    out, workspace = _paged_out_ws(cache, q, max_kv_len, chunk, out, workspace)
    L.check(L.lib().kvq_paged_decode_attend(
        C.byref(cache.struct), q.data_ptr(), _DTYPES[q.dtype], Hq, n_q, seq_lens.data_ptr(), max_kv_len,
        int(bool(causal)), float(attn_scale), chunk, out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)), "kvq_paged_decode_attend")
    return out


def paged_append_decode_attend(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                               seq_lens: torch.Tensor, max_kv_len: int, causal: bool = False,
                               attn_scale: float | None = None, chunk: int = 0, out: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_store at [seq_lens[b] - n_new, seq_lens[b]) then paged_decode_attend, in one call."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new)
    _need_cuda("q", q)
    _i32_vec("seq_lens", seq_lens, cache.batch)
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same shape and dtype")
    Bk, H, n_new, Dk = k_new.shape
    if (Bk, H, Dk) != (cache.batch, cache.n_kv_heads, cache.head_dim):
        raise ValueError("k_new shape does not match the cache")
    Hq, n_q, D = q.shape[1], q.shape[2], q.shape[3]
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    out, workspace = _paged_out_ws(cache, q, max_kv_len, chunk, out, workspace)
    L.check(L.lib().kvq_paged_append_decode_attend(
        C.byref(cache.struct), k_new.data_ptr(), v_new.data_ptr(), _DTYPES[k_new.dtype], n_new, q.data_ptr(),
        _DTYPES[q.dtype], Hq, n_q, seq_lens.data_ptr(), max_kv_len, int(bool(causal)), float(attn_scale), chunk,
        out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)),
        "kvq_paged_append_decode_attend")
    return out


def _need_host(name: str, t: torch.Tensor) -> None:
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor for the host-buffer call")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _host_out_ws(q, device, need, out, workspace):
    B, Hq, n_q, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, pin_memory=True)
    _need_host("out", out)
    if out.dtype != torch.float32 or tuple(out.shape) != (B, Hq, n_q, D):
        raise ValueError("out must be a float32 host tensor of q's shape")
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    _need_cuda("workspace", workspace)
    return out, workspace


def append_decode_attend_host_workspace_bytes(cache: KVCache, kv_dtype, n_new: int, q_dtype, n_q_heads: int,
                                              n_q: int, kv_len: int, chunk: int = 0) -> int:
    return L.lib().kvq_append_decode_attend_host_workspace_bytes(C.byref(cache.struct), _DTYPES[kv_dtype], n_new,
                                                                 _DTYPES[q_dtype], n_q_heads, n_q, kv_len, chunk)


def append_decode_attend_host(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, pos0: int, q: torch.Tensor,
                              kv_len: int, causal: bool = False, q_pos0: int = 0, attn_scale: float | None = None,
                              chunk: int = 0, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """append_decode_attend with host tensors (ideally pinned): the library copies k_new, v_new and
    q to device staging in the workspace, runs the step and copies the f32 result back into the
    host tensor `out`, returning once it is filled."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("q", q)):
        _need_host(n, t)
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same shape and dtype")
    Bk, H, n_new, Dk = k_new.shape
    B, Hq, n_q, D = q.shape
    if (Bk, H, Dk) != (cache.batch, cache.n_kv_heads, cache.head_dim) or B != cache.batch or D != cache.head_dim:
        raise ValueError("k_new/q shape does not match the cache")
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    need = 0 if workspace is not None else \
        append_decode_attend_host_workspace_bytes(cache, k_new.dtype, n_new, q.dtype, Hq, n_q, kv_len, chunk)
    out, workspace = _host_out_ws(q, cache.planes["k"]["payload"].device, need, out, workspace)
    L.check(L.lib().kvq_append_decode_attend_host(
        C.byref(cache.struct), k_new.data_ptr(), v_new.data_ptr(), _DTYPES[k_new.dtype], n_new, pos0, q.data_ptr(),
        _DTYPES[q.dtype], Hq, n_q, kv_len, int(bool(causal)), q_pos0, float(attn_scale), chunk, out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)),
        "kvq_append_decode_attend_host")
    return out


def paged_append_decode_attend_host_workspace_bytes(cache: PagedKVCache, kv_dtype, n_new: int, q_dtype,
                                                    n_q_heads: int, n_q: int, max_kv_len: int, chunk: int = 0) -> int:
    return L.lib().kvq_paged_append_decode_attend_host_workspace_bytes(
        C.byref(cache.struct), _DTYPES[kv_dtype], n_new, _DTYPES[q_dtype], n_q_heads, n_q, max_kv_len, chunk)


def paged_append_decode_attend_host(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                                    seq_lens: torch.Tensor, max_kv_len: int, causal: bool = False,
                                    attn_scale: float | None = None, chunk: int = 0,
                                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                    stream=None) -> torch.Tensor:
    """paged_append_decode_attend with host tensors (seq_lens: host int32 [batch]); returns once the
    host tensor `out` holds the result."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("q", q), ("seq_lens", seq_lens)):
        _need_host(n, t)
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != cache.batch:
        raise ValueError(f"seq_lens must be a host int32 tensor of {cache.batch} entries")
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same shape and dtype")
    Bk, H, n_new, Dk = k_new.shape
    B, Hq, n_q, D = q.shape
    if (Bk, H, Dk) != (cache.batch, cache.n_kv_heads, cache.head_dim) or B != cache.batch or D != cache.head_dim:
        raise ValueError("k_new/q shape does not match the cache")
    if attn_scale is None:
        attn_scale = 1.0 / math.sqrt(D)
    need = 0 if workspace is not None else \
        paged_append_decode_attend_host_workspace_bytes(cache, k_new.dtype, n_new, q.dtype, Hq, n_q, max_kv_len, chunk)
    out, workspace = _host_out_ws(q, cache.planes["k"]["payload"].device, need, out, workspace)
    L.check(L.lib().kvq_paged_append_decode_attend_host(
        C.byref(cache.struct), k_new.data_ptr(), v_new.data_ptr(), _DTYPES[k_new.dtype], n_new, q.data_ptr(),
        _DTYPES[q.dtype], Hq, n_q, seq_lens.data_ptr(), max_kv_len, int(bool(causal)), float(attn_scale), chunk,
        out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)),
        "kvq_paged_append_decode_attend_host")
    return out
