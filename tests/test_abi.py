"""The C ABI library loads and exports every entry point include/kvq.h declares; host-side
validation rejects bad arguments before touching the device (no GPU needed for these)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    from sub_byte_quantized_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from sub_byte_quantized_gb300.build import build_library
        build_library()
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 11
    from sub_byte_quantized_gb300._lib import EXPORTS
    assert sorted(EXPORTS) == names
    for n in names:
        assert hasattr(L, n), n


def test_sizes(L):
    assert L.kvq_row_bytes(0, 128) == 64 and L.kvq_row_bytes(1, 256) == 192
    assert L.kvq_row_bytes(2, 128) == 64 and L.kvq_row_bytes(3, 128) == 64
    assert L.kvq_row_bytes(0, 96) == 0 and L.kvq_row_bytes(9, 128) == 0
    out = (C.c_size_t * 4)()
    assert L.kvq_cache_bytes(0, 1, 8, 128, 131072, 0, out) == 0
    # 128K-token Llama-70B layer: 64 B payload + 8 B scales per token per kv head, K or V
    assert out[0] == 8 * 131072 * 64 and out[1] == 8 * 131072 * 8 and out[2] == 0 and out[3] == 0
    assert L.kvq_cache_bytes(2, 8, 8, 128, 4096, 64, out) == 0
    assert out[1] == 8 * 8 * 4096 * 4 and out[3] == 8 * 8 * 64 * 128 * 4
    assert L.kvq_cache_bytes(3, 1, 8, 128, 16, 0, out) == 0 and out[2] == 8 * 16 * 4 * 2


def _cache(layout=0, D=128, cap=64, ptr=4096):
    from sub_byte_quantized_gb300._lib import KvqCache
    return KvqCache(layout, 1, 2, D, cap, 0, ptr, ptr, ptr, ptr, ptr, ptr, None, None)


def test_validation_without_device(L):
    from sub_byte_quantized_gb300._lib import KvqCache
    p = C.byref
    # NULL cache
    assert L.kvq_store_q4_0(None, 16, 16, 1, 1, 0, None) == 1
    assert b"NULL" in L.kvq_last_error()
    # wrong layout for this store
    c = _cache(layout=1)
    assert L.kvq_store_q4_0(p(c), 16, 16, 1, 1, 0, None) == 4
    # capacity
    c = _cache()
    assert L.kvq_store_q4_0(p(c), 16, 16, 1, 10, 60, None) == 3
    # misaligned input
    assert L.kvq_store_q4_0(p(c), 17, 16, 1, 1, 0, None) == 5
    # bad head_dim
    c = _cache(D=96)
    assert L.kvq_store_q4_0(p(c), 16, 16, 1, 1, 0, None) == 2
    # misaligned plane
    c = _cache(ptr=4100)
    assert L.kvq_store_q4_0(p(c), 16, 16, 1, 1, 0, None) == 5
    # n_new == 0 is a no-op
    c = _cache()
    assert L.kvq_store_q4_0(p(c), None, None, 1, 0, 0, None) == 0
    # attention: kv_len 0, beyond capacity, H_q not a multiple of H_kv, causal bounds, workspace
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 1, 0, 0, 0, 1.0, 0, 16, 256, 1 << 20, None) == 1
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 1, 65, 0, 0, 1.0, 0, 16, 256, 1 << 20, None) == 3
    assert L.kvq_decode_attend(p(c), 16, 1, 7, 1, 8, 0, 0, 1.0, 0, 16, 256, 1 << 20, None) == 2
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 4, 8, 1, 6, 1.0, 0, 16, 256, 1 << 20, None) == 1
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 1, 8, 0, 0, 1.0, 100, 16, 256, 1 << 20, None) == 2
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 16, None) == 7
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 128 + 16, 1 << 20, None) == 5
    assert L.kvq_decode_attend(p(c), 16, 1, 8, 1, 8, 0, 0, float("nan"), 0, 16, 256, 1 << 20, None) == 1
    # debug scores only for the Hadamard layout
    assert L.kvq_debug_scores_i32(p(c), 16, 1, 8, 1, 8, 16, 16, None) == 4
    # score capture on the attention path: Hadamard only, outputs present and aligned
    assert L.kvq_debug_attend_scores_i32(p(c), 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 1 << 20, 16, 16, None) == 4
    ch = KvqCache(2, 1, 2, 128, 64, 0, 4096, 4096, 4096, 4096, None, None, None, None)
    assert L.kvq_debug_attend_scores_i32(p(ch), 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 1 << 20, None, 16, None) == 1
    assert L.kvq_debug_attend_scores_i32(p(ch), 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 1 << 20, 20, 16, None) == 5
    assert L.kvq_debug_attend_scores_i32(p(ch), 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 16, 16, 16, None) == 7
    # n_recent belongs to the Hadamard layout only
    c = KvqCache(0, 1, 2, 128, 64, 8, 4096, 4096, 4096, 4096, None, None, None, None)
    assert L.kvq_store_q4_0(p(c), 16, 16, 1, 1, 0, None) == 4
    assert L.kvq_status_string(7) == b"workspace too small"


def test_append_attend_validates_both_parts_first(L):
    """The combined append + attend call rejects a bad argument of either part before launching."""
    p = C.byref
    c = _cache()
    ws = 1 << 20
    # append part: capacity, misaligned k_new, unknown K/V dtype
    assert L.kvq_append_decode_attend(p(c), 16, 16, 1, 10, 60, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws, None) == 3
    assert L.kvq_append_decode_attend(p(c), 17, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws, None) == 5
    assert L.kvq_append_decode_attend(p(c), 16, 16, 9, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws, None) == 1
    # attention part (the append alone is valid): kv_len 0, workspace too small, misaligned q
    assert L.kvq_append_decode_attend(p(c), 16, 16, 1, 1, 7, 16, 1, 8, 1, 0, 0, 0, 1.0, 0, 16, 256, ws, None) == 1
    assert L.kvq_append_decode_attend(p(c), 16, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 16, None) == 7
    assert L.kvq_append_decode_attend(p(c), 16, 16, 1, 1, 7, 20, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws, None) == 5


def test_workspace_size_formula(L):
    c = _cache(cap=131072)
    # rows = 1*8*1, chunks = 256: m + l + o, each region rounded up to 256 bytes
    ws = L.kvq_attend_workspace_bytes(C.byref(c), 8, 1, 131072, 512)
    rows, Cc = 8, 256
    assert ws == 2 * ((rows * Cc * 4 + 255) // 256 * 256) + (rows * Cc * 128 * 4 + 255) // 256 * 256


def test_auto_chunk_is_a_multiple_of_64():
    c = _cache(cap=131072)
    for kv_len in (1, 100, 4096, 131072):
        ws = L_ws = None
        from sub_byte_quantized_gb300 import _lib
        Lb = _lib.lib()
        auto = Lb.kvq_attend_workspace_bytes(C.byref(c), 8, 1, kv_len, 0)
        assert auto > 0
        # the automatic chunk equals one of the explicit multiples of 64
        sizes = {Lb.kvq_attend_workspace_bytes(C.byref(c), 8, 1, kv_len, ch) for ch in range(64, 8193, 64)}
        assert auto in sizes


def _paged(layout=0, D=128, page=64, n_pages=8, mpp=4, ptr=4096, table=4096, n_recent=0):
    from sub_byte_quantized_gb300._lib import KvqPagedCache
    return KvqPagedCache(layout, 2, 2, D, page, n_pages, mpp, n_recent, ptr, ptr, ptr, ptr, ptr, ptr, None, None, table)


def test_paged_sizes(L):
    out = (C.c_size_t * 4)()
    assert L.kvq_paged_cache_bytes(0, 10, 8, 128, 64, 4, 0, out) == 0
    assert out[0] == 10 * 8 * 64 * 64 and out[1] == 10 * 8 * 64 * 8 and out[2] == 0 and out[3] == 0
    assert L.kvq_paged_cache_bytes(2, 10, 8, 128, 64, 4, 16, out) == 0
    assert out[1] == 10 * 8 * 64 * 4 and out[3] == 4 * 8 * 16 * 128 * 4
    assert L.kvq_paged_cache_bytes(3, 3, 2, 256, 128, 1, 0, out) == 0 and out[2] == 3 * 2 * 128 * 8 * 2
    assert L.kvq_paged_cache_bytes(9, 3, 2, 128, 64, 1, 0, out) == 1


def test_paged_validation_without_device(L):
    p = C.byref
    ws = 1 << 20
    # store: page size not a power of two / below 64, NULL table, misaligned table or positions
    for page in (48, 32, 96):
        assert L.kvq_paged_store(p(_paged(page=page)), 16, 16, 1, 1, 16, None) == 2
    assert L.kvq_paged_store(p(_paged(table=None)), 16, 16, 1, 1, 16, None) == 1
    assert L.kvq_paged_store(p(_paged(table=4100)), 16, 16, 1, 1, 16, None) == 5
    assert L.kvq_paged_store(p(_paged()), 16, 16, 1, 1, 20, None) == 5
    assert L.kvq_paged_store(p(_paged()), 16, 16, 1, 1, None, None) == 1
    assert L.kvq_paged_store(p(_paged(n_pages=0)), 16, 16, 1, 1, 16, None) == 1
    # more new rows than a sequence holds (4 pages x 64)
    assert L.kvq_paged_store(p(_paged()), 16, 16, 1, 257, 16, None) == 3
    assert L.kvq_paged_store(p(_paged()), None, None, 1, 0, None, None) == 0
    # n_recent on a non-Hadamard layout
    assert L.kvq_paged_store(p(_paged(n_recent=8)), 16, 16, 1, 1, 16, None) == 4
    # attention: max_kv_len 0 / beyond the sequence capacity, NULL or misaligned seq_lens, workspace
    c = _paged()
    assert L.kvq_paged_decode_attend(p(c), 16, 1, 8, 1, 16, 0, 0, 1.0, 0, 16, 256, ws, None) == 1
    assert L.kvq_paged_decode_attend(p(c), 16, 1, 8, 1, 16, 257, 0, 1.0, 0, 16, 256, ws, None) == 3
    assert L.kvq_paged_decode_attend(p(c), 16, 1, 8, 1, None, 64, 0, 1.0, 0, 16, 256, ws, None) == 1
    assert L.kvq_paged_decode_attend(p(c), 16, 1, 8, 1, 20, 64, 0, 1.0, 0, 16, 256, ws, None) == 5
    assert L.kvq_paged_decode_attend(p(c), 16, 1, 8, 1, 16, 64, 0, 1.0, 0, 16, 256, 16, None) == 7
    assert L.kvq_paged_decode_attend(p(c), 16, 1, 7, 1, 16, 64, 0, 1.0, 0, 16, 256, ws, None) == 2
    # the combined call validates both parts first
    assert L.kvq_paged_append_decode_attend(p(c), 17, 16, 1, 1, 16, 1, 8, 1, 16, 64, 0, 1.0, 0, 16, 256, ws,
                                            None) == 5
    assert L.kvq_paged_append_decode_attend(p(c), 16, 16, 1, 1, 16, 1, 8, 1, 16, 64, 0, 1.0, 0, 16, 256, 16,
                                            None) == 7
    # workspace: the contiguous formula at max_kv_len (rows = 2 sequences x 8 heads, 2 chunks)
    rows, Cc = 16, 2
    assert L.kvq_paged_attend_workspace_bytes(p(c), 8, 1, 256, 128) == \
        2 * ((rows * Cc * 4 + 255) // 256 * 256) + (rows * Cc * 128 * 4 + 255) // 256 * 256
    L.kvq_paged_attend_chunk.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_int32]
    assert L.kvq_paged_attend_chunk(p(c), 8, 1, 256, 0, 128) == 128
    # a ragged batch's total gives a chunk no larger than the max-length assumption's
    big = _paged(n_pages=4096, mpp=2048)
    auto_max = L.kvq_paged_attend_chunk(p(big), 8, 1, 131072, 0, 0)
    auto_tot = L.kvq_paged_attend_chunk(p(big), 8, 1, 131072, 40000, 0)
    assert auto_tot % 64 == 0 and 64 <= auto_tot <= auto_max


def test_mixed_layout_validation(L):
    from sub_byte_quantized_gb300._lib import KvqCache, mixed
    p = C.byref
    ok = KvqCache(mixed(0, 4), 1, 2, 128, 64, 0, 4096, 4096, 4096, 4096, None, None, None, None)
    # a per-layout store refuses a mixed cache (kvq_store takes any layout)
    assert L.kvq_store_q4_0(p(ok), 16, 16, 1, 1, 0, None) == 4
    assert b"kvq_store" in L.kvq_last_error()
    # a rotated K with an unrotated V, an unknown V layout
    bad = KvqCache(mixed(2, 0), 1, 2, 128, 64, 0, 4096, 4096, 4096, 4096, None, None, None, None)
    assert L.kvq_store(p(bad), 16, 16, 1, 1, 0, None) == 1
    bad = KvqCache(mixed(0, 9), 1, 2, 128, 64, 0, 4096, 4096, 4096, 4096, None, None, None, None)
    assert L.kvq_store(p(bad), 16, 16, 1, 1, 0, None) == 1
    # an asymmetric V plane needs its zero-point plane even when K has none
    za = KvqCache(mixed(0, 3), 1, 2, 128, 64, 0, 4096, 4096, 4096, 4096, None, None, None, None)
    assert L.kvq_store(p(za), 16, 16, 1, 1, 0, None) == 1
    za = KvqCache(mixed(0, 3), 1, 2, 128, 64, 0, 4096, 4096, 4096, 4096, None, 4096, None, None)
    assert L.kvq_store(p(za), 16, 16, 1, 10, 60, None) == 3          # valid planes, capacity error


def test_paged_plan_chunk(L):
    """The planner: the shortest multiple of 64 whose equal per-sequence chunks fit one wave."""
    import numpy as np
    p = C.byref
    L.kvq_paged_attend_plan_chunk.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p]
    c = _paged(mpp=2048, n_pages=8192)
    lens = np.array([131072, 5], np.int32)
    ch = L.kvq_paged_attend_plan_chunk(p(c), 8, 1, 1, lens.ctypes.data)
    assert ch % 64 == 0 and 64 <= ch <= 8192
    # fewer tokens never need a longer chunk
    small = np.array([4096, 5], np.int32)
    assert L.kvq_paged_attend_plan_chunk(p(c), 8, 1, 1, small.ctypes.data) <= ch
    assert L.kvq_paged_attend_plan_chunk(p(c), 8, 1, 1, None) == 0


def _r256(x):
    return (x + 255) // 256 * 256


def test_host_call_workspace_and_validation(L):
    """The host-buffer calls: workspace = the attention partials + device staging of k_new, v_new,
    q, out (and seq_lens); every argument is rejected before anything is enqueued."""
    p = C.byref
    c = _cache()                                           # batch 1, 2 kv heads, D 128, capacity 64
    att = L.kvq_attend_workspace_bytes(p(c), 8, 1, 64, 64)
    kvb, qb, ob = 1 * 2 * 3 * 128 * 2, 1 * 8 * 1 * 128 * 2, 1 * 8 * 1 * 128 * 4   # 3 bf16 rows, bf16 q
    assert L.kvq_append_decode_attend_host_workspace_bytes(p(c), 1, 3, 1, 8, 1, 64, 64) == \
        _r256(att) + 2 * _r256(kvb) + _r256(qb) + _r256(ob)
    # f32 q doubles the q staging; n_new 0 stages no rows; invalid dtypes size nothing
    assert L.kvq_append_decode_attend_host_workspace_bytes(p(c), 1, 0, 0, 8, 1, 64, 64) == \
        _r256(att) + _r256(2 * qb) + _r256(ob)
    assert L.kvq_append_decode_attend_host_workspace_bytes(p(c), 7, 3, 1, 8, 1, 64, 64) == 0
    assert L.kvq_append_decode_attend_host_workspace_bytes(p(c), 1, 3, 5, 8, 1, 64, 64) == 0
    ws = 1 << 20
    # NULL host q / out / k_new, unknown dtype, workspace too small or misaligned, capacity, shape
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 1, 7, None, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws,
                                           None) == 1
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, None, 256, ws,
                                           None) == 1
    assert L.kvq_append_decode_attend_host(p(c), None, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws,
                                           None) == 1
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 9, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws,
                                           None) == 1
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, 300,
                                           None) == 7
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 272, ws,
                                           None) == 5
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 10, 60, 16, 1, 8, 1, 8, 0, 0, 1.0, 0, 16, 256, ws,
                                           None) == 3
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 1, 7, 16, 1, 7, 1, 8, 0, 0, 1.0, 0, 16, 256, ws,
                                           None) == 2
    assert L.kvq_append_decode_attend_host(p(c), 16, 16, 1, 1, 7, 16, 1, 8, 1, 8, 0, 0, float("inf"), 0, 16, 256,
                                           ws, None) == 1
    # paged: NULL host seq_lens, staging sized with the lengths
    pc = _paged()
    att = L.kvq_paged_attend_workspace_bytes(p(pc), 8, 1, 256, 128)
    kvb, qb, ob = 2 * 2 * 1 * 128 * 2, 2 * 8 * 1 * 128 * 2, 2 * 8 * 1 * 128 * 4
    assert L.kvq_paged_append_decode_attend_host_workspace_bytes(p(pc), 1, 1, 1, 8, 1, 256, 128) == \
        _r256(att) + 2 * _r256(kvb) + _r256(qb) + _r256(ob) + 256
    assert L.kvq_paged_append_decode_attend_host(p(pc), 16, 16, 1, 1, 16, 1, 8, 1, None, 64, 0, 1.0, 0, 16, 256, ws,
                                                 None) == 1
    assert L.kvq_paged_append_decode_attend_host(p(pc), 16, 16, 1, 1, 16, 1, 8, 1, 16, 64, 0, 1.0, 0, 16, 256, 300,
                                                 None) == 7
    assert L.kvq_paged_append_decode_attend_host(p(pc), 16, 16, 1, 1, 16, 1, 8, 1, 16, 300, 0, 1.0, 0, 16, 256, ws,
                                                 None) == 3


def test_decode_chunk_follows_the_kernel(L):
    """The automatic chunk of a decode shape follows the phase-1 kernel that will run: the
    per-warp tensor-core kernel (Q4_0, Q8_0, Q4_0 keys + Q8_0 values, Hadamard int4) shares one
    rule; the asymmetric layout's CTA kernel and the row-side kernel (Hadamard int2) have others.
    Host-only: with no device the SM count defaults, the rules are the same."""
    from sub_byte_quantized_gb300._lib import KvqCache, mixed
    p = C.byref

    def chunk(layout, n_recent=0, rows=8):
        zero = 4096 if layout == 3 else None
        ring = 4096 if n_recent else None
        c = KvqCache(layout, 1, 8, 128, 131072, n_recent, 4096, 4096, 4096, 4096, zero, zero, ring, ring)
        return L.kvq_attend_chunk(p(c), 8 * rows, 1, 131072, 0)

    # the SM count the library sizes for: the device's, else its default of 148
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    up = lambda x, m: -(-x // m) * m
    # per-warp kernel: 12 resident warps per SM, each warp's slice whole 32-token stages, 4 warps per chunk
    per_warp = chunk(0)
    assert per_warp == 4 * up(-(-8 * 131072 // (12 * sms)), 32)
    assert chunk(4) == per_warp                      # Q8_0 on the per-warp kernel
    assert chunk(mixed(0, 4)) == per_warp            # Q4_0 keys + Q8_0 values
    assert chunk(3) != per_warp                      # asymmetric: one chunk per resident CTA
    # Hadamard int2: row-side kernel, decode form: one chunk per resident CTA (3 per SM) of the body
    # (the window is scored in phase 2)
    assert chunk(5, n_recent=256) == up(-(-(131072 - 256) // (3 * sms // 8)), 64)
    # more than eight rows per kv head leave the per-warp kernel
    assert chunk(4, rows=16) != chunk(4, rows=8)


def test_missing_library_fails_loudly(tmp_path):
    """Without libkvq.so the package raises on the first call: there is no CPU path to fall back to."""
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from sub_byte_quantized_gb300 import _lib\n"
        "_lib.LIB_PATH = %r\n"
        "import sub_byte_quantized_gb300 as kvq, torch\n"
        "try:\n"
        "    kvq.row_bytes('q4_0', 128)\n"
        "except RuntimeError as e:\n"
        "    print('raised:', 'missing' in str(e))\n"
        "else:\n"
        "    print('no error')\n"
    ) % (ROOT, str(tmp_path / "libkvq.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "raised: True" in r.stdout
