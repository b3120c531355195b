"""Paged KV pool through the C ABI vs the paged oracle: stored pool bytes bit-exact, attention
within |gpu - oracle| <= 2e-3 + 1e-3 * |oracle|, per-sequence lengths (ragged, empty, shorter
than the causal query block), permuted block tables, every phase-1 kernel family; and bitwise
invariants against the contiguous path and the two-call form.
"""
import math

import numpy as np
import pytest
import torch

import sub_byte_quantized_gb300 as kvq
from oracle.paged import OraclePagedCache
from synth import WORKLOADS, make_inputs
from tests.gpu_helpers import check_close, to_device

pytestmark = pytest.mark.gpu


def _tail(x, lens, n_new):
    """[B][H][n_new][D]: sequence b's tokens lens[b] - n_new .. lens[b] - 1 (zero rows before 0)."""
    B, H, S, D = x.shape
    out = np.zeros((B, H, n_new, D), x.dtype)
    for b in range(B):
        for j in range(n_new):
            t = int(lens[b]) - n_new + j
            if 0 <= t < S:
                out[b, :, j] = x[b, :, t]
    return out


def _dev(inp, arr_name, arr):
    """The device tensor of a host slice of one input, in the workload's dtype (the float32 values
    are exact in it, so the bits are those of the input)."""
    return to_device(arr, None, "f32", "cuda") if inp["dtype"] == "f32" else _bf16(arr)


def _bf16(arr):
    from synth import bf16_bits_from_f32
    bits = bf16_bits_from_f32(np.ascontiguousarray(arr, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def build(w, lens, page, n_q, n_new=5, seed=0, extra_pages=3, fused=False, chunk=0, q_dtype=None):
    """Fill a device pool and an oracle pool identically (bulk per sequence, then an n_new-token
    append at each sequence's end), attend, and return everything."""
    lens = np.asarray(lens, np.int64)
    S = max(int(lens.max()), 1)
    inp = make_inputs(w, kv_len=S, n_q=n_q)
    B, H, _, D = inp["k"].shape
    mpp = -(-S // page)
    n_pages = B * mpp + extra_pages
    rng = np.random.default_rng(1234 + seed)
    table = rng.permutation(n_pages)[:B * mpp].reshape(B, mpp)
    n_recent = w.n_recent
    dc = kvq.PagedKVCache(w.layout, B, H, D, page, n_pages, mpp, n_recent=n_recent)
    dc.set_block_table(table)
    oc = OraclePagedCache(w.layout, B, H, D, page, n_pages, mpp, n_recent, table=table)
    fill = np.maximum(lens - n_new, 0)
    for b in range(B):
        if fill[b]:
            pos = np.full(B, dc.capacity, np.int32)
            pos[b] = 0
            kk, vv = inp["k"][:, :, :fill[b]], inp["v"][:, :, :fill[b]]
            kvq.paged_store(dc, _dev(inp, "k", kk), _dev(inp, "v", vv), torch.from_numpy(pos).cuda())
            oc.store(kk, vv, pos)
    kt, vt = _tail(inp["k"], lens, n_new), _tail(inp["v"], lens, n_new)
    lens_dev = torch.from_numpy(lens.astype(np.int32)).cuda()
    q = _dev(inp, "q", inp["q"])
    qf = inp["q"]
    if q_dtype == "f32":
        q = q.float().contiguous()
    elif q_dtype == "f16":
        q = q.half().contiguous()
        qf = q.float().cpu().numpy()
    max_len = int(lens.max()) if lens.max() > 0 else 1
    if fused:
        out = kvq.paged_append_decode_attend(dc, _dev(inp, "k", kt), _dev(inp, "v", vt), q, lens_dev, max_len,
                                             causal=w.causal, attn_scale=w.alpha, chunk=chunk)
    else:
        kvq.paged_store(dc, _dev(inp, "k", kt), _dev(inp, "v", vt), (lens_dev - n_new).contiguous())
        out = kvq.paged_decode_attend(dc, q, lens_dev, max_len, causal=w.causal, attn_scale=w.alpha, chunk=chunk)
    oc.store(kt, vt, lens - n_new)
    torch.cuda.synchronize()
    ref = oc.attend(qf, w.alpha, lens, causal=w.causal)
    return dc, oc, out, ref


def pool_equal(dc, oc):
    for t in ("k", "v"):
        dp, op = dc.planes[t], oc.planes[t]
        for name in ("payload", "scale", "zero"):
            if name in op:
                got = dp[name].cpu().numpy()
                assert np.array_equal(got.view(np.uint8), op[name].view(np.uint8)), f"{t} {name} differs"
        if "ring" in op:
            assert np.array_equal(dp["recent"].cpu().numpy().view(np.uint32), op["ring"].view(np.uint32)), \
                f"{t} ring differs"


def _decode_w(layout, D=128, gqa=4, n_recent=0, causal=False):
    return WORKLOADS["c2_q4_0_llama3_8b"].scaled(layout=layout, head_dim=D, batch=4, n_kv_heads=2,
                                                 n_q_heads=2 * gqa, n_recent=n_recent, causal=causal)


@pytest.mark.parametrize("layout,D,page,chunk,n_recent", [
    ("q4_0", 128, 64, 0, 0),
    ("q4_0", 128, 256, 192, 0),
    ("had_int4", 128, 64, 0, 32),
    ("had_int4", 128, 128, 128, 0),
    ("had_int4", 256, 64, 0, 16),        # CUDA-core path with the query-prep kernel
    ("asym4_g32", 128, 64, 0, 0),        # 128-token stages over two 64-token pages
    ("asym4_g32", 128, 128, 192, 0),     # stages starting mid-page
    ("q6_0", 256, 128, 0, 0),
    ("q6_0", 128, 64, 128, 0),
    ("q8_0", 128, 64, 0, 0),
    ("had_int2", 128, 64, 0, 128),
    ("q4_0+q8_0", 128, 64, 0, 0),         # mixed K/V precision
])
def test_paged_decode(layout, D, page, chunk, n_recent):
    """Decode (one query row, GQA 4) over ragged sequences, one of them empty, one shorter than a
    page, one ending exactly on a page boundary; permuted pages with spares in the pool."""
    gqa = 4 if layout != "q6_0" else 2
    w = _decode_w(layout, D, gqa, n_recent)
    dc, oc, out, ref = build(w, [1000, 333, 0, 64], page, n_q=1, chunk=chunk)
    pool_equal(dc, oc)
    check_close(out.cpu().numpy(), ref, f"paged {layout}")
    assert not out[2].any()                               # the empty sequence


@pytest.mark.parametrize("layout,n_recent,q_dtype", [
    ("had_int4", 16, None), ("q4_0", 0, None), ("asym4_g32", 0, "f16"), ("q6_0", 0, None), ("q4_0", 0, "f32"),
])
def test_paged_prefill_rows(layout, n_recent, q_dtype):
    """Causal prefill blocks (40 rows x GQA 2) at each sequence's end; one sequence shorter than the
    block (its first rows see nothing), one empty. Row-side tensor-core kernel for Hadamard /
    Q4_0 / asym with 16-bit queries, the CUDA-core kernel otherwise."""
    w = WORKLOADS["c3_had_int4_prefill"].scaled(layout=layout, batch=4, n_kv_heads=2, n_q_heads=4,
                                                n_recent=n_recent)
    dc, oc, out, ref = build(w, [300, 150, 20, 0], 64, n_q=40, n_new=40, chunk=64, q_dtype=q_dtype)
    pool_equal(dc, oc)
    check_close(out.cpu().numpy(), ref, f"paged prefill {layout}")


def test_paged_many_rows_reduce():
    """Enough rows for phase 2's one-warp-per-row form, with per-sequence limits."""
    w = WORKLOADS["c3_had_int4_prefill"].scaled(layout="q4_0", batch=4, n_kv_heads=4, n_q_heads=16, n_recent=0)
    dc, oc, out, ref = build(w, [300, 80, 41, 299], 64, n_q=80, n_new=80, chunk=64)
    check_close(out.cpu().numpy(), ref, "paged many rows")


@pytest.mark.parametrize("layout", ["q4_0", "had_int4", "asym4_g32", "q6_0", "q8_0", "q4_0+q8_0"])
def test_paged_append_attend_matches_two_calls(layout):
    """paged_append_decode_attend == paged_store + paged_decode_attend, bit for bit."""
    D = 256 if layout == "q6_0" else 128
    w = _decode_w(layout, D, 2 if layout == "q6_0" else 4, 32 if layout == "had_int4" else 0)
    a = build(w, [700, 129, 64, 1], 64, n_q=1, fused=False)
    b = build(w, [700, 129, 64, 1], 64, n_q=1, fused=True)
    pool_equal(b[0], b[1])
    assert torch.equal(a[2], b[2])
    check_close(b[2].cpu().numpy(), b[3], f"paged fused {layout}")


@pytest.mark.parametrize("layout", ["q4_0", "had_int4", "asym4_g32", "q6_0", "q8_0", "q4_0+q8_0"])
def test_paged_equals_contiguous_bitwise(layout):
    """With equal lengths, a permuted paged pool gives the contiguous cache's output bit for bit
    (same kernels, same chunking: only the row addresses differ)."""
    D = 256 if layout == "q6_0" else 128
    n_recent = 32 if layout == "had_int4" else 0
    w = _decode_w(layout, D, 2 if layout == "q6_0" else 4, n_recent)
    S = 900
    inp = make_inputs(w, kv_len=S, n_q=1)
    B, H, _, _ = inp["k"].shape
    k, v, q = _dev(inp, "k", inp["k"]), _dev(inp, "v", inp["v"]), _dev(inp, "q", inp["q"])
    cc = kvq.KVCache(w.layout, B, H, D, S, n_recent=n_recent)
    kvq.store(cc, k, v, 0)
    ref = kvq.decode_attend(cc, q, S, attn_scale=w.alpha, chunk=128)
    page = 64
    mpp = -(-S // page)
    table = np.random.default_rng(5).permutation(B * mpp).reshape(B, mpp)
    pc = kvq.PagedKVCache(w.layout, B, H, D, page, B * mpp, mpp, n_recent=n_recent)
    pc.set_block_table(table)
    kvq.paged_store(pc, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    got = kvq.paged_decode_attend(pc, q, lens, S, attn_scale=w.alpha, chunk=128)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("layout,n_recent", [("q4_0", 0), ("asym4_g32", 0), ("had_int4", 32), ("q8_0", 0)])
def test_paged_planned_chunk_ragged(layout, n_recent):
    """A ragged batch with the chunk from kvq_paged_attend_plan_chunk: each sequence's body in equal
    chunks (its last chunk no longer a sliver), against the oracle."""
    w = _decode_w(layout, 128, 4, n_recent)
    lens = [1000, 130, 64, 777]
    S = max(lens)
    probe = kvq.PagedKVCache(w.layout, 4, 2, 128, 64, 4 * (-(-S // 64)), -(-S // 64), n_recent=n_recent)
    chunk = kvq.paged_attend_plan_chunk(probe, 8, 1, lens)
    assert chunk % 64 == 0 and 64 <= chunk <= 8192
    del probe
    dc, oc, out, ref = build(w, lens, 64, n_q=1, chunk=chunk)
    check_close(out.cpu().numpy(), ref, f"paged planned chunk {layout} ({chunk})")
