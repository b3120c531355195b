"""Host-buffer append + attend calls: with host k_new, v_new, q (pinned or pageable) the result and
the stored cache bytes are bit-identical to the device-buffer call on the same inputs, and within
|gpu - oracle| <= 2e-3 + 1e-3 * |oracle| of the oracle."""
import numpy as np
import pytest
import torch

import sub_byte_quantized_gb300 as kvq
from oracle.paged import OraclePagedCache
from synth import WORKLOADS, make_inputs
from tests.gpu_helpers import check_close, device_inputs, fill_both

pytestmark = pytest.mark.gpu


def _planes_equal(a, b):
    for t in ("k", "v"):
        for name, x in a.planes[t].items():
            assert torch.equal(x, b.planes[t][name]), f"{t} {name} differs"


@pytest.mark.parametrize("layout,n_recent,pinned", [("q4_0", 0, True), ("had_int4", 32, False),
                                                    ("q8_0", 0, True), ("asym4_g32", 0, False)])
def test_host_call_matches_device_call(layout, n_recent, pinned):
    w = WORKLOADS["c2_q4_0_llama3_8b"].scaled(layout=layout, batch=2, n_kv_heads=2, n_q_heads=8, n_recent=n_recent)
    inp = make_inputs(w, kv_len=700, n_q=1)
    B, H, S, D = inp["k"].shape
    n_new = 3
    fill = S - n_new
    dc, oc, d = fill_both(w, inp, fill=fill)                # device cache holds all S tokens
    dc2, _, _ = fill_both(w, inp, fill=fill)
    # rewind: both device caches re-append the last n_new rows through the two call forms
    kn, vn = d["k"][:, :, fill:].contiguous(), d["v"][:, :, fill:].contiguous()
    ref_dev = kvq.append_decode_attend(dc, kn, vn, fill, d["q"], S, attn_scale=w.alpha)
    hk, hv, hq = kn.cpu(), vn.cpu(), d["q"].cpu()
    if pinned:
        hk, hv, hq = hk.pin_memory(), hv.pin_memory(), hq.pin_memory()
    got = kvq.append_decode_attend_host(dc2, hk, hv, fill, hq, S, attn_scale=w.alpha)
    torch.cuda.synchronize()
    assert not got.is_cuda
    assert torch.equal(got, ref_dev.cpu())
    _planes_equal(dc, dc2)
    r = oc.attend(inp["q"], w.alpha, S)
    check_close(got.numpy(), r[0] if isinstance(r, tuple) else r, f"host call {layout}")


@pytest.mark.parametrize("layout", ["q4_0", "had_int4"])
def test_host_call_back_to_back_inputs(layout):
    """k_new, v_new and q as consecutive views of one pinned allocation (the call then moves them with
    one copy): the same result and stored bytes as the device-buffer call, twice in a row with
    different inputs in the same buffer."""
    w = WORKLOADS["c2_q4_0_llama3_8b"].scaled(layout=layout, batch=2, n_kv_heads=2, n_q_heads=8,
                                              n_recent=16 if layout == "had_int4" else 0)
    inp = make_inputs(w, kv_len=600, n_q=1)
    S = inp["k"].shape[2]
    n_new = 2
    fill = S - n_new
    dc, oc, d = fill_both(w, inp, fill=fill)
    dc2, _, _ = fill_both(w, inp, fill=fill)
    kn, vn, q = d["k"][:, :, fill:].contiguous(), d["v"][:, :, fill:].contiguous(), d["q"]
    n_k = kn.numel()
    packed = torch.empty(2 * n_k + q.numel(), dtype=kn.dtype).pin_memory()
    hk, hv, hq = packed[:n_k].view(kn.shape), packed[n_k:2 * n_k].view(vn.shape), packed[2 * n_k:].view(q.shape)
    for qq in (q, torch.flip(q, dims=[1]).contiguous()):
        hk.copy_(kn.cpu())
        hv.copy_(vn.cpu())
        hq.copy_(qq.cpu())
        ref = kvq.append_decode_attend(dc, kn, vn, fill, qq, S, attn_scale=w.alpha)
        got = kvq.append_decode_attend_host(dc2, hk, hv, fill, hq, S, attn_scale=w.alpha)
        torch.cuda.synchronize()
        assert torch.equal(got, ref.cpu())
        _planes_equal(dc, dc2)


def test_host_call_causal_rows_and_no_append():
    """Several causal query rows, and n_new == 0 (a plain attention through the host call)."""
    w = WORKLOADS["c3_had_int4_prefill"].scaled(layout="q4_0", batch=1, n_kv_heads=2, n_q_heads=4, n_recent=0)
    inp = make_inputs(w, kv_len=300, n_q=24)
    S = inp["k"].shape[2]
    dc, oc, d = fill_both(w, inp, fill=S)
    q0 = S - 24
    ref = kvq.decode_attend(dc, d["q"], S, causal=True, q_pos0=q0, attn_scale=w.alpha)
    empty = torch.empty((1, 2, 0, 128), dtype=d["k"].dtype)
    got = kvq.append_decode_attend_host(dc, empty, empty, S, d["q"].cpu(), S, causal=True, q_pos0=q0,
                                        attn_scale=w.alpha)
    assert torch.equal(got, ref.cpu())
    r = oc.attend(inp["q"], w.alpha, S, True, q0)
    check_close(got.numpy(), r[0] if isinstance(r, tuple) else r, "host call causal")


def test_paged_host_call_matches_device_call():
    w = WORKLOADS["c2_q4_0_llama3_8b"].scaled(layout="q4_0", batch=3, n_kv_heads=2, n_q_heads=8)
    lens = np.array([900, 65, 300], np.int64)
    S = int(lens.max())
    inp = make_inputs(w, kv_len=S, n_q=1)
    B, H, _, D = inp["k"].shape
    page, mpp = 64, -(-S // 64)
    table = np.random.default_rng(3).permutation(B * mpp).reshape(B, mpp)
    d = device_inputs(inp)
    n_new = 2
    pools = []
    for _ in range(2):
        pc = kvq.PagedKVCache("q4_0", B, H, D, page, B * mpp, mpp)
        pc.set_block_table(table)
        pos = torch.zeros(B, dtype=torch.int32, device="cuda")
        kvq.paged_store(pc, d["k"][:, :, :S - n_new].contiguous(), d["v"][:, :, :S - n_new].contiguous(), pos)
        pools.append(pc)
    # the appended rows sit at each sequence's end: seq_lens[b] - n_new + j
    kt = torch.stack([d["k"][b, :, int(lens[b]) - n_new:int(lens[b])] for b in range(B)]).contiguous()
    vt = torch.stack([d["v"][b, :, int(lens[b]) - n_new:int(lens[b])] for b in range(B)]).contiguous()
    lens_dev = torch.from_numpy(lens.astype(np.int32)).cuda()
    ref = kvq.paged_append_decode_attend(pools[0], kt, vt, d["q"], lens_dev, S, attn_scale=w.alpha)
    got = kvq.paged_append_decode_attend_host(pools[1], kt.cpu().pin_memory(), vt.cpu().pin_memory(),
                                              d["q"].cpu().pin_memory(), torch.from_numpy(lens.astype(np.int32)),
                                              S, attn_scale=w.alpha)
    torch.cuda.synchronize()
    assert torch.equal(got, ref.cpu())
    _planes_equal(pools[0], pools[1])
    oc = OraclePagedCache("q4_0", B, H, D, page, B * mpp, mpp, table=table)
    oc.store(inp["k"][:, :, :S - n_new], inp["v"][:, :, :S - n_new], np.zeros(B, np.int64))
    oc.store(kt.float().cpu().numpy(), vt.float().cpu().numpy(), lens - n_new)
    check_close(got.numpy(), oc.attend(inp["q"], w.alpha, lens), "paged host call")


@pytest.mark.parametrize("inputs,out_kind", [("pinned", "pageable"), ("pageable", "pinned"),
                                             ("pinned_unaligned", "pinned"), ("pinned", "pinned")])
def test_host_call_buffer_kinds(inputs, out_kind):
    """Pinned, 16-byte aligned host buffers are used in place (the store reads k_new / v_new and the
    reduce writes out over the host link); pageable or unaligned ones go through the workspace
    staging. Every mix gives the device-buffer call's result and stored bytes exactly."""
    w = WORKLOADS["c2_q4_0_llama3_8b"].scaled(layout="q4_0", batch=2, n_kv_heads=2, n_q_heads=8)
    inp = make_inputs(w, kv_len=500, n_q=1)
    S = inp["k"].shape[2]
    n_new = 2
    fill = S - n_new
    dc, _, d = fill_both(w, inp, fill=fill)
    dc2, _, _ = fill_both(w, inp, fill=fill)
    kn, vn, q = d["k"][:, :, fill:].contiguous(), d["v"][:, :, fill:].contiguous(), d["q"]
    if inputs == "pinned_unaligned":
        # views 2 bf16 elements (4 bytes) into pinned allocations: not 16-byte aligned
        hk = torch.empty(kn.numel() + 2, dtype=kn.dtype).pin_memory()[2:].view(kn.shape)
        hv = torch.empty(vn.numel() + 2, dtype=vn.dtype).pin_memory()[2:].view(vn.shape)
        hk.copy_(kn.cpu())
        hv.copy_(vn.cpu())
        hq = q.cpu().pin_memory()
    else:
        hk, hv, hq = kn.cpu(), vn.cpu(), q.cpu()
        if inputs == "pinned":
            hk, hv, hq = hk.pin_memory(), hv.pin_memory(), hq.pin_memory()
    out = torch.empty(q.shape, dtype=torch.float32)
    if out_kind == "pinned":
        out = out.pin_memory()
    ref = kvq.append_decode_attend(dc, kn, vn, fill, q, S, attn_scale=w.alpha)
    got = kvq.append_decode_attend_host(dc2, hk, hv, fill, hq, S, attn_scale=w.alpha, out=out)
    torch.cuda.synchronize()
    assert got.data_ptr() == out.data_ptr()
    assert torch.equal(got, ref.cpu())
    _planes_equal(dc, dc2)
