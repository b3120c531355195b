"""Store kernels vs the oracle: packed bytes, scales, zero-points and the f32 window bit-exact."""
import zlib

import numpy as np
import pytest
import torch

import sub_byte_quantized_gb300 as kvq
from oracle import attention as OA
from synth import WORKLOADS, make_inputs
from tests.gpu_helpers import fill_both, planes_equal

pytestmark = pytest.mark.gpu

LAYOUTS = ["q4_0", "q6_0", "had_int4", "asym4_g32", "q8_0", "had_int2"]
HADAMARD = ("had_int4", "had_int2")


def special_rows(rng, n, D):
    """Rows that stress the quantisers: zeros, -0.0, exact half steps, fp16 underflow and
    overflow of the scale, a single spike, constant groups."""
    x = (rng.standard_t(4, (n, D)) * rng.uniform(0.1, 4, (n, 1))).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2] = (np.arange(D) % 17 - 8 + 0.5).astype(np.float32)          # halves on a grid of step 1
    x[3] = 1e-9 * rng.standard_normal(D).astype(np.float32)            # scale underflows fp16
    x[4] = 3e6 * rng.standard_normal(D).astype(np.float32)             # scale saturates at 65504
    x[5] = 0.0
    x[5, 7] = -5.0                                                      # single spike
    x[6] = 0.75                                                         # constant groups
    x[7, :32] = np.linspace(-1, 1, 32, dtype=np.float32)
    return x


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_store_bit_exact(layout, D, dtype):
    rng = np.random.default_rng(zlib.crc32(f"{layout}/{D}/{dtype}".encode()))
    B, H, cap, pos0, n = 2, 3, 64, 5, 37
    k = special_rows(rng, B * H * n, D).reshape(B, H, n, D)
    v = rng.standard_t(3, (B, H, n, D)).astype(np.float32)
    v[:, :, :, 9] *= 30
    if dtype == "bf16":
        k = (torch.from_numpy(k).to(torch.bfloat16)).float().numpy()
        v = (torch.from_numpy(v).to(torch.bfloat16)).float().numpy()
        tdt = torch.bfloat16
    elif dtype == "f16":
        k = np.clip(k, -6e4, 6e4).astype(np.float16).astype(np.float32)
        v = v.astype(np.float16).astype(np.float32)
        tdt = torch.float16
    else:
        tdt = torch.float32
    n_recent = 16 if layout in HADAMARD else 0
    dc = kvq.KVCache(layout, B, H, D, cap, n_recent=n_recent)
    oc = OA.OracleCache(layout, B, H, D, cap, n_recent=n_recent)
    kd = torch.from_numpy(k).to(tdt).cuda()
    vd = torch.from_numpy(v).to(tdt).cuda()
    kvq.store(dc, kd, vd, pos0)
    oc.store(k, v, pos0)
    torch.cuda.synchronize()
    planes_equal(dc, oc)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_store_appends_and_restore_is_identical(layout):
    rng = np.random.default_rng(3)
    B, H, D, cap = 1, 2, 128, 300
    n_recent = 24 if layout in HADAMARD else 0
    x = rng.standard_t(4, (B, H, cap, D)).astype(np.float32)
    y = rng.standard_t(4, (B, H, cap, D)).astype(np.float32)
    dc = kvq.KVCache(layout, B, H, D, cap, n_recent=n_recent)
    oc = OA.OracleCache(layout, B, H, D, cap, n_recent=n_recent)
    xd, yd = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    # ragged appends: 1, 7, 100 (> n_recent), 1, 50
    pos = 0
    for n in (1, 7, 100, 1, 50):
        kvq.store(dc, xd[:, :, pos:pos + n].contiguous(), yd[:, :, pos:pos + n].contiguous(), pos)
        oc.store(x[:, :, pos:pos + n], y[:, :, pos:pos + n], pos)
        pos += n
    torch.cuda.synchronize()
    planes_equal(dc, oc, pos)
    before = {t: dc.planes[t]["payload"].clone() for t in "kv"}
    # storing the same token again writes identical bytes
    kvq.store(dc, xd[:, :, pos - 1:pos].contiguous(), yd[:, :, pos - 1:pos].contiguous(), pos - 1)
    torch.cuda.synchronize()
    for t in "kv":
        assert torch.equal(before[t], dc.planes[t]["payload"])


@pytest.mark.parametrize("name", ["c2_q4_0_llama3_8b", "c4_q6_0_gemma", "c3_had_int4_decode"])
def test_store_workload_sizes_bit_exact(name):
    w = WORKLOADS[name]
    inp = make_inputs(w, kv_len=1024 if w.kv_len > 1024 else None)
    dc, oc, _ = fill_both(w, inp, fill=inp["k"].shape[2] - 1)
    torch.cuda.synchronize()
    planes_equal(dc, oc, inp["k"].shape[2])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["c5_q4_0_llama70b_128k", "c5_asym4_g32_llama70b_128k"])
def test_store_full_128k_sampled(name):
    """Full 128K-token fill + 1-token append in the benchmark's launch shape; sampled rows
    (every quantised row depends only on its own values) compared bit-exactly."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    from tests.gpu_helpers import device_inputs
    d = device_inputs(inp)
    B, H, S, D = inp["k"].shape
    dc = kvq.KVCache(w.layout, B, H, D, S)
    kvq.store(dc, d["k"][:, :, :S - 1].contiguous(), d["v"][:, :, :S - 1].contiguous(), 0)
    kvq.store(dc, d["k"][:, :, S - 1:].contiguous(), d["v"][:, :, S - 1:].contiguous(), S - 1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    toks = np.unique(np.concatenate([rng.integers(0, S, 2000), [0, S - 2, S - 1]]))
    from oracle import quant as Q
    for t, name_ in (("k", "k"), ("v", "v")):
        planes = Q.quantize(w.layout, inp[name_][:, :, toks])
        got_p = dc.planes[t]["payload"][:, :, toks].cpu().numpy()
        assert np.array_equal(got_p, planes["payload"])
        got_s = dc.planes[t]["scale"][:, :, toks].cpu().numpy()
        assert np.array_equal(got_s.view(np.uint16), planes["scale"].view(np.uint16))
        if "zero" in planes:
            assert np.array_equal(dc.planes[t]["zero"][:, :, toks].cpu().numpy().view(np.uint16),
                                  planes["zero"].view(np.uint16))


@pytest.mark.parametrize("layout", ["q4_0+q8_0", "asym4_g32+q6_0", "had_int4+had_int2"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_store_mixed_bit_exact(layout, dtype):
    """A mixed K/V cache: one launch per plane, each plane bit-identical to the oracle's."""
    rng = np.random.default_rng(zlib.crc32(f"{layout}/{dtype}".encode()))
    B, H, D, cap, pos0, n = 2, 3, 128, 64, 5, 37
    k = special_rows(rng, B * H * n, D).reshape(B, H, n, D)
    v = rng.standard_t(3, (B, H, n, D)).astype(np.float32)
    tdt = torch.float32
    if dtype == "bf16":
        k = torch.from_numpy(k).to(torch.bfloat16).float().numpy()
        v = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
        tdt = torch.bfloat16
    n_recent = 16 if layout.startswith("had") else 0
    dc = kvq.KVCache(layout, B, H, D, cap, n_recent=n_recent)
    oc = OA.OracleCache(layout, B, H, D, cap, n_recent=n_recent)
    kvq.store(dc, torch.from_numpy(k).to(tdt).cuda(), torch.from_numpy(v).to(tdt).cuda(), pos0)
    oc.store(k, v, pos0)
    torch.cuda.synchronize()
    planes_equal(dc, oc)
