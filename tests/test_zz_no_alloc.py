"""The allocation-free attention entry point (kvq_decode_attend_static), called through the C
ABI, gives the same outputs as kvq_decode_attend with a caller workspace, on two calls in a row.
Both run the same kernels with the same chunking, only the partials' address differs, so the
outputs must be bitwise equal (the parity tolerance would hide a scratch layout or offset bug).

The entry point serves callers that cannot allocate device memory themselves (e.g. a plugin
inside an engine that owns the device memory pool); its partials live in a device array built
into the library. This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes as C

import pytest
import torch

import sub_byte_quantized_gb300 as kvq
from sub_byte_quantized_gb300 import _lib
from synth import WORKLOADS, make_inputs
from tests.gpu_helpers import fill_both

pytestmark = pytest.mark.gpu


def _static_call(dc, q, kv_len, alpha, out, chunk=0, causal=0, q_pos0=0):
    L = _lib.lib()
    st = L.kvq_decode_attend_static(C.byref(dc.struct), q.data_ptr(), _lib.KVQ_BF16 if q.dtype == torch.bfloat16
                                    else _lib.KVQ_F32, q.shape[1], q.shape[2], kv_len, causal, q_pos0,
                                    float(alpha), chunk, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st


# the Hadamard case has a 64-token exact-f32 window, scored in phase 2 from the same scratch
@pytest.mark.parametrize("name,kv_len", [("c2_q4_0_llama3_8b", 3000), ("c3_had_int4_decode", 1100)])
def test_static_matches_workspace_entry_point_twice(name, kv_len):
    w = WORKLOADS[name].scaled(batch=2)
    inp = make_inputs(w, kv_len=kv_len)
    dc, _, d = fill_both(w, inp)
    q2 = torch.flip(d["q"], dims=[1]).contiguous()       # a second, different query batch
    for q in (d["q"], q2):                                # two calls in a row share the scratch
        ref = kvq.decode_attend(dc, q, kv_len, attn_scale=w.alpha)
        out = torch.full_like(ref, float("nan"))
        st = _static_call(dc, q, kv_len, w.alpha, out)
        torch.cuda.synchronize()
        assert st == 0, _lib.lib().kvq_last_error()
        assert torch.equal(out, ref)


def test_static_rejects_calls_beyond_its_scratch():
    w = WORKLOADS["c5_q4_0_llama70b_128k"]
    B, H, D = 1, 8, 128
    dc = kvq.KVCache("q4_0", B, H, D, 131072)
    q = torch.zeros((B, 64 * 8, 1, D), dtype=torch.bfloat16, device="cuda")   # 8x the query heads
    out = torch.empty((B, 64 * 8, 1, D), dtype=torch.float32, device="cuda")
    need = kvq.attend_workspace_bytes(dc, 64 * 8, 1, 131072, 64)
    assert need > _lib.STATIC_SCRATCH_BYTES
    st = _static_call(dc, q, 131072, w.alpha, out, chunk=64)
    assert st == 7 and b"scratch" in _lib.lib().kvq_last_error()
