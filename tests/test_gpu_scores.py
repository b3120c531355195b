"""Exact integer-domain scores of the Hadamard layouts, taken from the kernels that run.

tract discussion #2402, "What's done": the body score is the integer dot int8(q_rot) . int4(k_rot)
-> i32, an exact integer, so every summation order gives the same value. The score-capture call
(kvq_debug_attend_scores_i32) runs the ordinary attention launches; the tensor-core kernel that
scores the body (the per-warp decode kernel for int4 and int2, the row-side prefill kernel, the
tcgen05 prefill kernel) also writes the integer it holds before scaling. Those integers and the int8 query scales must equal the
oracle's bit for bit; the attention output of the same call is checked at the usual tolerance.

An entry (row, t) is checked wherever row sees t (t <= its causal limit). Elsewhere the kernels may
still have computed it (a tile's rows share their tokens): then it must also equal the oracle, else
it keeps the fill value.
"""
import numpy as np
import pytest
import torch

import sub_byte_quantized_gb300 as kvq
from oracle import attention as OA
from synth import WORKLOADS, make_inputs
from tests.gpu_helpers import check_close, fill_both

pytestmark = pytest.mark.gpu

FILL = -(2 ** 31)


def _limits(n_q, kv_len, causal, q_pos0):
    return np.minimum(kv_len - 1, q_pos0 + np.arange(n_q)) if causal else np.full(n_q, kv_len - 1)


def check_scores(w, kv_len, n_q, fill, chunk=0, causal=None, q_pos0=None):
    causal = w.causal if causal is None else causal
    q_pos0 = (kv_len - n_q if causal else 0) if q_pos0 is None else q_pos0
    inp = make_inputs(w, kv_len=kv_len, n_q=n_q)
    dc, oc, d = fill_both(w, inp, fill=fill)
    out, scores, s_q = kvq.debug_attend_scores_i32(dc, d["q"], kv_len, causal=causal, q_pos0=q_pos0,
                                                   attn_scale=w.alpha, chunk=chunk, fill=FILL)
    torch.cuda.synchronize()
    ref_out, ref_scores = oc.attend(inp["q"], w.alpha, kv_len, causal=causal, q_pos0=q_pos0)
    _, ref_sq, _ = OA.prep_q_hadamard(inp["q"])
    got_sq = s_q.cpu().numpy()
    assert np.array_equal(got_sq.view(np.uint32), ref_sq.view(np.uint32)), "int8 query scales differ"
    got = scores.cpu().numpy().astype(np.int64)
    n_body = ref_scores.shape[-1]
    assert got.shape == ref_scores.shape
    lim = _limits(n_q, kv_len, causal, q_pos0)
    seen = np.arange(n_body)[None, :] <= lim[:, None]                      # [n_q][n_body]
    seen = np.broadcast_to(seen, got.shape)
    if not np.array_equal(got[seen], ref_scores[seen]):
        idx = tuple(np.argwhere(seen & (got != ref_scores))[0])
        raise AssertionError(f"{w.name}: integer score at {idx}: got {got[idx]} want {ref_scores[idx]}")
    rest = ~seen
    assert np.all((got[rest] == ref_scores[rest]) | (got[rest] == FILL)), "a score outside the visible set is wrong"
    check_close(out.cpu().numpy(), ref_out, w.name)
    return int(seen.sum())


def test_c3_decode_full_size():
    """The C3 Hadamard decode step at full size: B8, 16 query / 8 kv heads (GQA 2), one row,
    4096 tokens with the 64-token window (per-warp decode kernel)."""
    w = WORKLOADS["c3_had_int4_decode"]
    n = check_scores(w, w.kv_len, 1, w.n_fill)
    assert n == 8 * 16 * (4096 - 64)


def test_c3_prefill_chunk():
    """The C3 causal prefill chunk: 256 rows appended at 3840 over 4096 tokens with the 64-token
    window (row-side kernel, four 64-row blocks per kv head); batch 2 of the 8 to keep the oracle
    quick (the kernels see the same per-head work)."""
    w = WORKLOADS["c3_had_int4_prefill"].scaled(batch=2)
    check_scores(w, 4096, 256, 3840)


def test_int2_wide_window_decode():
    """Hadamard int2 body with a 256-token exact-f32 window, decode (per-warp decode kernel)."""
    w = WORKLOADS["c3_had_int2_decode_w256"].scaled(batch=2)
    check_scores(w, 4096, 1, 4095)


def test_int2_prefill_rows():
    """Hadamard int2, 96 causal rows (two row blocks, the second ragged)."""
    w = WORKLOADS["c3_had_int2_decode_w256"].scaled(batch=1, causal=True, n_recent=32)
    check_scores(w, 1500, 96, 1404)


@pytest.mark.parametrize("layout", ["had_int4", "had_int2"])
@pytest.mark.parametrize("kv_len,n_q,chunk", [(1000, 1, 64), (1000, 1, 0), (777, 3, 192), (1000, 40, 128)])
def test_ragged_final_stage(layout, kv_len, n_q, chunk):
    """Bodies that end inside a stage (the zero-filled tail rows must not produce scores), odd
    chunk counts, several query rows (GQA 2 x n_q), causal rows."""
    w = WORKLOADS["c3_had_int4_decode"].scaled(layout=layout, batch=2, n_recent=24, causal=n_q > 1)
    check_scores(w, kv_len, n_q, kv_len - n_q, chunk=chunk)


def test_capture_refused_elsewhere():
    """Score capture exists only where a tensor-core kernel scores a Hadamard body."""
    w = WORKLOADS["c1_q4_0_tiny"]
    inp = make_inputs(w)
    dc, _, d = fill_both(w, inp)
    with pytest.raises(kvq.KvqError) as e:
        kvq.debug_attend_scores_i32(dc, d["q"], 512)
    assert e.value.status == 4
