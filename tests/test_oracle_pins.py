"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: sizes the pages print
(tests/golden/page_sizes.json), the pages' read-side formulas applied to every code,
single-element position probes, values constructed on an exact grid, IEEE half rounding
done by Python's struct module, closed forms (Sylvester Hadamard matrix, orthogonality),
and pure-Python brute force on tiny inputs.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant as Q
from oracle import attention as A

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_sizes.json")))


def py_half(x: float) -> float:
    """IEEE binary16 rounding (half-to-even) by the standard library, independent of numpy."""
    return struct.unpack("<e", struct.pack("<e", x))[0]


def nibble(payload, i):
    b = int(payload[i // 2])
    return (b >> (4 * (i % 2))) & 0xF


# ------------------------------------------------------------------ sizes the pages print
def test_bytes_per_element_and_token():
    D = 128
    q4 = (Q.row_bytes("q4_0", D) + Q.param_bytes("q4_0", D)) / D
    q6 = (Q.row_bytes("q6_0", D) + Q.param_bytes("q6_0", D)) / D
    assert q4 == GOLD["q4_0_bytes_per_element"]["value"]
    assert q6 == GOLD["q6_0_bytes_per_element"]["value"]
    # bytes/token table: 10240 elements per token for every scheme (20480 B at bf16)
    table = GOLD["bytes_per_token_table"]["value"]
    n_el = table["bf16"] // 2
    assert n_el * q4 == table["q4_0"]
    assert n_el * q6 == table["q6_0"]
    assert n_el * GOLD["q8_0_bytes_per_element"]["value"] == table["q8_0"]


def test_hadamard_per_head_bytes():
    D = 128
    per_token_kv = 2 * (Q.row_bytes("had_int4", D) + Q.param_bytes("had_int4", D))
    g = GOLD["per_head_bytes_kib"]["value"]
    for T, f16, i4 in zip(g["T"], g["f16"], g["int4"]):
        assert T * 2 * D * 2 == f16 * 1024
        assert T * per_token_kv == i4 * 1024
    ratio = (2 * D * 4) / per_token_kv
    assert round(ratio, 1) == GOLD["int4_vs_f32_memory_ratio"]["value"]
    assert 28 * 2 * 8 * 128 * 2 == GOLD["qwen3_1p7b_f16_bytes_per_token"]["value"]


def test_asym_compression_ratio():
    D = 128
    fp16_bytes = D * 2
    asym = Q.row_bytes("asym4_g32", D) + Q.param_bytes("asym4_g32", D)
    assert fp16_bytes / asym == GOLD["asym4_g32_compression_vs_fp16"]["value"]


# ------------------------------------------------------------------ Q4_0
def test_q4_0_every_code_through_read_formula():
    # all 16 codes on an exact grid: s = 0.25, amax = 2.0 (code -8) so scale = 2/8 exactly
    codes = np.array(list(range(-8, 8)) * 2, np.float32)
    x = codes * np.float32(0.25)
    p, s = Q.quantize_q4_0(x[None])
    assert float(s[0, 0]) == 0.25
    got = [((nibble(p[0], i) ^ 0x8) - 0x8) for i in range(32)]        # the page's read formula
    assert got == [int(c) for c in codes]
    assert np.array_equal(Q.dequantize_q4_0(p, s)[0], x.astype(np.float64))


@pytest.mark.parametrize("i", range(32))
def test_q4_0_nibble_position(i):
    # value 2j -> low nibble of byte j, value 2j+1 -> high nibble
    x = np.zeros(32, np.float32)
    x[i] = -3.0                          # amax 3 -> scale 3/8, code -8
    x[(i + 5) % 32] = 1.5                # code 4 at another position
    p, s = Q.quantize_q4_0(x[None])
    assert float(s[0, 0]) == py_half(3.0 / 8.0)
    for j in range(32):
        want = {i: (-8) & 0xF, (i + 5) % 32: 4}.get(j, 0)
        assert nibble(p[0], j) == want


def test_q4_0_saturation_and_half_even():
    x = np.zeros(32, np.float32)
    x[0], x[1] = 8.0, -8.0                           # scale 1: +amax -> 8 clamps to 7, -amax -> -8
    halves = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 6.5, -6.5]
    x[2:2 + len(halves)] = halves
    p, s = Q.quantize_q4_0(x[None])
    assert float(s[0, 0]) == 1.0
    dec = [((nibble(p[0], i) ^ 8) - 8) for i in range(32)]
    assert dec[0] == 7 and dec[1] == -8
    assert dec[2:2 + len(halves)] == [0, 2, 2, 0, -2, -2, 4, 6, -6]   # round half to even


def test_q4_0_zero_and_underflow_blocks():
    z = np.zeros((2, 32), np.float32)
    z[0, 3] = -0.0
    z[1, 7] = 1e-9                                     # amax/8 underflows fp16 -> scale 0, codes 0
    p, s = Q.quantize_q4_0(z)
    assert not p.any() and not s.astype(np.float32).any()


def test_q4_0_scale_is_ieee_half_of_amax_over_8():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 32)) * rng.uniform(0.01, 300, (64, 1))).astype(np.float32)
    _, s = Q.quantize_q4_0(x)
    for r in range(64):
        amax = float(np.max(np.abs(x[r])))
        assert float(s[r, 0]) == py_half(amax / 8.0)


def test_q4_0_error_bound():
    rng = np.random.default_rng(8)
    x = rng.standard_t(4, (256, 128)).astype(np.float32)
    p, s = Q.quantize_q4_0(x)
    xb = x.reshape(256, 4, 32).astype(np.float64)
    xh = Q.dequantize_q4_0(p, s).reshape(256, 4, 32)
    sc = np.repeat(s.astype(np.float64)[..., None], 32, -1)
    r = xb / sc
    inner = (r >= -8.5) & (r <= 7.5)
    # inside the code range: within half a step of the stored scale
    assert np.all(np.abs(xh - xb)[inner] <= 0.5 * sc[inner] * (1 + 1e-6))
    # beyond it: saturated at the end codes 7 / -8 (only the block's +amax can exceed 7.5 steps)
    assert np.all(xh[r > 7.5] == 7 * sc[r > 7.5])
    assert np.all(xh[r < -8.5] == -8 * sc[r < -8.5])


# ------------------------------------------------------------------ Q6_0
def test_q6_0_every_code_through_read_formula():
    codes = np.array(list(range(-32, 32)), np.float32)
    x = (codes * np.float32(0.125)).reshape(2, 32)    # two blocks; each has amax 4 (code -32)
    x[1, 0] = -32 * 0.125                              # make the second block's amax 4 as well
    codes2 = codes.reshape(2, 32).copy()
    codes2[1, 0] = -32
    p, s = Q.quantize_q6_0(x.reshape(1, 64))
    assert s.shape == (1, 2) and np.all(s.astype(np.float32) == 0.125)
    for b in range(2):
        blk = p[0, 24 * b: 24 * b + 24]
        for i in range(32):
            lo = nibble(blk[:16], i)
            hi = (int(blk[16 + i // 4]) >> (2 * (i % 4))) & 3
            v = lo | (hi << 4)
            assert ((v ^ 0x20) - 0x20) == int(codes2[b, i])         # the page's read formula


@pytest.mark.parametrize("i", range(32))
def test_q6_0_plane_positions(i):
    x = np.zeros(32, np.float32)
    x[i] = -4.0            # amax 4 -> scale 1/8, code -32 = 0b100000: low nibble 0, top bits 2
    x[(i + 3) % 32] = 2.375  # code 19 = 0b010011: low nibble 3, top bits 1
    p, s = Q.quantize_q6_0(x[None])
    blk = p[0]
    for j in range(32):
        code = {i: -32, (i + 3) % 32: 19}.get(j, 0) & 0x3F
        assert nibble(blk[:16], j) == code & 0xF
        assert (int(blk[16 + j // 4]) >> (2 * (j % 4))) & 3 == code >> 4


def test_q6_0_saturation():
    x = np.zeros(32, np.float32)
    x[5], x[6] = 32.0, -32.0
    p, s = Q.quantize_q6_0(x[None])
    v = Q.q6_0_fields(p, 1)[0, 0]
    assert Q.read_q6_0(v[5]) == 31 and Q.read_q6_0(v[6]) == -32


# ------------------------------------------------------------------ FWHT / Hadamard int4
@pytest.mark.parametrize("D", [2, 8, 32, 128, 256])
def test_fwht_equals_dense_sylvester(D):
    rng = np.random.default_rng(D)
    x = rng.standard_normal((5, D))
    H = Q.hadamard_matrix(D)
    # closed form of the Sylvester matrix, entry by entry
    for i in range(0, D, max(1, D // 8)):
        for j in range(0, D, max(1, D // 8)):
            assert H[i, j] == (-1) ** bin(i & j).count("1")
    assert np.allclose(H @ H, D * np.eye(D))
    got = Q.fwht(x, np.float64)
    assert np.allclose(got, x @ H.T, rtol=0, atol=1e-12 * np.abs(x).sum())


def test_rotation_preserves_scores():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 128))
    k = rng.standard_normal((9, 128))
    c = 1.0 / math.sqrt(128)
    qr, kr = Q.fwht(q, np.float64) * c, Q.fwht(k, np.float64) * c
    assert np.allclose(qr @ kr.T, q @ k.T, rtol=0, atol=1e-10)       # (QH)(KH)^T = QK^T


@pytest.mark.parametrize("D", [128, 256])
def test_inv_sqrt_is_nearest_float32(D):
    c = Q.inv_sqrt_f32(D)
    below = np.nextafter(c, np.float32(0))
    above = np.nextafter(c, np.float32(1))
    target = Fraction(1) / Fraction(D)                                  # compare squares exactly
    err = lambda v: abs(Fraction(float(v)) ** 2 - target)
    assert err(c) <= err(below) and err(c) <= err(above)


def test_hadamard_int4_codes_and_scale():
    rng = np.random.default_rng(5)
    x = rng.standard_t(4, (64, 128)).astype(np.float32)
    x[:, 7] *= 10
    p, s, y = Q.quantize_hadamard_int4(x)
    assert p.shape == (64, 64) and s.dtype == np.float32
    codes = Q.hadamard_codes(p, 128)
    assert codes.min() >= -7 and codes.max() <= 7
    assert np.all(np.max(np.abs(codes), axis=1) == 7)                 # the amax element maps to +-7
    assert np.all(s == (np.max(np.abs(y), axis=1) / np.float32(7)))
    err = np.abs(codes * s[:, None].astype(np.float64) - y)
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-6))
    # the rotated row is the orthonormal rotation of x
    ref = Q.fwht(x.astype(np.float64), np.float64) / math.sqrt(128)
    assert np.allclose(y, ref, rtol=0, atol=1e-5 * np.abs(ref).max())


# ------------------------------------------------------------------ asymmetric g=32
def test_asym_exact_grid():
    qv = np.array(list(range(16)) * 2, np.float32)
    x = np.float32(-1.0) + qv * np.float32(0.125)       # min -1 (code 0), max 0.875 (code 15)
    p, s, z = Q.quantize_asym4_g32(x[None])
    assert float(s[0, 0]) == 0.125 and float(z[0, 0]) == -1.0
    got = [nibble(p[0], i) for i in range(32)]
    assert got == [int(v) for v in qv]
    assert np.array_equal(Q.dequantize_asym4_g32(p, s, z)[0], x.astype(np.float64))


def test_asym_constant_group_and_bound():
    x = np.full((1, 32), 0.3, np.float32)
    p, s, z = Q.quantize_asym4_g32(x)
    assert float(s[0, 0]) == 0.0 and not p.any() and float(z[0, 0]) == py_half(float(np.float32(0.3)))
    rng = np.random.default_rng(11)
    y = rng.standard_t(4, (128, 128)).astype(np.float32)
    p, s, z = Q.quantize_asym4_g32(y)
    yh = Q.dequantize_asym4_g32(p, s, z).reshape(128, 4, 32)
    yb = y.reshape(128, 4, 32)
    sc = s.astype(np.float64)[..., None]
    zshift = np.abs(yb.min(-1) - z.astype(np.float64))[..., None]
    assert np.all(np.abs(yh - yb) <= 0.5 * sc + zshift + 1e-6)
    codes = Q.unpack_nibbles(p.reshape(128, 4, 16), 32)
    assert np.all(codes[np.arange(128)[:, None], np.arange(4)[None, :], yb.argmin(-1)] <= 1)
    assert np.all(codes[np.arange(128)[:, None], np.arange(4)[None, :], yb.argmax(-1)] >= 14)


# ------------------------------------------------------------------ attention
def brute_attention(q, K, V, alpha, visible):
    """Pure-Python softmax attention of one query row (tiny inputs)."""
    idx = [t for t in range(len(K)) if visible(t)]
    s = [alpha * sum(q[d] * K[t][d] for d in range(len(q))) for t in idx]
    m = max(s)
    w = [math.exp(v - m) for v in s]
    L = sum(w)
    return [sum(w[j] * V[idx[j]][d] for j in range(len(idx))) / L for d in range(len(q))]


def test_attention_brute_force_gqa_causal():
    rng = np.random.default_rng(21)
    B, Hq, Hkv, nq, S, D = 1, 4, 2, 3, 40, 8
    q = rng.standard_normal((B, Hq, nq, D))
    K = rng.standard_normal((B, Hkv, S, D))
    V = rng.standard_normal((B, Hkv, S, D))
    alpha, q_pos0 = 0.37, 30
    got = A.attend_dense(q, K, V, alpha, S, causal=True, q_pos0=q_pos0)
    for h in range(Hq):
        for i in range(nq):
            ref = brute_attention(q[0, h, i].tolist(), K[0, h // 2].tolist(), V[0, h // 2].tolist(), alpha,
                                  lambda t: t <= q_pos0 + i)
            assert np.allclose(got[0, h, i], ref, rtol=1e-12, atol=1e-12)


def test_gqa_mapping_reads_kv_head_q_over_gqa():
    B, Hq, Hkv, S, D = 1, 8, 2, 5, 4
    q = np.ones((B, Hq, 1, D))
    K = np.zeros((B, Hkv, S, D))
    V = np.stack([np.full((S, D), 10.0 * (h + 1)) for h in range(Hkv)])[None]
    out = A.attend_dense(q, K, V, 1.0, S)
    assert np.allclose(out[0, :, 0, 0], [10, 10, 10, 10, 20, 20, 20, 20])


@pytest.mark.parametrize("chunk", [1, 7, 16, 64, 512])
def test_split_k_equals_single_pass(chunk):
    rng = np.random.default_rng(chunk)
    B, Hq, Hkv, nq, S, D = 2, 4, 2, 5, 150, 16
    q = rng.standard_normal((B, Hq, nq, D)) * 2
    K = rng.standard_normal((B, Hkv, S, D))
    V = rng.standard_normal((B, Hkv, S, D))
    for causal in (False, True):
        a = A.attend_dense(q, K, V, 0.5, S, causal, q_pos0=40)
        b = A.attend_split(q, K, V, 0.5, S, causal, q_pos0=40, chunk=chunk)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_causal_skip_equals_compute_then_mask():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, nq, S, D = 1, 2, 1, 16, 64, 8
    q = rng.standard_normal((B, Hq, nq, D))
    K = rng.standard_normal((B, Hkv, S, D))
    V = rng.standard_normal((B, Hkv, S, D))
    a = A.attend_dense(q, K, V, 0.3, S, causal=True, q_pos0=48)
    b = A.attend_causal_skip(q, K, V, 0.3, S, q_pos0=48)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)


def test_integer_scores_brute_force():
    rng = np.random.default_rng(4)
    q8 = rng.integers(-127, 128, (3, 32)).astype(np.int8)
    kc = rng.integers(-7, 8, (10, 32))
    got = A.scores_int(q8, kc)
    for r in range(3):
        for t in range(10):
            assert got[r, t] == sum(int(q8[r, d]) * int(kc[t, d]) for d in range(32))


def test_hadamard_full_window_is_exact_attention():
    # n_recent >= kv_len: every token is scored and weighted in exact f32 rotated values,
    # so the result is unquantised attention (tract discussion #2402 Appendix 7: "full f32 window 0.000").
    rng = np.random.default_rng(12)
    B, Hq, Hkv, S, D = 1, 4, 2, 48, 128
    k = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    v = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, 1, D)).astype(np.float32)
    c = A.OracleCache("had_int4", B, Hkv, D, S, n_recent=64)
    c.store(k, v, 0)
    out, _ = c.attend(q, 1 / math.sqrt(D), S)
    ref = A.attend_dense(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), 1 / math.sqrt(D), S)
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-5)


def test_hadamard_body_on_exact_grid_matches_plain_attention():
    # Rows built so that rotation + int4/int8 quantisation are lossless: the integer-domain score
    # times the scales and the un-rotated P.V must then equal plain attention of the inputs.
    rng = np.random.default_rng(13)
    D, S = 128, 20
    H = Q.hadamard_matrix(D) / math.sqrt(D)
    kc = rng.integers(-7, 8, (S, D)).astype(np.float64)
    kc[:, 0] = 7
    vc = rng.integers(-7, 8, (S, D)).astype(np.float64)
    vc[:, 1] = -7
    qc = rng.integers(-127, 128, (1, D)).astype(np.float64)
    qc[:, 2] = 127
    sk, sv, sq = 0.0625, 0.125, 1.0 / 256
    k = (kc * sk) @ H          # rotate(k) = k H^T / ... = kc * sk exactly up to fp32 rounding
    v = (vc * sv) @ H
    q = (qc * sq) @ H
    c = A.OracleCache("had_int4", 1, 1, D, S, n_recent=0)
    c.store(k[None, None].astype(np.float32), v[None, None].astype(np.float32), 0)
    assert np.array_equal(Q.hadamard_codes(c.planes["k"]["payload"][0, 0], D), kc)
    out, si = c.attend(q[None, None].astype(np.float32), 0.02, S)
    assert np.array_equal(si[0, 0, 0], (qc @ kc.T)[0].astype(np.int64))
    ref = A.attend_dense(q[None, None], k[None, None], v[None, None], 0.02, S)
    assert np.allclose(out, ref, rtol=2e-5, atol=2e-5)


def test_error_envelopes():
    # sanity band around the pages' kernel-level relative errors on kurtotic K/V
    # (q4_0 0.094, q6_0 0.024: FreeToken PR #268 Validation table; int4+H 0.115:
    # tract discussion #2402 Appendix 7). The definition is not stated, so only a band.
    rng = np.random.default_rng(31)
    B, Hq, Hkv, S, D = 1, 8, 2, 1024, 128
    k = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    v = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    k[:, :, :, [3, 50]] *= 10
    q = rng.standard_normal((B, Hq, 1, D)).astype(np.float32)
    alpha = 1 / math.sqrt(D)
    ref = A.attend_dense(q, k, v, alpha, S)
    errs = {}
    for lay in ("q4_0", "q6_0", "asym4_g32"):
        c = A.OracleCache(lay, B, Hkv, D, S)
        c.store(k, v, 0)
        out = c.attend(q, alpha, S)
        errs[lay] = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    c = A.OracleCache("had_int4", B, Hkv, D, S)
    c.store(k, v, 0)
    out, _ = c.attend(q, alpha, S)
    errs["had"] = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert 0.02 < errs["q4_0"] < 0.3
    assert 0.02 < errs["had"] < 0.3
    assert errs["q6_0"] < errs["q4_0"] / 2.5
    assert errs["asym4_g32"] < 0.3


def test_recent_window_semantics():
    # the newest n_recent tokens come from the ring, older ones from the packed body
    rng = np.random.default_rng(2)
    D, S, nr = 128, 40, 8
    k = rng.standard_normal((1, 1, S, D)).astype(np.float32)
    v = rng.standard_normal((1, 1, S, D)).astype(np.float32)
    c = A.OracleCache("had_int4", 1, 1, D, 64, n_recent=nr)
    c.store(k[:, :, :30], v[:, :, :30], 0)
    c.store(k[:, :, 30:], v[:, :, 30:], 30)
    for t in range(S - nr, S):
        assert np.array_equal(c.planes["k"]["ring"][0, 0, t % nr], Q.rotate(k[0, 0, t]))
    q = rng.standard_normal((1, 2, 1, D)).astype(np.float32)
    out_w, _ = c.attend(q, 0.1, S)
    c0 = A.OracleCache("had_int4", 1, 1, D, 64, n_recent=0)
    c0.store(k, v, 0)
    out_0, _ = c0.attend(q, 0.1, S)
    assert not np.allclose(out_w, out_0)       # the window changes the result ...
    ref = A.attend_dense(q, k, v, 0.1, S)
    assert np.linalg.norm(out_w - ref) < np.linalg.norm(out_0 - ref)   # ... towards exact attention


# ------------------------------------------------------------------ Q8_0 (reading R24)
def test_q8_0_density_is_the_pages():
    D = 128
    q8 = (Q.row_bytes("q8_0", D) + Q.param_bytes("q8_0", D)) / D
    assert q8 == GOLD["q8_0_bytes_per_element"]["value"]
    assert (GOLD["bytes_per_token_table"]["value"]["bf16"] // 2) * q8 == GOLD["bytes_per_token_table"]["value"]["q8_0"]


def test_q8_0_every_code_through_read_formula():
    # all 256 codes on an exact grid: 8 blocks of 32; each block holds -128 so amax = 128 s, s = 1/16
    codes = np.arange(-128, 128, dtype=np.float32).reshape(8, 32)
    codes[:, 0] = -128
    x = codes * np.float32(0.0625)
    p, s = Q.quantize_q8_0(x.reshape(1, 256))
    assert np.all(s.astype(np.float32) == 0.0625)
    got = [((int(p[0, i]) ^ 0x80) - 0x80) for i in range(256)]        # two's-complement byte i
    assert got == [int(c) for c in codes.reshape(-1)]
    assert np.array_equal(Q.dequantize_q8_0(p, s)[0], x.reshape(-1).astype(np.float64))


@pytest.mark.parametrize("i", [0, 1, 7, 16, 31])
def test_q8_0_byte_position_and_saturation(i):
    x = np.zeros(32, np.float32)
    x[i] = 12.8                     # amax -> scale fp16(0.1); 12.8 / scale rounds to 128 -> clamps to 127
    x[(i + 9) % 32] = -12.8         # -amax -> -128
    x[(i + 3) % 32] = 0.25          # an ordinary code
    p, s = Q.quantize_q8_0(x[None])
    sc = py_half(12.8 / 128.0)
    assert float(s[0, 0]) == sc
    want = {i: 127, (i + 9) % 32: -128, (i + 3) % 32: int(round(0.25 / sc))}
    for j in range(32):
        assert Q.read_q8_0(p[0, j]) == want.get(j, 0)


def test_q8_0_half_even_and_zero_block():
    x = np.zeros((2, 32), np.float32)
    x[0, 0] = 128.0                                      # scale 1
    x[0, 1:6] = [0.5, 1.5, 2.5, -0.5, -2.5]
    p, s = Q.quantize_q8_0(x)
    assert [int(Q.read_q8_0(p[0, j])) for j in range(1, 6)] == [0, 2, 2, 0, -2]
    assert not p[1].any() and float(s[1, 0]) == 0.0


# ------------------------------------------------------------------ Hadamard int2 (reading R25)
def test_int2_read_formula_every_field():
    # the four 2-bit fields through (v ^ 2) - 2: 0 -> 0, 1 -> 1, 2 -> -2, 3 -> -1
    assert [int(Q.read_int2(v)) for v in range(4)] == [0, 1, -2, -1]


@pytest.mark.parametrize("i", [0, 1, 2, 3, 4, 126, 127])
def test_int2_field_positions(i):
    # value 4j+i at bits 2i..2i+1 of byte j: pack a single -1 (field 0b11) at position i
    f = np.zeros(128, np.int32)
    f[i] = -1
    b = Q.pack_pairs_of_bits(f & 3)
    assert b.shape == (32,)
    for j in range(32):
        assert int(b[j]) == (3 << (2 * (i % 4)) if j == i // 4 else 0)
    assert np.array_equal(Q.hadamard_int2_codes(b, 128), f)


def test_hadamard_int2_codes_and_scale():
    rng = np.random.default_rng(6)
    x = rng.standard_t(4, (64, 128)).astype(np.float32)
    p, s, y = Q.quantize_hadamard_int2(x)
    assert p.shape == (64, 32) and s.dtype == np.float32
    codes = Q.hadamard_int2_codes(p, 128)
    assert set(np.unique(codes)) <= {-1, 0, 1}
    assert np.all(s == np.max(np.abs(y), axis=1))                       # scale = amax / 1
    # code = the nearest of {-1, 0, 1} to y / s (half-to-even at +-0.5: to 0)
    r = y.astype(np.float64) / s[:, None]
    want = np.where(r > 0.5, 1, np.where(r < -0.5, -1, 0))
    assert np.array_equal(codes, want)


def test_hadamard_int2_full_window_is_exact_attention():
    # every token in the exact-f32 window: the int2 body is never read
    rng = np.random.default_rng(14)
    B, Hq, Hkv, S, D = 1, 4, 2, 40, 128
    k = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    v = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, 1, D)).astype(np.float32)
    c = A.OracleCache("had_int2", B, Hkv, D, S, n_recent=64)
    c.store(k, v, 0)
    out, _ = c.attend(q, 1 / math.sqrt(D), S)
    ref = A.attend_dense(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), 1 / math.sqrt(D), S)
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-5)


def test_hadamard_int2_body_scores_brute_force():
    # the body scores are the exact integer dots of the int8 query codes and the int2 key codes
    rng = np.random.default_rng(15)
    D, S = 128, 12
    k = rng.standard_normal((1, 1, S, D)).astype(np.float32)
    c = A.OracleCache("had_int2", 1, 1, D, S, n_recent=0)
    c.store(k, k, 0)
    q = rng.standard_normal((1, 1, 2, D)).astype(np.float32)
    _, si = c.attend(q, 0.1, S)
    _, _, q8 = A.prep_q_hadamard(q)
    kc = Q.hadamard_int2_codes(c.planes["k"]["payload"][0, 0], D)
    for r in range(2):
        for t in range(S):
            assert si[0, 0, r, t] == sum(int(q8[0, 0, r, d]) * int(kc[t, d]) for d in range(D))


def test_int2_needs_the_window():
    # the reason for the window: int2 alone is far off exact attention, and a window over the
    # newest tokens brings it closer (tract discussion #2402, "Why this quant scheme")
    rng = np.random.default_rng(16)
    D, S = 128, 96
    k = rng.standard_t(4, (1, 2, S, D)).astype(np.float32)
    v = rng.standard_t(4, (1, 2, S, D)).astype(np.float32)
    q = (rng.standard_normal((1, 4, 1, D)) * 2).astype(np.float32)
    ref = A.attend_dense(q, k, v, 1 / math.sqrt(D), S)
    errs = {}
    for nr in (0, 32):
        c = A.OracleCache("had_int2", 1, 2, D, S, n_recent=nr)
        c.store(k, v, 0)
        out, _ = c.attend(q, 1 / math.sqrt(D), S)
        errs[nr] = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    c4 = A.OracleCache("had_int4", 1, 2, D, S)
    c4.store(k, v, 0)
    e4 = np.linalg.norm(c4.attend(q, 1 / math.sqrt(D), S)[0] - ref) / np.linalg.norm(ref)
    assert errs[0] > e4 and errs[32] < errs[0]


# ------------------------------------------------------------------ mixed K/V precision
def test_mixed_planes_are_the_single_layout_planes():
    """A "k+v" cache stores K exactly as a cache of the K layout and V exactly as one of the V layout."""
    rng = np.random.default_rng(21)
    k = rng.standard_t(4, (1, 2, 40, 128)).astype(np.float32)
    v = rng.standard_t(4, (1, 2, 40, 128)).astype(np.float32)
    for kl, vl in (("q4_0", "q8_0"), ("q8_0", "q4_0"), ("asym4_g32", "q6_0"), ("had_int2", "had_int4")):
        m = A.OracleCache(f"{kl}+{vl}", 1, 2, 128, 40, n_recent=8 if kl.startswith("had") else 0)
        m.store(k, v, 0)
        for lay, t, x in ((kl, "k", k), (vl, "v", v)):
            single = A.OracleCache(lay, 1, 2, 128, 40, n_recent=8 if lay.startswith("had") else 0)
            single.store(x, x, 0)
            for name, arr in single.planes[t].items():
                assert np.array_equal(m.planes[t][name], arr), (kl, vl, t, name)


def test_mixed_attention_is_attention_of_each_planes_dequantisation():
    rng = np.random.default_rng(22)
    B, Hq, Hkv, S, D = 1, 4, 2, 50, 128
    k = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    v = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, 2, D)).astype(np.float32)
    m = A.OracleCache("q4_0+q8_0", B, Hkv, D, S)
    m.store(k, v, 0)
    got = m.attend(q, 0.1, S, causal=True, q_pos0=S - 2)
    kd = Q.dequantize("q4_0", Q.quantize("q4_0", k), D)
    vd = Q.dequantize("q8_0", Q.quantize("q8_0", v), D)
    ref = A.attend_dense(q, kd, vd, 0.1, S, causal=True, q_pos0=S - 2)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_mixed_rejects_a_rotated_and_an_unrotated_plane():
    with pytest.raises(ValueError):
        A.OracleCache("q4_0+had_int4", 1, 1, 128, 8)


def test_value_precision_matters_more_than_key_precision():
    """Open-TQ-Metal, Section 5: value errors reach the output directly, key errors pass through the
    softmax; on heavy-tailed data the 4-bit K + 8-bit V cache is the closer of the two mixes."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, S, D = 1, 8, 2, 256, 128
    k = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    v = rng.standard_t(4, (B, Hkv, S, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, 1, D)).astype(np.float32)
    ref = A.attend_dense(q, k, v, 1 / math.sqrt(D), S)
    err = {}
    for lay in ("q4_0+q8_0", "q8_0+q4_0"):
        c = A.OracleCache(lay, B, Hkv, D, S)
        c.store(k, v, 0)
        err[lay] = np.linalg.norm(c.attend(q, 1 / math.sqrt(D), S) - ref) / np.linalg.norm(ref)
    assert err["q4_0+q8_0"] < err["q8_0+q4_0"]
