"""Pins of the paged-cache oracle (oracle/paged.py).

The paged model is pinned to things other than itself: hand-computed pool locations of single
probe tokens, the (separately pinned) contiguous oracle filled with each sequence's tokens
directly, invariance under a permuted block table, and the degenerate cases (an empty sequence,
causal rows before a short sequence's start, positions beyond the capacity).
"""
import numpy as np
import pytest

from oracle import quant as Q
from oracle.attention import OracleCache
from oracle.paged import OraclePagedCache

LAYOUTS = ["q4_0", "q6_0", "had_int4", "asym4_g32"]


def _rows(rng, B, H, n, D):
    return rng.standard_normal((B, H, n, D)).astype(np.float32)


def test_probe_token_lands_at_table_page_and_row():
    """Token t of sequence b is row t % P of pool page table[b][t // P] (hand-computed cases)."""
    P, D = 64, 128
    table = np.array([[5, 2, 9], [0, 7, 3]])
    pc = OraclePagedCache("q4_0", 2, 1, D, P, 10, 3, table=table)
    cases = [(0, 0, 5, 0), (0, 70, 2, 6), (0, 191, 9, 63), (1, 64, 7, 0), (1, 130, 3, 2)]
    for b, t, page, row in cases:
        before = pc.planes["k"]["scale"].copy()
        x = np.zeros((2, 1, 1, D), np.float32)
        x[b, 0, 0, :] = 3.0 + t                              # only sequence b's row is non-zero
        pos = np.array([t, t])
        pc.store(x, x, pos)
        changed = np.argwhere(np.any(pc.planes["k"]["scale"] != before, axis=-1))
        assert changed.tolist() == [[page, 0, row]], (b, t, changed)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_paged_equals_contiguous_per_sequence(layout):
    """Each sequence of the paged pool (ragged lengths, permuted table, fill + append) attends
    exactly as a contiguous one-sequence cache filled with the same rows by the contiguous store."""
    rng = np.random.default_rng(7)
    B, H, Hq, D, P = 3, 2, 4, 128, 64
    n_recent = 16 if layout == "had_int4" else 0
    lens = np.array([150, 64, 0])
    mpp = 3
    table = rng.permutation(B * mpp + 2)[:B * mpp].reshape(B, mpp)
    pc = OraclePagedCache(layout, B, H, D, P, B * mpp + 2, mpp, n_recent, table=table)
    S = int(lens.max())
    k, v = _rows(rng, B, H, S, D), _rows(rng, B, H, S, D)
    fill = np.maximum(lens - 5, 0)
    # bulk fill of each sequence's first fill[b] tokens, one sequence per call (the others'
    # positions lie past the capacity, so their rows are dropped), then the last 5 tokens of
    # every sequence as one append
    for b in range(B):
        if fill[b]:
            pos0 = np.full(B, pc.cap)
            pos0[b] = 0
            pc.store(k[:, :, :fill[b]], v[:, :, :fill[b]], pos0)
    tail_k = np.stack([k[b, :, fill[b]:fill[b] + 5] if lens[b] else np.zeros((H, 5, D), np.float32) for b in range(B)])
    tail_v = np.stack([v[b, :, fill[b]:fill[b] + 5] if lens[b] else np.zeros((H, 5, D), np.float32) for b in range(B)])
    pc.store(tail_k, tail_v, np.where(lens > 0, fill, pc.cap))
    q = _rows(rng, B, Hq, 3, D)
    for causal in (False, True):
        got = pc.attend(q, 0.125, lens, causal)
        for b in range(B):
            L = int(lens[b])
            if L == 0:
                assert not got[b].any()
                continue
            c = OracleCache(layout, 1, H, D, L, n_recent)
            c.store(k[b:b + 1, :, :L - 5], v[b:b + 1, :, :L - 5], 0)
            c.store(k[b:b + 1, :, L - 5:L], v[b:b + 1, :, L - 5:L], L - 5)
            want = c.attend(q[b:b + 1], 0.125, L, causal, L - 3)
            want = want[0] if isinstance(want, tuple) else want
            np.testing.assert_array_equal(got[b], want[0])


@pytest.mark.parametrize("layout", ["q4_0", "had_int4"])
def test_permuted_table_does_not_change_results(layout):
    """The same rows stored through two different block tables give identical attention, and the
    pool rows are the same bytes at the table-mapped places."""
    rng = np.random.default_rng(11)
    B, H, D, P, mpp = 2, 2, 128, 64, 4
    n_recent = 8 if layout == "had_int4" else 0
    k, v, q = _rows(rng, B, H, 200, D), _rows(rng, B, H, 200, D), _rows(rng, B, 4, 2, D)
    lens = np.array([200, 131])
    outs, caches = [], []
    for table in (np.arange(B * mpp).reshape(B, mpp), rng.permutation(B * mpp).reshape(B, mpp)):
        pc = OraclePagedCache(layout, B, H, D, P, B * mpp, mpp, n_recent, table=table)
        pc.store(k, v, np.zeros(B, np.int64))
        outs.append(pc.attend(q, 0.1, lens, causal=True))
        caches.append(pc)
    np.testing.assert_array_equal(outs[0], outs[1])
    for b in range(B):
        for t in range(0, 200, 37):
            (p0, r0), (p1, r1) = caches[0].locate(b, t), caches[1].locate(b, t)
            np.testing.assert_array_equal(caches[0].planes["v"]["payload"][p0, :, r0],
                                          caches[1].planes["v"]["payload"][p1, :, r1])


def test_short_causal_sequence_rows_before_start_are_zero():
    """Causal rows at negative positions (sequence shorter than n_q) see nothing -> zeros; the
    others equal a direct softmax over the dequantised rows."""
    rng = np.random.default_rng(3)
    H, D, P = 1, 128, 64
    pc = OraclePagedCache("q4_0", 1, H, D, P, 2, 2, table=np.array([[1, 0]]))
    k, v = _rows(rng, 1, H, 3, D), _rows(rng, 1, H, 3, D)
    pc.store(k, v, np.array([0]))
    q = _rows(rng, 1, H, 5, D)                               # 5 query rows, 3 tokens
    out = pc.attend(q, 0.2, np.array([3]), causal=True)
    assert not out[0, 0, :2].any()                           # positions -2, -1
    kd = Q.dequantize("q4_0", Q.quantize("q4_0", k[0, 0]), D).astype(np.float64)
    vd = Q.dequantize("q4_0", Q.quantize("q4_0", v[0, 0]), D).astype(np.float64)
    for i in range(2, 5):
        n = i - 1                                            # row i at position i - 2 sees t <= i - 2
        s = 0.2 * kd[:n] @ q[0, 0, i].astype(np.float64)
        p = np.exp(s - s.max())
        np.testing.assert_allclose(out[0, 0, i], p @ vd[:n] / p.sum(), rtol=1e-12, atol=1e-12)


def test_store_beyond_capacity_is_dropped():
    rng = np.random.default_rng(5)
    pc = OraclePagedCache("asym4_g32", 2, 1, 128, 64, 4, 1, table=np.array([[0], [1]]))
    x = _rows(rng, 2, 1, 4, 128)
    pc.store(x, x, np.array([62, -1]))                      # seq 0: rows 62, 63 fit; seq 1: row -1 dropped
    assert pc.planes["k"]["scale"][0, 0, 62:].any()
    assert not pc.planes["k"]["scale"][2:].any()
    assert pc.planes["k"]["scale"][1, 0, :3].any() and not pc.planes["k"]["scale"][1, 0, 3:].any()
