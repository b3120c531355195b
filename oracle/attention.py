"""Oracle decode attention over a packed KV cache, accumulated in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

`OracleCache` models the cache a caller owns: per (batch, kv head) rows of packed payload,
fp16 (or f32) scales, fp16 zero-points and, for the Hadamard layout, the float32 ring of the
newest `n_recent` rotated rows. `store` appends rows exactly as the quantizers in
`oracle.quant` define; `attend` computes scaled-dot-product attention from the exactly
dequantised rows.

Definitions followed:
  * score_t = alpha * q . k_hat_t, softmax over the visible tokens, out = sum_t p_t v_hat_t
    (standard attention; "score = alpha * q^T k", Open-TQ-Metal Section 4).
  * GQA: query head h reads kv head h // (H_q / H_kv) (Open-TQ-Metal Section 3, "SIMD and
    threadgroup organization").
  * causal: query row i (absolute position q_pos0 + i) sees tokens t <= q_pos0 + i
    (tract discussion #2402, "Causality & mixed precision").
  * split-K: chunks of `chunk` tokens from t = 0 each give (m_c, l_c, o_c) and a second phase
    combines them by the online-softmax correction (Open-TQ-Metal Section 3.2). Reading R15:
    M = max m_c, L = sum l_c e^(m_c - M), O = sum o_c e^(m_c - M) / L; a chunk with no visible
    token (m_c = -inf) weighs zero.
  * Hadamard layout (tract discussion #2402, "Architecture: Data flow (decode)"): Q is rotated
    by the same FWHT, quantised to int8 with one float32 scale per query row (reading R8:
    s_q = amax / 127, codes clamped to +-127), body scores are the exact integer dot
    int8(q_rot) . int4(k_rot) times alpha * s_q * s_k; the newest n_recent tokens are scored
    and weighted in exact float32 rotated values (reading R13); P.V runs in the rotated basis
    and the output is un-rotated by H / sqrt(D) (dense matrix here).
  * n_recent (reading R11/R12): a cache property; with kv_len tokens cached, tokens
    t >= kv_len - n_recent are read from ring slot t mod n_recent. Every token is also
    quantised when it is stored.
"""
from __future__ import annotations

import math

import numpy as np

from . import quant as Q


# ------------------------------------------------------------------ plain attention
def visible_mask(n_q: int, kv_len: int, causal: bool, q_pos0: int) -> np.ndarray:
    """[n_q][kv_len] bool: row i sees t < kv_len and, if causal, t <= q_pos0 + i."""
    t = np.arange(kv_len)[None, :]
    if not causal:
        return np.ones((n_q, kv_len), bool)
    return t <= (q_pos0 + np.arange(n_q))[:, None]


def _softmax_rows(s: np.ndarray, vis: np.ndarray):
    """p = exp(s - max) over visible entries (0 elsewhere) and its row sum."""
    s = np.where(vis, s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.where(vis, np.exp(s - m), 0.0)
    return p, p.sum(axis=-1, keepdims=True)


def attend_dense(q, k_hat, v_hat, alpha, kv_len, causal=False, q_pos0=0):
    """Single-pass softmax attention.

    q [B][H_q][n_q][D], k_hat/v_hat [B][H_kv][S][D] (any float; used as float64).
    Returns float64 [B][H_q][n_q][D]. Rows with no visible token return zeros.
    """
    q = np.asarray(q, np.float64)
    B, Hq, nq, D = q.shape
    Hkv = k_hat.shape[1]
    g = Hq // Hkv
    vis = visible_mask(nq, kv_len, causal, q_pos0)
    out = np.zeros((B, Hq, nq, D))
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            K = np.asarray(k_hat[b, kh, :kv_len], np.float64)
            V = np.asarray(v_hat[b, kh, :kv_len], np.float64)
            s = alpha * (q[b, h] @ K.T)
            p, l = _softmax_rows(s, vis)
            with np.errstate(invalid="ignore", divide="ignore"):
                out[b, h] = np.where(l > 0, (p @ V) / l, 0.0)
    return out


def chunk_partials(s: np.ndarray, vis: np.ndarray, V: np.ndarray, lo: int, hi: int):
    """(m_c, l_c, o_c) of one chunk [lo, hi) for score rows s[n][S] (phase one of split-K)."""
    sc = np.where(vis[:, lo:hi], s[:, lo:hi], -np.inf)
    m = np.max(sc, axis=-1) if hi > lo else np.full(s.shape[0], -np.inf)
    fin = np.isfinite(m)
    mm = np.where(fin, m, 0.0)
    p = np.where(vis[:, lo:hi], np.exp(sc - mm[:, None]), 0.0)
    return m, p.sum(axis=-1), p @ V[lo:hi]


def lse_combine(ms, ls, os_):
    """Phase two of split-K: combine chunk partials by the online-softmax correction (R15)."""
    ms = np.asarray(ms)            # [C][n]
    ls = np.asarray(ls)            # [C][n]
    os_ = np.asarray(os_)          # [C][n][D]
    M = np.max(ms, axis=0)
    Mf = np.where(np.isfinite(M), M, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - Mf[None, :]), 0.0)
    L = np.sum(ls * w, axis=0)
    O = np.sum(os_ * w[:, :, None], axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(L[:, None] > 0, O / L[:, None], 0.0)


def attend_split(q, k_hat, v_hat, alpha, kv_len, causal=False, q_pos0=0, chunk=512):
    """Split-K attention: chunks [c*chunk, (c+1)*chunk) (last one partial), LSE-combined."""
    q = np.asarray(q, np.float64)
    B, Hq, nq, D = q.shape
    Hkv = k_hat.shape[1]
    g = Hq // Hkv
    vis = visible_mask(nq, kv_len, causal, q_pos0)
    out = np.zeros((B, Hq, nq, D))
    C = -(-kv_len // chunk)
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            K = np.asarray(k_hat[b, kh, :kv_len], np.float64)
            V = np.asarray(v_hat[b, kh, :kv_len], np.float64)
            s = alpha * (q[b, h] @ K.T)
            parts = [chunk_partials(s, vis, V, c * chunk, min(kv_len, (c + 1) * chunk)) for c in range(C)]
            out[b, h] = lse_combine([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
    return out


def attend_causal_skip(q, k_hat, v_hat, alpha, kv_len, q_pos0=0):
    """Causal attention computed only over each row's visible prefix (no mask): row i reads
    tokens [0, min(kv_len, q_pos0 + i + 1)) (causal-skip, tract discussion #2402)."""
    q = np.asarray(q, np.float64)
    B, Hq, nq, D = q.shape
    g = Hq // k_hat.shape[1]
    out = np.zeros((B, Hq, nq, D))
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            for i in range(nq):
                n = min(kv_len, q_pos0 + i + 1)
                if n <= 0:
                    continue
                K = np.asarray(k_hat[b, kh, :n], np.float64)
                V = np.asarray(v_hat[b, kh, :n], np.float64)
                s = alpha * (K @ q[b, h, i])
                p = np.exp(s - s.max())
                out[b, h, i] = (p @ V) / p.sum()
    return out


# ------------------------------------------------------------------ Hadamard path
def prep_q_hadamard(q32: np.ndarray):
    """Query preparation for the integer-domain score (reading R8).

    q_rot = rotate(q) in float32; s_q = amax(|q_rot|) / 127 in float32 per row;
    q8 = clamp(rint(q_rot / s_q), -127, 127) (all zero when s_q == 0).
    Returns (q_rot float32, s_q float32, q8 int8).
    """
    q_rot = Q.rotate(q32)
    amax = np.max(np.abs(q_rot), axis=-1)
    s_q = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(q_rot / s_q[..., None])
    q8 = np.where(s_q[..., None] > 0, np.clip(r, -127, 127), 0.0).astype(np.int8)
    return q_rot, s_q, q8


def scores_int(q8: np.ndarray, k_codes: np.ndarray) -> np.ndarray:
    """Exact integer dots int8(q) . int4(k): q8 [..., R, D], k_codes [..., S, D] -> int64 [..., R, S]."""
    return np.matmul(q8.astype(np.int64), np.swapaxes(k_codes.astype(np.int64), -1, -2))


def attend_hadamard(q32, k_payload, k_scale, v_payload, v_scale, k_ring, v_ring, n_recent,
                    alpha, kv_len, causal=False, q_pos0=0, layout="had_int4", v_layout=None):
    """Hadamard-int4 attention with the exact float32 recent window, float64 accumulation.

    q32 [B][H_q][n_q][D] float32; k/v_payload [B][H_kv][S][row bytes] uint8 of `layout` (K) and
    `v_layout` (V, default the same; had_int4: D/2 bytes, had_int2: D/4); k/v_scale [B][H_kv][S]
    float32; k/v_ring [B][H_kv][n_recent][D] float32 (rotated rows) or None.
    Returns (out float64 [B][H_q][n_q][D], scores_i32 int64 [B][H_q][n_q][n_body]).
    """
    q32 = np.asarray(q32, np.float32)
    B, Hq, nq, D = q32.shape
    Hkv = k_payload.shape[1]
    g = Hq // Hkv
    nw = min(n_recent, kv_len)
    n_body = kv_len - nw
    q_rot, s_q, q8 = prep_q_hadamard(q32)
    Hd = Q.hadamard_matrix(D) / math.sqrt(D)
    vis = visible_mask(nq, kv_len, causal, q_pos0)
    out = np.zeros((B, Hq, nq, D))
    si = np.zeros((B, Hq, nq, n_body), np.int64)
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            kc = Q.hadamard_layout_codes(layout, k_payload[b, kh, :n_body], D)
            vc = Q.hadamard_layout_codes(v_layout or layout, v_payload[b, kh, :n_body], D).astype(np.float64)
            ks = np.asarray(k_scale[b, kh, :n_body], np.float64)
            vs = np.asarray(v_scale[b, kh, :n_body], np.float64)
            i32 = scores_int(q8[b, h], kc)                                   # [nq][n_body]
            si[b, h] = i32
            s_body = alpha * s_q[b, h].astype(np.float64)[:, None] * ks[None, :] * i32
            V_body = vc * vs[:, None]
            if nw:
                slots = np.arange(n_body, kv_len) % n_recent
                Kw = np.asarray(k_ring[b, kh, slots], np.float64)
                Vw = np.asarray(v_ring[b, kh, slots], np.float64)
                s_win = alpha * (q_rot[b, h].astype(np.float64) @ Kw.T)
                s = np.concatenate([s_body, s_win], axis=1)
                V = np.concatenate([V_body, Vw], axis=0)
            else:
                s, V = s_body, V_body
            p, l = _softmax_rows(s, vis)
            with np.errstate(invalid="ignore", divide="ignore"):
                o_rot = np.where(l > 0, (p @ V) / l, 0.0)
            out[b, h] = o_rot @ Hd.T                                         # un-rotate
    return out, si


# ------------------------------------------------------------------ cache model
class OracleCache:
    """CPU model of a caller-owned packed cache [B][H_kv][capacity][...].

    Planes: payload uint8 [B][H_kv][cap][row_bytes]; scale float16 [B][H_kv][cap][D/32]
    (float32 [B][H_kv][cap] for Hadamard); zero float16 [B][H_kv][cap][D/32] (asymmetric);
    ring float32 [B][H_kv][n_recent][D] (Hadamard with n_recent > 0). K and V each.
    """

    def __init__(self, layout, batch, n_kv_heads, head_dim, capacity, n_recent=0):
        self.layout, self.B, self.H, self.D, self.cap = layout, batch, n_kv_heads, head_dim, capacity
        self.lay = dict(zip(("k", "v"), Q.plane_layouts(layout)))      # each plane's own layout
        self.n_recent = n_recent if Q.is_hadamard(layout) else 0
        nb = head_dim // Q.BLOCK
        self.planes = {}
        for t in ("k", "v"):
            lt = self.lay[t]
            rb = Q.row_bytes(lt, head_dim)
            p = {"payload": np.zeros((batch, n_kv_heads, capacity, rb), np.uint8)}
            if lt in Q.HADAMARD:
                p["scale"] = np.zeros((batch, n_kv_heads, capacity), np.float32)
                if self.n_recent:
                    p["ring"] = np.zeros((batch, n_kv_heads, self.n_recent, head_dim), np.float32)
            else:
                p["scale"] = np.zeros((batch, n_kv_heads, capacity, nb), np.float16)
                if lt == "asym4_g32":
                    p["zero"] = np.zeros((batch, n_kv_heads, capacity, nb), np.float16)
            self.planes[t] = p

    def store(self, k_new, v_new, pos0):
        """Append rows k_new/v_new [B][H_kv][n_new][D] (float32 values) at [pos0, pos0+n_new).
        Hadamard: the last min(n_new, n_recent) of them also go to ring slot t mod n_recent."""
        n_new = k_new.shape[2]
        if pos0 < 0 or pos0 + n_new > self.cap:
            raise ValueError("store beyond capacity")
        for t, x in (("k", k_new), ("v", v_new)):
            st = Q.quantize(self.lay[t], np.asarray(x, np.float32))
            pl = self.planes[t]
            for name in ("payload", "scale", "zero"):
                if name in st and name in pl:
                    pl[name][:, :, pos0:pos0 + n_new] = st[name]
            if self.n_recent:
                first = max(0, n_new - self.n_recent)
                for j in range(first, n_new):
                    pl["ring"][:, :, (pos0 + j) % self.n_recent] = st["rot"][:, :, j]

    def dequantized(self, t, kv_len):
        pl = self.planes[t]
        sub = {k: v[:, :, :kv_len] for k, v in pl.items() if k != "ring"}
        return Q.dequantize(self.lay[t], sub, self.D)

    def attend(self, q, alpha, kv_len, causal=False, q_pos0=0, chunk=None):
        """Attention of q [B][H_q][n_q][D] (float32 values) over the first kv_len tokens.
        Returns float64 [B][H_q][n_q][D] (and int64 body scores for Hadamard as a 2-tuple)."""
        if Q.is_hadamard(self.layout):
            k, v = self.planes["k"], self.planes["v"]
            return attend_hadamard(q, k["payload"], k["scale"], v["payload"], v["scale"],
                                   k.get("ring"), v.get("ring"), self.n_recent, alpha, kv_len,
                                   causal, q_pos0, self.lay["k"], self.lay["v"])
        K = self.dequantized("k", kv_len)
        V = self.dequantized("v", kv_len)
        if chunk:
            return attend_split(q, K, V, alpha, kv_len, causal, q_pos0, chunk)
        return attend_dense(q, K, V, alpha, kv_len, causal, q_pos0)
