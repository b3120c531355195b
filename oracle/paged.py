"""Oracle of the paged KV cache: a page pool shared by the sequences of a batch, a block table,
and one length per sequence.

TEST INFRASTRUCTURE ONLY (see the package docstring).

FreeToken PR #268 ("Scope": only the paged full-attention KV pool is quantized; "Changes":
mha_pool allocates the packed buffer plus a separate scale buffer per spec) keeps the quantized
cache in a paged pool. The pages leave the pool's shape open; the reading taken here (and by the
library) is:
  * planes [n_pages][H_kv][page_size][...] with the contiguous cache's per-row byte layout;
  * block table [batch][max_pages_per_seq]: token t of sequence b is row t % page_size of pool
    page table[b][t // page_size];
  * every sequence has its own length L_b; a causal call's n_q query rows are the sequence's
    newest tokens (query row i sits at position L_b - n_q + i); the Hadamard exact-f32 window
    is the newest min(n_recent, L_b) tokens of each sequence, in a ring per sequence.

The model is deliberately plain: a store scatters each quantized row to its page; attention
gathers each sequence's rows back into a contiguous `OracleCache` of that one sequence and runs
the contiguous oracle on it. A row that sees no token gets zeros.
"""
from __future__ import annotations

import numpy as np

from . import quant as Q
from .attention import OracleCache


class OraclePagedCache:
    """CPU model of a caller-owned paged pool and its block table."""

    def __init__(self, layout, batch, n_kv_heads, head_dim, page_size, n_pages, max_pages_per_seq, n_recent=0,
                 table=None):
        self.layout, self.B, self.H, self.D = layout, batch, n_kv_heads, head_dim
        self.P, self.n_pages, self.max_pages = page_size, n_pages, max_pages_per_seq
        self.cap = page_size * max_pages_per_seq
        self.lay = dict(zip(("k", "v"), Q.plane_layouts(layout)))      # each plane's own layout
        self.n_recent = n_recent if Q.is_hadamard(layout) else 0
        nb = head_dim // Q.BLOCK
        pool = (n_pages, n_kv_heads, page_size)
        self.planes = {}
        for t in ("k", "v"):
            lt = self.lay[t]
            p = {"payload": np.zeros(pool + (Q.row_bytes(lt, head_dim),), np.uint8)}
            if lt in Q.HADAMARD:
                p["scale"] = np.zeros(pool, np.float32)
                if self.n_recent:
                    p["ring"] = np.zeros((batch, n_kv_heads, self.n_recent, head_dim), np.float32)
            else:
                p["scale"] = np.zeros(pool + (nb,), np.float16)
                if lt == "asym4_g32":
                    p["zero"] = np.zeros(pool + (nb,), np.float16)
            self.planes[t] = p
        self.table = np.zeros((batch, max_pages_per_seq), np.int64) if table is None else np.asarray(table, np.int64)

    def locate(self, b: int, t: int):
        """(pool page, row within the page) of token t of sequence b."""
        return int(self.table[b, t // self.P]), t % self.P

    def store(self, k_new, v_new, positions):
        """Append rows k_new/v_new [B][H_kv][n_new][D] (float32 values): sequence b's row j goes to
        position positions[b] + j. Rows outside [0, capacity) are dropped. Hadamard: the last
        min(n_new, n_recent) rows of each sequence also go to its ring slot (position mod n_recent)."""
        n_new = k_new.shape[2]
        for t, x in (("k", k_new), ("v", v_new)):
            st = Q.quantize(self.lay[t], np.asarray(x, np.float32))
            pl = self.planes[t]
            for b in range(self.B):
                for j in range(n_new):
                    pos = int(positions[b]) + j
                    if not 0 <= pos < self.cap:
                        continue
                    pg, r = self.locate(b, pos)
                    for name in ("payload", "scale", "zero"):
                        if name in st and name in pl:
                            pl[name][pg, :, r] = st[name][b, :, j]
                    if self.n_recent and j >= n_new - self.n_recent:
                        pl["ring"][b, :, pos % self.n_recent] = st["rot"][b, :, j]

    def sequence(self, b: int, length: int) -> OracleCache:
        """The first `length` tokens of sequence b as a contiguous one-sequence cache."""
        c = OracleCache(self.layout, 1, self.H, self.D, max(length, 1), self.n_recent)
        for t in ("k", "v"):
            src, dst = self.planes[t], c.planes[t]
            for pos in range(length):
                pg, r = self.locate(b, pos)
                for name in ("payload", "scale", "zero"):
                    if name in src:
                        dst[name][0, :, pos] = src[name][pg, :, r]
            if self.n_recent:
                dst["ring"][0] = src["ring"][b]
        return c

    def attend(self, q, alpha, seq_lens, causal=False):
        """Attention of q [B][H_q][n_q][D] (float32 values): sequence b over its first seq_lens[b]
        tokens; causal rows at positions seq_lens[b] - n_q + i. Float64 [B][H_q][n_q][D]."""
        q = np.asarray(q, np.float32)
        B, Hq, nq, D = q.shape
        out = np.zeros((B, Hq, nq, D))
        for b in range(B):
            L = int(seq_lens[b])
            if L <= 0:
                continue
            r = self.sequence(b, L).attend(q[b:b + 1], alpha, L, causal, L - nq)
            out[b] = (r[0] if isinstance(r, tuple) else r)[0]
        return out
