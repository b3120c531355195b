"""Planted mistakes in the oracle (on the CPU) must be caught by the pins.

Each case patches one plausible error into the oracle: a swapped nibble order, a wrong
magnitude or scale divisor (Q4_0, Q6_0, Q8_0, Hadamard int4, the int8 query, asymmetric), a
transposed high-plane field, a wrong GQA index, a dropped window term, a window ring slot off by
one, a missing rescale in the chunk combine, a rotation without its 1/sqrt(D), an asymmetric
zero-point taken at the maximum or subtracted, a paged token located at the wrong page or row. Cases inside a function body replace one
expression of the oracle's own source for the test's duration (`_mutant`). It then runs the pin
tests that should fail and checks that at least one does.
"""
import numpy as np
import pytest

import oracle.attention as A
import oracle.quant as Q
from tests import test_oracle_pins as P


def _fails(*tests):
    for t in tests:
        try:
            t()
        except AssertionError:
            return True
    return False


def test_swapped_nibble_order_is_caught(monkeypatch):
    def bad_pack(n):
        n = np.asarray(n).astype(np.uint8) & 0xF
        return (n[..., 1::2] | (n[..., 0::2] << 4)).astype(np.uint8)
    monkeypatch.setattr(Q, "pack_nibbles", bad_pack)
    assert _fails(lambda: P.test_q4_0_nibble_position(3))


def test_magnitude_7_is_caught(monkeypatch):
    orig = Q._symmetric_codes

    def bad_quant(x):
        xb = Q._blocks(x)
        amax = np.max(np.abs(xb), axis=-1)
        s16 = Q.fp16_round(amax / np.float32(7.0))
        q = orig(xb, s16.astype(np.float32), -8, 7)
        return Q.pack_nibbles(q & 0xF).reshape(x.shape[:-1] + (-1,)), s16
    monkeypatch.setattr(Q, "quantize_q4_0", bad_quant)
    assert _fails(P.test_q4_0_every_code_through_read_formula, P.test_q4_0_saturation_and_half_even)


def test_q6_high_plane_interleave_is_caught(monkeypatch):
    orig = Q.quantize_q6_0

    def bad(x):
        p, s = orig(x)
        pb = p.reshape(p.shape[:-1] + (-1, 24)).copy()
        hb = pb[..., 16:].astype(np.uint16)
        # bit pairs in the reverse order inside each high byte
        rev = ((hb & 3) << 6) | (((hb >> 2) & 3) << 4) | (((hb >> 4) & 3) << 2) | ((hb >> 6) & 3)
        pb[..., 16:] = rev.astype(np.uint8)
        return pb.reshape(p.shape), s
    monkeypatch.setattr(Q, "quantize_q6_0", bad)
    assert _fails(lambda: P.test_q6_0_plane_positions(1))


def test_fwht_sign_error_is_caught(monkeypatch):
    orig = Q.fwht

    def bad(x, dtype=np.float32):
        y = orig(x, dtype)
        y[..., -1] = -y[..., -1]
        return y
    monkeypatch.setattr(Q, "fwht", bad)
    assert _fails(lambda: P.test_fwht_equals_dense_sylvester(8))


def test_wrong_gqa_index_is_caught(monkeypatch):
    def bad(q, k_hat, v_hat, alpha, kv_len, causal=False, q_pos0=0):
        Hkv = k_hat.shape[1]
        # query head h reading kv head h % H_kv instead of h // (H_q / H_kv)
        perm = np.array([h % Hkv for h in range(q.shape[1])])
        g = q.shape[1] // Hkv
        k2 = np.repeat(k_hat, g, axis=1)[:, [p * g for p in perm]]
        v2 = np.repeat(v_hat, g, axis=1)[:, [p * g for p in perm]]
        return orig(q, k2, v2, alpha, kv_len, causal, q_pos0)
    orig = A.attend_dense
    monkeypatch.setattr(A, "attend_dense", bad)
    assert _fails(P.test_gqa_mapping_reads_kv_head_q_over_gqa)


def test_dropped_window_is_caught(monkeypatch):
    orig = A.attend_hadamard

    def bad(q32, k_payload, k_scale, v_payload, v_scale, k_ring, v_ring, n_recent, *a, **kw):
        return orig(q32, k_payload, k_scale, v_payload, v_scale, None, None, 0, *a, **kw)
    monkeypatch.setattr(A, "attend_hadamard", bad)
    assert _fails(P.test_hadamard_full_window_is_exact_attention)


def test_combine_without_rescale_is_caught(monkeypatch):
    def bad(ms, ls, os_):
        ls, os_ = np.asarray(ls), np.asarray(os_)
        return np.sum(os_, axis=0) / np.sum(ls, axis=0)[:, None]
    monkeypatch.setattr(A, "lse_combine", bad)
    assert _fails(lambda: P.test_split_k_equals_single_pass(16))


def test_transposed_causal_limit_is_caught(monkeypatch):
    def bad(n_q, kv_len, causal, q_pos0):
        t = np.arange(kv_len)[None, :]
        if not causal:
            return np.ones((n_q, kv_len), bool)
        return t < (q_pos0 + np.arange(n_q))[:, None]          # off by one: excludes the diagonal
    monkeypatch.setattr(A, "visible_mask", bad)
    assert _fails(P.test_attention_brute_force_gqa_causal)


def test_q8_0_magnitude_127_is_caught(monkeypatch):
    # the GGUF-style amax / 127 instead of the family rule's amax / 128
    def bad(x):
        xb = Q._blocks(x)
        amax = np.max(np.abs(xb), axis=-1)
        d16 = Q.fp16_round(amax / np.float32(127.0))
        d = d16.astype(np.float32)[..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.rint(xb / d)
        q = np.where(d > 0, np.clip(r, -128, 127), 0.0).astype(np.int32)
        return (q & 0xFF).astype(np.uint8).reshape(x.shape[:-1] + (-1,)), d16
    monkeypatch.setattr(Q, "quantize_q8_0", bad)
    assert _fails(P.test_q8_0_every_code_through_read_formula, lambda: P.test_q8_0_byte_position_and_saturation(1))


def test_int2_field_order_is_caught(monkeypatch):
    # value 4j+i at bits 6-2i instead of 2i
    def bad(f):
        f = np.asarray(f, dtype=np.uint8) & 0x3
        f = f.reshape(f.shape[:-1] + (-1, 4))
        return (f[..., 3] | (f[..., 2] << 2) | (f[..., 1] << 4) | (f[..., 0] << 6)).astype(np.uint8)
    monkeypatch.setattr(Q, "pack_pairs_of_bits", bad)
    assert _fails(lambda: P.test_int2_field_positions(1))


def test_int2_read_without_sign_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "read_int2", lambda v: np.asarray(v).astype(np.int32))
    assert _fails(P.test_int2_read_formula_every_field, P.test_hadamard_int2_codes_and_scale)


def _mutant(mod, name, old, new):
    """`mod.name` with one expression of its source replaced (a planted mistake for one test)."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(getattr(mod, name)))
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(mod))
    exec(compile(src.replace(old, new), f"<mutant {mod.__name__}.{name}>", "exec"), ns)
    return ns[name]


def test_asym_scale_over_16_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "quantize_asym4_g32",
                        _mutant(Q, "quantize_asym4_g32", "rng / np.float32(15.0)", "rng / np.float32(16.0)"))
    assert _fails(P.test_asym_exact_grid, P.test_asym_constant_group_and_bound)


def test_asym_zero_point_at_the_maximum_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "quantize_asym4_g32", _mutant(Q, "quantize_asym4_g32", "z16 = fp16_round(mn)",
                                                         "z16 = fp16_round(mx)"))
    assert _fails(P.test_asym_exact_grid, P.test_asym_constant_group_and_bound)


def test_asym_reconstruction_sign_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "dequantize_asym4_g32",
                        _mutant(Q, "dequantize_asym4_g32", "[..., None] + np.asarray(zero)",
                                "[..., None] - np.asarray(zero)"))
    assert _fails(P.test_asym_exact_grid, P.test_asym_constant_group_and_bound)


def test_hadamard_int4_scale_over_8_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "quantize_hadamard_int4",
                        _mutant(Q, "quantize_hadamard_int4", "amax / np.float32(7.0)", "amax / np.float32(8.0)"))
    assert _fails(P.test_hadamard_int4_codes_and_scale)


def test_rotation_without_normalisation_is_caught(monkeypatch):
    import inspect
    src = inspect.getsource(Q.rotate)
    # the rotation's 1/sqrt(D) factor, whatever name it has in the source, becomes 1
    body = [ln for ln in src.splitlines() if "inv_sqrt_f32" in ln]
    assert body, "rotate() scales by inv_sqrt_f32(D)"
    monkeypatch.setattr(Q, "inv_sqrt_f32", lambda d: np.float32(1.0))
    assert _fails(P.test_hadamard_int4_codes_and_scale, P.test_rotation_preserves_scores)


def test_window_ring_slot_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(A, "attend_hadamard",
                        _mutant(A, "attend_hadamard", "slots = np.arange(n_body, kv_len) % n_recent",
                                "slots = np.arange(n_body + 1, kv_len + 1) % n_recent"))
    assert _fails(P.test_recent_window_semantics, P.test_hadamard_full_window_is_exact_attention)


def test_combine_without_rescaled_sums_is_caught(monkeypatch):
    monkeypatch.setattr(A, "lse_combine", _mutant(A, "lse_combine", "L = np.sum(ls * w, axis=0)",
                                                  "L = np.sum(ls, axis=0)"))
    assert _fails(lambda: P.test_split_k_equals_single_pass(64), lambda: P.test_split_k_equals_single_pass(7))


def test_query_scale_over_128_is_caught(monkeypatch):
    monkeypatch.setattr(A, "prep_q_hadamard", _mutant(A, "prep_q_hadamard", "amax / np.float32(127.0)",
                                                      "amax / np.float32(128.0)"))
    assert _fails(P.test_integer_scores_brute_force, P.test_hadamard_body_on_exact_grid_matches_plain_attention,
                  P.test_error_envelopes)


def test_q6_0_magnitude_31_is_caught(monkeypatch):
    monkeypatch.setattr(Q, "quantize_q6_0", _mutant(Q, "quantize_q6_0", "amax / np.float32(32.0)",
                                                    "amax / np.float32(31.0)"))
    assert _fails(P.test_q6_0_every_code_through_read_formula, P.test_q6_0_saturation)


def test_paged_row_and_page_swapped_is_caught(monkeypatch):
    from oracle import paged as PG
    from tests import test_oracle_paged as PP
    monkeypatch.setattr(PG.OraclePagedCache, "locate",
                        _mutant(PG.OraclePagedCache, "locate", "int(self.table[b, t // self.P]), t % self.P",
                                "int(self.table[b, min(t % self.P, self.max_pages - 1)]), "
                                "min(t // self.P, self.P - 1)"))
    assert _fails(PP.test_probe_token_lands_at_table_page_and_row)


def test_paged_page_off_by_one_is_caught(monkeypatch):
    from oracle import paged as PG
    from tests import test_oracle_paged as PP
    monkeypatch.setattr(PG.OraclePagedCache, "locate",
                        _mutant(PG.OraclePagedCache, "locate", "self.table[b, t // self.P]",
                                "self.table[b, min(t // self.P + 1, self.max_pages - 1)]"))
    assert _fails(PP.test_probe_token_lands_at_table_page_and_row)
