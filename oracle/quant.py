"""Oracle quantizers: Q4_0, Q6_0, Q8_0, per-token Hadamard int4 / int2 and per-group
asymmetric int4.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain numpy, float32 IEEE arithmetic
with round-half-to-even, one operation at a time in the order written below. Every function
returns the exact bytes/scales that a conforming store must produce.

Readings of points the pages leave open (each one a single constant or step here):
  R1  x / scale is rounded half-to-even to an integer (numpy `rint`).
  R2  x / scale is a correctly rounded float32 division (not a multiply by a reciprocal).
  R3  codes are computed against the *stored* fp16 scale, so writer and reader agree.
  R4  Q4_0: scale = amax / 8, codes clamped to [-8, 7] (so +amax saturates to 7).
  R5  Q6_0: scale = amax / 32, codes clamped to [-32, 31].
  R6  Q6_0 high plane: the top two bits of value 4k+i sit at bits 2i..2i+1 of high byte k.
  R7  Hadamard int4: symmetric, zero-point free, scale = amax / 7, codes in [-7, 7].
  R9  FWHT: radix-2 butterflies (a, b) -> (a + b, a - b), half-span 1, 2, 4, ..., D/2 in that
      order, natural (Sylvester) ordering, then each output multiplied by the float32 nearest
      to 1/sqrt(D).
  R10 asymmetric g=32: scale = (max - min) / 15 and zero = min, both stored as fp16; codes
      q = rint((x - zero) / scale) clamped to [0, 15], stored unsigned.
  R17 all-zero block (or a scale that rounds to fp16 zero) -> every code 0; fp16 scales and
      zeros saturate at +-65504; -0.0 quantises to code 0. Non-finite inputs are unspecified.
  R24 Q8_0 (the pages give only its density, 1.0625 bytes/element): per 32 values 32 int8 code
      bytes and one fp16 scale; by the family rule of R4/R5 (magnitude 2^(bits-1)) scale =
      amax / 128 and codes clamped to [-128, 127], byte i = value i in two's complement, read
      back as (v ^ 0x80) - 0x80.
  R25 Hadamard int2 (the body below four bits that needs the exact-f32 window): the int4 layout
      of R7 with two bits: symmetric, zero-point free, scale = amax / 1, codes in [-1, 1]; four
      codes per byte, value 4j+i at bits 2i..2i+1 of byte j (two's complement), read back as
      (v ^ 2) - 2.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 32                     # values per Q4_0/Q6_0/asym block along head_dim
F16_MAX = np.float32(65504.0)

LAYOUTS = ("q4_0", "q6_0", "had_int4", "asym4_g32", "q8_0", "had_int2")
HADAMARD = ("had_int4", "had_int2")       # layouts in the rotated basis with a per-token f32 scale


def plane_layouts(layout: str):
    """(K layout, V layout) of a cache layout name. Mixed K/V precision (Open-TQ-Metal, Section 5:
    value quantisation costs more output quality than key quantisation) is written "k+v", e.g.
    "q4_0+q8_0"; both planes are block layouts, or both are Hadamard layouts (one rotated basis)."""
    k, _, v = layout.partition("+")
    v = v or k
    if k not in LAYOUTS or v not in LAYOUTS or ((k in HADAMARD) != (v in HADAMARD)):
        raise ValueError(f"unsupported layout {layout!r}")
    return k, v


def is_hadamard(layout: str) -> bool:
    return plane_layouts(layout)[0] in HADAMARD


# ------------------------------------------------------------------ sizes (closed forms)
def row_bytes(layout: str, head_dim: int) -> int:
    """Packed payload bytes of one token row of one head.

    Q4_0: 16 payload bytes per 32 values; Q6_0: 24 (16-byte low plane + 8-byte high plane)
    ("Storage layouts", FreeToken PR #268). Hadamard int4: ceil(D/2) bytes per token
    (tract discussion #2402, "Architecture: State"). Asymmetric g=32: two values per byte
    (Open-TQ-Metal, per-group asymmetric int4 background paragraph).
    """
    nb = head_dim // BLOCK
    return {"q4_0": 16 * nb, "q6_0": 24 * nb, "had_int4": (head_dim + 1) // 2,
            "asym4_g32": 16 * nb, "q8_0": 32 * nb, "had_int2": (head_dim + 3) // 4}[layout]


def param_bytes(layout: str, head_dim: int) -> int:
    """Bytes of scale (+ zero-point) per token row of one head."""
    nb = head_dim // BLOCK
    return {"q4_0": 2 * nb, "q6_0": 2 * nb, "had_int4": 4, "asym4_g32": 4 * nb, "q8_0": 2 * nb,
            "had_int2": 4}[layout]


# ------------------------------------------------------------------ helpers
def fp16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest float16 (half-to-even), saturating at +-65504. Returns float16."""
    x = np.asarray(x, dtype=np.float32)
    return np.clip(x, -F16_MAX, F16_MAX).astype(np.float16)


def inv_sqrt_f32(d: int) -> np.float32:
    """The float32 nearest to 1/sqrt(d) (R9)."""
    return np.float32(1.0 / math.sqrt(d))


def read_q4_0(v: np.ndarray) -> np.ndarray:
    """Read-side sign extension of a Q4_0 nibble: (v ^ 0x8) - 0x8 ("Storage layouts", q4_0)."""
    v = np.asarray(v).astype(np.int32)
    return (v ^ 0x8) - 0x8


def read_q6_0(v: np.ndarray) -> np.ndarray:
    """Read-side sign extension of a 6-bit Q6_0 value: (v ^ 0x20) - 0x20 ("Storage layouts", q6_0)."""
    v = np.asarray(v).astype(np.int32)
    return (v ^ 0x20) - 0x20


def pack_nibbles(n: np.ndarray) -> np.ndarray:
    """Byte j holds value 2j in its low nibble and value 2j+1 in its high nibble."""
    n = np.asarray(n).astype(np.uint8) & 0xF
    if n.shape[-1] % 2:
        n = np.concatenate([n, np.zeros(n.shape[:-1] + (1,), np.uint8)], axis=-1)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(b: np.ndarray, count: int) -> np.ndarray:
    """Inverse of pack_nibbles: the raw 4-bit fields, in value order."""
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out[..., :count]


def _blocks(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    if D % BLOCK:
        raise ValueError("head_dim must be a multiple of 32")
    return x.reshape(x.shape[:-1] + (D // BLOCK, BLOCK))


def _symmetric_codes(xb: np.ndarray, s: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """q = clamp(rint(x / s), lo, hi) per element, all-zero where s == 0 (R1, R2, R17)."""
    s_b = s[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(xb / s_b)          # float32 division, correctly rounded; then half-even
    q = np.clip(r, lo, hi)
    q = np.where(s_b > 0, q, 0.0)
    return q.astype(np.int32)


# ------------------------------------------------------------------ Q4_0
def quantize_q4_0(x: np.ndarray):
    """Q4_0 store of rows x[..., D] (float32 values).

    Per 32 values along head_dim one fp16 scale and 16 payload bytes ("Storage layouts",
    FreeToken PR #268): magnitude 8, range [-8, 7] (R4); byte j = value 2j low nibble,
    value 2j+1 high nibble; the nibble is the two's-complement low four bits of the code,
    which the page's read formula (v ^ 0x8) - 0x8 sign-extends.

    Returns (payload uint8 [..., 16*nb], scale float16 [..., nb]).
    """
    xb = _blocks(x)
    amax = np.max(np.abs(xb), axis=-1)
    d = amax / np.float32(8.0)
    s16 = fp16_round(d)
    s = s16.astype(np.float32)
    q = _symmetric_codes(xb, s, -8, 7)
    payload = pack_nibbles(q & 0xF)                          # [..., nb, 16]
    return payload.reshape(x.shape[:-1] + (-1,)), s16


def dequantize_q4_0(payload: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x_hat = ((v ^ 8) - 8) * scale, in float64 (exact)."""
    payload = np.asarray(payload, np.uint8)
    nb = scale.shape[-1]
    v = unpack_nibbles(payload.reshape(payload.shape[:-1] + (nb, 16)), BLOCK)
    code = read_q4_0(v).astype(np.float64)
    x = code * np.asarray(scale).astype(np.float64)[..., None]
    return x.reshape(payload.shape[:-1] + (nb * BLOCK,))


# ------------------------------------------------------------------ Q6_0
def quantize_q6_0(x: np.ndarray):
    """Q6_0 store: per 32 values a 16-byte low plane (low four bits, Q4_0 nibble order) then an
    8-byte high plane (top two bits, four values per byte at bit positions 0, 2, 4, 6) and one
    fp16 scale ("Storage layouts", FreeToken PR #268). Magnitude 32, range [-32, 31] (R5);
    value 4k+i goes to bits 2i of high byte k (R6).

    Returns (payload uint8 [..., 24*nb], scale float16 [..., nb]).
    """
    xb = _blocks(x)
    amax = np.max(np.abs(xb), axis=-1)
    d = amax / np.float32(32.0)
    s16 = fp16_round(d)
    s = s16.astype(np.float32)
    q = _symmetric_codes(xb, s, -32, 31)
    u = (q & 0x3F).astype(np.uint8)                            # 6-bit two's complement
    low = pack_nibbles(u & 0xF)                                # [..., nb, 16]
    top = (u >> 4) & 0x3                                       # [..., nb, 32]
    top4 = top.reshape(top.shape[:-1] + (8, 4)).astype(np.uint8)
    high = (top4[..., 0] | (top4[..., 1] << 2) | (top4[..., 2] << 4) | (top4[..., 3] << 6)).astype(np.uint8)
    payload = np.concatenate([low, high], axis=-1)             # [..., nb, 24]
    return payload.reshape(x.shape[:-1] + (-1,)), s16


def q6_0_fields(payload: np.ndarray, nb: int) -> np.ndarray:
    """The 6-bit stored values v = low | high << 4 of each block, in value order."""
    p = np.asarray(payload, np.uint8).reshape(payload.shape[:-1] + (nb, 24))
    low = unpack_nibbles(p[..., :16], BLOCK).astype(np.int32)
    hb = p[..., 16:].astype(np.int32)                          # [..., nb, 8]
    top = np.stack([(hb >> (2 * i)) & 3 for i in range(4)], axis=-1).reshape(hb.shape[:-1] + (BLOCK,))
    return low | (top << 4)


def dequantize_q6_0(payload: np.ndarray, scale: np.ndarray) -> np.ndarray:
    nb = scale.shape[-1]
    v = q6_0_fields(payload, nb)
    code = read_q6_0(v).astype(np.float64)
    x = code * np.asarray(scale).astype(np.float64)[..., None]
    return x.reshape(np.asarray(payload).shape[:-1] + (nb * BLOCK,))


# ------------------------------------------------------------------ FWHT + Hadamard int4
def fwht(x: np.ndarray, dtype=np.float32) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis (R9).

    O(D log D) radix-2 butterflies (the rotation of tract discussion #2402, "What's done":
    "FWHT, O(D log D)"). Stage with half-span h pairs element j with j + h inside each block
    of 2h and replaces (a, b) by (a + b, a - b); h runs 1, 2, 4, ..., D/2. Every add/subtract
    is rounded in `dtype`. The result equals the Sylvester matrix H (H_ij = (-1)^popcount(i&j))
    times x, up to rounding.
    """
    y = np.array(x, dtype=dtype, copy=True)
    D = y.shape[-1]
    if D & (D - 1):
        raise ValueError("FWHT length must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < D:
        y = y.reshape(lead + (D // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(lead + (D,))
        h *= 2
    return y


def rotate(x: np.ndarray) -> np.ndarray:
    """Orthonormal rotation y = FWHT(x) * fp32(1/sqrt(D)), in float32 (R9)."""
    x = np.asarray(x, dtype=np.float32)
    return (fwht(x, np.float32) * inv_sqrt_f32(x.shape[-1])).astype(np.float32)


def hadamard_matrix(d: int) -> np.ndarray:
    """Dense Sylvester Hadamard matrix H_ij = (-1)^popcount(i & j), float64 (unnormalised)."""
    i = np.arange(d)
    pc = np.vectorize(lambda t: bin(int(t)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def quantize_hadamard_int4(x: np.ndarray):
    """Per-token symmetric int4 in a fixed Hadamard basis (tract discussion #2402, "What's done"
    and "Architecture: Data flow (decode)": rotate (FWHT) -> per-token symmetric int4 -> pack).

    y = rotate(x); s = amax(|y|) / 7 (float32, R7); q = clamp(rint(y / s), -7, 7); the codes
    are packed two per byte in the Q4_0 nibble order (ceil(D/2) bytes per token) and s is
    stored as float32 ("State = ... packed int4 K/V (ceil(D/2) bytes/token) + one f32
    scale/token + the f32 recent window").

    Returns (payload uint8 [..., ceil(D/2)], scale float32 [...], y float32 [..., D]).
    """
    y = rotate(x)
    amax = np.max(np.abs(y), axis=-1)
    s = (amax / np.float32(7.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(y / s[..., None])
    q = np.where(s[..., None] > 0, np.clip(r, -7, 7), 0.0).astype(np.int32)
    return pack_nibbles(q & 0xF), s, y


def hadamard_codes(payload: np.ndarray, head_dim: int) -> np.ndarray:
    """Signed int4 codes of a Hadamard-int4 row (same read formula as Q4_0)."""
    return read_q4_0(unpack_nibbles(payload, head_dim))


def dequantize_hadamard_int4(payload: np.ndarray, scale: np.ndarray, head_dim: int) -> np.ndarray:
    """Rotated-basis reconstruction y_hat = code * s (float64)."""
    return hadamard_codes(payload, head_dim).astype(np.float64) * np.asarray(scale, np.float64)[..., None]


# ------------------------------------------------------------------ asymmetric g=32
def quantize_asym4_g32(x: np.ndarray):
    """Per-group asymmetric int4, g = 32 consecutive values, per-group scale and zero-point
    (Open-TQ-Metal, background "Per-group asymmetric int4 quantization": two values per byte,
    3.2x at g=32 including scale and zero-point). Formula reading R10:
      s = fp16((max - min) / 15), z = fp16(min), q = clamp(rint((x - z) / s), 0, 15),
    computed as a float32 subtraction then a float32 division, each rounded.
    Reconstruction x_hat = q * s + z.

    Returns (payload uint8 [..., 16*nb], scale float16 [..., nb], zero float16 [..., nb]).
    """
    xb = _blocks(x)
    mn = np.min(xb, axis=-1)
    mx = np.max(xb, axis=-1)
    rng = (mx - mn).astype(np.float32)
    s16 = fp16_round(rng / np.float32(15.0))
    z16 = fp16_round(mn)
    s = s16.astype(np.float32)[..., None]
    z = z16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint((xb - z) / s)
    q = np.where(s > 0, np.clip(r, 0, 15), 0.0).astype(np.int32)
    payload = pack_nibbles(q)
    return payload.reshape(x.shape[:-1] + (-1,)), s16, z16


def dequantize_asym4_g32(payload: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    payload = np.asarray(payload, np.uint8)
    nb = scale.shape[-1]
    q = unpack_nibbles(payload.reshape(payload.shape[:-1] + (nb, 16)), BLOCK).astype(np.float64)
    x = q * np.asarray(scale).astype(np.float64)[..., None] + np.asarray(zero).astype(np.float64)[..., None]
    return x.reshape(payload.shape[:-1] + (nb * BLOCK,))


# ------------------------------------------------------------------ Q8_0
def quantize_q8_0(x: np.ndarray):
    """Q8_0 (R24): per 32 values d = amax / 128 stored as fp16 (R3), q = clamp(rint(x / d),
    -128, 127) (R1, R2), byte i of the block = q_i as a two's-complement byte.

    Returns (payload uint8 [..., 32 * nb], scale float16 [..., nb]).
    """
    xb = _blocks(x)
    amax = np.max(np.abs(xb), axis=-1)
    d16 = fp16_round(amax / np.float32(128.0))
    d = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(xb / d)
    q = np.where(d > 0, np.clip(r, -128, 127), 0.0).astype(np.int32)
    payload = (q & 0xFF).astype(np.uint8)
    return payload.reshape(x.shape[:-1] + (-1,)), d16


def read_q8_0(v: np.ndarray) -> np.ndarray:
    """Read-side sign extension of a Q8_0 byte: (v ^ 0x80) - 0x80 (R24)."""
    v = np.asarray(v).astype(np.int32)
    return (v ^ 0x80) - 0x80


def dequantize_q8_0(payload: np.ndarray, scale: np.ndarray) -> np.ndarray:
    nb = scale.shape[-1]
    p = np.asarray(payload, np.uint8).reshape(np.asarray(payload).shape[:-1] + (nb, BLOCK))
    x = read_q8_0(p).astype(np.float64) * np.asarray(scale).astype(np.float64)[..., None]
    return x.reshape(np.asarray(payload).shape[:-1] + (nb * BLOCK,))


# ------------------------------------------------------------------ Hadamard int2
def pack_pairs_of_bits(f: np.ndarray) -> np.ndarray:
    """Four 2-bit fields per byte: field 4j+i at bits 2i..2i+1 of byte j (R25)."""
    f = np.asarray(f, dtype=np.uint8) & 0x3
    D = f.shape[-1]
    pad = (-D) % 4
    if pad:
        f = np.concatenate([f, np.zeros(f.shape[:-1] + (pad,), np.uint8)], axis=-1)
    f = f.reshape(f.shape[:-1] + (-1, 4))
    return (f[..., 0] | (f[..., 1] << 2) | (f[..., 2] << 4) | (f[..., 3] << 6)).astype(np.uint8)


def unpack_pairs_of_bits(b: np.ndarray, count: int) -> np.ndarray:
    """Inverse of pack_pairs_of_bits: the raw 2-bit fields in value order."""
    b = np.asarray(b, dtype=np.uint8)
    f = np.stack([(b >> (2 * i)) & 0x3 for i in range(4)], axis=-1)
    return f.reshape(b.shape[:-1] + (4 * b.shape[-1],))[..., :count]


def quantize_hadamard_int2(x: np.ndarray):
    """Per-token symmetric int2 in the Hadamard basis (R25; tract discussion #2402, "Why this quant
    scheme" and "Causality & mixed precision": int2 is usable only with the exact-f32 window).

    y = rotate(x); s = amax(|y|) (float32); q = clamp(rint(y / s), -1, 1); four codes per byte.
    Returns (payload uint8 [..., ceil(D/4)], scale float32 [...], y float32 [..., D]).
    """
    y = rotate(x)
    s = np.max(np.abs(y), axis=-1).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(y / s[..., None])
    q = np.where(s[..., None] > 0, np.clip(r, -1, 1), 0.0).astype(np.int32)
    return pack_pairs_of_bits(q & 0x3), s, y


def read_int2(v: np.ndarray) -> np.ndarray:
    """Read-side sign extension of a 2-bit field: (v ^ 2) - 2 (R25)."""
    v = np.asarray(v).astype(np.int32)
    return (v ^ 0x2) - 0x2


def hadamard_int2_codes(payload: np.ndarray, head_dim: int) -> np.ndarray:
    return read_int2(unpack_pairs_of_bits(payload, head_dim))


def hadamard_layout_codes(layout: str, payload: np.ndarray, head_dim: int) -> np.ndarray:
    """Signed codes of a Hadamard-layout row (int4 or int2)."""
    return hadamard_codes(payload, head_dim) if layout == "had_int4" else hadamard_int2_codes(payload, head_dim)


# ------------------------------------------------------------------ generic entry points
def quantize(layout: str, x: np.ndarray) -> dict:
    """Quantize rows x[..., D]; returns a dict of the stored planes for `layout`."""
    if layout == "q4_0":
        p, s = quantize_q4_0(x)
        return {"payload": p, "scale": s}
    if layout == "q6_0":
        p, s = quantize_q6_0(x)
        return {"payload": p, "scale": s}
    if layout == "had_int4":
        p, s, y = quantize_hadamard_int4(x)
        return {"payload": p, "scale": s, "rot": y}
    if layout == "asym4_g32":
        p, s, z = quantize_asym4_g32(x)
        return {"payload": p, "scale": s, "zero": z}
    if layout == "q8_0":
        p, s = quantize_q8_0(x)
        return {"payload": p, "scale": s}
    if layout == "had_int2":
        p, s, y = quantize_hadamard_int2(x)
        return {"payload": p, "scale": s, "rot": y}
    raise ValueError(layout)


def dequantize(layout: str, planes: dict, head_dim: int) -> np.ndarray:
    """float64 reconstruction of stored rows (Hadamard: in the rotated basis)."""
    if layout == "q4_0":
        return dequantize_q4_0(planes["payload"], planes["scale"])
    if layout == "q6_0":
        return dequantize_q6_0(planes["payload"], planes["scale"])
    if layout == "had_int4":
        return dequantize_hadamard_int4(planes["payload"], planes["scale"], head_dim)
    if layout == "asym4_g32":
        return dequantize_asym4_g32(planes["payload"], planes["scale"], planes["zero"])
    if layout == "q8_0":
        return dequantize_q8_0(planes["payload"], planes["scale"])
    if layout == "had_int2":
        return hadamard_int2_codes(planes["payload"], head_dim).astype(np.float64) * \
            np.asarray(planes["scale"], np.float64)[..., None]
    raise ValueError(layout)
