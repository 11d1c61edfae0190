"""NVFP4 codec of the oracle (test infrastructure only; see ``oracle/__init__``).

NVFP4, as read here: a tensor X is stored as
  * one FP32 *global scale* ``gs`` (an encode multiplier),
  * one unsigned E4M3 *block scale* per 16 consecutive elements along K,
  * one 4-bit E2M1 code per element, two codes per byte (even element in the
    low nibble),
and an element decodes to ``e2m1(code) * e4m3(scale) / gs``.

The pages name the operation ("quantize_activation_nvfp4", Test Plan Phase 1
of "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4") and require the global
scale to come from the measured amax rather than a stored input_scale
("Current Bug: vLLM produces NaN from layer 0", "What we've tried" item 1 and
"Key evidence").  They do not spell out the arithmetic; the readings taken are:

  A1  gs = fl32(448 * 6 / amax): the largest block scale (448, E4M3 max) times
      the largest element (6, E2M1 max) maps to the tensor amax.
  A2  amax is taken over the whole tensor.
  A3  fixed float32 operation order, each op correctly rounded:
        s   = fl32(fl32(amax_b * gs) / 6)
        s8  = e4m3_rne_satfinite(s),  sd = decode(s8)
        enc = fl32(gs / sd)
        q_i = fl32(x_i * enc),  code_i = e2m1_rne_satfinite(q_i)
      and an all-zero block scale (sd == 0) gives all-zero (+0) codes.
  A4  the E2M1 sign bit is the sign bit of q_i (a negative value that rounds
      to zero is code 0x8).
  A5  even element in the low nibble.

Bit formats (OCP Microscaling Formats v1.0):
  E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
        {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no Inf/NaN.
  E4M3 ("E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no Inf;
        S.1111.111 is NaN; max finite 448; min normal 2^-6; min subnormal 2^-9.
"""

from __future__ import annotations

import numpy as np

#: E2M1 magnitude for each 3-bit magnitude code 0..7.
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

#: 448 (largest E4M3) * 6 (largest E2M1): the global scale maps amax onto it.
GLOBAL_SCALE_NUMERATOR = 448.0 * 6.0

E4M3_MAX = 448.0
BLOCK = 16


# --------------------------------------------------------------------------
# E2M1
# --------------------------------------------------------------------------
def e2m1_decode(codes) -> np.ndarray:
    """4-bit E2M1 code (0..15) -> float64 value.  Bit 3 is the sign."""
    c = np.asarray(codes).astype(np.int64)
    mag = E2M1_GRID[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """float32 value -> 4-bit E2M1 code, round-to-nearest-even, saturating.

    The grid midpoints are 0.25, 0.75, 1.25, 1.75, 2.5, 3.5 and 5.  A value on
    a midpoint goes to the neighbour with the even code (even mantissa bit):
    0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0,
    5 -> 4.0.  So the comparison is strict ('>') where the lower neighbour has
    the even code and inclusive ('>=') where the upper one has it.  Anything
    above 5 saturates to 6 (satfinite).  The sign bit is copied from the input
    (reading A4), so -0.1 encodes to 0x8.
    """
    x = np.asarray(v, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    mag = (
        (a > 0.25).astype(np.uint8)
        + (a >= 0.75)
        + (a > 1.25)
        + (a >= 1.75)
        + (a > 2.5)
        + (a >= 3.5)
        + (a > 5.0)
    ).astype(np.uint8)
    return (mag | (np.signbit(x).astype(np.uint8) << 3)).astype(np.uint8)


# --------------------------------------------------------------------------
# E4M3 (E4M3FN)
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """8-bit E4M3FN code -> float64 value (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(v) -> np.ndarray:
    """float value -> E4M3FN code, round-to-nearest-even, saturating to 448.

    Subnormals are multiples of 2^-9 (codes 0..7); rounding a subnormal
    upward to 8 * 2^-9 gives code 8, which is exactly 2^-6, the smallest
    normal.  For normals ``a = (1 + f) * 2^E`` the 3-bit fraction ``f * 8`` is
    rounded half-to-even, carrying into the exponent when it reaches 8.
    Magnitudes >= 448 give 448 (code 0x7E): the format has no Inf and its only
    pattern above 448 is NaN.  NaN input is outside the contract.
    """
    x = np.asarray(v, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros(a.shape, dtype=np.int64)

    sub = a < 2.0**-6
    out[sub] = np.rint(a[sub] * 2.0**9).astype(np.int64)  # 0..8, half-even

    nrm = (~sub) & (a < E4M3_MAX)
    m, e = np.frexp(a[nrm])  # a = m * 2^e, m in [0.5, 1)
    E = e.astype(np.int64) - 1
    f8 = np.rint((2.0 * m - 1.0) * 8.0).astype(np.int64)  # half-even
    carry = f8 == 8
    E = E + carry
    f8 = np.where(carry, 0, f8)
    out[nrm] = ((E + 7) << 3) | f8

    out[a >= E4M3_MAX] = 0x7E
    out = np.minimum(out, 0x7E)
    out = out | (np.signbit(x).astype(np.int64) << 7)
    return out.astype(np.uint8)


# --------------------------------------------------------------------------
# bf16
# --------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """float64 -> nearest bf16 value (returned as float64), ties to even.

    bf16 keeps 8 significant bits.  With x = m * 2^e, 0.5 <= |m| < 1, the
    result is rint(m * 2^8) * 2^(e - 8) (np.rint is half-to-even).  Values
    outside the normal bf16 range are outside the contract.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


# --------------------------------------------------------------------------
# packing and the tensor codec
# --------------------------------------------------------------------------
def pack_nibbles(codes) -> np.ndarray:
    """[..., K] 4-bit codes -> [..., K/2] bytes, element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] 4-bit codes (inverse of pack_nibbles)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def global_scale(amax) -> np.float32:
    """gs = fl32(2688 / amax); gs = 1 for an all-zero tensor (reading A1)."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(GLOBAL_SCALE_NUMERATOR) / amax


def quantize(x, amax=None):
    """Quantise a [rows, K] tensor to NVFP4 (readings A1-A5 above).

    ``x`` holds float32 values (bf16 inputs are exact in float32).  ``amax``
    defaults to max|x| over the whole tensor; a caller passes it to take the
    amax over a subset (the valid rows of the intermediate).  Returns
    ``(codes [rows, K/2] uint8, scales [rows, K/16] uint8 (E4M3 bytes),
    gs float32, amax float32)``.
    """
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % BLOCK:
        raise ValueError("quantize expects [rows, K] with K a multiple of 16")
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite input is outside the contract")
    rows, K = x.shape
    if amax is None:
        amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    amax = np.float32(amax)
    gs = global_scale(amax)
    if not np.isfinite(gs):
        raise ValueError("amax too small: the global scale overflows float32")

    blocks = x.reshape(rows, K // BLOCK, BLOCK)
    amax_b = np.max(np.abs(blocks), axis=2)  # exact
    s = (amax_b * gs) / np.float32(6.0)  # two float32 ops, each rounded
    s8 = e4m3_encode(s)
    sd = e4m3_decode(s8).astype(np.float32)  # exact
    nz = sd > 0
    enc = np.where(nz, gs / np.where(nz, sd, np.float32(1)), np.float32(0)).astype(np.float32)
    q = (blocks * enc[..., None]).astype(np.float32)
    codes = e2m1_encode(q)
    codes[~nz] = 0
    return pack_nibbles(codes.reshape(rows, K)), s8, gs, amax


def _byte_tables():
    """Value tables built from the scalar decoders: code byte -> E2M1 value of
    its low nibble (even element) and of its high nibble (odd element); scale
    byte -> E4M3 value."""
    b = np.arange(256)
    return e2m1_decode(b & 0xF), e2m1_decode(b >> 4), e4m3_decode(b)


_LO_TABLE, _HI_TABLE, _SCALE_TABLE = _byte_tables()


def dequantize(codes, scales, gs) -> np.ndarray:
    """NVFP4 -> float64: e2m1(code) * e4m3(scale) / gs, element by element.

    Each code byte holds elements 2i (low nibble) and 2i+1 (high nibble); each
    nibble is decoded by table lookup.
    """
    c = np.asarray(codes, dtype=np.uint8)
    rows, half = c.shape
    K = half * 2
    v = np.empty((rows, K))
    v[:, 0::2] = _LO_TABLE[c]
    v[:, 1::2] = _HI_TABLE[c]
    sd = _SCALE_TABLE[np.asarray(scales, dtype=np.uint8)][..., None]
    return (v.reshape(rows, K // BLOCK, BLOCK) * sd / np.float64(gs)).reshape(rows, K)


# --------------------------------------------------------------------------
# MMA scale-factor layout (used only to read back the GPU's swizzled scales)
# --------------------------------------------------------------------------
def swizzle_scales(scales, rows_pad=None) -> np.ndarray:
    """Row-major [rows, K/16] scales -> the 128-row x 4-block atom layout.

    Atoms of 512 bytes hold 128 rows x 4 consecutive 16-element blocks (one
    64-element slice of K).  Atom (a, c) covers rows a*128 .. a*128+127 and
    blocks 4c .. 4c+3; inside it, row r = a*128 + 32*j + i and block 4c + b
    sit at byte i*16 + j*4 + b.  Atoms are stored [row-group a][slice c].
    Rows are padded to a multiple of 128 (``rows_pad``) with zero bytes.
    """
    s = np.asarray(scales, dtype=np.uint8)
    rows, nb = s.shape
    if nb % 4:
        raise ValueError("K/16 must be a multiple of 4")
    if rows_pad is None:
        rows_pad = -(-rows // 128) * 128
    full = np.zeros((rows_pad, nb), dtype=np.uint8)
    full[:rows] = s
    # [a, j, i, c, b] -> [a, c, i, j, b]
    t = full.reshape(rows_pad // 128, 4, 32, nb // 4, 4)
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def unswizzle_scales(buf, rows, nb) -> np.ndarray:
    """Inverse of swizzle_scales: atom-layout bytes -> [rows, nb] row-major."""
    b = np.asarray(buf, dtype=np.uint8).reshape(-1)
    rows_pad = -(-rows // 128) * 128
    t = b[: rows_pad * nb].reshape(rows_pad // 128, nb // 4, 32, 4, 4)
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(rows_pad, nb)[:rows]
