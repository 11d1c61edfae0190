"""Pins for the oracle's NVFP4 codec (CPU only).

Each test checks the oracle against something other than itself: hand
tables derived from the OCP MX v1.0 bit layouts (tests/golden/), an
exhaustive brute-force nearest-value search, torch's own float8/bfloat16
casts, and closed-form lossless cases.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4 as q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                a, b = line.split()
                rows.append((a, b))
    return rows


def test_e2m1_decode_matches_hand_table():
    for code, val in _read_table("e2m1_table.txt"):
        got = q.e2m1_decode(int(code, 16))
        assert float(got) == float(val)
        assert np.signbit(got) == val.startswith("-")


def test_e2m1_encode_matches_hand_rounding_table():
    for val, code in _read_table("e2m1_rounding.txt"):
        got = int(q.e2m1_encode(np.float32(float(val))))
        assert got == int(code, 16), (val, hex(got), code)


def test_e2m1_encode_exhaustive_against_brute_force_nearest():
    # every float32 in [-8, 8] on a 2^-12 grid, plus the grid midpoints
    # nudged by one float32 ulp either way
    v = np.arange(-8 * 4096, 8 * 4096 + 1, dtype=np.float64) / 4096.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    extra = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                            np.nextafter(mids.astype(np.float32), np.float32(10))])
    v = np.concatenate([v, extra, -extra]).astype(np.float32)
    got = q.e2m1_encode(v)
    # brute force: distance to each of the 8 magnitudes, smallest wins,
    # ties to the even code index
    a = np.abs(v.astype(np.float64))[:, None]
    dist = np.abs(a - np.array([0, .5, 1, 1.5, 2, 3, 4, 6])[None, :])
    best = np.full(v.shape, -1)
    bestd = np.full(v.shape, np.inf)
    for c in range(8):
        better = (dist[:, c] < bestd) | ((dist[:, c] == bestd) & (c % 2 == 0))
        best = np.where(better, c, best)
        bestd = np.where(better, dist[:, c], bestd)
    want = best | (np.signbit(v).astype(np.int64) << 3)
    assert np.array_equal(got.astype(np.int64), want)


def test_e4m3_matches_hand_points():
    for val, code in _read_table("e4m3_points.txt"):
        got = int(q.e4m3_encode(np.float64(float(val))))
        assert got == int(code, 16), (val, hex(got), code)


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = q.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], theirs[~nan])


def test_e4m3_encode_is_identity_on_decoded_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(q.e4m3_encode(q.e4m3_decode(codes)), codes)


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    # random values across the whole finite range plus every midpoint
    v = np.exp(rng.uniform(np.log(2.0**-12), np.log(447.0), 200_000)).astype(np.float32)
    finite = q.e4m3_decode(np.arange(0, 0x7F))
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, finite.astype(np.float32)])
    ours = q.e4m3_encode(v)
    theirs = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(100_000) * np.exp(rng.uniform(-20, 20, 100_000))).astype(np.float32)
    ours = q.bf16_round(v.astype(np.float64))
    theirs = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs)


def test_bf16_round_is_a_single_rounding_from_float64():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7; a hair above it must
    # round up.  Rounding through float32 first would land on the midpoint
    # and go to 1.0 (even): the oracle rounds float64 -> bf16 directly.
    x = 1.0 + 2.0**-8 + 2.0**-30
    assert q.bf16_round(x) == 1.0 + 2.0**-7
    assert q.bf16_round(1.0 + 2.0**-8) == 1.0
    assert q.bf16_round(-(1.0 + 3 * 2.0**-8)) == -(1.0 + 2.0**-6)


def test_pack_nibbles_low_nibble_is_even_element():
    codes = np.array([[0x1, 0xF, 0x7, 0x8]], dtype=np.uint8)
    packed = q.pack_nibbles(codes)
    assert packed.tolist() == [[0xF1, 0x87]]
    assert np.array_equal(q.unpack_nibbles(packed), codes)


def test_quantize_worked_example():
    # gs = 2688 / 2688 = 1.  Block 0 = [3, -1.2, 0.1, 0, ...]:
    #   amax_b = 3 -> s = 3 / 6 = 0.5 -> E4M3 0x30; enc = 1 / 0.5 = 2;
    #   3 -> 6 -> 0x7, -1.2 -> -2.4 -> -2 -> 0xC, 0.1 -> 0.2 -> +0 -> 0x0.
    # Block 1 holds the tensor amax 2688: s = 448 -> 0x7E; 2688/448 = 6 -> 0x7.
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :3] = [3.0, -1.2, 0.1]
    x[0, 16] = 2688.0
    codes, scales, gs, amax = q.quantize(x)
    assert gs == np.float32(1.0) and amax == np.float32(2688.0)
    assert scales.tolist() == [[0x30, 0x7E]]
    c = q.unpack_nibbles(codes)[0]
    assert c[:4].tolist() == [0x7, 0xC, 0x0, 0x0]
    assert c[16] == 0x7 and np.all(c[17:] == 0)


def test_quantize_all_zero_tensor_and_tiny_block():
    codes, scales, gs, amax = q.quantize(np.zeros((2, 32), np.float32))
    assert gs == 1.0 and amax == 0.0 and not codes.any() and not scales.any()
    # a block whose scale underflows E4M3 to zero: all codes +0 (even negative)
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1000.0
    x[0, 16:20] = [-1e-5, 1e-5, -2e-5, 0]
    codes, scales, gs, _ = q.quantize(x)
    assert scales[0, 1] == 0
    assert not q.unpack_nibbles(codes)[0, 16:].any()


def test_quantize_lossless_special_case():
    # gs = 2688 / 2.625 = 1024 exactly.  Blocks built as grid value * sd / gs
    # with sd a power of two and a +-6 in every block quantise to themselves:
    # amax_b * gs / 6 = sd exactly, enc = gs / sd exact, x * enc = grid value.
    rng = np.random.default_rng(3)
    rows, K = 8, 64
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -.5, -1, -1.5, -2, -3, -4, -6])
    vals = rng.choice(grid, (rows, K // 16, 16))
    vals[:, :, 0] = rng.choice([6.0, -6.0], (rows, K // 16))
    sd = 2.0 ** rng.integers(-4, 8, (rows, K // 16, 1))
    x = (vals * sd / 1024.0).reshape(rows, K).astype(np.float32)
    codes, scales, gs, _ = q.quantize(x, amax=2.625)
    assert gs == np.float32(1024.0)
    assert np.array_equal(q.dequantize(codes, scales, gs), x.astype(np.float64))


def test_quantize_error_within_the_grid_bound():
    # From the definitions alone: the block scale sd is the E4M3 round-to-
    # nearest of s = amax_b * gs / 6, so each block's largest encoded
    # magnitude amax_b * gs / sd = 6 s / sd lies in [6/(1+2^-4), 6/(1-2^-4)]
    # (3 mantissa bits; every s here is an E4M3 normal), and it is exactly 6
    # (scale 448 = 0x7E) in the block holding the tensor amax.  Every element
    # then decodes within half an E2M1 step of its encoded value x * gs / sd
    # (steps 0.5 below 2, 1 below 4, 2 up to 6), or to 6 when it lies above.
    rng = np.random.default_rng(11)
    rows, K = 64, 256
    mag = np.exp2(rng.integers(-5, 6, (rows, 1)).astype(np.float64))
    x = (rng.standard_normal((rows, K)) * mag).astype(np.float32)
    x[7, 32:48] = 0.0  # an all-zero block
    codes, s8, gs, amax = q.quantize(x)
    assert amax == np.float32(np.abs(x).max())
    sd = q.e4m3_decode(s8).astype(np.float64)
    blocks = x.astype(np.float64).reshape(rows, K // 16, 16)
    amax_b = np.abs(blocks).max(axis=2)
    zero = amax_b == 0
    assert np.array_equal(zero, sd == 0)
    s = amax_b * np.float64(gs) / 6.0
    assert np.all(s[~zero] >= 2.0 ** -6)
    qmax = np.where(zero, 0.0, 6.0 * s / np.where(zero, 1.0, sd))
    assert np.all(qmax[~zero] >= 6.0 / (1 + 2.0 ** -4) * (1 - 1e-6))
    assert np.all(qmax[~zero] <= 6.0 / (1 - 2.0 ** -4) * (1 + 1e-6))
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert s8[r, c // 16] == 0x7E and abs(qmax[r, c // 16] - 6.0) < 1e-6  # gs rounded to fp32
    enc = np.where(zero, 0.0, np.float64(gs) / np.where(zero, 1.0, sd))[..., None]
    qv = np.abs(blocks) * enc
    allowed = np.where(qv > 6, qv - 6, np.where(qv < 2, 0.25, np.where(qv < 4, 0.5, 1.0)))
    xh = q.dequantize(codes, s8, gs).reshape(rows, K // 16, 16)
    err = np.abs(xh - blocks) * enc
    assert np.all(err <= allowed * (1 + 1e-6) + 1e-9)
    assert not xh[7, 2].any()


def test_swizzle_layout_position_and_roundtrip():
    rows, nb = 200, 8  # K = 128
    s = (np.arange(rows * nb) % 251).astype(np.uint8).reshape(rows, nb)
    buf = q.swizzle_scales(s)
    assert buf.size == 256 * nb
    # row 33 = 32*1 + 1, block 5 = 4*1 + 1: atom (0, 1), byte 1*16 + 1*4 + 1
    assert buf[1 * 512 + 16 + 4 + 1] == s[33, 5]
    # row 130 = 128 + 2 (atom row-group 1), block 2: atom (1, 0), byte 2*16 + 2
    assert buf[(1 * (nb // 4) + 0) * 512 + 2 * 16 + 0 * 4 + 2] == s[130, 2]
    assert np.array_equal(q.unswizzle_scales(buf, rows, nb), s)
