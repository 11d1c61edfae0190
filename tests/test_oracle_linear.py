"""Pins for the oracle's dense NVFP4 linear layer (CPU only).

* a lossless closed form: activations and weights built directly on the
  NVFP4 grid (codes and scale bytes from the OCP MX v1.0 bit layouts, not
  from the oracle's encoder) must give exactly the plain float64 matmul of
  the values they were built from;
* the pages' evidence about the activation global scale: a stored
  input_scale of 0.00025141 (multiplier 3977.6) saturates the E4M3 block
  scales of activations with amax 2-8, while the measured amax does not.
"""

import numpy as np

import oracle
from oracle import nvfp4 as q

# E2M1 magnitude -> 3-bit code, and E4M3 byte of 2^n for normal n (bias 7):
# both read off the OCP MX v1.0 bit layouts, independent of the oracle.
MAG_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def pow2_e4m3_byte(n):
    assert -6 <= n <= 8
    return (n + 7) << 3


def grid_matrix(rng, rows, K):
    """Values on the NVFP4 grid with a +-6 in every block and a power-of-two
    block scale 2^n: returns (values / 2^0 before the global scale, codes,
    scale bytes)."""
    mags = np.array(list(MAG_CODE))
    v = rng.choice(mags, (rows, K // 16, 16)) * rng.choice([-1.0, 1.0], (rows, K // 16, 16))
    v[:, :, 0] = rng.choice([6.0, -6.0], (rows, K // 16))
    n = rng.integers(-3, 5, (rows, K // 16))
    nib = np.vectorize(lambda a: MAG_CODE[abs(a)] | (8 if a < 0 or (a == 0 and np.signbit(a)) else 0))(v)
    nib = nib.reshape(rows, K).astype(np.uint8)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    scales = np.vectorize(pow2_e4m3_byte)(n).astype(np.uint8)
    vals = (v * np.exp2(n)[..., None]).reshape(rows, K)
    return vals, codes, scales


def test_linear_lossless_equals_plain_matmul():
    rng = np.random.default_rng(11)
    T, K, N = 12, 256, 48
    # activations: grid values * 2^n / 1024 with amax pinned to 2.625 below,
    # so gs_x = 2688 / 2.625 = 1024 and every block re-quantises to itself
    xv, _, _ = grid_matrix(rng, T, K)
    x = (xv / 1024.0).astype(np.float32)
    gs_w = np.float32(512.0)
    wv, w_codes, w_scales = grid_matrix(rng, N, K)
    w = wv / 512.0
    out, inter = oracle.linear(x, w_codes, w_scales, gs_w, amax=2.625, round_bf16=False)
    assert inter["gs_x"] == np.float32(1024.0)
    assert np.array_equal(out, x.astype(np.float64) @ w.T)
    # rows and columns are not swapped: a one-hot activation picks a weight column
    e = np.zeros((1, K), np.float32)
    e[0, 5] = 6.0 / 1024.0
    out1, _ = oracle.linear(e, w_codes, w_scales, gs_w, amax=2.625, round_bf16=False)
    assert np.array_equal(out1[0], w[:, 5] * 6.0 / 1024.0)
    # the default output is that product rounded once to bf16
    out_bf16, _ = oracle.linear(x, w_codes, w_scales, gs_w, amax=2.625)
    assert np.array_equal(out_bf16, q.bf16_round(out)) and np.any(out_bf16 != out)


def test_linear_measured_amax_avoids_the_stored_scale_overflow():
    rng = np.random.default_rng(12)
    T, K, N = 16, 512, 64
    x = (rng.standard_normal((T, K)) * 0.9).astype(np.float32)
    x[3, 17] = 7.5  # activations of amax ~2-8
    _, w_codes, w_scales = grid_matrix(rng, N, K)
    gs_w = np.float32(512.0)
    exact = x.astype(np.float64) @ (q.dequantize(w_codes, w_scales, gs_w)).T
    measured, mi = oracle.linear(x, w_codes, w_scales, gs_w, round_bf16=False)
    stored_amax = 2688.0 * 0.00025141  # gs = 1 / input_scale = 3977.6
    stored, si = oracle.linear(x, w_codes, w_scales, gs_w, amax=stored_amax, round_bf16=False)
    assert abs(float(si["gs_x"]) - 3977.6) < 0.1
    # the stored scale saturates block scales (E4M3 max 448 = byte 0x7E) ...
    assert np.mean(si["x_scales"] == 0x7E) > 0.9
    # (with the measured amax only the block holding the tensor's amax reaches 448)
    amax_b = np.abs(x).reshape(T, K // 16, 16).max(axis=2)
    assert np.array_equal(mi["x_scales"] == 0x7E, amax_b == np.abs(x).max())
    err = lambda o: np.linalg.norm(o - exact) / np.linalg.norm(exact)
    # ... and wrecks the product, while the measured amax keeps NVFP4 accuracy
    assert err(measured) < 0.15
    assert err(stored) > 0.3 and err(stored) > 4 * err(measured)
