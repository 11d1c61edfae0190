"""The BFP16 model of tests/helpers.py (the storage of the forward's L2
output y: uint16 values u = q + 32768 with one power-of-two exponent per 16
rows x 8 columns, element = q * 2^s) pinned to hand values, and the error
budget it leaves against the float64 oracle's forward.  CPU only."""

import numpy as np

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs
from helpers import (BFP16_NONFINITE, MAX_ABS_OF_RMS, REL_L2, bf16_half_ulp, bfp16_decode,
                     bfp16_encode, bfp16_exponents)


def _group(vals):
    """One group: 16 rows x 8 columns, filled row by row."""
    g = np.zeros(128, np.float32)
    g[:len(vals)] = vals
    return g.reshape(16, 8)


def _q(u):
    return u.astype(np.int64) - 32768


def test_exponent_puts_the_group_max_just_below_2_to_15():
    # max 1.0: floor(log2) = 0, s = -14, q = v * 2^14
    u, s = bfp16_encode(_group([1.0, -0.5, 0.25, 3e-5]))
    assert s.shape == (1, 1) and s[0, 0] == -14
    assert list(_q(u[0, :4])) == [16384, -8192, 4096, round(3e-5 * 16384)]
    assert u[0, 0] == 16384 + 32768 and u[1, 0] == 32768  # a zero stores 32768
    # max 3.0 (floor(log2) = 1): s = -13, q = 3 * 2^13 = 24576
    u, s = bfp16_encode(_group([3.0, 1.0]))
    assert s[0, 0] == -13 and _q(u[0, 0]) == 24576 and _q(u[0, 1]) == 8192
    # a max whose scaled value would round to 2^15 takes the next exponent
    u, s = bfp16_encode(_group([np.nextafter(np.float32(2.0), np.float32(0)), -2.0 + 2 ** -23]))
    assert s[0, 0] == -13 and _q(u[0, 0]) == 16384 and _q(u[0, 1]) == -16384
    u, s = bfp16_encode(_group([1.99996]))  # fl32(1.99996) * 2^14 = 32767.34
    assert s[0, 0] == -14 and _q(u[0, 0]) == 32767
    u, s = bfp16_encode(_group([1.99997]))  # fl32(1.99997) * 2^14 = 32767.51
    assert s[0, 0] == -13 and _q(u[0, 0]) == 16384
    # ties go to even: v * 2^14 = 8192.5 -> 8192, 8193.5 -> 8194
    u, s = bfp16_encode(_group([1.0, 0.5 + 2.0 ** -15, 0.5 + 3 * 2.0 ** -15]))
    assert _q(u[0, 1]) == 8192 and _q(u[0, 2]) == 8194


def test_groups_are_16_rows_by_8_columns():
    v = np.zeros((32, 16), np.float32)
    v[3, 0], v[20, 7], v[5, 9] = 1.0, 4.0, 0.5
    assert bfp16_exponents(v).tolist() == [[-14, -15], [-12, 0]]
    # rows outside `valid` take no part in the exponent
    valid = np.ones(32, bool)
    valid[3] = False
    assert bfp16_exponents(v, valid).tolist() == [[0, -15], [-12, 0]]


def test_zero_group_huge_and_tiny_values():
    u, s = bfp16_encode(_group([]))
    assert s[0, 0] == 0 and np.all(u == 32768)
    # the largest float32: E = 127, s = 113, and its scaled value rounds to
    # 2^15, so s = 114 and q = 16384 (a value within 2^-16 of the maximum)
    big = np.finfo(np.float32).max
    u, s = bfp16_encode(_group([big, -big / 2]))
    assert s[0, 0] == 114 and _q(u[0, 0]) == 16384 and _q(u[0, 1]) == -8192
    # a large value below that keeps 15 bits
    u, s = bfp16_encode(_group([3e37]))
    assert abs(bfp16_decode(u, s)[0, 0] - 3e37) <= 3e37 * 2.0 ** -15
    # tiny groups clamp at -126 (q = v * 2^126)
    u, s = bfp16_encode(_group([1e-37, 3e-38]))
    assert s[0, 0] == -126 and _q(u[0, 0]) == round(1e-37 * 2.0 ** 126)


def test_non_finite_groups_pass_through_as_fp16():
    u, s = bfp16_encode(_group([1.0, np.nan, -np.inf]))
    assert s[0, 0] == BFP16_NONFINITE
    back = bfp16_decode(u, s)
    assert back[0, 0] == 1.0 and np.isnan(back[0, 1]) and back[0, 2] == -np.inf
    assert back[0, 3] == 0.0
    # other groups are unaffected
    v = np.zeros((16, 16), np.float32)
    v[0, 0] = np.nan
    v[9, 9] = 2.0
    u, s = bfp16_encode(v)
    assert list(s[0]) == [BFP16_NONFINITE, -13] and bfp16_decode(u, s)[9, 9] == 2.0


def test_round_trip_error_is_half_a_unit_of_the_group():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    u, s = bfp16_encode(v)
    back = bfp16_decode(u, s)
    unit = np.ldexp(1.0, np.repeat(np.repeat(s.astype(np.int64), 16, axis=0), 8, axis=1))
    assert np.all(np.abs(back - v.astype(np.float64)) <= unit / 2)  # half a unit of the group
    # each group's max keeps 15 significant bits
    m = np.abs(v).reshape(4, 16, 32, 8).max(axis=(1, 3))
    assert np.all(m.astype(np.float64) / unit[::16, ::8] >= 16383.75)


def test_bfp16_y_leaves_the_forward_well_inside_the_stated_tolerance():
    """The oracle's forward with its fp32-rounded y stored as BFP16 (valid
    rows choosing each group's exponent) and then combined exactly: against
    the float64 output, the error is under a quarter of the tolerance the
    GPU parity tests apply, on a batch whose experts hold many rows and on
    the one-token expert slice at the real width."""
    cfgs = [inputs.MoEConfig("bfp16_mid", 16, 4, 1024, 512, 256, "zipf", seed=8),
            inputs.CONFIGS["slice1"]]
    for cfg in cfgs:
        x = inputs.make_activations(cfg).float().numpy()
        ids, w = inputs.make_routing(cfg)
        ex = inputs.ExpertSet(cfg, inputs.make_all_experts(cfg))
        out, inter = oracle.forward(x, ids.numpy(), w.numpy(), ex, pad=cfg.pad,
                                    return_intermediates=True)
        rt = inter["routing"]
        y32 = np.asarray(inter["y"], dtype=np.float32)
        yb = bfp16_decode(*bfp16_encode(y32, rt.row_src >= 0))
        got = oracle.bf16_round(oracle.combine(yb, w.numpy(), rt.slot_dst, round_bf16=False))
        want = inter["out_f64"]
        ref = oracle.bf16_round(want)
        err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        excess = np.maximum(np.abs(got - want) - bf16_half_ulp(want), 0).max()
        rms = np.sqrt(np.mean(want ** 2))
        assert err <= REL_L2 / 4, (cfg.name, err)
        assert excess <= MAX_ABS_OF_RMS * rms / 4, (cfg.name, excess / rms)
