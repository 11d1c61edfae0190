"""The checkers of the GPU forward tests, on the CPU: each accepts the
oracle's own forward and rejects planted mistakes (a wrong requantised
code, swapped routing weights, another token's output)."""

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs
from helpers import check_forward, check_sampled_tokens


@pytest.fixture(scope="module")
def tiny_forward():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.make_activations(cfg).float().numpy()
    ids, w = inputs.make_routing(cfg)
    experts = inputs.ExpertSet(cfg)
    out, inter = oracle.forward(x, ids.numpy(), w.numpy(), experts, pad=32,
                                return_intermediates=True)
    return cfg, experts, ids.numpy(), w.numpy(), out, inter


def _check(fw, tokens, ids=None, w=None, hq=None, out=None):
    cfg, experts, ids0, w0, out0, inter = fw
    check_sampled_tokens(experts, ids0 if ids is None else ids, w0 if w is None else w,
                         inter["routing"].slot_dst, inter["h"],
                         inter["hq_codes"] if hq is None else hq, inter["hq_scales"],
                         inter["gs_h"], inter["amax_h"], out0 if out is None else out, tokens)


def test_accepts_the_oracle_forward(tiny_forward):
    _check(tiny_forward, np.arange(tiny_forward[0].T))


def test_rejects_a_wrong_requantised_code(tiny_forward):
    cfg, _, _, _, _, inter = tiny_forward
    hq = inter["hq_codes"].copy()
    r = int(inter["routing"].slot_dst[3 * cfg.k])
    hq[r, 5] ^= 0x01
    with pytest.raises(AssertionError, match="codes"):
        _check(tiny_forward, [3], hq=hq)


def test_rejects_swapped_routing_weights(tiny_forward):
    cfg, _, _, w, _, _ = tiny_forward
    w2 = w.copy()
    t = int(np.argmax(np.abs(w[:, 0] - w[:, 1])))
    w2[t, [0, 1]] = w2[t, [1, 0]]
    with pytest.raises(AssertionError):
        _check(tiny_forward, [t], w=w2)


def test_rejects_another_tokens_output(tiny_forward):
    out = tiny_forward[4].copy()
    out[[2, 7]] = out[[7, 2]]
    with pytest.raises(AssertionError):
        _check(tiny_forward, [2, 7], out=out)


class _Stages:
    """Stands in for a forward: its intermediates are the oracle's own, with
    NaN in the padding rows of h as a forward may leave them."""

    def __init__(self, inter):
        valid = inter["routing"].row_src >= 0
        h = torch.from_numpy(inter["h"].astype(np.float32)).to(torch.bfloat16)
        h[torch.from_numpy(~valid)] = float("nan")
        self.v = {"h": h, "hq_codes": torch.from_numpy(inter["hq_codes"].copy()),
                  "hq_sf": torch.from_numpy(inter["hq_scales"].copy()),
                  "slot_dst": torch.from_numpy(inter["routing"].slot_dst.astype(np.int32)),
                  "amax_h": torch.tensor([float(inter["amax_h"])], dtype=torch.float32),
                  "gs_h": torch.tensor([float(inter["gs_h"])], dtype=torch.float32)}

    def intermediates(self):
        return self.v


def _plant_requant_flip(inter, st):
    """Move one h value of a valid row by bf16 ulps until the row's
    requantisation (with the forward's amax) changes a code: a flip that an
    h difference explains, as an fp32 forward can produce.  Returns the
    token that owns the row."""
    from oracle import nvfp4 as q

    rt = inter["routing"]
    r = int(rt.slot_dst[0])
    h = st.v["h"]
    row = h[r].float().numpy().astype(np.float64)
    for c in range(row.size):
        for steps in range(1, 6):
            cand = row.copy()
            a = abs(cand[c]) if cand[c] != 0 else 2.0 ** -20
            cand[c] = cand[c] + steps * np.ldexp(1.0, int(np.floor(np.log2(a))) - 7)
            cand = q.bf16_round(cand)
            if np.abs(cand).max() > float(inter["amax_h"]):
                continue
            hc, hs, _, _ = q.quantize(cand[None].astype(np.float32), amax=inter["amax_h"])
            if not np.array_equal(hc[0], inter["hq_codes"][r]):
                h[r] = torch.from_numpy(cand.astype(np.float32)).to(torch.bfloat16)
                st.v["hq_codes"][r] = torch.from_numpy(hc[0])
                st.v["hq_sf"][r] = torch.from_numpy(hs[0])
                return int(rt.row_src[r]) // (rt.slot_dst.size // len(inter["out_f64"]))
    raise AssertionError("no flip found")


def test_forward_check_accepts_the_oracle_with_unwritten_padding(tiny_forward):
    cfg, ex, ids, w, out, inter = tiny_forward
    assert (inter["routing"].row_src < 0).any()
    out_t = torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16)
    check_forward(_Stages(inter), out_t, inter, ex, ids, w)


def test_forward_check_rejects_a_requant_flip_without_an_h_difference(tiny_forward):
    cfg, ex, ids, w, out, inter = tiny_forward
    st = _Stages(inter)
    r = int(inter["routing"].slot_dst[0])
    st.v["hq_codes"][r, 0] ^= 0x01
    out_t = torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16)
    with pytest.raises(AssertionError, match="without an h difference"):
        check_forward(st, out_t, inter, ex, ids, w)


def test_forward_check_rejects_a_wrong_output_token(tiny_forward):
    cfg, ex, ids, w, out, inter = tiny_forward
    bad = out.astype(np.float32).copy()
    bad[5] = -bad[5]
    with pytest.raises(AssertionError):
        check_forward(_Stages(inter), torch.from_numpy(bad).to(torch.bfloat16), inter, ex, ids, w)


def test_forward_check_rechecks_a_token_that_owns_a_requant_flip(tiny_forward):
    """A token whose requantised h differs (explained by an h difference) is
    not dropped: it is recomputed from the forward's own h, so its correct
    output passes and a wrong one fails."""
    from oracle import nvfp4 as q

    cfg, ex, ids, w, out, inter = tiny_forward
    st = _Stages(inter)
    t = _plant_requant_flip(inter, st)
    # the stand-in's output of token t follows its own requantised rows, as a
    # forward's does
    k = ids.shape[1]
    acc = np.zeros(out.shape[1])
    for j in range(k):
        r = int(inter["routing"].slot_dst[t * k + j])
        e = ex[int(ids[t, j])]
        hq = q.dequantize(st.v["hq_codes"][r:r + 1].numpy(), st.v["hq_sf"][r:r + 1].numpy(),
                          inter["gs_h"])
        acc += float(w[t, j]) * (hq @ q.dequantize(e["w2_codes"], e["w2_scales"], e["w2_gs"]).T)[0]
    out = out.copy()
    out[t] = q.bf16_round(acc)
    out_t = torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16)
    check_forward(st, out_t, inter, ex, ids, w)
    bad = out.astype(np.float32).copy()
    bad[t] = -bad[t]
    with pytest.raises(AssertionError, match="requant flip"):
        check_forward(st, torch.from_numpy(bad).to(torch.bfloat16), inter, ex, ids, w)


def test_forward_check_on_a_token_sample(tiny_forward):
    """The sample mode: the oracle runs on a subset of the tokens with the
    whole batch's global amax values; the forward's rows of those tokens are
    found through its own slot map.  A wrong output among the sampled tokens
    fails; one outside the sample is not looked at."""
    cfg, ex, ids, w, out, inter = tiny_forward
    x = inputs.make_activations(cfg).float().numpy()
    sample = np.array([1, 4, 9, 30, 63])
    _, sub = oracle.forward(x[sample], ids[sample], w[sample], ex, pad=32,
                            return_intermediates=True, amax_x=inter["amax_x"],
                            amax_h=inter["amax_h"])
    out_t = torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16)
    check_forward(_Stages(inter), out_t, sub, ex, ids, w, tokens=sample)
    bad = out.astype(np.float32).copy()
    bad[2] = -bad[2]  # not sampled
    check_forward(_Stages(inter), torch.from_numpy(bad).to(torch.bfloat16), sub, ex, ids, w,
                  tokens=sample)
    bad[9] = -bad[9]  # sampled
    with pytest.raises(AssertionError):
        check_forward(_Stages(inter), torch.from_numpy(bad).to(torch.bfloat16), sub, ex, ids, w,
                      tokens=sample)


def test_tolerance_checks_accept_rounding_and_reject_errors():
    from helpers import assert_close, assert_close_bf16, bf16_round

    rng = np.random.default_rng(2)
    want = rng.standard_normal(4096)
    # fp32 output: exact and fp32-rounded pass; 3e-3 relative noise, one
    # outlier of 2e-2 rms, a NaN or a swapped pair fail
    assert_close(want.astype(np.float32), want)
    for bad in (want * (1 + 3e-3 * rng.standard_normal(want.size)),
                np.where(np.arange(want.size) == 7, want + 0.02, want),
                np.where(np.arange(want.size) == 7, np.nan, want),
                want[np.r_[1, 0, 2:want.size]]):
        with pytest.raises(AssertionError):
            assert_close(bad, want)
    # bf16 output: the oracle's own rounding passes, and so does the other
    # neighbour of a value that sits next to a rounding midpoint; two ulps off
    # a large value do not
    got = bf16_round(want)
    assert_close_bf16(got, want)
    i = int(np.argmax(np.abs(want)))
    ulp = np.ldexp(1.0, int(np.floor(np.log2(abs(want[i])))) - 7)
    mid = want.copy()
    mid[i] = got[i] + np.sign(want[i] - got[i] or 1.0) * ulp * 0.499
    other = bf16_round(mid)
    other[i] = got[i] + np.sign(want[i] - got[i] or 1.0) * ulp
    assert_close_bf16(other, mid)
    far = got.copy()
    far[i] += 2 * ulp * np.sign(want[i])
    with pytest.raises(AssertionError):
        assert_close_bf16(far, want)
