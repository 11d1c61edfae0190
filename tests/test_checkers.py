"""The sampled-token checker of the full-size GPU tests, on the CPU: it
accepts the oracle's own forward and rejects planted mistakes (a wrong
requantised code, swapped routing weights, another token's output)."""

import numpy as np
import pytest

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs
from helpers import check_sampled_tokens


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
