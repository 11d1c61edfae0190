"""megamoe_router_topk against the oracle's router (ids bit-exact, weights
to fp32 rounding), and the forward with a shared expert (run as expert E
that every token visits with weight 1) against the oracle, both through its
routed formulation and its dense one."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import check_forward

pytestmark = pytest.mark.gpu


def _check_router(logits, bias, k, shared=-1):
    ids, w = megamoe.router_topk(logits.cuda(), k, None if bias is None else bias.cuda(),
                                 shared_expert=shared)
    torch.cuda.synchronize()
    want_ids, want_w = oracle.router_topk(logits.numpy(), k,
                                          None if bias is None else bias.numpy(),
                                          shared_expert=None if shared < 0 else shared)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    assert np.allclose(w.cpu().numpy(), want_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name", ["tiny", "decode", "decode1", "prefill", "large"])
def test_router_matches_oracle_on_workloads(cuda_lib, name):
    cfg = inputs.CONFIGS[name]
    logits, bias = inputs.make_router_logits(cfg)
    _check_router(logits, bias, cfg.k)
    _check_router(logits, bias, cfg.k, shared=cfg.E)


@pytest.mark.parametrize("E,k,T", [(33, 3, 17), (1024, 16, 100), (64, 1, 5), (200, 8, 9)])
def test_router_shapes_and_ties(cuda_lib, E, k, T):
    g = torch.Generator().manual_seed(E * 7 + k)
    logits = torch.randn(T, E, generator=g)
    _check_router(logits, None, k)
    # heavy ties: a coarse grid of values, with and without a bias
    tied = torch.randint(-3, 4, (T, E), generator=g).float()
    _check_router(tied, None, k)
    _check_router(tied, torch.randint(-1, 2, (E,), generator=g).float() * 0.5, k)


def test_router_argument_errors(cuda_lib):
    lib = megamoe.load()
    logits = torch.zeros(4, 8, device="cuda")
    ids = torch.empty(4, 9, dtype=torch.int32, device="cuda")
    w = torch.empty(4, 9, device="cuda")
    p = megamoe._p
    assert lib.megamoe_router_topk(p(logits), 4, 8, 8, None, 9, -1, p(ids), p(w), None) == 1
    assert lib.megamoe_router_topk(p(logits), 4, 8, 8, None, 0, -1, p(ids), p(w), None) == 1
    assert lib.megamoe_router_topk(p(logits), 4, 8, 4, None, 2, -1, p(ids), p(w), None) == 1
    assert lib.megamoe_router_topk(p(logits), 0, 8, 8, None, 2, -1, p(ids), p(w), None) == 0


@pytest.mark.parametrize("name,pad", [("tiny", 32), ("decode", 32), ("slice", 128)])
def test_forward_with_shared_expert(cuda_lib, name, pad):
    """router (k routed + the shared column) -> megamoe_forward over E + 1
    experts; the oracle's forward on the oracle router's ids, and its dense
    shared-expert form, agree with it."""
    base = inputs.CONFIGS[name]
    cfg = inputs.with_shared_expert(base)
    torch.cuda.empty_cache()
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(base)
    logits, bias = inputs.make_router_logits(base)
    ids, w = megamoe.router_topk(logits.cuda(), base.k, None if bias is None else bias.cuda(),
                                 shared_expert=base.E)
    fwd = megamoe.Forward(weights, base.T, cfg.k, pad=pad)
    out = fwd(x.cuda(), ids, w)
    assert fwd.read_status() == 0
    ids_o, w_o = oracle.router_topk(logits.numpy(), base.k,
                                    None if bias is None else bias.numpy(), shared_expert=base.E)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    experts = inputs.ExpertSet(cfg, raw)
    # the oracle's forward takes the GPU router's fp32 weights (the router
    # itself is checked above), so the comparison isolates the forward
    w_gpu = w.cpu().numpy()
    _, inter = oracle.forward(x.float().numpy(), ids_o, w_gpu, experts, pad=pad,
                              return_intermediates=True)
    check_forward(cfg, fwd, out, inter, what=cfg.name)
    routed = inputs.ExpertSet(replace(base), raw)
    _, out64 = oracle.forward_with_shared(x.float().numpy(), ids_o[:, :base.k],
                                          w_gpu[:, :base.k], routed, experts[base.E], pad=pad)
    assert np.allclose(out64, inter["out_f64"], rtol=0, atol=1e-9 * np.abs(out64).max())
