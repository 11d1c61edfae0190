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
    check_forward(fwd, out, inter, experts, ids_o, w_gpu, what=cfg.name)
    routed = inputs.ExpertSet(replace(base), raw)
    _, out64 = oracle.forward_with_shared(x.float().numpy(), ids_o[:, :base.k],
                                          w_gpu[:, :base.k], routed, experts[base.E], pad=pad)
    assert np.allclose(out64, inter["out_f64"], rtol=0, atol=1e-9 * np.abs(out64).max())


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("decode1", None),
                                    ("prefill_mid", None)])
def test_forward_from_logits_equals_router_then_forward(cuda_lib, name, T):
    """megamoe_forward_from_logits (router fused into the first block for
    small batches, its own kernel for large ones) gives exactly the output
    of megamoe_router_topk followed by megamoe_forward, and its ids are the
    oracle router's."""
    if name == "prefill_mid":  # 512 tokens x 1024: the router runs as its own kernel
        base = inputs.MoEConfig("prefill_mid", 64, 6, 1024, 512, 512, "zipf", seed=78)
    else:
        base = inputs.CONFIGS[name]
    cfg = inputs.with_shared_expert(base)
    torch.cuda.empty_cache()
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(base).cuda()
    logits, bias = inputs.make_router_logits(base, device="cuda")
    fwd_a = megamoe.Forward(weights, base.T, cfg.k, pad=32)
    ids, w = megamoe.router_topk(logits, base.k, bias, shared_expert=base.E)
    out_a = fwd_a(x, ids, w).clone()
    fwd_b = megamoe.Forward(weights, base.T, cfg.k, pad=32)
    out_b = fwd_b.from_logits(x, logits, base.k, bias, shared_expert=base.E).clone()
    torch.cuda.synchronize()
    assert fwd_a.read_status() == 0 and fwd_b.read_status() == 0
    assert torch.equal(out_a, out_b)
    want_ids, _ = oracle.router_topk(logits.cpu().numpy(), base.k,
                                     None if bias is None else bias.cpu().numpy(),
                                     shared_expert=base.E)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    # without a shared expert too
    fwd_c = megamoe.Forward(weights, base.T, base.k, pad=32)
    ids2, w2 = megamoe.router_topk(logits, base.k, bias)
    out_c = fwd_c(x, ids2, w2).clone()
    out_d = megamoe.Forward(weights, base.T, base.k, pad=32).from_logits(x, logits, base.k, bias)
    assert torch.equal(out_c, out_d)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_forward_from_logits_matches_oracle(cuda_lib, name):
    """The layer from router logits (router fused ahead of the routing, one
    shared expert) against the oracle alone: the oracle's router picks the
    ids and weights, the oracle's forward runs on them, and the whole output
    and every stage of the fused call meet the forward checks."""
    base = inputs.CONFIGS[name]
    cfg = inputs.with_shared_expert(base)
    torch.cuda.empty_cache()
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(base)
    logits, bias = inputs.make_router_logits(base)
    fwd = megamoe.Forward(weights, base.T, cfg.k, pad=32)
    out = fwd.from_logits(x.cuda(), logits.cuda(), base.k,
                          None if bias is None else bias.cuda(), shared_expert=base.E)
    assert fwd.read_status() == 0
    ids_o, w_o = oracle.router_topk(logits.numpy(), base.k,
                                    None if bias is None else bias.numpy(), shared_expert=base.E)
    experts = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids_o, w_o, experts, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, experts, ids_o, w_o, what=f"{name} from logits")
