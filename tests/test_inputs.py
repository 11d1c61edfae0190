"""The seeded input generators (CPU): any subset of experts regenerates
identically, draws are reproducible, and the derived workloads keep their
stated shapes.  The generators hold none of the method's arithmetic."""

import numpy as np
import torch

from nvfp4_block_scaled_topk_gb300 import inputs


def test_each_expert_regenerates_identically_alone_and_in_the_stack():
    cfg = inputs.CONFIGS["tiny"]
    stack = inputs.make_all_experts(cfg)
    for e in (0, 3, cfg.E - 1):
        one = inputs.make_expert(cfg, e)
        for k, v in one.items():
            assert torch.equal(stack[k][e].reshape(v.shape), v), (e, k)


def test_draws_are_reproducible_and_shaped():
    cfg = inputs.CONFIGS["tiny"]
    x1, x2 = inputs.make_activations(cfg), inputs.make_activations(cfg)
    assert torch.equal(x1, x2) and x1.shape == (cfg.T, cfg.d) and x1.dtype == torch.bfloat16
    assert float(x1.float().abs().max()) <= 1.3  # the tiny workload's clip
    ids, w = inputs.make_routing(cfg)
    assert ids.shape == (cfg.T, cfg.k) and w.shape == (cfg.T, cfg.k)
    assert torch.allclose(w.sum(1), torch.ones(cfg.T))
    assert all(len(set(r)) == cfg.k for r in ids.tolist())  # distinct experts per token
    lg1, b1 = inputs.make_router_logits(inputs.CONFIGS["prefill"].with_tokens(16))
    lg2, b2 = inputs.make_router_logits(inputs.CONFIGS["prefill"].with_tokens(16))
    assert torch.equal(lg1, lg2) and torch.equal(b1, b2) and lg1.shape == (16, 384)
    assert sorted(np.round(np.exp(-b1.numpy() / 1.1)).astype(int).tolist()) == list(range(1, 385))


def test_shared_expert_workload_and_linear_workloads():
    base = inputs.CONFIGS["decode"]
    s = inputs.with_shared_expert(base)
    assert (s.E, s.k, s.T, s.d, s.I) == (base.E + 1, base.k + 1, base.T, base.d, base.I)
    # the shared expert is expert E of the enlarged set, drawn like the others
    tiny = inputs.with_shared_expert(inputs.CONFIGS["tiny"])
    shared = inputs.make_expert(tiny, tiny.E - 1)
    again = inputs.make_expert(inputs.CONFIGS["tiny"], tiny.E - 1)
    assert all(torch.equal(shared[k], again[k]) for k in shared)
    for name, cfg in inputs.LINEAR_CONFIGS.items():
        assert cfg.K % 256 == 0 and cfg.N % 128 == 0, name
    x, c, sc, gs = inputs.make_linear(inputs.LINEAR_CONFIGS["linear_tiny"])
    lc = inputs.LINEAR_CONFIGS["linear_tiny"]
    assert x.shape == (lc.T, lc.K) and c.shape == (lc.N, lc.K // 2) and sc.shape == (lc.N, lc.K // 16)
    assert 2688 / 0.12 <= gs <= 2688 / 0.105 + 1e-3


def test_recipe_statistics():
    """Each statistic the recipe states, on the CPU draws."""
    from oracle import nvfp4 as q

    x = inputs.make_activations(inputs.CONFIGS["decode"]).float()
    assert abs(float(x.std()) - 0.09) < 0.002 and float(x.abs().max()) < 0.6
    p = inputs.CONFIGS["prefill"]
    xp = inputs.make_activations(p).float()
    assert abs(float((xp.abs() == 8).float().mean()) - 1e-3) < 1e-5
    ids, _ = inputs.make_routing(p)
    load = np.bincount(ids.numpy().reshape(-1), minlength=p.E)
    assert (load > 0).sum() == 126 and load.max() > 10 * load[load > 0].mean()
    big = inputs.CONFIGS["large"]
    ids, _ = inputs.make_routing(big)
    assert np.all(np.bincount(ids.numpy().reshape(-1), minlength=big.E) > 0)
    e = inputs.make_expert(inputs.CONFIGS["decode"], 5)
    mags = q.unpack_nibbles(e["w2_codes"].numpy()) & 7
    hist = np.bincount(mags.reshape(-1), minlength=8) / mags.size
    assert np.allclose(hist, np.array(inputs.MAG_COUNTS) / 128, atol=2e-3)
    w2 = q.dequantize(e["w2_codes"].numpy(), e["w2_scales"].numpy(), float(e["w2_gs"][0]))
    assert 0.020 < w2.std() < 0.023
