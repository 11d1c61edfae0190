"""megamoe_forward end to end against the oracle's forward, on the MegaMoE
workloads (full size where the oracle finishes in seconds, sampled stages
and invariants otherwise), plus robustness cases: poisoned workspace,
stress routings, skipped and out-of-range ids."""

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4 as q
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import (assert_close, assert_close_bf16, bf16_to_np, check_forward,
                     check_sampled_tokens)

pytestmark = pytest.mark.gpu

_CACHE = {}


def _weights(cfg):
    """All experts generated on the GPU (torch RNG) and prepared once."""
    key = (cfg.E, cfg.d, cfg.I, cfg.seed)
    if key not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        raw = inputs.make_all_experts(cfg, device="cuda")
        _CACHE[key] = (raw, megamoe.Weights.prepare(raw))
    return _CACHE[key]


def _run(cfg, pad, x=None, ids=None, w=None, poison=False):
    raw, weights = _weights(cfg)
    x = inputs.make_activations(cfg) if x is None else x
    if ids is None:
        ids, w = inputs.make_routing(cfg)
    fwd = megamoe.Forward(weights, x.shape[0], ids.shape[1], pad=pad)
    if poison:
        fwd.ws.fill_(0xFF)
    out = fwd(x.cuda(), ids.cuda(), w.cuda())
    bits = fwd.read_status()
    return raw, fwd, x, ids, w, out, bits


@pytest.mark.parametrize("name,pad", [("tiny", 32), ("tiny", 128), ("decode", 32),
                                      ("decode1", 32), ("slice", 128), ("slice1", 128)])
def test_forward_matches_oracle(cuda_lib, name, pad):
    cfg = inputs.CONFIGS[name]
    raw, fwd, x, ids, w, out, bits = _run(cfg, pad)
    assert bits == 0
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                              inputs.ExpertSet(cfg, raw), pad=pad, return_intermediates=True)
    check_forward(cfg, fwd, out, inter, what=name)


def test_forward_prefill_shaped_mid_size(cuda_lib):
    """Zipf-skewed routing with hot and empty experts, outliers, several
    token tiles per expert; small enough for the full oracle."""
    cfg = inputs.MoEConfig("prefill_mid", 64, 6, 2048, 1024, 512, "zipf", seed=77,
                           outlier_frac=1e-3)
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                              inputs.ExpertSet(cfg, raw), pad=32, return_intermediates=True)
    check_forward(cfg, fwd, out, inter, what="prefill_mid")


@pytest.mark.parametrize("name", ["prefill", "large"])
def test_forward_full_size_prefill_stages(cuda_lib, name):
    """Full-size prefill: routing and activation quantisation bit-exact, the
    L1 output on sampled rows against the oracle, the L1 amax bounds the
    sample, the output is finite, and sampled output tokens match the
    oracle's L2 and combine over the forward's own h."""
    cfg = inputs.CONFIGS[name]
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    o = bf16_to_np(out)
    assert np.all(np.isfinite(o)) and np.any(o != 0)
    v = fwd.intermediates()
    rt = oracle.route(ids.numpy(), cfg.E, 32)
    R = int(rt.padded_offsets[-1])
    assert np.array_equal(v["padded_offsets"].cpu().numpy(), rt.padded_offsets)
    assert np.array_equal(v["row_src"].cpu().numpy()[:R], rt.row_src)
    xc, xs, xg, xa = q.quantize(x.float().numpy())
    assert np.float32(v["gs_x"].item()) == xg
    assert np.array_equal(v["xq_codes"].cpu().numpy()[:R][rt.row_src >= 0],
                          xc[rt.row_src[rt.row_src >= 0] // cfg.k])
    if name == "prefill":
        # requantisation of the GPU's own h (valid rows), bit-exact
        valid = rt.row_src >= 0
        h_all = v["h"][:R].float().cpu().numpy()[valid]
        amax_h0 = np.float32(v["amax_h"].item())
        assert amax_h0 == np.float32(np.abs(h_all).max())
        hc, hs, hg, _ = q.quantize(h_all, amax=amax_h0)
        assert np.float32(v["gs_h"].item()) == hg
        assert np.array_equal(v["hq_codes"].cpu().numpy()[:R][valid], hc)
        assert np.array_equal(v["hq_sf"].cpu().numpy()[:R][valid], hs)
    # sampled rows of h, one or two per expert, computed by the oracle alone
    rng = np.random.default_rng(5)
    experts = inputs.ExpertSet(cfg, raw)
    rows = []
    for e in rng.choice(np.nonzero(rt.counts)[0], size=min(12, int((rt.counts > 0).sum())),
                        replace=False):
        r0 = int(rt.padded_offsets[e])
        rows += [r0, r0 + int(rt.counts[e]) - 1]
    h_gpu = v["h"].float().cpu().numpy()
    amax_h = v["amax_h"].item()
    for r in rows:
        t = int(rt.row_src[r]) // cfg.k
        e = int(np.searchsorted(rt.padded_offsets, r, side="right") - 1)
        ew = experts[e]
        xh = q.dequantize(xc[t:t + 1], xs[t:t + 1], xg)
        gate = q.dequantize(ew["w13_codes"][:cfg.I], ew["w13_scales"][:cfg.I], ew["w13_gs"][0])
        up = q.dequantize(ew["w13_codes"][cfg.I:], ew["w13_scales"][cfg.I:], ew["w13_gs"][1])
        hw64 = (oracle.silu(xh @ gate.T) * (xh @ up.T))[0]
        assert_close_bf16(h_gpu[r], hw64, what=f"h row {r}")
        assert amax_h >= np.abs(q.bf16_round(hw64)).max()
    # sampled output tokens from the forward's own h: the slot mapping
    # bit-exact, then requantised rows, L2 and the combine token by token
    assert np.array_equal(v["slot_dst"].cpu().numpy(), rt.slot_dst)
    check_sampled_tokens(experts, ids.numpy(), w.numpy(), rt.slot_dst, h_gpu,
                         v["hq_codes"].cpu().numpy(), v["hq_sf"].cpu().numpy(),
                         v["gs_h"].item(), amax_h, o, rng.choice(cfg.T, size=4, replace=False),
                         what=name)


def test_forward_ignores_poisoned_workspace(cuda_lib):
    cfg = inputs.CONFIGS["tiny"]
    _, _, _, _, _, clean, b0 = _run(cfg, 32)
    clean = clean.clone()
    _, _, _, _, _, dirty, b1 = _run(cfg, 32, poison=True)
    assert b0 == 0 and b1 == 0
    assert torch.equal(clean, dirty)


@pytest.mark.parametrize("case", ["all_one_expert", "one_nonempty", "skipped_slots",
                                  "bad_ids", "no_tokens"])
def test_forward_stress_routings(cuda_lib, case):
    cfg = inputs.CONFIGS["tiny"]
    raw, weights = _weights(cfg)
    x = inputs.make_activations(cfg)
    ids, w = inputs.make_routing(cfg)
    ids = ids.clone()
    if case == "all_one_expert":
        ids[:] = 3
        ids[:, 1] = 3
    elif case == "one_nonempty":
        ids[:] = 7
    elif case == "skipped_slots":
        ids[::3, 1] = -1
        ids[5] = -1
    elif case == "bad_ids":
        ids[2, 0] = 8
        ids[9, 1] = 100
    elif case == "no_tokens":
        x, ids, w = x[:0], ids[:0], w[:0]
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32, x=x, ids=ids, w=w)
    if case == "bad_ids":
        assert bits & megamoe.DEV_BAD_EXPERT_ID
        ids_ok = torch.where(ids >= cfg.E, torch.full_like(ids, -1), ids)
    else:
        assert bits == 0
        ids_ok = ids
    _, inter = oracle.forward(x.float().numpy(), ids_ok.numpy(), w.numpy(),
                              inputs.ExpertSet(cfg, raw), pad=32, return_intermediates=True)
    check_forward(cfg, fwd, out, inter, what=case)


def test_forward_captures_in_a_cuda_graph(cuda_lib):
    """The forward records into a CUDA graph (every launch is stream-ordered,
    no host synchronisation) and replays give exactly the eager results, also
    for new inputs written into the captured buffers."""
    cfg = inputs.CONFIGS["tiny"]
    raw, weights = _weights(cfg)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    ids, w = ids.cuda(), w.cuda()
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    want = fwd(x, ids, w).clone()
    out = torch.empty_like(want)
    g = torch.cuda.CUDAGraph()
    fwd(x, ids, w, out=out)  # warm-up on the capture's buffers
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fwd(x, ids, w, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    # new inputs in the same buffers: the replay follows them
    x2 = inputs.make_activations(inputs.MoEConfig("tiny2", 8, 2, 256, 512, 64, "logits", seed=9))
    ids2, w2 = inputs.make_routing(inputs.MoEConfig("tiny2", 8, 2, 256, 512, 64, "logits", seed=9))
    want2 = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)(x2.cuda(), ids2.cuda(), w2.cuda()).clone()
    x.copy_(x2)
    ids.copy_(ids2)
    w.copy_(w2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want2)
    assert fwd.read_status() == 0


@pytest.mark.parametrize("E,k,T,d,I,pad", [(1024, 16, 40, 256, 256, 64),
                                            (384, 16, 12, 7168, 2048, 32)])
def test_forward_at_the_interface_maxima(cuda_lib, E, k, T, d, I, pad):
    """1024 experts (the most the interface takes) and top-16 (the most
    slots per token), against the oracle's forward."""
    cfg = inputs.MoEConfig("maxima", E, k, d, I, T, "uniform", seed=501, pad=pad)
    torch.cuda.empty_cache()
    _CACHE.clear()
    raw, fwd, x, ids, w, out, bits = _run(cfg, pad)
    assert bits == 0
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                              inputs.ExpertSet(cfg, raw), pad=pad, return_intermediates=True)
    check_forward(cfg, fwd, out, inter, what=f"E={E} k={k}")
