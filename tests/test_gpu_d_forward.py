"""megamoe_forward end to end against the oracle's forward, on the MegaMoE
workloads: every workload at full size, against the oracle's whole forward
(the 16384-token batch on a 256-token seeded sample with the batch's global
scales), every stage bit-exact where it is integer or byte work; plus
robustness cases: poisoned workspace, stress routings, skipped and
out-of-range ids, CUDA-graph capture, the interface maxima."""

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4 as q
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import check_forward

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
    _stage_checks(cfg, fwd, x, ids, pad)
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=pad,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what=name)


@pytest.mark.parametrize("T", [36, 37])
def test_forward_around_the_prologue_limit(cuda_lib, T):
    """The two sides of the one-block prologue's limit at d = 7168: 36 tokens
    (the largest batch whose routing and amax(x) one thread block takes) and
    37 (the routing and amax kernels).  Every stage bit-exact, then the
    whole forward against the oracle."""
    cfg = inputs.MoEConfig("decode_mid", 16, 6, 7168, 512, T, "uniform", seed=900 + T)
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    _stage_checks(cfg, fwd, x, ids)
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what=f"decode_mid T={T}")


@pytest.mark.parametrize("T,routing", [(80, "uniform"), (160, "uniform"), (2000, "zipf")])
def test_forward_at_shapes_off_the_powers_of_two(cuda_lib, T, routing):
    """d = 1280 and I = 768, multiples of 256 that are not powers of two: the
    gate+up GEMM has 5 K steps and 6 feature tiles of 256 (12 of 128), the
    down GEMM 3 K steps (fewer than any stage count, so every tile's loads
    run on into the next tile's) and 10 feature tiles.  12 experts, top-3:
    T = 80, 160 and 2000 give 32- and 64-token tiles and, at 2000 with a
    Zipf-skewed load, 128-token tiles (token-major for L1).  Every stage
    bit-exact, then the whole forward against the oracle."""
    cfg = inputs.MoEConfig("off_pow2", 12, 3, 1280, 768, T, routing, seed=1300 + T)
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    _stage_checks(cfg, fwd, x, ids)
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what=f"off_pow2 T={T}")


def test_forward_prefill_shaped_mid_size(cuda_lib):
    """Zipf-skewed routing with hot and empty experts, outliers, several
    token tiles per expert; small enough for the full oracle."""
    cfg = inputs.MoEConfig("prefill_mid", 64, 6, 2048, 1024, 512, "zipf", seed=77,
                           outlier_frac=1e-3)
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what="prefill_mid")


def _stage_checks(cfg, fwd, x, ids, pad=32):
    """Routing and the quantised x bit-exact, amax(h) = max |h| over the
    forward's own valid rows, and the requantisation of the forward's own h
    bit-exact (all rows)."""
    v = fwd.intermediates()
    rt = oracle.route(ids.numpy(), cfg.E, pad)
    R = int(rt.padded_offsets[-1])
    assert np.array_equal(v["padded_offsets"].cpu().numpy(), rt.padded_offsets)
    assert np.array_equal(v["row_src"].cpu().numpy()[:R], rt.row_src)
    assert np.array_equal(v["slot_dst"].cpu().numpy(), rt.slot_dst)
    xc, xs, xg, xa = q.quantize(x.float().numpy())
    assert np.float32(v["amax_x"].item()) == xa and np.float32(v["gs_x"].item()) == xg
    valid = rt.row_src >= 0
    assert np.array_equal(v["xq_codes"].cpu().numpy()[:R][valid],
                          xc[rt.row_src[valid] // cfg.k])
    assert np.array_equal(v["xq_sf"].cpu().numpy()[:R][valid], xs[rt.row_src[valid] // cfg.k])
    h_all = v["h"][:R][torch.from_numpy(valid).cuda()].float().cpu().numpy()
    amax_h = np.float32(v["amax_h"].item())
    assert amax_h == np.float32(np.abs(h_all).max())
    hc, hs, hg, _ = q.quantize(h_all, amax=amax_h)
    assert np.float32(v["gs_h"].item()) == hg
    assert np.array_equal(v["hq_codes"].cpu().numpy()[:R][valid], hc)
    assert np.array_equal(v["hq_sf"].cpu().numpy()[:R][valid], hs)
    return xa, amax_h


def test_forward_full_size_prefill_against_the_full_oracle(cuda_lib):
    """4096-token prefill (Zipf-skewed load, outliers, ~130 active experts,
    several token tiles per hot expert) at full size: every stage checked,
    then the whole output against the oracle's forward over all 4096 tokens
    (float64 on ~130 experts; a minute or two on the host)."""
    cfg = inputs.CONFIGS["prefill"]
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    _stage_checks(cfg, fwd, x, ids)
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what="prefill")


def test_forward_full_size_large_on_a_token_sample(cuda_lib):
    """16384 tokens, uniform routing over all 384 experts, at full size: every
    stage checked on all rows, then 256 seeded tokens against the oracle's
    forward over those tokens with the batch's amax of x (the oracle's own,
    over all tokens) and the forward's amax of h (which the stage checks tie
    to the forward's h and the oracle's requantiser)."""
    cfg = inputs.CONFIGS["large"]
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32)
    assert bits == 0
    amax_x, amax_h = _stage_checks(cfg, fwd, x, ids)
    sample = np.sort(np.random.default_rng(5).choice(cfg.T, size=256, replace=False))
    ex = inputs.ExpertSet(cfg, raw)
    xs = x.float().numpy()[sample]
    _, inter = oracle.forward(xs, ids.numpy()[sample], w.numpy()[sample], ex, pad=32,
                              return_intermediates=True, amax_x=amax_x, amax_h=amax_h)
    # the batch's amax(h) bounds the sample's (to a bf16 ulp: an h value at the
    # maximum may round one ulp apart)
    assert amax_h >= np.float32(inter["amax_h_own"]) * (1 - 2.0 ** -8)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), tokens=sample, what="large")


def test_forward_ignores_poisoned_workspace(cuda_lib):
    cfg = inputs.CONFIGS["tiny"]
    _, _, _, _, _, clean, b0 = _run(cfg, 32)
    clean = clean.clone()
    _, _, _, _, _, dirty, b1 = _run(cfg, 32, poison=True)
    assert b0 == 0 and b1 == 0
    assert torch.equal(clean, dirty)


@pytest.mark.parametrize("case", ["all_one_expert", "one_nonempty", "skipped_slots",
                                  "bad_ids", "no_tokens", "all_skipped", "zero_x"])
def test_forward_stress_routings(cuda_lib, case):
    """Degenerate routings and inputs against the oracle.  all_skipped: every
    id is -1, so no expert has a row and every output is exactly 0.  zero_x:
    amax(x) = 0 gives gs = 1 and all-zero blocks (scale 0, codes 0), then
    h = 0, amax(h) = 0 and again gs = 1: the output is exactly 0."""
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
    elif case == "all_skipped":
        ids[:] = -1
    elif case == "zero_x":
        x = torch.zeros_like(x)
    raw, fwd, x, ids, w, out, bits = _run(cfg, 32, x=x, ids=ids, w=w)
    if case == "bad_ids":
        assert bits & megamoe.DEV_BAD_EXPERT_ID
        ids_ok = torch.where(ids >= cfg.E, torch.full_like(ids, -1), ids)
    else:
        assert bits == 0
        ids_ok = ids
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids_ok.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids_ok.numpy(), w.numpy(), what=case)
    if case in ("all_skipped", "zero_x"):
        assert not out.any()
        v = fwd.intermediates()
        if case == "zero_x":
            assert v["amax_x"].item() == 0 and v["gs_x"].item() == 1
            assert v["amax_h"].item() == 0 and v["gs_h"].item() == 1
        else:
            assert v["padded_offsets"][-1].item() == 0


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
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=pad,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what=f"E={E} k={k}")


@pytest.mark.parametrize("E,k,d,I,T", [(384, 6, 7168, 2048, 8), (64, 6, 2048, 1024, 1024)])
def test_fused_requant_equals_the_separate_kernel(cuda_lib, E, k, d, I, T):
    """The requantisation of h inside the L1 kernel (megamoe_set_fused_requant)
    against the default separate kernel: the same requantised codes, block
    scales, global scale and output, bit for bit, with the 32-token tiles of
    decode and the token-major tiles of larger batches."""
    cfg = inputs.MoEConfig("fused_rq", E, k, d, I, T, "uniform", seed=612)
    torch.cuda.empty_cache()
    _CACHE.clear()
    raw, weights = _weights(cfg)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    ids, w = ids.cuda(), w.cuda()
    res = []
    for fused in (False, True):
        fwd = megamoe.Forward(weights, T, k, pad=32)
        try:
            megamoe.set_fused_requant(fused)
            out = fwd(x, ids, w).clone()
        finally:
            megamoe.set_fused_requant(False)
        assert fwd.read_status() == 0
        v = fwd.intermediates()
        R = int(v["padded_offsets"][-1].item())
        valid = v["row_src"][:R] >= 0
        res.append((out, v["hq_codes"][:R][valid].clone(), v["hq_sf"][:R][valid].clone(),
                    v["gs_h"].item()))
    (o0, c0, s0, g0), (o1, c1, s1, g1) = res
    assert g0 == g1
    assert torch.equal(c0, c1) and torch.equal(s0, s1)
    assert torch.equal(o0, o1)


def test_forward_with_edge_blocks_in_the_weights(cuda_lib):
    """The workloads' weight bytes come from fixed histograms with no zero or
    subnormal block scales; here every expert matrix also holds blocks whose
    E4M3 scale is 0x00 (the block decodes to zero) or subnormal (0x01..0x07),
    and blocks of +-6 codes, through the whole forward against the oracle."""
    cfg = inputs.MoEConfig("edges", 16, 4, 1024, 512, 96, "uniform", seed=808)
    raw = inputs.make_all_experts(cfg, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(9)
    for cname, sname in (("w13_codes", "w13_scales"), ("w2_codes", "w2_scales")):
        sc, co = raw[sname], raw[cname]
        n = sc.numel()
        pick = torch.randperm(n, generator=g, device="cuda")[: 3 * (n // 40)]
        sc.view(-1)[pick[: n // 40]] = 0
        sc.view(-1)[pick[n // 40: 2 * (n // 40)]] = torch.randint(
            1, 8, (n // 40,), generator=g, device="cuda", dtype=torch.uint8)
        six = pick[2 * (n // 40):]
        rows, blk = six // sc.shape[-1], six % sc.shape[-1]
        flat = co.view(-1, co.shape[-1])
        for b in range(8):  # the block's 8 code bytes: +-6 pairs
            flat.view(-1, co.shape[-1])[rows, 8 * blk + b] = torch.tensor(
                [0x77, 0xFF, 0x7F, 0xF7][b % 4], dtype=torch.uint8, device="cuda")
    assert (raw["w13_scales"] == 0).any() and ((raw["w2_scales"] > 0) & (raw["w2_scales"] < 8)).any()
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg)
    ids, w = inputs.make_routing(cfg)
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    out = fwd(x.cuda(), ids.cuda(), w.cuda())
    assert fwd.read_status() == 0
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what="edge blocks")


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_stage_scan_finds_the_stage_that_holds_a_nan(cuda_lib, name):
    """megamoe_forward_scan_stages (the pages' stage-by-stage NaN hunt): clean
    on a clean forward, also with NaN in the unwritten padding rows; a
    non-finite value planted in a valid row of one stage sets that stage's
    bit and no other."""
    cfg = inputs.CONFIGS[name]
    raw, weights = _weights(cfg)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    fwd.ws.fill_(0xFF)  # padding rows keep NaN patterns
    out = fwd(x, ids.cuda(), w.cuda())
    assert fwd.read_status() == 0
    assert fwd.scan_stages() == 0
    v = fwd.intermediates()
    R = int(v["padded_offsets"][-1].item())
    valid = torch.nonzero(v["row_src"][:R] >= 0).flatten()
    assert (v["row_src"][:R] < 0).any() or R == valid.numel()
    r = int(valid[valid.numel() // 2].item())
    cases = [("xq_sf", megamoe.STAGE_XQ_SCALE, 0x7F), ("h", megamoe.STAGE_H, float("nan")),
             ("hq_sf", megamoe.STAGE_HQ_SCALE, 0xFF),
             ("y_exp", megamoe.STAGE_Y, 127)]  # a BFP16 group holding Inf or NaN
    for key, bit, bad in cases:
        t = v[key]
        i = r // 16 if key == "y_exp" else r  # one exponent row per 16 rows
        keep = t[i, 3].clone()
        t[i, 3] = bad
        assert fwd.scan_stages() == bit, key
        t[i, 3] = keep
    assert fwd.scan_stages() == 0
    keep = out[1, 5].clone()
    out[1, 5] = float("nan")
    assert fwd.scan_stages(out) == megamoe.STAGE_OUT
    out[1, 5] = keep
