"""Failure detection on the GPU without a GPU fault: a bounded wait that runs
out sets MEGAMOE_DEV_TIMEOUT, the kernel unwinds (copies in flight land,
tensor memory is freed) and the context stays usable."""

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import check_forward

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_sets_timeout_and_context_survives(cuda_lib):
    cfg = inputs.CONFIGS["tiny"]
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg)
    ids, w = inputs.make_routing(cfg)
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    try:
        # 100 ns: every pipeline wait that is not already satisfied runs out
        megamoe.set_wait_limit_ns(100)
        fwd(x.cuda(), ids.cuda(), w.cuda())
        bits = fwd.read_status()
    finally:
        megamoe.set_wait_limit_ns(0)
    assert bits & megamoe.DEV_TIMEOUT
    # the context is intact: the next forward is correct and clean
    out = fwd(x.cuda(), ids.cuda(), w.cuda())
    assert fwd.read_status() == 0
    ex = inputs.ExpertSet(cfg, raw)
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(), ex, pad=32,
                              return_intermediates=True)
    check_forward(fwd, out, inter, ex, ids.numpy(), w.numpy(), what="after timeout")


@pytest.mark.parametrize("tile_n", [128, 256])
def test_grouped_gemm_wait_that_runs_out_unwinds(cuda_lib, tile_n):
    """The same for the grouped GEMM alone, in both tile orientations
    (weights on M with 128-token tiles; token-major 128 x 256 tiles): the
    status word gets the timeout bit, and the next launch is exact."""
    cfg = inputs.MoEConfig("fail_gemm", 8, 2, 512, 512, 256, "uniform", seed=77)
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    fwd(x, ids.cuda(), w.cuda())
    v = fwd.intermediates()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        return megamoe.grouped_gemm(v["xq_codes"], v["xq_sf"], v["gs_x"], weights.w13_codes,
                                    weights.w13_scales, weights.w13_gs, v["offsets"],
                                    v["padded_offsets"], megamoe.EPI_SILU_MUL, tile_n=tile_n,
                                    status=status)

    want, _ = run()
    want = want.clone()
    torch.cuda.synchronize()
    assert status.item() == 0
    try:
        megamoe.set_wait_limit_ns(100)
        run()
        torch.cuda.synchronize()
    finally:
        megamoe.set_wait_limit_ns(0)
    assert status.item() & megamoe.DEV_TIMEOUT
    status.zero_()
    got, _ = run()
    torch.cuda.synchronize()
    assert status.item() == 0
    valid = v["row_src"][:int(v["padded_offsets"][-1].item())] >= 0
    assert torch.equal(got[:valid.numel()][valid], want[:valid.numel()][valid])


def test_fused_requant_barrier_that_runs_out(cuda_lib):
    """The forward with the requantisation of h fused into its L1 kernel
    (token-major tiles, a grid-wide arrival count behind the last tile):
    with a 100 ns limit every wait, that one included, runs out; the timeout
    bit is set, the kernel returns, and the next forward equals a clean one."""
    cfg = inputs.MoEConfig("fail_fused", 8, 2, 512, 512, 256, "uniform", seed=78)
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    ids, w = ids.cuda(), w.cuda()
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    try:
        megamoe.set_fused_requant(True)
        want = fwd(x, ids, w).clone()
        assert fwd.read_status() == 0
        try:
            megamoe.set_wait_limit_ns(100)
            fwd(x, ids, w)
            bits = fwd.read_status()
        finally:
            megamoe.set_wait_limit_ns(0)
        assert bits & megamoe.DEV_TIMEOUT
        out = fwd(x, ids, w)
        assert fwd.read_status() == 0
        assert torch.equal(out, want)
    finally:
        megamoe.set_fused_requant(False)
