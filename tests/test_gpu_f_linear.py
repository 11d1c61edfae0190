"""megamoe_linear_nvfp4 (the dense NVFP4 linear with a measured-amax
activation scale) against the oracle's linear: the measured amax and global
scale bit-exact, the output within the stated tolerance, on tiny and
attention-projection shapes (full where the oracle is quick, sampled rows at
4096 tokens), both output types, and the edge cases."""

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


def _prepared(cfg):
    x, c, s, gs = inputs.make_linear(cfg, device="cuda")
    return x, c, s, gs, megamoe.LinearWeights.prepare(c, s, gs)


def _run(x, w, out_dtype=megamoe.EPI_BF16):
    out, ws = megamoe.linear_nvfp4(x, w, out_dtype)
    torch.cuda.synchronize()
    scal = ws[:12].cpu().numpy()
    amax, gs = scal[:8].view(np.float32)
    status = int(scal[8:12].view(np.uint32)[0])
    return out, np.float32(amax), np.float32(gs), status


@pytest.mark.parametrize("name,T", [("linear_tiny", None), ("linear_qa_decode", None),
                                    ("linear_qa_decode", 1), ("linear_qa_decode", 300)])
@pytest.mark.parametrize("out_dtype", [megamoe.EPI_BF16, megamoe.EPI_F32])
def test_linear_matches_oracle(cuda_lib, name, T, out_dtype):
    cfg = inputs.LINEAR_CONFIGS[name]
    if T is not None:
        from dataclasses import replace
        cfg = replace(cfg, T=T)
    x, c, s, gs, w = _prepared(cfg)
    out, amax, gsx, status = _run(x, w, out_dtype)
    assert status == 0
    want, inter = oracle.linear(x.float().cpu().numpy(), c.cpu().numpy(), s.cpu().numpy(), gs,
                                round_bf16=False)
    assert amax == inter["amax_x"] and gsx == inter["gs_x"]
    got = out.float().cpu().numpy()
    if out_dtype == megamoe.EPI_BF16:
        assert_close_bf16(got, want, what=f"{name} T={cfg.T} bf16")
    else:
        assert_close(got, want, what=f"{name} T={cfg.T} f32")


@pytest.mark.parametrize("name", ["linear_qa_prefill", "linear_qb_prefill"])
def test_linear_full_size_sampled_rows(cuda_lib, name):
    """4096 tokens: amax and gs bit-exact against the whole x, 48 sampled
    rows (the first and last included) against the oracle computed row by row
    with that amax, and the whole output finite."""
    cfg = inputs.LINEAR_CONFIGS[name]
    x, c, s, gs, w = _prepared(cfg)
    out, amax, gsx, status = _run(x, w)
    assert status == 0
    xf = x.float().cpu().numpy()
    assert amax == np.float32(np.abs(xf).max())
    assert gsx == np.float32(2688.0) / amax
    o = out.float()
    assert bool(torch.isfinite(o).all())
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, 46, replace=False)]))
    want, _ = oracle.linear(xf[rows], c.cpu().numpy(), s.cpu().numpy(), gs, amax=amax,
                            round_bf16=False)
    assert_close_bf16(o[torch.from_numpy(rows).cuda()].cpu().numpy(), want, what=name)


def test_linear_nonfinite_input_sets_status(cuda_lib):
    cfg = inputs.LINEAR_CONFIGS["linear_tiny"]
    x, c, s, gs, w = _prepared(cfg)
    x = x.clone()
    x[3, 9] = float("nan")
    _, _, _, status = _run(x, w)
    assert status & megamoe.DEV_NONFINITE


def test_linear_large_batch_amax_path(cuda_lib):
    """Above one block's share (T*K > 262144) the amax is reduced by k_amax."""
    cfg = inputs.LinearConfig("linear_mid", 600, 512, 128, seed=2005)
    x, c, s, gs, w = _prepared(cfg)
    out, amax, gsx, status = _run(x, w)
    assert status == 0
    want, inter = oracle.linear(x.float().cpu().numpy(), c.cpu().numpy(), s.cpu().numpy(), gs,
                                round_bf16=False)
    assert amax == inter["amax_x"] and gsx == inter["gs_x"]
    assert_close_bf16(out.float().cpu().numpy(), want, what="linear_mid")


def test_linear_edge_cases(cuda_lib):
    lib = megamoe.load()
    cfg = inputs.LINEAR_CONFIGS["linear_tiny"]
    x, c, s, gs, w = _prepared(cfg)
    out, ws = megamoe.linear_nvfp4(x[:0], w)
    assert out.shape == (0, cfg.N)
    ws = torch.empty(megamoe.linear_workspace_size(cfg.T, cfg.K, cfg.N), dtype=torch.uint8, device="cuda")
    o = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device="cuda")
    p = megamoe._p
    # K not a multiple of 256, N not a multiple of 128, short workspace, bad dtype
    assert lib.megamoe_linear_nvfp4(p(x), cfg.T, 128, cfg.K, p(w.codes), p(w.scales), p(w.gs),
                                    cfg.N, megamoe.EPI_BF16, p(o), cfg.N, p(ws), ws.numel(),
                                    None) == 2
    assert lib.megamoe_linear_nvfp4(p(x), cfg.T, cfg.K, cfg.K, p(w.codes), p(w.scales), p(w.gs),
                                    64, megamoe.EPI_BF16, p(o), cfg.N, p(ws), ws.numel(),
                                    None) == 2
    assert lib.megamoe_linear_nvfp4(p(x), cfg.T, cfg.K, cfg.K, p(w.codes), p(w.scales), p(w.gs),
                                    cfg.N, megamoe.EPI_BF16, p(o), cfg.N, p(ws), 100, None) == 3
    assert lib.megamoe_linear_nvfp4(p(x), cfg.T, cfg.K, cfg.K, p(w.codes), p(w.scales), p(w.gs),
                                    cfg.N, megamoe.EPI_SILU_MUL, p(o), cfg.N, p(ws), ws.numel(),
                                    None) == 1


def test_linear_strided_input_and_output(cuda_lib):
    """x is a column slice of a wider buffer (ld_x > K) and out a slice of a
    wider one (ld_out > N): the strides are honoured and nothing outside the
    slices is written."""
    cfg = inputs.LINEAR_CONFIGS["linear_tiny"]
    x, c, s, gs, w = _prepared(cfg)
    xb = torch.zeros(cfg.T, cfg.K + 64, dtype=torch.bfloat16, device="cuda")
    xb[:, 32:32 + cfg.K] = x
    ob = torch.full((cfg.T, cfg.N + 128), 7.0, dtype=torch.bfloat16, device="cuda")
    xs, os_ = xb[:, 32:32 + cfg.K], ob[:, 64:64 + cfg.N]
    assert xs.stride(0) == cfg.K + 64 and os_.stride(0) == cfg.N + 128
    megamoe.linear_nvfp4(xs, w, out=os_)
    torch.cuda.synchronize()
    ref, _ = megamoe.linear_nvfp4(x.contiguous(), w)
    assert torch.equal(os_, ref)
    assert bool((ob[:, :64] == 7.0).all()) and bool((ob[:, 64 + cfg.N:] == 7.0).all())
