"""megamoe_forward_static: the forward for callers that cannot allocate.

Callers such as plugins in a process that owns all device memory, embedded
callers with no allocator at hand, or loops that must never enter the
allocator use the library's fixed internal workspace instead of one they pass
in.  This file is collected last on purpose.  It checks, through the C ABI,
that two calls in a row match megamoe_forward on the same inputs (and, on the
small workload, the oracle), and that a shape too large for the fixed
workspace is refused, after the forward's own shape checks.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_static_workspace_forward_matches_forward_twice(cuda_lib, name):
    cfg = inputs.CONFIGS[name]
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    ids, w = ids.cuda(), w.cuda()
    ref = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)(x, ids, w).float().cpu().numpy()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = megamoe.forward_static(weights, x, ids, w, pad=32, status_out=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        got = out.float().cpu().numpy()
        assert_close(got, ref, what=f"static workspace {name}")
        assert np.array_equal(got, ref)  # same kernels on the same inputs
    if name == "tiny":
        want = oracle.forward(x.float().cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(),
                              inputs.ExpertSet(cfg, raw), pad=32, return_intermediates=True)[1]
        assert_close_bf16(got[:cfg.T].astype(np.float64), want["out_f64"],
                          what="static workspace against the oracle")
    del raw, weights
    torch.cuda.empty_cache()


def test_static_workspace_refuses_oversized_shapes(cuda_lib):
    cfg = inputs.CONFIGS["decode"]
    lib = megamoe.load()
    fake = ctypes.c_void_p(256)
    cw = megamoe.CWeights(cfg.E, cfg.d, cfg.I, 256, 256, 256, 256, 256, 256)
    # 64 tokens of the MegaMoE decode shape need more than the fixed 64 MiB
    assert megamoe.workspace_size(64, 6, cfg.E, cfg.d, cfg.I, 32) > (64 << 20)
    code = lib.megamoe_forward_static(ctypes.byref(cw), fake, fake, fake, 64, 6, 32, fake, None,
                                      None)
    assert code == 3  # MEGAMOE_ERR_WORKSPACE_TOO_SMALL


def test_static_workspace_reports_shape_errors_before_the_size(cuda_lib):
    """A shape the forward cannot take (d not a multiple of 256) that would
    also overflow the fixed workspace is reported as unsupported, not as a
    workspace limit; a valid oversized shape is the workspace limit."""
    lib = megamoe.load()
    fake = ctypes.c_void_p(256)
    cw = megamoe.CWeights(384, 7168 + 128, 2048, 256, 256, 256, 256, 256, 256)
    code = lib.megamoe_forward_static(ctypes.byref(cw), fake, fake, fake, 4096, 6, 32, fake, None,
                                      None)
    assert code == 2  # MEGAMOE_ERR_UNSUPPORTED_SHAPE
    cw = megamoe.CWeights(384, 7168, 2048, 256, 256, 256, 256, 256, 256)
    code = lib.megamoe_forward_static(ctypes.byref(cw), fake, fake, fake, 4096, 6, 32, fake, None,
                                      None)
    assert code == 3  # MEGAMOE_ERR_WORKSPACE_TOO_SMALL
