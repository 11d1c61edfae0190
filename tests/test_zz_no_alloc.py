"""megamoe_forward_static: the forward for callers that cannot allocate.

Callers such as code inside a CUDA stream capture, plugins in a process that
owns all device memory, or loops that must never enter the allocator use the
library's fixed internal workspace instead of one they pass in.  This file is
collected last on purpose.  It checks, through the C ABI, that two calls in a
row match megamoe_forward on the same inputs, and that a shape too large for
the fixed workspace is refused.
"""

import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import assert_close

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
