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
