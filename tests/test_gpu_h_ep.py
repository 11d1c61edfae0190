"""The expert-parallel shard calls on one GPU, through the C ABI.

G shards of one layer run one after another on the same GPU (no kernel of
one shard waits on another's), with the exchange steps done on the device
between them: the all-gather is the shared input, the all-reduce(max) of
amax(h) a maximum over the shards' workspaces, the reduce-scatter(sum) a sum
of their fp32 partial outputs in shard order, then one bf16 rounding by the
library.  The result must meet the oracle's single-device forward (and
megamoe_forward) within the stated tolerance; on the MegaMoE decode batch
the shards are the pages' EP8 slices of 48 experts.
"""

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import ep, inputs, megamoe
from helpers import assert_close_bf16, bf16_to_np

pytestmark = pytest.mark.gpu


def _ep_forward(weights, E_total, G, x, ids, w, pad):
    T, k = ids.shape
    shards = []
    for g in range(G):
        base, n = ep.shard_range(E_total, G, g)
        shards.append(megamoe.ShardForward(weights.shard(base, n), base, E_total, T, k, pad))
    amax = [s.begin(x, ids) for s in shards]
    top = torch.stack(amax).max(dim=0).values
    for a in amax:
        a.copy_(top)
    total = torch.zeros(T, weights.d, dtype=torch.float32, device=x.device)
    for s in shards:
        total += s.end(w)
    out = megamoe.round_bf16(total)
    torch.cuda.synchronize()
    assert all(s.read_status() == 0 for s in shards)
    return out, shards, top.item()


@pytest.mark.parametrize("name,G", [("tiny", 2), ("tiny", 4), ("decode", 8), ("decode1", 8)])
def test_sharded_forward_matches_oracle_and_forward(cuda_lib, name, G):
    cfg = inputs.CONFIGS[name]
    torch.cuda.empty_cache()
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg)
    ids, w = inputs.make_routing(cfg)
    xd, idsd, wd = x.cuda(), ids.cuda(), w.cuda()
    out, shards, amax_h = _ep_forward(weights, cfg.E, G, xd, idsd, wd, pad=32)
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=32)
    ref = fwd(xd, idsd, wd)
    assert fwd.read_status() == 0
    # the shards' L1 outputs are the single-device forward's rows: the same
    # global scale of h and, row for row, the same bits
    assert amax_h == fwd.intermediates()["amax_h"].item()
    got = bf16_to_np(out)
    # only the order of the fp32 additions across shards differs
    assert np.mean(got == bf16_to_np(ref)) > 0.99
    _, inter = oracle.forward(x.float().numpy(), ids.numpy(), w.numpy(),
                              inputs.ExpertSet(cfg, raw), pad=32, return_intermediates=True)
    assert_close_bf16(got, inter["out_f64"], what=f"{name} over {G} shards")


def test_shard_flags_ids_outside_the_layer(cuda_lib):
    cfg = inputs.CONFIGS["tiny"]
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    ids = ids.clone()
    ids[3, 0] = cfg.E + 5  # not an expert of the layer
    s = megamoe.ShardForward(weights.shard(0, 4), 0, cfg.E, cfg.T, cfg.k, 32)
    s.begin(x, ids.cuda())
    s.end(w.cuda())
    assert s.read_status() & megamoe.DEV_BAD_EXPERT_ID
    s2 = megamoe.ShardForward(weights.shard(4, 4), 4, cfg.E, cfg.T, cfg.k, 32)
    s2.begin(x, ids.cuda())
    assert s2.read_status() & megamoe.DEV_BAD_EXPERT_ID


def test_round_bf16_matches_oracle(cuda_lib):
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    got = megamoe.round_bf16(torch.from_numpy(v).cuda()).float().cpu().numpy()
    assert np.array_equal(got.astype(np.float64), oracle.bf16_round(v.astype(np.float64)))
