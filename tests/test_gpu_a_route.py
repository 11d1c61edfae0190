"""megamoe_route_permute against the oracle's stable counting sort: bit-exact
counts, offsets, padded offsets, row_src and slot_dst."""

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe

pytestmark = pytest.mark.gpu


def _check(ids_np, E, pad):
    ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = megamoe.route_permute(ids, E, pad, status=status)
    torch.cuda.synchronize()
    want = oracle.route(np.where(ids_np >= E, -1, ids_np), E, pad)
    R = int(want.padded_offsets[-1])
    assert np.array_equal(r["counts"].cpu().numpy(), want.counts)
    assert np.array_equal(r["offsets"].cpu().numpy(), want.offsets)
    assert np.array_equal(r["padded_offsets"].cpu().numpy(), want.padded_offsets)
    rs = r["row_src"].cpu().numpy()
    assert np.array_equal(rs[:R], want.row_src)
    assert np.all(rs[R:] == -1)
    assert np.array_equal(r["slot_dst"].cpu().numpy(), want.slot_dst)
    return int(status.item())


@pytest.mark.parametrize("name,pad", [("tiny", 1), ("tiny", 32), ("tiny", 128), ("decode", 32),
                                      ("decode1", 32), ("slice", 128), ("slice1", 128),
                                      ("prefill", 32), ("large", 32), ("large", 1)])
def test_route_bit_exact_on_workloads(cuda_lib, name, pad):
    cfg = inputs.CONFIGS[name]
    ids, _ = inputs.make_routing(cfg)
    assert _check(ids.numpy(), cfg.E, pad) == 0


@pytest.mark.parametrize("case", ["all_one_expert", "one_nonempty", "negatives", "dups_k16",
                                  "single_expert", "empty_tokens", "ragged_big"])
def test_route_edge_cases(cuda_lib, case):
    rng = np.random.default_rng(11)
    if case == "all_one_expert":
        ids, E = np.full((300, 6), 5), 384
    elif case == "one_nonempty":
        ids, E = np.full((7, 3), 47), 48
    elif case == "negatives":
        ids, E = rng.integers(-1, 16, (100, 4)), 16
    elif case == "dups_k16":
        ids, E = rng.integers(0, 3, (33, 16)), 3
    elif case == "single_expert":
        ids, E = np.zeros((5, 1), dtype=np.int64), 1
    elif case == "empty_tokens":
        ids, E = np.zeros((0, 6), dtype=np.int64), 384
    else:
        ids, E = rng.integers(0, 1024, (5000, 8)), 1024
    for pad in (1, 32, 128):
        assert _check(ids, E, pad) == 0


def test_route_flags_and_skips_out_of_range_ids(cuda_lib):
    rng = np.random.default_rng(12)
    ids = rng.integers(0, 10, (40, 4))
    ids[3, 1] = 10
    ids[17, 0] = 1000
    assert _check(ids, 10, 32) & megamoe.DEV_BAD_EXPERT_ID


@pytest.mark.parametrize("case", ["uniform", "all_one_expert", "skipped_and_bad", "zipf_1024"])
def test_multi_block_routing_in_the_forward(cuda_lib, case):
    """From 16384 slots on, the forward routes over many blocks (per-block
    histograms, one-block offsets, per-block stable scatter); its routing
    views must equal the oracle's stable sort exactly, padding and all."""
    E, k, T = (1024, 8, 4096) if case == "zipf_1024" else (64, 6, 4096)
    routing = "zipf" if case == "zipf_1024" else "uniform"
    cfg = inputs.MoEConfig("route_multi", E, k, 256, 256, T, routing, seed=321)
    raw = inputs.make_all_experts(cfg, device="cuda")
    weights = megamoe.Weights.prepare(raw)
    x = inputs.make_activations(cfg).cuda()
    ids, w = inputs.make_routing(cfg)
    ids = ids.clone()
    if case == "all_one_expert":
        ids[:, 0] = 5
        ids[:, 1:] = -1
    elif case == "skipped_and_bad":
        g = torch.Generator().manual_seed(3)
        ids[torch.rand(ids.shape, generator=g) < 0.2] = -1
        ids[torch.rand(ids.shape, generator=g) < 0.01] = E + 7
    assert T * k >= 16384
    fwd = megamoe.Forward(weights, T, k, pad=32)
    fwd(x, ids.cuda(), w.cuda())
    bits = fwd.read_status()
    assert bool(bits & megamoe.DEV_BAD_EXPERT_ID) == (case == "skipped_and_bad")
    ids_np = ids.numpy()
    want = oracle.route(np.where(ids_np >= E, -1, ids_np), E, 32)
    v = fwd.intermediates()
    R = int(want.padded_offsets[-1])
    assert np.array_equal(v["counts"].cpu().numpy(), want.counts)
    assert np.array_equal(v["offsets"].cpu().numpy(), want.offsets)
    assert np.array_equal(v["padded_offsets"].cpu().numpy(), want.padded_offsets)
    rs = v["row_src"].cpu().numpy()
    assert np.array_equal(rs[:R], want.row_src)
    assert np.all(rs[R:] == -1)
    assert np.array_equal(v["slot_dst"].cpu().numpy(), want.slot_dst)
