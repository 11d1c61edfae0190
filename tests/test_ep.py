"""The expert-parallel forward's exchange on CPU ranks (gloo, world size 2).

Each rank holds half of the experts and runs its two halves of the forward
with the oracle standing in for the library (no GPU here); the orchestration
under test is the product's (``ep.ExpertParallelForward``): the token
all-gather, the all-reduce(max) of amax(h) between L1 and the
requantisation, and the reduce-scatter(sum) of the partial outputs.  The
ranks' outputs together must equal the oracle's single-device forward; with
the amax(h) exchange taken out they must not.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from nvfp4_block_scaled_topk_gb300 import inputs


class _SliceExperts:
    """Experts [base, base + n) of an expert set, under local ids 0..n-1."""

    def __init__(self, experts, base, n):
        self.ex, self.base = experts, base
        self.num_experts, self.d, self.I = n, experts.d, experts.I

    def __getitem__(self, e):
        return self.ex[self.base + int(e)]


class OracleShard:
    """One rank's halves of the forward computed by the oracle (float64):
    begin -> the shard's amax(h); end -> the shard's combine before rounding,
    with the (exchanged) amax(h) it is handed back."""

    def __init__(self, experts, base, n, pad):
        self.ex = _SliceExperts(experts, base, n)
        self.base, self.n, self.pad = base, n, pad

    def _local(self, ids):
        ids = ids.numpy()
        return np.where((ids >= self.base) & (ids < self.base + self.n), ids - self.base, -1)

    def begin(self, x, ids):
        self.x = x.float().numpy()
        self.ids = self._local(ids)
        # the shard's own amax of h (its valid rows): L1 with the whole batch's x
        _, inter = oracle.forward(self.x, self.ids, np.zeros(self.ids.shape), self.ex,
                                  pad=self.pad, return_intermediates=True)
        self.amax_h = torch.tensor([float(inter["amax_h_own"])], dtype=torch.float32)
        return self.amax_h

    def end(self, w):
        _, inter = oracle.forward(self.x, self.ids, w.numpy(), self.ex, pad=self.pad,
                                  return_intermediates=True, amax_h=self.amax_h.item())
        return torch.from_numpy(inter["out_f64"])

    def round(self, total):
        return torch.from_numpy(oracle.bf16_round(total.numpy()))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q, skip_amax_exchange):
    import torch.distributed as dist

    from nvfp4_block_scaled_topk_gb300 import ep

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if skip_amax_exchange:  # a planted mistake: each rank keeps its own amax(h)
            real = dist.all_reduce

            def all_reduce(t, op=dist.ReduceOp.SUM, group=None):
                if op == dist.ReduceOp.MAX:
                    return None
                return real(t, op=op, group=group)

            dist.all_reduce = all_reduce
        cfg = inputs.CONFIGS["tiny"]
        x = inputs.make_activations(cfg)
        ids, w = inputs.make_routing(cfg)
        Tl = cfg.T // world
        sl = slice(rank * Tl, (rank + 1) * Tl)
        base, n = ep.shard_range(cfg.E, world, rank)
        shard = OracleShard(inputs.ExpertSet(cfg), base, n, pad=32)
        f = ep.ExpertParallelForward(shard, Tl)
        out, total = f(x[sl].float(), ids[sl], w[sl].double(), return_sum=True)
        q.put((rank, out.numpy(), total.numpy()))
    finally:
        dist.destroy_process_group()


def _run(skip_amax_exchange=False):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q, skip_amax_exchange))
             for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (o, t)) for r, o, t in (q.get(timeout=300) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out = np.concatenate([res[r][0] for r in range(world)])
    total = np.concatenate([res[r][1] for r in range(world)])
    return out, total


@pytest.fixture(scope="module")
def single_device():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.make_activations(cfg).float().numpy()
    ids, w = inputs.make_routing(cfg)
    out, inter = oracle.forward(x, ids.numpy(), w.numpy(), inputs.ExpertSet(cfg), pad=32,
                                return_intermediates=True)
    return out, inter


def test_two_ranks_equal_the_single_device_forward(single_device):
    out1, inter = single_device
    out, total = _run()
    # the sums agree to float64 rounding (shard order vs slot order), and so
    # do the bf16 outputs
    np.testing.assert_allclose(total, inter["out_f64"], rtol=0,
                               atol=1e-12 * np.abs(inter["out_f64"]).max())
    assert np.mean(out == out1) > 0.999
    from helpers import assert_close_bf16

    assert_close_bf16(out, inter["out_f64"], what="expert-parallel forward")


def test_the_amax_exchange_is_needed(single_device):
    _, inter = single_device
    _, total = _run(skip_amax_exchange=True)
    err = np.abs(total - inter["out_f64"]).max() / np.abs(inter["out_f64"]).max()
    assert err > 1e-6, "each rank's own amax(h) should change the result"


def test_shard_ranges_cover_the_experts():
    from nvfp4_block_scaled_topk_gb300 import ep

    assert [ep.shard_range(384, 8, r) for r in range(8)] == [(48 * r, 48) for r in range(8)]
    with pytest.raises(ValueError):
        ep.shard_range(10, 4, 0)
