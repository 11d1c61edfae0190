"""Expert-parallel MoE forward: the experts sharded over a process group.

"CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Test Plan -- Finding the
NaN", Phase 2 runs the MoE as EP8: each of 8 GPUs holds 48 of the 384
experts.  Rank g of G owns experts [g E/G, (g+1) E/G).  One forward:

  1. all-gather the layer's tokens (x, topk_ids, topk_weights; every rank
     brings T_local tokens), so every rank sees all T = G T_local tokens;
  2. each rank routes the slots of its own experts, quantises x (its amax is
     over all T tokens, the same on every rank) and runs the L1 GEMM with
     SiLU(gate)*up (megamoe_ep_forward_begin);
  3. all-reduce(max) of amax(h): h has one global scale over every valid row
     of the layer's intermediate, whichever rank holds the row (without this
     exchange the shards' requantised h, and so the output, would depend on
     the sharding);
  4. each rank requantises its h rows with that scale, runs the L2 GEMM and
     the combine of its own slots in fp32 (megamoe_ep_forward_end);
  5. reduce-scatter(sum) of the fp32 partial outputs: rank g receives the
     sums of its own T_local tokens, rounded once to bf16.

The data plane of steps 1, 3 and 5 is the process group's backend (NCCL
between GPUs); everything else runs in the library's kernels.  The result
equals the single-device forward up to the order of the fp32 additions
across ranks.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import megamoe


def shard_range(num_experts: int, world: int, rank: int) -> tuple[int, int]:
    """(first expert, number of experts) of `rank`: equal contiguous slices."""
    if world < 1 or num_experts % world:
        raise ValueError("the experts must divide evenly over the ranks")
    n = num_experts // world
    return rank * n, n


class LibraryShard:
    """One rank's two halves of the forward, on its GPU (the library)."""

    def __init__(self, weights_shard: megamoe.Weights, expert_base: int, num_experts_total: int,
                 T: int, k: int, pad: int = 32):
        self.f = megamoe.ShardForward(weights_shard, expert_base, num_experts_total, T, k, pad)

    def begin(self, x, topk_ids) -> torch.Tensor:
        return self.f.begin(x, topk_ids)

    def end(self, topk_weights) -> torch.Tensor:
        return self.f.end(topk_weights)

    def round(self, total: torch.Tensor) -> torch.Tensor:
        return megamoe.round_bf16(total)


class ExpertParallelForward:
    """One rank's MoE forward with the experts sharded over `group`.

    ``shard`` runs the rank's halves of the forward (``LibraryShard``);
    every rank calls with its own T_local tokens and receives their output.
    """

    def __init__(self, shard, T_local: int, group=None):
        self.shard = shard
        self.T_local = T_local
        self.group = group

    def _gather(self, t: torch.Tensor) -> torch.Tensor:
        world = dist.get_world_size(self.group)
        out = torch.empty((world * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype,
                          device=t.device)
        dist.all_gather_into_tensor(out, t.contiguous(), group=self.group)
        return out

    def __call__(self, x_local, topk_ids_local, topk_weights_local, return_sum=False):
        if x_local.shape[0] != self.T_local:
            raise ValueError("every rank brings T_local tokens")
        # 1. the layer's tokens on every rank
        x = self._gather(x_local)
        ids = self._gather(topk_ids_local)
        w = self._gather(topk_weights_local)
        # 2-3. L1 on the rank's experts, then one global scale for h
        amax_h = self.shard.begin(x, ids)
        dist.all_reduce(amax_h, op=dist.ReduceOp.MAX, group=self.group)
        # 4-5. L2 and the rank's share of the combine, summed over the ranks
        partial = self.shard.end(w)
        mine = torch.empty((self.T_local,) + tuple(partial.shape[1:]), dtype=partial.dtype,
                           device=partial.device)
        dist.reduce_scatter_tensor(mine, partial.contiguous(), op=dist.ReduceOp.SUM,
                                   group=self.group)
        out = self.shard.round(mine)
        return (out, mine) if return_sum else out
