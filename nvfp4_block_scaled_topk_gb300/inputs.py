"""Seeded synthetic workloads for the MegaMoE routed-expert forward.

This module is the only code that both the CUDA path's tests/benchmark and the
CPU oracle consume.  It draws random inputs and holds none of the method's
arithmetic (no quantiser, no GEMM, no routing sort): the NVFP4 expert weights
are drawn directly as code bytes from fixed histograms.

Workloads (the five shapes of the MegaMoE study; 384 experts / top-6 is the
"Architecture: DeepSeek-V4 MegaMoE" section of "CURRENT_BUG.md -- DeepSeek-V4
Blackwell NVFP4"; the 48-expert slice with 1-8 tokens padded to 128 rows is
its "Test Plan" Phase 2; the activation statistics amax 1.27 / std 0.09 are
"Key evidence" of "Current Bug: vLLM produces NaN from layer 0"):

  tiny      8 experts, top-2, d=256,  I=512,  64 tokens, x ~ N(0, 0.09)
            clipped to |x| <= 1.3, ids = top-2 of N(0,1) logits
  decode    384 experts, top-6, d=7168, I=2048, 8 tokens (decode1: 1 token),
            uniform random distinct ids
  slice     48 experts, top-6, d=7168, I=2048, 8 tokens (slice1: 1 token),
            uniform random distinct ids, rows padded to 128 per expert
  prefill   384 experts, top-6, d=7168, I=2048, 4096 tokens, 0.1 % of x set
            to +-8, ids = top-6 of N(0,1) logits + bias_e, bias_e =
            -1.1 ln(rank_e) (rank from a seeded permutation; Zipf-1.1 load)
  large     384 experts, top-6, d=7168, I=2048, 16384 tokens, uniform ids
  prefill64 64 experts, top-6, d=7168, I=2048, 2048 tokens, uniform ids: a
            prefill-shaped case (about 192 tokens per expert) whose weights
            (about 1.5 GB) are small enough for multi-pass profiler captures

topk_weights are the softmax of the N(0,1) logits at the selected ids.

Expert weights (NVFP4, per expert: W13 [2I, d] = gate rows then up rows,
W2 [d, I]) are drawn per (expert, matrix) from their own generator, so any
subset of experts regenerates identically:
  * each 4-bit element code: sign uniform; magnitude code 0..7 with
    probabilities MAG_COUNTS / 128,
  * each E4M3 block-scale byte from SCALE_COUNTS / 256,
  * global scale gs = 2688 / amax_w with amax_w ~ U(0.105, 0.12).
The two histograms were measured on a block-quantised N(0, 0.02) tensor of
4096 x 7168 elements (gs = 2688 / amax), rounded to the counts below, so the
weights have the statistics of "N(0, 0.02) then NVFP4-quantised" without any
quantiser running here (the coarse counts put the dequantised standard
deviation at about 0.021-0.022).

Every draw depends on its generator's device as well as its seed: torch's
CPU and CUDA generators give different streams.  The same workload drawn on
the GPU and on the CPU is therefore two samples of one recipe (the prefill
routing activates 130 experts drawn on the GPU and 126 drawn on the CPU);
each comparison with the oracle uses the draws of its own run.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

#: magnitude-code histogram (codes 0..7 = 0, .5, 1, 1.5, 2, 3, 4, 6), out of 128
MAG_COUNTS = (9, 17, 16, 15, 19, 20, 18, 14)
#: E4M3 block-scale byte histogram, out of 256
SCALE_COUNTS = {
    0x6B: 1, 0x6C: 2, 0x6D: 4, 0x6E: 6, 0x6F: 10, 0x70: 20, 0x71: 37, 0x72: 42,
    0x73: 40, 0x74: 32, 0x75: 24, 0x76: 16, 0x77: 10, 0x78: 7, 0x79: 4, 0x7A: 1,
}
assert sum(MAG_COUNTS) == 128 and sum(SCALE_COUNTS.values()) == 256


def _mag_lut() -> torch.Tensor:
    lut = []
    for code, n in enumerate(MAG_COUNTS):
        lut += [code] * n
    return torch.tensor(lut, dtype=torch.uint8)


def _scale_lut() -> torch.Tensor:
    lut = []
    for byte, n in sorted(SCALE_COUNTS.items()):
        lut += [byte] * n
    return torch.tensor(lut, dtype=torch.uint8)


@dataclass(frozen=True)
class MoEConfig:
    name: str
    E: int
    k: int
    d: int
    I: int
    T: int
    routing: str  # "logits" | "uniform" | "zipf"
    seed: int
    pad: int = 32
    x_sigma: float = 0.09
    x_clip: float | None = None
    outlier_frac: float = 0.0
    outlier_value: float = 8.0

    @property
    def slots(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T)


CONFIGS = {
    "tiny": MoEConfig("tiny", 8, 2, 256, 512, 64, "logits", seed=0, x_clip=1.3),
    "decode": MoEConfig("decode", 384, 6, 7168, 2048, 8, "uniform", seed=1002),
    "decode1": MoEConfig("decode1", 384, 6, 7168, 2048, 1, "uniform", seed=1012),
    "slice": MoEConfig("slice", 48, 6, 7168, 2048, 8, "uniform", seed=1003, pad=128),
    "slice1": MoEConfig("slice1", 48, 6, 7168, 2048, 1, "uniform", seed=1013, pad=128),
    "prefill": MoEConfig("prefill", 384, 6, 7168, 2048, 4096, "zipf", seed=1004,
                         outlier_frac=1e-3),
    "large": MoEConfig("large", 384, 6, 7168, 2048, 16384, "uniform", seed=1005),
    # prefill-shaped case small enough for multi-pass profiler captures:
    # 64 experts hold about 1.5 GB of weights, ~192 tokens per expert
    "prefill64": MoEConfig("prefill64", 64, 6, 7168, 2048, 2048, "uniform", seed=1006),
}


@dataclass(frozen=True)
class LinearConfig:
    """A dense NVFP4 linear layer x [T, K] @ W[N, K].T."""

    name: str
    T: int
    K: int
    N: int
    seed: int
    x_sigma: float = 0.09
    outlier_frac: float = 0.0
    outlier_value: float = 8.0


#: attention-projection-shaped linear layers.  The pages name the NVFP4
#: projections (q_a, kv, q_b, o_b) but give no sizes; these take the
#: DeepSeek-style hidden 7168 -> q_a rank 1536 and 1536 -> 128 heads x 192.
LINEAR_CONFIGS = {
    "linear_tiny": LinearConfig("linear_tiny", 40, 512, 256, seed=2001),
    "linear_qa_decode": LinearConfig("linear_qa_decode", 8, 7168, 1536, seed=2002),
    "linear_qa_prefill": LinearConfig("linear_qa_prefill", 4096, 7168, 1536, seed=2003,
                                      outlier_frac=1e-3),
    "linear_qb_prefill": LinearConfig("linear_qb_prefill", 4096, 1536, 24576, seed=2004),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _mix(*vals: int) -> int:
    """A fixed 63-bit mix of integers, used to derive per-stream seeds."""
    h = 0x243F6A8885A308D3
    for v in vals:
        h ^= (int(v) + 0x9E3779B97F4A7C15 + (h << 6) + (h >> 2)) & 0xFFFF_FFFF_FFFF_FFFF
        h &= 0x7FFF_FFFF_FFFF_FFFF
    return h


# --------------------------------------------------------------------------
# activations and routing
# --------------------------------------------------------------------------
def make_activations(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """hidden_states [T, d] bf16."""
    g = _gen(_mix(cfg.seed, 1), device)
    x = torch.randn(cfg.T, cfg.d, generator=g, device=device, dtype=torch.float32) * cfg.x_sigma
    if cfg.x_clip is not None:
        x = x.clamp(-cfg.x_clip, cfg.x_clip)
    if cfg.outlier_frac > 0 and x.numel():
        n = max(1, int(round(cfg.outlier_frac * x.numel())))
        pos = torch.randperm(x.numel(), generator=g, device=device)[:n]
        sign = torch.randint(0, 2, (n,), generator=g, device=device).float() * 2 - 1
        x.view(-1)[pos] = sign * cfg.outlier_value
    return x.to(torch.bfloat16)


def make_routing(cfg: MoEConfig, device="cpu"):
    """(topk_ids [T, k] int32, topk_weights [T, k] float32)."""
    g = _gen(_mix(cfg.seed, 2), device)
    T, E, k = cfg.T, cfg.E, cfg.k
    if cfg.routing == "uniform":
        u = torch.rand(T, E, generator=g, device=device)
        ids = torch.argsort(u, dim=1)[:, :k]
        logits = torch.randn(T, k, generator=g, device=device)
    elif cfg.routing in ("logits", "zipf"):
        logits_all = torch.randn(T, E, generator=g, device=device)
        score = logits_all
        if cfg.routing == "zipf":
            rank = torch.randperm(E, generator=g, device=device).float() + 1.0
            score = logits_all - 1.1 * torch.log(rank)[None, :]
        ids = torch.topk(score, k, dim=1).indices
        logits = torch.gather(logits_all, 1, ids)
    else:
        raise ValueError(cfg.routing)
    w = torch.softmax(logits.float(), dim=1)
    return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def make_router_logits(cfg: MoEConfig, device="cpu"):
    """(logits [T, E] float32 ~ N(0, 1), bias [E] float32 or None): the
    router's inputs, from their own stream; for the Zipf-loaded configs the
    bias is -1.1 ln(rank_e) with rank from a seeded permutation."""
    g = _gen(_mix(cfg.seed, 5), device)
    logits = torch.randn(cfg.T, cfg.E, generator=g, device=device, dtype=torch.float32)
    bias = None
    if cfg.routing == "zipf":
        rank = torch.randperm(cfg.E, generator=g, device=device).float() + 1.0
        bias = (-1.1 * torch.log(rank)).to(torch.float32)
    return logits, bias


def with_shared_expert(cfg: MoEConfig) -> MoEConfig:
    """The same workload with one shared expert: expert index cfg.E (drawn
    like the routed experts, from its own stream), visited by every token
    with weight 1 as slot k; so E + 1 experts and k + 1 slots per token."""
    return replace(cfg, name=cfg.name + "+shared", E=cfg.E + 1, k=cfg.k + 1)


# --------------------------------------------------------------------------
# NVFP4 expert weights
# --------------------------------------------------------------------------
def _nvfp4_matrix(seed: int, rows: int, K: int, device):
    g = _gen(seed, device)
    mag = _mag_lut().to(device)
    sc = _scale_lut().to(device)
    r = torch.randint(0, 256, (2, rows, K // 2), generator=g, device=device, dtype=torch.int32)
    lo = mag[(r[0] & 127).long()] | ((r[0] >> 7) << 3).to(torch.uint8)
    hi = mag[(r[1] & 127).long()] | ((r[1] >> 7) << 3).to(torch.uint8)
    codes = (lo | (hi << 4)).to(torch.uint8)
    s = torch.randint(0, 256, (rows, K // 16), generator=g, device=device, dtype=torch.int32)
    scales = sc[s.long()]
    amax = 0.105 + 0.015 * torch.rand((), generator=g, device=device, dtype=torch.float64).item()
    gs = np.float32(2688.0) / np.float32(amax)
    return codes, scales, float(gs)


def make_expert(cfg: MoEConfig, e: int, device="cpu") -> dict:
    """Expert e's NVFP4 weights as torch tensors on ``device``.

    w13_codes [2I, d/2] u8, w13_scales [2I, d/16] u8 (row-major E4M3 bytes),
    w13_gs [2] f32 (gate, up), w2_codes [d, I/2], w2_scales [d, I/16],
    w2_gs [1] f32.
    """
    d, I = cfg.d, cfg.I
    gc, gsc, ggs = _nvfp4_matrix(_mix(cfg.seed, 3, e, 0), I, d, device)
    uc, usc, ugs = _nvfp4_matrix(_mix(cfg.seed, 3, e, 1), I, d, device)
    dc, dsc, dgs = _nvfp4_matrix(_mix(cfg.seed, 3, e, 2), d, I, device)
    return dict(
        w13_codes=torch.cat([gc, uc], 0),
        w13_scales=torch.cat([gsc, usc], 0),
        w13_gs=torch.tensor([ggs, ugs], dtype=torch.float32, device=device),
        w2_codes=dc,
        w2_scales=dsc,
        w2_gs=torch.tensor([dgs], dtype=torch.float32, device=device),
    )


def make_all_experts(cfg: MoEConfig, device="cpu") -> dict:
    """All experts stacked: w13_codes [E, 2I, d/2], ..., w2_gs [E]."""
    E, d, I = cfg.E, cfg.d, cfg.I
    out = dict(
        w13_codes=torch.empty(E, 2 * I, d // 2, dtype=torch.uint8, device=device),
        w13_scales=torch.empty(E, 2 * I, d // 16, dtype=torch.uint8, device=device),
        w13_gs=torch.empty(E, 2, dtype=torch.float32, device=device),
        w2_codes=torch.empty(E, d, I // 2, dtype=torch.uint8, device=device),
        w2_scales=torch.empty(E, d, I // 16, dtype=torch.uint8, device=device),
        w2_gs=torch.empty(E, dtype=torch.float32, device=device),
    )
    for e in range(E):
        w = make_expert(cfg, e, device)
        for key, v in w.items():
            out[key][e] = v.reshape(out[key][e].shape)
    return out


def make_linear(cfg: LinearConfig, device="cpu"):
    """(x [T, K] bf16, codes [N, K/2] u8, scales [N, K/16] u8, gs float) with
    x ~ N(0, x_sigma) (plus +-outlier_value at outlier_frac of the entries)
    and the weight drawn like the experts' (NVFP4 bytes from the fixed
    histograms)."""
    g = _gen(_mix(cfg.seed, 1), device)
    x = torch.randn(cfg.T, cfg.K, generator=g, device=device, dtype=torch.float32) * cfg.x_sigma
    if cfg.outlier_frac > 0 and x.numel():
        n = max(1, int(round(cfg.outlier_frac * x.numel())))
        pos = torch.randperm(x.numel(), generator=g, device=device)[:n]
        sign = torch.randint(0, 2, (n,), generator=g, device=device).float() * 2 - 1
        x.view(-1)[pos] = sign * cfg.outlier_value
    codes, scales, gs = _nvfp4_matrix(_mix(cfg.seed, 4), cfg.N, cfg.K, device)
    return x.to(torch.bfloat16), codes, scales, gs


class ExpertSet:
    """Expert weights as NumPy arrays for the CPU oracle, fetched lazily.

    ``source`` is either a stacked dict (as from ``make_all_experts``, on any
    device) or None, in which case expert e is drawn on the CPU on first use.
    Only the experts actually touched are materialised on the host.
    """

    def __init__(self, cfg: MoEConfig, source: dict | None = None):
        self.cfg = cfg
        self.num_experts = cfg.E
        self.d = cfg.d
        self.I = cfg.I
        self._src = source
        self._cache: dict[int, dict] = {}

    def __len__(self):
        return self.num_experts

    def __getitem__(self, e: int) -> dict:
        e = int(e)
        if e not in self._cache:
            if self._src is None:
                w = make_expert(self.cfg, e, "cpu")
                w = {k: v.numpy() for k, v in w.items()}
            else:
                w = {k: v[e].detach().cpu().numpy() for k, v in self._src.items()}
            w["w2_gs"] = np.float32(np.asarray(w["w2_gs"]).reshape(-1)[0])
            self._cache[e] = w
        return self._cache[e]


def expected_tokens_per_expert(cfg: MoEConfig) -> float:
    return cfg.slots / cfg.E


def algorithmic_bytes(cfg: MoEConfig, active_experts: int) -> int:
    """Bytes one forward must move at least: each active expert's NVFP4
    weights once (0.5 B code + 1/16 B scale per element), x read and out
    written in bf16, and the routing inputs."""
    w = active_experts * 3 * cfg.d * cfg.I * (0.5 + 1.0 / 16)
    return int(w + 2 * cfg.T * cfg.d * 2 + cfg.T * cfg.k * 8)


def algorithmic_flops(cfg: MoEConfig, valid_slots: int) -> int:
    """6 d I per valid slot: gate, up and down GEMMs, 2 flops per MAC."""
    return 6 * cfg.d * cfg.I * valid_slots

