"""Routed-expert forward of the oracle (test infrastructure only).

Follows "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4":
  * "Architecture: DeepSeek-V4 MegaMoE": experts with top-k routing, one
    grouped GEMM problem per expert;
  * "What's Been Verified": L1 is the gate+up GEMM, L2 the down GEMM;
  * "Test Plan -- Finding the NaN", Phase 1: inputs hidden_states, topk_ids,
    topk_weights; per-expert token counts padded to 128 rows; activation quant
    before the grouped GEMM; L1 GEMM -> SiLU -> L2 GEMM;
  * same section, Phase 2: zero-token experts; expert_offsets and
    padded_expert_offsets;
and "Current Bug: vLLM produces NaN from layer 0", "What we've tried" item 1:
the activation global scale comes from the measured amax.

Readings taken where the pages are silent:
  A6  the L1 output h = SiLU(gate) * up is rounded to bf16 before it is
      re-quantised; its global scale comes from the amax of bf16 h over the
      valid rows only.
  A8  rows are ordered per expert by ascending flat slot index t*k + j (a
      stable counting sort).
  A9  padding rows carry no token (row_src = -1) and do not enter any amax.
  A10 ids < 0 are skipped; ids >= E are an error; a duplicate id in one
      token is two separate slots.
  A11 topk_weights are used as given (no renormalisation).
  A12 gate, up and down matrices each have their own global scale.
  A15 the combine sums j = 0..k-1 in float64 and rounds once to bf16.

All GEMMs here are float64 matmuls of dequantised operands; SiLU is
g / (1 + exp(-g)) in float64.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .nvfp4 import bf16_round, dequantize, quantize


@dataclass
class Routing:
    """Result of ``route``: the token-permutation metadata.

    counts[E]            valid slots per expert
    offsets[E+1]         exclusive prefix sum of counts (expert_offsets)
    padded_offsets[E+1]  exclusive prefix sum of counts rounded up to ``pad``
                         (padded_expert_offsets); a zero count stays zero
    row_src[R_pad]       flat slot t*k+j held by each padded row, -1 for padding
    slot_dst[T*k]        padded row of each slot, -1 for a skipped slot (id < 0)
    """

    counts: np.ndarray
    offsets: np.ndarray
    padded_offsets: np.ndarray
    row_src: np.ndarray
    slot_dst: np.ndarray
    pad: int


def route(topk_ids, num_experts: int, pad: int = 1) -> Routing:
    """Stable counting sort of the flat slots by expert id (readings A8-A10).

    Slot s = t*k + j goes to expert topk_ids[t, j].  Within an expert the slots
    keep ascending s order.  Expert e owns padded rows
    [padded_offsets[e], padded_offsets[e+1]); its first counts[e] rows hold its
    slots and the rest are padding.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    if ids.ndim != 2:
        raise ValueError("topk_ids must be [T, k]")
    if pad < 1:
        raise ValueError("pad must be >= 1")
    flat = ids.reshape(-1)
    if np.any(flat >= num_experts):
        raise ValueError("expert id >= number of experts")
    counts = np.zeros(num_experts, dtype=np.int64)
    for e in flat[flat >= 0]:
        counts[e] += 1
    offsets = np.concatenate([[0], np.cumsum(counts)])
    padded = (counts + pad - 1) // pad * pad
    padded_offsets = np.concatenate([[0], np.cumsum(padded)])
    row_src = np.full(int(padded_offsets[-1]), -1, dtype=np.int64)
    slot_dst = np.full(flat.size, -1, dtype=np.int64)
    for e in range(num_experts):
        slots = np.nonzero(flat == e)[0]  # ascending slot order
        rows = padded_offsets[e] + np.arange(slots.size)
        row_src[rows] = slots
        slot_dst[slots] = rows
    return Routing(counts, offsets, padded_offsets, row_src, slot_dst, pad)


def silu(g):
    """SiLU in float64: g / (1 + exp(-g))."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def grouped_gemm(a_codes, a_scales, a_gs, experts, which, routing: Routing,
                 epilogue: str = "f32", return_unrounded: bool = False):
    """One grouped block-scaled GEMM over all experts (float64 on dequantised data).

    Expert e multiplies its valid rows of A (the quantised activations in
    padded-row order) by the transpose of its weight matrix:
        out[r, :] = Ahat[r, :] @ What_e.T,   r in the valid rows of e.
    ``which`` picks the matrix: "w13" ([2I, d]: gate rows 0..I-1, up rows
    I..2I-1, global scales (gate, up)) or "w2" ([d, I], one global scale).
    ``experts`` is an expert set: ``experts.num_experts``, ``experts.d``,
    ``experts.I`` and ``experts[e]`` -> dict with w13_codes [2I, d/2],
    w13_scales [2I, d/16], w13_gs [2], w2_codes [d, I/2], w2_scales [d, I/16],
    w2_gs (scalar).

    epilogue "f32":       returns out [R_pad, N] float64 (padding rows NaN).
    epilogue "silu_mul":  ``which`` must be "w13"; returns
        (h [R_pad, I] float64 holding bf16 values, amax_h) with
        h = bf16(silu(gate) * up), padding rows 0, amax over valid rows;
        with return_unrounded also silu(gate) * up before the rounding.
    """
    ahat = dequantize(a_codes, a_scales, a_gs)
    R_pad = ahat.shape[0]
    n_out = 2 * experts.I if which == "w13" else experts.d
    out = np.full((R_pad, n_out), np.nan)
    for e in range(routing.counts.size):
        m = int(routing.counts[e])
        if m == 0:
            continue
        r0 = int(routing.padded_offsets[e])
        w = experts[e]
        if which == "w13":
            I = experts.I
            gate = dequantize(w["w13_codes"][:I], w["w13_scales"][:I], w["w13_gs"][0])
            up = dequantize(w["w13_codes"][I:], w["w13_scales"][I:], w["w13_gs"][1])
            wm = np.concatenate([gate, up], axis=0)
        elif which == "w2":
            wm = dequantize(w["w2_codes"], w["w2_scales"], w["w2_gs"])
        else:
            raise ValueError(which)
        out[r0:r0 + m] = ahat[r0:r0 + m] @ wm.T
    if epilogue == "f32":
        return out
    if epilogue == "silu_mul":
        if which != "w13":
            raise ValueError("silu_mul needs the gate+up matrix")
        I = experts.I
        h = np.zeros((R_pad, I))
        h64 = np.zeros((R_pad, I))
        amax = 0.0
        for e in range(routing.counts.size):
            m = int(routing.counts[e])
            if m == 0:
                continue
            r0 = int(routing.padded_offsets[e])
            v = out[r0:r0 + m]
            hu = silu(v[:, :I]) * v[:, I:]
            hv = bf16_round(hu)
            h[r0:r0 + m] = hv
            h64[r0:r0 + m] = hu
            amax = max(amax, float(np.max(np.abs(hv))))
        if return_unrounded:
            return h, np.float32(amax), h64
        return h, np.float32(amax)
    raise ValueError(epilogue)


def combine(y, topk_weights, slot_dst, round_bf16=True):
    """out[t] = bf16( sum_j w[t, j] * y[slot_dst[t*k + j]] ), j ascending, float64.

    Skipped slots (slot_dst = -1) contribute nothing; a token without a valid
    slot gives a zero row.  With round_bf16=False the float64 sum is returned
    before the final rounding.
    """
    w = np.asarray(topk_weights, dtype=np.float64)
    T, k = w.shape
    d = y.shape[1]
    out = np.zeros((T, d))
    for t in range(T):
        acc = np.zeros(d)
        for j in range(k):
            r = int(slot_dst[t * k + j])
            if r >= 0:
                acc = acc + w[t, j] * y[r]
        out[t] = acc
    return bf16_round(out) if round_bf16 else out


def forward(x, topk_ids, topk_weights, experts, pad: int = 1, return_intermediates=False,
            amax_x=None, amax_h=None):
    """The routed-expert forward, step by step as the pages order it.

    1. route: bucket slots per expert (expert_offsets / padded offsets);
    2. quantise the activations with gs from the measured amax of x;
    3. L1 grouped GEMM (gate+up), SiLU(gate)*up, round to bf16;
    4. re-quantise h with gs from the amax of h over valid rows;
    5. L2 grouped GEMM (down);
    6. top-k weighted combine, rounded once to bf16.
    ``x`` is [T, d] (bf16 values as float32); ``experts[e]`` holds expert e's
    NVFP4 weights.  Returns the [T, d] output as float64 bf16 values.

    ``amax_x`` / ``amax_h``: when the given tokens are a sample of a larger
    batch, the amax of the whole batch's x and of its whole intermediate
    (reading A2: one global scale per tensor, so a sampled token is quantised
    with the batch's scales); by default both are measured over the tokens
    given.  Every other step is unchanged: each token's output depends on the
    batch only through these two scalars.
    """
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    E = experts.num_experts
    rt = route(ids, E, pad)
    R_pad = int(rt.padded_offsets[-1])
    d = x.shape[1]

    xq_codes, xq_scales, gs_x, amax_x = quantize(x, amax=amax_x)
    # gather quantised token rows into padded-row order (padding rows zero)
    a_codes = np.zeros((R_pad, d // 2), dtype=np.uint8)
    a_scales = np.zeros((R_pad, d // 16), dtype=np.uint8)
    valid = rt.row_src >= 0
    a_codes[valid] = xq_codes[rt.row_src[valid] // k]
    a_scales[valid] = xq_scales[rt.row_src[valid] // k]

    h, amax_h_own, h64 = grouped_gemm(a_codes, a_scales, gs_x, experts, "w13", rt, "silu_mul",
                                      return_unrounded=True)
    if amax_h is None:
        amax_h = amax_h_own
    hq_codes, hq_scales, gs_h, _ = quantize(h.astype(np.float32), amax=amax_h)
    hq_codes[~valid] = 0
    hq_scales[~valid] = 0
    y = grouped_gemm(hq_codes, hq_scales, gs_h, experts, "w2", rt, "f32")
    out64 = combine(y, topk_weights, rt.slot_dst, round_bf16=False)
    out = bf16_round(out64)
    if return_intermediates:
        return out, dict(routing=rt, out_f64=out64, h_f64=h64, gs_x=gs_x, amax_x=amax_x, xq_codes=xq_codes,
                         xq_scales=xq_scales, a_codes=a_codes, a_scales=a_scales,
                         h=h, amax_h=np.float32(amax_h), amax_h_own=amax_h_own, gs_h=gs_h,
                         hq_codes=hq_codes,
                         hq_scales=hq_scales, y=y)
    return out


def forward_with_shared(x, topk_ids, topk_weights, experts, shared, pad: int = 1):
    """The MoE layer with a shared expert, the shared part computed densely.

    out[t] = bf16( sum_j w[t, j] * y[row(t, j)] + y_s[t] ), with y_s the
    shared expert's SiLU-gated MLP applied to every token.  The pages name
    shared experts ("What's Been Verified", row "E2E 61-layer (shared
    experts)") without detail; the reading taken: the shared expert has its
    own NVFP4 weights (``shared``: the dict of one expert), sees the same
    NVFP4 activations x as the routed experts, and its h is requantised
    together with theirs (one global scale over every valid row of the
    intermediate, routed and shared); its term is added last.  Returns
    (out, out_f64).
    """
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    E = experts.num_experts
    I = experts.I
    rt = route(ids, E, pad)
    R_pad = int(rt.padded_offsets[-1])
    d = x.shape[1]
    xq_codes, xq_scales, gs_x, _ = quantize(x)
    a_codes = np.zeros((R_pad, d // 2), dtype=np.uint8)
    a_scales = np.zeros((R_pad, d // 16), dtype=np.uint8)
    valid = rt.row_src >= 0
    a_codes[valid] = xq_codes[rt.row_src[valid] // k]
    a_scales[valid] = xq_scales[rt.row_src[valid] // k]
    h, amax_r = grouped_gemm(a_codes, a_scales, gs_x, experts, "w13", rt, "silu_mul")
    # the shared expert over all tokens, as plain matrix products
    xhat = dequantize(xq_codes, xq_scales, gs_x)
    gate = dequantize(shared["w13_codes"][:I], shared["w13_scales"][:I], shared["w13_gs"][0])
    up = dequantize(shared["w13_codes"][I:], shared["w13_scales"][I:], shared["w13_gs"][1])
    h_s = bf16_round(silu(xhat @ gate.T) * (xhat @ up.T))
    amax_h = np.float32(max(float(amax_r), float(np.max(np.abs(h_s))) if T else 0.0))
    hq_codes, hq_scales, gs_h, _ = quantize(h.astype(np.float32), amax=amax_h)
    hq_codes[~valid] = 0
    hq_scales[~valid] = 0
    y = grouped_gemm(hq_codes, hq_scales, gs_h, experts, "w2", rt, "f32")
    hs_codes, hs_scales, _, _ = quantize(h_s.astype(np.float32), amax=amax_h)
    w2_gs = np.float32(np.asarray(shared["w2_gs"]).reshape(-1)[0])
    y_s = dequantize(hs_codes, hs_scales, gs_h) @ dequantize(
        shared["w2_codes"], shared["w2_scales"], w2_gs).T
    out64 = combine(y, topk_weights, rt.slot_dst, round_bf16=False) + y_s
    return bf16_round(out64), out64


def forward_unquantized(x, topk_ids, topk_weights, experts):
    """The same MoE with no activation quantisation and no bf16 rounding.

    Weights are the dequantised NVFP4 weights (exact); x and h stay float64.
    Used only as the high-precision comparison point for the accuracy pin.
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids)
    w = np.asarray(topk_weights, dtype=np.float64)
    T, k = ids.shape
    out = np.zeros_like(x)
    cache = {}
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            if e not in cache:
                ew = experts[e]
                I = ew["w13_codes"].shape[0] // 2
                cache[e] = (
                    dequantize(ew["w13_codes"][:I], ew["w13_scales"][:I], ew["w13_gs"][0]),
                    dequantize(ew["w13_codes"][I:], ew["w13_scales"][I:], ew["w13_gs"][1]),
                    dequantize(ew["w2_codes"], ew["w2_scales"], ew["w2_gs"]),
                )
            g_w, u_w, d_w = cache[e]
            hv = silu(g_w @ x[t]) * (u_w @ x[t])
            out[t] += w[t, j] * (d_w @ hv)
    return out
