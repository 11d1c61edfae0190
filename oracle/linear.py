"""Dense NVFP4 linear layer of the oracle (test infrastructure only).

Follows "Current Bug: vLLM produces NaN from layer 0" (blame @2fc81cc):
  * "Root Cause": the attention projections are NVFP4 linear layers whose
    activations are quantised to NVFP4 with a global scale, and the stored
    checkpoint input_scale used as that scale overflows;
  * "Key evidence": input_scale 0.00025141 (q_a) gives a multiplier of
    3977.6 for activations of amax about 2-8;
  * "What we've tried", item 1: taking the global scale from the measured
    amax instead.
and "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", table "What's Been
Verified" (NVFP4 linear projections q_a, kv, q_b, o_b).

The layer is the one-group case of the MoE's grouped GEMM:
    out[t, n] = sum_k xhat[t, k] * what[n, k]
with xhat = dequant(quantize(x)) (gs_x from the measured amax of x, or from
a given amax) and what the dequantised weight, in float64, then rounded once
to bf16 (or returned unrounded).
"""

from __future__ import annotations

import numpy as np

from .nvfp4 import bf16_round, dequantize, quantize


def linear(x, w_codes, w_scales, w_gs, amax=None, round_bf16=True):
    """NVFP4 linear: returns (out [T, N] float64, dict of intermediates).

    ``x`` is [T, K] (bf16 values as float32); ``w_codes`` [N, K/2],
    ``w_scales`` [N, K/16] E4M3 bytes, ``w_gs`` the weight's global scale.
    ``amax`` (optional) replaces the measured max|x| in the activation global
    scale gs_x = 2688 / amax -- the way a stored input_scale enters
    (amax = 2688 * input_scale).
    """
    x = np.asarray(x, dtype=np.float32)
    codes, scales, gs_x, amax_x = quantize(x, amax=amax)
    xhat = dequantize(codes, scales, gs_x)
    what = dequantize(w_codes, w_scales, np.float32(w_gs))
    out = xhat @ what.T
    inter = dict(x_codes=codes, x_scales=scales, gs_x=gs_x, amax_x=amax_x, out_f64=out)
    return (bf16_round(out) if round_bf16 else out), inter
