"""CPU oracle for the NVFP4 MegaMoE routed-expert forward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never imports,
links or executes anything in this package, and this package imports nothing
from the product path.  The two share no code: this package restates the
method from the source pages in plain NumPy so that a reader can check it
against them by eye.

Sources (titles and sections of the pages this follows):

* "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4" (nvfp4-megamoe-kernel, src
  @2e65594):
    - section "Architecture: DeepSeek-V4 MegaMoE": 384 experts, top-6 routing,
      grouped GEMM with one problem per expert;
    - table "What's Been Verified": the MoE is an L1 gate+up GEMM followed by
      an L2 down GEMM;
    - section "Test Plan -- Finding the NaN", Phase 1: the runner takes
      hidden_states, topk_ids, topk_weights and variable per-expert token
      counts padded to 128 rows; L1 GEMM -> SiLU activation -> L2 GEMM;
      activations are quantised to NVFP4 before the grouped GEMM;
    - same section, Phase 2: zero-token experts, expert_offsets and
      padded_expert_offsets.
* "Current Bug: vLLM produces NaN from layer 0" (blame @2fc81cc):
    - "What we've tried", item 1: the MoE works when the activation global
      scale comes from a warm-up (measured amax);
    - "Root Cause" and "Key evidence": a stored checkpoint input_scale used as
      the activation global scale overflows, so it is never used here.

The pages never define NVFP4 arithmetic.  The oracle takes the plain
two-level reading (E2M1 element codes, one E4M3 scale per 16 elements, one
FP32 global scale per tensor) with the OCP Microscaling v1.0 bit formats for
E2M1 and E4M3.  Every reading the pages leave open is stated at the function
that takes it.

Precision: the GEMMs, SiLU and combine run in float64 on dequantised
operands.  The quantiser's decisions (scale byte, element code) are taken in
IEEE float32 with one correctly rounded operation per step, in a fixed order,
because those decisions are integers that both sides must reach from the
same values.

Parity status: every public function here is pinned by a CPU test in
``tests/test_oracle_*.py`` (hand tables, exhaustive brute force, closed forms,
invariants, library cross-checks).  No function is "parity unpinned".
"""

from .nvfp4 import (  # noqa: F401
    E2M1_GRID,
    GLOBAL_SCALE_NUMERATOR,
    bf16_round,
    dequantize,
    e2m1_decode,
    e2m1_encode,
    e4m3_decode,
    e4m3_encode,
    pack_nibbles,
    quantize,
    swizzle_scales,
    unpack_nibbles,
    unswizzle_scales,
)
from .linear import linear  # noqa: F401
from .router import router_topk  # noqa: F401
from .moe import (  # noqa: F401
    Routing,
    combine,
    forward,
    forward_unquantized,
    forward_with_shared,
    grouped_gemm,
    route,
    silu,
)
