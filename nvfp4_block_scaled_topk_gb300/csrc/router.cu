// Router top-k and softmax ahead of the routing ("CURRENT_BUG.md -- DeepSeek-V4
// Blackwell NVFP4", "Architecture: DeepSeek-V4 MegaMoE": 384 experts, top-6;
// "Test Plan -- Finding the NaN", Phase 1 item 1: topk_ids and topk_weights
// come from the router).
//
// One warp per token.  Lane l holds the scores of experts l, l + 32, ...
// (score = logit + bias[e], an fp32 add).  k rounds of a warp argmax pick the
// experts in descending score, ties to the lower expert index; the weights are
// the softmax of the selected (unbiased) logits in fp32.  An optional shared
// expert is appended as one more column with weight 1.
#include <cuda_runtime.h>

#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace megamoe {

constexpr int kRouterWarps = 8;

template <int PER>
__global__ void __launch_bounds__(kRouterWarps * 32)
    k_router(const float* __restrict__ logits, int64_t T, int E, int64_t ld,
             const float* __restrict__ bias, int k, int shared, int32_t* __restrict__ ids,
             float* __restrict__ weights) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouterWarps + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform
  const int k_out = k + (shared >= 0 ? 1 : 0);
  float sc[PER], lg[PER];
  uint32_t live = 0;  // bit i: expert lane + 32 i exists and is not taken yet
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    lg[i] = 0.f;
    sc[i] = -FLT_MAX;
    if (e < E) {
      lg[i] = __ldg(logits + t * ld + e);
      sc[i] = bias ? __fadd_rn(lg[i], __ldg(bias + e)) : lg[i];
      live |= 1u << i;
    }
  }
  int my_id = -1;      // lane j < k: the j-th selected expert
  float my_logit = 0.f;
  for (int j = 0; j < k; ++j) {
    // this lane's best live expert (experts ascend with i, so strict > keeps
    // the lower index on ties)
    float bv = 0.f, bl = 0.f;
    int be = -1;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (((live >> i) & 1u) && (be < 0 || sc[i] > bv)) {
        bv = sc[i];
        bl = lg[i];
        be = lane + 32 * i;
      }
    }
    // warp argmax: higher score first, then the lower expert index
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const bool take = oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be));
      if (take) {
        bv = ov;
        bl = ol;
        be = oe;
      }
    }
    if (be < 0) break;  // fewer than k experts (k > E is refused on the host)
    if ((be & 31) == lane) live &= ~(1u << (be >> 5));
    if (lane == j) {
      my_id = be;
      my_logit = bl;
    }
  }
  // softmax of the selected logits
  float m = lane < k ? my_logit : -FLT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ex = lane < k ? expf(my_logit - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    ids[t * k_out + lane] = my_id;
    weights[t * k_out + lane] = ex / sum;
  } else if (lane == k && shared >= 0) {
    ids[t * k_out + lane] = shared;
    weights[t * k_out + lane] = 1.f;
  }
}

cudaError_t launch_router(const float* logits, int64_t T, int E, int64_t ld, const float* bias,
                          int k, int shared, int32_t* ids, float* weights, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((T + kRouterWarps - 1) / kRouterWarps));
  const dim3 block(kRouterWarps * 32);
  const int per = (E + 31) / 32;
#define MEGAMOE_ROUTER_CASE(P)                                                                  \
  if (per <= P)                                                                               \
    return launch_pdl(k_router<P>, grid, block, 0, stream, logits, T, E, ld, bias, k, shared, \
                      ids, weights);
  MEGAMOE_ROUTER_CASE(4)
  MEGAMOE_ROUTER_CASE(8)
  MEGAMOE_ROUTER_CASE(12)
  MEGAMOE_ROUTER_CASE(16)
  MEGAMOE_ROUTER_CASE(32)
#undef MEGAMOE_ROUTER_CASE
  return cudaErrorInvalidValue;
}

}  // namespace megamoe
