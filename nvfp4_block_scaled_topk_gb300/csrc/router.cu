// Router top-k and softmax ahead of the routing ("CURRENT_BUG.md -- DeepSeek-V4
// Blackwell NVFP4", "Architecture: DeepSeek-V4 MegaMoE": 384 experts, top-6;
// "Test Plan -- Finding the NaN", Phase 1 item 1: topk_ids and topk_weights
// come from the router).
//
// One warp per token (router_token in router.cuh): the token's scores
// (logit + bias[e], an fp32 add) are staged in shared memory and k rounds of
// a warp argmax pick the experts in descending score, ties to the lower
// expert index; the weights are the softmax of the selected (unbiased) logits
// in fp32.  An optional shared expert is appended as one more column with
// weight 1.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "router.cuh"

namespace megamoe {

constexpr int kRouterWarps = 8;

__global__ void __launch_bounds__(kRouterWarps * 32)
    k_router(const float* __restrict__ logits, int64_t T, int E, int64_t ld,
             const float* __restrict__ bias, int k, int shared, int32_t* __restrict__ ids,
             float* __restrict__ weights) {
  extern __shared__ float s_rows[];  // [kRouterWarps][E]
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouterWarps + warp;
  if (t >= T) return;  // warp-uniform
  const int k_out = k + (shared >= 0 ? 1 : 0);
  router_token(logits + t * ld, bias, E, k, shared, s_rows + warp * E, ids + t * k_out,
               weights + t * k_out, lane);
}

cudaError_t launch_router(const float* logits, int64_t T, int E, int64_t ld, const float* bias,
                          int k, int shared, int32_t* ids, float* weights, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((T + kRouterWarps - 1) / kRouterWarps));
  const dim3 block(kRouterWarps * 32);
  const size_t smem = sizeof(float) * kRouterWarps * E;
  cudaError_t err = cudaFuncSetAttribute(k_router, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(k_router, grid, block, smem, stream, logits, T, E, ld, bias, k, shared, ids,
                    weights);
}

}  // namespace megamoe
