// Top-k weighted combine: out[t] = bf16( sum_j w[t, j] * y[slot_dst[t*k + j]] )
// (the topk_weights input of "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4",
// "Test Plan -- Finding the NaN", Phase 1).  One thread per 4 consecutive
// features of one token: 128-bit loads of each routed row of y, fp32 sums in
// ascending j, one bf16 rounding, 64-bit stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace megamoe {

__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ y, int64_t ld_y,
                                                 const int32_t* __restrict__ slot_dst,
                                                 const float* __restrict__ w, int T, int k, int d,
                                                 uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int vecs = d / 4;
  const int64_t total = static_cast<int64_t>(T) * vecs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / vecs);
    const int v = static_cast<int>(i - static_cast<int64_t>(t) * vecs);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int r = __ldg(slot_dst + static_cast<int64_t>(t) * k + j);
      if (r < 0) continue;
      const float wt = __ldg(w + static_cast<int64_t>(t) * k + j);
      const float4 yv = __ldg(reinterpret_cast<const float4*>(y + r * ld_y) + v);
      acc.x = fmaf(wt, yv.x, acc.x);
      acc.y = fmaf(wt, yv.y, acc.y);
      acc.z = fmaf(wt, yv.z, acc.z);
      acc.w = fmaf(wt, yv.w, acc.w);
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * d)[v] = pk;
  }
}

cudaError_t launch_combine(const float* y, int64_t ld_y, const int32_t* slot_dst, const float* w,
                           int T, int k, int d, uint16_t* out, cudaStream_t stream) {
  const int64_t tasks = static_cast<int64_t>(T) * (d / 4);
  if (tasks == 0) return cudaSuccess;
  int64_t blocks = (tasks + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  return launch_pdl(k_combine, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, y, ld_y,
                    slot_dst, w, T, k, d, out);
}

}  // namespace megamoe
