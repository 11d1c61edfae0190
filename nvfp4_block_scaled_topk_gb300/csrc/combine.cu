// Top-k weighted combine: out[t] = bf16( sum_j w[t, j] * y[slot_dst[t*k + j]] )
// (the topk_weights input of "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4",
// "Test Plan -- Finding the NaN", Phase 1).  One thread per 4 consecutive
// features of one token: 128-bit loads of each routed row of y (up to eight
// slots' loads in flight at once), fp32 sums in ascending j, one bf16
// rounding, 64-bit stores.  An expert-parallel shard writes the fp32 sum of
// its own slots instead, and the shards' sums are added and rounded once
// after the exchange (k_round_bf16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace megamoe {

template <bool F32_OUT>
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ y, int64_t ld_y,
                                                 const int32_t* __restrict__ slot_dst,
                                                 const float* __restrict__ w, int T, int k, int d,
                                                 void* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int vecs = d / 4;
  const int64_t total = static_cast<int64_t>(T) * vecs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = (i >> 32) == 0 ? static_cast<int>(static_cast<uint32_t>(i) / static_cast<uint32_t>(vecs))
                                 : static_cast<int>(i / vecs);
    const int v = static_cast<int>(i - static_cast<int64_t>(t) * vecs);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // eight slots at a time: all their row indices and weights, then all
    // their rows of y, are in flight together; the sums stay in ascending j
    for (int j0 = 0; j0 < k; j0 += 8) {
      int r[8];
      float wt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        r[j] = j0 + j < k ? __ldg(slot_dst + static_cast<int64_t>(t) * k + j0 + j) : -1;
        wt[j] = j0 + j < k ? __ldg(w + static_cast<int64_t>(t) * k + j0 + j) : 0.f;
      }
      float4 yv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        yv[j] = r[j] >= 0 ? __ldg(reinterpret_cast<const float4*>(y + r[j] * ld_y) + v)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (r[j] < 0) continue;
        acc.x = fmaf(wt[j], yv[j].x, acc.x);
        acc.y = fmaf(wt[j], yv[j].y, acc.y);
        acc.z = fmaf(wt[j], yv[j].z, acc.z);
        acc.w = fmaf(wt[j], yv[j].w, acc.w);
      }
    }
    if (F32_OUT) {  // the sum before its rounding (one shard's share of the output)
      float* o = static_cast<float*>(out) + static_cast<int64_t>(t) * d + 4 * v;
      __stcs(reinterpret_cast<float4*>(o), acc);
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + static_cast<int64_t>(t) * d)[v] = pk;
    }
  }
}

// out[i] = bf16_rne(in[i]): four elements per thread, grid-stride.
__global__ void __launch_bounds__(256) k_round_bf16(const float4* __restrict__ in, int64_t n4,
                                                    uint2* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(in + i);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    out[i] = pk;
  }
}

// Up to 16 resident blocks of 256 threads per SM, grid-stride beyond that.
static unsigned stream_blocks(int64_t tasks) {
  int64_t blocks = (tasks + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<unsigned>(blocks > cap ? cap : blocks);
}

cudaError_t launch_combine(const float* y, int64_t ld_y, const int32_t* slot_dst, const float* w,
                           int T, int k, int d, void* out, bool out_f32, cudaStream_t stream) {
  const int64_t tasks = static_cast<int64_t>(T) * (d / 4);
  if (tasks == 0) return cudaSuccess;
  const dim3 grid(stream_blocks(tasks));
  if (out_f32)
    return launch_pdl(k_combine<true>, grid, dim3(256), 0, stream, y, ld_y, slot_dst, w, T, k, d,
                      out);
  return launch_pdl(k_combine<false>, grid, dim3(256), 0, stream, y, ld_y, slot_dst, w, T, k, d,
                    out);
}

cudaError_t launch_round_bf16(const float* in, int64_t n, uint16_t* out, cudaStream_t stream) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  return launch_pdl(k_round_bf16, dim3(stream_blocks(n4)), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(in), n4, reinterpret_cast<uint2*>(out));
}

}  // namespace megamoe
