// Top-k weighted combine: out[t] = bf16( sum_j w[t, j] * y[slot_dst[t*k + j]] )
// (the topk_weights input of "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4",
// "Test Plan -- Finding the NaN", Phase 1).  One thread per 4 consecutive
// features of one token: 128-bit loads of each routed row of y (up to eight
// slots' loads in flight at once), fp32 sums in ascending j, one bf16
// rounding, 64-bit stores.  y is fp32 (megamoe_combine), or (the forward)
// BFP16, then one thread per 8 features (k_combine_bfp16).  An expert-parallel
// shard writes the fp32 sum of its own slots instead, and the shards' sums
// are added and rounded once after the exchange (k_round_bf16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace megamoe {

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
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + static_cast<int64_t>(t) * d)[v] = pk;
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

// The combine over a BFP16 y: one thread per 8 consecutive features of one
// token, which are one exponent group of each routed row.  Per slot one
// 16-byte load of values and one exponent byte, up to eight slots in flight;
// the slot's power of two is folded into its weight (w * 2^s is exact), so
// each element costs a byte permute, an exact subtraction and one fused
// multiply-add into the fp32 sum (the same sum as decoding first), in
// ascending j; one bf16 rounding, two 8-byte stores (or the fp32 sum of a
// shard's slots).
template <bool F32_OUT>
__global__ void __launch_bounds__(256) k_combine_bfp16(const uint16_t* __restrict__ y,
                                                       const int8_t* __restrict__ y_exp,
                                                       int64_t ld_y, int64_t y_rows,
                                                       const int32_t* __restrict__ slot_dst,
                                                       const float* __restrict__ w, int T, int k,
                                                       int d, void* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int vecs = d / 8;
  const int64_t total = static_cast<int64_t>(T) * vecs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = (i >> 32) == 0 ? static_cast<int>(static_cast<uint32_t>(i) / static_cast<uint32_t>(vecs))
                                 : static_cast<int>(i / vecs);
    const int v = static_cast<int>(i - static_cast<int64_t>(t) * vecs);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      int r[8];
      float wt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        r[j] = j0 + j < k ? __ldg(slot_dst + static_cast<int64_t>(t) * k + j0 + j) : -1;
        if (r[j] >= y_rows) r[j] = -1;  // outside y: skipped like a -1 slot
        wt[j] = j0 + j < k ? __ldg(w + static_cast<int64_t>(t) * k + j0 + j) : 0.f;
      }
      uint4 qv[8];
      int sv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (r[j] >= 0) {
          qv[j] = __ldg(reinterpret_cast<const uint4*>(y + r[j] * ld_y) + v);
          sv[j] = __ldg(y_exp + (r[j] >> 4) * (ld_y / 8) + v);
        } else {
          qv[j] = make_uint4(0u, 0u, 0u, 0u);
          sv[j] = 0;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (r[j] < 0) continue;
        const uint32_t qw[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
        if (sv[j] == kBfp16NonFinite) {  // a group holding Inf or NaN: fp16 values
#pragma unroll
          for (int e = 0; e < 8; ++e)
            acc[e] = fmaf(wt[j], bfp16_decode(qw[e >> 1], e & 1, sv[j]), acc[e]);
          continue;
        }
        const float wp = wt[j] * bfp16_pow2(sv[j]);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wp, bfp16_offset_value(qw[e >> 1], e & 1), acc[e]);
      }
    }
    if (F32_OUT) {  // the sum before its rounding (one shard's share of the output)
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<int64_t>(t) * d + 8 * v);
      __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
      __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
    } else {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
        pk[e] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      uint2* o = reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + static_cast<int64_t>(t) * d + 8 * v);
      o[0] = make_uint2(pk[0], pk[1]);
      o[1] = make_uint2(pk[2], pk[3]);
    }
  }
}

// Up to 16 resident blocks of 256 threads per SM, grid-stride beyond that.
static unsigned stream_blocks(int64_t tasks) {
  int64_t blocks = (tasks + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<unsigned>(blocks > cap ? cap : blocks);
}

cudaError_t launch_combine(const void* y, const int8_t* y_exp, int64_t ld_y, int64_t y_rows,
                           const int32_t* slot_dst, const float* w, int T, int k, int d,
                           void* out, bool out_f32, cudaStream_t stream) {
  if (y_exp) {
    const int64_t tasks = static_cast<int64_t>(T) * (d / 8);
    if (tasks == 0) return cudaSuccess;
    const dim3 grid(stream_blocks(tasks));
    const uint16_t* yq = static_cast<const uint16_t*>(y);
    if (out_f32)
      return launch_pdl(k_combine_bfp16<true>, grid, dim3(256), 0, stream, yq, y_exp, ld_y,
                        y_rows, slot_dst, w, T, k, d, out);
    return launch_pdl(k_combine_bfp16<false>, grid, dim3(256), 0, stream, yq, y_exp, ld_y,
                      y_rows, slot_dst, w, T, k, d, out);
  }
  // an fp32 y (megamoe_combine) always gives the bf16 output
  if (out_f32) return cudaErrorInvalidValue;
  const int64_t tasks = static_cast<int64_t>(T) * (d / 4);
  if (tasks == 0) return cudaSuccess;
  const dim3 grid(stream_blocks(tasks));
  return launch_pdl(k_combine, grid, dim3(256), 0, stream, static_cast<const float*>(y), ld_y,
                    slot_dst, w, T, k, d, out);
}

cudaError_t launch_round_bf16(const float* in, int64_t n, uint16_t* out, cudaStream_t stream) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  return launch_pdl(k_round_bf16, dim3(stream_blocks(n4)), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(in), n4, reinterpret_cast<uint2*>(out));
}

}  // namespace megamoe
