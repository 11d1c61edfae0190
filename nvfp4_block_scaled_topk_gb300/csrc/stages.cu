// Debug scan of a finished forward's stage outputs for non-finite values
// ("CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Test Plan -- Finding the
// NaN", Phase 1 item 3: check the activations after the L1 GEMM and SiLU and
// after the L2 GEMM, stage by stage, to find where a NaN first appears).
//
// One grid-stride pass per stage over the valid rows only (padding rows are
// never written by the forward and may hold anything):
//   block scales of the quantised x and of the requantised h: an E4M3 byte
//   with all exponent and mantissa bits set (0x7F / 0xFF) is NaN;
//   h (bf16): an all-ones exponent is Inf or NaN;
//   y (BFP16): a group exponent of 127 marks a group holding Inf or NaN
//   (a 16-row group holds valid rows when its first row does: an expert's
//   valid rows come first in its padded range, and pads are multiples of 32);
//   the output (bf16), every row.
// Each stage found sets its bit in *flags with an atomicOr; flags are cleared
// by the launcher first.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace megamoe {

struct StageScan {
  const int32_t* row_src;         // [R]: -1 for padding rows
  const int32_t* padded_total;    // device scalar: R
  const uint8_t* xq_sf;           // [rows, d/16]
  const uint16_t* h;              // [rows, I]
  const uint8_t* hq_sf;           // [rows, I/16]
  const int8_t* y_exp;           // exponents of the BFP16 y [rows/16, d/8]
  const uint16_t* out;            // [T, d]
  int T, d, I;
  uint32_t* flags;
};

__global__ void __launch_bounds__(256) k_stage_scan(const StageScan a) {
  pdl_wait();
  pdl_trigger();
  const int64_t R = *a.padded_total;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  uint32_t found = 0;
  // 16-byte words per row of each region
  const int w_xs = a.d / 16 / 16, w_h = a.I * 2 / 16, w_hs = a.I / 16 / 16;
  const int per_row = w_xs + w_h + w_hs;
  for (int64_t i = tid; i < R * per_row; i += stride) {
    const int64_t row = i / per_row;
    int c = static_cast<int>(i - row * per_row);
    if (__ldg(a.row_src + row) < 0) continue;
    uint4 v;
    uint32_t bit;
    if (c < w_xs) {
      v = __ldg(reinterpret_cast<const uint4*>(a.xq_sf + row * (a.d / 16)) + c);
      bit = MEGAMOE_STAGE_XQ_SCALE;
      const uint32_t m[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4; ++j)
        for (int b = 0; b < 4; ++b)
          if (((m[j] >> (8 * b)) & 0x7Fu) == 0x7Fu) found |= bit;
      continue;
    }
    c -= w_xs;
    if (c < w_h) {
      v = __ldg(reinterpret_cast<const uint4*>(a.h + row * a.I) + c);
      const uint32_t m[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4; ++j)
        if ((m[j] & 0x7F80u) == 0x7F80u || (m[j] & 0x7F800000u) == 0x7F800000u)
          found |= MEGAMOE_STAGE_H;
      continue;
    }
    c -= w_h;
    if (c < w_hs) {
      v = __ldg(reinterpret_cast<const uint4*>(a.hq_sf + row * (a.I / 16)) + c);
      const uint32_t m[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4; ++j)
        for (int b = 0; b < 4; ++b)
          if (((m[j] >> (8 * b)) & 0x7Fu) == 0x7Fu) found |= MEGAMOE_STAGE_HQ_SCALE;
      continue;
    }
  }
  const int w_y = a.d / 128;  // 16-byte words of exponents per 16-row group (d/8 bytes)
  for (int64_t i = tid; i < (R / 16) * w_y; i += stride) {
    const int64_t grp = i / w_y;
    if (__ldg(a.row_src + 16 * grp) < 0) continue;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.y_exp + grp * (a.d / 8)) + (i - grp * w_y));
    const uint32_t m[4] = {v.x, v.y, v.z, v.w};
    for (int j = 0; j < 4; ++j)
      for (int b = 0; b < 4; ++b)
        if (((m[j] >> (8 * b)) & 0xFFu) == static_cast<uint32_t>(kBfp16NonFinite))
          found |= MEGAMOE_STAGE_Y;
  }
  const int64_t w_out = static_cast<int64_t>(a.T) * a.d * 2 / 16;
  for (int64_t i = tid; i < w_out; i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.out) + i);
    const uint32_t m[4] = {v.x, v.y, v.z, v.w};
    for (int j = 0; j < 4; ++j)
      if ((m[j] & 0x7F80u) == 0x7F80u || (m[j] & 0x7F800000u) == 0x7F800000u)
        found |= MEGAMOE_STAGE_OUT;
  }
  found = __reduce_or_sync(0xffffffffu, found);
  if ((threadIdx.x & 31) == 0 && found) atomicOr(a.flags, found);
}

cudaError_t launch_stage_scan(const int32_t* row_src, const int32_t* padded_total,
                              const uint8_t* xq_sf, const uint16_t* h, const uint8_t* hq_sf,
                              const int8_t* y_exp, const uint16_t* out, int T, int d, int I,
                              uint32_t* flags, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  StageScan a{row_src, padded_total, xq_sf, h, hq_sf, y_exp, out, T, d, I, flags};
  return launch_pdl(k_stage_scan, dim3(num_sms() * 8), dim3(256), 0, stream, a);
}

}  // namespace megamoe
