// Host-side launchers of the MegaMoE kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace megamoe {

size_t route_smem_bytes(int E);
cudaError_t launch_route(const int32_t* ids, int n_slots, int E, int pad, int32_t* counts,
                         int32_t* offsets, int32_t* padded_offsets, int32_t* row_src,
                         int64_t row_capacity, int32_t* slot_dst, uint32_t* status,
                         cudaStream_t stream);

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int K, int64_t ld, float* amax,
                        uint32_t* status, cudaStream_t stream);
cudaError_t launch_quant(const uint16_t* x, int64_t rows_in, int K, int64_t ld,
                         const int32_t* slot_dst, int k, const int32_t* row_src,
                         const int32_t* live_rows, int64_t out_rows, const float* amax,
                         float* gs_out, uint8_t* codes, uint8_t* scales, int scale_layout,
                         cudaStream_t stream);
cudaError_t launch_swizzle(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                           cudaStream_t stream);

cudaError_t launch_pack(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                        cudaStream_t stream);

struct GemmLaunch {
  const uint8_t* act_codes;
  const uint8_t* act_scales;  // atom layout
  const float* act_gs;
  int64_t act_rows;
  const uint8_t* w_codes;   // tile-major (k_pack)
  const uint8_t* w_scales;  // atom layout
  const float* w_gs;
  int E, N, K;
  const int32_t* offsets;
  const int32_t* padded_offsets;
  int epilogue;
  void* out;
  int64_t ld_out;
  float* out_amax;
  int tile_n;
  uint32_t* status;
};
// Encodes the tensor maps and launches the persistent grouped GEMM.
cudaError_t launch_grouped_gemm(const GemmLaunch& g, cudaStream_t stream);
int pick_tile_n(double expected_tokens_per_expert);

cudaError_t launch_combine(const float* y, int64_t ld_y, const int32_t* slot_dst,
                           const float* w, int T, int k, int d, uint16_t* out,
                           cudaStream_t stream);

}  // namespace megamoe
