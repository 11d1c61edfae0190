// Pieces shared by the grouped-GEMM kernels (internal to the library): the
// launch arguments, the token tile's tensor maps, and the persistent tile
// schedule over the experts.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace megamoe {

constexpr int kGemmThreads = 448;
constexpr int kSfWarp0 = 6;    // warps 6..9 write block scales into TMEM
constexpr int kEpiWarp1 = 10;  // warps 2..5 and 10..13 drain the accumulators
constexpr int kEpiWarps = 8;

struct GemmArgs {
  const uint8_t* w_codes;  // packed, pre-swizzled 16 KB blocks (megamoe_pack_weight_codes)
  const uint8_t* w_sf;  // atom layout [E*N/128][K/64][512]
  const float* w_gs;    // [E][G]
  const float* a_gs;    // device scalar
  const int32_t* offsets;
  const int32_t* padded_offsets;
  void* out;
  int64_t ld_out;
  float* out_amax;
  uint32_t* status;
  uint64_t wait_limit_ns;  // bound of every pipeline wait (unwinding waits use 4 s)
  int E, N, K;
  // 1: the routing offsets were complete before the preceding kernel started
  // (the forward's order), so the tile schedule is built and the first weight
  // stages are prefetched into L2 while that kernel still runs
  int early_weights;
  // split-K (kernels instantiated with kEpiPartial*): each tile's K range is
  // cut into ksplit pieces; piece ks of a tile writes acc * alpha as fp32 to
  // plane ks of `partial` ([ksplit][offsets[E]][N], rows unpadded:
  // row - padded_offsets[e] + offsets[e]); k_splitk_finish sums the planes
  int ksplit;
  float* partial;
  int64_t partial_plane;  // elements per plane
};

// Tensor maps of the token tile: codes (128-byte swizzle) and row-major
// block scales, boxes of the tile's token rows.
struct TokenMaps {
  CUtensorMap codes;
  CUtensorMap scales;
};

// Token-major tiles (tokens on the MMA's M side, 256 weight rows on N).
cudaError_t launch_grouped_gemm_tm(const TokenMaps& maps, const GemmArgs& a, int epilogue,
                                   cudaStream_t stream);

// Internal epilogue codes of the split-K kernels (G = 1 and G = 2 operands).
constexpr int kEpiPartial1 = 16;
constexpr int kEpiPartial2 = 17;

struct TileInfo {
  int e, mt, nt, ntiles;  // expert, feature tile, token tile, token tiles of e
};

// Tile -> (expert, feature tile, token tile) from the tile prefix s_toff alone;
// the expert is searched in [lo, E - 1] (a CTA's tiles never go back in e).
__device__ __forceinline__ TileInfo decode_tile(int tile, const int* s_toff, int E, int MT,
                                                int lo = 0) {
  int hi = E - 1;
  while (lo < hi) {  // largest e with s_toff[e] <= tile; it always owns tiles
    const int mid = (lo + hi + 1) >> 1;
    if (s_toff[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo t;
  t.e = lo;
  t.ntiles = (s_toff[lo + 1] - s_toff[lo]) / MT;
  const int local = tile - s_toff[lo];
  t.mt = local / t.ntiles;
  t.nt = local - t.mt * t.ntiles;
  return t;
}

// s_toff[e] = first tile of expert e, s_toff[E] = total tiles.  All threads.
template <int BN>
__device__ void build_tile_offsets(const int32_t* offsets, int E, int MT, int* s_toff,
                                   int* s_scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + kGemmThreads - 1) / kGemmThreads;
  const int e0 = tid * per, e1 = min(E, e0 + per);
  int sum = 0;
  for (int e = e0; e < e1; ++e) {
    const int cnt = __ldcg(offsets + e + 1) - __ldcg(offsets + e);
    const int t = cnt > 0 ? (cnt + BN - 1) / BN * MT : 0;
    s_toff[e] = t;
    sum += t;
  }
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_scan[warp] = x;
  __syncthreads();
  int base = x - sum;
  for (int w = 0; w < warp; ++w) base += s_scan[w];
  for (int e = e0; e < e1; ++e) {
    const int t = s_toff[e];
    s_toff[e] = base;
    base += t;
  }
  if (tid == kGemmThreads - 1) s_toff[E] = base;
  __syncthreads();
}

// Waits that ignore the abort flag (used only while unwinding).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitTimeoutNs) break;
  }
}

}  // namespace megamoe
