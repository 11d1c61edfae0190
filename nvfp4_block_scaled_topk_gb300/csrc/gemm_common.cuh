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
  // Requantisation of h fused into the SiLU*up kernel (null: not fused).
  // After its last tile every CTA with tiles adds one to *rq_arrivals (zeroed
  // before the launch) and waits, bounded, until all of them have; then each
  // encodes the h rows of its own tiles with gs = 2688 / amax(h) into
  // rq_codes [rows, N/4] and row-major rq_scales [rows, N/32], and CTA 0
  // stores gs in *rq_gs.
  uint32_t* rq_arrivals;
  uint8_t* rq_codes;
  uint8_t* rq_scales;
  float* rq_gs;
  // MEGAMOE_EPI_BFP16: the int8 exponents [rows / 16, ld_out / 8] after the
  // uint16 values at `out`
  int8_t* out_exp;
};

// Tensor maps of the token tile: codes (128-byte swizzle) and row-major
// block scales, boxes of the tile's token rows.  Token-major launches also
// carry 32- and 64-row boxes over the same matrices: an expert's last tile
// that holds at most 32 (64) valid rows loads only those.
struct TokenMaps {
  CUtensorMap codes;
  CUtensorMap scales;
  CUtensorMap codes32, scales32, codes64, scales64;
};

// Rows of the token box for a 128-row tile with `rows` valid rows.
__device__ __forceinline__ int short_box_rows(int rows) {
  return rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
}

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

// Grid-wide arrival of this CTA (thread 0 only), then a bounded wait until
// `expected` CTAs have arrived.  The fence before the arrival publishes this
// CTA's earlier writes (ordered before by the caller's __syncthreads); the
// acquire load and the fence after it make every arrived CTA's writes
// visible.  False (with MEGAMOE_DEV_TIMEOUT set) if the wait ran out.
__device__ __forceinline__ bool grid_arrive_and_wait(uint32_t* arrivals, uint32_t expected,
                                                     uint32_t* status, uint64_t limit_ns) {
  __threadfence();
  atomicAdd(arrivals, 1u);
  const uint64_t t0 = globaltimer();
  while (true) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(arrivals) : "memory");
    if (v >= expected) break;
    if (globaltimer() - t0 > limit_ns) {
      set_status(status, MEGAMOE_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  __threadfence();
  return true;
}

// The fused requantisation of h (GemmArgs::rq_*), by every thread of a CTA
// that had tiles, after its last tile's epilogue and a __syncthreads.  Tiles
// are BN token rows x 128 features of h (h = the kernel's bf16 output,
// ld_out = N/2); two tasks per row of a tile, each four 16-element blocks:
// 32 bytes of codes and one 4-byte word of scales, encoded exactly as
// k_quant does (encode_block, gs = fl32(2688 / amax)).
__device__ __forceinline__ void fused_requant(const GemmArgs& p, const int* s_toff, int MT,
                                              int total, int BN, int* s_ok) {
  if (threadIdx.x == 0) {
    const uint32_t expected = static_cast<uint32_t>(min(static_cast<int>(gridDim.x), total));
    *s_ok = grid_arrive_and_wait(p.rq_arrivals, expected, p.status, p.wait_limit_ns) ? 1 : 0;
  }
  __syncthreads();
  if (!*s_ok) return;
  const float amax = __ldcg(p.out_amax);
  const float gs = amax == 0.f ? 1.f : __fdiv_rn(2688.0f, amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.rq_gs = gs;
  const int I = p.N / 2;
  const uint16_t* h = static_cast<const uint16_t*>(p.out);
  int e_lo = 0;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const TileInfo ti = decode_tile(tile, s_toff, p.E, MT, e_lo);
    e_lo = ti.e;
    const int cnt = __ldg(p.offsets + ti.e + 1) - __ldg(p.offsets + ti.e);
    const int m_valid = min(BN, cnt - ti.nt * BN);
    const int64_t row0 = __ldg(p.padded_offsets + ti.e) + static_cast<int64_t>(ti.nt) * BN;
    for (int t = threadIdx.x; t < 2 * m_valid; t += blockDim.x) {
      const int64_t row = row0 + (t >> 1);
      const int f = ti.mt * 128 + (t & 1) * 64;  // first of four 16-element blocks
      // h was written by this CTA in this kernel: read through L2, not the
      // non-coherent path
      const uint4* src = reinterpret_cast<const uint4*>(h + row * p.ld_out + f);
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __ldcg(src + i);
      uint2 c[4];
      uint32_t s8[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) encode_block(v[2 * j], v[2 * j + 1], gs, c[j], s8[j]);
      uint4* cd = reinterpret_cast<uint4*>(p.rq_codes + row * (I / 2) + f / 2);
      cd[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
      cd[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
      *reinterpret_cast<uint32_t*>(p.rq_scales + row * (I / 16) + f / 16) =
          s8[0] | (s8[1] << 8) | (s8[2] << 16) | (s8[3] << 24);
    }
  }
}

}  // namespace megamoe
