// Token-major grouped block-scaled NVFP4 GEMM tiles for large batches.
//
// "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Architecture: DeepSeek-V4
// MegaMoE": one GEMM problem per expert, persistent tile scheduling, a large
// token tile for prefill; "What's Been Verified": L1 gate+up and L2 down.
//
// Shape of one tile (tokens on the MMA's M side, weights on N):
//   D[128 tokens, 256 weight rows] = A[tokens, K] x W_e[rows, K]^T
// For the L1 GEMM the 256 weight rows are the gate rows and the up rows of
// the same 128 features (adjacent in the packed layout), so one MMA per K
// slice produces both and SiLU(gate) * up is a per-lane epilogue; for the
// other epilogues they are 256 consecutive output features.
//
// Why this orientation at large batches: a stage's shared-memory traffic is
// the TMA writes plus the tensor cores' operand reads.  With weights on M the
// L1 tile issues two 128 x 128 MMAs per K slice that both read the token tile
// (16 KB of operand reads per slice); here one 128 x 256 MMA reads the token
// tile once and the weights once (12 KB).  The epilogue's lanes are token
// rows, so each thread stores a contiguous run of its row's features without
// staging through shared memory, and the fp32 epilogue's tiles cover 256
// features instead of 128.
//
// Roles (448 threads, one CTA per SM, grid = number of SMs) as in the
// weights-on-M kernel: warp 0 producer, warp 1 TMEM allocator and MMA issuer,
// warps 6..9 write the stage's block scales into tensor memory (token scales:
// 4 columns per 64-K slice, column j = token rows 32 j .. 32 j + 31; weight
// scales: 8 columns per slice, column j = weight rows 32 j .. 32 j + 31),
// warps 2..5 and 10..13 drain the accumulator (two warps per 32-lane quarter,
// each taking half of the 256 columns).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace megamoe {

template <int EPI, int STAGES>
struct TmCfg {
  static constexpr bool SILU = EPI == MEGAMOE_EPI_SILU_MUL;
  static constexpr int BM = 128;              // token rows per tile (MMA M)
  static constexpr int A_TILE = BM * 128;     // tokens: 128 rows x 128 bytes (one 256-K step)
  static constexpr int B_TILE = 256 * 128;    // weights: two pre-swizzled 16 KB blocks
  static constexpr int SFW = 2 * 2048;        // weight scale atoms: 2 row groups x 4 slices
  static constexpr int SFA_RAW = BM * 16;     // token scales as loaded: 128 rows x 16 bytes
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = A_TILE;
  static constexpr int OFF_SFW = OFF_B + B_TILE;
  static constexpr int OFF_SFA_RAW = OFF_SFW + SFW;
  static constexpr int STAGE = (OFF_SFA_RAW + SFA_RAW + 1023) / 1024 * 1024;
  static constexpr uint32_t TX = A_TILE + B_TILE;  // codes (full barrier)
  static constexpr uint32_t SF_TX = SFW + SFA_RAW;  // scales (sf_full barrier)
  static constexpr int ACC_COLS = 256;              // one fp32 accumulator slot
  static constexpr int SF_COLS = 16 + 32;           // per stage: token + weight scales
  static constexpr int SF_COL0 = ACC_COLS;
  static constexpr int BAR_OFF = STAGES * STAGE;
  static constexpr int TOFF_OFF = BAR_OFF + 512;
  static constexpr int SMEM = 1024 + TOFF_OFF + 4 * (MEGAMOE_MAX_EXPERTS + 1);
  static constexpr uint32_t IDESC = idesc_nvf4(128, 256);
  static_assert(SF_COL0 + STAGES * SF_COLS <= 512, "tensor memory budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert((4 * STAGES + 3) * 8 + 8 <= 512, "barrier area");
};

template <int EPI, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_grouped_gemm_tm(const __grid_constant__ TokenMaps maps, const GemmArgs p) {
  using C = TmCfg<EPI, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_ready = empty + STAGES;
  uint64_t* sf_full = sf_ready + STAGES;
  uint64_t* acc_full = sf_full + STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_toff = reinterpret_cast<int*>(smem + C::TOFF_OFF);
  __shared__ int s_scan[kGemmThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, N = p.N, K = p.K;
  // feature tiles per expert: 128 features (gate + up rows) for L1, else 256
  const int MT = C::SILU ? (N / 2) / 128 : N / 256;
  const int KT = K / 256;
  const int slices = K / 64;
  // first weight row of feature tile mt of expert e, and its second 128-row
  // group (the up rows for L1, the next 128 features otherwise)
  auto w_rows = [&](int e, int mt, int* r0, int* r1) {
    if (C::SILU) {
      *r0 = e * N + mt * 128;
      *r1 = e * N + N / 2 + mt * 128;
    } else {
      *r0 = e * N + mt * 256;
      *r1 = *r0 + 128;
    }
  };

  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.codes);
    prefetch_tensormap(&maps.scales);
    prefetch_tensormap(&maps.codes32);
    prefetch_tensormap(&maps.scales32);
    prefetch_tensormap(&maps.codes64);
    prefetch_tensormap(&maps.scales64);
  }
  if (p.early_weights) {
    build_tile_offsets<128>(p.offsets, E, MT, s_toff, s_scan);
    if (warp == 2 && lane < min(2 * STAGES, KT) && static_cast<int>(blockIdx.x) < s_toff[E]) {
      // the first (up to) 2 x STAGES weight stages of this CTA's first tile
      const TileInfo t0 = decode_tile(blockIdx.x, s_toff, E, MT);
      int r0, r1;
      w_rows(t0.e, t0.mt, &r0, &r1);
      if (C::SILU) {
        const int blk = ((t0.e * MT + t0.mt) * KT + lane) * 2;
        bulk_prefetch_l2(p.w_codes + static_cast<int64_t>(blk) * 16384, 32768);
      } else {
        bulk_prefetch_l2(p.w_codes + (static_cast<int64_t>(r0 >> 7) * KT + lane) * 16384, 16384);
        bulk_prefetch_l2(p.w_codes + (static_cast<int64_t>(r1 >> 7) * KT + lane) * 16384, 16384);
      }
    }
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_wait();
    pdl_trigger();
    build_tile_offsets<128>(p.offsets, E, MT, s_toff, s_scan);
  }
  const int total = s_toff[E];
  if (static_cast<int>(blockIdx.x) >= total) return;  // uniform: no work for this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 4);
      mbar_init(&sf_full[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol_w_once = policy_evict_first();
      const uint64_t pol_w_reused = policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      auto rows_of = [&](const TileInfo& t) {
        return __ldg(p.offsets + t.e + 1) - __ldg(p.offsets + t.e);
      };
      TileInfo ti_next = decode_tile(blockIdx.x, s_toff, E, MT);
      int poff_next = __ldg(p.padded_offsets + ti_next.e);
      int cnt_next = rows_of(ti_next);
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = ti_next;
        const int poff = poff_next;
        const int cnt = cnt_next;
        if (tile + static_cast<int>(gridDim.x) < total) {
          ti_next = decode_tile(tile + gridDim.x, s_toff, E, MT, ti.e);
          poff_next = __ldg(p.padded_offsets + ti_next.e);
          cnt_next = rows_of(ti_next);
        }
        // an expert's last tile with at most 32 (64) valid rows loads only a
        // 32 (64)-row token box; the MMA still computes 128 rows, and the
        // rows past the box (stale shared memory) are never stored
        const int box = short_box_rows(cnt - ti.nt * C::BM);
        const CUtensorMap* map_c =
            box == 32 ? &maps.codes32 : box == 64 ? &maps.codes64 : &maps.codes;
        const CUtensorMap* map_s =
            box == 32 ? &maps.scales32 : box == 64 ? &maps.scales64 : &maps.scales;
        int r0, r1;
        w_rows(ti.e, ti.mt, &r0, &r1);
        const int a_row0 = poff + ti.nt * C::BM;
        const uint64_t pol_w = ti.ntiles > 1 ? pol_w_reused : pol_w_once;
        const uint8_t* sfw0 = p.w_sf + static_cast<int64_t>(r0 >> 7) * slices * 512;
        const uint8_t* sfw1 = p.w_sf + static_cast<int64_t>(r1 >> 7) * slices * 512;
        // K = 0 code blocks: the adjacent gate/up pair (L1), or the first
        // block of each 128-row group
        const uint8_t* wc0 = C::SILU
            ? p.w_codes + static_cast<int64_t>((ti.e * MT + ti.mt) * KT) * 2 * 16384
            : p.w_codes + static_cast<int64_t>(r0 >> 7) * KT * 16384;
        const uint8_t* wc1 = p.w_codes + static_cast<int64_t>(r1 >> 7) * KT * 16384;
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE;
          mbar_arrive_expect_tx(&sf_full[stage], C::SFW + box * 16);
          bulk_load(sb + C::OFF_SFW, sfw0 + kt * 2048, 2048, &sf_full[stage], pol_w);
          bulk_load(sb + C::OFF_SFW + 2048, sfw1 + kt * 2048, 2048, &sf_full[stage], pol_w);
          tma_load_2d(sb + C::OFF_SFA_RAW, map_s, &sf_full[stage], kt * 16, a_row0, pol_a);
          mbar_arrive_expect_tx(&full[stage], C::B_TILE + box * 128);
          if (C::SILU) {
            bulk_load(sb + C::OFF_B, wc0 + kt * 32768, 32768, &full[stage], pol_w);
          } else {
            bulk_load(sb + C::OFF_B, wc0 + kt * 16384, 16384, &full[stage], pol_w);
            bulk_load(sb + C::OFF_B + 16384, wc1 + kt * 16384, 16384, &full[stage], pol_w);
          }
          tma_load_2d(sb + C::OFF_A, map_c, &full[stage], kt * 128, a_row0, pol_a);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // unwinding: let every copy already in flight land first
        for (int s = 0; s < STAGES && s < issued; ++s) {
          const uint32_t parity = static_cast<uint32_t>((issued - 1 - s) / STAGES) & 1u;
          mbar_drain(&full[s], parity);
          mbar_drain(&sf_full[s], parity);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, p.wait_limit_ns) ||
              !mbar_wait(&sf_ready[stage], phase, abort_flag, p.status, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* sb = smem + stage * C::STAGE;
          const uint32_t sf_col = tmem + C::SF_COL0 + stage * C::SF_COLS;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint64_t adesc = sdesc_sw128(smem_u32(sb + C::OFF_A) + 32 * c);
            const uint64_t bdesc = sdesc_sw128(smem_u32(sb + C::OFF_B) + 32 * c);
            mma_nvf4(tmem, adesc, bdesc, C::IDESC, sf_col + 4 * c, sf_col + 16 + 8 * c,
                     (kt != 0 || c != 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_phase ^= 1u;
      }
      // every MMA issued so far must finish before tensor memory is released
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= kSfWarp0 && warp < kEpiWarp1) {
    // --------------------------------------------------------- scale writers
    // Token scales arrive row-major (row n: 16 bytes = 4 slices x 4 blocks):
    // lane i takes rows 32 j + i and writes slice c's word to column 4 c + j.
    // Weight atom of slice c, row group g: byte 16 i + 4 j + b = row 32 j + i,
    // block 4c + b; lane i writes word j to column 16 + 8 c + 4 g + j.
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait(&sf_full[stage], phase, abort_flag, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint8_t* sb = smem + stage * C::STAGE;
        const uint32_t sf_col = tmem + lane_off + C::SF_COL0 + stage * C::SF_COLS;
        const uint4* raw = reinterpret_cast<const uint4*>(sb + C::OFF_SFA_RAW);
        uint4 r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) r[j] = raw[32 * j + lane];
        tmem_st_32x32b_x4(sf_col + 0, r[0].x, r[1].x, r[2].x, r[3].x);
        tmem_st_32x32b_x4(sf_col + 4, r[0].y, r[1].y, r[2].y, r[3].y);
        tmem_st_32x32b_x4(sf_col + 8, r[0].z, r[1].z, r[2].z, r[3].z);
        tmem_st_32x32b_x4(sf_col + 12, r[0].w, r[1].w, r[2].w, r[3].w);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 a =
                reinterpret_cast<const uint4*>(sb + C::OFF_SFW + g * 2048 + c * 512)[lane];
            tmem_st_32x32b_x4(sf_col + 16 + 8 * c + 4 * g, a.x, a.y, a.z, a.w);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Lane i of a warp in quarter q holds token row 32 q + i of the tile;
    // the two warps of a quarter take halves of the 256 accumulator columns
    // (for L1: gate features [64 half, 64 half + 64) and their up columns).
    const int q = warp & 3;
    const int half = warp >= kEpiWarp1 ? 1 : 0;
    const int row_in_tile = q * 32 + lane;
    const float a_gs = __ldg(p.a_gs);
    uint32_t acc_phase = 0;
    float amax = 0.f;
    struct ExpertInfo {
      TileInfo ti;
      int count, poff;
      float gs0, gs1;
    };
    auto fetch = [&](int tile, int e_lo) {
      ExpertInfo x;
      x.ti = decode_tile(tile, s_toff, E, MT, e_lo);
      const int e = x.ti.e;
      x.count = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
      x.poff = __ldg(p.padded_offsets + e);
      x.gs0 = __ldg(p.w_gs + (C::SILU ? 2 * e : e));
      x.gs1 = C::SILU ? __ldg(p.w_gs + 2 * e + 1) : 1.f;
      return x;
    };
    ExpertInfo next = fetch(blockIdx.x, 0);
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const ExpertInfo cur = next;
      const TileInfo& ti = cur.ti;
      if (tile + static_cast<int>(gridDim.x) < total) next = fetch(tile + gridDim.x, ti.e);
      const bool valid = ti.nt * C::BM + row_in_tile < cur.count;
      const int64_t row = cur.poff + static_cast<int64_t>(ti.nt) * C::BM + row_in_tile;
      const float alpha0 = 1.0f / (a_gs * cur.gs0);
      const float alpha1 = C::SILU ? 1.0f / (a_gs * cur.gs1) : 0.f;
      if (!mbar_wait(acc_full, acc_phase, abort_flag, p.status, p.wait_limit_ns)) break;
      tc_fence_after();
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
      if (C::SILU) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + row * p.ld_out + ti.mt * 128;
#pragma unroll 1
        for (int f0 = 64 * half; f0 < 64 * half + 64; f0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld_32x32b_x16(lane_base + f0, g);
          tmem_ld_32x32b_x16(lane_base + 128 + f0, u);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float hv[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const float gv = __uint_as_float(g[j + t]) * alpha0;
              const float uv = __uint_as_float(u[j + t]) * alpha1;
              // SiLU(g) * u = g * u / (1 + e^-g); e^-g = inf gives the limit 0
              const __nv_bfloat16 hb = __float2bfloat16_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
              hv[t] = __bfloat162float(hb);
            }
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(hv[0], hv[1]);
            pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            if (valid) amax = fmaxf(amax, fmaxf(fabsf(hv[0]), fabsf(hv[1])));
          }
          if (valid) {
            reinterpret_cast<uint4*>(out + f0)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            reinterpret_cast<uint4*>(out + f0)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else if (EPI == MEGAMOE_EPI_BF16) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + row * p.ld_out + ti.mt * 256;
#pragma unroll 1
        for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(lane_base + c0, v);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[j]) * alpha0,
                                                            __uint_as_float(v[j + 1]) * alpha0);
            pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          if (valid) {
            reinterpret_cast<uint4*>(out + c0)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            reinterpret_cast<uint4*>(out + c0)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
        float* out = reinterpret_cast<float*>(p.out) + row * p.ld_out + ti.mt * 256;
#pragma unroll 1
        for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(lane_base + c0, v);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(out + c0 + j) =
                  make_float4(__uint_as_float(v[j]) * alpha0, __uint_as_float(v[j + 1]) * alpha0,
                              __uint_as_float(v[j + 2]) * alpha0,
                              __uint_as_float(v[j + 3]) * alpha0);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      acc_phase ^= 1u;
    }
    if (C::SILU) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0 && amax > 0.f)
        atomicMax(reinterpret_cast<unsigned int*>(p.out_amax), __float_as_uint(amax));
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (C::SILU && p.rq_arrivals) {
    __shared__ int s_rq_ok;
    fused_requant(p, s_toff, MT, total, C::BM, &s_rq_ok);
  }
}

template <int EPI, int STAGES>
static cudaError_t launch_tm_cfg(const TokenMaps& maps, const GemmArgs& a, cudaStream_t stream) {
  using C = TmCfg<EPI, STAGES>;
  auto kern = k_grouped_gemm_tm<EPI, STAGES>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(num_sms()), dim3(kGemmThreads), C::SMEM, stream, maps, a);
}

cudaError_t launch_grouped_gemm_tm(const TokenMaps& maps, const GemmArgs& a, int epilogue,
                                   cudaStream_t stream) {
  switch (epilogue) {
    case MEGAMOE_EPI_SILU_MUL: return launch_tm_cfg<MEGAMOE_EPI_SILU_MUL, 4>(maps, a, stream);
    case MEGAMOE_EPI_BF16: return launch_tm_cfg<MEGAMOE_EPI_BF16, 4>(maps, a, stream);
    case MEGAMOE_EPI_F32: return launch_tm_cfg<MEGAMOE_EPI_F32, 4>(maps, a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace megamoe
