// Persistent grouped block-scaled NVFP4 GEMM on tcgen05 tensor cores.
//
// "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Architecture: DeepSeek-V4
// MegaMoE": one GEMM problem per expert, persistent tile scheduling across the
// experts, a token tile chosen from the expected tokens per expert (small for
// decode, large for prefill); "What's Been Verified": L1 gate+up and L2 down.
//
// Shape of one tile (weights on the MMA's M side, tokens on N):
//   D[128 output features, BN tokens] = W_e[features, K] x A[tokens, K]^T
// with E2M1 operands and one E4M3 scale per 16 elements of each operand,
// accumulated in fp32 in tensor memory (tcgen05.mma kind::mxf4nvf4,
// scale_vec::4X, M = 128, K = 64 per instruction).  For the L1 GEMM a tile
// holds the gate AND the up accumulators of the same 128 features (two MMAs
// per K step into two TMEM ranges), so SiLU(gate) * up is a per-lane epilogue.
//
// Roles (448 threads, one CTA per SM, grid = number of SMs):
//   warp 0      producer (one lane): per stage, the weights' block-scale atoms
//               (bulk copies) and the token tile's row-major block scales
//               (tensor map) on one barrier, then the stage's weight codes
//               (one bulk copy of pre-swizzled blocks) and token codes
//               (tensor map, 128-byte swizzle) on another, into a
//               STAGES-deep ring;
//   warp 1      TMEM allocator; one lane issues tcgen05.mma and commits
//               stage-free / accumulator-ready;
//   warps 2..5, 10..13  epilogue, two warps per 32-lane TMEM quarter taking
//               alternate 16-column chunks: tcgen05.ld, alpha scaling,
//               SiLU * up -> bf16 + amax (L1), bf16, or fp32 (L2), staged
//               through shared memory into 16-byte stores;
//   warps 6..9  scale writers: each writes the stage's weight and token block
//               scales into its own 32-lane quarter of tensor memory with
//               tcgen05.st (every quarter holds the same copy, the layout the
//               block-scaled MMA reads).  Scales do not go through the tensor
//               pipe (a tcgen05.cp costs about as much as an MMA), and the
//               token tile's first row always lands in the first scale
//               column whatever row the tile starts at.
// Split-K (kEpiPartial* instantiations, used by the dense linear when it has
// fewer tiles than SMs): each tile's K range is cut into pieces whose fp32
// partial sums go to planes that k_splitk_finish adds in a fixed order.
// Every expert's weights live in one buffer, packed once into blocks of 128
// rows x 128 bytes already in the 128-byte swizzle ([E*N/128][K/256] blocks;
// for L1 the gate and up blocks of the same features and K step adjacent), so
// the expert is an offset, not a new descriptor, and a stage's weights are one
// contiguous 16 KB (L2) or 32 KB (L1) bulk copy.  Token tiles use tensor maps.
// Tiles are numbered expert-major, weight-tile-major, token-tile-minor, so CTAs
// working on the same expert's weight tile run together and share it in L2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace megamoe {

template <int BN, int EPI, int STAGES>
struct GemmCfg {
  static constexpr int G = (EPI == MEGAMOE_EPI_SILU_MUL || EPI == kEpiPartial2) ? 2 : 1;
  static constexpr bool PARTIAL = EPI >= kEpiPartial1;
  // Two accumulator slots (the MMA fills one while the epilogue drains the
  // other) whenever tensor memory has room for them.
  static constexpr int ACC_STAGES = (2 * G * BN + STAGES * (16 * G + 16) <= 512) ? 2 : 1;
  static constexpr int A_TILE = 128 * 128;  // one weight matrix, 128 rows x 128 bytes
  static constexpr int B_TILE = BN * 128;
  static constexpr int SFW = 2048;     // 4 atoms of 512 bytes (one per 64-element slice)
  static constexpr int SFA_RAW = BN * 16;  // token scales as loaded: BN rows x 16 bytes
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = G * A_TILE;
  static constexpr int OFF_SFW = OFF_B + B_TILE;
  static constexpr int OFF_SFA_RAW = OFF_SFW + G * SFW;
  static constexpr int STAGE = (OFF_SFA_RAW + SFA_RAW + 1023) / 1024 * 1024;
  static constexpr uint32_t TX = G * A_TILE + B_TILE;     // codes (full barrier)
  static constexpr uint32_t SF_TX = G * SFW + SFA_RAW;     // scales (sf_full barrier)
  static constexpr int ACC_COLS = G * BN;
  static constexpr int SF_COLS = 16 * G + 16;  // per stage: weight scales + token scales
  static constexpr int SF_COL0 = ACC_STAGES * ACC_COLS;
  static constexpr int BAR_OFF = STAGES * STAGE;
  static constexpr int TOFF_OFF = BAR_OFF + 512;
  // per epilogue warp: STG_ROWS token rows x 32 features of output, staged so
  // that global stores are 16-byte vectors along the feature axis (512 bytes
  // for bf16, 2 KB for float)
  static constexpr bool BF16_OUT = EPI == MEGAMOE_EPI_SILU_MUL || EPI == MEGAMOE_EPI_BF16;
  static constexpr bool BFP16 = EPI == MEGAMOE_EPI_BFP16;
  // (the fp32 and BFP16 epilogues store straight from registers: for each
  // token a warp's 32 lanes hold 32 consecutive features, one 128- or 64-byte
  // run, so they need no staging and their shared memory goes to pipeline
  // stages; a lane's 16 tokens of one feature share a BFP16 exponent group
  // with those of 7 neighbouring lanes)
  static constexpr bool STAGED = BF16_OUT || PARTIAL;
  static constexpr int STG_ROWS = BF16_OUT ? 8 : 16;
  static constexpr int STG_BYTES = STAGED ? STG_ROWS * 32 * (BF16_OUT ? 2 : 4) : 0;
  static constexpr int STG_OFF = (TOFF_OFF + 4 * (MEGAMOE_MAX_EXPERTS + 1) + 15) / 16 * 16;
  static constexpr int SMEM = 1024 + STG_OFF + kEpiWarps * STG_BYTES;
  static constexpr uint32_t IDESC = idesc_nvf4(128, BN);
  static_assert(SF_COL0 + STAGES * SF_COLS <= 512, "tensor memory budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert((4 * STAGES + 2 * ACC_STAGES + 1) * 8 + 8 <= 512, "barrier area");
};

template <int BN, int EPI, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_grouped_gemm(const __grid_constant__ TokenMaps maps, const GemmArgs p) {
  using C = GemmCfg<BN, EPI, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_ready = empty + STAGES;
  uint64_t* sf_full = sf_ready + STAGES;   // the stage's block scales have landed
  uint64_t* acc_full = sf_full + STAGES;   // [ACC_STAGES]
  uint64_t* acc_empty = acc_full + C::ACC_STAGES;  // [ACC_STAGES]
  uint64_t* drain = acc_empty + C::ACC_STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_toff = reinterpret_cast<int*>(smem + C::TOFF_OFF);
  __shared__ int s_scan[kGemmThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, N = p.N, K = p.K;
  const int MT = (C::G == 2 ? N / 2 : N) / 128;
  const int KT = K / 256;
  const int slices = K / 64;
  // pieces per tile (1 unless split-K); piece q -> tile q / S, K range
  // [ks * KT / S, (ks + 1) * KT / S) with ks = q % S
  const int S = C::PARTIAL ? p.ksplit : 1;

  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.codes);
    prefetch_tensormap(&maps.scales);
  }
  // The activations and their global scale come from the preceding kernel,
  // the routing offsets from it or (early_weights) from an earlier one.
  if (p.early_weights) {
    build_tile_offsets<BN>(p.offsets, E, MT, s_toff, s_scan);
    if (warp == 2 && lane < min(2 * STAGES, KT / S) &&
        static_cast<int>(blockIdx.x) < s_toff[E] * S) {
      // the first (up to) 2 x STAGES weight stages of this CTA's first piece
      const int tile0 = static_cast<int>(blockIdx.x) / S;
      const TileInfo t0 = decode_tile(tile0, s_toff, E, MT);
      const int kt0 = (static_cast<int>(blockIdx.x) - tile0 * S) * KT / S;
      const int blk0 = C::G == 2 ? ((t0.e * MT + t0.mt) * KT) * 2
                                 : ((t0.e * N + t0.mt * 128) >> 7) * KT;
      bulk_prefetch_l2(p.w_codes + static_cast<int64_t>(blk0 + (kt0 + lane) * C::G) * 16384,
                       C::G * C::A_TILE);
    }
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_wait();
    pdl_trigger();
    build_tile_offsets<BN>(p.offsets, E, MT, s_toff, s_scan);
  }
  const int total = s_toff[E] * S;  // pieces
  if (static_cast<int>(blockIdx.x) >= total) return;  // uniform: no work for this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 4);
      mbar_init(&sf_full[s], 1);
    }
    for (int a = 0; a < C::ACC_STAGES; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
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
      // A weight tile read by one token tile is dead after it (evict first);
      // one that the expert's next token tiles re-read stays (evict normal).
      const uint64_t pol_w_once = policy_evict_first();
      const uint64_t pol_w_reused = policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // stages issued; issue i used slot i % STAGES, parity (i / STAGES) & 1
      bool ok = true;
      // the next tile and its expert's first padded row are found one tile ahead
      TileInfo ti_next = decode_tile(static_cast<int>(blockIdx.x) / S, s_toff, E, MT);
      int poff_next = __ldg(p.padded_offsets + ti_next.e);
      for (int piece = blockIdx.x; ok && piece < total; piece += gridDim.x) {
        const TileInfo ti = ti_next;
        const int poff = poff_next;
        const int ks = piece - (piece / S) * S;
        const int k0 = ks * KT / S, k1 = (ks + 1) * KT / S;
        if (piece + static_cast<int>(gridDim.x) < total) {
          ti_next = decode_tile((piece + static_cast<int>(gridDim.x)) / S, s_toff, E, MT, ti.e);
          poff_next = __ldg(p.padded_offsets + ti_next.e);
        }
        const int w_row0 = ti.e * N + ti.mt * 128;
        const int w_row1 = ti.e * N + N / 2 + ti.mt * 128;  // up rows (L1 only)
        // first 128-row code block of this tile's K = 0 step (paired for L1)
        const int w_blk0 = C::G == 2 ? ((ti.e * MT + ti.mt) * KT) * 2 : (w_row0 >> 7) * KT;
        const int a_row0 = poff + ti.nt * BN;
        const uint64_t pol_w = ti.ntiles > 1 ? pol_w_reused : pol_w_once;
        // this tile's K = 0 weight scales (gate, up) and codes; each K step
        // advances them by 4 atoms and by G code blocks
        const uint8_t* sfw0 = p.w_sf + static_cast<int64_t>(w_row0 >> 7) * slices * 512;
        const uint8_t* sfw1 = p.w_sf + static_cast<int64_t>(w_row1 >> 7) * slices * 512;
        const uint8_t* wcod = p.w_codes + static_cast<int64_t>(w_blk0) * 16384;
        for (int kt = k0; kt < k1; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE;
          // scales first, on their own barrier: the scale warps move them into
          // tensor memory while the codes are still landing
          mbar_arrive_expect_tx(&sf_full[stage], C::SF_TX);
          bulk_load(sb + C::OFF_SFW, sfw0 + kt * 2048, C::SFW, &sf_full[stage], pol_w);
          if (C::G == 2)
            bulk_load(sb + C::OFF_SFW + C::SFW, sfw1 + kt * 2048, C::SFW, &sf_full[stage], pol_w);
          tma_load_2d(sb + C::OFF_SFA_RAW, &maps.scales, &sf_full[stage], kt * 16, a_row0, pol_a);
          mbar_arrive_expect_tx(&full[stage], C::TX);
          // the stage's weight blocks (gate then up for L1) are contiguous and
          // pre-swizzled: one bulk copy
          bulk_load(sb + C::OFF_A, wcod + kt * (C::G * 16384), C::G * C::A_TILE, &full[stage], pol_w);
          tma_load_2d(sb + C::OFF_B, &maps.codes, &full[stage], kt * 128, a_row0, pol_a);
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
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int piece = blockIdx.x; ok && piece < total; piece += gridDim.x) {
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
        tc_fence_after();
        const uint32_t d_col = tmem + acc * C::ACC_COLS;
        const int ks = piece - (piece / S) * S;
        const int k0 = ks * KT / S, k1 = (ks + 1) * KT / S;
        for (int kt = k0; kt < k1; ++kt) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, p.wait_limit_ns) ||
              !mbar_wait(&sf_ready[stage], phase, abort_flag, p.status, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* sb = smem + stage * C::STAGE;
          const uint32_t sf_col = tmem + C::SF_COL0 + stage * C::SF_COLS;
          const uint32_t sfa_col = sf_col + 16 * C::G;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint64_t bdesc = sdesc_sw128(smem_u32(sb + C::OFF_B) + 32 * c);
#pragma unroll
            for (int g = 0; g < C::G; ++g) {
              const uint64_t adesc = sdesc_sw128(smem_u32(sb + C::OFF_A + g * C::A_TILE) + 32 * c);
              mma_nvf4(d_col + g * BN, adesc, bdesc, C::IDESC, sf_col + 16 * g + 4 * c,
                       sfa_col + 4 * c, (kt != k0 || c != 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued so far must finish before tensor memory is released
      tc_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= kSfWarp0 && warp < kEpiWarp1) {
    // --------------------------------------------------------- scale writers
    // Weight atom of slice c: byte 16 i + 4 j + b = row 32 j + i, block 4c + b;
    // lane i writes word j to column (4c + j) of lane quarter*32 + i.  Token
    // scales arrive row-major (row n: 16 bytes = 4 slices x 4 blocks) and are
    // regrouped the same way in registers.
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int piece = blockIdx.x; ok && piece < total; piece += gridDim.x) {
      const int ks = piece - (piece / S) * S;
      const int nk = (ks + 1) * KT / S - ks * KT / S;
      for (int kt = 0; kt < nk; ++kt) {
        if (!mbar_wait(&sf_full[stage], phase, abort_flag, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint8_t* sb = smem + stage * C::STAGE;
        const uint32_t sf_col = tmem + lane_off + C::SF_COL0 + stage * C::SF_COLS;
#pragma unroll
        for (int g = 0; g < C::G; ++g) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 a = reinterpret_cast<const uint4*>(sb + C::OFF_SFW + g * C::SFW + c * 512)[lane];
            tmem_st_32x32b_x4(sf_col + 16 * g + 4 * c, a.x, a.y, a.z, a.w);
          }
        }
        const uint4* raw = reinterpret_cast<const uint4*>(sb + C::OFF_SFA_RAW);
        const uint32_t sfa_col = sf_col + 16 * C::G;
        uint4 r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          r[j] = (32 * j + lane < BN) ? raw[32 * j + lane] : make_uint4(0u, 0u, 0u, 0u);
        tmem_st_32x32b_x4(sfa_col + 0, r[0].x, r[1].x, r[2].x, r[3].x);
        tmem_st_32x32b_x4(sfa_col + 4, r[0].y, r[1].y, r[2].y, r[3].y);
        tmem_st_32x32b_x4(sfa_col + 8, r[0].z, r[1].z, r[2].z, r[3].z);
        tmem_st_32x32b_x4(sfa_col + 12, r[0].w, r[1].w, r[2].w, r[3].w);
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
    // Two warps per TMEM lane quarter (a warp reaches only quarter warp % 4)
    // take alternate 16-column chunks of the tile.  Lane i holds feature i of
    // the quarter for 16 tokens; the chunk is transposed through the warp's
    // staging buffer so that each global store is a 16-byte run of features.
    const int q = warp & 3;
    const int half = warp >= kEpiWarp1 ? 1 : 0;
    uint8_t* stg = smem + C::STG_OFF + (half * 4 + q) * C::STG_BYTES;
    const float a_gs = __ldg(p.a_gs);
    int acc = 0;
    uint32_t acc_phase = 0;
    float amax = 0.f;
    // an expert's row count, first padded row and global scales, fetched one
    // tile ahead so that their latency hides behind the current tile
    struct ExpertInfo {
      TileInfo ti;
      int count, poff, off;  // valid rows, first padded row, first unpadded row
      float gs0, gs1;
    };
    auto fetch = [&](int tile, int e_lo) {
      ExpertInfo x;
      x.ti = decode_tile(tile, s_toff, E, MT, e_lo);
      const int e = x.ti.e;
      x.count = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
      x.poff = __ldg(p.padded_offsets + e);
      x.off = __ldg(p.offsets + e);
      x.gs0 = __ldg(p.w_gs + C::G * e);
      x.gs1 = C::G == 2 ? __ldg(p.w_gs + 2 * e + 1) : 1.f;
      return x;
    };
    ExpertInfo next = fetch(static_cast<int>(blockIdx.x) / S, 0);
    for (int piece = blockIdx.x; piece < total; piece += gridDim.x) {
      const ExpertInfo cur = next;
      const TileInfo& ti = cur.ti;
      const int ks = piece - (piece / S) * S;
      if (piece + static_cast<int>(gridDim.x) < total)
        next = fetch((piece + static_cast<int>(gridDim.x)) / S, ti.e);
      const int m_valid = min(BN, cur.count - ti.nt * BN);
      const int64_t row0 = cur.poff + static_cast<int64_t>(ti.nt) * BN;
      const int f0 = ti.mt * 128 + q * 32;  // first feature of this warp's quarter
      const float alpha0 = 1.0f / (a_gs * cur.gs0);
      const float alpha1 = C::G == 2 ? 1.0f / (a_gs * cur.gs1) : 0.f;
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.status, p.wait_limit_ns)) break;
      tc_fence_after();
      const uint32_t lane_base =
          tmem + acc * C::ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      for (int n0 = 16 * half; n0 < m_valid; n0 += 32) {
        const int rows = min(16, m_valid - n0);
        if (C::PARTIAL) {
          // split-K piece: acc * alpha of each operand matrix, fp32, to plane
          // ks at the unpadded rows; gate columns [0, N/2), up [N/2, N)
          float* plane = p.partial + ks * p.partial_plane;
          const int64_t urow = cur.off + static_cast<int64_t>(ti.nt) * BN + n0;
#pragma unroll
          for (int m = 0; m < C::G; ++m) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(lane_base + m * BN + n0, v);
            tmem_ld_wait();
            const float al = m == 0 ? alpha0 : alpha1;
            float* st = reinterpret_cast<float*>(stg);
#pragma unroll
            for (int j = 0; j < 16; ++j) st[j * 32 + lane] = __uint_as_float(v[j]) * al;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = lane + 32 * i, r = c >> 3;
              if (r < rows)
                *reinterpret_cast<uint4*>(plane + (urow + r) * N + m * (N / 2) + f0 + 4 * (c & 7)) =
                    reinterpret_cast<const uint4*>(stg)[c];
            }
            __syncwarp();
          }
          continue;
        }
        uint32_t g[16];
        tmem_ld_32x32b_x16(lane_base + n0, g);
        if (C::G == 2) {
          uint32_t u[16];
          tmem_ld_32x32b_x16(lane_base + BN + n0, u);
          tmem_ld_wait();
          __nv_bfloat16* s = reinterpret_cast<__nv_bfloat16*>(stg);
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int h8 = 0; h8 < 16; h8 += 8) {  // two staged halves of 8 rows
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float gv = __uint_as_float(g[h8 + j]) * alpha0;
              const float uv = __uint_as_float(u[h8 + j]) * alpha1;
              // SiLU(g) * u = g * u / (1 + e^-g); e^-g = inf gives the limit 0
              const __nv_bfloat16 hb =
                  __float2bfloat16_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
              if (h8 + j < rows) amax = fmaxf(amax, fabsf(__bfloat162float(hb)));
              s[j * 32 + lane] = hb;
            }
            __syncwarp();
            // 8 rows x 64 bytes = 32 chunks of 16 bytes, one per lane
            const int r = h8 + (lane >> 2);
            if (r < rows)
              *reinterpret_cast<uint4*>(out + (row0 + n0 + r) * p.ld_out + f0 + 8 * (lane & 3)) =
                  reinterpret_cast<const uint4*>(stg)[lane];
            __syncwarp();
          }
        } else if (C::BF16_OUT) {
          tmem_ld_wait();
          __nv_bfloat16* s = reinterpret_cast<__nv_bfloat16*>(stg);
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int h8 = 0; h8 < 16; h8 += 8) {  // two staged halves of 8 rows
#pragma unroll
            for (int j = 0; j < 8; ++j)
              s[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(g[h8 + j]) * alpha0);
            __syncwarp();
            const int r = h8 + (lane >> 2);
            if (r < rows)
              *reinterpret_cast<uint4*>(out + (row0 + n0 + r) * p.ld_out + f0 + 8 * (lane & 3)) =
                  reinterpret_cast<const uint4*>(stg)[lane];
            __syncwarp();
          }
        } else if (C::BFP16) {
          tmem_ld_wait();
          // rows row0 + n0 .. + 15 (16-aligned: pads and tiles are multiples
          // of 16) of features 8c .. 8c + 7 (8 consecutive lanes) are one
          // exponent group: the max |v| of this lane's written rows, then of
          // the 8 lanes; per token one 64-byte run of values across the warp,
          // and one exponent byte per 8 lanes
          float v[16];
          uint32_t mbits = 0u;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            v[j] = __uint_as_float(g[j]) * alpha0;
            if (j < rows) mbits = max(mbits, __float_as_uint(v[j]) & 0x7fffffffu);
          }
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) mbits = max(mbits, __shfl_xor_sync(0xffffffffu, mbits, o));
          const int sg = bfp16_exponent(mbits);
          uint16_t* q = reinterpret_cast<uint16_t*>(p.out) + (row0 + n0) * p.ld_out + f0 + lane;
          if (sg != kBfp16NonFinite) {
            const float sc = bfp16_pow2(-sg);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < rows) q[j * p.ld_out] = bfp16_round_int(v[j] * sc);
          } else {  // a group holding Inf or NaN: fp16 bits
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < rows) q[j * p.ld_out] = __half_as_ushort(__float2half_rn(v[j]));
          }
          if ((lane & 7) == 0)
            p.out_exp[((row0 + n0) >> 4) * (p.ld_out / 8) + ((f0 + lane) >> 3)] = static_cast<int8_t>(sg);
        } else {
          tmem_ld_wait();
          // token n0 + j: lanes write features f0 .. f0 + 31, one 128-byte run
          float* out = reinterpret_cast<float*>(p.out) + (row0 + n0) * p.ld_out + f0 + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < rows) out[j * p.ld_out] = __uint_as_float(g[j]) * alpha0;
        }
        __syncwarp();  // the staging buffer is rewritten by the next chunk
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (EPI == MEGAMOE_EPI_SILU_MUL) {
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
  if (EPI == MEGAMOE_EPI_SILU_MUL && p.rq_arrivals) {  // never split (S = 1)
    __shared__ int s_rq_ok;
    fused_requant(p, s_toff, MT, total, BN, &s_rq_ok);
  }
}

// Finishes a split-K GEMM: sums the fp32 planes in plane order and applies
// the epilogue (SiLU(gate) * up -> bf16 with amax, bf16, or fp32) at the
// padded output row.  One thread per (valid row, 4 output columns).
template <int EPI>
__global__ void __launch_bounds__(256)
    k_splitk_finish(const float* __restrict__ partial, int S, int64_t plane,
                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ padded_offsets,
                    int E, int N, void* out, int64_t ld_out, float* out_amax) {
  pdl_wait();
  pdl_trigger();
  const int width = EPI == MEGAMOE_EPI_SILU_MUL ? N / 2 : N;
  const int vecs = width / 4;
  const int64_t total = static_cast<int64_t>(__ldg(offsets + E)) * vecs;
  float amax = 0.f;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t u = (i >> 32) == 0
                          ? static_cast<int64_t>(static_cast<uint32_t>(i) / static_cast<uint32_t>(vecs))
                          : i / vecs;
    const int v = static_cast<int>(i - u * vecs);
    int lo = 0, hi = E - 1;  // largest e with offsets[e] <= u: the expert owning row u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(offsets + mid) <= u) lo = mid;
      else hi = mid - 1;
    }
    const int64_t row = __ldg(padded_offsets + lo) + (u - __ldg(offsets + lo));
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    for (int ks = 0; ks < S; ++ks) {
      const float* pl = partial + ks * plane + u * N + 4 * v;
      const float4 x = __ldg(reinterpret_cast<const float4*>(pl));
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      if (EPI == MEGAMOE_EPI_SILU_MUL) {
        const float4 y = __ldg(reinterpret_cast<const float4*>(pl + N / 2));
        b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
      }
    }
    if (EPI == MEGAMOE_EPI_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + row * ld_out + 4 * v) = a;
      continue;
    }
    float r[4] = {a.x, a.y, a.z, a.w};
    if (EPI == MEGAMOE_EPI_SILU_MUL) {
      const float up[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) r[j] = __fdividef(r[j], 1.0f + __expf(-r[j])) * up[j];
    }
    uint16_t hb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 q = __float2bfloat16_rn(r[j]);
      hb[j] = *reinterpret_cast<const uint16_t*>(&q);
      if (EPI == MEGAMOE_EPI_SILU_MUL) amax = fmaxf(amax, fabsf(__bfloat162float(q)));
    }
    uint2 pk;
    pk.x = hb[0] | (static_cast<uint32_t>(hb[1]) << 16);
    pk.y = hb[2] | (static_cast<uint32_t>(hb[3]) << 16);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + row * ld_out + 4 * v) = pk;
  }
  if (EPI == MEGAMOE_EPI_SILU_MUL) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0 && amax > 0.f)
      atomicMax(reinterpret_cast<unsigned int*>(out_amax), __float_as_uint(amax));
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D map over a [rows, row_bytes] byte matrix, boxes of box_rows x 128 bytes
// in the 128-byte swizzle the MMA descriptors expect.
static bool make_codes_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                           uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// 2-D map over row-major block scales [rows, K/16] bytes, boxes of
// box_rows x 16 bytes (the four 64-element slices of one 256-element K step).
static bool make_scales_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                            uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {16, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int EPI, int STAGES>
static cudaError_t launch_cfg(const TokenMaps& maps, const GemmArgs& a, cudaStream_t stream) {
  using C = GemmCfg<BN, EPI, STAGES>;
  auto kern = k_grouped_gemm<BN, EPI, STAGES>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(num_sms()), dim3(kGemmThreads), C::SMEM, stream, maps, a);
}

static uint64_t g_wait_limit_ns = kWaitTimeoutNs;

void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns ? ns : kWaitTimeoutNs; }
uint64_t wait_limit_ns() { return g_wait_limit_ns; }

// Token tile from the expected tokens per expert: 32 for decode-sized
// batches; 128 once experts hold more than ~48 tokens (a 128-wide MMA costs
// 68 cycles against 51 for 64 wide, so per token it is 1.5x cheaper).
int pick_ksplit(double tiles, int KT) {
  if (tiles <= 0) return 1;
  const int sms = num_sms();
  if (sms < 8) return 1;
  int best = 1;
  double best_waves = std::ceil(tiles / sms);
  for (int S = 2; S <= 8 && KT / S >= 2; ++S) {
    const double waves = std::ceil(tiles * S / sms) / S;
    if (waves < best_waves * 0.95) {  // a split must win by more than its overhead
      best = S;
      best_waves = waves;
    }
  }
  return best;
}

int pick_tile_n(double expected) {
  if (expected <= 24.0) return 32;
  if (expected <= 48.0) return 64;
  return 128;
}

cudaError_t launch_grouped_gemm(const GemmLaunch& g, cudaStream_t stream) {
  if (g.act_rows == 0 || g.E == 0) return cudaSuccess;
  const bool bfp16 = g.epilogue == MEGAMOE_EPI_BFP16;
  // BFP16 runs on weights-on-M tiles, whole K
  const int bn = bfp16 && g.tile_n == 256 ? 128 : g.tile_n;
  if (bfp16 && (g.ksplit > 1 || g.ld_out % 32 != 0)) return cudaErrorInvalidValue;
  // token-major tiles (256): 128-row boxes; otherwise BN-row boxes
  TokenMaps maps;
  const uint32_t box = bn == 256 ? 128u : static_cast<uint32_t>(bn);
  const uint64_t rows = static_cast<uint64_t>(g.act_rows);
  if (!make_codes_map(&maps.codes, g.act_codes, rows, g.K / 2, box) ||
      !make_scales_map(&maps.scales, g.act_scales, rows, g.K / 16, box))
    return cudaErrorInvalidValue;
  if (bn == 256) {  // short boxes for an expert's last tile of few rows
    if (!make_codes_map(&maps.codes32, g.act_codes, rows, g.K / 2, 32) ||
        !make_scales_map(&maps.scales32, g.act_scales, rows, g.K / 16, 32) ||
        !make_codes_map(&maps.codes64, g.act_codes, rows, g.K / 2, 64) ||
        !make_scales_map(&maps.scales64, g.act_scales, rows, g.K / 16, 64))
      return cudaErrorInvalidValue;
  } else {  // unused by weights-on-M tiles
    maps.codes32 = maps.codes64 = maps.codes;
    maps.scales32 = maps.scales64 = maps.scales;
  }
  GemmArgs a{g.w_codes,        g.w_scales, g.w_gs,     g.act_gs, g.offsets,
             g.padded_offsets, g.out,      g.ld_out,   g.out_amax, g.status,
             wait_limit_ns(),  g.E,        g.N,        g.K,          g.early_weights ? 1 : 0,
             g.ksplit,         g.partial,  g.partial_plane};
  if (bfp16)
    a.out_exp = reinterpret_cast<int8_t*>(g.out) + g.act_rows * g.ld_out * 2;
  if (g.epilogue == MEGAMOE_EPI_SILU_MUL && g.ksplit <= 1 && g.rq_arrivals) {
    if (!g.rq_codes || !g.rq_scales || !g.rq_gs || !g.out_amax) return cudaErrorInvalidValue;
    a.rq_arrivals = g.rq_arrivals;
    a.rq_codes = g.rq_codes;
    a.rq_scales = g.rq_scales;
    a.rq_gs = g.rq_gs;
  }
  if (bn == 256) {  // token-major tiles: 128 token rows x 256 weight rows
    if (g.ksplit > 1) return cudaErrorInvalidValue;
    if (g.epilogue == MEGAMOE_EPI_SILU_MUL && g.out_amax && g.zero_amax) {
      cudaError_t err = cudaMemsetAsync(g.out_amax, 0, sizeof(float), stream);
      if (err != cudaSuccess) return err;
    }
    return launch_grouped_gemm_tm(maps, a, g.epilogue, stream);
  }
  if (g.ksplit > 1) {
    if (!g.partial || bn > 64) return cudaErrorInvalidValue;
    cudaError_t err = cudaSuccess;
    if (g.epilogue == MEGAMOE_EPI_SILU_MUL) {
      if (g.out_amax && g.zero_amax) err = cudaMemsetAsync(g.out_amax, 0, sizeof(float), stream);
      if (err == cudaSuccess)
        err = bn == 32 ? launch_cfg<32, kEpiPartial2, 5>(maps, a, stream)
                       : launch_cfg<64, kEpiPartial2, 4>(maps, a, stream);
    } else {
      err = bn == 32 ? launch_cfg<32, kEpiPartial1, 8>(maps, a, stream)
                     : launch_cfg<64, kEpiPartial1, 7>(maps, a, stream);
    }
    if (err != cudaSuccess) return err;
    const int width = g.epilogue == MEGAMOE_EPI_SILU_MUL ? g.N / 2 : g.N;
    // valid rows are at most act_rows, and at most the plane's rows
    const int64_t rows = std::min<int64_t>(g.act_rows, g.partial_plane / g.N);
    const int64_t tasks = rows * (width / 4);
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((tasks + 255) / 256, num_sms() * 8));
    switch (g.epilogue) {
      case MEGAMOE_EPI_SILU_MUL:
        return launch_pdl(k_splitk_finish<MEGAMOE_EPI_SILU_MUL>, dim3(blocks), dim3(256), 0,
                          stream, g.partial, g.ksplit, g.partial_plane, g.offsets,
                          g.padded_offsets, g.E, g.N, g.out, g.ld_out, g.out_amax);
      case MEGAMOE_EPI_BF16:
        return launch_pdl(k_splitk_finish<MEGAMOE_EPI_BF16>, dim3(blocks), dim3(256), 0,
                          stream, g.partial, g.ksplit, g.partial_plane, g.offsets,
                          g.padded_offsets, g.E, g.N, g.out, g.ld_out, g.out_amax);
      default:
        return launch_pdl(k_splitk_finish<MEGAMOE_EPI_F32>, dim3(blocks), dim3(256), 0,
                          stream, g.partial, g.ksplit, g.partial_plane, g.offsets,
                          g.padded_offsets, g.E, g.N, g.out, g.ld_out, g.out_amax);
    }
  }
  if (g.epilogue == MEGAMOE_EPI_SILU_MUL) {
    if (g.out_amax && g.zero_amax) {
      cudaError_t err = cudaMemsetAsync(g.out_amax, 0, sizeof(float), stream);
      if (err != cudaSuccess) return err;
    }
    switch (bn) {
      case 32: return launch_cfg<32, MEGAMOE_EPI_SILU_MUL, 5>(maps, a, stream);
      case 64: return launch_cfg<64, MEGAMOE_EPI_SILU_MUL, 4>(maps, a, stream);
      case 128: return launch_cfg<128, MEGAMOE_EPI_SILU_MUL, 4>(maps, a, stream);
    }
  } else if (g.epilogue == MEGAMOE_EPI_BF16) {
    switch (bn) {
      case 32: return launch_cfg<32, MEGAMOE_EPI_BF16, 8>(maps, a, stream);
      case 64: return launch_cfg<64, MEGAMOE_EPI_BF16, 7>(maps, a, stream);
      case 128: return launch_cfg<128, MEGAMOE_EPI_BF16, 5>(maps, a, stream);
    }
  } else if (bfp16) {
    switch (bn) {
      case 32: return launch_cfg<32, MEGAMOE_EPI_BFP16, 9>(maps, a, stream);
      case 64: return launch_cfg<64, MEGAMOE_EPI_BFP16, 8>(maps, a, stream);
      case 128: return launch_cfg<128, MEGAMOE_EPI_BFP16, 6>(maps, a, stream);
    }
  } else {
    switch (bn) {
      case 32: return launch_cfg<32, MEGAMOE_EPI_F32, 9>(maps, a, stream);
      case 64: return launch_cfg<64, MEGAMOE_EPI_F32, 8>(maps, a, stream);
      case 128: return launch_cfg<128, MEGAMOE_EPI_F32, 6>(maps, a, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace megamoe
