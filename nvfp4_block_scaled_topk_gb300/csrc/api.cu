// C ABI of the MegaMoE library: argument checks, workspace layout and the
// forward orchestration.  No allocation, no synchronisation on the compute
// path; every launch goes to the caller's stream.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "../../include/megamoe.h"
#include "kernels.h"

using namespace megamoe;

namespace {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// NVTX range around the enqueueing of a stage (named "megamoe.<stage>"), so a
// profiler's timeline groups each stage's launches; no-ops unless a tool is
// attached.
struct StageRange {
  explicit StageRange(const char* name) { nvtxRangePushA(name); }
  ~StageRange() { nvtxRangePop(); }
};

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline megamoe_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? MEGAMOE_OK : MEGAMOE_ERR_CUDA;
}

// Workspace of megamoe_forward, every region 256-byte aligned.
struct Workspace {
  uint32_t* status;
  float* amax_x;
  float* gs_x;
  float* amax_h;
  float* gs_h;
  uint32_t* l1_arrivals;  // the fused requantisation's grid-wide arrival count
  int32_t* counts;
  int32_t* offsets;
  int32_t* padded_offsets;
  int32_t* slot_dst;
  int32_t* row_src;
  uint8_t* xq_codes;
  uint8_t* xq_sf;
  uint16_t* h;
  uint8_t* hq_codes;
  uint8_t* hq_sf;
  uint16_t* y;     // the L2 output: a BFP16 [rows, d] matrix (int16 values ...
  int8_t* y_exp;   // ... then the exponents [rows, d / 32])
  float* partial;  // split-K planes of L1
  int32_t* r_ids;  // router outputs of megamoe_forward_from_logits [T, k]
  float* r_w;
  int32_t* route_hist;  // per-block expert histograms of the multi-block routing
  int ks1, ks2;    // split-K of L1 and L2 (1 = none)
  int64_t rows;    // padded-row capacity
  size_t bytes;
};

// Token tile of the forward's grouped GEMMs: chosen from the expected tokens
// per expert; the MEGAMOE_TILE_N environment variable (32/64/128/256)
// overrides.
int tile_n_setting(double expected) {
  static const int forced = [] {
    const char* e = std::getenv("MEGAMOE_TILE_N");
    return (e && *e) ? std::atoi(e) : 0;
  }();
  if (forced == 32 || forced == 64 || forced == 128 || forced == 256) return forced;
  return pick_tile_n(expected);
}

// Split-K of a grouped GEMM of about `tiles` tiles: chosen by pick_ksplit;
// the MEGAMOE_KSPLIT environment variable (1-8) overrides.
int ksplit_setting(double tiles, int KT, int tile_n) {
  static const int forced = [] {
    const char* e = std::getenv("MEGAMOE_KSPLIT");
    return (e && *e) ? std::atoi(e) : 0;
  }();
  if (tile_n > 64 || KT < 4) return 1;
  if (forced >= 1 && forced <= 8) return std::min(forced, KT / 2);
  return pick_ksplit(tiles, KT);
}

// The forward's split-K of L1 and L2.  Measured on the MegaMoE decode
// shapes, splitting did not shorten the grouped GEMMs (their time at these
// sizes is start-up latency and the weight stream, not idle SMs) while the
// finishing kernels cost more, so the forward splits only when the
// MEGAMOE_KSPLIT environment variable asks for it.
void forward_splits(int T, int k, int E, int d, int I, int* ks1, int* ks2) {
  *ks1 = *ks2 = 1;
  static const int forced = [] {
    const char* e = std::getenv("MEGAMOE_KSPLIT");
    return (e && *e) ? std::atoi(e) : 0;
  }();
  const int64_t slots = static_cast<int64_t>(T) * k;
  if (slots == 0 || forced < 2) return;
  const int tile_n = tile_n_setting(static_cast<double>(slots) / E);
  *ks1 = ksplit_setting(0.0, d / 256, tile_n);
  // L2 writes the BFP16 y, whose exponent groups need whole-K sums: not split
  *ks2 = 1;
}

Workspace carve(void* base, int T, int k, int E, int d, int I, int pad) {
  Workspace w{};
  const int64_t rows = megamoe_max_padded_rows(T, k, E, pad);
  w.rows = rows;
  size_t off = 0;
  auto take = [&](size_t bytes) -> uint8_t* {
    uint8_t* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
    off = round_up(off + bytes, 256);
    return p;
  };
  uint8_t* hdr = take(256);
  if (hdr) {
    w.status = reinterpret_cast<uint32_t*>(hdr);
    w.amax_x = reinterpret_cast<float*>(hdr + 4);
    w.gs_x = reinterpret_cast<float*>(hdr + 8);
    w.amax_h = reinterpret_cast<float*>(hdr + 12);
    w.gs_h = reinterpret_cast<float*>(hdr + 16);
    w.l1_arrivals = reinterpret_cast<uint32_t*>(hdr + 20);
  }
  w.counts = reinterpret_cast<int32_t*>(take(4 * static_cast<size_t>(E)));
  w.offsets = reinterpret_cast<int32_t*>(take(4 * static_cast<size_t>(E + 1)));
  w.padded_offsets = reinterpret_cast<int32_t*>(take(4 * static_cast<size_t>(E + 1)));
  w.slot_dst = reinterpret_cast<int32_t*>(take(4 * static_cast<size_t>(T) * k));
  w.row_src = reinterpret_cast<int32_t*>(take(4 * static_cast<size_t>(rows)));
  w.xq_codes = take(static_cast<size_t>(rows) * (d / 2));
  w.xq_sf = take(static_cast<size_t>(rows) * (d / 16));
  w.h = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(rows) * I * 2));
  w.hq_codes = take(static_cast<size_t>(rows) * (I / 2));
  w.hq_sf = take(static_cast<size_t>(rows) * (I / 16));
  uint8_t* y = take(MEGAMOE_BFP16_BYTES(rows, d));
  w.y = reinterpret_cast<uint16_t*>(y);
  w.y_exp = y ? reinterpret_cast<int8_t*>(y + static_cast<size_t>(rows) * d * 2) : nullptr;
  forward_splits(T, k, E, d, I, &w.ks1, &w.ks2);
  const size_t slots = static_cast<size_t>(T) * k;
  const size_t p1 = w.ks1 > 1 ? w.ks1 * slots * 2 * I : 0;
  w.partial = reinterpret_cast<float*>(take(p1 * 4));
  w.r_ids = reinterpret_cast<int32_t*>(take(4 * slots));
  w.r_w = reinterpret_cast<float*>(take(4 * slots));
  w.route_hist = reinterpret_cast<int32_t*>(
      take(slots >= static_cast<size_t>(kRouteMultiMinSlots)
               ? 4 * static_cast<size_t>(kRouteMaxBlocks) * E
               : 0));
  w.bytes = off;
  return w;
}

// The L1 GEMM's tiles: where 128-token tiles are chosen, token-major tiles
// (128 tokens x the gate and up rows of 128 features in one MMA) instead;
// measured on the 4096- and 16384-token MegaMoE batches they take 5-6 % off
// the L1 GEMM, while for the L2 GEMM (8 K steps per tile) token-major tiles
// were slower, so L2 keeps the tile of tile_n_setting.
int l1_tile(int tile_n) { return tile_n == 128 ? 256 : tile_n; }

megamoe_status check_route_args(int T, int k, int E, int pad) {
  if (T < 0 || k < 1 || E < 1 || pad < 1) return MEGAMOE_ERR_INVALID_ARG;
  if (E > MEGAMOE_MAX_EXPERTS || k > MEGAMOE_MAX_TOPK) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(T) * k > (int64_t{1} << 30)) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  // padded offsets and row indices of the kernels are int32
  if (megamoe_max_padded_rows(T, k, E, pad) >= (int64_t{1} << 31))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return MEGAMOE_OK;
}

}  // namespace

namespace megamoe {

megamoe_status check_forward_shape(const megamoe_weights* w, int T, int k, int pad) {
  if (!w) return MEGAMOE_ERR_INVALID_ARG;
  const int E = w->num_experts, d = w->hidden, I = w->intermediate;
  megamoe_status st = check_route_args(T, k, E, pad);
  if (st != MEGAMOE_OK) return st;
  if (d <= 0 || I <= 0) return MEGAMOE_ERR_INVALID_ARG;
  if (d % 256 != 0 || I % 256 != 0 || pad % 32 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (!w->w13_codes || !w->w13_scales || !w->w13_gs || !w->w2_codes || !w->w2_scales ||
      !w->w2_gs)
    return MEGAMOE_ERR_INVALID_ARG;
  if (!aligned(w->w13_codes, 16) || !aligned(w->w2_codes, 16) || !aligned(w->w13_scales, 16) ||
      !aligned(w->w2_scales, 16))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return MEGAMOE_OK;
}

megamoe_status check_forward_args(const megamoe_weights* w, const uint16_t* x,
                                  const int32_t* topk_ids, const float* topk_weights, int T, int k,
                                  int pad, const uint16_t* out, bool router) {
  megamoe_status st = check_forward_shape(w, T, k, pad);
  if (st != MEGAMOE_OK) return st;
  if (T > 0 && (!x || (!router && (!topk_ids || !topk_weights)) || !out))
    return MEGAMOE_ERR_INVALID_ARG;
  if ((x && !aligned(x, 16)) || (out && !aligned(out, 8))) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return MEGAMOE_OK;
}

}  // namespace megamoe

extern "C" {

const char* megamoe_status_string(megamoe_status s) {
  switch (s) {
    case MEGAMOE_OK: return "ok";
    case MEGAMOE_ERR_INVALID_ARG: return "invalid argument";
    case MEGAMOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MEGAMOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MEGAMOE_ERR_CUDA: return "CUDA error";
    case MEGAMOE_ERR_DEVICE_STATUS: return "device reported an error";
  }
  return "unknown status";
}

int64_t megamoe_max_padded_rows(int T, int k, int E, int pad) {
  if (T < 0 || k < 1 || E < 1 || pad < 1) return 0;
  const int64_t slots = static_cast<int64_t>(T) * k;
  return slots + std::min<int64_t>(E, slots) * (pad - 1);
}

megamoe_status megamoe_route_permute(const int32_t* topk_ids, int T, int k, int E, int pad,
                                     int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                                     int32_t* row_src, int64_t row_capacity, int32_t* slot_dst,
                                     uint32_t* status, megamoe_stream_t stream) {
  megamoe_status st = check_route_args(T, k, E, pad);
  if (st != MEGAMOE_OK) return st;
  if (!counts || !offsets || !padded_offsets || (T > 0 && (!topk_ids || !slot_dst)))
    return MEGAMOE_ERR_INVALID_ARG;
  const int64_t need = megamoe_max_padded_rows(T, k, E, pad);
  if (row_capacity < need || (row_capacity > 0 && !row_src)) return MEGAMOE_ERR_INVALID_ARG;
  return cuda_status(launch_route(topk_ids, T * k, E, pad, counts, offsets, padded_offsets,
                                  row_src, row_capacity, slot_dst, status, nullptr, 0,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

megamoe_status megamoe_quantize_nvfp4(const uint16_t* x, int64_t rows, int K, int64_t ld,
                                      const int32_t* slot_dst, int k, const int32_t* row_src,
                                      const int32_t* live_rows, int64_t out_rows,
                                      const float* amax_in, float* amax_out, float* gs_out,
                                      uint8_t* codes, uint8_t* scales, int scale_layout,
                                      uint32_t* status, megamoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rows < 0 || out_rows < 0 || K <= 0 || ld < K) return MEGAMOE_ERR_INVALID_ARG;
  if (scale_layout != MEGAMOE_SCALES_ROWMAJOR && scale_layout != MEGAMOE_SCALES_MMA)
    return MEGAMOE_ERR_INVALID_ARG;
  if (K % 64 != 0 || ld % 8 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (!gs_out || (!amax_in && !amax_out)) return MEGAMOE_ERR_INVALID_ARG;
  if (slot_dst) {
    if (k < 1 || k > MEGAMOE_MAX_TOPK) return MEGAMOE_ERR_INVALID_ARG;
  } else if (rows < out_rows) {
    return MEGAMOE_ERR_INVALID_ARG;
  }
  if ((rows > 0 && !x) || (out_rows > 0 && (!codes || !scales))) return MEGAMOE_ERR_INVALID_ARG;
  if (x && !aligned(x, 16)) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if ((codes && !aligned(codes, 16)) || (scales && !aligned(scales, 4)))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  const float* amax = amax_in;
  if (!amax_in) {
    cudaError_t e = launch_amax(x, rows, K, ld, amax_out, status, true, s);
    if (e != cudaSuccess) return MEGAMOE_ERR_CUDA;
    amax = amax_out;
  } else if (amax_out && amax_out != amax_in) {
    if (cudaMemcpyAsync(amax_out, amax_in, sizeof(float), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return MEGAMOE_ERR_CUDA;
  }
  return cuda_status(launch_quant(x, rows, K, ld, slot_dst, k, row_src, live_rows, out_rows, amax,
                                  gs_out, codes, scales, scale_layout, s));
}

megamoe_status megamoe_swizzle_scales(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                                      megamoe_stream_t stream) {
  if (rows < 0 || K <= 0) return MEGAMOE_ERR_INVALID_ARG;
  if (K % 64 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (rows > 0 && (!src || !dst)) return MEGAMOE_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned(src, 4) || !aligned(dst, 4))) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_swizzle(src, rows, K, dst, reinterpret_cast<cudaStream_t>(stream)));
}

megamoe_status megamoe_pack_weight_codes(const uint8_t* src, int64_t rows, int K, int half_rows,
                                         uint8_t* dst, megamoe_stream_t stream) {
  if (rows < 0 || K <= 0 || half_rows < 0) return MEGAMOE_ERR_INVALID_ARG;
  if (K % 256 != 0 || rows % 128 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (half_rows > 0 && (half_rows % 128 != 0 || rows % (2 * static_cast<int64_t>(half_rows))))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (rows > 0 && (!src || !dst)) return MEGAMOE_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned(src, 16) || !aligned(dst, 16))) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(
      launch_pack(src, rows, K, half_rows, dst, reinterpret_cast<cudaStream_t>(stream)));
}

megamoe_status megamoe_grouped_gemm(const uint8_t* act_codes, const uint8_t* act_scales,
                                    const float* act_gs, int64_t act_rows, const uint8_t* w_codes,
                                    const uint8_t* w_scales, const float* w_gs, int E, int N,
                                    int K, const int32_t* offsets, const int32_t* padded_offsets,
                                    int epilogue, void* out, int64_t ld_out, float* out_amax,
                                    int tile_n, double expected_tokens, uint32_t* status,
                                    megamoe_stream_t stream) {
  if (act_rows < 0 || E < 1 || N <= 0 || K <= 0) return MEGAMOE_ERR_INVALID_ARG;
  if (epilogue != MEGAMOE_EPI_F32 && epilogue != MEGAMOE_EPI_SILU_MUL &&
      epilogue != MEGAMOE_EPI_BF16 && epilogue != MEGAMOE_EPI_BFP16)
    return MEGAMOE_ERR_INVALID_ARG;
  if (E > MEGAMOE_MAX_EXPERTS || K % 256 != 0 || N % (epilogue == MEGAMOE_EPI_SILU_MUL ? 256 : 128))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(E) * N * (K / 256) >= (int64_t{1} << 31) ||
      act_rows >= (int64_t{1} << 31))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (tile_n != 0 && tile_n != 32 && tile_n != 64 && tile_n != 128 && tile_n != 256)
    return MEGAMOE_ERR_INVALID_ARG;
  // token-major tiles hold 256 weight rows (128 gate + 128 up features for SILU_MUL)
  if (tile_n == 256 && N % 256 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  const int width = epilogue == MEGAMOE_EPI_SILU_MUL ? N / 2 : N;
  if (ld_out < width) return MEGAMOE_ERR_INVALID_ARG;
  // output rows start on 16-byte boundaries: the epilogue stores 16-byte vectors
  // (BFP16: whole 32-column exponent groups)
  if (ld_out % (epilogue == MEGAMOE_EPI_F32 ? 4 : epilogue == MEGAMOE_EPI_BFP16 ? 32 : 8) != 0)
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (!w_codes || !w_scales || !w_gs || !offsets || !padded_offsets ||
      (act_rows > 0 && (!act_codes || !act_scales || !act_gs || !out)))
    return MEGAMOE_ERR_INVALID_ARG;
  if (epilogue == MEGAMOE_EPI_SILU_MUL && !out_amax) return MEGAMOE_ERR_INVALID_ARG;
  if (!aligned(w_codes, 16) || !aligned(w_scales, 16) || (act_codes && !aligned(act_codes, 16)) ||
      (act_scales && !aligned(act_scales, 16)) || (out && !aligned(out, 16)))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  GemmLaunch g{};
  g.act_codes = act_codes;
  g.act_scales = act_scales;
  g.act_gs = act_gs;
  g.act_rows = act_rows;
  g.w_codes = w_codes;
  g.w_scales = w_scales;
  g.w_gs = w_gs;
  g.E = E;
  g.N = N;
  g.K = K;
  g.offsets = offsets;
  g.padded_offsets = padded_offsets;
  g.epilogue = epilogue;
  g.out = out;
  g.ld_out = ld_out;
  g.out_amax = out_amax;
  // the automatic choice is the forward's: token-major tiles for the gate+up
  // GEMM where 128-token tiles would be chosen
  g.tile_n = tile_n ? tile_n
                    : (epilogue == MEGAMOE_EPI_SILU_MUL ? l1_tile(pick_tile_n(expected_tokens))
                                                        : pick_tile_n(expected_tokens));
  g.status = status;
  return cuda_status(launch_grouped_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

megamoe_status megamoe_combine(const float* y, int64_t ld_y, const int32_t* slot_dst,
                               const float* topk_weights, int T, int k, int d, uint16_t* out,
                               megamoe_stream_t stream) {
  if (T < 0 || k < 1 || k > MEGAMOE_MAX_TOPK || d <= 0 || ld_y < d) return MEGAMOE_ERR_INVALID_ARG;
  if (d % 4 != 0 || ld_y % 4 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!y || !slot_dst || !topk_weights || !out)) return MEGAMOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned(y, 16) || !aligned(out, 8))) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(
      launch_combine(y, nullptr, ld_y, 0, slot_dst, topk_weights, T, k, d, out, false,
                     reinterpret_cast<cudaStream_t>(stream)));
}

megamoe_status megamoe_combine_bfp16(const void* y, int64_t ld_y, int64_t y_rows,
                                     const int32_t* slot_dst, const float* topk_weights, int T,
                                     int k, int d, uint16_t* out, megamoe_stream_t stream) {
  if (T < 0 || k < 1 || k > MEGAMOE_MAX_TOPK || d <= 0 || ld_y < d || y_rows < 0)
    return MEGAMOE_ERR_INVALID_ARG;
  if (d % 32 != 0 || ld_y % 32 != 0) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!y || !slot_dst || !topk_weights || !out)) return MEGAMOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned(y, 16) || !aligned(out, 8))) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  const int8_t* y_exp = static_cast<const int8_t*>(y) + y_rows * ld_y * 2;
  return cuda_status(launch_combine(y, y_exp, ld_y, y_rows, slot_dst, topk_weights, T, k, d, out,
                                    false, reinterpret_cast<cudaStream_t>(stream)));
}

size_t megamoe_workspace_size(int T, int k, int E, int d, int I, int pad) {
  if (T < 0 || k < 1 || E < 1 || d <= 0 || I <= 0 || pad < 1) return 0;
  return carve(nullptr, T, k, E, d, I, pad).bytes;
}

}  // extern "C"

namespace {

// The forward; with `router` the ids and weights are computed here from the
// router logits (into the workspace) instead of being passed in.
// Steps 0-4 of the forward: (router,) route, amax of x, quantise x into its
// routed rows, L1 gate+up grouped GEMM with SiLU(gate)*up -> bf16 h and
// amax(h).  `expected` is the caller's expected rows per expert (the token
// tile's choice).
cudaError_t forward_l1(const megamoe_weights* w, const uint16_t* x, const int32_t* topk_ids,
                       int T, int k, int pad, const Workspace& wk, cudaStream_t s,
                       RouterArgs* router, int tile_n, bool fuse_requant) {
  const int E = w->num_experts, d = w->hidden, I = w->intermediate;
  cudaError_t e = cudaSuccess;
  // 0-3. (router,) route (its first act clears the status word and the amax
  //      accumulators), amax of x, quantise x into its routed rows.  Padding
  //      rows are left as they are: each output column of the grouped GEMM
  //      depends on one token row, and columns of padding rows are never
  //      stored.  Small batches route (and run the router) and take the amax
  //      in one thread block.
  if (prologue_fits(T, d)) {
    StageRange r("megamoe.route+amax_x");
    e = launch_prologue(topk_ids, T, k, E, pad, wk.counts, wk.offsets, wk.padded_offsets,
                        wk.row_src, wk.rows, wk.slot_dst, wk.status, wk.status, 6, x, d,
                        wk.amax_x, s, router);
  } else {
    if (router) {
      StageRange r("megamoe.router");
      e = launch_router(router->logits, T, router->n_logits, router->ld, router->bias,
                        router->k_routed, router->shared, wk.r_ids, wk.r_w, s);
    }
    if (e != cudaSuccess) return e;
    StageRange r("megamoe.route");
    e = launch_route(topk_ids, T * k, E, pad, wk.counts, wk.offsets, wk.padded_offsets,
                     wk.row_src, wk.rows, wk.slot_dst, wk.status, wk.status, 6, s,
                     wk.route_hist);
    if (e != cudaSuccess) return e;
    StageRange ra("megamoe.amax_x");
    e = launch_amax(x, T, d, d, wk.amax_x, wk.status, false, s);
  }
  if (e != cudaSuccess) return e;
  {
    StageRange r("megamoe.quant_x");
    e = launch_quant(x, T, d, d, wk.slot_dst, k, nullptr, wk.padded_offsets + E, wk.rows,
                     wk.amax_x, wk.gs_x, wk.xq_codes, wk.xq_sf, MEGAMOE_SCALES_ROWMAJOR, s);
  }
  if (e != cudaSuccess) return e;
  // 4. L1 gate+up grouped GEMM, SiLU(gate)*up -> bf16 h, amax(h)
  GemmLaunch g{};
  g.act_codes = wk.xq_codes;
  g.act_scales = wk.xq_sf;
  g.act_gs = wk.gs_x;
  g.act_rows = wk.rows;
  g.w_codes = w->w13_codes;
  g.w_scales = w->w13_scales;
  g.w_gs = w->w13_gs;
  g.E = E;
  g.N = 2 * I;
  g.K = d;
  g.offsets = wk.offsets;
  g.padded_offsets = wk.padded_offsets;
  g.epilogue = MEGAMOE_EPI_SILU_MUL;
  g.out = wk.h;
  g.ld_out = I;
  g.out_amax = wk.amax_h;
  g.tile_n = tile_n;
  g.status = wk.status;
  g.zero_amax = false;
  // The kernel reads the routing offsets before its grid-dependency wait
  // (its tile schedule and first weight stages start early).  Sound only with
  // a kernel in between: the quantiser lets this kernel launch after its own
  // wait, which returns once the routing kernel has completed and its writes
  // are visible.  Launched straight after the routing, it could read offsets
  // still being written.
  g.early_weights = true;
  g.ksplit = wk.ks1;
  g.partial = wk.partial;
  g.partial_plane = static_cast<int64_t>(T) * k * 2 * I;
  if (fuse_requant) {  // 5. (fused) requantise h inside the L1 kernel
    g.rq_arrivals = wk.l1_arrivals;
    g.rq_codes = wk.hq_codes;
    g.rq_scales = wk.hq_sf;
    g.rq_gs = wk.gs_h;
  }
  StageRange r("megamoe.l1_gemm");
  return launch_grouped_gemm(g, s);
}

// Whether the forward requantises h inside the L1 kernel (behind a grid-wide
// arrival count) instead of in its own kernel after it: only when asked
// (megamoe_set_fused_requant) and the L1 GEMM is not split along K.
// Measured on GB300 the separate kernel is faster: 3.72 against 4.01 ms at
// 16384 tokens, 1.20 against 1.28 ms at 4096, 182 against 190 us at 8 --
// CTAs that finish their last tile early exit and free their SM for the next
// kernel's start, while behind the grid-wide wait every CTA holds its SM
// until the slowest is done.
bool g_fused_requant = false;
bool requant_fused(const Workspace& wk) { return g_fused_requant && wk.ks1 <= 1; }

// Steps 5-7: requantise h with gs from the amax(h) held in the workspace, L2
// down grouped GEMM -> BFP16 y, top-k weighted combine (bf16 out, or the fp32
// sum before its rounding with out_f32).
cudaError_t forward_l2(const megamoe_weights* w, const float* topk_weights, int T, int k,
                       void* out, bool out_f32, const Workspace& wk, cudaStream_t s,
                       int tile_n, bool requant_done) {
  const int E = w->num_experts, d = w->hidden, I = w->intermediate;
  cudaError_t e = cudaSuccess;
  // 5. requantise the valid rows of h with gs from amax(h) (slot by slot),
  //    unless the L1 kernel already did
  if (!requant_done) {
    StageRange r("megamoe.requant_h");
    e = launch_quant(wk.h, static_cast<int64_t>(T) * k, I, I, wk.slot_dst, 1, nullptr,
                     wk.padded_offsets + E, wk.rows, wk.amax_h, wk.gs_h, wk.hq_codes, wk.hq_sf,
                     MEGAMOE_SCALES_ROWMAJOR, s, /*slot_rows=*/true);
    if (e != cudaSuccess) return e;
  }
  // 6. L2 down grouped GEMM -> BFP16 y
  GemmLaunch g{};
  g.act_codes = wk.hq_codes;
  g.act_scales = wk.hq_sf;
  g.act_gs = wk.gs_h;
  g.act_rows = wk.rows;
  g.w_codes = w->w2_codes;
  g.w_scales = w->w2_scales;
  g.w_gs = w->w2_gs;
  g.E = E;
  g.N = d;
  g.K = I;
  g.offsets = wk.offsets;
  g.padded_offsets = wk.padded_offsets;
  g.epilogue = MEGAMOE_EPI_BFP16;
  g.out = wk.y;
  g.ld_out = d;
  g.out_amax = nullptr;
  g.tile_n = tile_n;
  g.status = wk.status;
  g.early_weights = true;
  {
    StageRange r("megamoe.l2_gemm");
    e = launch_grouped_gemm(g, s);
  }
  if (e != cudaSuccess) return e;
  // 7. top-k weighted combine
  StageRange r("megamoe.combine");
  return launch_combine(wk.y, wk.y_exp, d, wk.rows, wk.slot_dst, topk_weights, T, k, d, out,
                        out_f32, s);
}

// The forward; with `router` the ids and weights are computed here from the
// router logits (into the workspace) instead of being passed in.
megamoe_status forward_impl(const megamoe_weights* w, const uint16_t* x, const int32_t* topk_ids,
                            const float* topk_weights, int T, int k, int pad, uint16_t* out,
                            void* ws, size_t ws_bytes, cudaStream_t s, RouterArgs* router) {
  megamoe_status st =
      megamoe::check_forward_args(w, x, topk_ids, topk_weights, T, k, pad, out, router != nullptr);
  if (st != MEGAMOE_OK) return st;
  if (!ws || !aligned(ws, 256)) return MEGAMOE_ERR_INVALID_ARG;
  const int E = w->num_experts, d = w->hidden, I = w->intermediate;
  Workspace wk = carve(ws, T, k, E, d, I, pad);
  if (ws_bytes < wk.bytes) return MEGAMOE_ERR_WORKSPACE_TOO_SMALL;

  if (T == 0) return cudaMemsetAsync(wk.status, 0, 256, s) == cudaSuccess ? MEGAMOE_OK
                                                                         : MEGAMOE_ERR_CUDA;
  const int tile_n = tile_n_setting(static_cast<double>(T) * k / E);
  StageRange whole("megamoe.forward");
  if (router) {  // the ids and weights land in the workspace
    router->ids_out = wk.r_ids;
    router->w_out = wk.r_w;
    topk_ids = wk.r_ids;
    topk_weights = wk.r_w;
  }
  const bool fused = requant_fused(wk);
  cudaError_t e = forward_l1(w, x, topk_ids, T, k, pad, wk, s, router, l1_tile(tile_n), fused);
  if (e == cudaSuccess) e = forward_l2(w, topk_weights, T, k, out, false, wk, s, tile_n, fused);
  return cuda_status(e);
}

// Checks and workspace of one expert-parallel shard (the shard's weights hold
// its experts only; ids are global).
megamoe_status ep_setup(const megamoe_weights* w, int T, int k, int expert_base,
                        int num_experts_total, int pad, void* ws, size_t ws_bytes, Workspace* wk) {
  megamoe_status st = megamoe::check_forward_shape(w, T, k, pad);
  if (st != MEGAMOE_OK) return st;
  if (expert_base < 0 || num_experts_total < 1 || num_experts_total > MEGAMOE_MAX_EXPERTS ||
      static_cast<int64_t>(expert_base) + w->num_experts > num_experts_total)
    return MEGAMOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return MEGAMOE_ERR_INVALID_ARG;
  *wk = carve(ws, T, k, w->num_experts, w->hidden, w->intermediate, pad);
  if (ws_bytes < wk->bytes) return MEGAMOE_ERR_WORKSPACE_TOO_SMALL;
  return MEGAMOE_OK;
}

// Token tile of a shard: the expected rows per expert of the whole layer
// (each shard holds E / G experts and receives about T k / G of the slots).
int ep_tile_n(int T, int k, int num_experts_total) {
  return tile_n_setting(static_cast<double>(T) * k / num_experts_total);
}

}  // namespace

extern "C" {

megamoe_status megamoe_forward(const megamoe_weights* w, const uint16_t* x,
                               const int32_t* topk_ids, const float* topk_weights, int T, int k,
                               int pad, uint16_t* out, void* ws, size_t ws_bytes,
                               megamoe_stream_t stream) {
  return forward_impl(w, x, topk_ids, topk_weights, T, k, pad, out, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream), nullptr);
}

megamoe_status megamoe_ep_forward_begin(const megamoe_weights* w_shard, const uint16_t* x,
                                        const int32_t* topk_ids, int T, int k, int expert_base,
                                        int num_experts_total, int pad, void* ws, size_t ws_bytes,
                                        megamoe_stream_t stream) {
  Workspace wk{};
  megamoe_status st =
      ep_setup(w_shard, T, k, expert_base, num_experts_total, pad, ws, ws_bytes, &wk);
  if (st != MEGAMOE_OK) return st;
  if (T > 0 && (!x || !topk_ids)) return MEGAMOE_ERR_INVALID_ARG;
  if (x && !aligned(x, 16)) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) return cudaMemsetAsync(wk.status, 0, 256, s) == cudaSuccess ? MEGAMOE_OK
                                                                         : MEGAMOE_ERR_CUDA;
  // global ids -> this shard's local ids (other shards' experts skipped)
  cudaError_t e = launch_ep_remap(topk_ids, static_cast<int64_t>(T) * k, expert_base,
                                  w_shard->num_experts, num_experts_total, wk.r_ids, s);
  if (e == cudaSuccess)
    // the shard's h is requantised only after the amax(h) exchange
    e = forward_l1(w_shard, x, wk.r_ids, T, k, pad, wk, s, nullptr,
                   l1_tile(ep_tile_n(T, k, num_experts_total)), false);
  return cuda_status(e);
}

megamoe_status megamoe_ep_forward_end(const megamoe_weights* w_shard, const float* topk_weights,
                                      int T, int k, int num_experts_total, int pad,
                                      float* out_partial, void* ws, size_t ws_bytes,
                                      megamoe_stream_t stream) {
  Workspace wk{};
  megamoe_status st = ep_setup(w_shard, T, k, 0, num_experts_total, pad, ws, ws_bytes, &wk);
  if (st != MEGAMOE_OK) return st;
  if (T > 0 && (!topk_weights || !out_partial)) return MEGAMOE_ERR_INVALID_ARG;
  if (out_partial && !aligned(out_partial, 16)) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MEGAMOE_OK;
  return cuda_status(forward_l2(w_shard, topk_weights, T, k, out_partial, true, wk,
                                reinterpret_cast<cudaStream_t>(stream),
                                ep_tile_n(T, k, num_experts_total), false));
}

megamoe_status megamoe_forward_scan_stages(const megamoe_weights* w, int T, int k, int pad,
                                           const uint16_t* out, const void* ws, size_t ws_bytes,
                                           uint32_t* flags, megamoe_stream_t stream) {
  megamoe_status st = megamoe::check_forward_shape(w, T, k, pad);
  if (st != MEGAMOE_OK) return st;
  if (!ws || !aligned(ws, 256) || !flags || (T > 0 && !out)) return MEGAMOE_ERR_INVALID_ARG;
  if (out && !aligned(out, 16)) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  Workspace wk = carve(const_cast<void*>(ws), T, k, w->num_experts, w->hidden, w->intermediate,
                       pad);
  if (ws_bytes < wk.bytes) return MEGAMOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) return cuda_status(cudaMemsetAsync(flags, 0, sizeof(uint32_t), s));
  return cuda_status(launch_stage_scan(wk.row_src, wk.padded_offsets + w->num_experts, wk.xq_sf,
                                       wk.h, wk.hq_sf, wk.y_exp, out, T, w->hidden, w->intermediate,
                                       flags, s));
}

megamoe_status megamoe_round_bf16(const float* in, int64_t n, uint16_t* out,
                                  megamoe_stream_t stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return MEGAMOE_ERR_INVALID_ARG;
  if (n % 4 != 0 || (in && !aligned(in, 16)) || (out && !aligned(out, 8)))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_round_bf16(in, n, out, reinterpret_cast<cudaStream_t>(stream)));
}

megamoe_status megamoe_forward_from_logits(const megamoe_weights* w, const uint16_t* x,
                                           const float* logits, int64_t ld_logits,
                                           const float* bias, int n_logits, int k,
                                           int shared_expert, int T, int pad, uint16_t* out,
                                           void* ws, size_t ws_bytes, megamoe_stream_t stream) {
  if (!w || n_logits < 1 || n_logits > w->num_experts || ld_logits < n_logits || k < 1 ||
      k > n_logits)
    return MEGAMOE_ERR_INVALID_ARG;
  if (shared_expert >= 0 && (shared_expert < n_logits || shared_expert >= w->num_experts))
    return MEGAMOE_ERR_INVALID_ARG;
  if (T > 0 && !logits) return MEGAMOE_ERR_INVALID_ARG;
  if ((logits && !aligned(logits, 4)) || (bias && !aligned(bias, 4)))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  const int k_out = k + (shared_expert >= 0 ? 1 : 0);
  if (k_out > MEGAMOE_MAX_TOPK) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  RouterArgs r;
  r.logits = logits;
  r.ld = ld_logits;
  r.bias = bias;
  r.n_logits = n_logits;
  r.k_routed = k;
  r.shared = shared_expert;
  return forward_impl(w, x, nullptr, nullptr, T, k_out, pad, out, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream), &r);
}

void megamoe_set_wait_limit_ns(uint64_t ns) { set_wait_limit_ns(ns); }

void megamoe_set_fused_requant(int enable) { g_fused_requant = enable != 0; }

megamoe_status megamoe_router_topk(const float* logits, int64_t T, int E, int64_t ld_logits,
                                   const float* bias, int k, int shared_expert,
                                   int32_t* topk_ids, float* topk_weights,
                                   megamoe_stream_t stream) {
  if (T < 0 || E < 1 || ld_logits < E || k < 1 || k > MEGAMOE_MAX_TOPK || k > E)
    return MEGAMOE_ERR_INVALID_ARG;
  if (E > MEGAMOE_MAX_EXPERTS || T >= (int64_t{1} << 40)) return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!logits || !topk_ids || !topk_weights)) return MEGAMOE_ERR_INVALID_ARG;
  if ((logits && !aligned(logits, 4)) || (bias && !aligned(bias, 4)) ||
      (topk_ids && !aligned(topk_ids, 4)) || (topk_weights && !aligned(topk_weights, 4)))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(launch_router(logits, T, E, ld_logits, bias, k, shared_expert, topk_ids,
                                   topk_weights, reinterpret_cast<cudaStream_t>(stream)));
}

static size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// The dense linear's split-K, from its shape (one group of T rows).
static int linear_ksplit(int64_t T, int K, int N) {
  const int tile_n = tile_n_setting(static_cast<double>(T));
  const double tiles = std::ceil(static_cast<double>(T) / tile_n) * (N / 128);
  return ksplit_setting(tiles, K / 256, tile_n);
}

size_t megamoe_linear_workspace_size(int64_t T, int K, int N) {
  if (T < 0 || K <= 0 || N <= 0) return 0;
  const int S = linear_ksplit(T, K, N);
  return 256 + align256(static_cast<size_t>(T) * (K / 2)) + align256(static_cast<size_t>(T) * (K / 16)) +
         (S > 1 ? align256(static_cast<size_t>(S) * T * N * 4) : 0);
}

megamoe_status megamoe_linear_nvfp4(const uint16_t* x, int64_t T, int K, int64_t ld_x,
                                    const uint8_t* w_codes, const uint8_t* w_scales,
                                    const float* w_gs, int N, int out_dtype, void* out,
                                    int64_t ld_out, void* ws, size_t ws_bytes,
                                    megamoe_stream_t stream) {
  if (T < 0 || K <= 0 || N <= 0 || ld_x < K || ld_out < N) return MEGAMOE_ERR_INVALID_ARG;
  if (out_dtype != MEGAMOE_EPI_BF16 && out_dtype != MEGAMOE_EPI_F32) return MEGAMOE_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 128 != 0 || ld_x % 8 != 0 ||
      ld_out % (out_dtype == MEGAMOE_EPI_F32 ? 4 : 8) != 0)
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (T >= (int64_t{1} << 31) || static_cast<int64_t>(N) * (K / 256) >= (int64_t{1} << 31))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (!w_codes || !w_scales || !w_gs || !ws || (T > 0 && (!x || !out)))
    return MEGAMOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || !aligned(w_codes, 16) || !aligned(w_scales, 16) ||
      (x && !aligned(x, 16)) || (out && !aligned(out, 16)))
    return MEGAMOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < megamoe_linear_workspace_size(T, K, N)) return MEGAMOE_ERR_WORKSPACE_TOO_SMALL;
  if (T == 0) return MEGAMOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* amax = reinterpret_cast<float*>(base);
  float* gs = reinterpret_cast<float*>(base + 4);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + 8);
  int32_t* groups = reinterpret_cast<int32_t*>(base + 16);  // offsets[2], padded_offsets[2]
  uint8_t* codes = base + 256;
  uint8_t* scales = codes + align256(static_cast<size_t>(T) * (K / 2));
  float* partial = reinterpret_cast<float*>(scales + align256(static_cast<size_t>(T) * (K / 16)));
  // 1. status, group offsets, amax (one block when x is small, else k_amax)
  cudaError_t e = launch_linear_prologue(x, T, K, ld_x, amax, status, groups, s);
  if (e == cudaSuccess && !linear_prologue_full_amax(T, K))
    e = launch_amax(x, T, K, ld_x, amax, status, false, s);
  // 2. x -> NVFP4 with gs = 2688 / amax
  if (e == cudaSuccess)
    e = launch_quant(x, T, K, ld_x, nullptr, 1, nullptr, nullptr, T, amax, gs, codes, scales,
                     MEGAMOE_SCALES_ROWMAJOR, s);
  if (e != cudaSuccess) return MEGAMOE_ERR_CUDA;
  // 3. the one-group GEMM
  GemmLaunch g{};
  g.act_codes = codes;
  g.act_scales = scales;
  g.act_gs = gs;
  g.act_rows = T;
  g.w_codes = w_codes;
  g.w_scales = w_scales;
  g.w_gs = w_gs;
  g.E = 1;
  g.N = N;
  g.K = K;
  g.offsets = groups;
  g.padded_offsets = groups + 2;
  g.epilogue = out_dtype;
  g.out = out;
  g.ld_out = ld_out;
  g.out_amax = nullptr;
  g.tile_n = tile_n_setting(static_cast<double>(T));
  g.status = status;
  // the offsets were written by the prologue, which finished before the quantiser
  g.early_weights = true;
  g.ksplit = linear_ksplit(T, K, N);
  g.partial = partial;
  g.partial_plane = T * N;
  return cuda_status(launch_grouped_gemm(g, s));
}

megamoe_status megamoe_read_status(const uint32_t* status, uint32_t* bits,
                                   megamoe_stream_t stream) {
  if (!status || !bits) return MEGAMOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MEGAMOE_ERR_CUDA;
  if (cudaMemcpy(bits, status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MEGAMOE_ERR_CUDA;
  return *bits ? MEGAMOE_ERR_DEVICE_STATUS : MEGAMOE_OK;
}

}  // extern "C"
