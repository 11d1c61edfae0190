// Host-side launchers of the MegaMoE kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/megamoe.h"

namespace megamoe {

// Launch on `stream` with programmatic stream serialization: the kernel may be
// scheduled while its predecessor finishes; every kernel of this library
// executes griddepcontrol.wait before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

size_t route_smem_bytes(int E);
// Routing over many blocks (three passes) from this many slots on, when the
// caller passes a block_hist scratch of kRouteMaxBlocks * E ints.
constexpr int kRouteMultiMinSlots = 16384;
constexpr int kRouteMaxBlocks = 256;
// zero_words (may be null): n_zero 32-bit words cleared before anything else
// (the forward's status word and amax accumulators).
cudaError_t launch_route(const int32_t* ids, int n_slots, int E, int pad, int32_t* counts,
                         int32_t* offsets, int32_t* padded_offsets, int32_t* row_src,
                         int64_t row_capacity, int32_t* slot_dst, uint32_t* status,
                         uint32_t* zero_words, int n_zero, cudaStream_t stream,
                         int32_t* block_hist = nullptr);

// zero_first: clear *amax first (false when the caller already cleared it).
cudaError_t launch_amax(const uint16_t* x, int64_t rows, int K, int64_t ld, float* amax,
                        uint32_t* status, bool zero_first, cudaStream_t stream);
// Dense linear prologue (one block): status cleared, single-group offsets
// {0, rows, 0, rows}, and the amax of x when linear_prologue_full_amax (else
// amax = 0 for a following launch_amax with zero_first = false).
bool linear_prologue_full_amax(int64_t rows, int K);
cudaError_t launch_linear_prologue(const uint16_t* x, int64_t rows, int K, int64_t ld,
                                   float* amax, uint32_t* status, int32_t* groups,
                                   cudaStream_t stream);
cudaError_t launch_quant(const uint16_t* x, int64_t rows_in, int K, int64_t ld,
                         const int32_t* slot_dst, int k, const int32_t* row_src,
                         const int32_t* live_rows, int64_t out_rows, const float* amax,
                         float* gs_out, uint8_t* codes, uint8_t* scales, int scale_layout,
                         cudaStream_t stream, bool slot_rows = false);

// Small-batch prologue of the forward in one thread block: route and the amax
// of x.  Used when prologue_fits(T, d).
bool prologue_fits(int T, int d);
// Router fused into the prologue: ids/weights [T, k] (k = k_routed + shared
// column) are written from logits [T, ld] over n_logits experts, then routed.
struct RouterArgs {
  const float* logits = nullptr;
  int64_t ld = 0;
  const float* bias = nullptr;
  int n_logits = 0;
  int k_routed = 0;
  int shared = -1;
  int32_t* ids_out = nullptr;
  float* w_out = nullptr;
};
cudaError_t launch_prologue(const int32_t* ids, int T, int k, int E, int pad, int32_t* counts,
                            int32_t* offsets, int32_t* padded_offsets, int32_t* row_src,
                            int64_t row_capacity, int32_t* slot_dst, uint32_t* status,
                            uint32_t* zero_words, int n_zero, const uint16_t* x, int d,
                            float* amax, cudaStream_t stream, const RouterArgs* router = nullptr);
cudaError_t launch_swizzle(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                           cudaStream_t stream);

cudaError_t launch_pack(const uint8_t* src, int64_t rows, int K, int half_rows, uint8_t* dst,
                        cudaStream_t stream);

struct GemmLaunch {
  const uint8_t* act_codes;
  const uint8_t* act_scales;  // atom layout
  const float* act_gs;
  int64_t act_rows;
  const uint8_t* w_codes;   // tile-major (k_pack; gate/up paired for SILU_MUL)
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
  bool zero_amax = true;  // false when the caller already cleared out_amax
  // true only when the offsets were written by a kernel that finished before
  // the one immediately preceding the GEMM (the forward's order): the GEMM
  // then prefetches its first weight stages while that kernel runs
  bool early_weights = false;
  // split-K: ksplit > 1 cuts each tile's K range into ksplit pieces (token
  // tiles of 32 or 64 only); `partial` holds ksplit planes of
  // partial_plane >= offsets[E] * N floats; a finishing kernel sums them
  int ksplit = 1;
  float* partial = nullptr;
  int64_t partial_plane = 0;
  // requantisation of h fused into the SILU_MUL kernel (ksplit 1 only):
  // arrival counter zeroed before the launch, codes [rows, N/4], row-major
  // scales [rows, N/32], global scale out (all null: not fused)
  uint32_t* rq_arrivals = nullptr;
  uint8_t* rq_codes = nullptr;
  uint8_t* rq_scales = nullptr;
  float* rq_gs = nullptr;
};
// Split-K choice for a GEMM of about `tiles` whole-K tiles of KT K steps: the
// smallest ksplit (<= 8, >= 2 K steps a piece) that minimises the waves of
// pieces over the SMs, in units of a whole tile.
int pick_ksplit(double tiles, int KT);
// Encodes the tensor maps and launches the persistent grouped GEMM.
cudaError_t launch_grouped_gemm(const GemmLaunch& g, cudaStream_t stream);
int pick_tile_n(double expected_tokens_per_expert);
// Bound of the grouped GEMM's pipeline waits (0 restores the default 4 s).
void set_wait_limit_ns(uint64_t ns);
uint64_t wait_limit_ns();

// Router: ids/weights [T, k (+1 with a shared expert)] from fp32 logits.
cudaError_t launch_router(const float* logits, int64_t T, int E, int64_t ld, const float* bias,
                          int k, int shared, int32_t* ids, float* weights, cudaStream_t stream);

// Shape and weight-pointer checks of megamoe_forward.
megamoe_status check_forward_shape(const megamoe_weights* w, int T, int k, int pad);
// Argument and shape checks of megamoe_forward that do not involve the
// workspace (router: the ids and weights come from a fused router).
megamoe_status check_forward_args(const megamoe_weights* w, const uint16_t* x,
                                  const int32_t* topk_ids, const float* topk_weights, int T, int k,
                                  int pad, const uint16_t* out, bool router);

// Number of SMs of the current device (at least 1).
int num_sms();

// out: bf16 [T, d] (one rounding of the fp32 sum), or with out_f32 the fp32
// sum itself.
// y fp32 [*, ld_y] (y_exp null) or BFP16 (uint16 values at y, exponents
// [rows / 16, ld_y / 8] at y_exp)
// (y_rows: rows of a BFP16 y; slots at or past it are skipped)
cudaError_t launch_combine(const void* y, const int8_t* y_exp, int64_t ld_y, int64_t y_rows,
                           const int32_t* slot_dst, const float* w, int T, int k, int d,
                           void* out, bool out_f32, cudaStream_t stream);
// Non-finite scan of a forward's stage outputs (MEGAMOE_STAGE_* bits in
// *flags, cleared first); valid rows only, every output row.
cudaError_t launch_stage_scan(const int32_t* row_src, const int32_t* padded_total,
                              const uint8_t* xq_sf, const uint16_t* h, const uint8_t* hq_sf,
                              const int8_t* y_exp, const uint16_t* out, int T, int d, int I,
                              uint32_t* flags, cudaStream_t stream);
// out[i] = bf16_rne(in[i]), n a multiple of 4.
cudaError_t launch_round_bf16(const float* in, int64_t n, uint16_t* out, cudaStream_t stream);
// Expert-parallel shard: ids in [base, base + E_local) -> id - base; other
// valid ids and ids < 0 -> -1 (skipped); ids >= E_total -> E_local (out of
// range for the shard, so the routing flags and skips them).
cudaError_t launch_ep_remap(const int32_t* ids, int64_t n, int base, int E_local, int E_total,
                            int32_t* out, cudaStream_t stream);

}  // namespace megamoe
