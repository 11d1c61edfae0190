/*
 * megamoe.h -- C ABI of the GB300 (sm_103a) NVFP4 MegaMoE routed-expert forward,
 * with, around it, the router (megamoe_router_topk, and
 * megamoe_forward_from_logits for the whole layer from router logits, a
 * shared expert included) and the dense NVFP4 linear with a measured-amax
 * activation scale (megamoe_linear_nvfp4).
 *
 * What it computes (sources are the titles and sections of the pages the
 * method is taken from):
 *   "CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4"
 *     - "Architecture: DeepSeek-V4 MegaMoE": 384 experts with top-6 routing
 *       and a persistent grouped GEMM whose groups are the experts;
 *     - "What's Been Verified": the MoE is the L1 gate+up GEMM and the L2 down
 *       GEMM, both NVFP4;
 *     - "Test Plan -- Finding the NaN", Phase 1: the runner takes
 *       hidden_states, topk_ids, topk_weights and variable per-expert token
 *       counts padded to 128 rows, quantises the activations to NVFP4, and
 *       runs L1 GEMM -> SiLU -> L2 GEMM; Phase 2: zero-token experts and the
 *       expert_offsets / padded_expert_offsets arrays.
 *   "Current Bug: vLLM produces NaN from layer 0"
 *     - "What we've tried" item 1 and "Key evidence": the activation global
 *       scale must come from the measured amax, never from a stored
 *       input_scale.
 *
 * NVFP4 here: E2M1 element codes (two per byte, even element in the low
 * nibble), one unsigned E4M3 block scale per 16 elements along K, one FP32
 * global scale gs per tensor.  An element decodes to
 * e2m1(code) * e4m3(scale) / gs.  Activations are encoded with
 * gs = 2688 / amax (448 * 6), and with the float32 steps
 * s = (amax_b * gs) / 6, s8 = e4m3_rne_satfinite(s), enc = gs / decode(s8),
 * code = e2m1_rne_satfinite(x * enc), each a correctly rounded operation.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless a parameter says "host".  The
 *     caller owns every buffer (workspace included); the library never
 *     allocates or frees memory and never synchronises on the compute path.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).
 *   - Argument and shape errors are returned synchronously, before anything
 *     is enqueued.  A failed launch returns MEGAMOE_ERR_CUDA.  Problems only
 *     the device can see (an expert id >= E, a non-finite input, a spin-wait
 *     that ran out) set bits in a device status word and never trap; read it
 *     with megamoe_read_status.
 *   - Matrices are row-major.  "Atom layout" (MEGAMOE_SCALES_MMA) stores block
 *     scales in 512-byte atoms of 128 rows x 4 blocks: atom (a, c) covers rows
 *     128a..128a+127 and blocks 4c..4c+3 and holds row 128a + 32j + i, block
 *     4c + b at byte 16i + 4j + b; atoms are ordered [a][c].  This is the
 *     layout the tensor cores read block scales in.
 */
#ifndef MEGAMOE_H
#define MEGAMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* megamoe_stream_t; /* == cudaStream_t */

typedef enum megamoe_status {
  MEGAMOE_OK = 0,
  MEGAMOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum */
  MEGAMOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set      */
  MEGAMOE_ERR_WORKSPACE_TOO_SMALL = 3,
  MEGAMOE_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed     */
  MEGAMOE_ERR_DEVICE_STATUS = 5      /* megamoe_read_status found bits set    */
} megamoe_status;

/* Bits of the device status word. */
#define MEGAMOE_DEV_BAD_EXPERT_ID 0x1u /* a topk id >= E was seen (slot skipped) */
#define MEGAMOE_DEV_NONFINITE 0x2u     /* the amax of an input was not finite    */
#define MEGAMOE_DEV_TIMEOUT 0x4u       /* a bounded device wait gave up          */

/* Scale layouts. */
#define MEGAMOE_SCALES_ROWMAJOR 0 /* [rows, K/16] bytes                         */
#define MEGAMOE_SCALES_MMA 1      /* atom layout, ceil(rows/128)*128 rows          */

/* Grouped-GEMM epilogues. */
#define MEGAMOE_EPI_F32 0      /* out[r, n] = fp32 accumulator * alpha            */
#define MEGAMOE_EPI_SILU_MUL 1 /* out[r, i] = bf16(silu(gate) * up), amax of it   */
#define MEGAMOE_EPI_BF16 2     /* out[r, n] = bf16(fp32 accumulator * alpha)      */
#define MEGAMOE_EPI_BFP16 3    /* out = BFP16 matrix of fp32 accumulator * alpha */

/*
 * BFP16 (16-bit block floating point): the storage of the forward's L2
 * output y between the down GEMM and the combine (the pages fix no type for
 * it; fp32 would double its round trip through HBM).  A [rows, ld] BFP16
 * matrix (ld a multiple of 32) holds one power-of-two exponent per group of
 * 16 rows x 8 columns (rows 16g .. 16g + 15, columns 8c .. 8c + 7).  It is one
 * buffer of MEGAMOE_BFP16_BYTES(rows, ld) bytes:
 *   bytes [0, 2*rows*ld)                          uint16 values u[r*ld + c]
 *   bytes [2*rows*ld, + ceil(rows/16)*(ld/8))     int8 exponents s[(r/16)*(ld/8) + c/8]
 *   element (r, c) = (u - 32768) * 2^s              (s <= 114)
 *                  = fp16 value of the bits of u    (s = 127)
 * Writing the fp32 values v of a group's written rows: with m = max |v| and
 * E = floor(log2 m), s = max(E - 14, -126), plus one when m * 2^-s >= 32767.5,
 * and u = rint(v * 2^-s) + 32768 (ties to even; |rint| <= 32767), so the
 * group's largest values keep 15 significant bits (v * 2^-s is exact; the
 * only rounding is to the integer); s = 0 and u = 32768 when all are zero.
 * A group holding Inf or NaN gets s = 127 and the fp16 encoding of each
 * value, so non-finite values pass through.  Rows that are not written
 * (padding rows) take no part in their group's exponent.  (A value within
 * 2^-16 of the largest float decodes to Inf.)
 */
#define MEGAMOE_BFP16_BYTES(rows, ld) \
  ((size_t)(rows) * (size_t)(ld) * 2 + ((size_t)(rows) + 15) / 16 * ((size_t)(ld) / 8))

/* Limits. */
#define MEGAMOE_MAX_EXPERTS 1024
#define MEGAMOE_MAX_TOPK 16

/*
 * NVFP4 expert weights.  Expert e of W13 is [2I, d]: rows 0..I-1 are the gate
 * projection, rows I..2I-1 the up projection ("What's Been Verified": L1
 * gate+up).  W2 is [d, I] per expert (L2 down).
 *   w13_codes   [E*2I, d/2] E2M1 codes packed by megamoe_pack_weight_codes
 *               with half_rows = I
 *   w13_scales  atom layout of [E*2I, d/16] (from megamoe_swizzle_scales)
 *   w13_gs      [E, 2] float            global scales (gate, up)
 *   w2_codes    [E*d, I/2] packed by megamoe_pack_weight_codes, half_rows = 0
 *   w2_scales   atom layout of [E*d, I/16]
 *   w2_gs       [E] float
 * Supported: 1 <= E <= 1024, d and I multiples of 256.
 */
typedef struct megamoe_weights {
  int32_t num_experts;
  int32_t hidden;       /* d */
  int32_t intermediate; /* I */
  const uint8_t* w13_codes;
  const uint8_t* w13_scales;
  const float* w13_gs;
  const uint8_t* w2_codes;
  const uint8_t* w2_scales;
  const float* w2_gs;
} megamoe_weights;

/* Human-readable name of a status code (static storage). */
const char* megamoe_status_string(megamoe_status s);

/*
 * Largest number of padded rows routing can produce:
 * T*k + min(E, T*k) * (pad - 1).  Host-only, no device work.
 */
int64_t megamoe_max_padded_rows(int T, int k, int E, int pad);

/*
 * megamoe_route_permute -- bucket the (token, slot) pairs by expert.
 * ("Test Plan -- Finding the NaN", Phase 1: variable token counts per expert
 * padded to 128; Phase 2: zero-token experts, expert_offsets and
 * padded_expert_offsets.)
 *
 * Slot s = t*k + j is routed to expert topk_ids[t*k + j].  Slots are grouped
 * by expert with a stable counting sort (ascending s inside an expert).
 *   topk_ids        [T, k] int32; ids < 0 are skipped; ids >= E are skipped and
 *                   set MEGAMOE_DEV_BAD_EXPERT_ID in *status
 *   counts          [E]    valid slots per expert (out)
 *   offsets         [E+1]  exclusive prefix sum of counts (out)
 *   padded_offsets  [E+1]  exclusive prefix sum of counts rounded up to pad;
 *                          a zero count stays zero (out)
 *   row_src         [row_capacity] flat slot held by each padded row, -1 for
 *                   padding and for every row >= padded_offsets[E] (out)
 *   slot_dst        [T*k]  padded row of each slot, -1 if skipped (out)
 *   status          device uint32 status word (bits are OR-ed in; may be NULL)
 * Requires 1 <= E <= 1024, 1 <= k <= 16, pad >= 1, T >= 0 and
 * row_capacity >= megamoe_max_padded_rows(T, k, E, pad).  T*k above 2^30 or
 * megamoe_max_padded_rows at or above 2^31 (offsets are int32) returns
 * MEGAMOE_ERR_UNSUPPORTED_SHAPE; the forward checks the same.  One thread
 * block.
 */
megamoe_status megamoe_route_permute(const int32_t* topk_ids, int T, int k, int E, int pad,
                                     int32_t* counts, int32_t* offsets,
                                     int32_t* padded_offsets, int32_t* row_src,
                                     int64_t row_capacity, int32_t* slot_dst,
                                     uint32_t* status, megamoe_stream_t stream);

/*
 * megamoe_quantize_nvfp4 -- bf16 activations -> NVFP4
 * ("Test Plan -- Finding the NaN", Phase 1 item 4: quantize_activation_nvfp4;
 * global scale from the measured amax per "Current Bug: vLLM produces NaN
 * from layer 0", "What we've tried" item 1).
 *
 *   x          [rows, K] bf16 with row stride ld (elements), ld >= K
 *   amax_in    if non-NULL, the amax to use (device float, e.g. the amax the
 *              L1 epilogue measured); if NULL the amax of x over all rows is
 *              measured here (one extra read of x)
 *   amax_out   device float: the amax used (out; may be NULL if amax_in given)
 *   gs_out     device float: gs = 2688 / amax, or 1 if amax == 0 (out)
 *   codes      [out_rows, K/2] (out), scales in `scale_layout` (out)
 * Row mapping:
 *   slot_dst == NULL: out row r is x row r (out_rows == rows).
 *   slot_dst != NULL: x row t is written to out rows slot_dst[t*k + j],
 *                     j = 0..k-1, skipping -1 (the routed gather).
 *   row_src != NULL:  out rows with row_src[r] < 0 are written as zero codes
 *                     and zero scales instead (padding rows).
 *   live_rows != NULL: device int32; out rows >= *live_rows are not touched.
 * Requires rows >= 0, out_rows >= 0, ld >= K and, with slot_dst == NULL,
 * rows >= out_rows (else MEGAMOE_ERR_INVALID_ARG); K a multiple of 64, ld a
 * multiple of 8, x and codes 16-byte aligned, scales 4-byte aligned (else
 * MEGAMOE_ERR_UNSUPPORTED_SHAPE).
 */
megamoe_status megamoe_quantize_nvfp4(const uint16_t* x, int64_t rows, int K, int64_t ld,
                                      const int32_t* slot_dst, int k, const int32_t* row_src,
                                      const int32_t* live_rows, int64_t out_rows,
                                      const float* amax_in, float* amax_out, float* gs_out,
                                      uint8_t* codes, uint8_t* scales, int scale_layout,
                                      uint32_t* status, megamoe_stream_t stream);

/*
 * megamoe_swizzle_scales -- one-time weight preparation: row-major block
 * scales [rows, K/16] -> atom layout (see the file comment).  Rows are padded
 * to a multiple of 128 with zero bytes; dst holds ceil(rows/128)*128*K/16
 * bytes.  Requires K a multiple of 64 and 4-byte aligned src and dst.
 */
megamoe_status megamoe_swizzle_scales(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                                      megamoe_stream_t stream);

/*
 * megamoe_pack_weight_codes -- one-time weight preparation: row-major E2M1
 * codes [rows, K/2] -> tile-major blocks of 128 rows x 128 bytes (256
 * elements of K).  Within a block, row i sits at byte 128*i and its 16-byte
 * chunk j at chunk j XOR (i % 8): the 128-byte swizzle the tensor cores read
 * K-major operands in, so the GEMM copies a block to shared memory as is.
 *   half_rows == 0: blocks ordered [rows/128][K/256] (the W2 layout).
 *   half_rows == H: rows come in groups of 2H, H gate rows then H up rows (one
 *                   expert of W13, H = I); the gate and up blocks of the same
 *                   128 features and K step are adjacent:
 *                   [rows/2H][H/128][K/256][gate, up] (the W13 layout).
 * A stage of the grouped GEMM then reads one contiguous 16 KB (W2) or 32 KB
 * (W13) block with a single bulk copy.  Requires rows a multiple of 128 (of 2H when H > 0), H a
 * multiple of 128, K a multiple of 256, 16-byte alignment.
 */
megamoe_status megamoe_pack_weight_codes(const uint8_t* src, int64_t rows, int K, int half_rows,
                                         uint8_t* dst, megamoe_stream_t stream);

/*
 * megamoe_grouped_gemm -- one persistent grouped block-scaled GEMM over all
 * experts ("Architecture: DeepSeek-V4 MegaMoE": one problem per expert,
 * persistent tile scheduling across groups, token tile chosen from the
 * expected tokens per expert).  On tcgen05 tensor cores with TMEM
 * accumulators and TMA loads.
 *
 * For every expert e and every valid row r of e
 * (padded_offsets[e] <= r < padded_offsets[e] + offsets[e+1] - offsets[e]):
 *   acc[r, n] = sum_K dequant(act)[r, :] . dequant(w_e)[n, :]   (fp32 accumulate)
 *   act_codes   [act_rows, K/2]; act_scales row-major [act_rows, K/16];
 *               act_gs device float (one global scale)
 *   w_codes     [E*N, K/2] packed by megamoe_pack_weight_codes (half_rows =
 *               N/2 for MEGAMOE_EPI_SILU_MUL, 0 otherwise);
 *               w_scales atom layout of [E*N, K/16] (megamoe_swizzle_scales)
 *   w_gs        [E, G] float: G = 2 (gate, up) for MEGAMOE_EPI_SILU_MUL, else 1
 *   offsets, padded_offsets  [E+1] int32 as produced by megamoe_route_permute
 *               with a pad that is a multiple of 32
 * Epilogues:
 *   MEGAMOE_EPI_F32:      out float [act_rows, ld_out], out[r, n] = acc * alpha,
 *                         alpha = 1 / (act_gs * w_gs[e]).
 *   MEGAMOE_EPI_BF16:     out bf16 [act_rows, ld_out], out[r, n] = bf16(acc * alpha).
 *   MEGAMOE_EPI_BFP16:    out BFP16 [act_rows, ld_out] of acc * alpha (the
 *                         format above; ld_out a multiple of 32; a group's
 *                         rows are 16 padded rows of one expert; weights-on-M
 *                         tiles only: tile_n 256 runs as 128).
 *   MEGAMOE_EPI_SILU_MUL: N = 2I; out bf16 [act_rows, ld_out],
 *                         out[r, i] = bf16(silu(acc[r, i] * alpha_gate) *
 *                                          (acc[r, I + i] * alpha_up)),
 *                         out_amax (device float, zeroed here) = max |out| over
 *                         valid rows.
 * Padding rows of `out` are not written.  tile_n selects the tile shape
 * (0 = choose from the expected tokens per expert, expected_tokens = rows the
 * caller expects per active expert, may be 0):
 *   32, 64, 128  tiles of 128 weight rows x tile_n token rows (weights on the
 *                MMA's M side, tokens on N);
 *   256          token-major tiles: 128 token rows x 256 weight rows (tokens on
 *                M, weights on N; for SILU_MUL the gate and up rows of 128
 *                features in one MMA); requires N a multiple of 256.
 * Requires N a multiple of 128 (256 for SILU_MUL), K a multiple of 256,
 * 1 <= E <= 1024, 16-byte aligned pointers, ld_out >= output width and a
 * multiple of 16 bytes (4 floats, 8 bf16), else MEGAMOE_ERR_UNSUPPORTED_SHAPE.
 */
megamoe_status megamoe_grouped_gemm(const uint8_t* act_codes, const uint8_t* act_scales,
                                    const float* act_gs, int64_t act_rows,
                                    const uint8_t* w_codes, const uint8_t* w_scales,
                                    const float* w_gs, int E, int N, int K,
                                    const int32_t* offsets, const int32_t* padded_offsets,
                                    int epilogue, void* out, int64_t ld_out, float* out_amax,
                                    int tile_n, double expected_tokens, uint32_t* status,
                                    megamoe_stream_t stream);

/*
 * megamoe_router_topk -- the router step ahead of megamoe_route_permute
 * ("CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Test Plan -- Finding the
 * NaN", Phase 1 item 1: topk_ids and topk_weights come from the router; the
 * pages do not spell the router out: this is the plain top-k + softmax):
 *   score[t, e] = fl32(logits[t, e] + bias[e])   (bias nullable: score = logit)
 *   topk_ids[t, 0..k-1]     = the k experts of highest score, in descending
 *                             score, ties to the lower expert index
 *   topk_weights[t, j]      = softmax over the k selected *logits* (fp32)
 * With shared_expert >= 0 one more column is appended to both outputs:
 * id shared_expert with weight 1 (a shared expert that every token visits,
 * to be run by megamoe_forward as one more expert).
 *   logits        float [T, ld_logits] (ld_logits >= E)
 *   topk_ids      int32 [T, k_out], topk_weights float [T, k_out],
 *                 k_out = k + (shared_expert >= 0)
 * Requires 1 <= k <= min(E, 16), E <= 1024, 4-byte aligned pointers.
 */
megamoe_status megamoe_router_topk(const float* logits, int64_t T, int E, int64_t ld_logits,
                                   const float* bias, int k, int shared_expert,
                                   int32_t* topk_ids, float* topk_weights,
                                   megamoe_stream_t stream);

/*
 * megamoe_forward_from_logits -- the MoE layer from router logits: the router
 * step of megamoe_router_topk (k routed experts among the first n_logits,
 * plus, with shared_expert >= 0, that expert for every token with weight 1)
 * followed by megamoe_forward over w's experts with k_out = k + (shared_expert
 * >= 0) slots per token.  For small batches (T * hidden <= 262144) the router
 * runs inside the forward's first thread block, ahead of the routing; larger
 * batches run it as its own kernel.  The ids and weights are written into the
 * workspace (sized by megamoe_workspace_size(T, k_out, w->num_experts, ...)).
 *   logits   float [T, ld_logits], n_logits <= w->num_experts columns used;
 *   bias     float [n_logits] or NULL (selection only)
 *   shared_expert  -1, or an expert index in [n_logits, w->num_experts)
 * Otherwise as megamoe_forward; k_out <= 16.
 */
megamoe_status megamoe_forward_from_logits(const megamoe_weights* w, const uint16_t* x,
                                           const float* logits, int64_t ld_logits,
                                           const float* bias, int n_logits, int k,
                                           int shared_expert, int T, int pad, uint16_t* out,
                                           void* ws, size_t ws_bytes, megamoe_stream_t stream);

/*
 * megamoe_linear_nvfp4 -- a dense NVFP4 linear layer whose activation global
 * scale comes from the measured amax of x, not from a stored input scale
 * ("Current Bug: vLLM produces NaN from layer 0", "Root Cause" and "Key
 * evidence": the attention projections quantised activations with the
 * checkpoint's input_scale, whose inverse (~4e3 to 1.6e4) overflowed
 * activations of amax 2-8).  The one-group case of the grouped GEMM:
 *   amax = max |x|, gs_x = 2688 / amax (1 if amax = 0), x -> NVFP4 as
 *   megamoe_quantize_nvfp4 does, then
 *   out[t, n] = sum_K dequant(x)[t, :] . dequant(w)[n, :]   (fp32 accumulate)
 * written as bf16 (out_dtype MEGAMOE_EPI_BF16) or float (MEGAMOE_EPI_F32).
 *   x          bf16 [T, K], row stride ld_x elements
 *   w_codes    [N, K/2] packed by megamoe_pack_weight_codes (half_rows 0)
 *   w_scales   atom layout of [N, K/16] (megamoe_swizzle_scales)
 *   w_gs       device float: the weight's global scale
 *   out        [T, ld_out] of out_dtype
 *   ws         device workspace of megamoe_linear_workspace_size(T, K, N) bytes,
 *              256-byte aligned, owned by the caller; it also receives the
 *              measured amax (float at ws + 0) and gs_x (float at ws + 4) and
 *              the status word (uint32 at ws + 8, read with megamoe_read_status)
 * Requires K a multiple of 256, N a multiple of 128, ld_x a multiple of 8
 * and ld_out of 16 bytes, 16-byte aligned pointers.  Argument errors return
 * before anything is enqueued; non-finite x sets MEGAMOE_DEV_NONFINITE.
 */
size_t megamoe_linear_workspace_size(int64_t T, int K, int N);
megamoe_status megamoe_linear_nvfp4(const uint16_t* x, int64_t T, int K, int64_t ld_x,
                                    const uint8_t* w_codes, const uint8_t* w_scales,
                                    const float* w_gs, int N, int out_dtype, void* out,
                                    int64_t ld_out, void* ws, size_t ws_bytes,
                                    megamoe_stream_t stream);

/*
 * megamoe_combine -- top-k weighted combine (topk_weights input of "Test Plan
 * -- Finding the NaN", Phase 1):
 *   out[t, :] = bf16( sum_{j=0..k-1, slot_dst[t*k+j] >= 0}
 *                     topk_weights[t*k+j] * y[slot_dst[t*k+j], :] )
 * summed in fp32 in ascending j.  y is float [*, ld_y]; out bf16 [T, d].
 * Requires d and ld_y multiples of 4, y 16-byte and out 8-byte aligned
 * (else MEGAMOE_ERR_UNSUPPORTED_SHAPE).
 */
megamoe_status megamoe_combine(const float* y, int64_t ld_y, const int32_t* slot_dst,
                               const float* topk_weights, int T, int k, int d, uint16_t* out,
                               megamoe_stream_t stream);

/*
 * megamoe_combine_bfp16 -- the same combine over a BFP16 y of y_rows rows and
 * leading dimension ld_y (the forward's own form of y): each element is
 * decoded exactly into fp32, then summed in fp32 in ascending j and rounded
 * once to bf16.  Requires d and ld_y multiples of 32, y 16-byte and out
 * 8-byte aligned (else MEGAMOE_ERR_UNSUPPORTED_SHAPE); a slot_dst entry at or
 * past y_rows is skipped like a negative one.
 */
megamoe_status megamoe_combine_bfp16(const void* y, int64_t ld_y, int64_t y_rows,
                                     const int32_t* slot_dst, const float* topk_weights, int T,
                                     int k, int d, uint16_t* out, megamoe_stream_t stream);

/*
 * Workspace bytes megamoe_forward needs for these sizes (host-only).
 */
size_t megamoe_workspace_size(int T, int k, int E, int d, int I, int pad);

/*
 * megamoe_forward -- the whole routed-expert forward on one stream:
 * route -> amax(x) -> quantise x into routed rows -> L1 grouped GEMM with
 * SiLU(gate)*up and amax(h) in its epilogue -> requantise h -> L2 grouped
 * GEMM into a BFP16 y -> top-k weighted combine (y decoded exactly, fp32
 * sums, one bf16 rounding).
 *   x             [T, d] bf16 hidden_states
 *   topk_ids      [T, k] int32 (ids < 0 skipped)
 *   topk_weights  [T, k] float (used as given)
 *   pad           rows per expert are padded to a multiple of pad; must be a
 *                 multiple of 32 (32, 64, 128, ...)
 *   out           [T, d] bf16 (out)
 *   ws, ws_bytes  workspace, at least megamoe_workspace_size(...) bytes,
 *                 256-byte aligned; its first 4 bytes are the device status
 *                 word, cleared at the start of every call.
 * Requires the weight shapes above, 1 <= k <= 16, T >= 0, x and the weight
 * codes and scales 16-byte aligned, out 8-byte aligned.  Every step is a
 * kernel launch on `stream` (no host synchronisation, no memory allocation),
 * so the call can be recorded into a CUDA graph and replayed.
 */
megamoe_status megamoe_forward(const megamoe_weights* w, const uint16_t* x,
                               const int32_t* topk_ids, const float* topk_weights, int T, int k,
                               int pad, uint16_t* out, void* ws, size_t ws_bytes,
                               megamoe_stream_t stream);

/*
 * megamoe_set_wait_limit_ns -- bound of every pipeline wait inside the
 * grouped GEMM kernels launched afterwards (host setting of this library,
 * all devices; 0 restores the default of 4 s).  A wait that runs out raises
 * the kernel's abort flag and MEGAMOE_DEV_TIMEOUT; the kernel then lets its
 * copies and MMAs in flight land (waiting up to 4 s), frees its tensor memory
 * and returns, so the context stays usable.  For failure-detection tests and
 * diagnosis; the default never fires in normal operation.
 */
void megamoe_set_wait_limit_ns(uint64_t ns);

/*
 * megamoe_set_fused_requant -- where megamoe_forward / _from_logits /
 * _static requantise h (the requantisation fused into the L1 GEMM's
 * epilogue, or after it; host setting of this library, all devices, for
 * forwards launched afterwards):
 *   0 (default)  a separate kernel after the L1 GEMM reads h once and encodes
 *                it with the global scale of amax(h);
 *   1            the L1 GEMM kernel does it: after its last tile each CTA
 *                arrives on a grid-wide count in the workspace and waits
 *                (bounded by the pipeline wait limit; MEGAMOE_DEV_TIMEOUT on
 *                expiry) until every CTA with tiles has, so amax(h) is
 *                final, then encodes the h rows of its own tiles.
 * Both give bit-identical results.  The default is the faster on GB300 (the
 * separate kernel lets CTAs that finish early free their SM for the next
 * kernel); an L1 GEMM split along K always uses the separate kernel.
 */
void megamoe_set_fused_requant(int enable);

/*
 * Expert-parallel forward, one shard (one process and GPU) of G: the shard
 * holds experts [expert_base, expert_base + w_shard->num_experts) of
 * num_experts_total ("CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Test
 * Plan -- Finding the NaN", Phase 2: the EP8 slice of 48 of the 384 experts).
 * The layer's tokens are first gathered on every shard (x, topk_ids and
 * topk_weights of all T tokens, global expert ids); then:
 *
 *   megamoe_ep_forward_begin  routes the shard's slots (ids of other shards
 *     skipped, ids >= num_experts_total flagged MEGAMOE_DEV_BAD_EXPERT_ID and
 *     skipped), takes amax(x) over all T tokens (the same on every shard, so
 *     x's global scale needs no exchange), quantises x and runs the L1 GEMM
 *     with SiLU(gate)*up; the shard's amax(h) is left as a float at bytes
 *     [12, 16) of ws.
 *   The caller replaces that float on every shard by the maximum over all
 *     shards (an all-reduce(max) of 4 bytes): h has one global scale over
 *     every valid row of the layer's intermediate, whichever shard holds it.
 *   megamoe_ep_forward_end  requantises h with that global amax, runs the L2
 *     GEMM and writes out_partial [T, d] fp32 = sum over the shard's slots j
 *     (ascending) of topk_weights[t, j] * y (0 for tokens with no slot on the
 *     shard), before any rounding.
 *   The caller sums the shards' out_partial (an all-reduce or reduce-scatter)
 *     and rounds once with megamoe_round_bf16.
 *
 * With the same inputs the result equals megamoe_forward's up to the order of
 * the fp32 additions across shards.  w_shard, T, k, pad and ws are those of
 * megamoe_forward on the shard's experts (ws: megamoe_workspace_size(T, k,
 * w_shard->num_experts, d, I, pad) bytes, 256-byte aligned, the same buffer
 * for begin and end); out_partial is 16-byte aligned.  Errors as
 * megamoe_forward, plus MEGAMOE_ERR_INVALID_ARG when the shard's range does
 * not fit in [0, num_experts_total).
 */
megamoe_status megamoe_ep_forward_begin(const megamoe_weights* w_shard, const uint16_t* x,
                                        const int32_t* topk_ids, int T, int k, int expert_base,
                                        int num_experts_total, int pad, void* ws, size_t ws_bytes,
                                        megamoe_stream_t stream);
megamoe_status megamoe_ep_forward_end(const megamoe_weights* w_shard, const float* topk_weights,
                                      int T, int k, int num_experts_total, int pad,
                                      float* out_partial, void* ws, size_t ws_bytes,
                                      megamoe_stream_t stream);

/*
 * megamoe_round_bf16 -- out[i] = bf16(in[i]), round to nearest even, i < n
 * (the single rounding of the expert-parallel sum).  n a multiple of 4, in
 * 16-byte and out 8-byte aligned, else MEGAMOE_ERR_UNSUPPORTED_SHAPE.
 */
megamoe_status megamoe_round_bf16(const float* in, int64_t n, uint16_t* out,
                                  megamoe_stream_t stream);

/*
 * megamoe_forward_scan_stages -- debug aid: which stage of the last forward
 * run with this workspace produced a non-finite value ("CURRENT_BUG.md --
 * DeepSeek-V4 Blackwell NVFP4", "Test Plan -- Finding the NaN", Phase 1
 * item 3: check after the L1 GEMM and SiLU, and after the L2 GEMM).  ws and
 * (T, k, E = w->num_experts, d, I, pad) are those of a megamoe_forward /
 * _from_logits call already enqueued on `stream`; out its output.  Scans
 * the valid rows (padding rows are never written and may hold anything) and
 * writes to *flags (device uint32, cleared here) the bits of every stage
 * that holds one:
 *   MEGAMOE_STAGE_XQ_SCALE  a block scale of the quantised x is an E4M3 NaN byte
 *   MEGAMOE_STAGE_H         h = bf16(SiLU(gate) * up) holds Inf or NaN
 *   MEGAMOE_STAGE_HQ_SCALE  a block scale of the requantised h is an E4M3 NaN byte
 *   MEGAMOE_STAGE_Y         the L2 output y holds Inf or NaN (a BFP16 group
 *                           of valid rows with exponent 127)
 *   MEGAMOE_STAGE_OUT       the combined output holds Inf or NaN
 * Reads every intermediate once (~3.7 GB at 16384 tokens): for diagnosis,
 * not the forward's path.  Asynchronous on `stream`.
 */
#define MEGAMOE_STAGE_XQ_SCALE 0x01u
#define MEGAMOE_STAGE_H 0x02u
#define MEGAMOE_STAGE_HQ_SCALE 0x04u
#define MEGAMOE_STAGE_Y 0x08u
#define MEGAMOE_STAGE_OUT 0x10u
megamoe_status megamoe_forward_scan_stages(const megamoe_weights* w, int T, int k, int pad,
                                           const uint16_t* out, const void* ws, size_t ws_bytes,
                                           uint32_t* flags, megamoe_stream_t stream);

/*
 * megamoe_read_status -- synchronise `stream`, copy the device status word at
 * `status` (for megamoe_forward: the first 4 bytes of ws) into *bits (host),
 * and return MEGAMOE_ERR_DEVICE_STATUS if any bit is set, else MEGAMOE_OK.
 */
megamoe_status megamoe_read_status(const uint32_t* status, uint32_t* bits,
                                   megamoe_stream_t stream);

/*
 * megamoe_forward_static -- megamoe_forward without a caller-provided
 * workspace, for callers that cannot allocate device memory where they run
 * the forward: plugins in a host process that owns every device allocation
 * (an inference server with its own memory pool, which forbids side
 * allocations), embedded callers that link only this library and have no
 * allocator at hand, hot loops that must never enter the allocator.  (The
 * source pages have no counterpart: this is a deployment variant of
 * megamoe_forward, not a step of the method.)
 *
 * The workspace is a fixed device array inside the library of
 * MEGAMOE_STATIC_WS_BYTES (64 MiB), held by every GPU that loads the library
 * until the process exits.  Nothing is allocated or freed by this call.
 * Arguments are those of megamoe_forward, minus ws/ws_bytes, plus:
 *   status_out  device uint32 (may be NULL): receives the forward's device
 *               status word (see MEGAMOE_DEV_*), copied on `stream`; written
 *               only when the call returns MEGAMOE_OK.
 * Argument and shape errors are those of megamoe_forward and are reported
 * first; then MEGAMOE_ERR_WORKSPACE_TOO_SMALL when
 * megamoe_workspace_size(T, k, E, d, I, pad) exceeds MEGAMOE_STATIC_WS_BYTES
 * (for E = 384, d = 7168, I = 2048, k = 6, pad = 32 that is T > 9 tokens).
 * The first call on a device looks the array up for that device (with it
 * current) and should come before any stream capture; a call under a new
 * driver context of the device (after cudaDeviceReset, or a context made
 * current through the driver API) looks it up again.  All calls share the
 * array: calls that overlap on the GPU race, so the caller serialises them
 * (one stream per device, or its own ordering).
 */
#define MEGAMOE_STATIC_WS_BYTES (64u << 20)
megamoe_status megamoe_forward_static(const megamoe_weights* w, const uint16_t* x,
                                      const int32_t* topk_ids, const float* topk_weights, int T,
                                      int k, int pad, uint16_t* out, uint32_t* status_out,
                                      megamoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MEGAMOE_H */
