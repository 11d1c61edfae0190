// NVFP4 activation quantisation with a global scale from the measured amax
// ("CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4", "Test Plan -- Finding the
// NaN", Phase 1 item 4: quantize_activation_nvfp4; "Current Bug: vLLM
// produces NaN from layer 0", "What we've tried" item 1 and "Key evidence":
// the global scale comes from the measured amax, never a stored input_scale).
//
// k_amax    one streaming read of the bf16 tensor with 128-bit loads; the
//           |x| maximum is taken on the bf16 bit patterns with packed 16-bit
//           integer max (monotone for finite values), reduced with warp
//           shuffles and one atomicMax per block.
// k_quant   one thread per (row, 16-element block): 32 bytes of bf16 in
//           (2 x 128-bit loads), 8 bytes of E2M1 codes and one E4M3 scale
//           byte out.  The routed gather is fused: a token row is encoded
//           once and written to each of its k expert rows.
// k_swizzle row-major block scales -> the tensor-core atom layout (weights,
//           once, off the hot path).
// k_pack    row-major E2M1 codes -> tile-major blocks of 128 rows x 128 bytes,
//           pre-swizzled (weights, once): the grouped GEMM fetches a stage's
//           weights with one contiguous bulk copy.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace megamoe {

// t / n for a non-negative task index: 32-bit division whenever t fits (the
// 64-bit one is a long software sequence).
__device__ __forceinline__ int64_t task_div(int64_t t, int n) {
  return (t >> 32) == 0 ? static_cast<int64_t>(static_cast<uint32_t>(t) / static_cast<uint32_t>(n))
                        : t / n;
}

__global__ void __launch_bounds__(256) k_amax(const uint16_t* __restrict__ x, int64_t rows, int K,
                                              int64_t ld, float* amax, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int vecs = K / 8;
  const int64_t total = rows * vecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint32_t m2 = 0;  // two packed |bf16| maxima
  // four loads in flight per thread per round
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i0 < total;
       i0 += 4 * stride) {
    uint4 q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = i0 + j * stride;
      const int64_t r = task_div(i, vecs);
      q[j] = i < total ? __ldg(reinterpret_cast<const uint4*>(x + r * ld) + (i - r * vecs))
                       : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m2 = __vmaxu2(m2, q[j].x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q[j].y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q[j].z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q[j].w & 0x7FFF7FFFu);
    }
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (blockDim.x >> 5); ++w) m = max(m, red[w]);
    if (m >= 0x7F80u) {  // Inf or NaN
      set_status(status, MEGAMOE_DEV_NONFINITE);
      m = 0x7F7Fu;  // keep the scale finite; the result is flagged anyway
    }
    atomicMax(reinterpret_cast<unsigned int*>(amax), m << 16);
  }
}

struct QuantArgs {
  const uint16_t* x;
  int64_t rows_in;
  int K;
  int64_t ld;
  const int32_t* slot_dst;
  int k;
  const int32_t* row_src;
  const int32_t* live_rows;
  int64_t out_rows;
  const float* amax;
  float* gs_out;
  uint8_t* codes;
  uint8_t* scales;
  int scale_layout;
  // true: task rows come from slot_dst (rows_in = number of slots); slot s
  // with slot_dst[s] >= 0 encodes x row slot_dst[s] into the same out row
  bool slot_rows;
};


__device__ __forceinline__ void store_block(const QuantArgs& a, int64_t out_row, int b, uint2 c,
                                            uint32_t s8) {
  *reinterpret_cast<uint2*>(a.codes + out_row * (a.K / 2) + 8 * b) = c;
  const int64_t so = a.scale_layout == MEGAMOE_SCALES_MMA
                         ? sf_atom_offset(out_row, b >> 2, a.K / 64) + (b & 3)
                         : out_row * (a.K / 16) + b;
  a.scales[so] = static_cast<uint8_t>(s8);
}

// One thread per (row, group of BPT 16-element blocks).  Tasks (NB = K/16
// blocks per row, in groups of BPT):
//  * slot_rows: [0, rows_in*NB): slot s encodes row slot_dst[s] in place;
//  * slot_dst:  [0, rows_in*NB) are token rows, scattered to their routed
//    rows, then, if row_src is given, [rows_in*NB, (rows_in+out_rows)*NB)
//    zero the padding rows;
//  * otherwise  [0, out_rows*NB) map out row r <- x row r (padding rows
//    zeroed when row_src is given).
// BPT consecutive 16-element blocks of one row per task: BPT = 1 for small
// launches (many short tasks over many SMs), 4 for large ones (32 bytes of
// codes and one 4-byte scale word per store, fewer index loads).
template <int BPT>
struct Group {
  uint2 c[BPT];
  uint32_t s8[BPT];
};

template <int BPT>
__device__ __forceinline__ Group<BPT> encode_group(const uint16_t* src, float gs) {
  uint4 v[2 * BPT];
#pragma unroll
  for (int i = 0; i < 2 * BPT; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
  Group<BPT> g;
#pragma unroll
  for (int j = 0; j < BPT; ++j) encode_block(v[2 * j], v[2 * j + 1], gs, g.c[j], g.s8[j]);
  return g;
}

template <int BPT>
__device__ __forceinline__ void store_group(const QuantArgs& a, int64_t out_row, int b0,
                                            const Group<BPT>& g) {
  if (BPT == 1) {
    store_block(a, out_row, b0, g.c[0], g.s8[0]);
    return;
  }
  // BPT = 4: b0 is a multiple of 4, so the codes are 32 aligned bytes and the
  // four scale bytes one aligned word in either layout
  uint4* cd = reinterpret_cast<uint4*>(a.codes + out_row * (a.K / 2) + 8 * b0);
  cd[0] = make_uint4(g.c[0].x, g.c[0].y, g.c[1].x, g.c[1].y);
  cd[1] = make_uint4(g.c[2].x, g.c[2].y, g.c[3].x, g.c[3].y);
  const uint32_t w = g.s8[0] | (g.s8[1] << 8) | (g.s8[2] << 16) | (g.s8[3] << 24);
  const int64_t so = a.scale_layout == MEGAMOE_SCALES_MMA
                         ? sf_atom_offset(out_row, b0 >> 2, a.K / 64)
                         : out_row * (a.K / 16) + b0;
  *reinterpret_cast<uint32_t*>(a.scales + so) = w;
}

template <int BPT>
__device__ __forceinline__ Group<BPT> zero_group() {
  Group<BPT> g;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    g.c[j] = make_uint2(0u, 0u);
    g.s8[j] = 0u;
  }
  return g;
}

template <int BPT>
__global__ void __launch_bounds__(256) k_quant(const QuantArgs a) {
  pdl_wait();
  pdl_trigger();
  const int NG = a.K / 16 / BPT;  // tasks per row
  const float amax = *a.amax;
  const float gs = amax == 0.f ? 1.f : __fdiv_rn(2688.0f, amax);
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.gs_out) *a.gs_out = gs;
  const int64_t live = a.live_rows ? static_cast<int64_t>(*a.live_rows) : a.out_rows;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (a.slot_rows) {
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
         t < a.rows_in * NG; t += stride) {
      const int64_t slot = task_div(t, NG);
      const int b0 = static_cast<int>(t - slot * NG) * BPT;
      const int64_t row = a.slot_dst[slot];
      if (row < 0 || row >= live) continue;
      store_group<BPT>(a, row, b0, encode_group<BPT>(a.x + row * a.ld + 16 * b0, gs));
    }
    return;
  }
  const int64_t token_tasks = a.slot_dst ? a.rows_in * NG : 0;
  const int64_t total = token_tasks + ((a.slot_dst && !a.row_src) ? 0 : a.out_rows * NG);
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
       t += stride) {
    const bool token_task = t < token_tasks;
    const int64_t u = token_task ? t : t - token_tasks;
    const int64_t row = task_div(u, NG);
    const int b0 = static_cast<int>(u - row * NG) * BPT;
    if (!token_task) {
      if (row >= live) continue;
      const bool pad_row = a.row_src && a.row_src[row] < 0;
      if (a.slot_dst && !pad_row) continue;  // written by its token task
      if (pad_row) {
        store_group<BPT>(a, row, b0, zero_group<BPT>());
        continue;
      }
    }
    const Group<BPT> g = encode_group<BPT>(a.x + row * a.ld + 16 * b0, gs);
    if (token_task) {
      for (int j = 0; j < a.k; ++j) {
        const int dst = a.slot_dst[row * a.k + j];
        if (dst >= 0 && dst < live) store_group<BPT>(a, dst, b0, g);
      }
    } else {
      store_group<BPT>(a, row, b0, g);
    }
  }
}

__global__ void __launch_bounds__(256) k_swizzle(const uint8_t* __restrict__ src, int64_t rows,
                                                 int K, uint8_t* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  const int S = K / 64;
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  const int64_t total = rows_pad * S;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = t / S;
    const int c = static_cast<int>(t - r * S);
    const uint32_t w =
        r < rows ? *reinterpret_cast<const uint32_t*>(src + r * (K / 16) + 4 * c) : 0u;
    *reinterpret_cast<uint32_t*>(dst + sf_atom_offset(r, c, S)) = w;
  }
}

// half_rows == 0: blocks ordered [rows/128][K/256].  half_rows == H > 0: rows
// come in groups of 2H (gate rows then up rows of one expert) and the gate and
// up blocks of the same 128 features and K step sit side by side:
// [group][H/128][K/256][gate, up], so the L1 GEMM reads 32 KB contiguous.
__global__ void __launch_bounds__(256) k_pack(const uint8_t* __restrict__ src, int64_t rows, int K,
                                              int half_rows, uint8_t* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  const int chunks = K / 32;  // 16-byte chunks per row
  const int KT = K / 256;     // 128-byte K blocks per row
  const int64_t total = rows * chunks;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = t / chunks;
    const int c = static_cast<int>(t - r * chunks);
    const int kt = c >> 3;
    int64_t block;
    if (half_rows > 0) {
      const int64_t group = r / (2 * half_rows);
      const int64_t in = r - group * 2 * half_rows;
      const int g = in >= half_rows ? 1 : 0;
      const int64_t mt = (in - g * half_rows) >> 7;
      block = ((group * (half_rows >> 7) + mt) * KT + kt) * 2 + g;
    } else {
      block = (r >> 7) * KT + kt;
    }
    // 16-byte chunk j of row r goes to chunk j ^ (r % 8): the 128-byte swizzle
    // the tensor cores read, so a plain bulk copy lands the block ready to use
    const int64_t o = (block * 128 + (r & 127)) * 128 + (((c & 7) ^ (r & 7)) * 16);
    *reinterpret_cast<uint4*>(dst + o) =
        __ldg(reinterpret_cast<const uint4*>(src + r * (K / 2)) + c);
  }
}

static int grid_for(int64_t tasks, int threads) {
  int64_t b = (tasks + threads - 1) / threads;
  const int64_t cap = 152 * 32;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

// Prologue of the dense NVFP4 linear, one block: clears the status word,
// writes the single group's offsets ({0, rows} as offsets and as padded
// offsets) and either the amax of x (full_amax: x small enough for one block)
// or 0, which k_amax's atomics then raise.
constexpr int kLinearPrologueThreads = 1024;
constexpr int64_t kLinearPrologueMaxElems = 262144;

__global__ void __launch_bounds__(kLinearPrologueThreads)
    k_linear_prologue(const uint16_t* __restrict__ x, int64_t rows, int K, int64_t ld,
                      float* amax, uint32_t* status, int32_t* groups, int full_amax) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t red[kLinearPrologueThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    groups[0] = 0;
    groups[1] = static_cast<int32_t>(rows);
    groups[2] = 0;
    groups[3] = static_cast<int32_t>(rows);
  }
  uint32_t m = 0;
  if (full_amax) {
    // at most 32 vectors a thread (rows * K <= 262144): issued 8 at a time so
    // that their latencies overlap
    const int vecs = K / 8;
    const int total = static_cast<int>(rows) * vecs;
    uint32_t m2 = 0;
    for (int base = tid; base < total; base += 8 * kLinearPrologueThreads) {
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * kLinearPrologueThreads;
        const int r = i / vecs;
        q[j] = i < total ? __ldg(reinterpret_cast<const uint4*>(x + r * ld) + (i - r * vecs))
                         : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m2 = __vmaxu2(m2, q[j].x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, q[j].y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, q[j].z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, q[j].w & 0x7FFF7FFFu);
      }
    }
    m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
  }
  if (tid == 0) {
    uint32_t bits = 0;
    if (full_amax) {
      for (int w = 1; w < kLinearPrologueThreads / 32; ++w) m = max(m, red[w]);
      if (m >= 0x7F80u) {  // Inf or NaN
        bits = MEGAMOE_DEV_NONFINITE;
        m = 0x7F7Fu;
      }
    }
    *status = bits;
    *amax = __uint_as_float(m << 16);
  }
}

bool linear_prologue_full_amax(int64_t rows, int K) {
  return rows * static_cast<int64_t>(K) <= kLinearPrologueMaxElems;
}

cudaError_t launch_linear_prologue(const uint16_t* x, int64_t rows, int K, int64_t ld,
                                   float* amax, uint32_t* status, int32_t* groups,
                                   cudaStream_t stream) {
  return launch_pdl(k_linear_prologue, dim3(1), dim3(kLinearPrologueThreads), 0, stream, x, rows,
                    K, ld, amax, status, groups,
                    linear_prologue_full_amax(rows, K) ? 1 : 0);
}

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int K, int64_t ld, float* amax,
                        uint32_t* status, bool zero_first, cudaStream_t stream) {
  if (zero_first) {
    cudaError_t err = cudaMemsetAsync(amax, 0, sizeof(float), stream);
    if (err != cudaSuccess) return err;
  }
  if (rows == 0) return cudaSuccess;
  return launch_pdl(k_amax, dim3(grid_for(rows * (K / 8), 256)), dim3(256), 0, stream, x, rows,
                    K, ld, amax, status);
}

cudaError_t launch_quant(const uint16_t* x, int64_t rows_in, int K, int64_t ld,
                         const int32_t* slot_dst, int k, const int32_t* row_src,
                         const int32_t* live_rows, int64_t out_rows, const float* amax,
                         float* gs_out, uint8_t* codes, uint8_t* scales, int scale_layout,
                         cudaStream_t stream, bool slot_rows) {
  QuantArgs a{x,        rows_in, K,      ld,     slot_dst,     k,        row_src, live_rows,
              out_rows, amax,    gs_out, codes,  scales,       scale_layout, slot_rows};
  const int64_t tasks =
      slot_rows ? rows_in * (K / 16)
                : ((slot_dst ? rows_in : 0) + ((slot_dst && !row_src) ? 0 : out_rows)) * (K / 16);
  if (tasks == 0) return cudaSuccess;
  // encoding is ALU work: few tasks go in small blocks spread over many SMs,
  // one 16-element block each; many tasks go four blocks to a thread
  if (tasks > 152 * 256 * 4)
    return launch_pdl(k_quant<4>, dim3(grid_for(tasks / 4, 256)), dim3(256), 0, stream, a);
  const int threads = tasks <= 152 * 256 ? 64 : 256;
  return launch_pdl(k_quant<1>, dim3(grid_for(tasks, threads)), dim3(threads), 0, stream, a);
}

cudaError_t launch_swizzle(const uint8_t* src, int64_t rows, int K, uint8_t* dst,
                           cudaStream_t stream) {
  const int64_t tasks = (rows + 127) / 128 * 128 * (K / 64);
  if (tasks == 0) return cudaSuccess;
  return launch_pdl(k_swizzle, dim3(grid_for(tasks, 256)), dim3(256), 0, stream, src, rows, K,
                    dst);
}

cudaError_t launch_pack(const uint8_t* src, int64_t rows, int K, int half_rows, uint8_t* dst,
                        cudaStream_t stream) {
  const int64_t tasks = rows * (K / 32);
  if (tasks == 0) return cudaSuccess;
  return launch_pdl(k_pack, dim3(grid_for(tasks, 256)), dim3(256), 0, stream, src, rows, K,
                    half_rows, dst);
}

}  // namespace megamoe
