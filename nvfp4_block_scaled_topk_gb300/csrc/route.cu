// Token bucketing: per-expert counts, expert_offsets, padded_expert_offsets
// and the stable permutation ("CURRENT_BUG.md -- DeepSeek-V4 Blackwell NVFP4",
// "Test Plan -- Finding the NaN", Phase 1: variable token counts per expert
// padded to 128; Phase 2: zero-token experts, expert_offsets and
// padded_expert_offsets).
//
// One thread block of 32 warps.  Warp w owns a contiguous chunk of the flat
// slots, so the order "chunk, then position inside the chunk" is the flat slot
// order and the sort is stable without atomics deciding anything:
//   1. per-warp histograms hist[w][e] (shared-memory atomics; counts only);
//   2. per expert: the total, then hist[w][e] becomes the exclusive prefix over
//      warps; a block scan over experts gives offsets and padded offsets;
//   3. each warp walks its chunk 32 slots at a time; lanes with the same expert
//      find each other with __match_any_sync, rank = earlier peers + the running
//      count of that expert in this warp.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "router.cuh"

namespace megamoe {

constexpr int kRouteWarps = 32;
constexpr int kRouteThreads = kRouteWarps * 32;

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int t = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_sums[lane] = t - s;  // exclusive warp base
    if (lane == 31) *total = t;
  }
  __syncthreads();
  const int r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

// The routing itself, for one block of kRouteThreads threads.  `smem` holds
// 32*E + 2*E + 1 ints.  Ends with the block's global writes issued; callers
// that read them back in the same block synchronise first.
__device__ void route_block(const int32_t* ids, int n_slots, int E, int pad,
                            int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                            int32_t* row_src, int64_t row_capacity, int32_t* slot_dst,
                            uint32_t* status, uint32_t* zero_words, int n_zero, int* smem) {
  int* hist = smem;                        // [32][E]
  int* s_poff = hist + kRouteWarps * E;    // [E+1]
  int* s_cnt = s_poff + (E + 1);           // [E]
  __shared__ int warp_sums[32];
  __shared__ int totals[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < n_zero; i += kRouteThreads) zero_words[i] = 0u;
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();

  const int chunk = (n_slots + kRouteWarps - 1) / kRouteWarps;
  const int s_begin = warp * chunk;
  const int s_end = min(n_slots, s_begin + chunk);

  // 1. per-warp histograms (four 32-slot groups of ids loaded per round)
  bool bad = false;
  for (int b0 = s_begin; b0 < s_end; b0 += 128) {  // warp-uniform bounds
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int sv = b0 + 32 * u + lane;
      ev[u] = sv < s_end ? ids[sv] : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (ev[u] >= E) bad = true;
      else if (ev[u] >= 0) atomicAdd(&hist[warp * E + ev[u]], 1);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MEGAMOE_DEV_BAD_EXPERT_ID);
  __syncthreads();

  // 2. totals, per-warp exclusive bases, offsets (E <= 1024: one expert per thread)
  int cnt = 0, padded = 0;
  if (tid < E) {
    for (int w = 0; w < kRouteWarps; ++w) {
      const int h = hist[w * E + tid];
      hist[w * E + tid] = cnt;
      cnt += h;
    }
    padded = (cnt + pad - 1) / pad * pad;
  }
  const int off = block_exclusive_scan_1024(cnt, warp_sums, &totals[0]);
  const int poff = block_exclusive_scan_1024(padded, warp_sums, &totals[1]);
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = off;
    padded_offsets[tid] = poff;
    s_poff[tid] = poff;
    s_cnt[tid] = cnt;
  }
  if (tid == 0) {
    offsets[E] = totals[0];
    padded_offsets[E] = totals[1];
    s_poff[E] = totals[1];
  }
  __syncthreads();

  // 3. stable scatter, warp by warp over its own chunk, 32 slots at a time in
  //    order (the ids of four groups loaded per round)
  int ev[4];
  for (int base = s_begin; base < s_end; base += 32) {
    const int u = ((base - s_begin) >> 5) & 3;
    if (u == 0) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int sv = base + 32 * v + lane;
        ev[v] = sv < s_end ? ids[sv] : -1;
      }
    }
    const int s = base + lane;
    const bool in = s < s_end;
    int e = -1;
#pragma unroll
    for (int v = 0; v < 4; ++v)
      if (v == u) e = ev[v];
    if (e >= E) e = -1;
    const unsigned active = __ballot_sync(0xffffffffu, in);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (in) {
      if (e >= 0) {
        const unsigned lower = peers & ((1u << lane) - 1u);
        const int rank = hist[warp * E + e] + __popc(lower);
        const int row = s_poff[e] + rank;
        row_src[row] = s;
        slot_dst[s] = row;
      } else {
        slot_dst[s] = -1;
      }
    }
    __syncwarp();
    // the highest lane of each peer group advances that expert's running count
    if (in && e >= 0 && (31 - __clz(peers & active)) == lane)
      hist[warp * E + e] += __popc(peers & active);
    __syncwarp();
  }

  // padding rows of every expert, then everything past the last expert
  for (int e = tid; e < E; e += kRouteThreads) {
    for (int r = s_poff[e] + s_cnt[e]; r < s_poff[e + 1]; ++r) row_src[r] = -1;
  }
  for (int64_t r = s_poff[E] + tid; r < row_capacity; r += kRouteThreads) row_src[r] = -1;
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    k_route(const int32_t* ids, int n_slots, int E, int pad, int32_t* counts,
            int32_t* offsets, int32_t* padded_offsets, int32_t* row_src, int64_t row_capacity,
            int32_t* slot_dst, uint32_t* status, uint32_t* zero_words, int n_zero) {
  extern __shared__ int smem_route[];
  pdl_wait();
  pdl_trigger();
  route_block(ids, n_slots, E, pad, counts, offsets, padded_offsets, row_src, row_capacity,
              slot_dst, status, zero_words, n_zero, smem_route);
}

// ---------------------------------------------------------------------------
// Large batches: the same routing over many blocks, in three passes.  Block b
// owns the contiguous slot chunk [b * chunk, (b + 1) * chunk), so "block,
// then warp, then position" is still the flat slot order and the result is
// identical to route_block's:
//   1. k_route_hist: per-block expert histograms -> hist[e][b] (expert-major,
//      rows of bstride >= blocks ints, bstride a multiple of 4);
//   2. k_route_offsets (one block): counts, offsets, padded offsets, and each
//      block's exclusive base per expert (hist rewritten in place; thread e
//      walks its row in 16-byte loads, eight in flight);
//   3. k_route_scatter: per block, per-warp histograms of its chunk on top of
//      the block's bases, then the stable scatter as in route_block; the
//      padding rows are spread over the blocks; ids >= E are flagged here
//      (after pass 1 cleared the status word).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouteThreads) k_route_hist(const int32_t* __restrict__ ids,
                                                              int n_slots, int E, int chunk,
                                                              int bstride,
                                                              int32_t* __restrict__ hist,
                                                              uint32_t* zero_words, int n_zero) {
  extern __shared__ int sh_hist[];  // [E]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  if (blockIdx.x == 0)
    for (int i = tid; i < n_zero; i += kRouteThreads) zero_words[i] = 0u;
  for (int e = tid; e < E; e += kRouteThreads) sh_hist[e] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * chunk, s1 = min(n_slots, s0 + chunk);
  for (int sv = s0 + tid; sv < s1; sv += kRouteThreads) {
    const int e = __ldg(ids + sv);
    if (e >= 0 && e < E) atomicAdd(&sh_hist[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kRouteThreads)
    hist[static_cast<int64_t>(e) * bstride + blockIdx.x] = sh_hist[e];
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    k_route_offsets(int n_blocks, int bstride, int E, int pad, int32_t* __restrict__ hist,
                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ padded_offsets) {
  __shared__ int warp_sums[32];
  __shared__ int totals[2];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  int cnt = 0, padded = 0;
  if (tid < E) {  // E <= 1024: one expert per thread, its row of block counts
    int4* row = reinterpret_cast<int4*>(hist + static_cast<int64_t>(tid) * bstride);
    const int vecs = bstride / 4;
    for (int j0 = 0; j0 < vecs; j0 += 8) {
      int4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = j0 + i < vecs ? row[j0 + i] : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (j0 + i >= vecs) break;
        const int b = 4 * (j0 + i);  // entries past the last block are not counts
        int4 o;
        o.x = cnt;
        cnt += b + 0 < n_blocks ? v[i].x : 0;
        o.y = cnt;
        cnt += b + 1 < n_blocks ? v[i].y : 0;
        o.z = cnt;
        cnt += b + 2 < n_blocks ? v[i].z : 0;
        o.w = cnt;
        cnt += b + 3 < n_blocks ? v[i].w : 0;
        row[j0 + i] = o;
      }
    }
    padded = (cnt + pad - 1) / pad * pad;
  }
  const int off = block_exclusive_scan_1024(cnt, warp_sums, &totals[0]);
  const int poff = block_exclusive_scan_1024(padded, warp_sums, &totals[1]);
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = off;
    padded_offsets[tid] = poff;
  }
  if (tid == 0) {
    offsets[E] = totals[0];
    padded_offsets[E] = totals[1];
  }
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    k_route_scatter(const int32_t* __restrict__ ids, int n_slots, int E, int chunk, int bstride,
                    const int32_t* __restrict__ hist, const int32_t* __restrict__ counts,
                    const int32_t* __restrict__ padded_offsets, int32_t* row_src,
                    int64_t row_capacity, int32_t* slot_dst, uint32_t* status) {
  extern __shared__ int smem_sc[];
  int* whist = smem_sc;                 // [32][E]: per-warp running rows
  int* s_poff = whist + kRouteWarps * E;  // [E + 1]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) whist[i] = 0;
  for (int e = tid; e <= E; e += kRouteThreads) s_poff[e] = padded_offsets[e];
  __syncthreads();
  const int b0 = blockIdx.x * chunk, b1 = min(n_slots, b0 + chunk);
  const int wchunk = (max(b1 - b0, 0) + kRouteWarps - 1) / kRouteWarps;
  const int s_begin = min(b1, b0 + warp * wchunk);
  const int s_end = min(b1, s_begin + wchunk);
  // per-warp histograms of the warp's part of the chunk
  bool bad = false;
  for (int c0 = s_begin; c0 < s_end; c0 += 32) {  // warp-uniform bounds
    const int sv = c0 + lane;
    const int e = sv < s_end ? __ldg(ids + sv) : -1;
    if (e >= E) bad = true;
    else if (e >= 0) atomicAdd(&whist[warp * E + e], 1);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MEGAMOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  // exclusive over warps, on top of this block's base from pass 2
  for (int e = tid; e < E; e += kRouteThreads) {
    int base = hist[static_cast<int64_t>(e) * bstride + blockIdx.x];
    for (int w = 0; w < kRouteWarps; ++w) {
      const int h = whist[w * E + e];
      whist[w * E + e] = base;
      base += h;
    }
  }
  __syncthreads();
  // stable scatter, 32 slots at a time in order
  for (int c0 = s_begin; c0 < s_end; c0 += 32) {
    const int sv = c0 + lane;
    const bool in = sv < s_end;
    int e = in ? __ldg(ids + sv) : -1;
    if (e >= E) e = -1;
    const unsigned active = __ballot_sync(0xffffffffu, in);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (in) {
      if (e >= 0) {
        const unsigned lower = peers & ((1u << lane) - 1u);
        const int row = s_poff[e] + whist[warp * E + e] + __popc(lower);
        row_src[row] = sv;
        slot_dst[sv] = row;
      } else {
        slot_dst[sv] = -1;
      }
    }
    __syncwarp();
    if (in && e >= 0 && (31 - __clz(peers & active)) == lane)
      whist[warp * E + e] += __popc(peers & active);
    __syncwarp();
  }
  // padding rows of every expert, then everything past the last expert,
  // spread over the blocks
  const int gtid = blockIdx.x * kRouteThreads + tid;
  const int gthreads = gridDim.x * kRouteThreads;
  for (int e = gtid; e < E; e += gthreads) {
    const int c = __ldg(counts + e);
    for (int r = s_poff[e] + c; r < s_poff[e + 1]; ++r) row_src[r] = -1;
  }
  for (int64_t r = s_poff[E] + gtid; r < row_capacity; r += gthreads) row_src[r] = -1;
}

// Small batches: route and the amax of x in this one block (the quantisation
// itself, ALU-heavy, runs spread over many SMs in the next kernel).
constexpr int64_t kPrologueMaxElems = 262144;  // T * d read by one block

__global__ void __launch_bounds__(kRouteThreads, 1)
    k_prologue(const int32_t* ids, int T, int k, int E, int pad, int32_t* counts,
               int32_t* offsets, int32_t* padded_offsets, int32_t* row_src,
               int64_t row_capacity, int32_t* slot_dst, uint32_t* status, uint32_t* zero_words,
               int n_zero, const uint16_t* __restrict__ x, int d, float* amax_out,
               const RouterArgs r) {
  extern __shared__ int smem_route[];
  __shared__ uint32_t red[kRouteWarps];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // amax of x on the bf16 bit patterns (monotone for finite values); the
  // first kPre vectors per thread are loaded before the routing so that their
  // latency overlaps it
  constexpr int kPre = 8;
  const int64_t vecs = static_cast<int64_t>(T) * (d / 8);
  uint4 pre[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int64_t i = tid + static_cast<int64_t>(j) * kRouteThreads;
    pre[j] = i < vecs ? __ldg(reinterpret_cast<const uint4*>(x) + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (r.logits) {
    // the router first: warp w takes tokens w, w + 32, ...; its score row
    // lives in the routing histogram's shared memory, not yet in use
    float* s_row = reinterpret_cast<float*>(smem_route) + warp * r.n_logits;
    for (int t = warp; t < T; t += kRouteWarps)
      router_token(r.logits + static_cast<int64_t>(t) * r.ld, r.bias, r.n_logits, r.k_routed,
                   r.shared, s_row, r.ids_out + static_cast<int64_t>(t) * k,
                   r.w_out + static_cast<int64_t>(t) * k, lane);
    __syncthreads();  // the ids are read back below by every warp
    ids = r.ids_out;
  }
  route_block(ids, T * k, E, pad, counts, offsets, padded_offsets, row_src, row_capacity,
              slot_dst, status, zero_words, n_zero, smem_route);
  uint32_t m2 = 0;
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    m2 = __vmaxu2(m2, pre[j].x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, pre[j].y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, pre[j].z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, pre[j].w & 0x7FFF7FFFu);
  }
  for (int64_t i = tid + static_cast<int64_t>(kPre) * kRouteThreads; i < vecs;
       i += kRouteThreads) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + i);
    m2 = __vmaxu2(m2, q.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, q.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, q.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, q.w & 0x7FFF7FFFu);
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();  // also orders the status word's clearing before the write below
  if (tid == 0) {
    for (int w = 1; w < kRouteWarps; ++w) m = max(m, red[w]);
    if (m >= 0x7F80u) {  // Inf or NaN
      set_status(status, MEGAMOE_DEV_NONFINITE);
      m = 0x7F7Fu;
    }
    *amax_out = __uint_as_float(m << 16);
  }
}

// Expert-parallel shard (experts [base, base + E_local) of E_total): a global
// id becomes the shard's local id, -1 (skipped) when another shard owns it or
// it is negative, and E_local (out of the shard's range: flagged and skipped
// by the routing) when it is not a valid expert at all.
__global__ void __launch_bounds__(256) k_ep_remap(const int32_t* __restrict__ ids, int64_t n,
                                                  int base, int E_local, int E_total,
                                                  int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int id = __ldg(ids + i);
    int r = -1;
    if (id >= E_total) r = E_local;
    else if (id >= base && id < base + E_local) r = id - base;
    out[i] = r;
  }
}

cudaError_t launch_ep_remap(const int32_t* ids, int64_t n, int base, int E_local, int E_total,
                            int32_t* out, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(k_ep_remap, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, ids, n,
                    base, E_local, E_total, out);
}

size_t route_smem_bytes(int E) { return sizeof(int) * (static_cast<size_t>(kRouteWarps) * E + 2 * E + 1); }

cudaError_t launch_route(const int32_t* ids, int n_slots, int E, int pad, int32_t* counts,
                         int32_t* offsets, int32_t* padded_offsets, int32_t* row_src,
                         int64_t row_capacity, int32_t* slot_dst, uint32_t* status,
                         uint32_t* zero_words, int n_zero, cudaStream_t stream,
                         int32_t* block_hist) {
  const size_t smem = route_smem_bytes(E);
  if (block_hist && n_slots >= kRouteMultiMinSlots) {
    // chunks of at least 1024 slots, one per block, at most one block per SM
    const int blocks_max = std::min(kRouteMaxBlocks, num_sms());
    int chunk = (n_slots + blocks_max - 1) / blocks_max;
    chunk = std::max(1024, (chunk + 31) / 32 * 32);
    const int blocks = (n_slots + chunk - 1) / chunk;
    const int bstride = (blocks + 3) / 4 * 4;  // <= kRouteMaxBlocks
    cudaError_t err = launch_pdl(k_route_hist, dim3(blocks), dim3(kRouteThreads),
                                 sizeof(int) * static_cast<size_t>(E), stream, ids, n_slots, E,
                                 chunk, bstride, block_hist, zero_words, n_zero);
    if (err == cudaSuccess)
      err = launch_pdl(k_route_offsets, dim3(1), dim3(kRouteThreads), 0, stream, blocks, bstride,
                       E, pad, block_hist, counts, offsets, padded_offsets);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_route_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
    if (err == cudaSuccess)
      err = launch_pdl(k_route_scatter, dim3(blocks), dim3(kRouteThreads), smem, stream, ids,
                       n_slots, E, chunk, bstride, static_cast<const int32_t*>(block_hist),
                       static_cast<const int32_t*>(counts),
                       static_cast<const int32_t*>(padded_offsets), row_src, row_capacity,
                       slot_dst, status);
    return err;
  }
  cudaError_t err = cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(k_route, dim3(1), dim3(kRouteThreads), smem, stream, ids, n_slots, E, pad,
                    counts, offsets, padded_offsets, row_src, row_capacity, slot_dst, status,
                    zero_words, n_zero);
}

bool prologue_fits(int T, int d) {
  return static_cast<int64_t>(T) * d <= kPrologueMaxElems && d % 64 == 0;
}

cudaError_t launch_prologue(const int32_t* ids, int T, int k, int E, int pad, int32_t* counts,
                            int32_t* offsets, int32_t* padded_offsets, int32_t* row_src,
                            int64_t row_capacity, int32_t* slot_dst, uint32_t* status,
                            uint32_t* zero_words, int n_zero, const uint16_t* x, int d,
                            float* amax, cudaStream_t stream, const RouterArgs* router) {
  const size_t smem = route_smem_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(k_prologue, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const RouterArgs none{};
  return launch_pdl(k_prologue, dim3(1), dim3(kRouteThreads), smem, stream, ids, T, k, E, pad,
                    counts, offsets, padded_offsets, row_src, row_capacity, slot_dst, status,
                    zero_words, n_zero, x, d, amax, router ? *router : none);
}

}  // namespace megamoe
