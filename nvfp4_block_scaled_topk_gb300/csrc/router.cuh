// The router step for one token, run by one warp (used by the router kernel
// and by the small-batch prologue, so both select and weigh identically):
//   score[e] = fl32(logit[e] + bias[e]) (bias optional); the k experts of
//   highest score in descending order, ties to the lower expert index; the
//   weights are the softmax of the selected logits in fp32; an optional
//   shared expert is appended with weight 1.
// `s_row` is E floats of shared memory owned by the warp.
#pragma once

#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

namespace megamoe {

__device__ __forceinline__ void router_token(const float* __restrict__ lrow,
                                             const float* __restrict__ bias, int E, int k,
                                             int shared, float* s_row, int32_t* ids_row,
                                             float* w_row, int lane) {
  for (int e = lane; e < E; e += 32) {
    const float l = __ldg(lrow + e);
    s_row[e] = bias ? __fadd_rn(l, __ldg(bias + e)) : l;
  }
  __syncwarp();
  int my_id = -1;
  float my_logit = 0.f;
  for (int j = 0; j < k; ++j) {
    // this lane's best remaining expert (taken ones hold NaN); experts ascend
    // along the lane's walk, so strict > keeps the lower index on ties
    float bv = 0.f;
    int be = -1;
    for (int e = lane; e < E; e += 32) {
      const float v = s_row[e];
      if (v == v && (be < 0 || v > bv)) {
        bv = v;
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if (be < 0) break;  // fewer than k experts (refused on the host)
    if (lane == 0) s_row[be] = __int_as_float(0x7fc00000);  // taken
    if (lane == j) {
      my_id = be;
      my_logit = __ldg(lrow + be);
    }
    __syncwarp();
  }
  float m = lane < k ? my_logit : -FLT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ex = lane < k ? expf(my_logit - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    ids_row[lane] = my_id;
    w_row[lane] = ex / sum;
  } else if (lane == k && shared >= 0) {
    ids_row[lane] = shared;
    w_row[lane] = 1.f;
  }
  __syncwarp();  // s_row is reused for the warp's next token
}

}  // namespace megamoe
