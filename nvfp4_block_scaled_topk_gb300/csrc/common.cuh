// Device helpers shared by the MegaMoE kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA / bulk copies and the tcgen05
// (5th-generation tensor core + tensor memory) instructions, the shared-memory
// and instruction descriptors of the block-scaled NVFP4 MMA, and the NVFP4
// element/scale encoders.  Every spin-wait here is bounded: it gives up after
// kWaitTimeoutNs of %globaltimer time or when the kernel's abort flag is set,
// and the caller then records MEGAMOE_DEV_TIMEOUT and unwinds.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/megamoe.h"

namespace megamoe {

constexpr uint64_t kWaitTimeoutNs = 4ull * 1000ull * 1000ull * 1000ull;  // 4 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: wait until the preceding kernel in the stream
// has completed and its memory is visible (call before touching global
// memory), and let the next kernel be scheduled early (it still waits).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with parity `parity` of `bar` has completed.  Returns
// false if the abort flag was raised or the wait ran past `limit_ns` (in which
// case the abort flag is raised here and `status` gets the TIMEOUT bit).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status, uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      set_status(status, MEGAMOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA and bulk copies (global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Fire-and-forget copy of global memory into L2 (no completion to wait on).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T with per-16-element E4M3 scales of A and B
// in tensor memory; M = 128, K = 64 (NVFP4 packed), N from the descriptor.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i gets lane (quarter*32 + i).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Thread i of a warp writes 4 consecutive 32-bit columns of lane
// (quarter*32 + i); a warp may only address its own 32-lane quarter.
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b,
                                                  uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// (8 rows x 128 bytes per 1024-byte atom, atoms 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride offset: 8-row atoms
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}

// Instruction descriptor of the block-scaled MMA: A and B E2M1, K-major,
// E4M3 scales, fp32 accumulate, M x N tile.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7)                                  // A format: E2M1
         | (1u << 10)                               // B format: E2M1
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16 (scale format bit 23 = E4M3)
}

// ---------------------------------------------------------------------------
// BFP16 (uint16 values offset by 32768, one power-of-two exponent per 16 rows
// x 8 columns): the storage of the forward's L2 output between the down GEMM
// and the combine
// ---------------------------------------------------------------------------
constexpr int kBfp16NonFinite = 127;  // exponent of a group holding Inf or NaN
// 2^s for |s| <= 126: a normal float, so scaling by it is exact.
__device__ __forceinline__ float bfp16_pow2(int s) {
  return __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
}
// Exponent of a group from the bits of its max |v| (sign bit clear):
// s = max(floor(log2 m) - 14, -126), plus one when m * 2^-s >= 32767.5, so
// that every value rounds to at most 32767 units; 0 for an all-zero group,
// kBfp16NonFinite when the group holds Inf or NaN.
__device__ __forceinline__ int bfp16_exponent(uint32_t mbits) {
  if (mbits >= 0x7f800000u) return kBfp16NonFinite;
  if (mbits == 0u) return 0;
  const int be = static_cast<int>(mbits >> 23);
  const int s = max(-126, (be == 0 ? -127 : be - 127) - 14);  // subnormal m: below 2^-126
  return __uint_as_float(mbits) * bfp16_pow2(-s) >= 32767.5f ? s + 1 : s;
}
// x (already scaled by 2^-s, |x| < 32767.5) -> the stored value
// rint(x) + 32768 (ties to even): adding 1.5 * 2^23 + 2^15 in round-to-
// nearest mode leaves 0x4B400000 + 32768 + rint(x) as the sum's bits (valid
// for |x| < 2^22), whose low 16 bits are the stored value.  ALU work only.
__device__ __forceinline__ uint16_t bfp16_round_int(float x) {
  return static_cast<uint16_t>(__float_as_uint(__fadd_rn(x, 12615680.f)));
}
// A 32-bit word's low (hi = false) or high stored value -> u - 32768 as a
// float, exactly: one byte permute builds the bits 0x4B40:u of 1.5 * 2^23 +
// u, and subtracting 1.5 * 2^23 + 2^15 is exact.
__device__ __forceinline__ float bfp16_offset_value(uint32_t word, bool hi) {
  return __fsub_rn(__uint_as_float(__byte_perm(word, 0x4B40u, hi ? 0x5432u : 0x5410u)),
                   12615680.f);
}
// Any group: the element's value (fp16 bits when s = kBfp16NonFinite).
__device__ __forceinline__ float bfp16_decode(uint32_t word, bool hi, int s) {
  if (s == kBfp16NonFinite)
    return __half2float(__ushort_as_half(static_cast<uint16_t>(hi ? word >> 16 : word)));
  return bfp16_offset_value(word, hi) * bfp16_pow2(s);
}

// ---------------------------------------------------------------------------
// NVFP4 element and scale codecs (float32 decisions, as the oracle takes them)
// ---------------------------------------------------------------------------
// Two floats -> one byte of two E2M1 codes, `lo` in the low nibble: the
// hardware conversion rounds to nearest (ties to the even code) onto the grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}, saturates to +-6 and keeps the sign of zero.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Non-negative float -> E4M3 byte, round-to-nearest-even, saturating to 448.
__device__ __forceinline__ uint32_t e4m3_code(float s) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3));
}

// E4M3 byte (non-negative, finite) -> float, exactly.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));   // (1 + m/8) * 2^(e-7)
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// Encode one 16-element block of bf16 values (two 128-bit words): 16 E2M1
// codes (8 bytes, element 2i in the low nibble of byte i) and the E4M3 scale
// byte, following the fixed float32 order
//   s = (amax_b * gs) / 6, s8 = e4m3(s), enc = gs / decode(s8), code = e2m1(x * enc).
__device__ __forceinline__ void encode_block(uint4 v0, uint4 v1, float gs, uint2& codes,
                                             uint32_t& s8) {
  float xv[16];
  const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    xv[2 * j] = bf16_bits_to_float(u[j] & 0xFFFFu);
    xv[2 * j + 1] = bf16_bits_to_float(u[j] >> 16);
  }
  float amax_b = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(xv[i]));
  const float s = __fdiv_rn(__fmul_rn(amax_b, gs), 6.0f);
  s8 = e4m3_code(s);
  const float sd = e4m3_value(s8);
  uint32_t c0 = 0, c1 = 0;
  if (sd > 0.f) {
    const float enc = __fdiv_rn(gs, sd);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c0 |= e2m1x2(__fmul_rn(xv[2 * i], enc), __fmul_rn(xv[2 * i + 1], enc)) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c1 |= e2m1x2(__fmul_rn(xv[8 + 2 * i], enc), __fmul_rn(xv[9 + 2 * i], enc)) << (8 * i);
  }
  codes = make_uint2(c0, c1);
}

// Atom-layout byte offset of the 4-byte scale word of (row, 64-element slice).
__host__ __device__ __forceinline__ int64_t sf_atom_offset(int64_t row, int slice, int slices) {
  return ((row >> 7) * slices + slice) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

}  // namespace megamoe
