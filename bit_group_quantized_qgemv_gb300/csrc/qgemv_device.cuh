// qgemv_device.cuh -- device-side building blocks of the sm_103a kernels:
// bounded mbarrier waits, 1-D TMA bulk copies, the dequant-dot inner loops
// and the per-row epilogues.  GPU path only (shares nothing with the oracle).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "qgemv_args.h"

namespace qgemv {

// Library status bits kept in device memory (one word per translation unit).
constexpr unsigned kStatusWaitTimeout = 1u;

// 2^24 and 2^-24: the dot products below run on fp16 subnormal codes
// (q * 2^-24), so every partial sum carries a 2^-24 scale until the epilogue.
constexpr float kTwo24 = 16777216.0f;
constexpr float kTwoM24 = 5.9604644775390625e-08f;

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds; it
// resumes as soon as the phase completes, so a waiting warp does not spin
// through issue slots that computing warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after about one second of wall time (the only legitimate waits are for
// DRAM copies and sibling warps, microseconds at most), records the timeout
// in *status and returns false: kernels then stop instead of hanging.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned* status,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* status) {
  return mbar_wait_for(bar, parity, status, 1000000000ull);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// L2 policy for weights: streamed once, evict first so activations stay.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D TMA bulk copy global -> shared (this CTA), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Order-preserving 64-bit key of (fp32 value, index): larger value first,
// then the lower index; 0 is below every key.
__device__ __forceinline__ unsigned long long argmax_key(float v, int index) {
  unsigned b = __float_as_uint(v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(b) << 32) | static_cast<unsigned>(~index);
}

__device__ __forceinline__ unsigned long long max_key(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Programmatic dependent launch: let the next kernel of the stream start
// launching (its CTAs take SMs as this grid's CTAs exit), and wait until
// the previous kernel's grid has completed with its memory visible.  Both
// are no-ops for a launch without that dependency.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

// ---------------------------------------------------------- dequant dots
//
// A 4-bit word holds codes q_0..q_7 (k = 8i .. 8i+7) low nibble first.
// Masking with 0x000F000F keeps q_0 and q_4 in the low mantissa bits of two
// fp16 lanes with a zero exponent: the fp16 subnormals q_0 * 2^-24 and
// q_4 * 2^-24, exactly.  0x00F000F0 gives 16 q_1 * 2^-24 and 16 q_5 * 2^-24;
// the word shifted right by 8 gives (q_2, q_6) and (q_3, q_7) the same way.
// The mixed fma.rn.f32.f16 multiplies such a code by an fp16 activation
// exactly and accumulates in fp32, so
//   a accumulates q x 2^-24      over q_0, q_2, q_4, q_6
//   b accumulates 16 q x 2^-24   over q_1, q_3, q_5, q_7
// and (a + b / 16) * 2^24 = sum_k q_k x_k: the group's sum of code times
// activation with fp32 accumulation and no offset to cancel (every product
// is exact; the power-of-two scale leaves all roundings relative to
// sum |q x|).  The group then adds scale * that + bias * sum(x): the
// fma(q, scale*x, bias*x) form of the FMA-reordered dequantisation,
// factored over the 64 k of a group.
//
// The activations come packed in the same pairing as the code lanes:
// xp[j] = (x_{8i+j}, x_{8i+j+4}) for j = 0..3 (low half first), so every
// fma pairs the low (high) half of a code register with the low (high) half
// of an activation register; the fma reads either half directly, so no
// instruction unpacks anything.
__device__ __forceinline__ void dot_word4(uint32_t w, const uint32_t* xp, float& a, float& b) {
  asm("{\n"
      ".reg .b32 v0, v1, v2, v3, w8;\n"
      ".reg .b16 q0, q1, q2, q3, q4, q5, q6, q7;\n"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7;\n"
      "and.b32 v0, %2, 0x000F000F;\n"
      "and.b32 v1, %2, 0x00F000F0;\n"
      "shr.u32 w8, %2, 8;\n"
      "and.b32 v2, w8, 0x000F000F;\n"
      "and.b32 v3, w8, 0x00F000F0;\n"
      "mov.b32 {q0, q4}, v0;\n"
      "mov.b32 {q1, q5}, v1;\n"
      "mov.b32 {q2, q6}, v2;\n"
      "mov.b32 {q3, q7}, v3;\n"
      "mov.b32 {x0, x4}, %3;\n"
      "mov.b32 {x1, x5}, %4;\n"
      "mov.b32 {x2, x6}, %5;\n"
      "mov.b32 {x3, x7}, %6;\n"
      "fma.rn.f32.f16 %0, q0, x0, %0;\n"
      "fma.rn.f32.f16 %1, q1, x1, %1;\n"
      "fma.rn.f32.f16 %0, q4, x4, %0;\n"
      "fma.rn.f32.f16 %1, q5, x5, %1;\n"
      "fma.rn.f32.f16 %0, q2, x2, %0;\n"
      "fma.rn.f32.f16 %1, q3, x3, %1;\n"
      "fma.rn.f32.f16 %0, q6, x6, %0;\n"
      "fma.rn.f32.f16 %1, q7, x7, %1;\n"
      "}"
      : "+f"(a), "+f"(b)
      : "r"(w), "r"(xp[0]), "r"(xp[1]), "r"(xp[2]), "r"(xp[3]));
}

// A 2-bit word holds codes c_0..c_15 (k = 16i .. 16i+15), low bits first.
// Masks 0x00030003, 0x000C000C, 0x00300030, 0x00C000C0 (on the word and on
// the word >> 8) yield fp16 subnormals m * c * 2^-24 with m = 1, 4, 16, 64,
// lane pairs (c_j, c_{j+8}).  Class accumulators a (m=1), b (4), c (16),
// d (64):  sum_k c_k x_k = (a + b / 4 + c / 16 + d / 64) * 2^24.
// Activations packed xp[j] = (x_{16i+j}, x_{16i+j+8}) for j = 0..7.
__device__ __forceinline__ void dot_word2(uint32_t w, const uint32_t* xp, float& a, float& b,
                                          float& c, float& d) {
  asm("{\n"
      ".reg .b32 v0, v1, v2, v3, v4, v5, v6, v7, w8;\n"
      ".reg .b16 p0, p1, p2, p3, p4, p5, p6, p7, p8, p9, p10, p11, p12, p13, p14, p15;\n"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7, x8, x9, x10, x11, x12, x13, x14, x15;\n"
      "and.b32 v0, %4, 0x00030003;\n"
      "and.b32 v1, %4, 0x000C000C;\n"
      "and.b32 v2, %4, 0x00300030;\n"
      "and.b32 v3, %4, 0x00C000C0;\n"
      "shr.u32 w8, %4, 8;\n"
      "and.b32 v4, w8, 0x00030003;\n"
      "and.b32 v5, w8, 0x000C000C;\n"
      "and.b32 v6, w8, 0x00300030;\n"
      "and.b32 v7, w8, 0x00C000C0;\n"
      "mov.b32 {p0, p8}, v0;\n"
      "mov.b32 {p1, p9}, v1;\n"
      "mov.b32 {p2, p10}, v2;\n"
      "mov.b32 {p3, p11}, v3;\n"
      "mov.b32 {p4, p12}, v4;\n"
      "mov.b32 {p5, p13}, v5;\n"
      "mov.b32 {p6, p14}, v6;\n"
      "mov.b32 {p7, p15}, v7;\n"
      "mov.b32 {x0, x8}, %5;\n"
      "mov.b32 {x1, x9}, %6;\n"
      "mov.b32 {x2, x10}, %7;\n"
      "mov.b32 {x3, x11}, %8;\n"
      "mov.b32 {x4, x12}, %9;\n"
      "mov.b32 {x5, x13}, %10;\n"
      "mov.b32 {x6, x14}, %11;\n"
      "mov.b32 {x7, x15}, %12;\n"
      "fma.rn.f32.f16 %0, p0, x0, %0;\n"
      "fma.rn.f32.f16 %1, p1, x1, %1;\n"
      "fma.rn.f32.f16 %2, p2, x2, %2;\n"
      "fma.rn.f32.f16 %3, p3, x3, %3;\n"
      "fma.rn.f32.f16 %0, p8, x8, %0;\n"
      "fma.rn.f32.f16 %1, p9, x9, %1;\n"
      "fma.rn.f32.f16 %2, p10, x10, %2;\n"
      "fma.rn.f32.f16 %3, p11, x11, %3;\n"
      "fma.rn.f32.f16 %0, p4, x4, %0;\n"
      "fma.rn.f32.f16 %1, p5, x5, %1;\n"
      "fma.rn.f32.f16 %2, p6, x6, %2;\n"
      "fma.rn.f32.f16 %3, p7, x7, %3;\n"
      "fma.rn.f32.f16 %0, p12, x12, %0;\n"
      "fma.rn.f32.f16 %1, p13, x13, %1;\n"
      "fma.rn.f32.f16 %2, p14, x14, %2;\n"
      "fma.rn.f32.f16 %3, p15, x15, %3;\n"
      "}"
      : "+f"(a), "+f"(b), "+f"(c), "+f"(d)
      : "r"(w), "r"(xp[0]), "r"(xp[1]), "r"(xp[2]), "r"(xp[3]), "r"(xp[4]), "r"(xp[5]),
        "r"(xp[6]), "r"(xp[7]));
}

// An 8-bit word holds codes q_0..q_3 (k = 4i .. 4i+3), low byte first.
// Masking with 0x00FF00FF keeps q_0 and q_2 as fp16 subnormals q * 2^-24
// (exact: q < 1024), and the word shifted right by 8 gives q_1 and q_3 the
// same way, so one accumulator takes all four products: a += q x 2^-24.
// Activations packed xp[0] = (x_{4i}, x_{4i+2}), xp[1] = (x_{4i+1}, x_{4i+3}).
__device__ __forceinline__ void dot_word8(uint32_t w, const uint32_t* xp, float& a, float& b) {
  asm("{\n"
      ".reg .b32 v0, v1;\n"
      ".reg .b16 q0, q1, q2, q3, x0, x1, x2, x3;\n"
      "and.b32 v0, %2, 0x00FF00FF;\n"
      "shr.u32 v1, %2, 8;\n"
      "and.b32 v1, v1, 0x00FF00FF;\n"
      "mov.b32 {q0, q2}, v0;\n"
      "mov.b32 {q1, q3}, v1;\n"
      "mov.b32 {x0, x2}, %3;\n"
      "mov.b32 {x1, x3}, %4;\n"
      "fma.rn.f32.f16 %0, q0, x0, %0;\n"
      "fma.rn.f32.f16 %1, q1, x1, %1;\n"
      "fma.rn.f32.f16 %0, q2, x2, %0;\n"
      "fma.rn.f32.f16 %1, q3, x3, %1;\n"
      "}"
      : "+f"(a), "+f"(b)
      : "r"(w), "r"(xp[0]), "r"(xp[1]));
}

// Code q of k within a packed word (generic path).
template <int BITS>
__device__ __forceinline__ int unpack_code(uint32_t word, int j) {
  return static_cast<int>((word >> (BITS * j)) & ((1u << BITS) - 1u));
}

// ------------------------------------------------------------ epilogues

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

}  // namespace qgemv
