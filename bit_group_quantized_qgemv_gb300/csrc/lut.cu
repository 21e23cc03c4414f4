// lut.cu -- the LUT / palettised 4-bit GEMV: y[n] = sum_k lut[n / R][q[n][k]] x[k]
// (+ residual[n]), 4-bit codes 8 per uint32 (low nibble first) indexing a
// 16-entry fp16 table shared by R consecutive rows.
//
// Each warp takes RA rows at a time; lane l walks the 32-k chunks
// c = l + 32 j of those rows (one 16-byte load of codes per chunk and row).
// The table lookup runs in registers: a row's 16 entries become 8 byte
// planes (low and high bytes of entries 0-7 and 8-15), and one byte permute
// looks up 4 codes at once (their low 3 bits as the selector); a second
// permute turns bit 3 of each code into a byte mask that picks between the
// two halves of the table, and two more interleave the bytes into fp16
// pairs.  The products with the fp16 activations are exact in the mixed
// fma.rn.f32.f16 and accumulate in fp32.  x is staged in shared memory, its
// 16-byte pieces XOR-swizzled so that the 8 lanes of each quarter-warp read
// 8 different bank groups.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "epilogue_ops.h"
#include "qgemv_device.cuh"

namespace qgemv {
namespace {

constexpr int kLutThreads = 256;
constexpr int kLutWarps = kLutThreads / 32;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

// A table as byte planes: lo_a = low bytes of entries 0-3 / 4-7, lo_b of
// entries 8-11 / 12-15, hi_* the high bytes.
struct Planes {
  uint32_t lo_a0, lo_a1, lo_b0, lo_b1, hi_a0, hi_a1, hi_b0, hi_b1;
};

__device__ __forceinline__ Planes load_planes(const uint16_t* __restrict__ t) {
  const uint4 p = *reinterpret_cast<const uint4*>(t);      // entries 0..7
  const uint4 q = *reinterpret_cast<const uint4*>(t + 8);  // entries 8..15
  Planes L;
  L.lo_a0 = prmt(p.x, p.y, 0x6420u);
  L.hi_a0 = prmt(p.x, p.y, 0x7531u);
  L.lo_a1 = prmt(p.z, p.w, 0x6420u);
  L.hi_a1 = prmt(p.z, p.w, 0x7531u);
  L.lo_b0 = prmt(q.x, q.y, 0x6420u);
  L.hi_b0 = prmt(q.x, q.y, 0x7531u);
  L.lo_b1 = prmt(q.z, q.w, 0x6420u);
  L.hi_b1 = prmt(q.z, q.w, 0x7531u);
  return L;
}

// The entries of the 4 codes in the low 16 bits of v as fp16 pairs
// (e[q0], e[q1]) and (e[q2], e[q3]).
__device__ __forceinline__ void lookup4(const Planes& L, uint32_t v, uint32_t& p01,
                                        uint32_t& p23) {
  const uint32_t sel = v & 0x7777u;               // low 3 bits: byte within a half-table
  const uint32_t m = prmt(v << 4, v, 0xD9C8u);    // byte i = 0xFF when bit 3 of code i is set
  const uint32_t la = prmt(L.lo_a0, L.lo_a1, sel), lb = prmt(L.lo_b0, L.lo_b1, sel);
  const uint32_t ha = prmt(L.hi_a0, L.hi_a1, sel), hb = prmt(L.hi_b0, L.hi_b1, sel);
  const uint32_t lo = (la & ~m) | (lb & m);
  const uint32_t hi = (ha & ~m) | (hb & m);
  p01 = prmt(lo, hi, 0x5140u);
  p23 = prmt(lo, hi, 0x7362u);
}

// a += w_even * x_even, b += w_odd * x_odd over 8 weights: w and x as fp16
// pairs (k, k+1).
__device__ __forceinline__ void dot8(uint32_t w01, uint32_t w23, uint32_t w45, uint32_t w67,
                                     const uint4& x, float& a, float& b) {
  asm("{\n"
      ".reg .b16 w0, w1, w2, w3, w4, w5, w6, w7;\n"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7;\n"
      "mov.b32 {w0, w1}, %2;\n"
      "mov.b32 {w2, w3}, %3;\n"
      "mov.b32 {w4, w5}, %4;\n"
      "mov.b32 {w6, w7}, %5;\n"
      "mov.b32 {x0, x1}, %6;\n"
      "mov.b32 {x2, x3}, %7;\n"
      "mov.b32 {x4, x5}, %8;\n"
      "mov.b32 {x6, x7}, %9;\n"
      "fma.rn.f32.f16 %0, w0, x0, %0;\n"
      "fma.rn.f32.f16 %1, w1, x1, %1;\n"
      "fma.rn.f32.f16 %0, w2, x2, %0;\n"
      "fma.rn.f32.f16 %1, w3, x3, %1;\n"
      "fma.rn.f32.f16 %0, w4, x4, %0;\n"
      "fma.rn.f32.f16 %1, w5, x5, %1;\n"
      "fma.rn.f32.f16 %0, w6, x6, %0;\n"
      "fma.rn.f32.f16 %1, w7, x7, %1;\n"
      "}"
      : "+f"(a), "+f"(b)
      : "r"(w01), "r"(w23), "r"(w45), "r"(w67), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
}

// Physical index of 16-byte piece m (k = 32c + 8m .. +7) of chunk c of x.
__device__ __forceinline__ int x_piece(int c, int m) { return 4 * c + (m ^ ((c >> 1) & 3)); }

__device__ __forceinline__ void dot_chunk(const Planes& L, const uint4& w, const uint4* xs, int c,
                                          float& a, float& b) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t p01, p23, p45, p67;
    lookup4(L, words[m], p01, p23);
    lookup4(L, words[m] >> 16, p45, p67);
    dot8(p01, p23, p45, p67, xs[x_piece(c, m)], a, b);
  }
}

// RA rows per warp at a time; U chunks of each row per lane per step.
template <int RA, int U>
__global__ void __launch_bounds__(kLutThreads) lut_qgemv_kernel(
    const uint4* __restrict__ codes, const uint16_t* __restrict__ lut, int rows_per_lut,
    const uint4* __restrict__ x, const __half* __restrict__ residual, __half* __restrict__ y,
    int N, int K) {
  extern __shared__ __align__(16) uint4 xs[];  // K / 8 pieces, swizzled
  pdl_launch_dependents();
  const int C = K >> 5;  // 32-k chunks per row
  pdl_wait();            // x (and the residual) come from the previous kernel
  for (int p = threadIdx.x; p < (K >> 3); p += kLutThreads) xs[x_piece(p >> 2, p & 3)] = x[p];
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int groups = (N + RA - 1) / RA;
  const int stride = gridDim.x * kLutWarps;
  for (int g = blockIdx.x * kLutWarps + (threadIdx.x >> 5); g < groups; g += stride) {
    const int r0 = g * RA;
    Planes L[RA];
    float a[RA], b[RA];
#pragma unroll
    for (int r = 0; r < RA; ++r) {
      const int row = r0 + r < N ? r0 + r : N - 1;  // (a duplicate row is never stored)
      L[r] = load_planes(lut + static_cast<long long>(row / rows_per_lut) * 16);
      a[r] = 0.f;
      b[r] = 0.f;
    }
    for (int c0 = lane; c0 < C; c0 += 32 * U) {
      uint4 w[RA][U];
#pragma unroll
      for (int r = 0; r < RA; ++r) {
        const int row = r0 + r < N ? r0 + r : N - 1;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + 32 * u;
          w[r][u] = c < C ? __ldcs(codes + static_cast<long long>(row) * C + c)
                          : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c < C) {
#pragma unroll
          for (int r = 0; r < RA; ++r) dot_chunk(L[r], w[r][u], xs, c, a[r], b[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RA; ++r) {
      float s = a[r] + b[r];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const int row = r0 + r;
      if (lane == 0 && row < N) {
        if (residual) s += __half2float(residual[row]);
        y[row] = __float2half_rn(s);
      }
    }
  }
}

template <int RA, int U>
cudaError_t launch(const uint32_t* codes, const uint16_t* lut, int rows_per_lut, const __half* x,
                   const __half* residual, __half* y, int N, int K, int sms, cudaStream_t st) {
  const int smem = K * 2;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(lut_qgemv_kernel<RA, U>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  const long long groups = (static_cast<long long>(N) + RA - 1) / RA;
  long long blocks = (groups + kLutWarps - 1) / kLutWarps;
  const long long cap = static_cast<long long>(sms) * 4;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kLutThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lut_qgemv_kernel<RA, U>, reinterpret_cast<const uint4*>(codes),
                            lut, rows_per_lut, reinterpret_cast<const uint4*>(x), residual, y, N,
                            K);
}

}  // namespace

cudaError_t lut_qgemv_launch(const uint32_t* codes, const uint16_t* lut, int rows_per_lut,
                             const __half* x, const __half* residual, __half* y, int N, int K,
                             int sms, cudaStream_t st) {
  // Short rows: more rows in flight per warp; long rows: more chunks.
  if (K <= 2048) return launch<4, 1>(codes, lut, rows_per_lut, x, residual, y, N, K, sms, st);
  if (K <= 4096) return launch<2, 2>(codes, lut, rows_per_lut, x, residual, y, N, K, sms, st);
  return launch<1, 4>(codes, lut, rows_per_lut, x, residual, y, N, K, sms, st);
}

}  // namespace qgemv
