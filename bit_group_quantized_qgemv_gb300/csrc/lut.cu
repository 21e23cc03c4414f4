// lut.cu -- the LUT / palettised 4-bit GEMV: y[n] = sum_k lut[n / R][q[n][k]] x[k]
// (+ residual[n]), 4-bit codes 8 per uint32 (low nibble first) indexing a
// 16-entry fp16 table shared by R consecutive rows.
//
// Each warp walks its rows (warp w of W: rows w, w + W, ...) as a stream of
// items (row, j): lane l takes the 32-k chunk c = l + 32 j of the row, one
// 16-byte load of codes.  The loads run D items ahead of the arithmetic
// (a register ring unrolled by D), so every lane keeps D loads in flight
// whatever K is.  A row's table (32 bytes) is loaded by lanes 0 and 1 with
// the row's first item and handed to the warp by shuffles; one table for
// the whole tensor is read once.  The lookup runs in registers: the table
// as byte planes (low and high bytes of entries 0-7 and 8-15), one byte
// permute per 4 codes and plane with the codes' low 3 bits as selector, a
// permute-built byte mask from the codes' top bit to pick the half-table,
// and two permutes interleaving the bytes into fp16 pairs.  The products
// with the fp16 activations are exact in the mixed fma.rn.f32.f16 and
// accumulate in fp32.  x is staged in shared memory, its 16-byte pieces
// XOR-swizzled so that the 8 lanes of each quarter-warp read 8 different
// bank groups.
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

__device__ __forceinline__ Planes make_planes(const uint4& p, const uint4& q) {
  // p: entries 0..7, q: entries 8..15 (fp16 pairs, low entry in the low half)
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

// The table whose halves lanes 0 (entries 0..7) and 1 (8..15) hold in v.
__device__ __forceinline__ Planes planes_from_lanes(const uint4& v) {
  uint4 p, q;
  p.x = __shfl_sync(0xffffffffu, v.x, 0);
  p.y = __shfl_sync(0xffffffffu, v.y, 0);
  p.z = __shfl_sync(0xffffffffu, v.z, 0);
  p.w = __shfl_sync(0xffffffffu, v.w, 0);
  q.x = __shfl_sync(0xffffffffu, v.x, 1);
  q.y = __shfl_sync(0xffffffffu, v.y, 1);
  q.z = __shfl_sync(0xffffffffu, v.z, 1);
  q.w = __shfl_sync(0xffffffffu, v.w, 1);
  return make_planes(p, q);
}

// The entries of the 8 codes of w as fp16 pairs (e[q0], e[q1]), ...,
// (e[q6], e[q7]).
__device__ __forceinline__ void lookup8(const Planes& L, uint32_t w, uint32_t& p01, uint32_t& p23,
                                        uint32_t& p45, uint32_t& p67) {
  const uint32_t sl = w & 0x77777777u;   // low 3 bits of every code; a permute reads
  const uint32_t sh = sl >> 16;          // the low 4 selectors of its operand
  const uint32_t w4 = w << 4;
  const uint32_t ml = prmt(w4, w, 0xD9C8u);  // byte i = 0xFF when bit 3 of code i is set
  const uint32_t mh = prmt(w4, w, 0xFBEAu);  // the same for codes 4..7
  const uint32_t ll = (prmt(L.lo_a0, L.lo_a1, sl) & ~ml) | (prmt(L.lo_b0, L.lo_b1, sl) & ml);
  const uint32_t hl = (prmt(L.hi_a0, L.hi_a1, sl) & ~ml) | (prmt(L.hi_b0, L.hi_b1, sl) & ml);
  const uint32_t lh = (prmt(L.lo_a0, L.lo_a1, sh) & ~mh) | (prmt(L.lo_b0, L.lo_b1, sh) & mh);
  const uint32_t hh = (prmt(L.hi_a0, L.hi_a1, sh) & ~mh) | (prmt(L.hi_b0, L.hi_b1, sh) & mh);
  p01 = prmt(ll, hl, 0x5140u);
  p23 = prmt(ll, hl, 0x7362u);
  p45 = prmt(lh, hh, 0x5140u);
  p67 = prmt(lh, hh, 0x7362u);
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
    lookup8(L, words[m], p01, p23, p45, p67);
    dot8(p01, p23, p45, p67, xs[x_piece(c, m)], a, b);
  }
}

// The item pipeline: D loads of codes in flight per lane.  SHARED: one
// table serves every row (rows_per_lut >= N); it needs fewer registers, so
// four CTAs fit per SM instead of three.
template <int D, bool SHARED>
__global__ void __launch_bounds__(kLutThreads, SHARED ? 4 : 3) lut_qgemv_kernel(
    const uint4* __restrict__ codes, const uint16_t* __restrict__ lut, int rows_per_lut,
    const uint4* __restrict__ x, const __half* __restrict__ residual, __half* __restrict__ y,
    int N, int K) {
  extern __shared__ __align__(16) uint4 xs[];  // K / 8 pieces, swizzled
  pdl_launch_dependents();
  const int C = K >> 5;         // 32-k chunks per row
  const int J = (C + 31) >> 5;  // items per row
  const int lane = threadIdx.x & 31;
  const int W = gridDim.x * kLutWarps;
  const int gw = blockIdx.x * kLutWarps + (threadIdx.x >> 5);
  const long long rows_mine = gw < N ? (N - 1 - gw) / W + 1 : 0;
  const long long T = rows_mine * J;  // items of this warp

  uint4 bc[D], bl[D];
  // issue position: item (ir, ij) = row gw + ir W, chunk step ij
  long long ir = 0;
  int ij = 0;
  auto issue = [&](uint4& c_out, uint4& l_out) {
    if (ir < rows_mine) {
      const long long row = gw + ir * W;
      const int c = lane + 32 * ij;
      c_out = c < C ? __ldcs(codes + row * C + c) : make_uint4(0u, 0u, 0u, 0u);
      if (!SHARED && ij == 0 && lane < 2)
        l_out = *reinterpret_cast<const uint4*>(lut + (row / rows_per_lut) * 16 + 8 * lane);
      if (++ij == J) {
        ij = 0;
        ++ir;
      }
    }
  };
  // The weights do not depend on the previous kernel: start streaming them.
#pragma unroll
  for (int d = 0; d < D; ++d) issue(bc[d], bl[d]);
  Planes L{};
  if (SHARED)
    L = make_planes(*reinterpret_cast<const uint4*>(lut), *reinterpret_cast<const uint4*>(lut + 8));

  pdl_wait();  // x (and the residual) come from the previous kernel
  for (int p = threadIdx.x; p < (K >> 3); p += kLutThreads) xs[x_piece(p >> 2, p & 3)] = x[p];
  __syncthreads();

  // consume position
  long long cr = 0;
  int cj = 0;
  float a = 0.f, b = 0.f;
  for (long long t0 = 0; t0 < T; t0 += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (t0 + d < T) {  // uniform over the warp
        if (!SHARED && cj == 0) L = planes_from_lanes(bl[d]);
        const int c = lane + 32 * cj;
        if (c < C) dot_chunk(L, bc[d], xs, c, a, b);
        if (cj == J - 1) {
          float s = a + b;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          if (lane == 0) {
            const long long row = gw + cr * W;
            if (residual) s += __half2float(residual[row]);
            y[row] = __float2half_rn(s);
          }
          a = 0.f;
          b = 0.f;
          cj = 0;
          ++cr;
        } else {
          ++cj;
        }
        issue(bc[d], bl[d]);
      }
    }
  }
}

template <int D, bool SHARED>
cudaError_t launch(const uint32_t* codes, const uint16_t* lut, int rows_per_lut, const __half* x,
                   const __half* residual, __half* y, int N, int K, int sms, cudaStream_t st) {
  const int smem = K * 2;  // at most 32 KB
  long long blocks = (static_cast<long long>(N) + kLutWarps - 1) / kLutWarps;
  const long long cap = static_cast<long long>(sms) * (SHARED ? 4 : 3);  // CTAs resident per SM
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
  return cudaLaunchKernelEx(&cfg, lut_qgemv_kernel<D, SHARED>,
                            reinterpret_cast<const uint4*>(codes), lut, rows_per_lut,
                            reinterpret_cast<const uint4*>(x), residual, y, N, K);
}

}  // namespace

cudaError_t lut_qgemv_launch(const uint32_t* codes, const uint16_t* lut, int rows_per_lut,
                             const __half* x, const __half* residual, __half* y, int N, int K,
                             int sms, cudaStream_t st) {
  if (rows_per_lut >= N)
    return launch<4, true>(codes, lut, rows_per_lut, x, residual, y, N, K, sms, st);
  return launch<4, false>(codes, lut, rows_per_lut, x, residual, y, N, K, sms, st);
}

}  // namespace qgemv
