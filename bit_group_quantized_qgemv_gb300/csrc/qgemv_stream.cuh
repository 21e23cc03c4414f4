// qgemv_stream.cuh -- the streaming dequant-fused GEMV kernel for sm_103a.
//
// Design (GB300-first; the Metal simdgroup-per-row-band kernels the pages
// describe in INFERENCE_RESEARCH.md section 1 are prior art, not the plan):
//
//  * Persistent: one CTA per SM.  CTA b owns the contiguous row range
//    [b*R/P, (b+1)*R/P) of the R output rows (P CTAs), so every SM streams
//    the same number of bytes and a CTA's codes, scales and biases are three
//    contiguous blocks of memory.
//  * Warp 0 (one lane) is the producer: it streams the range in stages of RS
//    rows with 1-D TMA bulk copies (cp.async.bulk, L2 evict-first) into an
//    NS-deep shared-memory ring guarded by mbarriers.  No multicast.
//  * The other T threads are consumers.  Threads form tasks of TG threads;
//    thread uu of a task owns the same 16- or 32-byte slice ("unit") of
//    codes in every row, so its activations (32 or 64 fp16 values of x) sit
//    in registers for the whole kernel, loaded once.  S = T / TG tasks run
//    side by side; each thread handles JR rows of every stage.
//  * Inner loop: dot_word4 / dot_word2 (fp16-subnormal codes x fp16
//    activations with the mixed fma.rn.f32.f16, exact products, fp32 sums),
//    then scale * sum(q x) + bias * sum(x) per unit: the FMA-reordered
//    dequantisation of the hada.io page (topic 27758), factored per group.
//  * Row sums: a warp transpose-reduce of the JR row partials (log2 JR
//    split levels, then plain xor levels), one shared-memory slot per warp,
//    a consumer-only named barrier, and TG/32 adds by the finaliser thread
//    of each row, which applies the epilogue (residual, RMSNorm scale,
//    SwiGLU, MoE weights) and stores.
//  * Every mbarrier wait is bounded (about 1 s); a timeout sets a status bit
//    and the kernel stops instead of hanging.
#pragma once

#include <cuda_runtime.h>

#include "qgemv_args.h"
#include "qgemv_device.cuh"

namespace qgemv {

// Status word of this translation unit (bit kStatusWaitTimeout).
static __device__ unsigned g_status = 0;

template <int BITS, int UB>
struct Unit {
  static constexpr int kWords = UB / 4;               // uint32 words per row slice
  static constexpr int kCodesPerWord = 32 / BITS;
  static constexpr int kK = kWords * kCodesPerWord;   // k values per slice
  static constexpr int kPairs = kCodesPerWord / 2;    // packed x registers per word
  static constexpr int kXRegs = kWords * kPairs;
};

// Rows in the stage that starts at `row`: up to RS, never past the CTA's
// range, and (kMoeUp) never across an expert boundary.
template <int MODE>
__device__ __forceinline__ int stage_rows(long long row, long long r1, const StreamArgs& a) {
  long long n = r1 - row;
  if (n > a.RS) n = a.RS;
  if (MODE == kMoeUp) {
    const long long left = a.rows_per_expert - (row % a.rows_per_expert);
    if (n > left) n = left;
  }
  return static_cast<int>(n);
}

// Transpose-reduce JR row partials across a warp.  Returns, on lanes with
// lane % (32/JR) == 0, the warp's sum for row j = lane / (32/JR).
template <int JR>
__device__ __forceinline__ float warp_reduce_rows(float (&v)[JR], int lane) {
#pragma unroll
  for (int c = JR, o = 16; c > 1; c >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = upper ? v[i] : v[i + c / 2];
      const float keep = upper ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16 / JR; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// Sum of the thread's x slice, pairwise in fp32 (error ~ log2(64) ulp).
template <int N>
__device__ __forceinline__ float pairwise_sum(float (&v)[N]) {
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) v[i] += v[i + w];
  return v[0];
}

// One row slice: sum over the unit of w * x, in units of 2^-24.
template <int BITS, int UB>
__device__ __forceinline__ float unit_dot(const uint8_t* codes, const uint32_t* xp, float s,
                                          float b, float xs_scaled) {
  using U = Unit<BITS, UB>;
  uint32_t w[U::kWords];
#pragma unroll
  for (int i = 0; i < U::kWords / 4; ++i) {
    const uint4 v = reinterpret_cast<const uint4*>(codes)[i];
    w[4 * i + 0] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
  float t;
  if (BITS == 4) {
    float pa = 0.f, pb = 0.f, qa = 0.f, qb = 0.f;
#pragma unroll
    for (int i = 0; i < U::kWords; i += 2) {
      dot_word4(w[i], xp[4 * i], xp[4 * i + 1], xp[4 * i + 2], xp[4 * i + 3], pa, pb);
      if (i + 1 < U::kWords)
        dot_word4(w[i + 1], xp[4 * i + 4], xp[4 * i + 5], xp[4 * i + 6], xp[4 * i + 7], qa, qb);
    }
    t = fmaf(pb + qb, 0.0625f, pa + qa);
  } else {
    float ca = 0.f, cb = 0.f, cc = 0.f, cd = 0.f;
#pragma unroll
    for (int i = 0; i < U::kWords; ++i) dot_word2(w[i], xp + 8 * i, ca, cb, cc, cd);
    t = fmaf(cd, 0.015625f, fmaf(cc, 0.0625f, fmaf(cb, 0.25f, ca)));
  }
  return fmaf(s, t, b * xs_scaled);
}

template <int BITS, int UB, int MODE, int JR>
__global__ void __launch_bounds__(544, 1) stream_kernel(const StreamArgs a) {
  using U = Unit<BITS, UB>;
  constexpr int NMAT = (MODE == kSwiglu || MODE == kMoeUp) ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ float red[2][NMAT][kRedSlots];
  __shared__ float s_norm[17];
  __shared__ int s_eidx[kMaxTopK];
  __shared__ float s_ewt[kMaxTopK];
  __shared__ int s_abort;

  const int T = static_cast<int>(blockDim.x) - 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.NS;
  const long long r0 = static_cast<long long>(blockIdx.x) * a.rows / gridDim.x;
  const long long r1 = static_cast<long long>(blockIdx.x + 1) * a.rows / gridDim.x;
  const int rcb = a.K * BITS / 8;  // code bytes per row
  const int rgb = a.K / 32;        // scale (or bias) bytes per row
  const int MS = (MODE == kMoeDown) ? a.top_k : NMAT;  // matrices per stage
  const int codes_off = 0;
  const int scales_off = MS * a.RS * rcb;
  const int biases_off = scales_off + MS * a.RS * rgb;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), static_cast<uint32_t>(T / 32));
    }
    fence_mbar_init();
    if (MODE == kMoeUp || MODE == kMoeDown) {
      for (int k = 0; k < a.top_k; ++k) {
        const int e = a.idx[k];
        const bool ok = e >= 0 && e < a.n_experts;
        s_eidx[k] = ok ? e : -1;
        s_ewt[k] = ok ? a.wt[k] : 0.f;
        if (!ok && blockIdx.x == 0 && a.err_flag != nullptr) *a.err_flag = 1;
      }
    }
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int it = 0;
      for (long long row = r0; row < r1; ++it) {
        const int n = stage_rows<MODE>(row, r1, a);
        const int s = it % NS;
        if (!mbar_wait(smem_u32(&empty_bar[s]), ((it / NS) & 1) ^ 1, &g_status)) break;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t st = smem_u32(smem + static_cast<size_t>(s) * a.stage_bytes);
        // Sources of each matrix slot for rows [row, row + n).
        const uint8_t* cs[kMaxTopK];
        const __half* ss[kMaxTopK];
        const __half* bs[kMaxTopK];
        uint32_t bytes = 0;
        for (int m = 0; m < MS; ++m) {
          long long lrow = row;
          long long ec = 0, eg = 0;
          const int which = (MODE == kMoeDown) ? 0 : m;
          bool valid = true;
          if (MODE == kMoeUp) {
            const int e = s_eidx[row / a.rows_per_expert];
            valid = e >= 0;
            lrow = row % a.rows_per_expert;
            ec = static_cast<long long>(e) * a.ex_code_bytes;
            eg = static_cast<long long>(e) * a.ex_groups;
          } else if (MODE == kMoeDown) {
            const int e = s_eidx[m];
            valid = e >= 0;
            ec = static_cast<long long>(e) * a.ex_code_bytes;
            eg = static_cast<long long>(e) * a.ex_groups;
          }
          if (!valid) {
            cs[m] = nullptr;
            continue;
          }
          cs[m] = a.codes[which] + ec + lrow * rcb;
          ss[m] = a.scales[which] + eg + lrow * (rgb / 2);
          bs[m] = a.biases[which] + eg + lrow * (rgb / 2);
          bytes += static_cast<uint32_t>(n) * static_cast<uint32_t>(rcb + 2 * rgb);
        }
        mbar_arrive_expect_tx(fb, bytes);
        for (int m = 0; m < MS; ++m) {
          if (cs[m] == nullptr) continue;
          bulk_g2s(st + codes_off + m * a.RS * rcb, cs[m], n * rcb, fb, pol);
          bulk_g2s(st + scales_off + m * a.RS * rgb, ss[m], n * rgb, fb, pol);
          bulk_g2s(st + biases_off + m * a.RS * rgb, bs[m], n * rgb, fb, pol);
        }
        row += n;
      }
      // Drain: never leave while a copy into this CTA's shared memory is in flight.
      for (int j = (it > NS ? it - NS : 0); j < it; ++j)
        mbar_wait(smem_u32(&full_bar[j % NS]), (j / NS) & 1, &g_status);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int t = threadIdx.x - 32;
  const int TG = a.TG;
  const int S = a.S;
  const int slot = t / TG;
  const int uu = t - slot * TG;  // this thread's unit (row slice) index
  const int wit = uu >> 5;       // warp index within the task
  const int wpt = TG >> 5;       // warps per task
  int ek = 0, rbase = slot, rstep = S;
  if (MODE == kMoeDown) {
    ek = slot % a.top_k;
    rbase = slot / a.top_k;
    rstep = S / a.top_k;
  }
  const bool use_gamma = (MODE == kNorm) || (MODE == kSwiglu && a.gamma != nullptr);

  // RMS of x (kNorm, kSwiglu with gamma): every consumer sums a strided part.
  float rstd = 1.f;
  if (use_gamma) {
    float ss = 0.f;
    for (int k = t; k < a.K; k += T) {
      const float v = __half2float(a.x[k]);
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_norm[warp - 1] = ss;
    named_bar_sync(1, T);
    if (t == 0) {
      float tot = 0.f;
      for (int w = 0; w < T / 32; ++w) tot += s_norm[w];
      s_norm[16] = 1.0f / sqrtf(tot / static_cast<float>(a.K) + a.eps);
    }
    named_bar_sync(1, T);
    rstd = s_norm[16];
  }

  // This thread's activations, packed in the pairing the dot routines use,
  // and their sum (times 2^-24, the dot products' scale).
  uint32_t xp[U::kXRegs];
  float xs_scaled;
  {
    const int k0 = uu * U::kK;
    float xv[U::kK];
    if (MODE == kMoeDown) {
      const float4* src = reinterpret_cast<const float4*>(a.xf + static_cast<size_t>(ek) * a.K + k0);
#pragma unroll
      for (int i = 0; i < U::kK / 4; ++i) {
        const float4 v = src[i];
        xv[4 * i + 0] = v.x;
        xv[4 * i + 1] = v.y;
        xv[4 * i + 2] = v.z;
        xv[4 * i + 3] = v.w;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + k0);
#pragma unroll
      for (int i = 0; i < U::kK / 8; ++i) {
        const uint4 v = src[i];
        const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(h[j]);
          xv[8 * i + 2 * j] = f.x;
          xv[8 * i + 2 * j + 1] = f.y;
        }
      }
      if (use_gamma) {
        const uint4* gsrc = reinterpret_cast<const uint4*>(a.gamma + k0);
#pragma unroll
        for (int i = 0; i < U::kK / 8; ++i) {
          const uint4 v = gsrc[i];
          const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(h[j]);
            xv[8 * i + 2 * j] *= f.x;
            xv[8 * i + 2 * j + 1] *= f.y;
          }
        }
      }
    }
    // Round to fp16 once (the kernel multiplies fp16 activations).
    __half xh[U::kK];
#pragma unroll
    for (int k = 0; k < U::kK; ++k) {
      xh[k] = __float2half_rn(xv[k]);
      xv[k] = __half2float(xh[k]);
    }
    constexpr int cpw = U::kCodesPerWord;
#pragma unroll
    for (int i = 0; i < U::kWords; ++i)
#pragma unroll
      for (int j = 0; j < U::kPairs; ++j)
        xp[i * U::kPairs + j] = pack_half2(xh[i * cpw + j], xh[i * cpw + j + cpw / 2]);
    xs_scaled = pairwise_sum(xv) * kTwoM24;
  }
  const bool expert_ok = (MODE == kMoeDown) ? (s_eidx[ek] >= 0) : true;
  const int group_in_row = (uu * U::kK) / 64;

  // `alive` turns false for good once a wait has run out (here or in a
  // sibling warp, seen through s_abort after a barrier).  Every consumer then
  // keeps walking the same stages and barriers without waiting or working,
  // so no thread is ever left alone at a named barrier.
  bool alive = true;
  int it = 0, buf = 0;
  for (long long row = r0; row < r1; ++it) {
    const int n = stage_rows<MODE>(row, r1, a);
    const int s = it % NS;
    if (alive && __any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&s_abort) != 0))
      alive = false;
    if (alive) {
      const bool got = mbar_wait(smem_u32(&full_bar[s]), (it / NS) & 1, &g_status);
      alive = __all_sync(0xffffffffu, got);
      if (!alive && lane == 0) *reinterpret_cast<volatile int*>(&s_abort) = 1;
    }
    const uint8_t* st = smem + static_cast<size_t>(s) * a.stage_bytes;
    bool slot_ok = expert_ok;
    if (MODE == kMoeUp) slot_ok = s_eidx[row / a.rows_per_expert] >= 0;
    const bool work = alive && slot_ok;

    float acc[NMAT][JR];
#pragma unroll
    for (int j = 0; j < JR; ++j) {
      const int rl = rbase + j * rstep;
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        acc[m][j] = 0.f;
        if (rl < n && work) {
          const int ms = (MODE == kMoeDown) ? ek : m;
          const uint8_t* cp = st + codes_off + (ms * a.RS + rl) * rcb + uu * UB;
          const __half* sp =
              reinterpret_cast<const __half*>(st + scales_off + (ms * a.RS + rl) * rgb);
          const __half* bp =
              reinterpret_cast<const __half*>(st + biases_off + (ms * a.RS + rl) * rgb);
          acc[m][j] = unit_dot<BITS, UB>(cp, xp, __half2float(sp[group_in_row]),
                                         __half2float(bp[group_in_row]), xs_scaled);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && alive) mbar_arrive(smem_u32(&empty_bar[s]));

    constexpr int kLanesPerRow = 32 / JR;
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      const float v = warp_reduce_rows<JR>(acc[m], lane);
      if ((lane & (kLanesPerRow - 1)) == 0) {
        const int j = lane / kLanesPerRow;
        const int rl = rbase + j * rstep;
        const int task = (MODE == kMoeDown) ? rl * a.top_k + ek : rl;
        red[buf][m][task * wpt + wit] = v;
      }
    }
    named_bar_sync(1, T);

    if (t < n && alive) {
      const long long gr = row + t;
      float v[NMAT];
#pragma unroll
      for (int m = 0; m < NMAT; ++m) v[m] = 0.f;
      if (MODE == kMoeDown) {
        for (int k = 0; k < a.top_k; ++k) {
          float e = 0.f;
          for (int w = 0; w < wpt; ++w) e += red[buf][0][(t * a.top_k + k) * wpt + w];
          v[0] = fmaf(s_ewt[k], e, v[0]);
        }
      } else {
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          for (int w = 0; w < wpt; ++w) v[m] += red[buf][m][t * wpt + w];
      }
#pragma unroll
      for (int m = 0; m < NMAT; ++m) v[m] *= kTwo24;

      if (MODE == kPlain || MODE == kMoeDown) {
        float o = v[0];
        if (a.residual != nullptr) o += __half2float(a.residual[gr]);
        a.y[gr] = __float2half_rn(o);
      } else if (MODE == kNorm) {
        a.y[gr] = __float2half_rn(v[0] * rstd);
      } else if (MODE == kSwiglu) {
        const float g = v[0] * rstd, u = v[NMAT - 1] * rstd;
        a.y[gr] = __float2half_rn(silu_f(g) * u);
      } else if (MODE == kMoeUp) {
        a.yf[gr] = slot_ok ? silu_f(v[0]) * v[NMAT - 1] : 0.f;
      }
    }
    buf ^= 1;
    row += n;
  }
}

// Set the dynamic shared-memory limit once per (kernel, device).
template <typename F>
inline cudaError_t ensure_smem_attr(F* kernel, int bytes, unsigned* done_mask, int device) {
  if (device >= 0 && device < 32 && (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) >> device) & 1u)
    return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && device >= 0 && device < 32)
    __atomic_fetch_or(done_mask, 1u << device, __ATOMIC_ACQ_REL);
  return e;
}

template <int BITS, int UB, int MODE, int JR>
inline cudaError_t launch_stream_t(const StreamPlan& p, StreamArgs a, cudaStream_t stream,
                                   int device) {
  static unsigned done_mask = 0;
  auto* k = stream_kernel<BITS, UB, MODE, JR>;
  const int dyn = p.ns * p.stage_bytes;
  cudaError_t e = ensure_smem_attr(k, 220 * 1024, &done_mask, device);
  if (e != cudaSuccess) return e;
  a.TG = p.tg;
  a.S = p.s;
  a.RS = p.rs;
  a.NS = p.ns;
  a.stage_bytes = p.stage_bytes;
  k<<<p.grid, p.t + 32, dyn, stream>>>(a);
  return cudaGetLastError();
}

// Dispatch on the plan's unit size and rows per thread.
template <int BITS, int MODE>
inline cudaError_t launch_stream(const StreamPlan& p, const StreamArgs& a, cudaStream_t stream,
                                 int device) {
  if constexpr (BITS == 4) {
    if (p.ub == 32)
      return p.jr == 4 ? launch_stream_t<BITS, 32, MODE, 4>(p, a, stream, device)
                       : launch_stream_t<BITS, 32, MODE, 2>(p, a, stream, device);
  }
  return p.jr == 4 ? launch_stream_t<BITS, 16, MODE, 4>(p, a, stream, device)
                   : launch_stream_t<BITS, 16, MODE, 2>(p, a, stream, device);
}

// Read and clear this translation unit's status word (synchronous).
inline cudaError_t read_clear_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  *out |= v;
  return e;
}

}  // namespace qgemv
