// generic.cu -- warp-per-row kernels for every case the streaming kernel
// does not take: K not a multiple of 1024 (2048 for 2-bit), pointers that are
// not 16-byte aligned, and small batches M = 2..8.  Same arithmetic and the
// same fp16 roundings of the activations as the streaming kernel; slower
// (activations are re-read from L1/L2 for every row).
#include "qgemv_args.h"
#include "epilogue_ops.h"
#include "qgemv_device.cuh"

namespace qgemv {

static __device__ unsigned g_status_generic = 0;

constexpr int kGenericWarps = 8;
static_assert(kGenericWarps == 8, "generic_blocks() in qgemv_args.h counts 8 rows per CTA");

// The fp16-rounded activation value the kernels multiply by.
template <int MODE>
__device__ __forceinline__ float activation(const StreamArgs& a, int m, int k, bool use_gamma,
                                            int ek) {
  if (MODE == kMoeDown) return __half2float(__float2half_rn(a.xf[static_cast<size_t>(ek) * a.K + k]));
  float v = __half2float(a.x[static_cast<size_t>(m) * a.K + k]);
  if (use_gamma) v = __half2float(__float2half_rn(v * __half2float(a.gamma[k])));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int BITS, int MODE, int M>
__global__ void __launch_bounds__(32 * kGenericWarps) generic_kernel(const StreamArgs a) {
  constexpr int NMAT = (MODE == kSwiglu || MODE == kMoeUp) ? 2 : 1;
  constexpr int CPW = 32 / BITS;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((MODE == kMoeUp || MODE == kMoeDown) && blockIdx.x == 0 && threadIdx.x == 0 &&
      a.err_flag != nullptr) {
    for (int k = 0; k < a.top_k; ++k)
      if (a.idx[k] < 0 || a.idx[k] >= a.n_experts) *a.err_flag = 1;
  }
  // Opt-in trace of the (index, weight) pairs this CTA reads (every thread
  // reads the same words; thread 0 records them).
  if ((MODE == kMoeUp || MODE == kMoeDown) && a.trace != nullptr && threadIdx.x == 0 &&
      static_cast<int>(blockIdx.x) < a.trace_ctas) {
    for (int k = 0; k < a.top_k; ++k) {
      const int e = a.idx[k];
      const float w = a.wt[k];
      const bool ok = e >= 0 && e < a.n_experts;
      reinterpret_cast<uint4*>(a.trace)[blockIdx.x * a.top_k + k] =
          make_uint4(static_cast<unsigned>(e), __float_as_uint(w),
                     static_cast<unsigned>(ok ? e : -1), __float_as_uint(ok ? w : 0.f));
    }
  }
  const long long row = static_cast<long long>(blockIdx.x) * kGenericWarps + warp;
  if (row >= a.rows) return;
  const int K = a.K;
  const int words = K / CPW;
  const int G = K / 64;
  const bool use_gamma = (MODE == kNorm) || (MODE == kSwiglu && a.gamma != nullptr);

  float rstd = 1.f;
  if (use_gamma) {
    float ss = 0.f;
    for (int k = lane; k < K; k += 32) {
      const float v = __half2float(a.x[k]);
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    rstd = 1.0f / sqrtf(ss / static_cast<float>(K) + a.eps);
  }

  // Row pointers of each matrix this row reads.
  const uint32_t* wrow[NMAT];
  const __half* srow[NMAT];
  const __half* brow[NMAT];
  bool row_ok = true;
  if (MODE != kMoeDown) {
    long long lrow = row, ec = 0, eg = 0;
    if (MODE == kMoeUp) {
      const int e = a.idx[row / a.rows_per_expert];
      row_ok = e >= 0 && e < a.n_experts;
      lrow = row % a.rows_per_expert;
      ec = row_ok ? static_cast<long long>(e) * a.ex_code_bytes : 0;
      eg = row_ok ? static_cast<long long>(e) * a.ex_groups : 0;
    }
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      wrow[m] = reinterpret_cast<const uint32_t*>(a.codes[m] + ec) + lrow * words;
      srow[m] = a.scales[m] + eg + lrow * G;
      brow[m] = a.biases[m] + eg + lrow * G;
    }
  }

  float acc[NMAT][M];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int b = 0; b < M; ++b) acc[m][b] = 0.f;

  if (row_ok) {
    for (int w = lane; w < words; w += 32) {
      const int k0 = w * CPW;
      const int g = k0 / 64;
      if (MODE == kMoeDown) {
        for (int k = 0; k < a.top_k; ++k) {
          const int e = a.idx[k];
          if (e < 0 || e >= a.n_experts) continue;
          const long long ec = static_cast<long long>(e) * a.ex_code_bytes;
          const long long eg = static_cast<long long>(e) * a.ex_groups;
          const uint32_t word = reinterpret_cast<const uint32_t*>(a.codes[0] + ec)[row * words + w];
          const float s = __half2float(a.scales[0][eg + row * G + g]);
          const float b = __half2float(a.biases[0][eg + row * G + g]);
          float S = 0.f, X = 0.f;
#pragma unroll
          for (int j = 0; j < CPW; ++j) {
            const float xv = activation<MODE>(a, 0, k0 + j, false, k);
            S = fmaf(static_cast<float>(unpack_code<BITS>(word, j)), xv, S);
            X += xv;
          }
          acc[0][0] = fmaf(a.wt[k], fmaf(s, S, b * X), acc[0][0]);
        }
      } else {
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint32_t word = wrow[m][w];
          const float s = __half2float(srow[m][g]);
          const float b = __half2float(brow[m][g]);
#pragma unroll
          for (int bi = 0; bi < M; ++bi) {
            float S = 0.f, X = 0.f;
#pragma unroll
            for (int j = 0; j < CPW; ++j) {
              const float xv = activation<MODE>(a, bi, k0 + j, use_gamma, 0);
              S = fmaf(static_cast<float>(unpack_code<BITS>(word, j)), xv, S);
              X += xv;
            }
            acc[m][bi] = fmaf(s, S, fmaf(b, X, acc[m][bi]));
          }
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int b = 0; b < M; ++b) acc[m][b] = warp_sum(acc[m][b]);

  if (lane != 0) return;
  if (MODE == kPlain) {
#pragma unroll
    for (int b = 0; b < M; ++b) {
      float o = acc[0][b];
      const long long idx = static_cast<long long>(b) * a.rows + row;
      if (a.residual != nullptr) o += __half2float(a.residual[idx]);
      a.y[idx] = __float2half_rn(o);
    }
  } else if (MODE == kMoeDown) {
    float o = acc[0][0];
    if (a.residual != nullptr) o += __half2float(a.residual[row]);
    a.y[row] = __float2half_rn(o);
  } else if (MODE == kNorm) {
    a.y[row] = __float2half_rn(acc[0][0] * rstd);
  } else if (MODE == kSwiglu) {
    a.y[row] = __float2half_rn(silu_f(acc[0][0] * rstd) * (acc[NMAT - 1][0] * rstd));
  } else if (MODE == kMoeUp) {
    a.yf[row] = row_ok ? silu_f(acc[0][0]) * acc[NMAT - 1][0] : 0.f;
  }
}

template <int BITS, int MODE, int M>
static cudaError_t launch_generic_t(const StreamArgs& a, cudaStream_t st) {
  const long long blocks = (a.rows + kGenericWarps - 1) / kGenericWarps;
  generic_kernel<BITS, MODE, M><<<static_cast<unsigned>(blocks), 32 * kGenericWarps, 0, st>>>(a);
  return cudaGetLastError();
}

template <int BITS>
static cudaError_t launch_plain_m(const StreamArgs& a, cudaStream_t st) {
  switch (a.M) {
    case 1: return launch_generic_t<BITS, kPlain, 1>(a, st);
    case 2: return launch_generic_t<BITS, kPlain, 2>(a, st);
    case 3: return launch_generic_t<BITS, kPlain, 3>(a, st);
    case 4: return launch_generic_t<BITS, kPlain, 4>(a, st);
    case 5: return launch_generic_t<BITS, kPlain, 5>(a, st);
    case 6: return launch_generic_t<BITS, kPlain, 6>(a, st);
    case 7: return launch_generic_t<BITS, kPlain, 7>(a, st);
    case 8: return launch_generic_t<BITS, kPlain, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t generic_launch(int mode, int bits, const StreamArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  switch (mode) {
    case kPlain:
      return bits == 4 ? launch_plain_m<4>(a, st)
                       : (bits == 8 ? launch_plain_m<8>(a, st) : launch_plain_m<2>(a, st));
    case kNorm: return launch_generic_t<4, kNorm, 1>(a, st);
    case kSwiglu: return launch_generic_t<4, kSwiglu, 1>(a, st);
    case kMoeUp: return launch_generic_t<4, kMoeUp, 1>(a, st);
    case kMoeDown: return launch_generic_t<4, kMoeDown, 1>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------ seq-len-1 attention copy

__global__ void attention_seq1_kernel(const __half* __restrict__ qkv, __half* __restrict__ out,
                                      int n_q, int n_kv, int head_dim) {
  pdl_launch_dependents();
  pdl_wait();  // qkv comes from the previous kernel
  const long long total = static_cast<long long>(n_q) * head_dim;
  const int group = n_q / n_kv;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(i / head_dim);
    const int d = static_cast<int>(i % head_dim);
    out[i] = qkv[static_cast<long long>(n_q + n_kv + h / group) * head_dim + d];
  }
}

cudaError_t attention_seq1_launch(const __half* qkv, __half* out, int n_q, int n_kv,
                                  int head_dim, cudaStream_t st) {
  const long long total = static_cast<long long>(n_q) * head_dim;
  long long blocks = (total + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attention_seq1_kernel, qkv, out, n_q, n_kv, head_dim);
}

// Argmax of an fp16 vector by one CTA of 1024 threads (lowest index of the
// largest value, the same key as the streaming kernel's kArgmax epilogue).
__global__ void __launch_bounds__(1024) argmax_kernel(const __half* __restrict__ y, int n,
                                                      int* __restrict__ token) {
  __shared__ unsigned long long s_best[32];
  unsigned long long best = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    best = max_key(best, argmax_key(__half2float(y[i]), i));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) best = max_key(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) s_best[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x < 32) {
    best = threadIdx.x < blockDim.x / 32 ? s_best[threadIdx.x] : 0ull;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) best = max_key(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (threadIdx.x == 0) *token = static_cast<int>(~static_cast<unsigned>(best & 0xffffffffull));
  }
}

cudaError_t argmax_launch(const __half* y, int n, int* token, cudaStream_t st) {
  argmax_kernel<<<1, 1024, 0, st>>>(y, n, token);
  return cudaGetLastError();
}

__global__ void argmax_finalize_kernel(unsigned long long* key, int* token) {
  pdl_launch_dependents();
  pdl_wait();  // every CTA of the kArgmax grid has folded its key in
  const unsigned long long k = *reinterpret_cast<volatile unsigned long long*>(key);
  *token = static_cast<int>(~static_cast<unsigned>(k & 0xffffffffull));
  *key = 0ull;
}

cudaError_t argmax_finalize_launch(unsigned long long* key, int* token, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, argmax_finalize_kernel, key, token);
}

// MoE routing from fp16 router logits, one CTA of 1024 threads: the shared
// expert (shared >= 0), then the routed experts with the largest logits one
// at a time (the (value, index) key of argmax_key: the lower index wins a
// tie), then the softmax of the chosen logits in fp32.
__global__ void __launch_bounds__(1024) moe_route_kernel(const __half* __restrict__ logits, int E,
                                                         int top_k, int shared,
                                                         int* __restrict__ idx,
                                                         float* __restrict__ wt) {
  __shared__ unsigned long long s_red[32];
  __shared__ int s_chosen[kMaxTopK];
  pdl_launch_dependents();
  pdl_wait();  // the logits come from the previous kernel
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int n = 0;
  if (shared >= 0) {
    if (threadIdx.x == 0) s_chosen[0] = shared;
    n = 1;
  }
  __syncthreads();
  for (; n < top_k; ++n) {
    unsigned long long best = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      bool taken = false;
      for (int j = 0; j < n; ++j) taken = taken || (s_chosen[j] == e);
      if (!taken) best = max_key(best, argmax_key(__half2float(logits[e]), e));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) best = max_key(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (warp == 0) {
      best = lane < static_cast<int>(blockDim.x >> 5) ? s_red[lane] : 0ull;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        best = max_key(best, __shfl_xor_sync(0xffffffffu, best, o));
      if (lane == 0) s_chosen[n] = static_cast<int>(~static_cast<unsigned>(best & 0xffffffffull));
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    float v[kMaxTopK];
    float m = -INFINITY;
    for (int j = 0; j < top_k; ++j) {
      v[j] = __half2float(logits[s_chosen[j]]);
      m = fmaxf(m, v[j]);
    }
    float sum = 0.f;
    for (int j = 0; j < top_k; ++j) {
      v[j] = expf(v[j] - m);
      sum += v[j];
    }
    for (int j = 0; j < top_k; ++j) {
      idx[j] = s_chosen[j];
      wt[j] = v[j] / sum;
    }
  }
}

cudaError_t moe_route_launch(const __half* logits, int E, int top_k, int shared, int* idx,
                             float* wt, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_route_kernel, logits, E, top_k, shared, idx, wt);
}

// Residual add and RMSNorm as a standalone epilogue, one CTA of 1024
// threads: h = fp16(x + r) (exact sum, one rounding), xn = fp16(h * gamma *
// rstd(h)) with rstd = 1 / sqrt(mean(h^2) + eps) over the fp16 h.  r may be
// null (then h = x and it is not stored).
__global__ void __launch_bounds__(1024) residual_rmsnorm_kernel(
    const __half* __restrict__ x, const __half* __restrict__ r, const __half* __restrict__ gamma,
    float eps, int K, __half* __restrict__ h, __half* __restrict__ xn) {
  __shared__ float s_red[32];
  __shared__ float s_rstd;
  pdl_launch_dependents();
  pdl_wait();  // x and r may come from the previous kernel
  float sq = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v = __half2float(x[k]);
    if (r != nullptr) {
      const __half hv = __float2half_rn(v + __half2float(r[k]));
      h[k] = hv;
      v = __half2float(hv);
    }
    sq = fmaf(v, v, sq);
  }
  sq = warp_sum(sq);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = sq;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? s_red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) s_rstd = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
  }
  __syncthreads();
  const float rstd = s_rstd;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float v = __half2float(r != nullptr ? h[k] : x[k]);
    xn[k] = __float2half_rn(v * __half2float(gamma[k]) * rstd);
  }
}

cudaError_t residual_rmsnorm_launch(const __half* x, const __half* r, const __half* gamma,
                                    float eps, int K, __half* h, __half* xn, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, residual_rmsnorm_kernel, x, r, gamma, eps, K, h, xn);
}

// Self-test of the bounded waits: one thread waits on an mbarrier that no
// thread ever arrives on, with the given limit; the wait must give up, set
// the timeout bit and return, leaving the context usable.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    (void)mbar_wait_for(smem_u32(&bar), 0, &g_status_generic, limit_ns);
  }
}

cudaError_t selftest_wait_launch(uint64_t limit_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t status_generic(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_generic, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_status_generic, &zero, sizeof(zero));
  *out |= v;
  return e;
}

}  // namespace qgemv
