// sample.cu -- top-k sampling of the next token from fp16 logits on the GPU,
// so that only the token goes back to the host.
//
// One cluster of kCluster CTAs; CTA r holds slice r of the logits in shared
// memory as order-preserving 16-bit keys, counted into a fine (key >> 4)
// histogram as they arrive.  The k-th largest key T is found by radix
// selection on the cluster's histograms, read through distributed shared
// memory: the coarse bin (key >> 8), the fine bin inside it, then the low
// nibble of the keys in that fine bin.  Every key above T, and the
// lowest-index keys equal to T, claim slots in CTA 0 (one atomic per warp);
// threads whose largest key lies below the fine bin skip those passes.  CTA 0
// sorts the k candidates (descending value, ascending index), weights them
// by exp((l_j - l_0) / temperature) in fp32 and picks the token by inverse
// CDF against the caller's u in one warp.  The selection is exact (integer
// work on the fp16 bits); only the weights are floating point.  Three
// cluster barriers, no global scratch, no spin-waits: the cluster barriers
// are hardware barriers over co-scheduled CTAs.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "epilogue_ops.h"
#include "qgemv_device.cuh"

namespace cg = cooperative_groups;

namespace qgemv {
namespace {

constexpr int kCluster = 8;                  // CTAs in the cluster, one slice each
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kFine = 4096;                  // key >> 4
constexpr int kCoarse = 256;                 // key >> 8
constexpr int kRankSortMax = 256;            // k sorted by counting ranks up to here, bitonic above
constexpr int kFixedSmem = kFine * 4 + kCoarse * 4 + kMaxSampleK * 8 + kRankSortMax * 8;

// Larger key <=> larger fp16 value; -0 is folded onto +0 so that equal values
// have equal keys.
__device__ __forceinline__ unsigned key16(unsigned b) {
  if (b == 0x8000u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// key16 of both halves of a word: positive values get the sign bit set,
// negative ones are complemented; -0 (which becomes 0x7FFF) is then moved up
// to +0 (0x8000).
__device__ __forceinline__ unsigned key16x2(unsigned w) {
  const unsigned neg = ((w >> 15) & 0x00010001u) * 0xFFFFu;
  unsigned key = w ^ (neg | 0x80008000u);
  key += __vcmpeq2(key, 0x7FFF7FFFu) & 0x00010001u;
  return key;
}

__device__ __forceinline__ float key_value(unsigned k) {
  const unsigned short b =
      static_cast<unsigned short>((k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu));
  return __half2float(__ushort_as_half(b));
}

// Sort key of a candidate: value key above, complemented index below, so that
// a larger sort key is a larger value or, for equal values, a lower index.
__device__ __forceinline__ unsigned long long cand_key(unsigned k, unsigned idx) {
  return (static_cast<unsigned long long>(k) << 32) | static_cast<unsigned long long>(~idx);
}

// Inclusive block scan of a pair of counts (1024 threads, every thread of the
// CTA must call it); also returns the block totals.
__device__ __forceinline__ uint2 block_scan2(uint2 v, uint2* s_w, uint2* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned a = __shfl_up_sync(0xffffffffu, v.x, o);
    const unsigned b = __shfl_up_sync(0xffffffffu, v.y, o);
    if (lane >= o) { v.x += a; v.y += b; }
  }
  if (lane == 31) s_w[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint2 w = s_w[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned a = __shfl_up_sync(0xffffffffu, w.x, o);
      const unsigned b = __shfl_up_sync(0xffffffffu, w.y, o);
      if (lane >= o) { w.x += a; w.y += b; }
    }
    s_w[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  if (warp > 0) { v.x += s_w[warp - 1].x; v.y += s_w[warp - 1].y; }
  *total = s_w[kWarps - 1];
  return v;
}

__device__ __forceinline__ unsigned cand_index(unsigned long long c) {
  return ~static_cast<unsigned>(c & 0xffffffffull);
}

__device__ __forceinline__ unsigned key_at(const uint4& o, int e) {
  const unsigned w = e < 2 ? o.x : e < 4 ? o.y : e < 6 ? o.z : o.w;
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// n slots of CTA 0's candidate buffer for this thread: one atomic per warp.
// Every lane of the warp calls it.
__device__ __forceinline__ unsigned claim(unsigned n, unsigned* cnt0) {
  const int lane = threadIdx.x & 31;
  unsigned inc = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  unsigned base = 0;
  if (lane == 31 && inc != 0u) base = atomicAdd(cnt0, inc);
  base = __shfl_sync(0xffffffffu, base, 31);
  return base + inc - n;
}

__global__ void __launch_bounds__(kThreads) sample_topk_kernel(
    const __half* __restrict__ logits, int n, int slice, int top_k, float temperature,
    const float* __restrict__ u_ptr, int* __restrict__ token, int* __restrict__ out_idx,
    float* __restrict__ out_prob) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned* fine = reinterpret_cast<unsigned*>(smem);                              // [kFine]
  unsigned* coarse = fine + kFine;                                                 // [kCoarse]
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(coarse + kCoarse);  // [kMaxSampleK]
  unsigned long long* ranked = cand + kMaxSampleK;                                 // [kRankSortMax]
  unsigned short* keys = reinterpret_cast<unsigned short*>(ranked + kRankSortMax);  // [slice]

  __shared__ unsigned s_h2[16];        // this CTA's keys in the fine bin, by low nibble
  __shared__ unsigned s_all[kCluster][16];
  __shared__ unsigned s_f16[16];
  __shared__ unsigned s_w[kWarps];
  __shared__ uint2 s_w2[kWarps];
  __shared__ unsigned s_cnt;           // CTA 0: candidate slots claimed
  __shared__ unsigned s_B, s_above_B, s_bin, s_gt_bin, s_lo4, s_gt, s_base;

  pdl_launch_dependents();
  cg::cluster_group cl = cg::this_cluster();
  const unsigned rank = cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned k = static_cast<unsigned>(top_k);

  for (int i = tid; i < kFine; i += kThreads) fine[i] = 0u;
  cand[tid] = 0ull;
  if (tid < 16) s_h2[tid] = 0u;
  if (tid == 0) {
    s_cnt = 0u;
    s_B = s_above_B = s_bin = s_gt_bin = s_lo4 = s_gt = s_base = 0u;
  }
  const long long lo = static_cast<long long>(rank) * slice;
  const int n_loc = static_cast<int>(lo >= n ? 0 : (n - lo < slice ? n - lo : slice));
  const __half* src = logits + lo;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int nv = vec ? (n_loc >> 3) : 0;   // 8-key groups read as uint4
  const int done = nv << 3;                // keys [done, n_loc) read one by one
  uint4* k4 = reinterpret_cast<uint4*>(keys);
  // This thread's keys: groups v = tid (mod kThreads), then keys done + tid (mod kThreads).
  auto own = [&](auto&& f) {
    for (int v = tid; v < nv; v += kThreads) {
      const uint4 o = k4[v];
#pragma unroll
      for (int e = 0; e < 8; ++e) f(key_at(o, e), (v << 3) + e);
    }
    for (int i = done + tid; i < n_loc; i += kThreads) f(static_cast<unsigned>(keys[i]), i);
  };

  pdl_wait();  // the logits (and u) come from the previous kernel
  __syncthreads();  // the histogram is zero before anyone counts into it

  // Slice -> keys, each counted into the fine histogram; and the largest key
  // of each thread.
  unsigned tmax2 = 0u;  // two halves
  {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int base = tid; base < nv; base += 4 * kThreads) {
      uint4 d[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = base + j * kThreads;
        d[j] = v < nv ? s4[v] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = base + j * kThreads;
        if (v < nv) {
          uint4 o;
          o.x = key16x2(d[j].x);
          o.y = key16x2(d[j].y);
          o.z = key16x2(d[j].z);
          o.w = key16x2(d[j].w);
          k4[v] = o;
          tmax2 = __vmaxu2(tmax2, __vmaxu2(__vmaxu2(o.x, o.y), __vmaxu2(o.z, o.w)));
#pragma unroll
          for (int e = 0; e < 8; ++e) atomicAdd(&fine[key_at(o, e) >> 4], 1u);
        }
      }
    }
    for (int i = done + tid; i < n_loc; i += kThreads) {
      const unsigned kk = key16(__half_as_ushort(src[i]));
      keys[i] = static_cast<unsigned short>(kk);
      tmax2 = __vmaxu2(tmax2, kk);
      atomicAdd(&fine[kk >> 4], 1u);
    }
  }
  const unsigned tmax = max(tmax2 & 0xFFFFu, tmax2 >> 16);  // 0 when the thread has no keys
  __syncthreads();
  if (tid < kCoarse) {
    const uint4* f4 = reinterpret_cast<const uint4*>(fine + tid * 16);
    unsigned c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 a = f4[j];
      c += a.x + a.y + a.z + a.w;
    }
    coarse[tid] = c;
  }
  cl.sync();  // (1) every CTA's histograms are complete

  // The coarse bin B holding the k-th largest key of the cluster.
  {
    unsigned g = 0;
    if (tid < kCoarse) {
#pragma unroll
      for (int c = 0; c < kCluster; ++c) g += cl.map_shared_rank(coarse, c)[tid];
    }
    unsigned suf = g;  // suffix sum within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += t;
    }
    if (lane == 0 && warp < kCoarse / 32) s_w[warp] = suf;
    __syncthreads();
    if (tid < kCoarse) {
      for (int w = warp + 1; w < kCoarse / 32; ++w) suf += s_w[w];
      if (suf >= k && suf - g < k) {
        s_B = static_cast<unsigned>(tid);
        s_above_B = suf - g;
      }
    }
    __syncthreads();
  }
  // The fine bin inside B.
  {
    const unsigned B = s_B;
    if (tid < 16 * kCluster) {
      const int j = tid >> 3, c = tid & 7;
      unsigned v = cl.map_shared_rank(fine, c)[B * 16 + j];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (c == 0) s_f16[j] = v;
    }
    __syncthreads();
    if (warp == 0) {
      const unsigned v = lane < 16 ? s_f16[lane] : 0u;
      unsigned suf = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      const unsigned above = s_above_B;
      if (lane < 16 && above + suf >= k && above + suf - v < k) {
        s_bin = B * 16 + static_cast<unsigned>(lane);
        s_gt_bin = above + suf - v;
      }
    }
    __syncthreads();
  }
  const unsigned bin = s_bin;
  unsigned* cnt0 = cl.map_shared_rank(&s_cnt, 0);
  unsigned long long* cand0 = cl.map_shared_rank(cand, 0);
  const bool active = (tmax >> 4) >= bin;  // holds a key in the fine bin or above

  // Keys above the fine bin are in; keys inside it are counted by low nibble.
  {
    unsigned n_in = 0;
    if (active)
      own([&](unsigned kk, int) {
        if ((kk >> 4) > bin) ++n_in;
        else if ((kk >> 4) == bin) atomicAdd(&s_h2[kk & 15u], 1u);
      });
    unsigned slot = claim(n_in, cnt0);
    if (n_in != 0u)
      own([&](unsigned kk, int i) {
        if ((kk >> 4) > bin) {
          if (slot < k) cand0[slot] = cand_key(kk, static_cast<unsigned>(lo + i));
          ++slot;
        }
      });
  }
  cl.sync();  // (2)

  // T = the k-th largest key; the quota of keys equal to T for this CTA.
  if (tid < 16 * kCluster) {
    const int c = tid >> 4, j = tid & 15;
    s_all[c][j] = cl.map_shared_rank(s_h2, c)[j];
  }
  __syncthreads();
  if (warp == 0) {
    unsigned v = 0;
    if (lane < 16)
      for (int c = 0; c < kCluster; ++c) v += s_all[c][lane];
    unsigned suf = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += t;
    }
    const unsigned gtb = s_gt_bin;
    if (lane < 16 && gtb + suf >= k && gtb + suf - v < k) {
      s_lo4 = static_cast<unsigned>(lane);
      s_gt = gtb + suf - v;
    }
  }
  __syncthreads();
  const unsigned lo4 = s_lo4;
  const unsigned T = (bin << 4) | lo4;
  const unsigned need = k - s_gt;  // keys equal to T taken, lowest indices first
  unsigned eq_before = 0, above_mine = 0;
  for (unsigned c = 0; c < rank; ++c) eq_before += s_all[c][lo4];
  for (unsigned j = lo4 + 1; j < 16; ++j) above_mine += s_all[rank][j];
  const unsigned eq_mine = s_all[rank][lo4];
  const unsigned q = need > eq_before ? need - eq_before : 0u;
  const unsigned quota = q < eq_mine ? q : eq_mine;
  const bool take_all_eq = quota == eq_mine;  // then their order does not matter

  if (above_mine != 0u || quota != 0u) {  // uniform over the CTA
    auto taken = [&](unsigned kk) { return (kk >> 4) == bin && (kk > T || (kk == T && take_all_eq)); };
    unsigned n_in = 0;
    if (active)
      own([&](unsigned kk, int) { n_in += taken(kk); });
    unsigned slot = claim(n_in, cnt0);
    if (n_in != 0u)
      own([&](unsigned kk, int i) {
        if (taken(kk)) {
          if (slot < k) cand0[slot] = cand_key(kk, static_cast<unsigned>(lo + i));
          ++slot;
        }
      });
    if (!take_all_eq && quota != 0u) {
      // Only some of this CTA's keys equal to T are taken: the lowest
      // indices.  Each thread scans a contiguous run of indices, so an
      // exclusive scan of the per-thread counts ranks them by index.
      const int run = (n_loc + kThreads - 1) / kThreads;
      const int b = tid * run;
      const int e = b + run < n_loc ? b + run : n_loc;
      unsigned c = 0;
      for (int i = b; i < e; ++i) c += keys[i] == T;
      uint2 tot;
      const uint2 inc = block_scan2(make_uint2(c, 0u), s_w2, &tot);
      if (tid == 0) s_base = atomicAdd(cnt0, quota);
      __syncthreads();
      const unsigned base = s_base;
      unsigned r = inc.x - c;
      for (int i = b; i < e && r < quota; ++i) {
        if (keys[i] == T) {
          if (base + r < k) cand0[base + r] = cand_key(T, static_cast<unsigned>(lo + i));
          ++r;
        }
      }
    }
  }
  cl.sync();  // (3) after this no CTA touches another's shared memory
  if (rank != 0) return;

  // CTA 0: the k candidates are in cand[0, k), in claim order.  Sort them by
  // descending sort key: by counting ranks for small k, else bitonic.
  const unsigned long long* sorted = cand;
  if (top_k <= kRankSortMax) {
    if (tid < top_k) {
      const unsigned long long c = cand[tid];
      unsigned r = 0;
      int i = 0;
      for (; i + 4 <= top_k; i += 4)
        r += (cand[i] > c) + (cand[i + 1] > c) + (cand[i + 2] > c) + (cand[i + 3] > c);
      for (; i < top_k; ++i) r += cand[i] > c;
      ranked[r < k ? r : k - 1] = c;
    }
    __syncthreads();
    sorted = ranked;
  } else {
    // Bitonic over P = 512 or 1024 slots (zero keys pad, below every real
    // one), one per thread: partners closer than a warp by shuffle, farther
    // ones through shared memory.
    int P = 2;
    while (P < top_k) P <<= 1;
    unsigned long long x = cand[tid];
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        unsigned long long y;
        if (stride >= 32) {
          __syncthreads();
          cand[tid] = x;
          __syncthreads();
          y = cand[tid ^ stride];
        } else {
          y = __shfl_xor_sync(0xffffffffu, x, stride);
        }
        const bool lower = (tid & stride) == 0;
        const bool desc = (tid & size) == 0;
        x = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
      }
    }
    __syncthreads();
    cand[tid] = x;
    __syncthreads();
  }

  // Weights, their running sum and the inverse-CDF pick, in one warp: lane
  // l holds candidates [l E, l E + E).
  if (tid >= 32) return;
  float* wbuf = reinterpret_cast<float*>(fine);  // free in CTA 0 from here on
  const float l0 = key_value(static_cast<unsigned>(sorted[0] >> 32));
  const int E = (top_k + 31) >> 5;
  const int b = lane * E;
  const int e = b + E < top_k ? b + E : top_k;
  float part = 0.f;
  for (int i = b; i < e; ++i) {
    const float p = expf((key_value(static_cast<unsigned>(sorted[i] >> 32)) - l0) / temperature);
    wbuf[i] = p;
    part += p;
  }
  float inc = part;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  const float total = __shfl_sync(0xffffffffu, inc, 31);
  const float target = *u_ptr * total;
  float run = inc - part;
  int first = -1;
  for (int i = b; i < e; ++i) {
    run += wbuf[i];
    if (run > target) { first = i; break; }
  }
  const unsigned m = __ballot_sync(0xffffffffu, first >= 0);
  const int pick = m ? __shfl_sync(0xffffffffu, first, __ffs(m) - 1) : top_k - 1;
  if (lane == 0) *token = static_cast<int>(cand_index(sorted[pick]));
  for (int i = b; i < e; ++i) {
    if (out_idx) out_idx[i] = static_cast<int>(cand_index(sorted[i]));
    if (out_prob) out_prob[i] = wbuf[i] / total;
  }
}

std::atomic<int> g_smem_set[64];

}  // namespace

static int sample_slice(int n) {
  const int per = (n + kCluster - 1) / kCluster;
  return (per + 7) & ~7;
}

cudaError_t sample_topk_launch(const __half* logits, int n, int top_k, float temperature,
                               const float* u, int* token, int* out_idx, float* out_prob,
                               cudaStream_t st) {
  const int slice = sample_slice(n);
  const int smem = kFixedSmem + slice * 2;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && g_smem_set[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(sample_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFixedSmem + kMaxSampleSlice * 2);
    if (e != cudaSuccess) return e;
    g_smem_set[dev].store(1, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sample_topk_kernel, logits, n, slice, top_k, temperature, u,
                            token, out_idx, out_prob);
}

}  // namespace qgemv
