// qgemv_stream.cuh -- the streaming dequant-fused GEMV kernel for sm_103a.
//
// Design (GB300-first; the Metal simdgroup-per-row-band kernels the pages
// describe in INFERENCE_RESEARCH.md section 1 are prior art, not the plan):
//
//  * Persistent: one CTA per SM.  CTA b owns the contiguous row range
//    [b*R/P, (b+1)*R/P) of the R output rows (P CTAs), so every SM streams
//    the same number of bytes and a CTA's codes, scales and biases are
//    contiguous blocks of memory.
//  * Warp 0 (one lane) is the producer: it streams the range in stages of RS
//    rows (of every matrix the op reads) with 1-D TMA bulk copies
//    (cp.async.bulk, L2 evict-first) into an NS-deep shared-memory ring
//    guarded by mbarriers.  No multicast.
//  * The other T threads are consumers.  A stage holds MS x RS "tasks"
//    (matrix slot, row).  Threads form slots of TG = K/32 threads; thread uu
//    of a slot owns k in [32 uu, 32 uu + 32) of every row (KPT = 32, half a
//    quantisation group), so its activations sit in registers (16 packed
//    fp16 pairs) for the whole kernel.  The S = T/TG slots take the tasks
//    round-robin, JR per thread.  (Whole-group tasks, 64 k per thread,
//    measured slower on GB300: twice the activation registers and 32-byte
//    strided code loads.)
//  * Inner loop: dot_word4 / dot_word2 (fp16-subnormal codes x fp16
//    activations with the mixed fma.rn.f32.f16, exact products, fp32 sums),
//    then scale * sum(q x) + bias * sum(x) per slice: the FMA-reordered
//    dequantisation of the hada.io page (topic 27758), factored per group.
//  * Row sums: a warp transpose-reduce of the JR task partials (log2 JR
//    split levels, then plain xor levels) and one shared-memory slot per
//    warp and task.  Consumer warps never wait for each other: each stores
//    its partials and arrives on the stage's "partials" mbarrier.  Warp 1
//    is the epilogue warp: it waits for that barrier, sums the slots in a
//    fixed order (deterministic), applies the epilogue (residual, RMSNorm
//    scale, SwiGLU, MoE weights) and stores the rows.  A stage is released
//    to the producer only when every consumer warp and the epilogue warp
//    are done with it, so the slots are reused only after they were read.
//  * The consumers' row loop is branch-free: all JR slices of a stage are
//    computed (rows past the stage's end read stale but valid shared memory)
//    and masked afterwards, so the compiler can interleave the rows' FMA
//    chains and hoist their shared-memory loads.
//  * Every thread loads its own 32-k activation slice straight from global
//    memory (L2): no block-wide staging, so no barrier among the consumer
//    warps at all, and each starts as soon as its slice and stage are in.
//    The producer issues only the plan's first `prefill` stages (about 100
//    KB) before every consumer warp has its slice (the `xready` mbarrier):
//    activation loads issued behind a full ring of outstanding weight copies
//    waited about a microsecond longer.
//  * Every mbarrier wait is bounded (about 1 s); a timeout sets a status bit
//    and the waiting thread returns instead of hanging (no named barrier
//    exists, so nothing is left waiting).
#pragma once

#include <cuda_runtime.h>

#include "qgemv_args.h"
#include "qgemv_device.cuh"

namespace qgemv {

// Status word of this translation unit (bit kStatusWaitTimeout).
static __device__ unsigned g_status = 0;

// A thread's task: KPT consecutive k of one row (KPT = 32: half a
// quantisation group), its codes (KPT * BITS / 8 bytes) and its activations,
// held as KPT / 2 packed fp16 pairs.
template <int BITS, int KPT>
struct Task {
  static constexpr int kCodeBytes = KPT * BITS / 8;  // 16 / 32 (4-bit), 8 / 16 (2-bit)
  static constexpr int kXRegs = KPT / 2;
};

// Stage walker shared by the producer, the consumers and the epilogue warp:
// the rows of each stage, the ring slot and its phase parity.
//  * contiguous (stride == 0): the CTA walks its own row range [r0, r1) in
//    stages of up to RS rows (for kMoeUp never across an expert boundary);
//  * interleaved (stride > 0): stage g covers rows [g RS, g RS + RS) and the
//    CTA walks g = blockIdx.x, + P, + 2P, ..., so at any moment all SMs read
//    neighbouring stages of the same region of memory.  (Used when every
//    expert boundary falls on a stage boundary.)
// No divisions on the per-stage path except kMoeUp's interleaved expert
// lookup.
struct StageWalker {
  int row, r1, rs, ns;
  int rows_per_expert;  // kMoeUp only, else 0
  int expert_slot, left_in_expert;
  int stride;           // rows between this CTA's stages when interleaved, else 0
  int slot;
  uint32_t phase;

  __device__ __forceinline__ StageWalker(int r0_, int r1_, int rs_, int ns_, int rpe, int stride_)
      : row(r0_), r1(r1_), rs(rs_), ns(ns_), rows_per_expert(rpe), stride(stride_), slot(0),
        phase(0) {
    expert_slot = rpe > 0 ? r0_ / rpe : 0;
    left_in_expert = rpe > 0 ? rpe - (r0_ - expert_slot * rpe) : 0x7fffffff;
  }
  __device__ __forceinline__ bool more() const { return row < r1; }
  __device__ __forceinline__ int rows() const {
    int n = r1 - row;
    if (n > rs) n = rs;
    if (n > left_in_expert) n = left_in_expert;
    return n;
  }
  __device__ __forceinline__ void advance(int n) {
    if (stride > 0) {
      row += stride;
      if (rows_per_expert > 0 && row < r1) {
        expert_slot = row / rows_per_expert;
        left_in_expert = rows_per_expert - (row - expert_slot * rows_per_expert);
      }
    } else {
      row += n;
      if (rows_per_expert > 0) {
        left_in_expert -= n;
        if (left_in_expert == 0) {
          ++expert_slot;
          left_in_expert = rows_per_expert;
        }
      }
    }
    if (++slot == ns) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Transpose-reduce JR partials across a warp.  Returns, on lanes with
// lane % (32/JR) == 0, the warp's sum of partial j = lane / (32/JR).
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

// One task: sum over its KPT k of w * x, in units of 2^-24, as
// scale * sum(q x) + bias * sum(x) (xs_scaled = sum(x) * 2^-24).
template <int BITS, int KPT>
__device__ __forceinline__ float task_dot(const uint8_t* codes, const uint32_t* xp, float s,
                                          float b, float xs_scaled) {
  float t;
  if (BITS == 4) {
    float a0 = 0.f, b0 = 0.f, a1 = 0.f, b1 = 0.f;
#pragma unroll
    for (int q = 0; q < KPT / 32; ++q) {
      const uint4 c = *reinterpret_cast<const uint4*>(codes + 16 * q);
      dot_word4(c.x, xp + 16 * q + 0, a0, b0);
      dot_word4(c.y, xp + 16 * q + 4, a1, b1);
      dot_word4(c.z, xp + 16 * q + 8, a0, b0);
      dot_word4(c.w, xp + 16 * q + 12, a1, b1);
    }
    t = fmaf(b0 + b1, 0.0625f, a0 + a1);
  } else if (BITS == 8) {
    float a0 = 0.f, b0 = 0.f, a1 = 0.f, b1 = 0.f;
#pragma unroll
    for (int q = 0; q < KPT / 16; ++q) {
      const uint4 c = *reinterpret_cast<const uint4*>(codes + 16 * q);
      dot_word8(c.x, xp + 8 * q + 0, a0, b0);
      dot_word8(c.y, xp + 8 * q + 2, a1, b1);
      dot_word8(c.z, xp + 8 * q + 4, a0, b0);
      dot_word8(c.w, xp + 8 * q + 6, a1, b1);
    }
    t = (a0 + b0) + (a1 + b1);
  } else {
    float ca = 0.f, cb = 0.f, cc = 0.f, cd = 0.f;
#pragma unroll
    for (int q = 0; q < KPT / 32; ++q) {
      const uint2 c = *reinterpret_cast<const uint2*>(codes + 8 * q);
      dot_word2(c.x, xp + 16 * q + 0, ca, cb, cc, cd);
      dot_word2(c.y, xp + 16 * q + 8, ca, cb, cc, cd);
    }
    t = fmaf(cd, 0.015625f, fmaf(cc, 0.0625f, fmaf(cb, 0.25f, ca)));
  }
  return fmaf(s, t, b * xs_scaled);
}

// A thread's KPT activations k in [k0, k0 + KPT), read straight from global
// memory: fp16 x (times gamma when given) or fp32 xf, rounded to fp16 once
// (the kernels multiply fp16 activations) and packed in the pairing of the
// code lanes (4-bit: (x_{8i+j}, x_{8i+j+4}); 2-bit: (x_{16i+j}, x_{16i+j+8})),
// plus their sum times 2^-24 (the dot products' scale).  16-byte aligned.
// gpre: gamma[k0 .. k0 + KPT) already loaded (load_gamma), else read here;
// sq (optional) receives the sum of squares of the raw x (for RMSNorm).
template <int BITS, int KPT>
__device__ __forceinline__ void load_task_x(const __half* x, const __half* gamma, const float* xf,
                                            int k0, uint32_t (&xp)[KPT / 2], float& xs_scaled,
                                            const uint4* gpre = nullptr, float* sq = nullptr) {
  float part[KPT / 16];
  float sqa = 0.f;
#pragma unroll
  for (int c = 0; c < KPT / 16; ++c) {  // 16 activations at a time
    float xv[16];
    if (xf != nullptr) {
      const float4* src = reinterpret_cast<const float4*>(xf + k0 + 16 * c);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = src[i];
        xv[4 * i + 0] = f.x;
        xv[4 * i + 1] = f.y;
        xv[4 * i + 2] = f.z;
        xv[4 * i + 3] = f.w;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(x + k0 + 16 * c);
      uint4 raw[2] = {src[0], src[1]};
      uint4 graw[2];
      if (gpre != nullptr) {
        graw[0] = gpre[2 * c];
        graw[1] = gpre[2 * c + 1];
      } else if (gamma != nullptr) {
        const uint4* g = reinterpret_cast<const uint4*>(gamma + k0 + 16 * c);
        graw[0] = g[0];
        graw[1] = g[1];
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const __half2* h = reinterpret_cast<const __half2*>(&raw[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float2 f = __half22float2(h[j]);
          if (sq != nullptr) sqa = fmaf(f.x, f.x, fmaf(f.y, f.y, sqa));
          if (gamma != nullptr) {
            const float2 gf = __half22float2(reinterpret_cast<const __half2*>(&graw[i])[j]);
            f.x *= gf.x;
            f.y *= gf.y;
          }
          xv[8 * i + 2 * j] = f.x;
          xv[8 * i + 2 * j + 1] = f.y;
        }
      }
    }
    unsigned short hv[16];
    part[c] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const __half h = __float2half_rn(xv[k]);
      hv[k] = __half_as_ushort(h);
      part[c] += __half2float(h);
    }
    if (BITS == 4) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          xp[8 * c + 4 * i + j] = static_cast<uint32_t>(hv[8 * i + j]) |
                                  (static_cast<uint32_t>(hv[8 * i + j + 4]) << 16);
    } else if (BITS == 8) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // word i of the chunk: k = 4i .. 4i+3
        xp[8 * c + 2 * i] =
            static_cast<uint32_t>(hv[4 * i]) | (static_cast<uint32_t>(hv[4 * i + 2]) << 16);
        xp[8 * c + 2 * i + 1] =
            static_cast<uint32_t>(hv[4 * i + 1]) | (static_cast<uint32_t>(hv[4 * i + 3]) << 16);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        xp[8 * c + j] = static_cast<uint32_t>(hv[j]) | (static_cast<uint32_t>(hv[j + 8]) << 16);
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < KPT / 16; ++c) sum += part[c];
  xs_scaled = sum * kTwoM24;
  if (sq != nullptr) *sq = sqa;
}

// gamma[k0 .. k0 + KPT) into registers (a weight: no kernel writes it, so
// it may be read before the previous kernel's grid has completed).
template <int KPT>
__device__ __forceinline__ void load_gamma(const __half* gamma, int k0, uint4 (&g)[KPT / 8]) {
  const uint4* src = reinterpret_cast<const uint4*>(gamma + k0);
#pragma unroll
  for (int i = 0; i < KPT / 8; ++i) g[i] = src[i];
}

template <int BITS, int MODE, int JR, int KPT>
__global__ void __launch_bounds__(576, 1) stream_kernel(const StreamArgs a) {
  using TK = Task<BITS, KPT>;
  constexpr int NMAT = (MODE == kSwiglu || MODE == kMoeUp) ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t part_bar[kMaxStages];
  __shared__ __align__(8) uint64_t xready_bar;  // every consumer warp has its activations
  __shared__ int s_eidx[kMaxTopK];
  __shared__ float s_ewt[kMaxTopK];
  __shared__ float s_sq[16];  // RMSNorm modes: sums of x^2 of slot 0's consumer warps
  __shared__ float s_res[64];  // residual rows of a CTA's row band (at most 64 rows)

  const int T = static_cast<int>(blockDim.x) - 64;  // consumer threads
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.NS;
  const int stride = a.interleave ? static_cast<int>(gridDim.x) * a.RS : 0;
  const int r0 = a.interleave
                     ? static_cast<int>(blockIdx.x) * a.RS
                     : static_cast<int>(static_cast<long long>(blockIdx.x) * a.rows / gridDim.x);
  const int r1 = a.interleave
                     ? static_cast<int>(a.rows)
                     : static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.rows / gridDim.x);
  const int rpe = (MODE == kMoeUp) ? a.rows_per_expert : 0;
  const int rcb = a.K * BITS / 8;  // code bytes per row
  const int rgb = a.K / 32;        // scale (or bias) bytes per row
  const int MS = (MODE == kMoeDown) ? a.top_k : NMAT;  // matrices per stage
  const int codes_off = 0;
  const int scales_off = MS * a.RS * rcb;
  const int biases_off = scales_off + MS * a.RS * rgb;

  // The next kernel of the stream may start launching now: its producer
  // streams weights (which no kernel writes) while its consumers wait for
  // this grid (pdl_wait below).
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&part_bar[s]), static_cast<uint32_t>(T / 32));
      mbar_init(smem_u32(&empty_bar[s]), static_cast<uint32_t>(T / 32 + 1));
    }
    mbar_init(smem_u32(&xready_bar), static_cast<uint32_t>(T / 32));
    fence_mbar_init();
    if (MODE == kMoeUp || MODE == kMoeDown) {
      pdl_wait();  // the expert indices and weights may come from the previous kernel
      for (int k = 0; k < a.top_k; ++k) {
        const int e = a.idx[k];
        const float w = a.wt[k];
        const bool ok = e >= 0 && e < a.n_experts;
        s_eidx[k] = ok ? e : -1;
        s_ewt[k] = ok ? w : 0.f;
        if (!ok && blockIdx.x == 0 && a.err_flag != nullptr) *a.err_flag = 1;
        if (a.trace != nullptr && static_cast<int>(blockIdx.x) < a.trace_ctas)
          reinterpret_cast<uint4*>(a.trace)[blockIdx.x * a.top_k + k] =
              make_uint4(static_cast<unsigned>(e), __float_as_uint(w),
                         static_cast<unsigned>(s_eidx[k]), __float_as_uint(s_ewt[k]));
      }
    }
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (StageWalker wk(r0, r1, a.RS, NS, rpe, stride); wk.more();) {
        const int n = wk.rows();
        const int s = wk.slot;
        // After the first a.prefill stages, wait until the consumers hold
        // their activations: their loads would otherwise queue behind the
        // weight copies in flight.
        if (issued == a.prefill && !mbar_wait(smem_u32(&xready_bar), 0, &g_status)) break;
        if (!mbar_wait(smem_u32(&empty_bar[s]), wk.phase ^ 1u, &g_status)) break;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t st = smem_u32(smem + static_cast<size_t>(s) * a.stage_bytes);
        // Expected bytes of every valid matrix slot first, then the copies.
        uint32_t bytes = 0;
        for (int m = 0; m < MS; ++m) {
          const int e = (MODE == kMoeUp)     ? s_eidx[wk.expert_slot]
                        : (MODE == kMoeDown) ? s_eidx[m]
                                             : 0;
          if (e >= 0) bytes += static_cast<uint32_t>(n) * static_cast<uint32_t>(rcb + 2 * rgb);
        }
        mbar_arrive_expect_tx(fb, bytes);
        for (int m = 0; m < MS; ++m) {
          long long lrow = wk.row;
          int e = 0;
          if (MODE == kMoeUp) {
            e = s_eidx[wk.expert_slot];
            lrow = rpe - wk.left_in_expert;
          } else if (MODE == kMoeDown) {
            e = s_eidx[m];
          }
          if (e < 0) continue;
          const int which = (MODE == kMoeDown) ? 0 : m;
          const long long ec = static_cast<long long>(e) * a.ex_code_bytes;
          const long long eg = static_cast<long long>(e) * a.ex_groups;
          bulk_g2s(st + codes_off + m * a.RS * rcb, a.codes[which] + ec + lrow * rcb, n * rcb, fb,
                   pol);
          bulk_g2s(st + scales_off + m * a.RS * rgb, a.scales[which] + eg + lrow * (rgb / 2),
                   n * rgb, fb, pol);
          bulk_g2s(st + biases_off + m * a.RS * rgb, a.biases[which] + eg + lrow * (rgb / 2),
                   n * rgb, fb, pol);
        }
        ++issued;
        wk.advance(n);
      }
      const int it = issued;
      // Drain: never leave while a copy into this CTA's shared memory is in flight.
      for (int j = (it > NS ? it - NS : 0); j < it; ++j)
        mbar_wait(smem_u32(&full_bar[j % NS]), (j / NS) & 1, &g_status);
    }
    return;
  }

  // ------------------------------------------------- consumers and epilogue
  const bool epi = (warp == 1);           // the epilogue warp
  const int t = threadIdx.x - 64;         // consumer index (negative for warp 1)
  const int TG = a.TG;
  const int S = a.S;
  const int slot = epi ? 0 : t / TG;
  const int uu = epi ? 0 : t - slot * TG;  // this thread's slice index within a row
  const int wit = uu >> 5;       // warp index within the slot
  const int wpt = TG >> 5;       // warps per slot
  const int ek = (MODE == kMoeDown) ? slot % a.top_k : 0;  // kMoeDown: fixed expert slot
  const bool use_gamma = (MODE == kNorm) || (MODE == kSwiglu && a.gamma != nullptr);
  const int tasks = MS * a.RS;  // per stage
  // Per-stage partial-sum slots, after the ring: [NS][tasks][wpt].
  float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(NS) * a.stage_bytes);
  const int red_stage = (tasks * wpt + 3) & ~3;  // floats, 16-byte multiple

  if (epi) {
    // Epilogue warp: finish every stage's rows once all partials are in
    // (the RMS of the input, RMSNorm modes, from the consumers' sums of
    // squares).  It reads residuals and writes y, so it waits for the
    // previous kernel first.
    pdl_wait();
    unsigned long long am_best = 0;  // kArgmax: this lane's best (value, index) key
    float rstd = 1.f;
    if (use_gamma) {
      // Slot 0's warps store their sums of x^2 before arriving on xready,
      // so the RMS is ready while the first stage is being computed.
      if (!mbar_wait(smem_u32(&xready_bar), 0, &g_status)) return;
      float tot = 0.f;
      for (int w = 0; w < wpt; ++w) tot += s_sq[w];
      rstd = 1.0f / sqrtf(tot / static_cast<float>(a.K) + a.eps);
    }
    // A contiguous band of at most 64 rows: load its residual rows now, so
    // the last stage's tail does not wait for them.
    const bool res_pre = (MODE == kPlain || MODE == kMoeDown) && a.residual != nullptr &&
                         !a.interleave && r1 - r0 <= 64;
    if (res_pre) {
      for (int i = lane; i < r1 - r0; i += 32) s_res[i] = __half2float(a.residual[r0 + i]);
      __syncwarp();
    }
    for (StageWalker wk(r0, r1, a.RS, NS, rpe, stride); wk.more();) {
      const int n = wk.rows();
      const int s = wk.slot;
      const int row = wk.row;
      if (!mbar_wait(smem_u32(&part_bar[s]), wk.phase, &g_status)) return;
      const bool ok = (MODE == kMoeUp) ? (s_eidx[wk.expert_slot] >= 0) : true;
      const float* rs = red + static_cast<size_t>(s) * red_stage;
      for (int r = lane; r < n; r += 32) {
        const int gr = row + r;
        float v[NMAT];
        if (MODE == kMoeDown) {
          v[0] = 0.f;
          for (int k = 0; k < a.top_k; ++k) {
            float e = 0.f;
            for (int w = 0; w < wpt; ++w) e += rs[(r * a.top_k + k) * wpt + w];
            v[0] = fmaf(s_ewt[k], e, v[0]);
          }
        } else {
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            v[m] = 0.f;
            for (int w = 0; w < wpt; ++w) v[m] += rs[(m * a.RS + r) * wpt + w];
          }
        }
#pragma unroll
        for (int m = 0; m < NMAT; ++m) v[m] *= kTwo24;
        if (MODE == kPlain || MODE == kMoeDown) {
          float o = v[0];
          if (res_pre)
            o += s_res[gr - r0];
          else if (a.residual != nullptr)
            o += __half2float(a.residual[gr]);
          a.y[gr] = __float2half_rn(o);
        } else if (MODE == kArgmax) {
          const __half h = __float2half_rn(v[0]);
          a.y[gr] = h;
          am_best = max_key(am_best, argmax_key(__half2float(h), gr));
        } else if (MODE == kNorm) {
          a.y[gr] = __float2half_rn(v[0] * rstd);
        } else if (MODE == kSwiglu) {
          const float g = v[0] * rstd, u = v[NMAT - 1] * rstd;
          a.y[gr] = __float2half_rn(silu_f(g) * u);
        } else if (MODE == kMoeUp) {
          a.yf[gr] = ok ? silu_f(v[0]) * v[NMAT - 1] : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
      wk.advance(n);
    }
    if (MODE == kArgmax) {
      // The CTA's best (value, index) into the global key with a reduction
      // that returns nothing, so the CTA does not wait for it; the finalize
      // kernel that follows reads the key once this grid has completed.
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        am_best = max_key(am_best, __shfl_xor_sync(0xffffffffu, am_best, o));
      if (lane == 0)
        asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(a.am_key), "l"(am_best)
                     : "memory");
    }
    return;
  }

  // This thread's KPT activations, packed fp16 pairs, and their sum (times
  // 2^-24, the dot products' scale), straight from global memory: no
  // block-wide staging or barrier, so each warp starts on its own.
  uint32_t xp[TK::kXRegs];
  float xs_scaled;
  uint4 gpre[KPT / 8];
  if (use_gamma) load_gamma<KPT>(a.gamma, uu * KPT, gpre);  // before the wait: a weight
  pdl_wait();  // x may come from the previous kernel
  if (MODE == kMoeDown)
    load_task_x<BITS, KPT>(nullptr, nullptr, a.xf + static_cast<size_t>(ek) * a.K, uu * KPT, xp,
                           xs_scaled);
  else if (MODE == kPlain && a.gather_hd > 0) {
    // a KPT-k slice lies inside one head (head_dim % KPT == 0, host-checked)
    const int k0 = uu * KPT;
    const int head = k0 / a.gather_hd;
    const __half* src =
        a.x + static_cast<long long>(a.gather_nq + a.gather_nkv + head / (a.gather_nq / a.gather_nkv)) *
                  a.gather_hd +
        (k0 - head * a.gather_hd);
    load_task_x<BITS, KPT>(src, nullptr, nullptr, 0, xp, xs_scaled);
  } else if (use_gamma) {
    float sq;
    load_task_x<BITS, KPT>(a.x, a.gamma, nullptr, uu * KPT, xp, xs_scaled, gpre, &sq);
    if (slot == 0) {  // slot 0's threads cover K once: its warps' sums give mean(x^2)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0) s_sq[wit] = sq;
    }
  } else {
    load_task_x<BITS, KPT>(a.x, nullptr, nullptr, uu * KPT, xp, xs_scaled);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&xready_bar));
  const bool expert_ok = (MODE == kMoeDown) ? (s_eidx[ek] >= 0) : true;
  const int group_in_row = (uu * KPT) / 64;
  // Task j of this thread in every stage: matrix slot and row, and the
  // shared-memory offsets of its slice.
  int code_off[JR], group_off[JR];
#pragma unroll
  for (int j = 0; j < JR; ++j) {
    const int task = slot + j * S;
    int ms, rl;
    if (MODE == kMoeDown) {
      ms = ek;
      rl = task / a.top_k;
    } else {
      ms = task / a.RS;
      rl = task - ms * a.RS;
    }
    code_off[j] = (ms * a.RS + rl) * rcb + uu * TK::kCodeBytes;
    group_off[j] = (ms * a.RS + rl) * rgb + group_in_row * 2;
  }

  for (StageWalker wk(r0, r1, a.RS, NS, rpe, stride); wk.more();) {
    const int n = wk.rows();
    const int s = wk.slot;
    if (!mbar_wait(smem_u32(&full_bar[s]), wk.phase, &g_status)) return;
    const uint8_t* st = smem + static_cast<size_t>(s) * a.stage_bytes;
    const bool slot_ok = expert_ok;

    float acc[JR];
#pragma unroll
    for (int j = 0; j < JR; ++j) {
      const __half sv = *reinterpret_cast<const __half*>(st + scales_off + group_off[j]);
      const __half bv = *reinterpret_cast<const __half*>(st + biases_off + group_off[j]);
      const float v = task_dot<BITS, KPT>(st + codes_off + code_off[j], xp, __half2float(sv),
                                          __half2float(bv), xs_scaled);
      // Tasks of rows past a partial stage's end read stale (valid) shared
      // memory; their partials land in reduction slots the epilogue never
      // reads, so no mask.  An invalid MoE expert's partial must be zero:
      // its slot weight is zero, but its stale scale may not be finite.
      acc[j] = (MODE == kMoeDown && !slot_ok) ? 0.f : v;
    }

    // Warp partials of this stage's tasks into the stage's slots.
    float* rs = red + static_cast<size_t>(s) * red_stage;
    {
      constexpr int kLanesPerRow = 32 / JR;
      const float v = warp_reduce_rows<JR>(acc, lane);
      if ((lane & (kLanesPerRow - 1)) == 0) rs[(slot + (lane / kLanesPerRow) * S) * wpt + wit] = v;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&part_bar[s]));
      mbar_arrive(smem_u32(&empty_bar[s]));
    }
    wk.advance(n);
  }
}

// Launch with programmatic stream serialisation allowed, so the kernel may
// start while the previous kernel of the stream finishes (see
// pdl_launch_dependents / pdl_wait).
template <typename F>
inline cudaError_t launch_pdl(F* kernel, const StreamPlan& p, const StreamArgs& a,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(p.t + 64));
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
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

template <int BITS, int MODE, int JR, int KPT>
inline cudaError_t launch_stream_t(const StreamPlan& p, StreamArgs a, cudaStream_t stream,
                                   int device) {
  static unsigned done_mask = 0;
  auto* k = stream_kernel<BITS, MODE, JR, KPT>;
  cudaError_t e = ensure_smem_attr(k, 220 * 1024, &done_mask, device);
  if (e != cudaSuccess) return e;
  a.TG = p.tg;
  a.S = p.s;
  a.RS = p.rs;
  a.NS = p.ns;
  a.stage_bytes = p.stage_bytes;
  a.interleave = p.interleave;
  a.prefill = p.prefill;
  return launch_pdl(k, p, a, stream);
}

// Dispatch on the plan's tasks per thread.
template <int BITS, int MODE>
inline cudaError_t launch_stream(const StreamPlan& p, const StreamArgs& a, cudaStream_t stream,
                                 int device) {
  switch (p.jr) {
    case 8: return launch_stream_t<BITS, MODE, 8, 32>(p, a, stream, device);
    case 4: return launch_stream_t<BITS, MODE, 4, 32>(p, a, stream, device);
    case 2: return launch_stream_t<BITS, MODE, 2, 32>(p, a, stream, device);
    default: return launch_stream_t<BITS, MODE, 1, 32>(p, a, stream, device);
  }
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
