// stream_batch.cu -- small-batch streaming GEMV, Y[m] = W . X[m] (+ R[m])
// for M = 2..8 activation rows (INFERENCE_RESEARCH.md section 1: routing by
// M, the weights loaded once and applied to every row of the batch).
//
// Same ring as the M = 1 streaming kernel (producer warp, 1-D TMA bulk
// copies of whole rows, epilogue warp); the consumer threads differ: a
// thread owns KPT k of every row and holds its KPT activations of ALL MB
// batch rows in registers (packed fp16 pairs), decodes each code word once
// and feeds it to MB mixed fma.rn.f32.f16 chains.  Registers bound MB * KPT:
// MB = 2 and 4 use 32-k tasks, MB = 8 16-k tasks (K <= 4096; the host runs
// larger K as two 4-row passes).  Per task and row m the thread adds
// scale * T_m + bias * sum(x_m); a warp transpose-reduce leaves one partial
// per (task, m) and warp, which the epilogue warp sums in a fixed order.
#include "qgemv_stream.cuh"

namespace qgemv {
namespace {

// Code lanes of a 4-bit word (see dot_word4): (q0,q4), 16(q1,q5),
// (q2,q6), 16(q3,q7) as fp16 subnormals times 2^-24.
__device__ __forceinline__ void decode4(uint32_t w, uint32_t (&v)[4]) {
  v[0] = w & 0x000F000Fu;
  v[1] = w & 0x00F000F0u;
  const uint32_t w8 = w >> 8;
  v[2] = w8 & 0x000F000Fu;
  v[3] = w8 & 0x00F000F0u;
}

// The 8 products of one decoded 4-bit word with one batch row's packed
// activations xp[0..3] = (x_{8i+j}, x_{8i+j+4}).
__device__ __forceinline__ void fma_word4(const uint32_t (&v)[4], const uint32_t* xp, float& a,
                                          float& b) {
  asm("{\n"
      ".reg .b16 q0, q1, q2, q3, q4, q5, q6, q7;\n"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7;\n"
      "mov.b32 {q0, q4}, %2;\n"
      "mov.b32 {q1, q5}, %3;\n"
      "mov.b32 {q2, q6}, %4;\n"
      "mov.b32 {q3, q7}, %5;\n"
      "mov.b32 {x0, x4}, %6;\n"
      "mov.b32 {x1, x5}, %7;\n"
      "mov.b32 {x2, x6}, %8;\n"
      "mov.b32 {x3, x7}, %9;\n"
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
      : "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(xp[0]), "r"(xp[1]), "r"(xp[2]),
        "r"(xp[3]));
}

// Code lanes of a 2-bit word (see dot_word2): classes 1, 4, 16, 64 on the
// word and on the word >> 8.
__device__ __forceinline__ void decode2(uint32_t w, uint32_t (&v)[8]) {
  v[0] = w & 0x00030003u;
  v[1] = w & 0x000C000Cu;
  v[2] = w & 0x00300030u;
  v[3] = w & 0x00C000C0u;
  const uint32_t w8 = w >> 8;
  v[4] = w8 & 0x00030003u;
  v[5] = w8 & 0x000C000Cu;
  v[6] = w8 & 0x00300030u;
  v[7] = w8 & 0x00C000C0u;
}

// The 16 products of one decoded 2-bit word with one batch row's packed
// activations xp[0..7] = (x_{16i+j}, x_{16i+j+8}).
__device__ __forceinline__ void fma_word2(const uint32_t (&v)[8], const uint32_t* xp, float& a,
                                          float& b, float& c, float& d) {
  asm("{\n"
      ".reg .b16 p0, p1, p2, p3, p4, p5, p6, p7, p8, p9, p10, p11, p12, p13, p14, p15;\n"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7, x8, x9, x10, x11, x12, x13, x14, x15;\n"
      "mov.b32 {p0, p8}, %4;\n"
      "mov.b32 {p1, p9}, %5;\n"
      "mov.b32 {p2, p10}, %6;\n"
      "mov.b32 {p3, p11}, %7;\n"
      "mov.b32 {p4, p12}, %8;\n"
      "mov.b32 {p5, p13}, %9;\n"
      "mov.b32 {p6, p14}, %10;\n"
      "mov.b32 {p7, p15}, %11;\n"
      "mov.b32 {x0, x8}, %12;\n"
      "mov.b32 {x1, x9}, %13;\n"
      "mov.b32 {x2, x10}, %14;\n"
      "mov.b32 {x3, x11}, %15;\n"
      "mov.b32 {x4, x12}, %16;\n"
      "mov.b32 {x5, x13}, %17;\n"
      "mov.b32 {x6, x14}, %18;\n"
      "mov.b32 {x7, x15}, %19;\n"
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
      : "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(xp[0]), "r"(xp[1]), "r"(xp[2]), "r"(xp[3]), "r"(xp[4]), "r"(xp[5]), "r"(xp[6]),
        "r"(xp[7]));
}

// One task (KPT k of one row) against MB batch rows: out[m] = scale * T_m +
// bias * sum(x_m) in units of 2^-24.
template <int BITS, int KPT, int MB>
__device__ __forceinline__ void task_dot_batch(const uint8_t* codes,
                                               const uint32_t (&xp)[MB][KPT / 2], float s, float b,
                                               const float (&xs)[MB], float (&out)[MB]) {
  constexpr int NW = KPT * BITS / 32;  // code words of the task
  uint32_t w[NW];
  if (NW == 4) {
    const uint4 c = *reinterpret_cast<const uint4*>(codes);
    w[0] = c.x;
    w[1 % NW] = c.y;
    w[2 % NW] = c.z;
    w[3 % NW] = c.w;
  } else if (NW == 2) {
    const uint2 c = *reinterpret_cast<const uint2*>(codes);
    w[0] = c.x;
    w[1 % NW] = c.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(codes);
  }
  if (BITS == 4) {
    float A[MB], B[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) A[m] = B[m] = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      uint32_t v[4];
      decode4(w[i], v);
#pragma unroll
      for (int m = 0; m < MB; ++m) fma_word4(v, &xp[m][4 * i], A[m], B[m]);
    }
#pragma unroll
    for (int m = 0; m < MB; ++m) out[m] = fmaf(s, fmaf(B[m], 0.0625f, A[m]), b * xs[m]);
  } else {
    float A[MB], B[MB], C[MB], D[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) A[m] = B[m] = C[m] = D[m] = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      uint32_t v[8];
      decode2(w[i], v);
#pragma unroll
      for (int m = 0; m < MB; ++m) fma_word2(v, &xp[m][8 * i], A[m], B[m], C[m], D[m]);
    }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      const float t = fmaf(D[m], 0.015625f, fmaf(C[m], 0.0625f, fmaf(B[m], 0.25f, A[m])));
      out[m] = fmaf(s, t, b * xs[m]);
    }
  }
}

template <int BITS, int MB, int KPT, int JR>
__global__ void __launch_bounds__(MB == 8 ? 320 : (MB == 4 ? 512 : 576), 1)
    batch_kernel(const StreamArgs a) {
  constexpr int NV = JR * MB;  // partials per thread and stage
  static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "JR * MB must be a power of two <= 32");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t part_bar[kMaxStages];
  __shared__ __align__(8) uint64_t xready_bar;  // see stream_kernel

  const int T = static_cast<int>(blockDim.x) - 64;  // consumer threads
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.NS;
  const int M = a.M;
  const int N = static_cast<int>(a.rows);
  const int stride = a.interleave ? static_cast<int>(gridDim.x) * a.RS : 0;
  const int r0 = a.interleave
                     ? static_cast<int>(blockIdx.x) * a.RS
                     : static_cast<int>(static_cast<long long>(blockIdx.x) * a.rows / gridDim.x);
  const int r1 = a.interleave
                     ? N
                     : static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.rows / gridDim.x);
  const int rcb = a.K * BITS / 8;
  const int rgb = a.K / 32;
  const int scales_off = a.RS * rcb;
  const int biases_off = scales_off + a.RS * rgb;

  pdl_launch_dependents();  // see stream_kernel
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&part_bar[s]), static_cast<uint32_t>(T / 32));
      mbar_init(smem_u32(&empty_bar[s]), static_cast<uint32_t>(T / 32 + 1));
    }
    mbar_init(smem_u32(&xready_bar), static_cast<uint32_t>(T / 32));
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (StageWalker wk(r0, r1, a.RS, NS, 0, stride); wk.more();) {
        const int n = wk.rows();
        const int s = wk.slot;
        if (issued == a.prefill && !mbar_wait(smem_u32(&xready_bar), 0, &g_status)) break;
        if (!mbar_wait(smem_u32(&empty_bar[s]), wk.phase ^ 1u, &g_status)) break;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t st = smem_u32(smem + static_cast<size_t>(s) * a.stage_bytes);
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(n) * static_cast<uint32_t>(rcb + 2 * rgb));
        const long long row = wk.row;
        bulk_g2s(st, a.codes[0] + row * rcb, n * rcb, fb, pol);
        bulk_g2s(st + scales_off, a.scales[0] + row * (rgb / 2), n * rgb, fb, pol);
        bulk_g2s(st + biases_off, a.biases[0] + row * (rgb / 2), n * rgb, fb, pol);
        ++issued;
        wk.advance(n);
      }
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        mbar_wait(smem_u32(&full_bar[j % NS]), (j / NS) & 1, &g_status);
    }
    return;
  }

  const bool epi = (warp == 1);
  const int t = threadIdx.x - 64;
  const int TG = a.TG;
  const int S = a.S;
  const int slot = epi ? 0 : t / TG;
  const int uu = epi ? 0 : t - slot * TG;
  const int wit = uu >> 5, wpt = TG >> 5;
  // Per-stage partials after the ring: [NS][RS][MB][wpt].
  float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(NS) * a.stage_bytes);
  const int red_stage = (a.RS * MB * wpt + 3) & ~3;

  // ------------------------------------------------------------ epilogue
  if (epi) {
    pdl_wait();  // residuals and y belong to the stream order
    for (StageWalker wk(r0, r1, a.RS, NS, 0, stride); wk.more();) {
      const int n = wk.rows();
      const int s = wk.slot;
      const int row = wk.row;
      if (!mbar_wait(smem_u32(&part_bar[s]), wk.phase, &g_status)) return;
      const float* rs = red + static_cast<size_t>(s) * red_stage;
      for (int i = lane; i < n * M; i += 32) {
        const int r = i / M, m = i - r * M;
        float v = 0.f;
        for (int w = 0; w < wpt; ++w) v += rs[(r * MB + m) * wpt + w];
        v *= kTwo24;
        const size_t o = static_cast<size_t>(m) * N + row + r;
        if (a.residual != nullptr) v += __half2float(a.residual[o]);
        a.y[o] = __float2half_rn(v);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
      wk.advance(n);
    }
    return;
  }

  // ----------------------------------------------------------- consumers
  uint32_t xp[MB][KPT / 2];
  float xs[MB];
  pdl_wait();  // x may come from the previous kernel
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m < M) {
      load_task_x<BITS, KPT>(a.x + static_cast<size_t>(m) * a.K, nullptr, nullptr, uu * KPT, xp[m],
                             xs[m]);
    } else {
#pragma unroll
      for (int i = 0; i < KPT / 2; ++i) xp[m][i] = 0u;
      xs[m] = 0.f;
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&xready_bar));
  const int group_in_row = (uu * KPT) / 64;
  int code_off[JR], group_off[JR];
#pragma unroll
  for (int j = 0; j < JR; ++j) {
    const int rl = slot + j * S;
    code_off[j] = rl * rcb + uu * (KPT * BITS / 8);
    group_off[j] = rl * rgb + group_in_row * 2;
  }

  for (StageWalker wk(r0, r1, a.RS, NS, 0, stride); wk.more();) {
    const int n = wk.rows();
    const int s = wk.slot;
    if (!mbar_wait(smem_u32(&full_bar[s]), wk.phase, &g_status)) return;
    const uint8_t* st = smem + static_cast<size_t>(s) * a.stage_bytes;
    // Rows past a partial stage's end read stale (valid) shared memory;
    // their partials land in slots the epilogue never reads.
    float acc[NV];
#pragma unroll
    for (int j = 0; j < JR; ++j) {
      const float sv = __half2float(*reinterpret_cast<const __half*>(st + scales_off + group_off[j]));
      const float bv = __half2float(*reinterpret_cast<const __half*>(st + biases_off + group_off[j]));
      float out[MB];
      task_dot_batch<BITS, KPT, MB>(st + code_off[j], xp, sv, bv, xs, out);
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[j * MB + m] = out[m];
    }
    float* rs = red + static_cast<size_t>(s) * red_stage;
    constexpr int kLanesPerValue = 32 / NV;
    const float v = warp_reduce_rows<NV>(acc, lane);
    if ((lane & (kLanesPerValue - 1)) == 0) {
      const int vi = lane / kLanesPerValue;
      const int j = vi / MB, m = vi - j * MB;
      rs[((slot + j * S) * MB + m) * wpt + wit] = v;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&part_bar[s]));
      mbar_arrive(smem_u32(&empty_bar[s]));
    }
    wk.advance(n);
  }
}

template <int BITS, int MB, int KPT, int JR>
cudaError_t launch_batch_t(const StreamPlan& p, StreamArgs a, cudaStream_t stream, int device) {
  static unsigned done_mask = 0;
  auto* k = batch_kernel<BITS, MB, KPT, JR>;
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

template <int BITS>
cudaError_t launch_batch_bits(const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                              int device) {
  if (p.mb == 2) {
    if (p.jr == 8) return launch_batch_t<BITS, 2, 32, 8>(p, a, st, device);
    if (p.jr == 4) return launch_batch_t<BITS, 2, 32, 4>(p, a, st, device);
    if (p.jr == 2) return launch_batch_t<BITS, 2, 32, 2>(p, a, st, device);
    return launch_batch_t<BITS, 2, 32, 1>(p, a, st, device);
  }
  if (p.mb == 4) {
    if (p.jr == 4) return launch_batch_t<BITS, 4, 32, 4>(p, a, st, device);
    if (p.jr == 2) return launch_batch_t<BITS, 4, 32, 2>(p, a, st, device);
    return launch_batch_t<BITS, 4, 32, 1>(p, a, st, device);
  }
  if (p.jr == 4) return launch_batch_t<BITS, 8, 16, 4>(p, a, st, device);
  if (p.jr == 2) return launch_batch_t<BITS, 8, 16, 2>(p, a, st, device);
  return launch_batch_t<BITS, 8, 16, 1>(p, a, st, device);
}

}  // namespace

cudaError_t stream_batch(int bits, const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                         int device) {
  if (bits == 4) return launch_batch_bits<4>(p, a, st, device);
  return launch_batch_bits<2>(p, a, st, device);
}

cudaError_t status_batch(unsigned* out) { return read_clear_status(out); }

}  // namespace qgemv
