// stack.cu -- qgemv_decode_stack: one decode token through a whole stack of
// pre-norm transformer layers' quantized matvecs in ONE persistent launch.
//
// Per layer l (INFERENCE_RESEARCH.md section 1: one command buffer encoding
// the whole layer stack, fused kernels, no per-token overhead):
//   op 0  qkv  = W_qkv . (x_l * gamma1) * rstd(x_l)          (RMSNorm fused)
//   op 1  h    = x_l + W_o . attn,  attn = value heads of qkv (decode over
//                one cached position: softmax of one score is 1)
//   op 2  act  = silu(W_g . x~) * (W_u . x~),  x~ = h * gamma2 * rstd(h)
//   op 3  x_{l+1} = h + W_d . act
//
// Why one launch: each op alone streams 9-66 MB and pays a fixed launch,
// prologue and ring-fill cost of a few microseconds; 4 launches per layer
// (5 with the value-head copy) x 32 layers made those fixed costs a large
// part of the token.  Here the producer warp of every CTA streams the
// weights of all ops of all layers back to back through one TMA ring
// (weights never depend on activations), so the ring stays full across op
// boundaries.  Only the consumers of an op wait for the op that produces
// their input: the epilogue warp publishes each op's completion on a
// grid-wide counter (fence + atomic), one lane per CTA polls that counter
// (acquire) and passes it on to the CTA's consumer warps through a
// shared-memory mbarrier, and each consumer thread then loads its own
// 32-k input slice from global memory.  The launch is cooperative, so every
// CTA is resident and the counter waits can always complete; each wait is
// bounded (~1 s) and sets the library status bit instead of hanging.
#include <atomic>

#include "qgemv.h"
#include "qgemv_stream.cuh"

namespace qgemv {
namespace {

constexpr int kMaxStackLayers = 64;
constexpr int kStackJR = 4;
constexpr int kOps = 4;  // qkv, o, gate.up, down
constexpr int kResRows = 256;  // residual rows an epilogue prefetches per op

struct StackLayerDev {
  const uint8_t* w[5];  // qkv, o, gate, up, down codes
  const __half* s[5];
  const __half* b[5];
  const __half* g1;  // attention norm
  const __half* g2;  // MLP norm
};

struct OpPlanDev {
  int K, rows, TG, S, RS, MS, stage_bytes, interleave;
};

struct StackArgs {
  StackLayerDev layers[kMaxStackLayers];
  OpPlanDev plan[kOps];
  const __half* x_in;
  __half* y_out;
  __half* qkv;
  __half* h;
  __half* act;
  __half* xbuf[2];
  int* counters;  // [n_layers * 4] lines of 128 bytes, zero on entry
  int n_layers, H, n_q, n_kv, hd, I;
  float eps;
  int NS, slot_bytes, red_slot_floats;
};

// Ring position shared in lockstep by the three roles.
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  int ns;
  __device__ explicit Ring(int ns_) : ns(ns_) {}
  __device__ __forceinline__ void advance() {
    if (++slot == ns) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// This CTA's rows of an op: contiguous range, or interleaved stages.
struct OpRows {
  int r0, r1, stride;
};

__device__ __forceinline__ OpRows op_rows(const OpPlanDev& p) {
  OpRows o;
  if (p.interleave) {
    o.r0 = static_cast<int>(blockIdx.x) * p.RS;
    o.r1 = p.rows;
    o.stride = static_cast<int>(gridDim.x) * p.RS;
  } else {
    o.r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.rows / gridDim.x);
    o.r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.rows / gridDim.x);
    o.stride = 0;
  }
  return o;
}

__device__ __forceinline__ int next_row(const OpRows& o, int row, int n) {
  return o.stride ? row + o.stride : row + n;
}

// Index of the op whose output op (l, k) reads, or -1 (the stack input).
__device__ __forceinline__ int dependency(int l, int k) {
  if (k == 0) return l == 0 ? -1 : (l - 1) * kOps + 3;
  return l * kOps + k - 1;
}

// Bounded wait until *c >= target (gpu-scope acquire).
__device__ bool wait_counter(const int* c, int target) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) return true;
    __nanosleep(64);
    if (global_timer_ns() - t0 > 1000000000ull) {
      atomicOr(&g_status, kStatusWaitTimeout);
      return false;
    }
  }
}

// Grid completion counter of op c; each on its own 128-byte line, so the
// pollers of one op and the adders of the next do not share a line.
constexpr int kCounterStride = 32;
__device__ __forceinline__ int* counter(const StackArgs& a, int c) {
  return a.counters + c * kCounterStride;
}

__device__ __forceinline__ const __half* op_input(const StackArgs& a, int l, int k) {
  switch (k) {
    case 0: return l == 0 ? a.x_in : a.xbuf[l & 1];
    case 1: return a.qkv;
    case 2: return a.h;
    default: return a.act;
  }
}

__device__ __forceinline__ const __half* layer_input(const StackArgs& a, int l) {
  return l == 0 ? a.x_in : a.xbuf[l & 1];
}

// The consumer warps' share of op (l, k): each thread loads its KPT-k slice
// of the op's input straight from global memory (ops 0 and 2 multiply by
// gamma here; rstd is applied by the epilogue warp), then streams the op's
// stages from the ring.  Returns false after a timed-out wait.
template <int KPT, int JR>
__device__ __forceinline__ bool consume_op(const StackArgs& a, int l, int k, int t, int lane,
                                           Ring& ring, uint8_t* smem, float* red,
                                           uint64_t* full_bar, uint64_t* part_bar,
                                           uint64_t* empty_bar) {
  using TK = Task<4, KPT>;
  const OpPlanDev& p = a.plan[k];
  const StackLayerDev& L = a.layers[l];
  const int K = p.K;
  const int TG = p.TG, S = p.S;
  const bool active = t < S * TG;  // whole warps
  const int slot = active ? t / TG : 0;
  const int uu = active ? t - slot * TG : 0;
  const int wit = uu >> 5, wpt = TG >> 5;
  const int rcb = K / 2, rgb = K / 32;
  const int scales_off = p.MS * p.RS * rcb;
  const int biases_off = scales_off + p.MS * p.RS * rgb;
  uint32_t xp[TK::kXRegs];
  float xs_scaled = 0.f;
  if (active) {
    const int k0 = uu * KPT;
    if (k == 1) {
      // attention output = the value heads of qkv; a 32-k slice lies
      // inside one head (head_dim % 32 == 0, checked by the host)
      const int head = k0 / a.hd;
      const __half* src = a.qkv +
                          static_cast<long long>(a.n_q + a.n_kv + head / (a.n_q / a.n_kv)) * a.hd +
                          (k0 - head * a.hd);
      load_task_x<4, KPT>(src, nullptr, nullptr, 0, xp, xs_scaled);
    } else {
      const __half* gam = (k == 0) ? L.g1 : (k == 2) ? L.g2 : nullptr;
      load_task_x<4, KPT>(op_input(a, l, k), gam, nullptr, k0, xp, xs_scaled);
    }
  }
  int code_off[JR], group_off[JR];
  const int group_in_row = (uu * KPT) / 64;
#pragma unroll
  for (int j = 0; j < JR; ++j) {
    const int task = slot + j * S;
    const int ms = task / p.RS;
    const int rl = task - ms * p.RS;
    code_off[j] = (ms * p.RS + rl) * rcb + uu * TK::kCodeBytes;
    group_off[j] = (ms * p.RS + rl) * rgb + group_in_row * 2;
  }

  const OpRows o = op_rows(p);
  for (int row = o.r0; row < o.r1;) {
    const int n = min(p.RS, o.r1 - row);
    if (!mbar_wait(smem_u32(&full_bar[ring.slot]), ring.phase, &g_status)) return false;
    if (active) {
      const uint8_t* st = smem + static_cast<size_t>(ring.slot) * a.slot_bytes;
      float acc[JR];
#pragma unroll
      for (int j = 0; j < JR; ++j) {
        const __half sv = *reinterpret_cast<const __half*>(st + scales_off + group_off[j]);
        const __half bv = *reinterpret_cast<const __half*>(st + biases_off + group_off[j]);
        const float v = task_dot<4, KPT>(st + code_off[j], xp, __half2float(sv), __half2float(bv),
                                         xs_scaled);
        acc[j] = v;  // rows past a partial stage's end: partials never read
      }
      float* rs = red + static_cast<size_t>(ring.slot) * a.red_slot_floats;
      constexpr int kLanesPerRow = 32 / JR;
      const float v = warp_reduce_rows<JR>(acc, lane);
      if ((lane & (kLanesPerRow - 1)) == 0) rs[(slot + (lane / kLanesPerRow) * S) * wpt + wit] = v;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&part_bar[ring.slot]));
      mbar_arrive(smem_u32(&empty_bar[ring.slot]));
    }
    ring.advance();
    row = next_row(o, row, n);
  }
  return true;
}

__global__ void __launch_bounds__(576, 1) stack_kernel(const __grid_constant__ StackArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t part_bar[kMaxStages];
  // One phase per op: the epilogue warp's lane 0 acquires the grid counter of
  // the op's input and arrives here; the consumer warps wait here instead of
  // all polling the counter.
  __shared__ __align__(8) uint64_t dep_bar;
  __shared__ float res_sm[kResRows];  // epilogue: residual rows of the op

  const int T = static_cast<int>(blockDim.x) - 64;  // consumer threads
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.NS;
  const int P = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&part_bar[s]), static_cast<uint32_t>(T / 32));
      mbar_init(smem_u32(&empty_bar[s]), static_cast<uint32_t>(T / 32 + 1));
    }
    mbar_init(smem_u32(&dep_bar), 1);
    fence_mbar_init();
  }
  __syncthreads();

  float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(NS) * a.slot_bytes);

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      Ring ring(NS);
      int issued = 0;
      bool ok = true;
      for (int l = 0; l < a.n_layers && ok; ++l) {
        const StackLayerDev& L = a.layers[l];
        for (int k = 0; k < kOps && ok; ++k) {
          const OpPlanDev& p = a.plan[k];
          const int rcb = p.K / 2, rgb = p.K / 32;
          const int scales_off = p.MS * p.RS * rcb;
          const int biases_off = scales_off + p.MS * p.RS * rgb;
          const OpRows o = op_rows(p);
          for (int row = o.r0; row < o.r1;) {
            const int n = min(p.RS, o.r1 - row);
            if (!mbar_wait(smem_u32(&empty_bar[ring.slot]), ring.phase ^ 1u, &g_status)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&full_bar[ring.slot]);
            const uint32_t st = smem_u32(smem + static_cast<size_t>(ring.slot) * a.slot_bytes);
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(p.MS * n * (rcb + 2 * rgb)));
            for (int m = 0; m < p.MS; ++m) {
              const int wi = (k == 0) ? 0 : (k == 1) ? 1 : (k == 2) ? 2 + m : 4;
              bulk_g2s(st + m * p.RS * rcb, L.w[wi] + static_cast<long long>(row) * rcb, n * rcb,
                       fb, pol);
              bulk_g2s(st + scales_off + m * p.RS * rgb, L.s[wi] + static_cast<long long>(row) * (rgb / 2),
                       n * rgb, fb, pol);
              bulk_g2s(st + biases_off + m * p.RS * rgb, L.b[wi] + static_cast<long long>(row) * (rgb / 2),
                       n * rgb, fb, pol);
            }
            ++issued;
            ring.advance();
            row = next_row(o, row, n);
          }
        }
      }
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        mbar_wait(smem_u32(&full_bar[j % NS]), (j / NS) & 1, &g_status);
    }
    return;
  }

  // ------------------------------------------------------------ epilogue
  if (warp == 1) {
    Ring ring(NS);
    for (int l = 0; l < a.n_layers; ++l) {
      for (int k = 0; k < kOps; ++k) {
        const OpPlanDev& p = a.plan[k];
        const int dep = dependency(l, k);
        // Lane 0 acquires the producing op's completion (gpu scope), then
        // passes it on to this warp (__syncwarp) and to the consumer warps
        // (the dependency barrier's release/acquire).  On a timeout nothing
        // arrives and the consumers' own bounded wait ends them.
        int ok = 1;
        if (lane == 0 && dep >= 0) {
          ok = wait_counter(counter(a, dep), P);
          __threadfence();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&dep_bar));
        // RMS of the op's normalised input (ops 0 and 2).
        const float rstd = (k == 0)   ? warp_rstd(layer_input(a, l), a.H, a.eps, lane)
                           : (k == 2) ? warp_rstd(a.h, a.H, a.eps, lane)
                                      : 1.f;
        const int wpt = p.TG >> 5;
        const OpRows o = op_rows(p);
        __half* out = (k == 0) ? a.qkv
                      : (k == 1) ? a.h
                      : (k == 2) ? a.act
                                 : (l == a.n_layers - 1 ? a.y_out : a.xbuf[(l + 1) & 1]);
        const __half* resid = (k == 1) ? layer_input(a, l) : (k == 3) ? a.h : nullptr;
        // Residual rows of ops 1 and 3 (complete: their producer op was
        // acquired before), loaded all at once into shared memory so that the
        // per-stage work needs no global round trip.  Row index = stage * RS +
        // row in stage; rows past kResRows are read directly.
        if (resid != nullptr) {
          float rv[kResRows / 32];
#pragma unroll
          for (int i = 0; i < kResRows / 32; ++i) {
            const int idx = lane + 32 * i;
            const int g = idx / p.RS;
            const int gr = o.stride ? o.r0 + g * o.stride + (idx - g * p.RS) : o.r0 + idx;
            rv[i] = gr < o.r1 ? __half2float(resid[gr]) : 0.f;
          }
#pragma unroll
          for (int i = 0; i < kResRows / 32; ++i) res_sm[lane + 32 * i] = rv[i];
          __syncwarp();
        }
        int sidx = 0;  // stage * RS
        for (int row = o.r0; row < o.r1;) {
          const int n = min(p.RS, o.r1 - row);
          if (!mbar_wait(smem_u32(&part_bar[ring.slot]), ring.phase, &g_status)) return;
          const float* rs = red + static_cast<size_t>(ring.slot) * a.red_slot_floats;
          for (int r = lane; r < n; r += 32) {
            float v0 = 0.f, v1 = 0.f;
            for (int w = 0; w < wpt; ++w) v0 += rs[r * wpt + w];
            if (p.MS == 2)
              for (int w = 0; w < wpt; ++w) v1 += rs[(p.RS + r) * wpt + w];
            v0 *= kTwo24;
            v1 *= kTwo24;
            const int gr = row + r;
            float res;
            if (k == 0) {
              res = v0 * rstd;
            } else if (k == 2) {
              res = silu_f(v0 * rstd) * (v1 * rstd);
            } else {
              res = v0 + (sidx + r < kResRows ? res_sm[sidx + r] : __half2float(resid[gr]));
            }
            out[gr] = __float2half_rn(res);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty_bar[ring.slot]));
          ring.advance();
          row = next_row(o, row, n);
          sidx += p.RS;
        }
        // This CTA's rows of op (l, k) are written: publish.
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(counter(a, l * kOps + k), 1);
      }
    }
    return;
  }

  // ----------------------------------------------------------- consumers
  const int t = threadIdx.x - 64;
  Ring ring(NS);
  for (int l = 0; l < a.n_layers; ++l) {
    for (int k = 0; k < kOps; ++k) {
      const OpPlanDev& p = a.plan[k];
      // Input ready everywhere: the epilogue warp has acquired it.
      if (!mbar_wait(smem_u32(&dep_bar), static_cast<uint32_t>(l * kOps + k) & 1u, &g_status))
        return;
      if (!consume_op<kSliceK, kStackJR>(a, l, k, t, lane, ring, smem, red, full_bar, part_bar,
                                         empty_bar))
        return;
    }
  }
}

std::atomic<unsigned> g_attr_done{0};

}  // namespace
}  // namespace qgemv

extern "C" {

size_t qgemv_decode_stack_workspace_bytes(const qgemv_stack_shape* shape) {
  if (shape == nullptr || shape->n_layers < 1) return 0;
  auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  const size_t nqkv = static_cast<size_t>(shape->n_q + 2 * shape->n_kv) * shape->head_dim;
  return up(128 * 4 * static_cast<size_t>(shape->n_layers)) + up(2 * nqkv) +
         up(2 * static_cast<size_t>(shape->hidden)) + up(2 * static_cast<size_t>(shape->inter)) +
         2 * up(2 * static_cast<size_t>(shape->hidden));
}

int qgemv_decode_stack(const qgemv_stack_layer* layers, const qgemv_stack_shape* shape,
                       const uint16_t* x, uint16_t* y, void* workspace, size_t workspace_bytes,
                       void* stream) {
  using namespace qgemv;
  if (!layers || !shape || !x || !y || !workspace) return QGEMV_ENULL;
  const int H = shape->hidden, nq = shape->n_q, nkv = shape->n_kv, hd = shape->head_dim;
  const int I = shape->inter, NL = shape->n_layers;
  if (NL < 1 || NL > kMaxStackLayers || nq < 1 || nkv < 1 || nq % nkv != 0 || hd < 32 ||
      hd % 32 != 0 || !(shape->eps > 0.0f))
    return QGEMV_EINVAL;
  const int Dq = nq * hd;
  const int nqkv = (nq + 2 * nkv) * hd;
  for (int K : {H, Dq, I})
    if (K % 1024 != 0 || K / kSliceK > 512) return QGEMV_EINVAL;
  if (workspace_bytes < qgemv_decode_stack_workspace_bytes(shape)) return QGEMV_EINVAL;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(x) || !al16(y) || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return QGEMV_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return QGEMV_EDEVICE;

  StackArgs a{};
  for (int l = 0; l < NL; ++l) {
    const qgemv_stack_layer& s = layers[l];
    const uint32_t* w[5] = {s.qkv_codes, s.o_codes, s.gate_codes, s.up_codes, s.down_codes};
    const uint16_t* sc[5] = {s.qkv_scales, s.o_scales, s.gate_scales, s.up_scales, s.down_scales};
    const uint16_t* bi[5] = {s.qkv_biases, s.o_biases, s.gate_biases, s.up_biases, s.down_biases};
    for (int m = 0; m < 5; ++m) {
      if (!w[m] || !sc[m] || !bi[m]) return QGEMV_ENULL;
      if (!al16(w[m]) || !al16(sc[m]) || !al16(bi[m])) return QGEMV_EALIGN;
      a.layers[l].w[m] = reinterpret_cast<const uint8_t*>(w[m]);
      a.layers[l].s[m] = reinterpret_cast<const __half*>(sc[m]);
      a.layers[l].b[m] = reinterpret_cast<const __half*>(bi[m]);
    }
    if (!s.attn_norm || !s.mlp_norm) return QGEMV_ENULL;
    if (!al16(s.attn_norm) || !al16(s.mlp_norm)) return QGEMV_EALIGN;
    a.layers[l].g1 = reinterpret_cast<const __half*>(s.attn_norm);
    a.layers[l].g2 = reinterpret_cast<const __half*>(s.mlp_norm);
  }
  // Plans of the four ops (same for every layer), all with JR = 4.
  const int kinds[kOps] = {kNorm, kPlain, kSwiglu, kPlain};
  const int Ks[kOps] = {H, Dq, H, I};
  const int rows[kOps] = {nqkv, H, I, H};
  int slot_bytes = 0, red_floats = 0;
  for (int k = 0; k < kOps; ++k) {
    const StreamPlan p = make_stream_plan(kinds[k], 4, Ks[k], rows[k], 1, sms, 512, kStackJR);
    if (!p.ok || p.jr != kStackJR) return QGEMV_EINVAL;
    OpPlanDev& d = a.plan[k];
    d.K = Ks[k];
    d.rows = rows[k];
    d.TG = p.tg;
    d.S = p.s;
    d.RS = p.rs;
    d.MS = (k == 2) ? 2 : 1;
    d.stage_bytes = p.stage_bytes;
    d.interleave = p.interleave;
    slot_bytes = slot_bytes > p.stage_bytes ? slot_bytes : p.stage_bytes;
    const int rf = ((p.s * p.jr * (p.tg / 32)) + 3) & ~3;
    red_floats = red_floats > rf ? red_floats : rf;
  }
  int ns = (200 * 1024) / (slot_bytes + red_floats * 4);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return QGEMV_EINVAL;
  a.NS = ns;
  a.slot_bytes = slot_bytes;
  a.red_slot_floats = red_floats;
  const int smem = ns * (slot_bytes + red_floats * 4);

  // Workspace: counters, qkv, h, act, x ping-pong.
  auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  uint8_t* wp = static_cast<uint8_t*>(workspace);
  a.counters = reinterpret_cast<int*>(wp);
  wp += up(128 * 4 * static_cast<size_t>(NL));
  a.qkv = reinterpret_cast<__half*>(wp);
  wp += up(2 * static_cast<size_t>(nqkv));
  a.h = reinterpret_cast<__half*>(wp);
  wp += up(2 * static_cast<size_t>(H));
  a.act = reinterpret_cast<__half*>(wp);
  wp += up(2 * static_cast<size_t>(I));
  a.xbuf[0] = reinterpret_cast<__half*>(wp);
  wp += up(2 * static_cast<size_t>(H));
  a.xbuf[1] = reinterpret_cast<__half*>(wp);
  a.x_in = reinterpret_cast<const __half*>(x);
  a.y_out = reinterpret_cast<__half*>(y);
  a.n_layers = NL;
  a.H = H;
  a.n_q = nq;
  a.n_kv = nkv;
  a.hd = hd;
  a.I = I;
  a.eps = shape->eps;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* kern = stack_kernel;
  if (dev < 32 && !((g_attr_done.load(std::memory_order_acquire) >> dev) & 1u)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024) !=
        cudaSuccess)
      return QGEMV_ELAUNCH;
    g_attr_done.fetch_or(1u << dev, std::memory_order_acq_rel);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 576, smem) != cudaSuccess ||
      per_sm < 1)
    return QGEMV_ELAUNCH;
  if (cudaMemsetAsync(a.counters, 0, 128 * 4 * static_cast<size_t>(NL), st) != cudaSuccess)
    return QGEMV_ELAUNCH;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms));
  cfg.blockDim = dim3(576);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return QGEMV_ELAUNCH;
  return QGEMV_OK;
}

}  // extern "C"

namespace qgemv {
cudaError_t status_stack(unsigned* out) { return read_clear_status(out); }
}  // namespace qgemv
