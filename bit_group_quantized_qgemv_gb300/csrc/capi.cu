// capi.cu -- the extern "C" boundary of libqgemv.so (declared in
// include/qgemv.h).  Host code only: validates arguments, picks the
// streaming kernel or the generic kernel, and launches on the caller's
// stream.  Never allocates, frees or synchronises (except the diagnostic
// qgemv_device_status).
#include <stdint.h>

#include <atomic>
#include <cmath>

#include "qgemv.h"
#include "qgemv_args.h"
#include "epilogue_ops.h"

static_assert(QGEMV_SAMPLE_MAX_K == qgemv::kMaxSampleK, "sampler candidate limit");
static_assert(QGEMV_SAMPLE_MAX_N == qgemv::kMaxSampleN, "sampler logits limit");

namespace {

using qgemv::StreamArgs;
using qgemv::StreamPlan;

thread_local int t_last_cuda_error = 0;

// Multiprocessor count per device, read once.
std::atomic<int> g_sms[64];

int current_device(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return QGEMV_EDEVICE;
  if (*dev < 0 || *dev >= 64) return QGEMV_EDEVICE;
  int v = g_sms[*dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess || v <= 0)
      return QGEMV_EDEVICE;
    g_sms[*dev].store(v, std::memory_order_relaxed);
  }
  *sms = v;
  return QGEMV_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int finish(cudaError_t e) {
  if (e == cudaSuccess) return QGEMV_OK;
  t_last_cuda_error = static_cast<int>(e);
  return QGEMV_ELAUNCH;
}

bool valid_k(int K) { return K >= 64 && K % 64 == 0; }

int check_sample(const uint16_t* logits, int N, int top_k, float temperature, const float* u,
                 const int32_t* token, const int32_t* topk_idx, const float* topk_prob) {
  if (!logits || !u || !token) return QGEMV_ENULL;
  if (N < 1 || N > QGEMV_SAMPLE_MAX_N || top_k < 1 || top_k > QGEMV_SAMPLE_MAX_K || top_k > N)
    return QGEMV_EINVAL;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return QGEMV_EINVAL;
  if (!aligned(logits, 2) || !aligned(u, 4) || !aligned(token, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_prob, 4))
    return QGEMV_EALIGN;
  return QGEMV_OK;
}

int moe_impl(const uint32_t* gu_codes, const uint16_t* gu_scales, const uint16_t* gu_biases,
             const uint32_t* dn_codes, const uint16_t* dn_scales, const uint16_t* dn_biases,
             int n_experts, int H, int I, const int32_t* expert_idx, const float* expert_w,
             int top_k, const uint16_t* x, const uint16_t* residual, uint16_t* y,
             float* workspace, int* err_flag, uint32_t* trace, int trace_ctas,
             int* ctas_launched, void* stream);

// One activation row (the last pass of an odd batch): the M = 1 streaming
// kernel when it takes the shape, else the generic kernel.
cudaError_t launch_single_row(int bits, const StreamArgs& a, int sms, cudaStream_t st, int dev) {
  const StreamPlan p = qgemv::make_stream_plan(qgemv::kPlain, bits, a.K, a.rows, 1, sms);
  if (p.ok) return qgemv::stream_plain(bits, p, a, st, dev);
  return qgemv::generic_launch(qgemv::kPlain, bits, a, st);
}

StreamArgs blank_args() {
  StreamArgs a{};
  a.M = 1;
  a.top_k = 1;
  return a;
}

// Which kernels a qgemv_w4g64 / w2g64 / w8g64 call of this shape takes
// (plain_impl follows it; qgemv_plan_gemv reports it).  al16: codes, scales,
// biases and x 16-byte aligned; mma: the tensor-core kernel may be tried.
qgemv_gemv_plan route_plain(int bits, int M, long long N, int K, int sms, bool al16, bool mma) {
  qgemv_gemv_plan r{};
  r.path = QGEMV_PATH_GENERIC;
  r.passes = 1;
  r.cluster = 1;
  if (M == 1) {
    const StreamPlan p = qgemv::make_stream_plan(qgemv::kPlain, bits, K, N, 1, sms);
    if (p.ok && al16) {
      r.path = QGEMV_PATH_STREAM;
      r.stages = p.ns;
      r.smem_bytes = p.smem_bytes;
    }
    return r;
  }
  // Small batch on the tensor cores (M >= 3, and M = 2 on short ops): one
  // pass holding all M rows when their activations fit in shared memory,
  // else passes of at most 4 rows (a pass of 1 or 2 rows takes the
  // CUDA-core kernels).
  int mp = 0, smem = 0, ns = 0, cl = 1, kc = 0;
  if (al16 && mma && qgemv::batch_mma_plan(bits, K, N, M, sms, &mp, &smem, &ns, &cl, &kc)) {
    r.path = QGEMV_PATH_MMA;
  } else if (al16 && mma && M > 4 &&
             qgemv::batch_mma_plan(bits, K, N, 4, sms, &mp, &smem, &ns, &cl, &kc)) {
    r.path = QGEMV_PATH_MMA_PASSES;
    r.passes = (M + 3) / 4;
  }
  if (r.path != QGEMV_PATH_GENERIC) {
    r.m_pad = mp;
    r.cluster = cl;
    r.chunk_k = kc;
    r.stages = ns;
    r.smem_bytes = smem;
    return r;
  }
  // CUDA-core small-batch kernel, then the generic kernel.
  const StreamPlan p = qgemv::make_batch_plan(bits, K, N, M, sms);
  const StreamPlan p4 = qgemv::make_batch_plan(bits, K, N, 4, sms);
  if (al16 && p.ok) {
    r.path = QGEMV_PATH_BATCH;
    r.stages = p.ns;
    r.smem_bytes = p.smem_bytes;
  } else if (al16 && p4.ok) {
    r.path = QGEMV_PATH_BATCH_PASSES;
    r.passes = (M + 3) / 4;
    r.stages = p4.ns;
    r.smem_bytes = p4.smem_bytes;
  }
  return r;
}

int plain_impl(int bits, const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
               const uint16_t* x, uint16_t* y, int M, int N, int K, const uint16_t* residual,
               void* stream) {
  if (!codes || !scales || !biases || !x || !y) return QGEMV_ENULL;
  if (M < 1 || M > QGEMV_MAX_M || N < 1 || !valid_k(K)) return QGEMV_EINVAL;
  if (!aligned(codes, 4) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(x, 2) ||
      !aligned(y, 2) || !aligned(residual, 2))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  StreamArgs a = blank_args();
  a.codes[0] = reinterpret_cast<const uint8_t*>(codes);
  a.scales[0] = reinterpret_cast<const __half*>(scales);
  a.biases[0] = reinterpret_cast<const __half*>(biases);
  a.x = reinterpret_cast<const __half*>(x);
  a.y = reinterpret_cast<__half*>(y);
  a.residual = reinterpret_cast<const __half*>(residual);
  a.rows = N;
  a.K = K;
  a.M = M;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool al16 = aligned(codes, 16) && aligned(scales, 16) && aligned(biases, 16) &&
                    aligned(x, 16);
  qgemv_gemv_plan r = route_plain(bits, M, N, K, sms, al16, true);
  if (r.path == QGEMV_PATH_MMA) {
    const cudaError_t e = qgemv::stream_batch_mma(bits, a, sms, st, dev);
    // cudaErrorNotSupported: the device cannot host the plan's clusters (a
    // restricted SM partition, say); nothing was launched, so the CUDA-core
    // kernels take the call.
    if (e != cudaErrorNotSupported) return finish(e);
    cudaGetLastError();
    r = route_plain(bits, M, N, K, sms, al16, false);
  }
  auto pass = [&](int m0) {
    StreamArgs ap = a;
    ap.M = M - m0 < 4 ? M - m0 : 4;
    ap.x = a.x + static_cast<size_t>(m0) * K;
    ap.y = a.y + static_cast<size_t>(m0) * N;
    if (a.residual) ap.residual = a.residual + static_cast<size_t>(m0) * N;
    return ap;
  };
  switch (r.path) {
    case QGEMV_PATH_STREAM:
      return finish(qgemv::stream_plain(
          bits, qgemv::make_stream_plan(qgemv::kPlain, bits, K, N, 1, sms), a, st, dev));
    case QGEMV_PATH_MMA_PASSES:
      for (int m0 = 0; m0 < M; m0 += 4) {
        const StreamArgs ap = pass(m0);
        cudaError_t e;
        if (ap.M >= 3) {
          e = qgemv::stream_batch_mma(bits, ap, sms, st, dev);
        } else if (ap.M == 2) {
          const StreamPlan pm = qgemv::make_batch_plan(bits, K, N, 2, sms);
          e = pm.ok ? qgemv::stream_batch(bits, pm, ap, st, dev)
                    : qgemv::generic_launch(qgemv::kPlain, bits, ap, st);
        } else {
          e = launch_single_row(bits, ap, sms, st, dev);
        }
        if (e != cudaSuccess) return finish(e);
      }
      return QGEMV_OK;
    case QGEMV_PATH_BATCH:
      return finish(
          qgemv::stream_batch(bits, qgemv::make_batch_plan(bits, K, N, M, sms), a, st, dev));
    case QGEMV_PATH_BATCH_PASSES:
      for (int m0 = 0; m0 < M; m0 += 4) {
        const StreamArgs ap = pass(m0);
        const StreamPlan pp = qgemv::make_batch_plan(bits, K, N, ap.M < 2 ? 2 : ap.M, sms);
        const cudaError_t e = qgemv::stream_batch(bits, pp, ap, st, dev);
        if (e != cudaSuccess) return finish(e);
      }
      return QGEMV_OK;
    default:
      return finish(qgemv::generic_launch(qgemv::kPlain, bits, a, st));
  }
}

}  // namespace

extern "C" {

int qgemv_w4g64(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                const uint16_t* x, uint16_t* y, int M, int N, int K, const uint16_t* residual,
                void* stream) {
  return plain_impl(4, codes, scales, biases, x, y, M, N, K, residual, stream);
}

int qgemv_w2g64(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                const uint16_t* x, uint16_t* y, int M, int N, int K, const uint16_t* residual,
                void* stream) {
  return plain_impl(2, codes, scales, biases, x, y, M, N, K, residual, stream);
}

int qgemv_w8g64(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                const uint16_t* x, uint16_t* y, int M, int N, int K, const uint16_t* residual,
                void* stream) {
  return plain_impl(8, codes, scales, biases, x, y, M, N, K, residual, stream);
}

int rmsnorm_qgemv(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                  const uint16_t* x, const uint16_t* norm_weight, float eps, uint16_t* y, int N,
                  int K, void* stream) {
  if (!codes || !scales || !biases || !x || !norm_weight || !y) return QGEMV_ENULL;
  if (N < 1 || !valid_k(K) || !(eps > 0.0f) || eps > 1e30f) return QGEMV_EINVAL;
  if (!aligned(codes, 4) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(x, 2) ||
      !aligned(norm_weight, 2) || !aligned(y, 2))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  StreamArgs a = blank_args();
  a.codes[0] = reinterpret_cast<const uint8_t*>(codes);
  a.scales[0] = reinterpret_cast<const __half*>(scales);
  a.biases[0] = reinterpret_cast<const __half*>(biases);
  a.x = reinterpret_cast<const __half*>(x);
  a.gamma = reinterpret_cast<const __half*>(norm_weight);
  a.eps = eps;
  a.y = reinterpret_cast<__half*>(y);
  a.rows = N;
  a.K = K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const StreamPlan p = qgemv::make_stream_plan(qgemv::kNorm, 4, K, N, 1, sms);
  if (p.ok && aligned(codes, 16) && aligned(scales, 16) && aligned(biases, 16) &&
      aligned(x, 16) && aligned(norm_weight, 16))
    return finish(qgemv::stream_norm(p, a, st, dev));
  return finish(qgemv::generic_launch(qgemv::kNorm, 4, a, st));
}

int swiglu_qgemv(const uint32_t* gate_codes, const uint16_t* gate_scales,
                 const uint16_t* gate_biases, const uint32_t* up_codes, const uint16_t* up_scales,
                 const uint16_t* up_biases, const uint16_t* x, const uint16_t* norm_weight,
                 float eps, uint16_t* h, int I, int K, void* stream) {
  if (!gate_codes || !gate_scales || !gate_biases || !up_codes || !up_scales || !up_biases ||
      !x || !h)
    return QGEMV_ENULL;
  if (I < 1 || !valid_k(K)) return QGEMV_EINVAL;
  if (norm_weight && (!(eps > 0.0f) || eps > 1e30f)) return QGEMV_EINVAL;
  if (!aligned(gate_codes, 4) || !aligned(up_codes, 4) || !aligned(gate_scales, 2) ||
      !aligned(gate_biases, 2) || !aligned(up_scales, 2) || !aligned(up_biases, 2) ||
      !aligned(x, 2) || !aligned(norm_weight, 2) || !aligned(h, 2))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  StreamArgs a = blank_args();
  a.codes[0] = reinterpret_cast<const uint8_t*>(gate_codes);
  a.scales[0] = reinterpret_cast<const __half*>(gate_scales);
  a.biases[0] = reinterpret_cast<const __half*>(gate_biases);
  a.codes[1] = reinterpret_cast<const uint8_t*>(up_codes);
  a.scales[1] = reinterpret_cast<const __half*>(up_scales);
  a.biases[1] = reinterpret_cast<const __half*>(up_biases);
  a.x = reinterpret_cast<const __half*>(x);
  a.gamma = reinterpret_cast<const __half*>(norm_weight);
  a.eps = eps;
  a.y = reinterpret_cast<__half*>(h);
  a.rows = I;
  a.K = K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const StreamPlan p = qgemv::make_stream_plan(qgemv::kSwiglu, 4, K, I, 1, sms);
  if (p.ok && aligned(gate_codes, 16) && aligned(gate_scales, 16) && aligned(gate_biases, 16) &&
      aligned(up_codes, 16) && aligned(up_scales, 16) && aligned(up_biases, 16) &&
      aligned(x, 16) && (norm_weight == nullptr || aligned(norm_weight, 16)))
    return finish(qgemv::stream_swiglu(p, a, st, dev));
  return finish(qgemv::generic_launch(qgemv::kSwiglu, 4, a, st));
}

size_t qgemv_moe_workspace_bytes(int top_k, int I) {
  if (top_k < 1 || I < 1) return 0;
  return static_cast<size_t>(top_k) * static_cast<size_t>(I) * sizeof(float);
}

int moe_qgemv_combine(const uint32_t* gu_codes, const uint16_t* gu_scales,
                      const uint16_t* gu_biases, const uint32_t* dn_codes,
                      const uint16_t* dn_scales, const uint16_t* dn_biases, int n_experts, int H,
                      int I, const int32_t* expert_idx, const float* expert_w, int top_k,
                      const uint16_t* x, const uint16_t* residual, uint16_t* y, float* workspace,
                      int* err_flag, void* stream) {
  return moe_impl(gu_codes, gu_scales, gu_biases, dn_codes, dn_scales, dn_biases, n_experts, H, I,
                  expert_idx, expert_w, top_k, x, residual, y, workspace, err_flag, nullptr, 0,
                  nullptr, stream);
}

int moe_qgemv_combine_traced(const uint32_t* gu_codes, const uint16_t* gu_scales,
                             const uint16_t* gu_biases, const uint32_t* dn_codes,
                             const uint16_t* dn_scales, const uint16_t* dn_biases, int n_experts,
                             int H, int I, const int32_t* expert_idx, const float* expert_w,
                             int top_k, const uint16_t* x, const uint16_t* residual, uint16_t* y,
                             float* workspace, int* err_flag, uint32_t* trace, int trace_ctas,
                             int* ctas_launched, void* stream) {
  if (!trace || !ctas_launched) return QGEMV_ENULL;
  if (trace_ctas < 1) return QGEMV_EINVAL;
  if (!aligned(trace, 16)) return QGEMV_EALIGN;
  return moe_impl(gu_codes, gu_scales, gu_biases, dn_codes, dn_scales, dn_biases, n_experts, H, I,
                  expert_idx, expert_w, top_k, x, residual, y, workspace, err_flag, trace,
                  trace_ctas, ctas_launched, stream);
}

}  // extern "C"

namespace {

int moe_impl(const uint32_t* gu_codes, const uint16_t* gu_scales, const uint16_t* gu_biases,
             const uint32_t* dn_codes, const uint16_t* dn_scales, const uint16_t* dn_biases,
             int n_experts, int H, int I, const int32_t* expert_idx, const float* expert_w,
             int top_k, const uint16_t* x, const uint16_t* residual, uint16_t* y,
             float* workspace, int* err_flag, uint32_t* trace, int trace_ctas,
             int* ctas_launched, void* stream) {
  if (!gu_codes || !gu_scales || !gu_biases || !dn_codes || !dn_scales || !dn_biases ||
      !expert_idx || !expert_w || !x || !y || !workspace)
    return QGEMV_ENULL;
  if (n_experts < 1 || top_k < 1 || top_k > QGEMV_MAX_TOPK || !valid_k(H) || !valid_k(I))
    return QGEMV_EINVAL;
  if (!aligned(gu_codes, 4) || !aligned(dn_codes, 4) || !aligned(gu_scales, 2) ||
      !aligned(gu_biases, 2) || !aligned(dn_scales, 2) || !aligned(dn_biases, 2) ||
      !aligned(expert_idx, 4) || !aligned(expert_w, 4) || !aligned(x, 2) ||
      !aligned(residual, 2) || !aligned(y, 2) || !aligned(workspace, 4) || !aligned(err_flag, 4))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long gu_row_bytes = static_cast<long long>(H) / 2;  // 4-bit: H/8 words * 4 B
  const long long dn_row_bytes = static_cast<long long>(I) / 2;

  // Phase 1: h_k = silu(Wg[e_k] x) * (Wu[e_k] x) into the workspace.
  StreamArgs u = blank_args();
  u.codes[0] = reinterpret_cast<const uint8_t*>(gu_codes);
  u.codes[1] = reinterpret_cast<const uint8_t*>(gu_codes) + static_cast<long long>(I) * gu_row_bytes;
  u.scales[0] = reinterpret_cast<const __half*>(gu_scales);
  u.scales[1] = reinterpret_cast<const __half*>(gu_scales) + static_cast<long long>(I) * (H / 64);
  u.biases[0] = reinterpret_cast<const __half*>(gu_biases);
  u.biases[1] = reinterpret_cast<const __half*>(gu_biases) + static_cast<long long>(I) * (H / 64);
  u.ex_code_bytes = 2LL * I * gu_row_bytes;
  u.ex_groups = 2LL * I * (H / 64);
  u.x = reinterpret_cast<const __half*>(x);
  u.yf = workspace;
  u.idx = expert_idx;
  u.wt = expert_w;
  u.err_flag = err_flag;
  u.top_k = top_k;
  u.n_experts = n_experts;
  u.rows = static_cast<long long>(top_k) * I;
  u.rows_per_expert = I;
  u.K = H;
  u.trace = trace;
  u.trace_ctas = trace_ctas;
  const StreamPlan pu = qgemv::make_stream_plan(qgemv::kMoeUp, 4, H, u.rows, top_k, sms);
  cudaError_t e;
  if (pu.ok && aligned(gu_codes, 16) && aligned(gu_scales, 16) && aligned(gu_biases, 16) &&
      aligned(x, 16)) {
    if (ctas_launched) ctas_launched[0] = pu.grid;
    e = qgemv::stream_moe_up(pu, u, st, dev);
  } else {
    if (ctas_launched) ctas_launched[0] = qgemv::generic_blocks(u);
    e = qgemv::generic_launch(qgemv::kMoeUp, 4, u, st);
  }
  if (e != cudaSuccess) return finish(e);

  // Phase 2: y = r + sum_k wt_k Wd[e_k] h_k.
  StreamArgs d = blank_args();
  d.codes[0] = reinterpret_cast<const uint8_t*>(dn_codes);
  d.scales[0] = reinterpret_cast<const __half*>(dn_scales);
  d.biases[0] = reinterpret_cast<const __half*>(dn_biases);
  d.ex_code_bytes = static_cast<long long>(H) * dn_row_bytes;
  d.ex_groups = static_cast<long long>(H) * (I / 64);
  d.xf = workspace;
  d.residual = reinterpret_cast<const __half*>(residual);
  d.y = reinterpret_cast<__half*>(y);
  d.idx = expert_idx;
  d.wt = expert_w;
  d.err_flag = err_flag;
  d.top_k = top_k;
  d.n_experts = n_experts;
  d.rows = H;
  d.K = I;
  // the down phase's records follow the up phase's
  d.trace = trace ? trace + static_cast<size_t>(trace_ctas) * top_k * 4 : nullptr;
  d.trace_ctas = trace_ctas;
  const StreamPlan pd = qgemv::make_stream_plan(qgemv::kMoeDown, 4, I, H, top_k, sms);
  if (pd.ok && aligned(dn_codes, 16) && aligned(dn_scales, 16) && aligned(dn_biases, 16) &&
      aligned(workspace, 16)) {
    if (ctas_launched) ctas_launched[1] = pd.grid;
    e = qgemv::stream_moe_down(pd, d, st, dev);
  } else {
    if (ctas_launched) ctas_launched[1] = qgemv::generic_blocks(d);
    e = qgemv::generic_launch(qgemv::kMoeDown, 4, d, st);
  }
  return finish(e);
}

}  // namespace

extern "C" {

int decode_attention_seq1(const uint16_t* qkv, uint16_t* out, int n_q, int n_kv, int head_dim,
                          void* stream) {
  if (!qkv || !out) return QGEMV_ENULL;
  if (n_q < 1 || n_kv < 1 || head_dim < 1 || n_q % n_kv != 0) return QGEMV_EINVAL;
  if (!aligned(qkv, 2) || !aligned(out, 2)) return QGEMV_EALIGN;
  return finish(qgemv::attention_seq1_launch(reinterpret_cast<const __half*>(qkv),
                                             reinterpret_cast<__half*>(out), n_q, n_kv, head_dim,
                                             static_cast<cudaStream_t>(stream)));
}

const char* qgemv_strerror(int status) {
  switch (status) {
    case QGEMV_OK: return "ok";
    case QGEMV_EINVAL: return "invalid shape or scalar argument";
    case QGEMV_ENULL: return "required pointer is NULL";
    case QGEMV_EALIGN: return "pointer misaligned (codes need 4 bytes, fp16 2 bytes)";
    case QGEMV_ELAUNCH: return "CUDA reported an error at kernel launch";
    case QGEMV_EDEVICE: return "no usable CUDA device";
    case QGEMV_ESCRATCH: return "top_k * I exceeds the allocation-free scratch array";
    default: return "unknown status";
  }
}

int qgemv_last_cuda_error(void) { return t_last_cuda_error; }

int qgemv_device_status(unsigned* flags) {
  if (!flags) return QGEMV_ENULL;
  *flags = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return QGEMV_EDEVICE;
  unsigned v = 0;
  if (qgemv::status_plain(&v) != cudaSuccess || qgemv::status_norm_swiglu(&v) != cudaSuccess ||
      qgemv::status_moe(&v) != cudaSuccess || qgemv::status_generic(&v) != cudaSuccess ||
      qgemv::status_batch(&v) != cudaSuccess)
    return QGEMV_EDEVICE;
  *flags = v;
  return QGEMV_OK;
}

int qgemv_moe_router(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                     const uint16_t* x, int E, int H, int top_k, int shared_expert,
                     uint16_t* logits, int32_t* expert_idx, float* expert_w, void* stream) {
  if (!codes || !scales || !biases || !x || !logits || !expert_idx || !expert_w)
    return QGEMV_ENULL;
  if (E < 1 || top_k < 1 || top_k > qgemv::kMaxTopK || top_k > E || shared_expert < -1 ||
      shared_expert >= E || !valid_k(H))
    return QGEMV_EINVAL;
  if (!aligned(expert_idx, 4) || !aligned(expert_w, 4)) return QGEMV_EALIGN;
  const int rc = plain_impl(4, codes, scales, biases, x, logits, 1, E, H, nullptr, stream);
  if (rc != QGEMV_OK) return rc;
  return finish(qgemv::moe_route_launch(reinterpret_cast<const __half*>(logits), E, top_k,
                                        shared_expert, expert_idx, expert_w,
                                        static_cast<cudaStream_t>(stream)));
}

int qgemv_residual_rmsnorm(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma,
                           float eps, int K, uint16_t* h, uint16_t* xn, void* stream) {
  if (!x || !gamma || !xn || (residual && !h)) return QGEMV_ENULL;
  if (K < 1 || !(eps > 0.0f)) return QGEMV_EINVAL;
  if (!aligned(x, 2) || !aligned(residual, 2) || !aligned(gamma, 2) || !aligned(h, 2) ||
      !aligned(xn, 2))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  return finish(qgemv::residual_rmsnorm_launch(
      reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(residual),
      reinterpret_cast<const __half*>(gamma), eps, K, reinterpret_cast<__half*>(h),
      reinterpret_cast<__half*>(xn), static_cast<cudaStream_t>(stream)));
}

size_t qgemv_argmax_scratch_bytes(void) { return 16; }

int qgemv_lm_head_argmax(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                         const uint16_t* x, uint16_t* logits, int N, int K, void* scratch,
                         int32_t* token, void* stream) {
  if (!codes || !scales || !biases || !x || !logits || !scratch || !token) return QGEMV_ENULL;
  if (N < 1 || !valid_k(K)) return QGEMV_EINVAL;
  if (!aligned(codes, 4) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(x, 2) ||
      !aligned(logits, 2) || !aligned(scratch, 8) || !aligned(token, 4))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  StreamArgs a = blank_args();
  a.codes[0] = reinterpret_cast<const uint8_t*>(codes);
  a.scales[0] = reinterpret_cast<const __half*>(scales);
  a.biases[0] = reinterpret_cast<const __half*>(biases);
  a.x = reinterpret_cast<const __half*>(x);
  a.y = reinterpret_cast<__half*>(logits);
  a.rows = N;
  a.K = K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const StreamPlan p = qgemv::make_stream_plan(qgemv::kPlain, 4, K, N, 1, sms);
  if (p.ok && aligned(codes, 16) && aligned(scales, 16) && aligned(biases, 16) &&
      aligned(x, 16)) {
    a.am_key = static_cast<unsigned long long*>(scratch);
    const cudaError_t e = qgemv::stream_argmax(p, a, st, dev);
    if (e != cudaSuccess) return finish(e);
    return finish(qgemv::argmax_finalize_launch(a.am_key, token, st));
  }
  // Other shapes: the generic GEMV, then a one-CTA argmax over the logits.
  const cudaError_t e = qgemv::generic_launch(qgemv::kPlain, 4, a, st);
  if (e != cudaSuccess) return finish(e);
  return finish(qgemv::argmax_launch(a.y, N, token, st));
}

int qgemv_sample_topk(const uint16_t* logits, int N, int top_k, float temperature,
                      const float* u, int32_t* token, int32_t* topk_idx, float* topk_prob,
                      void* stream) {
  if (int rc = check_sample(logits, N, top_k, temperature, u, token, topk_idx, topk_prob)) return rc;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  return finish(qgemv::sample_topk_launch(reinterpret_cast<const __half*>(logits), N, top_k,
                                          temperature, u, token, topk_idx, topk_prob,
                                          static_cast<cudaStream_t>(stream)));
}

int qgemv_lm_head_sample(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                         const uint16_t* x, uint16_t* logits, int N, int K, int top_k,
                         float temperature, const float* u, int32_t* token, int32_t* topk_idx,
                         float* topk_prob, void* stream) {
  if (!codes || !scales || !biases || !x) return QGEMV_ENULL;
  if (int rc = check_sample(logits, N, top_k, temperature, u, token, topk_idx, topk_prob)) return rc;
  if (!valid_k(K)) return QGEMV_EINVAL;
  if (!aligned(codes, 4) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(x, 2))
    return QGEMV_EALIGN;
  if (int rc = plain_impl(4, codes, scales, biases, x, logits, 1, N, K, nullptr, stream)) return rc;
  return finish(qgemv::sample_topk_launch(reinterpret_cast<const __half*>(logits), N, top_k,
                                          temperature, u, token, topk_idx, topk_prob,
                                          static_cast<cudaStream_t>(stream)));
}

int qgemv_plan_gemv(int bits, int M, int N, int K, int sms, int aligned16, qgemv_gemv_plan* out) {
  if (!out) return QGEMV_ENULL;
  if ((bits != 2 && bits != 4 && bits != 8) || M < 1 || M > QGEMV_MAX_M || N < 1 ||
      !valid_k(K) || sms < 1)
    return QGEMV_EINVAL;
  *out = route_plain(bits, M, N, K, sms, aligned16 != 0, true);
  return QGEMV_OK;
}

int qgemv_lut4(const uint32_t* codes, const uint16_t* lut, int n_luts, int rows_per_lut,
               const uint16_t* x, uint16_t* y, int N, int K, const uint16_t* residual,
               void* stream) {
  if (!codes || !lut || !x || !y) return QGEMV_ENULL;
  if (N < 1 || !valid_k(K) || K > QGEMV_LUT_MAX_K || rows_per_lut < 1 || n_luts < 1)
    return QGEMV_EINVAL;
  if (static_cast<long long>(n_luts) * rows_per_lut < N) return QGEMV_EINVAL;
  if (!aligned(codes, 16) || !aligned(lut, 16) || !aligned(x, 16) || !aligned(y, 2) ||
      !aligned(residual, 2))
    return QGEMV_EALIGN;
  int dev, sms;
  if (int rc = current_device(&dev, &sms)) return rc;
  return finish(qgemv::lut_qgemv_launch(codes, lut, rows_per_lut,
                                        reinterpret_cast<const __half*>(x),
                                        reinterpret_cast<const __half*>(residual),
                                        reinterpret_cast<__half*>(y), N, K, sms,
                                        static_cast<cudaStream_t>(stream)));
}

int qgemv_selftest_wait_timeout(unsigned limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return QGEMV_EINVAL;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  return finish(qgemv::selftest_wait_launch(static_cast<uint64_t>(limit_us) * 1000ull,
                                            static_cast<cudaStream_t>(stream)));
}

int qgemv_version(void) { return 100; }

}  // extern "C"
