// stack.cu -- qgemv_decode_stack: one decode token through a stack of
// pre-norm transformer layers' quantized matvecs.
//
// Per layer l (INFERENCE_RESEARCH.md section 1: one command buffer encoding
// the whole layer stack, fused kernels, no per-token overhead):
//   op 0  qkv  = W_qkv . (x_l * gamma1) * rstd(x_l)          (RMSNorm fused)
//   op 1  h    = x_l + W_o . attn,  attn = value heads of qkv (decode over
//                one cached position: softmax of one score is 1), read by
//                the o_proj kernel straight from qkv (no copy)
//   op 2  act  = silu(W_g . x~) * (W_u . x~),  x~ = h * gamma2 * rstd(h)
//   op 3  x_{l+1} = h + W_d . act
//
// The 4 * n_layers ops are enqueued as streaming-kernel launches with
// programmatic dependent launch: each kernel lets its successor start as its
// own CTAs exit, so the successor's producer warps stream their weights
// (which no op writes) while the last CTAs of the previous op finish, and
// only its consumer and epilogue warps wait (griddepcontrol.wait) for the
// previous grid's output.  On GB300 this chain measured faster than one
// cooperative persistent kernel synchronising its CTAs through completion
// counters in global memory (1254 us against 1370 us per 32-layer token):
// the hardware's grid dependency resolves sooner than a fence, an atomic and
// a polled counter.  The launches themselves go through a CUDA-graph cache
// (below): eager launches cost more host time than the GPU needs for them.
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "qgemv.h"
#include "qgemv_args.h"

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t up256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// The 4 * n_layers launches of one call.  Arguments already validated.
int enqueue_stack(const qgemv_stack_layer* layers, const qgemv_stack_shape* shape,
                  const uint16_t* x, uint16_t* y, void* workspace, int dev, int sms,
                  cudaStream_t st);

// CUDA-graph cache of the decode stack.  A call enqueues 4 * n_layers
// kernels; issued eagerly and back to back, a 32-layer call on a GB300 node
// held its host thread for ~1050 us (as long as the GPU work, ~1075 us), so
// the host could not run ahead.  Each distinct argument set (device, shape,
// every pointer) is therefore captured once into a graph whose instance
// later calls replay with one cudaGraphLaunch (~9 us of host time per call
// back to back, ~18 us into an idle stream).  The kernels and their
// programmatic dependencies are the same either way.
constexpr int kGraphCacheSize = 4;

struct GraphEntry {
  std::vector<uintptr_t> key;
  cudaGraphExec_t exec = nullptr;
  unsigned long long last_use = 0;
};

std::mutex g_graph_mu;
GraphEntry g_graphs[kGraphCacheSize];
unsigned long long g_graph_clock = 0;
cudaStream_t g_capture_stream[64] = {};

std::vector<uintptr_t> graph_key(const qgemv_stack_layer* layers, const qgemv_stack_shape* shape,
                                 const uint16_t* x, const uint16_t* y, const void* workspace,
                                 int dev) {
  std::vector<uintptr_t> k;
  const int NL = shape->n_layers;
  k.reserve(12 + static_cast<size_t>(NL) * (sizeof(qgemv_stack_layer) / sizeof(uintptr_t) + 1));
  uint32_t eps_bits;
  memcpy(&eps_bits, &shape->eps, sizeof(eps_bits));
  const uintptr_t head[] = {static_cast<uintptr_t>(dev),          static_cast<uintptr_t>(shape->hidden),
                            static_cast<uintptr_t>(shape->n_q),   static_cast<uintptr_t>(shape->n_kv),
                            static_cast<uintptr_t>(shape->head_dim), static_cast<uintptr_t>(shape->inter),
                            static_cast<uintptr_t>(NL),           eps_bits,
                            reinterpret_cast<uintptr_t>(x),       reinterpret_cast<uintptr_t>(y),
                            reinterpret_cast<uintptr_t>(workspace)};
  k.insert(k.end(), head, head + sizeof(head) / sizeof(head[0]));
  for (int l = 0; l < NL; ++l) {
    const qgemv_stack_layer& s = layers[l];
    const void* p[17] = {s.qkv_codes,   s.qkv_scales,  s.qkv_biases,  s.attn_norm,  s.o_codes,
                         s.o_scales,    s.o_biases,    s.gate_codes,  s.gate_scales,
                         s.gate_biases, s.up_codes,    s.up_scales,   s.up_biases,  s.mlp_norm,
                         s.down_codes,  s.down_scales, s.down_biases};
    for (const void* q : p) k.push_back(reinterpret_cast<uintptr_t>(q));
  }
  return k;
}

// Capture the call's launches into a graph instance (nullptr on failure;
// the caller then launches eagerly).
cudaGraphExec_t capture_stack(const qgemv_stack_layer* layers, const qgemv_stack_shape* shape,
                              const uint16_t* x, uint16_t* y, void* workspace, int dev, int sms) {
  if (dev < 0 || dev >= 64) return nullptr;
  if (g_capture_stream[dev] == nullptr &&
      cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
    g_capture_stream[dev] = nullptr;
    cudaGetLastError();
    return nullptr;
  }
  cudaStream_t cap = g_capture_stream[dev];
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  const int rc = enqueue_stack(layers, shape, x, y, workspace, dev, sms, cap);
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cap, &graph);
  cudaGraphExec_t exec = nullptr;
  if (rc == QGEMV_OK && e == cudaSuccess && graph != nullptr &&
      cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
    exec = nullptr;
  if (graph != nullptr) cudaGraphDestroy(graph);
  cudaGetLastError();  // a failed capture leaves no sticky error behind
  return exec;
}

}  // namespace

extern "C" {

size_t qgemv_decode_stack_workspace_bytes(const qgemv_stack_shape* shape) {
  if (shape == nullptr || shape->n_layers < 1 || shape->hidden < 1 || shape->inter < 1 ||
      shape->n_q < 1 || shape->n_kv < 1 || shape->head_dim < 1)
    return 0;
  const size_t nqkv = static_cast<size_t>(shape->n_q + 2 * shape->n_kv) * shape->head_dim;
  const size_t H = static_cast<size_t>(shape->hidden), I = static_cast<size_t>(shape->inter);
  return up256(2 * nqkv) + up256(2 * H) + up256(2 * I) + 2 * up256(2 * H);
}

int qgemv_decode_stack(const qgemv_stack_layer* layers, const qgemv_stack_shape* shape,
                       const uint16_t* x, uint16_t* y, void* workspace, size_t workspace_bytes,
                       void* stream) {
  using namespace qgemv;
  if (!layers || !shape || !x || !y || !workspace) return QGEMV_ENULL;
  const int H = shape->hidden, nq = shape->n_q, nkv = shape->n_kv, hd = shape->head_dim;
  const int I = shape->inter, NL = shape->n_layers;
  if (NL < 1 || nq < 1 || nkv < 1 || nq % nkv != 0 || hd < 32 || hd % 32 != 0 ||
      !(shape->eps > 0.0f))
    return QGEMV_EINVAL;
  const int Dq = nq * hd;
  const int nqkv = (nq + 2 * nkv) * hd;
  if (workspace_bytes < qgemv_decode_stack_workspace_bytes(shape)) return QGEMV_EINVAL;
  if (!al16(x) || !al16(y) || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return QGEMV_EALIGN;
  for (int l = 0; l < NL; ++l) {
    const qgemv_stack_layer& s = layers[l];
    const void* p[17] = {s.qkv_codes,   s.qkv_scales,  s.qkv_biases,  s.attn_norm,  s.o_codes,
                         s.o_scales,    s.o_biases,    s.gate_codes,  s.gate_scales,
                         s.gate_biases, s.up_codes,    s.up_scales,   s.up_biases,  s.mlp_norm,
                         s.down_codes,  s.down_scales, s.down_biases};
    for (const void* q : p) {
      if (q == nullptr) return QGEMV_ENULL;
      if (!al16(q)) return QGEMV_EALIGN;
    }
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return QGEMV_EDEVICE;
  // Each op must take the streaming kernel (K a multiple of 1024, at most 16384).
  if (!make_stream_plan(kNorm, 4, H, nqkv, 1, sms).ok ||
      !make_stream_plan(kPlain, 4, Dq, H, 1, sms).ok ||
      !make_stream_plan(kSwiglu, 4, H, I, 1, sms).ok ||
      !make_stream_plan(kPlain, 4, I, H, 1, sms).ok)
    return QGEMV_EINVAL;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // A caller that is capturing its own graph gets the launches themselves.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return QGEMV_ELAUNCH;
  }
  if (cs != cudaStreamCaptureStatusNone)
    return enqueue_stack(layers, shape, x, y, workspace, dev, sms, st);

  const std::vector<uintptr_t> key = graph_key(layers, shape, x, y, workspace, dev);
  std::lock_guard<std::mutex> lock(g_graph_mu);
  GraphEntry* hit = nullptr;
  for (GraphEntry& g : g_graphs)
    if (g.exec != nullptr && g.key == key) hit = &g;
  if (hit == nullptr) {
    cudaGraphExec_t exec = capture_stack(layers, shape, x, y, workspace, dev, sms);
    if (exec == nullptr) return enqueue_stack(layers, shape, x, y, workspace, dev, sms, st);
    GraphEntry* victim = &g_graphs[0];
    for (GraphEntry& g : g_graphs)
      if (g.exec == nullptr || g.last_use < victim->last_use) victim = &g;
    if (victim->exec != nullptr) cudaGraphExecDestroy(victim->exec);
    victim->exec = exec;
    victim->key = key;
    hit = victim;
  }
  hit->last_use = ++g_graph_clock;
  if (cudaGraphLaunch(hit->exec, st) != cudaSuccess) {
    // A cached instance that no longer launches (its context was reset, say)
    // is dropped; this call launches eagerly and the next one re-captures.
    cudaGetLastError();
    cudaGraphExecDestroy(hit->exec);
    cudaGetLastError();
    hit->exec = nullptr;
    hit->key.clear();
    return enqueue_stack(layers, shape, x, y, workspace, dev, sms, st);
  }
  return QGEMV_OK;
}

}  // extern "C"

namespace {

int enqueue_stack(const qgemv_stack_layer* layers, const qgemv_stack_shape* shape,
                  const uint16_t* x, uint16_t* y, void* workspace, int dev, int sms,
                  cudaStream_t st) {
  using namespace qgemv;
  const int H = shape->hidden, nq = shape->n_q, nkv = shape->n_kv, hd = shape->head_dim;
  const int I = shape->inter, NL = shape->n_layers;
  const int Dq = nq * hd;
  const int nqkv = (nq + 2 * nkv) * hd;

  // The four ops' plans (the same for every layer).
  const StreamPlan p0 = make_stream_plan(kNorm, 4, H, nqkv, 1, sms);
  const StreamPlan p1 = make_stream_plan(kPlain, 4, Dq, H, 1, sms);
  const StreamPlan p2 = make_stream_plan(kSwiglu, 4, H, I, 1, sms);
  const StreamPlan p3 = make_stream_plan(kPlain, 4, I, H, 1, sms);
  if (!p0.ok || !p1.ok || !p2.ok || !p3.ok) return QGEMV_EINVAL;

  // Workspace: qkv, h, act, x ping-pong.
  uint8_t* wp = static_cast<uint8_t*>(workspace);
  __half* qkv = reinterpret_cast<__half*>(wp);
  wp += up256(2 * static_cast<size_t>(nqkv));
  __half* h = reinterpret_cast<__half*>(wp);
  wp += up256(2 * static_cast<size_t>(H));
  __half* act = reinterpret_cast<__half*>(wp);
  wp += up256(2 * static_cast<size_t>(I));
  __half* xbuf[2];
  xbuf[0] = reinterpret_cast<__half*>(wp);
  wp += up256(2 * static_cast<size_t>(H));
  xbuf[1] = reinterpret_cast<__half*>(wp);

  auto hp = [](const uint16_t* p) { return reinterpret_cast<const __half*>(p); };
  auto cp = [](const uint32_t* p) { return reinterpret_cast<const uint8_t*>(p); };
  for (int l = 0; l < NL; ++l) {
    const qgemv_stack_layer& L = layers[l];
    const __half* xl = (l == 0) ? hp(x) : xbuf[l & 1];
    StreamArgs a{};
    a.M = 1;
    a.top_k = 1;
    a.eps = shape->eps;

    // op 0: RMSNorm -> QKV
    StreamArgs a0 = a;
    a0.codes[0] = cp(L.qkv_codes);
    a0.scales[0] = hp(L.qkv_scales);
    a0.biases[0] = hp(L.qkv_biases);
    a0.x = xl;
    a0.gamma = hp(L.attn_norm);
    a0.y = qkv;
    a0.rows = nqkv;
    a0.K = H;
    if (stream_norm(p0, a0, st, dev) != cudaSuccess) return QGEMV_ELAUNCH;

    // op 1: o_proj over the value heads of qkv, + residual x_l
    StreamArgs a1 = a;
    a1.codes[0] = cp(L.o_codes);
    a1.scales[0] = hp(L.o_scales);
    a1.biases[0] = hp(L.o_biases);
    a1.x = qkv;
    a1.gather_nq = nq;
    a1.gather_nkv = nkv;
    a1.gather_hd = hd;
    a1.residual = xl;
    a1.y = h;
    a1.rows = H;
    a1.K = Dq;
    if (stream_plain(4, p1, a1, st, dev) != cudaSuccess) return QGEMV_ELAUNCH;

    // op 2: post-attention RMSNorm -> gate.up SwiGLU
    StreamArgs a2 = a;
    a2.codes[0] = cp(L.gate_codes);
    a2.scales[0] = hp(L.gate_scales);
    a2.biases[0] = hp(L.gate_biases);
    a2.codes[1] = cp(L.up_codes);
    a2.scales[1] = hp(L.up_scales);
    a2.biases[1] = hp(L.up_biases);
    a2.x = h;
    a2.gamma = hp(L.mlp_norm);
    a2.y = act;
    a2.rows = I;
    a2.K = H;
    if (stream_swiglu(p2, a2, st, dev) != cudaSuccess) return QGEMV_ELAUNCH;

    // op 3: down + residual h -> x_{l+1} (or y)
    StreamArgs a3 = a;
    a3.codes[0] = cp(L.down_codes);
    a3.scales[0] = hp(L.down_scales);
    a3.biases[0] = hp(L.down_biases);
    a3.x = act;
    a3.residual = h;
    a3.y = (l == NL - 1) ? reinterpret_cast<__half*>(y) : xbuf[(l + 1) & 1];
    a3.rows = H;
    a3.K = I;
    if (stream_plain(4, p3, a3, st, dev) != cudaSuccess) return QGEMV_ELAUNCH;
  }
  return QGEMV_OK;
}

}  // namespace
