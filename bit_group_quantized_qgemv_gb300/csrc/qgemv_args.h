// qgemv_args.h -- host/device-shared argument block, kernel modes and the
// host-side launch planner of the streaming kernels.  No device code.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qgemv {

// Kernel modes (what one output row computes).
enum Mode : int {
  kPlain = 0,    // y = W x (+ residual)
  kNorm = 1,     // y = W (x * gamma) * rstd(x)
  kSwiglu = 2,   // h = silu(Wg xt) * (Wu xt), xt optionally RMS-normalised
  kMoeUp = 3,    // per active expert: h_k = silu(Wg[e] x) * (Wu[e] x)  -> fp32 workspace
  kMoeDown = 4,  // y = r + sum_k wt_k Wd[e_k] h_k
  kArgmax = 5,   // y = W x, and the index of its largest element (greedy lm_head)
};

constexpr int kMaxStages = 16;
constexpr int kSliceK = 32;  // smallest k range of a row one streaming-kernel thread owns
constexpr int kMaxTopK = 8;
constexpr int kMaxM = 8;

struct StreamArgs {
  const uint8_t* codes[2];  // matrix 0 (or gate), matrix 1 (up); MoE: expert-0 bases
  const __half* scales[2];
  const __half* biases[2];
  long long ex_code_bytes;  // MoE: bytes between experts in the code stack
  long long ex_groups;      // MoE: fp16 elements between experts in scale/bias stacks
  const __half* x;          // fp16 activation [M][K] (all modes but kMoeDown)
  const float* xf;          // kMoeDown: fp32 workspace h [top_k][K]
  const __half* gamma;      // RMSNorm weight (kNorm; kSwiglu optional)
  float eps;
  const __half* residual;   // kPlain / kMoeDown, optional, [M][rows]
  __half* y;                // fp16 output [M][rows]
  float* yf;                // kMoeUp: fp32 output (workspace)
  const int* idx;           // MoE expert indices [top_k]
  const float* wt;          // MoE expert weights [top_k]
  int* err_flag;            // MoE: set to 1 on a bad index (nullable)
  // MoE, opt-in: CTA b < trace_ctas writes, per expert slot k, what it read
  // and used: {idx[k], bits of wt[k], expert used (-1: skipped), bits of the
  // weight used (0 when skipped)} at trace[(b * top_k + k) * 4] (nullable).
  unsigned* trace;
  int trace_ctas;
  int top_k, n_experts;
  long long rows;           // output rows: N, I, top_k*I (kMoeUp) or H (kMoeDown)
  int rows_per_expert;      // kMoeUp: I
  int K;                    // reduction length of every row
  int M;                    // batch (generic kPlain only; 1 elsewhere)
  int TG, S, RS, NS;        // launch plan of the streaming kernel
  int stage_bytes;
  int interleave;           // 1: CTAs take stages round-robin (see StageWalker)
  int prefill;              // stages the producer issues before the activations are in
  // kArgmax: the 64-bit (value, index) key the CTAs fold their rows into
  // (zero on entry; argmax_finalize_launch reads it and zeroes it again).
  unsigned long long* am_key;
  // kPlain: when gather_hd > 0, x is the attention output of a decode over
  // one cached position gathered from qkv (x points at qkv): query head h
  // reads value head h / (gather_nq / gather_nkv) of head_dim gather_hd.
  int gather_nq, gather_nkv, gather_hd;
};

struct StreamPlan {
  bool ok = false;
  int kpt = 0;  // k per thread and task (32: half a quantisation group)
  int mb = 1;   // batch rows a consumer thread holds (small-batch kernel)
  int ub = 0, tg = 0, t = 0, s = 0, jr = 0, rs = 0, ns = 0, stage_bytes = 0, grid = 0;
  int red_bytes = 0;   // partial-sum slots per stage
  int interleave = 0;  // 1: CTAs take stages round-robin
  int smem_bytes = 0;  // dynamic shared memory: ns * (stage_bytes + red_bytes)
  int prefill = 0;     // stages issued before every consumer warp has its activations
};

// Weight bytes a CTA's producer may have in flight before its consumers
// have loaded their activations.  A kernel starts (programmatic dependent
// launch) while its predecessor finishes; the activation loads, issued once
// the predecessor's output is visible, queue behind whatever weight copies
// are already outstanding, so issuing the whole ring at once delays them.
// About 100 KB per SM keeps HBM busy meanwhile: measured on GB300 (32-layer
// 8B stack) 1128 us with no limit, 1091 us with two 37 KB stages, 1078 us
// with two (QKV, gate.up) or three (down: 32 KB) stages.
constexpr int kPrefillBytes = 100 * 1024;

inline int prefill_stages(int stage_bytes, int ns) {
  int b = stage_bytes > 0 ? kPrefillBytes / stage_bytes : 1;
  if (b < 1) b = 1;
  return b < ns ? b : ns;
}

// Choose the thread counts, tasks per thread, rows per stage and ring depth
// of the streaming kernel.  ok = false when it does not apply (the generic
// kernel runs instead): K must be a multiple of 1024 and at most 16384, so
// that a row's TG = K/KPT tasks span whole warps and every scale row is a
// multiple of 16 bytes.
inline StreamPlan make_stream_plan(int mode, int bits, int K, long long rows, int top_k,
                                   int sms, int target_threads = 256, int max_jr = 8,
                                   int stage_limit = 40 * 1024, int ring_budget = 200 * 1024,
                                   bool interleave_ok = true) {
  StreamPlan p;
  if ((bits != 4 && bits != 2 && bits != 8) || K % 1024 != 0 || K / kSliceK > 512 || rows <= 0 ||
      sms <= 0)
    return p;
  const int kpt = kSliceK;
  const int tg = K / kpt;
  int s;
  if (mode == kMoeDown) {
    if (top_k < 1 || top_k > kMaxTopK || tg * top_k > 512) return p;
    int m = target_threads / (tg * top_k);
    if (m < 1) m = 1;
    s = top_k * m;
  } else {
    s = target_threads / tg;
    if (s < 1) s = 1;
  }
  const int t = s * tg;
  if (t > 512) return p;
  const int ms = (mode == kSwiglu || mode == kMoeUp) ? 2 : (mode == kMoeDown ? top_k : 1);
  const int task_bytes = K * bits / 8 + 2 * (K / 32);  // one row of one matrix
  int jr = max_jr;
  while (jr > 1 && (static_cast<long long>(s) * jr * task_bytes > stage_limit || (s * jr) % ms))
    jr /= 2;
  if ((s * jr) % ms) return p;
  // An op of at most one stage per CTA: the smallest stage that still holds
  // a CTA's rows (the tasks of rows past a CTA's end are computed and
  // discarded, so a mostly empty stage costs compute for nothing).
  if (mode == kPlain || mode == kNorm || mode == kSwiglu) {
    const long long rpc = (rows + sms - 1) / sms;
    while (jr > 1 && (s * (jr / 2)) % ms == 0 && static_cast<long long>(s) * (jr / 2) / ms >= rpc)
      jr /= 2;
  }
  const int tasks = s * jr;
  const int rs = tasks / ms;
  const long long stage = static_cast<long long>(tasks) * task_bytes;
  if (stage > 100 * 1024) return p;
  const int red = ((tasks * (tg / 32) + 3) & ~3) * static_cast<int>(sizeof(float));
  // (activations are held in registers, loaded straight from global memory:
  // shared memory is all ring)
  int ns = static_cast<int>(ring_budget / (stage + red));
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return p;
  p.ok = true;
  p.kpt = kpt;
  p.ub = kpt * bits / 8;
  p.tg = tg;
  p.t = t;
  p.s = s;
  p.jr = jr;
  p.rs = rs;
  p.ns = ns;
  p.stage_bytes = static_cast<int>(stage);
  p.red_bytes = red;
  p.smem_bytes = ns * (static_cast<int>(stage) + red);
  p.prefill = prefill_stages(p.stage_bytes, ns);
  p.grid = static_cast<int>(rows < sms ? rows : sms);
  // Interleave stages across CTAs when that keeps the SMs within one stage
  // of each other (and, for kMoeUp, stages never straddle experts).
  const long long stages = (rows + rs - 1) / rs;
  const bool experts_align = (mode != kMoeUp) || ((rows / (top_k > 0 ? top_k : 1)) % rs == 0);
  if (interleave_ok && experts_align && stages >= 4LL * sms) {
    p.interleave = 1;
    p.grid = sms;
  }
  return p;
}

// Plan of the small-batch kernel for M = 2..8 activation rows: a thread
// holds its k of all MB >= M rows in registers, so MB * KPT is bounded
// (MB = 2: KPT = 32, K <= 16384; MB = 4: KPT = 32, K <= 14336; MB = 8:
// KPT = 16 with at most 256 consumer threads, i.e. K <= 4096).  ok = false
// when it does not apply.
inline StreamPlan make_batch_plan(int bits, int K, long long rows, int M, int sms,
                                  int stage_limit = 40 * 1024, int ring_budget = 200 * 1024) {
  StreamPlan p;
  if ((bits != 4 && bits != 2) || M < 2 || M > kMaxM || rows <= 0 || sms <= 0) return p;
  const int mb = M <= 2 ? 2 : (M <= 4 ? 4 : 8);
  const int kpt = (mb == 8) ? 16 : 32;
  if (K % (32 * kpt) != 0) return p;
  const int tg = K / kpt;
  const int target = 256;
  if (tg > (mb == 8 ? 256 : (mb == 4 ? 448 : 512))) return p;  // the kernels' launch bounds
  int s = target / tg;
  if (s < 1) s = 1;
  const int t = s * tg;
  // Rows per slot and stage: 8 for MB = 2, 4 for MB = 4 and 8 (measured on
  // GB300: 2 rows for MB = 4 / 8 was 8-12 % slower, the per-stage handshake
  // and reduction spread over fewer FMAs; MB = 2 with 512 threads of 4 rows
  // 3 % slower; MB = 4 with 8 rows spills)
  int jr = (mb == 2) ? 8 : 4;
  const int task_bytes = K * bits / 8 + 2 * (K / 32);
  while (jr > 1 && static_cast<long long>(s) * jr * task_bytes > stage_limit) jr /= 2;
  const int rs = s * jr;
  const long long stage = static_cast<long long>(rs) * task_bytes;
  if (stage > 100 * 1024) return p;
  const int red = ((rs * mb * (tg / 32) + 3) & ~3) * static_cast<int>(sizeof(float));
  int ns = static_cast<int>(ring_budget / (stage + red));
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return p;
  p.ok = true;
  p.kpt = kpt;
  p.mb = mb;
  p.ub = kpt * bits / 8;
  p.tg = tg;
  p.t = t;
  p.s = s;
  p.jr = jr;
  p.rs = rs;
  p.ns = ns;
  p.stage_bytes = static_cast<int>(stage);
  p.red_bytes = red;
  p.smem_bytes = ns * (static_cast<int>(stage) + red);
  p.prefill = prefill_stages(p.stage_bytes, ns);
  p.grid = static_cast<int>(rows < sms ? rows : sms);
  const long long stages = (rows + rs - 1) / rs;
  if (stages >= 4LL * sms) {
    p.interleave = 1;
    p.grid = sms;
  }
  return p;
}

// Entry points of the kernel translation units (each returns the CUDA
// error of its launch).
cudaError_t stream_plain(int bits, const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                         int device);
cudaError_t stream_norm(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device);
cudaError_t stream_swiglu(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device);
cudaError_t stream_moe_up(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device);
cudaError_t stream_moe_down(const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                            int device);
cudaError_t stream_batch(int bits, const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                         int device);
// Tensor-core small-batch kernel (M = 3..8, and M = 2 on short ops, in one
// pass; K split across a cluster of up to 4 CTAs when the activations are
// large).  batch_mma_plan: whether it takes a pass of M rows (K a multiple
// of 512, the staged activations within their shared-memory budget), with
// its B columns, dynamic shared memory, ring depth, cluster size and chunk
// length (kc nullable); stream_batch_mma returns cudaErrorNotSupported when
// it does not.
bool batch_mma_plan(int bits, int K, long long N, int M, int sms, int* mp, int* smem, int* ns,
                    int* cl, int* kc = nullptr);
cudaError_t stream_batch_mma(int bits, const StreamArgs& a, int sms, cudaStream_t st, int device);
cudaError_t stream_argmax(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device);
// Single-CTA argmax of an fp16 vector (the fallback when the streaming kernel
// does not take the shape): token = lowest index of the largest element.
cudaError_t argmax_launch(const __half* y, int n, int* token, cudaStream_t st);
// MoE routing from fp16 logits [E] (one CTA, chained after the router
// GEMV): idx [top_k] = the shared expert (shared >= 0) and the routed
// experts with the largest logits, wt [top_k] = their softmax.
cudaError_t moe_route_launch(const __half* logits, int E, int top_k, int shared, int* idx,
                             float* wt, cudaStream_t st);
// After a kArgmax launch: once its grid has completed, token = the index in
// *key, and *key = 0 (programmatic dependent launch: one thread).
cudaError_t argmax_finalize_launch(unsigned long long* key, int* token, cudaStream_t st);
cudaError_t generic_launch(int mode, int bits, const StreamArgs& a, cudaStream_t st);
// CTAs generic_launch starts for these arguments (8 rows each).
inline int generic_blocks(const StreamArgs& a) { return static_cast<int>((a.rows + 7) / 8); }
cudaError_t selftest_wait_launch(uint64_t limit_ns, cudaStream_t st);
cudaError_t attention_seq1_launch(const __half* qkv, __half* out, int n_q, int n_kv,
                                  int head_dim, cudaStream_t st);

// Read and clear the device status word of each translation unit.
cudaError_t status_plain(unsigned* out);
cudaError_t status_norm_swiglu(unsigned* out);
cudaError_t status_moe(unsigned* out);
cudaError_t status_generic(unsigned* out);
cudaError_t status_batch(unsigned* out);

}  // namespace qgemv
