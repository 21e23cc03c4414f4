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
};

constexpr int kMaxStages = 16;
constexpr int kMaxTopK = 8;
constexpr int kMaxM = 8;
constexpr int kRedSlots = 128;  // JR * T / 32 <= 8 * 512 / 32

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
  int top_k, n_experts;
  long long rows;           // output rows: N, I, top_k*I (kMoeUp) or H (kMoeDown)
  int rows_per_expert;      // kMoeUp: I
  int K;                    // reduction length of every row
  int M;                    // batch (generic kPlain only; 1 elsewhere)
  int TG, S, RS, NS;        // launch plan of the streaming kernel
  int stage_bytes;
};

struct StreamPlan {
  bool ok = false;
  int ub = 0, tg = 0, t = 0, s = 0, jr = 0, rs = 0, ns = 0, stage_bytes = 0, grid = 0;
};

// Choose the unit size, thread counts, rows per stage and ring depth of the
// streaming kernel.  ok = false when it does not apply (the generic kernel
// runs instead): K must be a multiple of 1024 (2048 for 2-bit) so that each
// task spans whole warps and every scale row is a multiple of 16 bytes.
inline StreamPlan make_stream_plan(int mode, int bits, int K, long long rows, int top_k,
                                   int sms, int target_threads = 256) {
  StreamPlan p;
  if (K % 1024 != 0 || rows <= 0 || sms <= 0) return p;
  int tg = 0, ub = 0;
  if (bits == 4) {
    if ((K / 64) % 32 == 0 && K / 64 <= 512) {
      ub = 32;
      tg = K / 64;
    } else if ((K / 32) % 32 == 0 && K / 32 <= 512) {
      ub = 16;
      tg = K / 32;
    }
  } else if (bits == 2) {
    if ((K / 64) % 32 == 0 && K / 64 <= 512) {
      ub = 16;
      tg = K / 64;
    }
  }
  if (tg == 0) return p;
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
  const int nmat = (mode == kSwiglu || mode == kMoeUp) ? 2 : (mode == kMoeDown ? top_k : 1);
  const int rowstep = (mode == kMoeDown) ? s / top_k : s;
  const int row_bytes = nmat * (K * bits / 8 + 2 * (K / 32));
  int jr = 4;
  if (static_cast<long long>(jr) * rowstep * row_bytes > 40 * 1024) jr = 2;
  const int rs = jr * rowstep;
  const long long stage = static_cast<long long>(rs) * row_bytes;
  if (stage > 100 * 1024) return p;
  int ns = static_cast<int>((200 * 1024) / stage);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return p;
  if (jr * t / 32 > kRedSlots) return p;
  p.ok = true;
  p.ub = ub;
  p.tg = tg;
  p.t = t;
  p.s = s;
  p.jr = jr;
  p.rs = rs;
  p.ns = ns;
  p.stage_bytes = static_cast<int>(stage);
  p.grid = static_cast<int>(rows < sms ? rows : sms);
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
cudaError_t generic_launch(int mode, int bits, const StreamArgs& a, cudaStream_t st);
cudaError_t attention_seq1_launch(const __half* qkv, __half* out, int n_q, int n_kv,
                                  int head_dim, cudaStream_t st);

// Read and clear the device status word of each translation unit.
cudaError_t status_plain(unsigned* out);
cudaError_t status_norm_swiglu(unsigned* out);
cudaError_t status_moe(unsigned* out);
cudaError_t status_generic(unsigned* out);

}  // namespace qgemv
