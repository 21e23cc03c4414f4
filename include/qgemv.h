/*
 * qgemv.h -- C ABI of libqgemv.so: dequant-fused quantized matrix-vector
 * products for batch-1 (and small-batch) LLM decode on NVIDIA GB300 (sm_103a).
 *
 * Weight format (all entry points).  A weight W of N rows and K columns is
 * stored planar, MLX style ("Boosting inference speed on Apple Silicon",
 * INFERENCE_RESEARCH.md, section 3, item 4: 4-bit data packed in uint32 plus
 * separate scale and bias tensors, group 64; item 5: rows laid out along the
 * matvec's access direction, consumed as stored):
 *   codes   uint32 [N][K*bits/32]  row-major; code q[n][k] sits in word
 *           k / (32/bits) at bit offset bits * (k % (32/bits)), low bits first.
 *   scales  fp16   [N][K/64]       row-major, one per 64 consecutive k of a row.
 *   biases  fp16   [N][K/64]       same layout.
 *   w[n][k] = q[n][k] * scales[n][k/64] + biases[n][k/64].
 * fp16 values are IEEE binary16 passed as uint16_t bit patterns.  Activations
 * x are fp16 [M][K] and outputs fp16 [M][N], row-major, unit stride.  Every
 * product accumulates in fp32 and each fp16 output is rounded once (RNE).
 * The inner loop evaluates the dequantised product through the exact
 * rewrite of (q*scale + bias)*x as fma(q, scale*x, bias*x) given on the
 * hada.io page (topic 27758), "Noyau de dequantification optimise FMA",
 * factored per group of 64: scale * sum(q*x) + bias * sum(x).
 *
 * Conventions.
 *   - Every pointer argument except `stream` (and the host descriptor
 *     arrays of qgemv_decode_stack) is a DEVICE pointer owned by the caller.
 *     The library allocates no device memory per call and does not
 *     synchronise (qgemv_device_status excepted); work is only enqueued on
 *     `stream` (a cudaStream_t; NULL = legacy default).  It holds three
 *     things of its own for the life of the process: the fixed scratch
 *     array of moe_qgemv_combine_noalloc, and the CUDA graphs (at most 4)
 *     and the capture stream per device of qgemv_decode_stack.
 *   - Return value: QGEMV_OK (0) or a negative QGEMV_E* status.  Argument
 *     checks run on the host before any launch; on failure nothing is
 *     enqueued.  QGEMV_ELAUNCH reports a CUDA error seen right after the
 *     launch; its code is kept for qgemv_last_cuda_error().
 *   - Kernels never trap.  A device-side wait that runs out (it has a
 *     bounded spin) sets a library flag read by qgemv_device_status().
 *   - Inputs may not overlap outputs, except that `residual` may be the
 *     same pointer as `y` (an in-place residual add).
 *   - Calls are asynchronous and thread-compatible: concurrent calls on
 *     different streams are safe when their outputs do not overlap.
 *   - Launches are chained by programmatic dependent launch: a kernel may
 *     start while the kernel enqueued before it on `stream` is still
 *     running and may already read its weights (codes, scales, biases,
 *     tables, norm weights); it waits for that kernel to complete before it
 *     reads anything else (activations, residuals, expert indices and
 *     weights, logits, u) and before it writes.  So
 *     weights must not be written by the kernel enqueued immediately
 *     before the call on the same stream; anything earlier is ordered.
 */
#ifndef QGEMV_H_
#define QGEMV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QGEMV_OK 0
#define QGEMV_EINVAL (-1)  /* bad shape or scalar argument                   */
#define QGEMV_ENULL (-2)   /* a required pointer is NULL                      */
#define QGEMV_EALIGN (-3)  /* codes not 4-byte aligned, fp16 not 2-byte aligned */
#define QGEMV_ELAUNCH (-4) /* CUDA reported an error at launch                */
#define QGEMV_EDEVICE (-5) /* no usable CUDA device / device query failed     */
#define QGEMV_ESCRATCH (-6) /* top_k * I exceeds the allocation-free scratch    */

/* Largest supported small batch M and expert count top_k. */
#define QGEMV_MAX_M 8
#define QGEMV_MAX_TOPK 8

/*
 * qgemv_w4g64 -- y[m][n] = sum_k w[n][k] * x[m][k] (+ residual[m][n]),
 * 4-bit codes, group 64.  The dequant-fused GEMV of INFERENCE_RESEARCH.md
 * section 1 (dequantisation inside the inner loop, no f32 weights ever
 * materialised); small-batch M <= 8 follows the mat-vec branch of the
 * "routing by M" decision in the same section.
 *   codes    [N][K/8] uint32      scales, biases [N][K/64] fp16
 *   x        [M][K] fp16          y [M][N] fp16
 *   residual [M][N] fp16 or NULL (may equal y)
 *   1 <= M <= 8, N >= 1, K >= 64 and K % 64 == 0, else QGEMV_EINVAL.
 */
int qgemv_w4g64(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                const uint16_t *x, uint16_t *y, int M, int N, int K,
                const uint16_t *residual, void *stream);

/*
 * qgemv_w2g64 -- the same product with 2-bit codes (the 2-bit expert
 * configuration on the hada.io page, "Resultats de performance" and
 * "Shaders de calcul Metal"): codes [N][K/16] uint32, 16 codes per word,
 * low bits first.  Other arguments and checks as qgemv_w4g64.
 */
int qgemv_w2g64(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                const uint16_t *x, uint16_t *y, int M, int N, int K,
                const uint16_t *residual, void *stream);

/*
 * qgemv_w8g64 -- the same product with 8-bit codes (Q8 group 64, the other
 * quantisation level the BaseRT page, "BaseRT: Best-in-Class LLM Inference
 * on Apple Silicon via Native Metal", evaluates beside Q4, in the planar
 * layout of INFERENCE_RESEARCH.md section 3 item 4): codes [N][K/4] uint32,
 * 4 codes per word, low byte first; w = q * scale + bias with q in 0..255.
 * Other arguments and checks as qgemv_w4g64 (M > 1 takes the generic kernel).
 */
int qgemv_w8g64(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                const uint16_t *x, uint16_t *y, int M, int N, int K,
                const uint16_t *residual, void *stream);

/*
 * qgemv_plan_gemv -- which kernels qgemv_w4g64 / qgemv_w2g64 / qgemv_w8g64
 * launch for a shape, without touching the device (host-only; for callers
 * that size work or check a deployment, and for the host tests).  bits 2,
 * 4 or 8; M, N, K as those calls check them; sms: the device's
 * multiprocessor count; aligned16: 1 when codes, scales, biases and x are
 * 16-byte aligned (the fast kernels need it), else 0.  Fills *out:
 *   path        QGEMV_PATH_* below
 *   passes      launches of that kernel (passes of at most 4 batch rows)
 *   m_pad       tensor-core paths: B columns the batch is padded to (4, 8)
 *   cluster     tensor-core paths: CTAs that split K between them (1, 2, 4)
 *   chunk_k     tensor-core paths: k per ring stage
 *   stages      ring depth of the kernel (0 for the generic kernel)
 *   smem_bytes  its dynamic shared memory per CTA (0 for the generic kernel)
 * The tensor-core path can still fall back to the CUDA-core kernels at
 * launch when the device cannot host the plan's clusters.  Returns
 * QGEMV_ENULL (out NULL) or QGEMV_EINVAL (bits, M, N, K or sms out of
 * range), else QGEMV_OK.
 */
#define QGEMV_PATH_GENERIC 0      /* one thread block per 8 rows, any alignment */
#define QGEMV_PATH_STREAM 1       /* M = 1 streaming kernel */
#define QGEMV_PATH_MMA 2          /* tensor-core small batch, one pass */
#define QGEMV_PATH_MMA_PASSES 3   /* tensor-core small batch, passes of <= 4 rows */
#define QGEMV_PATH_BATCH 4        /* CUDA-core small batch, one pass */
#define QGEMV_PATH_BATCH_PASSES 5 /* CUDA-core small batch, passes of <= 4 rows */
typedef struct {
  int path, passes, m_pad, cluster, chunk_k, stages, smem_bytes;
} qgemv_gemv_plan;
int qgemv_plan_gemv(int bits, int M, int N, int K, int sms, int aligned16, qgemv_gemv_plan *out);

/*
 * rmsnorm_qgemv -- y = W . (x * gamma / sqrt(mean(x^2) + eps)), M = 1,
 * 4-bit g64.  The RMSNorm + QKV matvec fusion of INFERENCE_RESEARCH.md
 * section 1 (and the RMS normalisation shader on the hada.io page).
 *   x, norm_weight (gamma) [K] fp16; y [N] fp16; eps > 0 (else EINVAL).
 * The normalised activation x*gamma is rounded to fp16 once inside the
 * kernel and 1/sqrt(mean(x^2)+eps) is applied to the fp32 row sums.
 */
int rmsnorm_qgemv(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                  const uint16_t *x, const uint16_t *norm_weight, float eps,
                  uint16_t *y, int N, int K, void *stream);

/*
 * swiglu_qgemv -- h[i] = silu(g_i) * u_i with g = Wg . xt, u = Wu . xt,
 * xt = x, or xt = rmsnorm(x) * gamma when norm_weight is not NULL (the
 * post-attention norm fused in front).  The "gate.up SwiGLU in one kernel"
 * fusion of INFERENCE_RESEARCH.md section 1; silu(z) = z / (1 + e^-z).
 *   gate_*: Wg [I][K], up_*: Wu [I][K] (4-bit g64, separate pointers; a
 *   caller holding one [2I][K] matrix passes base and base + I rows).
 *   x [K] fp16, norm_weight [K] fp16 or NULL, eps > 0 when used; h [I] fp16.
 */
int swiglu_qgemv(const uint32_t *gate_codes, const uint16_t *gate_scales,
                 const uint16_t *gate_biases, const uint32_t *up_codes,
                 const uint16_t *up_scales, const uint16_t *up_biases,
                 const uint16_t *x, const uint16_t *norm_weight, float eps,
                 uint16_t *h, int I, int K, void *stream);

/*
 * moe_qgemv_combine -- MoE top-K expert matvec with weighted combine and
 * residual (hada.io page: 512 experts, K = 4 active per token including one
 * shared expert, hidden 4096, "Deferred GPU Expert Compute": combine +
 * residual on the GPU, result handed to the next layer):
 *   for k < top_k: e = expert_idx[k];
 *     h_k = silu(Wgu[e][0:I] . x) * (Wgu[e][I:2I] . x)      (fp32, workspace)
 *   y[n] = residual[n] + sum_k expert_w[k] * (Wd[e] . h_k)[n]   (fp16)
 *   gu_codes  [E][2I][H/8] uint32, gu_scales/gu_biases [E][2I][H/64] fp16
 *             (expert-contiguous; gate rows 0..I-1, then up rows I..2I-1)
 *   dn_codes  [E][H][I/8] uint32, dn_scales/dn_biases [E][H][I/64] fp16
 *   expert_idx [top_k] int32 and expert_w [top_k] fp32 are DEVICE arrays,
 *   read by the kernels (no host synchronisation).
 *   x, residual, y [H] fp16 (residual may equal y; NULL means zero).
 *   workspace: device fp32, >= qgemv_moe_workspace_bytes(top_k, I) bytes,
 *   4-byte aligned; its contents on entry are ignored.
 *   err_flag: device int or NULL.  An index outside [0, n_experts) sets
 *   *err_flag = 1 and that expert contributes nothing; the flag is never
 *   cleared by the library.  A repeated index contributes twice.
 *   Checks: n_experts >= 1, 1 <= top_k <= 8, H and I >= 64, multiples of 64.
 */
int moe_qgemv_combine(const uint32_t *gu_codes, const uint16_t *gu_scales,
                      const uint16_t *gu_biases, const uint32_t *dn_codes,
                      const uint16_t *dn_scales, const uint16_t *dn_biases,
                      int n_experts, int H, int I, const int32_t *expert_idx,
                      const float *expert_w, int top_k, const uint16_t *x,
                      const uint16_t *residual, uint16_t *y, float *workspace,
                      int *err_flag, void *stream);

/*
 * moe_qgemv_combine_traced -- moe_qgemv_combine that also records, for the
 * test suite and for debugging, which expert indices and weights each CTA
 * of its two kernels read and used (hada.io page, "Architecture du modele":
 * the expert indices are routing decisions and must be honoured exactly).
 * Same arguments, results and checks as moe_qgemv_combine, plus:
 *   trace: device, 16-byte aligned, 2 * trace_ctas * top_k * 4 uint32.
 *     CTA b < trace_ctas of phase p (0: gate.up + SwiGLU, 1: down + combine)
 *     writes, for each expert slot k, at trace[((p * trace_ctas + b) * top_k
 *     + k) * 4]: the int32 expert_idx[k] it read, the fp32 bits of
 *     expert_w[k] it read, the expert it used (-1 when the index is out of
 *     range and the slot is skipped) and the bits of the weight it used (0
 *     when skipped).  Records of CTAs that do not exist are left untouched.
 *   trace_ctas >= 1 (else EINVAL); ctas_launched: HOST int[2], set to the
 *   number of CTAs each phase launched (records exist for the first
 *   min(ctas_launched[p], trace_ctas) of them).  NULL trace or
 *   ctas_launched: ENULL.
 */
int moe_qgemv_combine_traced(const uint32_t *gu_codes, const uint16_t *gu_scales,
                             const uint16_t *gu_biases, const uint32_t *dn_codes,
                             const uint16_t *dn_scales, const uint16_t *dn_biases,
                             int n_experts, int H, int I, const int32_t *expert_idx,
                             const float *expert_w, int top_k, const uint16_t *x,
                             const uint16_t *residual, uint16_t *y, float *workspace,
                             int *err_flag, uint32_t *trace, int trace_ctas,
                             int *ctas_launched, void *stream);

/* Workspace bytes moe_qgemv_combine needs: top_k * I fp32 values. */
size_t qgemv_moe_workspace_bytes(int top_k, int I);

/* Capacity of the allocation-free entry point's scratch, in fp32 values. */
#define QGEMV_NOALLOC_MAX_SCRATCH 16384

/*
 * moe_qgemv_combine_noalloc -- moe_qgemv_combine without a workspace
 * argument, for callers that cannot allocate device memory: for instance a
 * plugin inside a host application that owns every device allocation and
 * gives the plugin no allocator, or a latency-critical loop that must not
 * allocate once it is running.  (The paper has no counterpart; this is an
 * interface convenience of this library.)
 *
 * Instead of a caller workspace it uses one fixed scratch array of
 * QGEMV_NOALLOC_MAX_SCRATCH fp32 values (64 KiB) in the library's own device
 * memory.  Every GPU that loads the library holds that array until the
 * process exits.  The call allocates nothing, and calls no cudaMalloc or
 * cudaFree.
 *   - Checks, in this order: a NULL required pointer gives QGEMV_ENULL;
 *     a bad n_experts, top_k, H or I (as moe_qgemv_combine) QGEMV_EINVAL;
 *     top_k * I above QGEMV_NOALLOC_MAX_SCRATCH QGEMV_ESCRATCH; then the
 *     alignment checks of moe_qgemv_combine (QGEMV_EALIGN).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and keeps it with the
 *     id of the device's current context; a call in another context (after
 *     cudaDeviceReset, say) looks it up again.  Make the first call on a
 *     device, and the first after a reset, outside any stream capture.
 *   - All calls share the array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero: the first kernel writes every
 *     value the second one reads.  Calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on the array; serialise them.
 * Results are identical to moe_qgemv_combine with a workspace.
 */
int moe_qgemv_combine_noalloc(const uint32_t *gu_codes, const uint16_t *gu_scales,
                              const uint16_t *gu_biases, const uint32_t *dn_codes,
                              const uint16_t *dn_scales, const uint16_t *dn_biases,
                              int n_experts, int H, int I, const int32_t *expert_idx,
                              const float *expert_w, int top_k, const uint16_t *x,
                              const uint16_t *residual, uint16_t *y, int *err_flag,
                              void *stream);

/* Bytes of the allocation-free entry point's scratch array. */
size_t qgemv_noalloc_max_scratch(void);

/*
 * decode_attention_seq1 -- attention of one query over a single cached
 * position: the softmax over one score is 1, so query head h returns value
 * head h / (n_q / n_kv) unchanged.  Copies those value heads out of a fused
 * QKV vector into the o_proj input:
 *   out[h*head_dim + d] = qkv[(n_q + n_kv + h / (n_q/n_kv)) * head_dim + d].
 * qkv [(n_q + 2 n_kv) * head_dim] fp16, out [n_q * head_dim] fp16.
 * n_q % n_kv == 0 else EINVAL.  (The decode-stack stand-in for attention;
 * attention proper is outside this library.)
 */
int decode_attention_seq1(const uint16_t *qkv, uint16_t *out, int n_q, int n_kv,
                          int head_dim, void *stream);

/*
 * Decode stack: one token through a stack of pre-norm transformer layers'
 * quantized matvecs in one call: 4 kernel launches per layer, chained by
 * programmatic dependent launch and replayed from a cached CUDA graph.
 * INFERENCE_RESEARCH.md section 1: encode the whole layer stack at once,
 * fused kernels, zero per-token overhead.
 * Per layer l, with 4-bit g64 weights and fp16 activations:
 *   qkv     = W_qkv . rmsnorm(x_l; attn_norm)              [(n_q+2 n_kv) hd]
 *   attn    = value heads of qkv, head h -> value head h/(n_q/n_kv)
 *             (decode over one cached position: softmax of one score is 1)
 *   h       = x_l + W_o . attn                              [hidden]
 *   act     = silu(W_gate . r) * (W_up . r), r = rmsnorm(h; mlp_norm)  [inter]
 *   x_{l+1} = h + W_down . act                              [hidden]
 * with rmsnorm(v; g) = v * g / sqrt(mean(v^2) + eps).  Same arithmetic and
 * roundings as rmsnorm_qgemv, decode_attention_seq1, qgemv_w4g64 and
 * swiglu_qgemv chained.
 */
typedef struct {
  const uint32_t *qkv_codes;   /* [(n_q + 2 n_kv) * head_dim][hidden/8]  */
  const uint16_t *qkv_scales, *qkv_biases;
  const uint16_t *attn_norm;   /* [hidden] fp16 */
  const uint32_t *o_codes;     /* [hidden][n_q * head_dim / 8]           */
  const uint16_t *o_scales, *o_biases;
  const uint16_t *mlp_norm;    /* [hidden] fp16 */
  const uint32_t *gate_codes;  /* [inter][hidden/8]                      */
  const uint16_t *gate_scales, *gate_biases;
  const uint32_t *up_codes;    /* [inter][hidden/8]                      */
  const uint16_t *up_scales, *up_biases;
  const uint32_t *down_codes;  /* [hidden][inter/8]                      */
  const uint16_t *down_scales, *down_biases;
} qgemv_stack_layer;

typedef struct {
  int hidden, n_q, n_kv, head_dim, inter, n_layers;
  float eps;
} qgemv_stack_shape;

/* Workspace bytes qgemv_decode_stack needs (qkv, h, act, x ping-pong). */
size_t qgemv_decode_stack_workspace_bytes(const qgemv_stack_shape *shape);

/*
 * qgemv_decode_stack -- y = stack(x).  `layers` is a HOST array of n_layers
 * descriptors of device pointers (all 16-byte aligned); x, y [hidden] fp16
 * device (16-byte aligned, may not overlap the workspace); workspace:
 * device, 256-byte aligned, >= qgemv_decode_stack_workspace_bytes bytes,
 * contents on entry ignored.  Checks: n_layers >= 1, n_q % n_kv == 0,
 * head_dim % 32 == 0, hidden, n_q*head_dim and inter multiples of 1024 and at
 * most 16384, eps > 0.  Enqueues 4 * n_layers streaming-kernel launches on
 * `stream` (programmatic dependent launch between them: each op's weights
 * start streaming while the previous op finishes); calls that share a
 * workspace must not overlap on the GPU.  The launches of each distinct
 * argument set (device, shape, every pointer) are captured once into a
 * CUDA graph (up to 4 kept, least recently used replaced) and later calls
 * replay it with one graph launch on `stream`; when `stream` is itself
 * being captured, the launches are enqueued on it directly.
 */
int qgemv_decode_stack(const qgemv_stack_layer *layers, const qgemv_stack_shape *shape,
                       const uint16_t *x, uint16_t *y, void *workspace, size_t workspace_bytes,
                       void *stream);

/* Human-readable text for a status code (static string). */
const char *qgemv_strerror(int status);

/* cudaError_t value of the last QGEMV_ELAUNCH on this host thread (0 if none). */
int qgemv_last_cuda_error(void);

/*
 * qgemv_device_status -- synchronously read and clear the library's
 * device-side status word on the current device: bit 0 = a bounded wait in a
 * kernel ran out.  *flags receives the word.  Diagnostic: it synchronises the
 * device.  Returns QGEMV_OK or QGEMV_EDEVICE.
 */
int qgemv_device_status(unsigned *flags);

/*
 * qgemv_residual_rmsnorm -- the residual add and the RMSNorm of a pre-norm
 * block as one standalone epilogue (INFERENCE_RESEARCH.md section 1: the
 * residual+norm fusion), for callers whose matvecs do not fuse them:
 *   h  = x + residual, rounded once to fp16 (h = x when residual is NULL,
 *        and then h is not written and may be NULL),
 *   xn = h * gamma / sqrt(mean(h^2) + eps), rounded once to fp16, the mean
 *        over the fp16 h.
 * x, residual, gamma, h, xn: fp16 [K] device.  Checks: K >= 1, eps > 0.
 * One CTA, chained by programmatic dependent launch.
 */
int qgemv_residual_rmsnorm(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma,
                           float eps, int K, uint16_t *h, uint16_t *xn, void *stream);

/*
 * qgemv_moe_router -- MoE routing of one token on the GPU (the hada.io page,
 * topic 27758, "Architecture du modele": K active experts of E, one shared;
 * INFERENCE_RESEARCH.md section 1: keep the routing on the device):
 * logits = Wr . x (4-bit g64 router weight [E][H], as qgemv_w4g64), then
 * expert_idx = the shared expert (shared_expert >= 0; -1 for none) followed
 * by the routed experts with the largest logits, in decreasing order, the
 * lower index winning a tie (the fp16 logits are compared), until top_k are
 * chosen; expert_w = softmax of the chosen logits (fp32).  expert_idx int32
 * [top_k] and expert_w fp32 [top_k] on the device are what
 * moe_qgemv_combine takes.  logits: fp16 [E] device output (required).
 * Checks: E >= 1, 1 <= top_k <= 8, top_k <= E, -1 <= shared_expert < E,
 * H >= 64 and H % 64 == 0.  Two launches (the GEMV, then a one-CTA
 * selection chained by programmatic dependent launch).
 */
int qgemv_moe_router(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                     const uint16_t *x, int E, int H, int top_k, int shared_expert,
                     uint16_t *logits, int32_t *expert_idx, float *expert_w, void *stream);

/*
 * qgemv_lm_head_argmax -- greedy decoding of the last matvec of a decode
 * step (INFERENCE_RESEARCH.md section 1: lm_head and sampling on the GPU,
 * only the token read back): logits = W . x exactly as qgemv_w4g64 (M = 1),
 * and *token = the lowest index n of the largest logits[n] (the fp16 values
 * compared; NaNs are not expected).  codes/scales/biases: 4-bit g64 as
 * qgemv_w4g64, N rows (the vocabulary), K columns; x fp16 [K]; logits fp16
 * [N] device output (required); token: device int32.  scratch: device,
 * 8-byte aligned, qgemv_argmax_scratch_bytes() bytes, zeroed by the caller
 * before its first use; every call leaves it zero again.  Calls sharing a
 * scratch must not overlap on the GPU.  When the streaming kernel takes the
 * shape (K a multiple of 1024, at most 16384, 16-byte-aligned operands) its
 * epilogue folds each CTA's rows into one 64-bit (value, index) key in the
 * scratch with a reduction that returns nothing, and a one-thread kernel
 * chained by programmatic dependent launch turns the key into the index;
 * otherwise the generic GEMV and a one-CTA argmax kernel.
 */
int qgemv_lm_head_argmax(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                         const uint16_t *x, uint16_t *logits, int N, int K, void *scratch,
                         int32_t *token, void *stream);

/* Bytes of the scratch qgemv_lm_head_argmax needs (16). */
size_t qgemv_argmax_scratch_bytes(void);

#define QGEMV_SAMPLE_MAX_K 1024
#define QGEMV_SAMPLE_MAX_N 786432

/*
 * qgemv_sample_topk -- top-k sampling of the next token from its logits on
 * the GPU (INFERENCE_RESEARCH.md section 1: the logits matvec followed by
 * top-k sampling on the GPU, only the token read back).  The candidates are
 * the top_k largest logits (the fp16 values compared, -0 equal to +0, the
 * lower index first among equal values), in decreasing order c_0 .. c_{k-1};
 * their weights p_j = exp((l[c_j] - l[c_0]) / temperature) (fp32); *token =
 * c_j for the first j whose running sum p_0 + .. + p_j exceeds
 * (*u) * (p_0 + .. + p_{k-1}), c_{k-1} when none does.  The random number is
 * the caller's: u is one fp32 on the device, read when the kernel runs (so a
 * captured graph samples afresh when the caller rewrites it), meant to be in
 * [0, 1).  The choice of candidates is exact; the weights are fp32, so a u
 * within about 1e-4 of a boundary of the running sum may fall to either
 * neighbour.  logits: fp16 [N] device; token: int32 device; topk_idx (int32
 * [top_k]) and topk_prob (fp32 [top_k], p_j / sum p) are optional device
 * outputs (NULL to skip).  Logits are expected finite: a non-finite logit
 * still yields one of the candidates, with unspecified weights.  Checks:
 * 1 <= N <= QGEMV_SAMPLE_MAX_N, 1 <= top_k <= min(N, QGEMV_SAMPLE_MAX_K),
 * temperature finite and > 0 (QGEMV_EINVAL); logits, u and token non-NULL
 * (QGEMV_ENULL); logits 2-byte, u, token, topk_idx and topk_prob 4-byte
 * aligned (QGEMV_EALIGN).  One launch of a cluster of 8 CTAs (each holds
 * N/8 logits in shared memory), chained to the previous kernel on `stream`
 * by programmatic dependent launch; no scratch, no allocation.
 */
int qgemv_sample_topk(const uint16_t *logits, int N, int top_k, float temperature,
                      const float *u, int32_t *token, int32_t *topk_idx, float *topk_prob,
                      void *stream);

/*
 * qgemv_lm_head_sample -- the lm_head matvec and top-k sampling as one call:
 * logits = W . x exactly as qgemv_w4g64 (M = 1; logits fp16 [N] device
 * output, required), then qgemv_sample_topk on those logits.  Arguments as
 * the two calls; every check of both is made before the first launch.  Two
 * launches, the second chained by programmatic dependent launch.
 */
int qgemv_lm_head_sample(const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                         const uint16_t *x, uint16_t *logits, int N, int K, int top_k,
                         float temperature, const float *u, int32_t *token, int32_t *topk_idx,
                         float *topk_prob, void *stream);

#define QGEMV_LUT_MAX_K 16384

/*
 * qgemv_lut4 -- the LUT / palettised 4-bit GEMV ("Boosting inference speed
 * on Apple Silicon", INFERENCE_RESEARCH.md section 3 item 4: a LUT /
 * palettised type, 4-bit indices and a 16-entry f16 LUT, Core ML style):
 *   y[n] = sum_k lut[n / rows_per_lut][q[n][k]] * x[k] (+ residual[n])
 * with fp32 accumulation and one round-to-nearest-even to fp16; every
 * product of a table entry and an activation is exact.
 * codes: device uint32 [N][K/8], 4-bit indices, 8 per word, low nibble
 * first along K (the qgemv_w4g64 code layout).  lut: device fp16
 * [n_luts][16]; table t serves rows t*rows_per_lut .. +rows_per_lut-1
 * (rows_per_lut = N: one table for the tensor; 1: one per row).  x: fp16
 * [K]; y: fp16 [N]; residual: fp16 [N] or NULL.  M = 1.
 * Checks: N >= 1, K >= 64, K % 64 == 0, K <= QGEMV_LUT_MAX_K, rows_per_lut
 * >= 1, n_luts * rows_per_lut >= N (QGEMV_EINVAL); codes, lut and x 16-byte
 * aligned, y and residual 2-byte aligned (QGEMV_EALIGN).  One launch,
 * chained by programmatic dependent launch.
 */
int qgemv_lut4(const uint32_t *codes, const uint16_t *lut, int n_luts, int rows_per_lut,
               const uint16_t *x, uint16_t *y, int N, int K, const uint16_t *residual,
               void *stream);

/*
 * qgemv_selftest_wait_timeout -- health check of the bounded device waits
 * every kernel uses: enqueues one tiny kernel on `stream` whose thread waits
 * on a shared-memory mbarrier that nothing ever arrives on, with a limit of
 * limit_us microseconds (1 .. 1000000) instead of the kernels' 1 s.  The
 * wait gives up, sets bit 0 of the status word read by qgemv_device_status
 * and the kernel returns: no trap, the context stays usable.  Returns
 * QGEMV_OK, QGEMV_EINVAL (limit out of range), QGEMV_EDEVICE or
 * QGEMV_ELAUNCH.
 */
int qgemv_selftest_wait_timeout(unsigned limit_us, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int qgemv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H_ */
