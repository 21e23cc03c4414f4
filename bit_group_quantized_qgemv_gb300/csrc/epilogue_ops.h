// epilogue_ops.h -- launch of the standalone epilogue kernels (csrc/generic.cu)
// that are not streaming kernels.  Host declarations only.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qgemv {

// h = x + r (fp16, one rounding), xn = RMSNorm(h) * gamma (fp16); one CTA,
// chained by programmatic dependent launch; r may be null (h = x, unstored).
cudaError_t residual_rmsnorm_launch(const __half* x, const __half* r, const __half* gamma,
                                    float eps, int K, __half* h, __half* xn, cudaStream_t st);

// Top-k sampling from fp16 logits (csrc/sample.cu): one cluster of 8 CTAs,
// chained by programmatic dependent launch.  1 <= top_k <= min(n,
// kMaxSampleK), n <= kMaxSampleN, temperature > 0; u is read on the device.
// token = the pick; out_idx / out_prob (nullable) = the k candidates in
// decreasing order and their normalised weights.
constexpr int kMaxSampleK = 1024;       // QGEMV_SAMPLE_MAX_K
constexpr int kMaxSampleSlice = 98304;  // logits held by one CTA
constexpr int kMaxSampleN = 8 * kMaxSampleSlice;  // QGEMV_SAMPLE_MAX_N
cudaError_t sample_topk_launch(const __half* logits, int n, int top_k, float temperature,
                               const float* u, int* token, int* out_idx, float* out_prob,
                               cudaStream_t st);

}  // namespace qgemv
