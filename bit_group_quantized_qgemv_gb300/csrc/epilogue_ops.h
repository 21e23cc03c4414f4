// epilogue_ops.h -- launch of the kernels that are not streaming kernels:
// the standalone epilogues (csrc/generic.cu), top-k sampling (csrc/sample.cu)
// and the LUT / palettised GEMV (csrc/lut.cu).  Host declarations only.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

// LUT / palettised 4-bit GEMV (csrc/lut.cu), M = 1: y[n] = sum_k
// lut[n / rows_per_lut][q[n][k]] x[k] (+ residual[n]); codes, lut and x
// 16-byte aligned; K a multiple of 64, at most 16384.  Chained by
// programmatic dependent launch.
cudaError_t lut_qgemv_launch(const uint32_t* codes, const uint16_t* lut, int rows_per_lut,
                             const __half* x, const __half* residual, __half* y, int N, int K,
                             int sms, cudaStream_t st);

}  // namespace qgemv
