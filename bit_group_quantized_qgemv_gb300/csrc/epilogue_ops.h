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

}  // namespace qgemv
