// Streaming kernels: RMSNorm -> GEMV and gate.up SwiGLU (4-bit).
#include "qgemv_stream.cuh"

namespace qgemv {

cudaError_t stream_norm(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device) {
  return launch_stream<4, kNorm>(p, a, st, device);
}

cudaError_t stream_swiglu(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device) {
  return launch_stream<4, kSwiglu>(p, a, st, device);
}

cudaError_t status_norm_swiglu(unsigned* out) { return read_clear_status(out); }

}  // namespace qgemv
