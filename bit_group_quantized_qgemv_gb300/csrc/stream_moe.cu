// Streaming kernels: the two phases of the MoE expert matvec with combine.
#include "qgemv_stream.cuh"

namespace qgemv {

cudaError_t stream_moe_up(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device) {
  return launch_stream<4, kMoeUp>(p, a, st, device);
}

cudaError_t stream_moe_down(const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                            int device) {
  return launch_stream<4, kMoeDown>(p, a, st, device);
}

cudaError_t status_moe(unsigned* out) { return read_clear_status(out); }

}  // namespace qgemv
