// Streaming kernels: plain 4-, 8- and 2-bit GEMV (optionally + residual), and
// the 4-bit GEMV with the index of its largest output (greedy lm_head).
#include "qgemv_stream.cuh"

namespace qgemv {

cudaError_t stream_plain(int bits, const StreamPlan& p, const StreamArgs& a, cudaStream_t st,
                         int device) {
  if (bits == 4) return launch_stream<4, kPlain>(p, a, st, device);
  if (bits == 8) return launch_stream<8, kPlain>(p, a, st, device);
  return launch_stream<2, kPlain>(p, a, st, device);
}

cudaError_t stream_argmax(const StreamPlan& p, const StreamArgs& a, cudaStream_t st, int device) {
  return launch_stream<4, kArgmax>(p, a, st, device);
}

cudaError_t status_plain(unsigned* out) { return read_clear_status(out); }

}  // namespace qgemv
