// noalloc.cu -- moe_qgemv_combine_noalloc: the MoE expert matvec with
// combine for callers that cannot allocate device memory.
//
// moe_qgemv_combine needs a caller-provided fp32 workspace for the
// intermediate activations h_k.  Some callers have no way to provide one:
// a plugin inside a host application that owns every device allocation and
// exposes no allocator, or a latency-critical loop that is not allowed to
// allocate once it has started.  This entry point uses a fixed scratch array
// that lives in this library's device memory instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in, not a device address, so the device address is taken
// with cudaGetSymbolAddress once per device (with that device current) and
// then passed to the kernels like any workspace.
#include <atomic>

#include "qgemv.h"
#include "qgemv_args.h"

namespace {

// Scratch for h_k: top_k * I fp32 values at most.
__device__ __align__(256) float g_moe_scratch[QGEMV_NOALLOC_MAX_SCRATCH];

constexpr int kMaxDevices = 64;
std::atomic<float*> g_scratch_addr[kMaxDevices];

// Device address of g_moe_scratch on the current device; looked up once per
// device.  Returns nullptr if the lookup fails.
float* scratch_on_current_device(int* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = QGEMV_EDEVICE;
    return nullptr;
  }
  float* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  void* addr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&addr, g_moe_scratch);
  if (e != cudaSuccess || addr == nullptr) {
    *status = QGEMV_EDEVICE;
    return nullptr;
  }
  p = static_cast<float*>(addr);
  g_scratch_addr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" {

size_t qgemv_noalloc_max_scratch(void) {
  return static_cast<size_t>(QGEMV_NOALLOC_MAX_SCRATCH) * sizeof(float);
}

int moe_qgemv_combine_noalloc(const uint32_t* gu_codes, const uint16_t* gu_scales,
                              const uint16_t* gu_biases, const uint32_t* dn_codes,
                              const uint16_t* dn_scales, const uint16_t* dn_biases,
                              int n_experts, int H, int I, const int32_t* expert_idx,
                              const float* expert_w, int top_k, const uint16_t* x,
                              const uint16_t* residual, uint16_t* y, int* err_flag,
                              void* stream) {
  if (top_k < 1 || top_k > QGEMV_MAX_TOPK || I < 1) return QGEMV_EINVAL;
  if (static_cast<long long>(top_k) * I > QGEMV_NOALLOC_MAX_SCRATCH) return QGEMV_ESCRATCH;
  int status = QGEMV_OK;
  float* scratch = scratch_on_current_device(&status);
  if (scratch == nullptr) return status;
  return moe_qgemv_combine(gu_codes, gu_scales, gu_biases, dn_codes, dn_scales, dn_biases,
                           n_experts, H, I, expert_idx, expert_w, top_k, x, residual, y, scratch,
                           err_flag, stream);
}

}  // extern "C"
