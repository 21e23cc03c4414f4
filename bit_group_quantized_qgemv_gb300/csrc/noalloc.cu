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
// with cudaGetSymbolAddress once per device and context (with that device
// current) and then passed to the kernels like any workspace.
#include <cuda.h>

#include <mutex>

#include "qgemv.h"
#include "qgemv_args.h"

namespace {

// Scratch for h_k: top_k * I fp32 values at most.
__device__ __align__(256) float g_moe_scratch[QGEMV_NOALLOC_MAX_SCRATCH];

constexpr int kMaxDevices = 64;

// Per device: the context the address was looked up in (its process-unique
// id from cuCtxGetId; 0 = none yet) and the array's device address there.
// A cudaDeviceReset destroys the context and unloads this library's device
// module; the next call runs in a new context with a new id, so the address
// is looked up again instead of reusing the old one.
struct ScratchSlot {
  unsigned long long ctx_id = 0;
  float* addr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_slots_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's cuCtxGetCurrent and cuCtxGetId, through the runtime (the
// library does not link the driver library itself); looked up once,
// thread-safely.
bool driver_ctx_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  struct Fns {
    CtxGetCurrentFn cur = nullptr;
    CtxGetIdFn id = nullptr;
  };
  static const Fns fns = [] {
    Fns r;
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault,
                                         &q0) == cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q0 == cudaDriverEntryPointSuccess && q1 == cudaDriverEntryPointSuccess && f0 && f1) {
      r.cur = reinterpret_cast<CtxGetCurrentFn>(f0);
      r.id = reinterpret_cast<CtxGetIdFn>(f1);
    } else {
      cudaGetLastError();
    }
    return r;
  }();
  if (fns.cur == nullptr || fns.id == nullptr) return false;
  *cur = fns.cur;
  *id = fns.id;
  return true;
}

// Id of the calling thread's current context, 0 if there is none yet.
unsigned long long current_ctx_id(CtxGetCurrentFn cur, CtxGetIdFn id) {
  CUcontext ctx = nullptr;
  unsigned long long v = 0;
  if (cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (id(ctx, &v) != CUDA_SUCCESS) return 0;
  return v;
}

// Device address of g_moe_scratch in the current context of the current
// device.  The address is looked up (cudaGetSymbolAddress, with the device
// current) on the first call on each device and again after that device's
// context has changed; otherwise the cached value is returned.  Returns
// nullptr (status QGEMV_EDEVICE) if no address can be had.
float* scratch_on_current_device(int* status) {
  *status = QGEMV_EDEVICE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrentFn cur = nullptr;
  CtxGetIdFn id = nullptr;
  if (!driver_ctx_fns(&cur, &id)) return nullptr;
  std::lock_guard<std::mutex> lock(g_slots_mu);
  unsigned long long ctx = current_ctx_id(cur, id);
  ScratchSlot& slot = g_slots[dev];
  if (ctx != 0 && slot.ctx_id == ctx && slot.addr != nullptr) {
    *status = QGEMV_OK;
    return slot.addr;
  }
  void* addr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&addr, g_moe_scratch);
  if (e != cudaSuccess || addr == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  // The lookup makes the device's primary context current if no context was.
  ctx = current_ctx_id(cur, id);
  if (ctx == 0) return nullptr;
  slot.ctx_id = ctx;
  slot.addr = static_cast<float*>(addr);
  *status = QGEMV_OK;
  return slot.addr;
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
  // Null pointers and shapes first, with the statuses of moe_qgemv_combine,
  // then the scratch capacity; alignment is checked by moe_qgemv_combine.
  if (!gu_codes || !gu_scales || !gu_biases || !dn_codes || !dn_scales || !dn_biases ||
      !expert_idx || !expert_w || !x || !y)
    return QGEMV_ENULL;
  if (n_experts < 1 || top_k < 1 || top_k > QGEMV_MAX_TOPK || H < 64 || H % 64 != 0 || I < 64 ||
      I % 64 != 0)
    return QGEMV_EINVAL;
  if (static_cast<long long>(top_k) * I > QGEMV_NOALLOC_MAX_SCRATCH) return QGEMV_ESCRATCH;
  int status = QGEMV_OK;
  float* scratch = scratch_on_current_device(&status);
  if (scratch == nullptr) return status;
  return moe_qgemv_combine(gu_codes, gu_scales, gu_biases, dn_codes, dn_scales, dn_biases,
                           n_experts, H, I, expert_idx, expert_w, top_k, x, residual, y, scratch,
                           err_flag, stream);
}

}  // extern "C"
