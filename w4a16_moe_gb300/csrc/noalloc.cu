// b4_fused_moe_noalloc: the fused layer for callers that cannot allocate.
//
// A plugin hook of an inference runtime, or a custom-op slot of a framework,
// is handed only its input and output buffers.  The host's own allocator owns
// all device memory there: a cudaMalloc from inside the hook would stall the
// whole device on the serving path and escape the host's accounting, so such
// hooks must not allocate, and they have no workspace to pass to
// b4_fused_moe.  This entry point runs the same kernels as b4_fused_moe with
// their scratch taken from one fixed array that this file declares in device
// memory.  The library never calls cudaMalloc, cudaFree or any allocating
// routine for it: the CUDA runtime places the array when it loads this
// library's device code onto a GPU, and the array stays there until the
// process exits.

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "b4moe.h"

namespace b4 {
void set_last_error(const char* fmt, ...);
}

// The scratch array.  In host code this name is only a host-side stand-in for
// the symbol, never a device address: the address a kernel may use comes from
// cudaGetSymbolAddress, per device and context, below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[B4_NOALLOC_SCRATCH_BYTES];

namespace {

// Driver entry points for the identity of the current context, fetched through
// the runtime (the library links no libcuda).  cuCtxGetId gives every context
// a process-unique id, so a context that replaced an earlier one (after a
// cudaDeviceReset, or a teardown and re-creation of the primary context) has
// a new id even where the driver reuses the old handle.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(p);
  return nullptr;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  unsigned long long ctx_id;
  void* addr;
};
Cached g_cache[kMaxDevices] = {};

// Device address of g_noalloc_scratch in the context now current on this
// device.  Set-up: the first call in each context (per device) looks the
// address up with cudaGetSymbolAddress, which allocates nothing but may load
// this library's device code into that context; later calls in the same
// context reuse it.  A new context (after cudaDeviceReset or a primary-context
// teardown) has a new id, so its first call looks the address up again and a
// stale address is never passed to a kernel.
b4_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    b4::set_last_error("b4_fused_moe_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    return B4_ERR_CUDA;
  }
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  auto current_id = [&](unsigned long long* id) {
    CUcontext ctx = nullptr;
    return dev >= 0 && dev < kMaxDevices && get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
           get_id(ctx, id) == CUDA_SUCCESS;
  };
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = 0;
  if (current_id(&id) && g_cache[dev].addr && g_cache[dev].ctx_id == id) {
    *out = g_cache[dev].addr;
    return B4_OK;
  }
  // (the lookup also binds the device's primary context when none is current yet)
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    b4::set_last_error("b4_fused_moe_noalloc: cudaGetSymbolAddress of the static scratch failed on device %d: %s",
                       dev, cudaGetErrorString(e));
    return B4_ERR_CUDA;
  }
  if (current_id(&id)) g_cache[dev] = Cached{id, p};  // without a context id, look up on every call
  *out = p;
  return B4_OK;
}

}  // namespace

extern "C" b4_status b4_fused_moe_noalloc(const b4_moe_config* cfg, const uint16_t* x, const uint8_t* w13,
                                          const uint8_t* s13, const float* gs13, const uint8_t* w2,
                                          const uint8_t* s2, const float* gs2, const int32_t* topk_ids,
                                          const float* topk_weights, int32_t activation, uint16_t* out,
                                          uint32_t* device_status, b4_stream_t stream) {
  // shape validation and the size check come first, so an oversized shape is
  // refused without touching any device
  const size_t need = b4_workspace_bytes(cfg, activation);
  if (need == 0) return B4_ERR_INVALID_ARGUMENT;  // b4_last_error already says why
  if (need > B4_NOALLOC_SCRATCH_BYTES) {
    b4::set_last_error(
        "b4_fused_moe_noalloc: this shape needs %zu bytes of scratch, more than the static array's %zu "
        "(B4_NOALLOC_SCRATCH_BYTES); call b4_fused_moe with a workspace instead",
        need, (size_t)B4_NOALLOC_SCRATCH_BYTES);
    return B4_ERR_WORKSPACE_TOO_SMALL;
  }
  if (device_status && reinterpret_cast<uintptr_t>(device_status) % 4) {
    b4::set_last_error("b4_fused_moe_noalloc: device_status must be 4-byte aligned");
    return B4_ERR_INVALID_ARGUMENT;
  }
  void* scratch = nullptr;
  b4_status st = scratch_address(&scratch);
  if (st != B4_OK) return st;
  // Every scratch region is written before it is read within one call (the
  // status word by the first kernel, the fp32 top-k accumulator by FC1 before
  // FC2 adds into it), so what the previous call left behind is never read.
  st = b4_fused_moe(cfg, x, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights, activation, out, scratch,
                    B4_NOALLOC_SCRATCH_BYTES, stream);
  if (st != B4_OK || !device_status) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // m == 0 launches nothing, so there is no status word of this call to copy
  const cudaError_t e = cfg->m == 0 ? cudaMemsetAsync(device_status, 0, 2 * sizeof(uint32_t), s)
                                    : cudaMemcpyAsync(device_status, scratch, 2 * sizeof(uint32_t),
                                                      cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) {
    b4::set_last_error("b4_fused_moe_noalloc: status copy failed: %s", cudaGetErrorString(e));
    return B4_ERR_CUDA;
  }
  return B4_OK;
}
