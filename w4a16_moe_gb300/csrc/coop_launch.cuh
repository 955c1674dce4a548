// Cooperative launch of the small-m kernels, with programmatic dependent
// launch (PDL) on top when the device accepts the combination: the kernel's
// launch and CTA set-up then overlap the tail of the kernel before it in the
// stream.  The kernels wait (griddepcontrol.wait) before they read any input
// or write anything, so the result is the same either way.  Whether the
// device takes the pair is learned per device on the first launch outside a
// stream capture (a refused launch is an ordinary, non-sticky launch error);
// until then, and inside a capture, the launch is cooperative only.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace b4 {

inline int& coop_pdl_state(int dev) {
  static int state[64] = {};  // 0 unknown, 1 accepted, -1 refused
  static int other = -1;      // devices past 64: never tried
  return dev >= 0 && dev < 64 ? state[dev] : other;
}

template <typename Kernel, typename Params>
cudaError_t launch_cooperative(Kernel kern, int grid, int block, size_t smem, cudaStream_t stream,
                               const Params& p) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  int state;
  {
    std::lock_guard<std::mutex> lock(mu);
    state = coop_pdl_state(dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  const bool try_pdl = state == 1 || (state == 0 && cap == cudaStreamCaptureStatusNone && dev >= 0 && dev < 64);
  if (try_pdl) {
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (state == 1) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (e == cudaSuccess) {
      coop_pdl_state(dev) = 1;
      return e;
    }
    (void)cudaGetLastError();  // the refused launch enqueued nothing
    coop_pdl_state(dev) = -1;
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace b4
