// Small kernels of the fused W4A16 MoE layer: the final conversion of the
// grouped path's fp32 top-k accumulator into the bf16 output.

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}


// ------------------------------------------------------------- finalize
// out = bf16(acc)
__global__ void finalize_grouped_kernel(const __grid_constant__ FinalizeParams p) {
  pdl_wait();
  const size_t total = (size_t)p.m * p.hidden;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i * 4 < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(p.acc)[i];
    ushort4 o;
    o.x = float_to_bf16_bits(a.x);
    o.y = float_to_bf16_bits(a.y);
    o.z = float_to_bf16_bits(a.z);
    o.w = float_to_bf16_bits(a.w);
    reinterpret_cast<ushort4*>(p.out)[i] = o;
  }
}

cudaError_t launch_finalize(const FinalizeParams& p, int num_sms, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  const size_t total = (size_t)p.m * p.hidden / 4;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 4 * num_sms) blocks = 4 * num_sms;
  if (blocks < 1) blocks = 1;
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, finalize_grouped_kernel, p);
}

}  // namespace b4
