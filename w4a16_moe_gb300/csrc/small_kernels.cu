// Small kernels of the grouped path of the fused W4A16 MoE layer: the final
// conversion of the fp32 top-k accumulator into the bf16 output (the copy of x
// rows into packed-route order is part of the route pack, route_pack.cu).

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------- finalize
// out = bf16(acc).  Each thread loads four float4s before it stores any: the
// compiler cannot move a load above a store to a buffer that might alias it,
// so one load per store would wait one round trip each.
__global__ void finalize_grouped_kernel(const __grid_constant__ FinalizeParams p) {
  constexpr int kLoads = 4;
  pdl_wait();
  const size_t n4 = (size_t)p.m * p.hidden / 4;  // H is a multiple of 64
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const float4* acc = reinterpret_cast<const float4*>(p.acc);
  ushort4* out = reinterpret_cast<ushort4*>(p.out);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += kLoads * stride) {
    float4 a[kLoads];
#pragma unroll
    for (int k = 0; k < kLoads; ++k)
      if (i + k * stride < n4) a[k] = acc[i + k * stride];
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      if (i + k * stride >= n4) break;
      ushort4 o;
      o.x = float_to_bf16_bits(a[k].x);
      o.y = float_to_bf16_bits(a[k].y);
      o.z = float_to_bf16_bits(a[k].z);
      o.w = float_to_bf16_bits(a[k].w);
      out[i + k * stride] = o;
    }
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
