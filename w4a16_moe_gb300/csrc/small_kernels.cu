// Small kernels of the grouped path of the fused W4A16 MoE layer: the copy of
// x rows into packed-route order (the FC1 B operand) and the final conversion
// of the fp32 top-k accumulator into the bf16 output.

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// --------------------------------------------------------- permute x rows
// xp[slot] = x[token of the route at packed slot], for the valid slots: the
// FC1 B operand becomes contiguous per expert chunk.  One warp per row, 16-byte
// copies, four loads in flight per lane before their stores (a store to a
// buffer that might alias the source keeps later loads behind it); slots past
// the valid count are left untouched (never loaded).
__global__ void permute_x_kernel(const __grid_constant__ GemmParams p) {
  constexpr int kLoads = 4;
  pdl_wait();  // sorted routes come from the route-pack kernel
  pdl_launch_dependents();
  const int valid = *p.valid_count;
  const int chunks = p.hidden / 8;  // 16-byte pieces of a row
  const int wpb = blockDim.x / 32;
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < valid; r += gridDim.x * wpb) {
    const int tok = __ldg(p.sorted_routes + r) / p.top_k;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)tok * p.hidden);
    uint4* dst = reinterpret_cast<uint4*>(p.xp + (size_t)r * p.hidden);
    for (int c = lane; c < chunks; c += 32 * kLoads) {
      uint4 v[kLoads];
#pragma unroll
      for (int k = 0; k < kLoads; ++k)
        if (c + 32 * k < chunks) v[k] = __ldg(src + c + 32 * k);
#pragma unroll
      for (int k = 0; k < kLoads; ++k)
        if (c + 32 * k < chunks) dst[c + 32 * k] = v[k];
    }
  }
}

cudaError_t launch_permute_x(const GemmParams& p, int num_sms, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * num_sms);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, permute_x_kernel, p);
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
