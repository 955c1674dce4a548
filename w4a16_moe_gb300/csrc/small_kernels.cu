// Small kernels of the fused W4A16 MoE layer: the final top-k combine into
// the bf16 output, for the grouped path (fp32 accumulator -> bf16) and the
// decode path (sum of the FC2 split-K partials of a token's routes -> bf16).

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}


// ------------------------------------------------------------- finalize
// Grouped: out = bf16(acc).  Decode: out[t, n] = bf16(sum_j sum_split q).
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

__global__ void finalize_decode_kernel(const __grid_constant__ FinalizeParams p) {
  // a block handles 256 consecutive outputs of one token; the token's routes
  // are resolved once into shared memory, then every partial load is independent
  __shared__ int s_valid[32];
  pdl_wait();
  const int R = p.m * p.top_k;
  const int blocks_per_token = cdiv(p.hidden, 256);
  for (int b = blockIdx.x; b < p.m * blocks_per_token; b += gridDim.x) {
    const int t = b / blocks_per_token;
    const int n = (b - t * blocks_per_token) * 256 + threadIdx.x;
    __syncthreads();
    if (threadIdx.x < p.top_k) {
      const int id = p.topk_ids[t * p.top_k + threadIdx.x];
      int ok = id >= 0 && id < p.num_global_experts;
      if (ok) {
        const int l = p.expert_map ? p.expert_map[id] : id;
        ok = l >= 0 && l < p.num_local_experts;
      }
      s_valid[threadIdx.x] = ok;
    }
    __syncthreads();
    if (n >= p.hidden) continue;
    float acc = 0.f;
    for (int j = 0; j < p.top_k; ++j) {
      if (!s_valid[j]) continue;
      const float* q = p.q + (size_t)(t * p.top_k + j) * p.hidden + n;
      for (int sp = 0; sp < p.splits; ++sp) acc += q[(size_t)sp * R * p.hidden];
    }
    p.out[(size_t)t * p.hidden + n] = float_to_bf16_bits(acc);
  }
}

cudaError_t launch_finalize(const FinalizeParams& p, bool grouped, int num_sms, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  const size_t total = grouped ? (size_t)p.m * p.hidden / 4 : (size_t)p.m * cdiv(p.hidden, 256) * 256;
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
  return grouped ? cudaLaunchKernelEx(&cfg, finalize_grouped_kernel, p)
                 : cudaLaunchKernelEx(&cfg, finalize_decode_kernel, p);
}

}  // namespace b4
