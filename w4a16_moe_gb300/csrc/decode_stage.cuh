// The decode path's per-thread stage arithmetic: 64 K elements of two weight
// rows dequantised in registers and multiplied with the activation slice on
// warp-level m16n8k16 bf16 MMAs (layout notes in decode_moe.cu).
#pragma once

#include <cstdint>

#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 block-scale multiplier of a serving scale byte, in one IMAD:
// NVFP4 bits (b << 4) + 0x5800 (= E4M3 value * 2^63), MXFP4 bits (b + 63) << 7
// (= 2^(e-127) * 2^63), in both halves.
template <int FMT>
__device__ __forceinline__ uint32_t d_scale(uint32_t b) {
  return FMT == 0 ? b * 0x00100010u + 0x58005800u : b * 0x00800080u + 0x1F801F80u;
}

// One thread's operands of one 64-wide stage: 8 code bytes (block t) of rows
// r0 and r1, their two scale bytes, and the 16 activations of block t.
struct StageIn {
  uint2 c0, c1;
  uint32_t b0, b1;
  uint4 xa, xb;
};

template <int SB>
__device__ __forceinline__ void load_stage(StageIn& in, const uint8_t* cs, const uint8_t* ss, const uint8_t* xr) {
  in.c0 = *reinterpret_cast<const uint2*>(cs);
  in.c1 = *reinterpret_cast<const uint2*>(cs + 8 * 16);
  in.b0 = ss[0];
  in.b1 = ss[8 * SB];
  in.xa = *reinterpret_cast<const uint4*>(xr);
  in.xb = *reinterpret_cast<const uint4*>(xr + 16);
}

// Dequantise the stage's 2 x 16 weights and run its four m16n8k16 MMAs
// (pairs 2j, 2j+1 of block t feed MMA j) into two accumulators.
template <int FMT>
__device__ __forceinline__ void compute_stage(const StageIn& in, float (&d)[4], float (&e)[4]) {
  const uint32_t sa = d_scale<FMT>(in.b0), sb = d_scale<FMT>(in.b1);
  uint32_t a0[8], a1[8];
  fp4x8_lookup(in.c0.x, a0[0], a0[1], a0[2], a0[3]);
  fp4x8_lookup(in.c0.y, a0[4], a0[5], a0[6], a0[7]);
  fp4x8_lookup(in.c1.x, a1[0], a1[1], a1[2], a1[3]);
  fp4x8_lookup(in.c1.y, a1[4], a1[5], a1[6], a1[7]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a0[i] = bf16x2_mul(a0[i], sa);
    a1[i] = bf16x2_mul(a1[i], sb);
  }
  mma_16816(d, a0[0], a1[0], a0[1], a1[1], in.xa.x, in.xa.y);
  mma_16816(e, a0[2], a1[2], a0[3], a1[3], in.xa.z, in.xa.w);
  mma_16816(d, a0[4], a1[4], a0[5], a1[5], in.xb.x, in.xb.y);
  mma_16816(e, a0[6], a1[6], a0[7], a1[7], in.xb.z, in.xb.w);
}

}  // namespace b4
