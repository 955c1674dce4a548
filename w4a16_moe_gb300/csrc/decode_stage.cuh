// The small-m kernels' per-thread stage arithmetic: weight rows dequantised in
// registers and multiplied with the activation slice on warp-level m16n8k16
// MMAs.  Here: the bf16 MMA and block-scale multiplier the route-grouped
// kernel feeds from the register table lookup (dequant.cuh), and the
// per-route kernel's stage: hardware FP4 conversion with f16 MMAs and
// block-diagonal activations.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

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

// ------------------------------------------------------------------ f16 stage
// The per-route small-m kernel's dequantiser: E2M1 codes are converted by the hardware
// FP4 conversion (two codes of one byte -> one f16x2, exact), the weight
// operand of f16 m16n8k16 MMAs.  The activation operand is block diagonal:
// MMA column c is nonzero only for the K positions of block c, so after the
// eight MMAs of a 128-wide slot column c holds the unscaled sum of block c,
// and the block scale (and the activations' power-of-two prescale) is applied
// to that fp32 sum.  Activations are converted to f16 after a prescale by a
// power of two per 128-wide slot, chosen so the slot's largest magnitude lands
// in [2^14, 2^15): every bf16 value within 2^24 of it is exact in f16.

// A prepared code word (prepare.cu): four bytes of two plain E2M1 nibbles
// each, byte 0 holding elements 0 (low nibble) and 2, byte 1 elements 1 and 3,
// byte 2 elements 4 and 6, byte 3 elements 5 and 7 -> four f16x2 (low nibble
// -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t v, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                                uint32_t& h3) {
  asm("{\n .reg .b8 c0, c1, c2, c3;\n mov.b32 {c0, c1, c2, c3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, c0;\n cvt.rn.f16x2.e2m1x2 %1, c1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, c2;\n cvt.rn.f16x2.e2m1x2 %3, c3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(v));
}

__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Power-of-two prescale exponent of a slot of activations whose largest
// magnitude is amax (>= 0, possibly Inf): the slot is multiplied by 2^-e.
__device__ __forceinline__ int slot_prescale(float amax) {
  const int E = (int)(__float_as_uint(amax) >> 23) - 127;  // floor(log2) for normal amax
  const int e = E - 14;
  return e < -110 ? -110 : e;
}
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// One lane's four activations of a slot, (v0, v1, v2, v3) = K positions
// 4l .. 4l+3, scaled by 2^-e and stored as f16 in the order the weight bytes
// pair them: (v0, v2) then (v1, v3).
__device__ __forceinline__ void store_x4_f16(uint8_t* dst, float v0, float v1, float v2, float v3, int e) {
  const float f = pow2_neg(e);
  const __half2 lo = __floats2half2_rn(v0 * f, v2 * f);
  const __half2 hi = __floats2half2_rn(v1 * f, v3 * f);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&lo);
  w.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = w;
}

// The f16 weight operand of one 64-wide stage for rows (r0, r0 + 8): codes
// w0 (row r0, elements 0..7 and 8..15 of this thread's block) and w1 (row r1).
struct F16Stage {
  uint32_t a[4], b[4], c[4], d[4];
};
__device__ __forceinline__ void dequant_stage_f16(const uint2& w0, const uint2& w1, F16Stage& f) {
  e2m1x8_to_f16x2(w0.x, f.a[0], f.a[1], f.a[2], f.a[3]);
  e2m1x8_to_f16x2(w1.x, f.b[0], f.b[1], f.b[2], f.b[3]);
  e2m1x8_to_f16x2(w0.y, f.c[0], f.c[1], f.c[2], f.c[3]);
  e2m1x8_to_f16x2(w1.y, f.d[0], f.d[1], f.d[2], f.d[3]);
}

// The four MMAs of one stage against the activation slices at bp (quarters
// q = 0..3, 8 bytes each; zeros for a thread whose column is not this
// stage's block).  Even quarters accumulate into de, odd into dq.
__device__ __forceinline__ void mma_stage_f16(const F16Stage& f, const uint8_t* bp, float (&de)[4], float (&dq)[4]) {
  const uint4 x01 = *reinterpret_cast<const uint4*>(bp);
  const uint4 x23 = *reinterpret_cast<const uint4*>(bp + 16);
  mma_16816_f16(de, f.a[0], f.b[0], f.a[1], f.b[1], x01.x, x01.y);
  mma_16816_f16(dq, f.a[2], f.b[2], f.a[3], f.b[3], x01.z, x01.w);
  mma_16816_f16(de, f.c[0], f.d[0], f.c[1], f.d[1], x23.x, x23.y);
  mma_16816_f16(dq, f.c[2], f.d[2], f.c[3], f.d[3], x23.z, x23.w);
}

__device__ __forceinline__ void stage_mma_f16(const uint2& w0, const uint2& w1, const uint8_t* bp, float (&de)[4],
                                              float (&dq)[4]) {
  F16Stage f;
  dequant_stage_f16(w0, w1, f);
  mma_stage_f16(f, bp, de, dq);
}

// fp32 block scale of a prepared scale byte b, times 2^xe (the activations'
// prescale): NVFP4 bits b * 2^20 + 0x38800000 are the E4M3 value, MXFP4 bits
// b << 23 are 2^(b - 127).
template <int FMT>
__device__ __forceinline__ float f32_scale(uint32_t b, int xe) {
  return FMT == 0 ? __uint_as_float(b * 0x100000u + 0x38800000u + ((uint32_t)xe << 23))
                  : __uint_as_float(b * 0x800000u + ((uint32_t)xe << 23));
}

}  // namespace b4
