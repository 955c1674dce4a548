// E2M1 x block-scale dequantisation to bf16 in registers (sm_103a).
//
// Shared by the GEMM kernels and the route-grouped small-m kernel; it reads
// the prepared layout that the prepare kernel writes (prepare.cu).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace b4 {

// One thread, one weight row, one 64-element stage: 32 bytes of prepared
// codes (two 16-byte chunks) and the re-encoded block scales -> 32 registers
// of packed bf16 pairs (column c holds elements 2c, 2c+1).
//
// A prepared code word holds eight plain E2M1 nibbles (s, e1, e0, m), byte 0
// elements 0 and 2, byte 1 elements 1 and 3, byte 2 elements 4 and 6, byte 3
// elements 5 and 7 (prepare.cu).  Exchanging bit pairs (2,3) and (4,5) of
// every byte gives the selector form: pair j of the word (elements 2j, 2j+1)
// at shift {0, 2, 16, 18}[j], the low element with (e0, m) at bits [1:0] and
// (s, e1) at [5:4], the high element at [9:8] and [13:12].  With 0x4040
// or-ed in, those 16 bits are a PRMT selector whose byte lookups in the table
// {00,40,80,C0 | 00,01,80,81} assemble the bf16 bit pattern
// s<<15 | e1<<8 | e0<<7 | m<<6 of each element: the E2M1 value times 2^-126.
// One bf16x2 multiply by (scale * 2^63) then yields value * scale * 2^-63.
__device__ __forceinline__ uint32_t nibbles_to_selectors(uint32_t v) {
  const uint32_t t = (v ^ (v >> 2)) & 0x0C0C0C0Cu;
  return v ^ t ^ (t << 2);
}

// The four pairs of one prepared code word, with the selectors formed on all
// 32 bits at once: after the exchange, (v & 0x33333333) | 0x40404040 holds
// the selectors of pairs 0 (low half) and 2 (high half), the same of v >> 2
// those of pairs 1 and 3, and a PRMT reads only the low 16 bits of its
// selector.
__device__ __forceinline__ void fp4x8_lookup(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  const uint32_t v = nibbles_to_selectors(w);
  const uint32_t s = (v & 0x33333333u) | 0x40404040u;
  const uint32_t t = ((v >> 2) & 0x33333333u) | 0x40404040u;
  p0 = __byte_perm(0xC0804000u, 0x81800100u, s);
  p1 = __byte_perm(0xC0804000u, 0x81800100u, t);
  p2 = __byte_perm(0xC0804000u, 0x81800100u, s >> 16);
  p3 = __byte_perm(0xC0804000u, 0x81800100u, t >> 16);
}

template <int FMT>
__device__ __forceinline__ void dequant_stage(const uint4& c0, const uint4& c1, uint32_t sc, uint32_t (&r)[32]) {
  uint32_t s[4];
  if constexpr (FMT == 0) {
    // NVFP4: byte b' -> bf16 bits (b' << 4) + 0x5800 == E4M3 value * 2^63
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t bits = (((sc >> (8 * b)) & 0xFFu) << 4) + 0x5800u;
      s[b] = bits * 0x10001u;
    }
  } else {
    // MXFP4: E8M0 e -> bf16 bits (e + 63) << 7 == 2^(e-127) * 2^63
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t bits = (((sc >> (8 * b)) & 0xFFu) + 63u) << 7;
      s[b] = bits * 0x10001u;
    }
    s[2] = s[3] = 0;
  }
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t sq = FMT == 0 ? s[q >> 1] : s[q >> 2];
    uint32_t p0, p1, p2, p3;
    fp4x8_lookup(w[q], p0, p1, p2, p3);
    r[4 * q + 0] = bf16x2_mul(p0, sq);
    r[4 * q + 1] = bf16x2_mul(p1, sq);
    r[4 * q + 2] = bf16x2_mul(p2, sq);
    r[4 * q + 3] = bf16x2_mul(p3, sq);
  }
}

// Half a stage of one row: the 16-byte chunk `half` (32 elements) -> 16
// registers of packed bf16 pairs, scaled by the row's block scales `sc` (as
// in dequant_stage).
template <int FMT>
__device__ __forceinline__ void dequant_half(const uint4& c, uint32_t sc, int half, uint32_t (&r)[16]) {
  uint32_t s0, s1;
  if constexpr (FMT == 0) {
    s0 = ((((sc >> (16 * half)) & 0xFFu) << 4) + 0x5800u) * 0x10001u;
    s1 = ((((sc >> (16 * half + 8)) & 0xFFu) << 4) + 0x5800u) * 0x10001u;
  } else {
    s0 = s1 = ((((sc >> (8 * half)) & 0xFFu) + 63u) << 7) * 0x10001u;
  }
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t sq = q < 2 ? s0 : s1;
    uint32_t p0, p1, p2, p3;
    fp4x8_lookup(w[q], p0, p1, p2, p3);
    r[4 * q + 0] = bf16x2_mul(p0, sq);
    r[4 * q + 1] = bf16x2_mul(p1, sq);
    r[4 * q + 2] = bf16x2_mul(p2, sq);
    r[4 * q + 3] = bf16x2_mul(p3, sq);
  }
}

}  // namespace b4
