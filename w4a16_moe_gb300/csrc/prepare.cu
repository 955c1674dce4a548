// Weight preparation: checkpoint layout -> serving layout of the GEMM kernels.
//
// flashinfer PR #4255, CodeRabbit walkthrough: ModelOpt / E8M0-K32
// preparation "with layout normalization, reusable buffers, scale packing, and
// W13 rotation"; the Tests section states preparation is bit-identical to its
// previous implementation.  Here the serving layout is this library's own:
//
// codes   [E][n_tiles][k_stages][chunk 0..1][row 0..127][16 bytes]
// scales  [E][n_tiles][k_stages][row 0..127][SB bytes]   SB = 4 (NVFP4), 2 (MXFP4)
//
// * a tile is 128 weight rows; a stage is 64 elements of K (two 16-byte
//   chunks of 32 codes per row), so each dequant thread reads its row's
//   chunk with one conflict-free 16-byte shared-memory load;
// * SwiGLU W13: tile t, row 32q + l holds gate row t*64 + 16q + l (l < 16)
//   or up row inter + t*64 + 16q + (l - 16) (l >= 16) -- gate and up rows of
//   the same output column sit 16 lanes apart in one warp ("W13 rotation");
// * rows and K are padded with zero codes and zero scales;
// * every 32-bit code word holds eight plain E2M1 nibbles (s, e1, e0, m) in
//   the order the hardware FP4 conversion pairs them: byte 0 holds elements 0
//   (low nibble) and 2, byte 1 elements 1 and 3, byte 2 elements 4 and 6,
//   byte 3 elements 5 and 7 (element e sits in nibble e with bits 0 and 1
//   swapped); the table-lookup dequantiser turns a word into its selectors
//   with one bit-pair exchange (dequant.cuh);
// * NVFP4 scales become b' with bf16 bits (b' << 4) + 0x5800 == scale * 2^63
//   (b' = 0 for a zero scale); MXFP4 keeps e, decoded as (e + 63) << 7;
// * a block with a zero scale stores zero codes; a negative E4M3 scale is
//   folded into the code signs.

#include "kernels.cuh"

namespace b4 {

__device__ __forceinline__ uint32_t src_code(const uint8_t* row, int k, int kvalid) {
  if (k >= kvalid) return 0;
  const uint8_t b = row[k >> 1];
  return (k & 1) ? (b >> 4) : (b & 0xF);
}

// E4M3 code -> serving byte b' (bf16 of scale * 2^63 == (b' << 4) + 0x5800).
// Returns -1 for NaN.  Sign handled by the caller.
__device__ __forceinline__ int nvfp4_scale_byte(uint32_t code) {
  const uint32_t mag = code & 0x7F;
  if (mag == 0x7F) return -1;
  if (mag == 0) return 0;
  if (mag >= 8) return (int)mag + 56;  // normal: exponent E + 183, mantissa m
  // subnormal m * 2^-9: renormalise
  static constexpr int sub[8] = {0, 40, 48, 52, 56, 58, 60, 62};
  return sub[mag];
}

__global__ void prepare_kernel(const __grid_constant__ PrepareParams p) {
  const TensorGeom g = tensor_geom(p.which, p.act, p.hidden, p.inter);
  const int group = p.fmt == 0 ? 16 : 32;
  const int SB = scale_bytes_per_row(p.fmt);
  const int src_kb = g.k_valid / group;  // scale blocks per source row
  const size_t total = (size_t)p.num_experts * g.n_tiles * g.k_stages * kTileRows;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx % kTileRows);
    size_t rest = idx / kTileRows;
    const int s = (int)(rest % g.k_stages);
    rest /= g.k_stages;
    const int t = (int)(rest % g.n_tiles);
    const int e = (int)(rest / g.n_tiles);

    int src_row;
    if (p.which == 0 && p.act == 0) {
      const int q = r >> 5, l = r & 31;
      const int i = t * 64 + q * 16 + (l & 15);
      src_row = i < p.inter ? (l < 16 ? i : p.inter + i) : -1;
    } else {
      const int n = t * kTileRows + r;
      src_row = n < g.rows_valid ? n : -1;
    }
    const uint8_t* crow =
        src_row >= 0 ? p.src_codes + ((size_t)e * g.rows_valid + src_row) * (g.k_valid / 2) : nullptr;
    const uint8_t* srow = src_row >= 0 ? p.src_scales + ((size_t)e * g.rows_valid + src_row) * src_kb : nullptr;

    // block scales of this stage
    const int nblk = kBK / group;  // 4 or 2
    uint32_t sbytes = 0;
    uint32_t flip = 0;    // per block: fold a negative scale into the code signs
    uint32_t zero = 0;    // per block: zero scale -> zero codes
    for (int b = 0; b < nblk; ++b) {
      const int kb = s * nblk + b;
      uint32_t out = 0;
      if (srow && kb < src_kb) {
        const uint32_t code = srow[kb];
        if (p.fmt == 0) {
          const int v = nvfp4_scale_byte(code);
          if (v < 0) {
            atomicAdd(p.bad, 1);
            zero |= 1u << b;
          } else {
            out = (uint32_t)v;
            if (v == 0) zero |= 1u << b;
            if (code & 0x80) flip |= 1u << b;
          }
        } else {
          out = code;
          bool any_nonzero = false;
          for (int k = kb * 32; k < kb * 32 + 32; ++k) any_nonzero |= (src_code(crow, k, g.k_valid) & 7) != 0;
          if (code >= 192 || (code < 65 && any_nonzero)) {
            atomicAdd(p.bad, 1);
            zero |= 1u << b;
            out = 127;
          }
        }
      } else {
        zero |= 1u << b;
      }
      sbytes |= out << (8 * b);
    }
    uint8_t* dsc = p.dst_scales + ((((size_t)e * g.n_tiles + t) * g.k_stages + s) * kTileRows + r) * SB;
    for (int b = 0; b < SB; ++b) dsc[b] = (uint8_t)(sbytes >> (8 * b));

    // 8 words of 8 codes each
    uint8_t* dco = p.dst_codes + (((size_t)e * g.n_tiles + t) * g.k_stages + s) * kCodeBytesPerStage;
    for (int q = 0; q < 8; ++q) {
      uint32_t word = 0;
      for (int el = 0; el < 8; ++el) {
        const int k = s * kBK + q * 8 + el;
        const int b = (k - s * kBK) / group;
        uint32_t c = crow ? src_code(crow, k, g.k_valid) : 0;
        if (zero & (1u << b)) c = 0;
        if (flip & (1u << b)) c ^= 8;
        const int nib = (el & 4) | ((el & 1) << 1) | ((el >> 1) & 1);  // bits 0 and 1 of el swapped
        word |= c << (4 * nib);
      }
      const int chunk = q >> 2, w4 = q & 3;
      *reinterpret_cast<uint32_t*>(dco + chunk * 2048 + r * 16 + w4 * 4) = word;
    }
  }
}

cudaError_t launch_prepare(const PrepareParams& p, int num_sms, cudaStream_t stream) {
  const TensorGeom g = tensor_geom(p.which, p.act, p.hidden, p.inter);
  const size_t total = (size_t)p.num_experts * g.n_tiles * g.k_stages * kTileRows;
  size_t blocks = (total + 255) / 256;
  if (blocks > (size_t)num_sms * 16) blocks = (size_t)num_sms * 16;
  if (blocks < 1) blocks = 1;
  prepare_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace b4
