// Test-only probes of the library's device building blocks (not part of
// libb4moe): a single tcgen05.mma with A in tensor memory and B in the
// library's shared-memory layout, and a dump of the register dequantiser.
// They pin the layout assumptions the GEMM kernel is built on.
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_stage.cuh"
#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tma.cuh"

using namespace b4;

// D[128][N] = A[128][64] x B[N][64]^T, A via tcgen05.st into TMEM, B in the
// no-swizzle K-major core-matrix layout (LBO 128 B, SBO 1024 B), four K=16
// MMAs, one commit.
__global__ void probe_mma_kernel(const uint16_t* A, const uint16_t* B, int N, float* D, uint32_t* status) {
  __shared__ __align__(1024) uint8_t sB[256 * 128];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  const Abort ab{status, &abort_flag};
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem, 512);
    tmem_relinquish();
  }
  for (int idx = tid; idx < N * 8; idx += blockDim.x) {
    const int n = idx >> 3, kc = idx & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(B + n * 64 + kc * 8);
    *reinterpret_cast<uint4*>(sB + (n >> 3) * 1024 + kc * 128 + (n & 7) * 16) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t base = tmem;
  uint32_t r[32];
  for (int c = 0; c < 32; ++c) r[c] = (uint32_t)A[tid * 64 + 2 * c] | ((uint32_t)A[tid * 64 + 2 * c + 1] << 16);
  tmem_st32(base + ((uint32_t)(32 * warp) << 16), r);
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_m128((uint32_t)N);
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16_ts(base + 128, base + kk * 8, smem_desc_noswizzle(smem_u32(sB) + kk * 256, 128, 1024), idesc,
                  kk > 0 ? 1u : 0u);
    mma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, ab, 100);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(base + ((uint32_t)(32 * warp) << 16) + 128 + c0, v);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j) D[tid * N + c0 + j] = __uint_as_float(v[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(base, 512);
}

// D[128][16] = A[128][64] x B^T where B's row 0 is the contiguous 64-element
// row `x` held in natural order and the descriptor uses a 16-byte K stride and
// a zero N stride (the decode path's single-row B operand).  Rows 1..15 of B
// then read shifted / repeated data: only column 0 (and its copy, column 8)
// is meaningful.
__global__ void probe_mma_rowb_kernel(const uint16_t* A, const uint16_t* x, float* D, uint32_t* status) {
  __shared__ __align__(1024) uint8_t sB[128 + 256];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  const Abort ab{status, &abort_flag};
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem, 256);
    tmem_relinquish();
  }
  for (int i = tid; i < (128 + 256) / 2; i += blockDim.x)
    reinterpret_cast<uint16_t*>(sB)[i] = i < 64 ? x[i] : (uint16_t)0x7FC0;  // NaN slack
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t base = tmem;
  uint32_t r[32];
  for (int c = 0; c < 32; ++c) r[c] = (uint32_t)A[tid * 64 + 2 * c] | ((uint32_t)A[tid * 64 + 2 * c + 1] << 16);
  tmem_st32(base + ((uint32_t)(32 * warp) << 16), r);
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_m128(16);
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16_ts(base + 128, base + kk * 8, smem_desc_noswizzle(smem_u32(sB) + kk * 32, 16, 0), idesc,
                  kk > 0 ? 1u : 0u);
    mma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, ab, 101);
  tc_fence_after();
  if (ok) {
    uint32_t v[16];
    tmem_ld16(base + ((uint32_t)(32 * warp) << 16) + 128, v);
    tmem_ld_wait();
    for (int j = 0; j < 16; ++j) D[tid * 16 + j] = __uint_as_float(v[j]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(base, 256);
}

// TMA probes: a 2-D tile box and a gather4 (4 rows) into 128-byte-swizzled
// shared memory, dumped raw so the test can check the swizzle pattern.
__global__ void probe_tma_kernel(const __grid_constant__ CUtensorMap tm, int mode, int c0, int r0, int r1, int r2,
                                 int r3, int box_rows, int dst_off, uint8_t* out, uint32_t* status) {
  __shared__ __align__(1024) uint8_t s[256 * 128];
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const Abort ab{status, &abort_flag};
  const int tid = threadIdx.x;
  for (int i = tid; i < 256 * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(s)[i] = 0xA5A5A5A5u;
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    if (mode == 0) {
      mbar_arrive_expect_tx(&bar, (uint32_t)box_rows * 128);
      tma_load_2d(s + dst_off, &tm, c0, r0, &bar);
    } else {
      mbar_arrive_expect_tx(&bar, 4 * 128);
      tma_gather4(s + dst_off, &tm, c0, r0, r1, r2, r3, &bar);
    }
  }
  const bool ok = mbar_wait(&bar, 0, ab, 110);
  __syncthreads();
  if (ok)
    for (int i = tid; i < 256 * 128; i += blockDim.x) out[i] = s[i];
}

// D[128][N] = A[128][64] x B[N][64]^T with B loaded by one TMA box into the
// 128-byte-swizzled K-major layout and read through a swizzled descriptor.
__global__ void probe_mma_sw128_kernel(const __grid_constant__ CUtensorMap tm, const uint16_t* A, int N, float* D,
                                       uint32_t* status) {
  __shared__ __align__(1024) uint8_t sB[256 * 128];
  __shared__ uint64_t bar, bar2;
  __shared__ uint32_t tmem;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  const Abort ab{status, &abort_flag};
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    mbar_init(&bar2, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t base = tmem;
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)N * 128);
    tma_load_2d(sB, &tm, 0, 0, &bar);
  }
  uint32_t r[32];
  for (int c = 0; c < 32; ++c) r[c] = (uint32_t)A[tid * 64 + 2 * c] | ((uint32_t)A[tid * 64 + 2 * c + 1] << 16);
  tmem_st32(base + ((uint32_t)(32 * warp) << 16), r);
  tmem_st_wait();
  tc_fence_before();
  bool ok = mbar_wait(&bar, 0, ab, 111);
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t idesc = idesc_bf16_m128((uint32_t)N);
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16_ts(base + 128, base + kk * 8, smem_desc_sw128(smem_u32(sB) + kk * 32), idesc, kk > 0 ? 1u : 0u);
    mma_commit(&bar2);
  }
  ok = mbar_wait(&bar2, 0, ab, 112) && ok;
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(base + ((uint32_t)(32 * warp) << 16) + 128 + c0, v);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j) D[tid * N + c0 + j] = __uint_as_float(v[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(base, 512);
}

// Dequantise prepared blocks (one 128-row x 64-element stage each) with the
// table-lookup dequantiser.
template <int FMT>
__global__ void probe_dequant_kernel(const uint8_t* codes, const uint8_t* scales, uint16_t* out) {
  const int blk = blockIdx.x, r = threadIdx.x;
  constexpr int SB = scale_bytes_per_row(FMT);
  const uint8_t* cs = codes + (size_t)blk * kCodeBytesPerStage;
  const uint4 c0 = *reinterpret_cast<const uint4*>(cs + r * 16);
  const uint4 c1 = *reinterpret_cast<const uint4*>(cs + 2048 + r * 16);
  const uint8_t* ss = scales + ((size_t)blk * kTileRows + r) * SB;
  uint32_t sc = 0;
  for (int b = 0; b < SB; ++b) sc |= (uint32_t)ss[b] << (8 * b);
  uint32_t v[32];
  dequant_stage<FMT>(c0, c1, sc, v);
  uint16_t* o = out + ((size_t)blk * kTileRows + r) * kBK;
  for (int c = 0; c < 32; ++c) {
    o[2 * c] = (uint16_t)(v[c] & 0xFFFF);
    o[2 * c + 1] = (uint16_t)(v[c] >> 16);
  }
}

// The per-route small-m kernel's dequantiser: prepared words (plain nibble
// pairs) -> hardware FP4 conversion to f16, times the fp32 block scale; one thread per
// weight row, one block per 64-wide stage, fp32 output in K order.
template <int FMT>
__global__ void probe_dequant_f16_kernel(const uint8_t* codes, const uint8_t* scales, float* out) {
  const int blk = blockIdx.x, r = threadIdx.x;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int G = FMT == 0 ? 16 : 32;
  const uint8_t* cs = codes + (size_t)blk * kCodeBytesPerStage;
  const uint8_t* ss = scales + ((size_t)blk * kTileRows + r) * SB;
  float* o = out + ((size_t)blk * kTileRows + r) * kBK;
  // byte b of a converted word holds elements (lo, hi) of the word's eight
  const int el_lo[4] = {0, 1, 4, 5}, el_hi[4] = {2, 3, 6, 7};
  for (int q = 0; q < 8; ++q) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(cs + (q >> 2) * 2048 + r * 16 + (q & 3) * 4);
    uint32_t h[4];
    e2m1x8_to_f16x2(w, h[0], h[1], h[2], h[3]);
    for (int b = 0; b < 4; ++b) {
      const __half2 v = *reinterpret_cast<const __half2*>(&h[b]);
      const int klo = q * 8 + el_lo[b], khi = q * 8 + el_hi[b];
      o[klo] = __low2float(v) * f32_scale<FMT>(ss[klo / G], 0);
      o[khi] = __high2float(v) * f32_scale<FMT>(ss[khi / G], 0);
    }
  }
}

// bf16x2 multiply on chosen bit patterns (subnormal-input behaviour).
__global__ void probe_bf16_mul_kernel(const uint32_t* a, const uint32_t* b, uint32_t* d, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) d[i] = bf16x2_mul(a[i], b[i]);
}

extern "C" {

int probe_mma_ts(const uint16_t* A, const uint16_t* B, int N, float* D, uint32_t* status) {
  if (N < 16 || N > 256 || N % 16) return -1;
  probe_mma_kernel<<<1, 128>>>(A, B, N, D, status);
  cudaError_t e = cudaDeviceSynchronize();
  return (int)e;
}

int probe_mma_rowb(const uint16_t* A, const uint16_t* x, float* D, uint32_t* status) {
  probe_mma_rowb_kernel<<<1, 128>>>(A, x, D, status);
  return (int)cudaDeviceSynchronize();
}

int probe_tma(const uint16_t* src, int rows, int cols, int mode, int c0, const int* r4, int box_rows, int dst_off,
              uint8_t* out, uint32_t* status) {
  CUtensorMap tm;
  if (!make_tmap_bf16_2d(&tm, src, (uint64_t)rows, (uint64_t)cols, mode == 0 ? (uint32_t)box_rows : 1u)) return -2;
  probe_tma_kernel<<<1, 128>>>(tm, mode, c0, r4[0], r4[1], r4[2], r4[3], box_rows, dst_off, out, status);
  return (int)cudaDeviceSynchronize();
}

int probe_mma_sw128(const uint16_t* A, const uint16_t* B, int N, float* D, uint32_t* status) {
  if (N < 16 || N > 256 || N % 16) return -1;
  CUtensorMap tm;
  if (!make_tmap_bf16_2d(&tm, B, (uint64_t)N, 64, (uint32_t)N)) return -2;
  probe_mma_sw128_kernel<<<1, 128>>>(tm, A, N, D, status);
  return (int)cudaDeviceSynchronize();
}

int probe_dequant(const uint8_t* codes, const uint8_t* scales, int fmt, int nblocks, uint16_t* out) {
  if (nblocks <= 0) return -1;
  if (fmt == 0) probe_dequant_kernel<0><<<nblocks, 128>>>(codes, scales, out);
  else probe_dequant_kernel<1><<<nblocks, 128>>>(codes, scales, out);
  return (int)cudaDeviceSynchronize();
}

int probe_dequant_f16(const uint8_t* codes, const uint8_t* scales, int fmt, int nblocks, float* out) {
  if (nblocks <= 0) return -1;
  if (fmt == 0) probe_dequant_f16_kernel<0><<<nblocks, 128>>>(codes, scales, out);
  else probe_dequant_f16_kernel<1><<<nblocks, 128>>>(codes, scales, out);
  return (int)cudaDeviceSynchronize();
}

int probe_bf16_mul(const uint32_t* a, const uint32_t* b, uint32_t* d, int n) {
  if (n <= 0) return -1;
  probe_bf16_mul_kernel<<<(n + 127) / 128, 128>>>(a, b, d, n);
  return (int)cudaDeviceSynchronize();
}

}  // extern "C"
