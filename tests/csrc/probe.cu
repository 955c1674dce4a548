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

// Latency microbenchmark of the tensor-memory building blocks (cycles):
// out[0] tcgen05.st 32x32b.x32 + wait::st, out[1] tcgen05.ld 32x32b.x16 +
// wait::ld (both per warp, averaged), out[2] four M128 N16 K16 MMAs + commit
// observed on the mbarrier, out[3] the same with N = 160.
__global__ void probe_tmem_latency_kernel(long long* out, uint32_t* status) {
  __shared__ __align__(1024) uint8_t sB[160 * 128];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  for (int i = tid; i < 160 * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sB)[i] = 0;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t base = tmem;
  const uint32_t lb = (uint32_t)(32 * warp) << 16;
  uint32_t r[32];
  for (int c = 0; c < 32; ++c) r[c] = 0x3F803F80u;
  long long t_st = 0, t_ld = 0;
  for (int it = 0; it < 64; ++it) {
    const long long t0 = clock64();
    tmem_st32(base + lb + (it % 6) * 32, r);
    tmem_st_wait();
    const long long t1 = clock64();
    uint32_t v[16];
    tmem_ld16(base + lb + 256, v);
    tmem_ld_wait();
    const long long t2 = clock64();
    t_st += t1 - t0;
    t_ld += t2 - t1;
    r[it & 31] ^= v[it & 15] & 1u;
  }
  if (lane == 0) {
    atomicAdd(reinterpret_cast<unsigned long long*>(&out[0]), (unsigned long long)(t_st / 64));
    atomicAdd(reinterpret_cast<unsigned long long*>(&out[1]), (unsigned long long)(t_ld / 64));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    uint32_t phase = 0;
    for (int which = 0; which < 2; ++which) {
      const uint32_t n = which == 0 ? 16u : 160u;
      const uint32_t idesc = idesc_bf16_m128(n);
      long long tot = 0;
      for (int it = 0; it < 32 && !ab.raised(); ++it) {
        const long long t0 = clock64();
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts(base + 192, base + kk * 8, smem_desc_noswizzle(smem_u32(sB) + kk * 256, 128, 1024), idesc,
                      kk > 0 ? 1u : 0u);
        mma_commit(&bar);
        if (!mbar_wait(&bar, phase, ab, 102)) break;
        phase ^= 1;
        tot += clock64() - t0;
      }
      out[2 + which] = tot / 32;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(base, 512);
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

// MMA issue throughput: 64 stages of `per` K=16 MMAs, one commit every
// `per_commit` MMAs (0: none until the end), timed from the first issue to
// the completion of the last (cycles).  variant bit 0: N = 160 (else 16);
// bit 1: A from shared memory (else TMEM); bit 2: per stage, also wait on an
// already-completed mbarrier and fence; bit 3: N = 256.
// Non-blocking test of a phase (mbarrier.test_wait): true when complete.
__device__ __forceinline__ bool probe_mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// 64 stages of four MMAs as the GEMM kernels issue them (see probe_mma_tput).
// rz is 0 at run time but unknown to the compiler, so the slot arithmetic is
// not folded away.  cyc[0] = issue time, cyc[1] = until the last completes.
template <int WAITS, bool A_TMEM>
__device__ __noinline__ void issue_loop(uint32_t base, uint32_t a_base, uint32_t b_base, uint32_t idesc, uint32_t rz,
                                        uint64_t* bar_stage, uint64_t* bar_ready, uint64_t* bar_done, const Abort& ab,
                                        long long* cyc) {
  const long long t0 = clock64();
  for (int s = 0; s < 64; ++s) {
    const uint32_t slot = ((uint32_t)s % 3u) * rz;
    if constexpr (WAITS == 1) {  // two bounded try_wait waits and a fence
      mbar_wait(bar_ready, 0, ab, 117);
      mbar_wait(bar_ready, 0, ab, 118);
      tc_fence_after();
    } else if constexpr (WAITS == 2) {  // two non-blocking tests first, then the fence
      if (!probe_mbar_test(bar_ready, 0)) mbar_wait(bar_ready, 0, ab, 119);
      if (!probe_mbar_test(bar_ready, 0)) mbar_wait(bar_ready, 0, ab, 120);
      tc_fence_after();
    } else if constexpr (WAITS == 3) {  // two bounded waits, no fence
      mbar_wait(bar_ready, 0, ab, 121);
      mbar_wait(bar_ready, 0, ab, 122);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t bdesc = smem_desc_sw128(b_base + slot * 32768u + kk * 32);
      if constexpr (A_TMEM) {
        mma_bf16_ts(base + ((kk & 1) ? 320u : 128u), base + (slot * 32u + kk * 8u), bdesc, idesc,
                    (s > 0 || kk > 1) ? 1u : 0u);
      } else {
        const uint64_t adesc = smem_desc_sw128(a_base + slot * 16384u + kk * 32);
        mma_bf16_ss(base + ((kk & 1) ? 256u : 0u), adesc, bdesc, idesc, (s > 0 || kk > 1) ? 1u : 0u);
      }
    }
    mma_commit(bar_stage);
  }
  const long long t1 = clock64();
  mma_commit(bar_done);
  mbar_wait(bar_done, 0, ab, 116);
  cyc[0] = t1 - t0;
  cyc[1] = clock64() - t0;
}

__global__ void probe_mma_tput_kernel(int variant, int per, int per_commit, long long* out, uint32_t* status) {
  __shared__ __align__(1024) uint8_t sB[256 * 128];  // B rows (N <= 256); A in shared memory reuses rows 0..127
  uint8_t* sA = sB;
  __shared__ uint64_t bar_stage, bar_done, bar_ready;
  __shared__ uint32_t tmem;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  const Abort ab{status, &abort_flag};
  for (int i = tid; i < 256 * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sB)[i] = 0;
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_stage, 1);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_ready, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t base = tmem;
  if (tid == 0) {
    mbar_arrive(&bar_ready);  // phase 0 complete: waits on it return at once
    const uint32_t n = (variant & 8) ? 256u : (variant & 1) ? 160u : (variant & 64) ? 128u : (variant & 128) ? 64u : 16u;
    const bool sw = (variant & 32) != 0;  // 128-byte-swizzled K-major operands (as in the GEMM kernels)
    // variant bit 256: M = 64 instead of 128 (A from shared memory)
    const uint32_t idesc = (variant & 256) ? ((idesc_bf16_m128(n) & ~(0x1Fu << 24)) | ((64u >> 4) << 24))
                                           : idesc_bf16_m128(n);
    if ((variant & 16384) && n > 128) {
      out[0] = out[1] = -1;  // the tensor-memory-A variant is laid out for N <= 128 only
    } else if (variant & 2048) {
      // as the GEMM kernels issue: descriptors rebuilt for every MMA from a
      // runtime ring slot, four MMAs per stage unrolled, one commit per stage;
      // bit 8192 adds two barrier waits and a fence per stage, bit 16384 takes
      // A from tensor memory.  Each combination is its own branch-free loop.
      // bits 8192 / 32768 / 65536: waits as try_wait + fence / test_wait first + fence / try_wait, no fence
      const int waits = (variant & 8192) ? 1 : (variant & 32768) ? 2 : (variant & 65536) ? 3 : 0;
      const uint32_t rz = (uint32_t)variant >> 30;
      long long cyc[2];
      const uint32_t sa = smem_u32(sA), sb = smem_u32(sB);
      if (variant & 16384) {
        switch (waits) {
          case 0: issue_loop<0, true>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
          case 1: issue_loop<1, true>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
          case 2: issue_loop<2, true>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
          default: issue_loop<3, true>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
        }
      } else {
        switch (waits) {
          case 0: issue_loop<0, false>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
          case 1: issue_loop<1, false>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
          case 2: issue_loop<2, false>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
          default: issue_loop<3, false>(base, sa, sb, idesc, rz, &bar_stage, &bar_ready, &bar_done, ab, cyc); break;
        }
      }
      out[0] = cyc[0];
      out[1] = cyc[1];
    } else if (variant & 512) {
      // descriptors computed before the loop, four MMAs per iteration
      // unrolled (A and B in shared memory, 128-byte swizzle, two accumulators)
      uint64_t ad[4], bd[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        ad[kk] = smem_desc_sw128(smem_u32(sA) + kk * 32);
        bd[kk] = smem_desc_sw128(smem_u32(sB) + kk * 32);
      }
      const long long t0b = clock64();
      for (int s = 0; s < 64; ++s) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(base + ((kk & 1) ? 256u : 0u), ad[kk], bd[kk], idesc, (s > 0 || kk > 1) ? 1u : 0u);
      }
      const long long t1b = clock64();
      mma_commit(&bar_done);
      mbar_wait(&bar_done, 0, ab, 115);
      out[0] = t1b - t0b;
      out[1] = clock64() - t0b;
    } else {
    const long long t0 = clock64();
    for (int s = 0; s < 64; ++s) {
      if (variant & 4) {
        mbar_wait(&bar_ready, 0, ab, 113);
        tc_fence_after();
      }
      for (int kk = 0; kk < per; ++kk) {
        const uint64_t bdesc = sw ? smem_desc_sw128(smem_u32(sB) + (kk & 3) * 32)
                                  : smem_desc_noswizzle(smem_u32(sB) + (kk & 3) * 256, 128, 1024);
        if (variant & 2) {
          // variant bit 16: MMAs alternate between two accumulators (columns 0 and 256)
          const uint32_t dcol = (variant & 16) ? ((kk & 1) ? 256u : 0u) : 192u;
          const uint64_t adesc = sw ? smem_desc_sw128(smem_u32(sA) + (kk & 3) * 32)
                                    : smem_desc_noswizzle(smem_u32(sA) + (kk & 3) * 256, 128, 1024);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(base + dcol),
              "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)(s > 0 || kk > 1))
              : "memory");
        } else {
          mma_bf16_ts(base + 192, base + (kk & 3) * 8, bdesc, idesc, (s > 0 || kk > 0) ? 1u : 0u);
        }
        if (per_commit > 0 && ((s * per + kk + 1) % per_commit) == 0) mma_commit(&bar_stage);
      }
    }
    const long long t1 = clock64();
    mma_commit(&bar_done);
    mbar_wait(&bar_done, 0, ab, 114);
    const long long t2 = clock64();
    out[0] = t1 - t0;  // issue time of 64 stages
    out[1] = t2 - t0;  // until the last completes
    }
  } else if ((variant & 131072) && warp >= 1) {
    // warps 1-3 store into tensor memory (columns 448..479 of their lane
    // quarters, away from the MMA operands and accumulators) while thread 0
    // issues the MMAs: the dequantiser warps' traffic in the GEMM kernels
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) r[c] = 0x3F803F80u + c;
    const uint32_t taddr = base + ((uint32_t)(32 * warp) << 16) + 448u;
    for (int it = 0; it < 400; ++it) {
      tmem_st32(taddr, r);
      tmem_st_wait();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(base, 512);
}

// Dequantise serving-layout blocks (one 128-row x 64-element stage each).
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

// bf16x2 multiply on chosen bit patterns (subnormal-input behaviour).
__global__ void probe_bf16_mul_kernel(const uint32_t* a, const uint32_t* b, uint32_t* d, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) d[i] = bf16x2_mul(a[i], b[i]);
}

// Steady-state cost of the decode path's stage arithmetic, without producers:
// every CTA (8 warps, 16 weight rows each) runs `stages` stages over
// shared-memory data that does not change.  Dynamic shared memory pads the
// CTA to set how many are resident per SM.  Variants: 0 as the decode kernel
// (two stages per step, four accumulators); 1 one stage per step; 2 the
// dequantisation alone (its results folded by bf16x2 adds); 3 the MMAs alone.
template <int V>
__global__ void __launch_bounds__(256) probe_decode_stage_kernel(int stages, float* out, long long* cyc) {
  extern __shared__ __align__(16) uint8_t sm[];
  uint8_t* codes = sm;                  // 4 slots x 2 stages x 4096
  uint8_t* scales = sm + 32768;         // 8 stages x 512
  uint8_t* xrow = sm + 32768 + 4096;    // 128 stages x 128 B
  for (int i = threadIdx.x; i < 32768 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(codes)[i] = 0x9E3779B9u * (uint32_t)(i + 1);
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) scales[i] = (uint8_t)(0x68 + (i % 23));
  for (int i = threadIdx.x; i < 128 * 128 / 2; i += blockDim.x)
    reinterpret_cast<uint16_t*>(xrow)[i] = (uint16_t)(0x3F80u + (i & 0x3F));
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = 16 * warp + g;
  const uint32_t code_off = (t >> 1) * 2048 + r0 * 16 + (t & 1) * 8;
  const uint32_t sc_off = r0 * 4 + t;
  float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
  float f[4] = {0.f, 0.f, 0.f, 0.f}, h4[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t fold = 0;
  const long long t0 = clock64();
  for (int s = 0; s < stages; s += 2) {
    const int slot = (s >> 1) & 3;
    const uint8_t* cs = codes + slot * 8192 + code_off;
    const uint8_t* ss = scales + (s & 7) * 512 + sc_off;
    const uint8_t* xr = xrow + t * 32 + (s & 126) * 128;
    if constexpr (V == 0) {
      StageIn a, b;
      load_stage<4>(a, cs, ss, xr);
      load_stage<4>(b, cs + 4096, ss + 512, xr + 128);
      compute_stage<0>(a, d, e);
      compute_stage<0>(b, f, h4);
    } else if constexpr (V == 1) {
#pragma unroll 1
      for (int st = 0; st < 2; ++st) {
        StageIn a;
        load_stage<4>(a, cs + st * 4096, ss + st * 512, xr + st * 128);
        compute_stage<0>(a, d, e);
      }
    } else if constexpr (V == 2) {
      for (int st = 0; st < 2; ++st) {
        StageIn a;
        load_stage<4>(a, cs + st * 4096, ss + st * 512, xr + st * 128);
        const uint32_t sa = d_scale<0>(a.b0), sb = d_scale<0>(a.b1);
        const uint32_t w[4] = {a.c0.x, a.c0.y, a.c1.x, a.c1.y};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t sq = q < 2 ? sa : sb;
          uint32_t v0 = bf16x2_mul(fp4x2_lookup(w[q]), sq);
          uint32_t v1 = bf16x2_mul(fp4x2_lookup((w[q] >> 2)), sq);
          uint32_t v2 = bf16x2_mul(fp4x2_lookup((w[q] >> 16)), sq);
          uint32_t v3 = bf16x2_mul(fp4x2_lookup((w[q] >> 18)), sq);
          asm("add.rn.bf16x2 %0, %0, %1;" : "+r"(fold) : "r"(v0));
          asm("add.rn.bf16x2 %0, %0, %1;" : "+r"(fold) : "r"(v1));
          asm("add.rn.bf16x2 %0, %0, %1;" : "+r"(fold) : "r"(v2));
          asm("add.rn.bf16x2 %0, %0, %1;" : "+r"(fold) : "r"(v3));
        }
      }
    } else {
      for (int st = 0; st < 2; ++st) {
        StageIn a;
        load_stage<4>(a, cs + st * 4096, ss + st * 512, xr + st * 128);
        mma_16816(st ? f : d, a.xa.x, a.xb.x, a.xa.y, a.xb.y, a.xa.z, a.xa.w);
        mma_16816(st ? h4 : e, a.xa.z, a.xb.z, a.xa.w, a.xb.w, a.xb.x, a.xb.y);
        mma_16816(st ? f : d, a.xb.x, a.xa.x, a.xb.y, a.xa.y, a.xa.x, a.xa.y);
        mma_16816(st ? h4 : e, a.xb.z, a.xa.z, a.xb.w, a.xa.w, a.xb.z, a.xb.w);
      }
    }
  }
  const long long t1 = clock64();
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
  out[blockIdx.x * blockDim.x + threadIdx.x] = d[0] + e[0] + f[2] + h4[2] + __uint_as_float(fold & 0x3FFFFFFFu);
}

// Issue rate of single instructions: 8 warps per CTA, one CTA per SM, eight
// independent dependency chains per thread.  op: 0 prmt, 1 lop3, 2 mul.hi.u32,
// 3 mul.rn.bf16x2, 4 shr.b32, 5 fma.rn.f32, 6 mul.rn.f16x2, 7 fma.rn.bf16x2,
// 8 mad.lo.u32, 9 iadd3 (add.u32).
template <int OP>
__global__ void __launch_bounds__(256) probe_op_tput_kernel(int iters, uint32_t k, uint32_t* out, long long* cyc) {
  uint32_t a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = threadIdx.x * 2654435761u + i * 40503u + k;
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (OP == 0) asm volatile("prmt.b32 %0, %0, %1, %2;" : "+r"(a[i]) : "r"(k), "r"(0x3210u ^ k));
      if constexpr (OP == 1) asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(a[i]) : "r"(k), "r"(a[(i + 1) & 7]));
      if constexpr (OP == 2) asm volatile("mul.hi.u32 %0, %0, %1;" : "+r"(a[i]) : "r"(k | 0x40000000u));
      if constexpr (OP == 3) asm volatile("mul.rn.bf16x2 %0, %0, %1;" : "+r"(a[i]) : "r"(0x3F803F80u ^ (k & 1)));
      if constexpr (OP == 4) asm volatile("shr.b32 %0, %0, %1;" : "+r"(a[i]) : "r"(k & 1));
      if constexpr (OP == 5) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+r"(a[i]) : "r"(0x3F800000u), "r"(k));
      if constexpr (OP == 6) asm volatile("mul.rn.f16x2 %0, %0, %1;" : "+r"(a[i]) : "r"(0x3C003C00u ^ (k & 1)));
      if constexpr (OP == 7)
        asm volatile("fma.rn.bf16x2 %0, %0, %1, %2;" : "+r"(a[i]) : "r"(0x3F803F80u ^ (k & 1)), "r"(0u));
      if constexpr (OP == 8) asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(a[i]) : "r"(k | 1u), "r"(k));
      if constexpr (OP == 9) asm volatile("add.u32 %0, %0, %1;" : "+r"(a[i]) : "r"(k));
    }
  }
  const long long t1 = clock64();
  uint32_t x = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) x ^= a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = x;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// Empty kernel for launch-latency measurements (grid, block, dynamic shared
// memory and the cooperative attribute chosen by the caller).
__global__ void probe_launch_kernel(int* out) {
  extern __shared__ int sm_launch[];
  if (threadIdx.x == 0 && blockIdx.x == 0 && out) out[0] = sm_launch[0] * 0 + 1;
}

// mma.sync m16n8k16 bf16 with every A element = a_bits and every B element =
// b_bits (one warp): out[lane * 4 + i] = D fragment element i.  With A a
// bf16 subnormal this shows whether the tensor core keeps subnormal inputs.
__global__ void probe_mma_sync_const_kernel(uint16_t a_bits, uint16_t b_bits, float* out) {
  const uint32_t a = (uint32_t)a_bits | ((uint32_t)a_bits << 16), b = (uint32_t)b_bits | ((uint32_t)b_bits << 16);
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  mma_16816(d, a, a, a, a, b, b);
  for (int i = 0; i < 4; ++i) out[threadIdx.x * 4 + i] = d[i];
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

int probe_tmem_latency(long long* out, uint32_t* status) {
  probe_tmem_latency_kernel<<<1, 128>>>(out, status);
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

int probe_mma_tput(int variant, int per, int per_commit, long long* out, uint32_t* status) {
  if (per < 1 || per > 16) return -1;
  probe_mma_tput_kernel<<<1, 128>>>(variant, per, per_commit, out, status);
  return (int)cudaDeviceSynchronize();
}

int probe_dequant(const uint8_t* codes, const uint8_t* scales, int fmt, int nblocks, uint16_t* out) {
  if (nblocks <= 0) return -1;
  if (fmt == 0) probe_dequant_kernel<0><<<nblocks, 128>>>(codes, scales, out);
  else probe_dequant_kernel<1><<<nblocks, 128>>>(codes, scales, out);
  return (int)cudaDeviceSynchronize();
}

int probe_bf16_mul(const uint32_t* a, const uint32_t* b, uint32_t* d, int n) {
  if (n <= 0) return -1;
  probe_bf16_mul_kernel<<<(n + 127) / 128, 128>>>(a, b, d, n);
  return (int)cudaDeviceSynchronize();
}

int probe_decode_stage(int variant, int stages, int grid, int smem_bytes, float* out, long long* cyc) {
  if (stages < 2 || stages % 2 || smem_bytes < 32768 + 4096 + 16384 || grid < 1) return -1;
  cudaError_t e = cudaSuccess;
#define B4_PROBE_STAGE(V)                                                                             \
  e = cudaFuncSetAttribute(probe_decode_stage_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           smem_bytes);                                                               \
  if (e == cudaSuccess) probe_decode_stage_kernel<V><<<grid, 256, smem_bytes>>>(stages, out, cyc);
  switch (variant) {
    case 0: B4_PROBE_STAGE(0); break;
    case 1: B4_PROBE_STAGE(1); break;
    case 2: B4_PROBE_STAGE(2); break;
    default: B4_PROBE_STAGE(3); break;
  }
#undef B4_PROBE_STAGE
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}

int probe_op_tput(int op, int iters, int grid, uint32_t k, uint32_t* out, long long* cyc) {
  switch (op) {
    case 0: probe_op_tput_kernel<0><<<grid, 256>>>(iters, k, out, cyc); break;
    case 1: probe_op_tput_kernel<1><<<grid, 256>>>(iters, k, out, cyc); break;
    case 2: probe_op_tput_kernel<2><<<grid, 256>>>(iters, k, out, cyc); break;
    case 3: probe_op_tput_kernel<3><<<grid, 256>>>(iters, k, out, cyc); break;
    case 4: probe_op_tput_kernel<4><<<grid, 256>>>(iters, k, out, cyc); break;
    case 5: probe_op_tput_kernel<5><<<grid, 256>>>(iters, k, out, cyc); break;
    case 6: probe_op_tput_kernel<6><<<grid, 256>>>(iters, k, out, cyc); break;
    case 7: probe_op_tput_kernel<7><<<grid, 256>>>(iters, k, out, cyc); break;
    case 8: probe_op_tput_kernel<8><<<grid, 256>>>(iters, k, out, cyc); break;
    default: probe_op_tput_kernel<9><<<grid, 256>>>(iters, k, out, cyc); break;
  }
  return (int)cudaDeviceSynchronize();
}

int probe_launch(int grid, int block, int smem_bytes, int cooperative, int* out, void* stream) {
  static int configured = 0;
  if (smem_bytes > configured) {
    cudaError_t e = cudaFuncSetAttribute(probe_launch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return (int)e;
    configured = smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 1 : 0;
  return (int)cudaLaunchKernelEx(&cfg, probe_launch_kernel, out);
}

int probe_mma_sync_const(int a_bits, int b_bits, float* out) {
  probe_mma_sync_const_kernel<<<1, 32>>>((uint16_t)a_bits, (uint16_t)b_bits, out);
  return (int)cudaDeviceSynchronize();
}

}  // extern "C"
