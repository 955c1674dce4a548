// Grouped W4A16 GEMMs of the fused MoE layer on tcgen05 (sm_103a).
//
// One persistent, warp-specialised kernel serves the two route-packed GEMMs
// (flashinfer PR #4255, Description: "Cooperative persistent launches for the
// fused FC1/FC2 kernel", "folding the top-k sum into the FC2 store
// epilogue"):
//
//   FC1  B = x rows of the routes of one expert chunk, copied into
//        packed-route order by the route pack; the epilogue applies
//        SiLU-SwiGLU or ReLU^2 (none for the dense linear layer, whose
//        B rows are x itself) and stores bf16 h in the same order.
//   FC2  B = h rows of the chunk; the epilogue multiplies by gs2 and the
//        router weight and adds into an fp32 [tokens, H] accumulator (the
//        top-k sum), which finalize_grouped_kernel rounds to bf16.
//
// A work unit is (expert chunk of <= 160 routes, 128-row weight tile).  The
// tensor-core operation is swapped: the 128 weight rows are the M operand, the
// chunk's routes are N (rounded up to 16).  Used when experts receive many
// routes (prefill); moe_gemm_wn.cu puts 256 weight rows on N instead, which
// issues half the MMAs when experts receive few routes.  Weights are dequantised from E2M1
// codes and E4M3 / E8M0 block scales to bf16 by eight dequant warps (one
// thread per weight row) and written straight into tensor memory with
// tcgen05.st, where tcgen05.mma reads them as its A operand; B sits in shared
// memory in the 128-byte-swizzled K-major layout, loaded by TMA in 80-row 2-D
// boxes, at most two per 160-row stage (both B operands are contiguous in
// packed-route order; rows past a chunk are read, or zero-filled past the
// tensor, and left unused: five 32-row boxes per stage measured 3 % slower on
// prefill, 7 % on the dense m = 2048 layer).  Roles, one CTA of 16 warps:
//   warp 0       bulk-copy (TMA engine) producer of packed codes and scales
//   warp 1       TMEM allocator and the single MMA-issuing thread
//   warp 2       B producer (TMA tile loads)
//   warps 4-11   dequantisers (two groups of four taking alternate stages)
//   warps 12-15  epilogue: tensor-memory accumulators -> outputs
// Rings: weights (10 stages); A slots in TMEM and B stages (6, one index, one
// release commit per stage); two accumulators, so the epilogue of one unit
// overlaps the next mainloop.
// Every wait is bounded (ptx.cuh).
//
// Dequantised weights carry a factor 2^-63 so that every product of an E2M1
// code and a block scale is a normal bf16; the epilogue multiplies by 2^63.

#include <cuda_bf16.h>

#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tma.cuh"

namespace b4 {

cudaError_t ensure_smem_limit(const void* func, size_t bytes);

constexpr int kNumA = 6;                 // A slots (K stages) held in tensor memory
constexpr int kThreads = 512;
constexpr int kAColsPerSlot = kBK / 2;   // 32 columns of packed bf16 pairs
constexpr int kNW = 10;                  // weight stages in flight
constexpr int kNB = 6;                   // B stages in flight
constexpr int kBN = kChunkRowsM;         // max tcgen05 N
constexpr int kBStage = kBN * kBK * 2;   // 160 rows x 128 bytes, swizzled
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol0 = kNumA * kAColsPerSlot;  // 192: two accumulators of kBN columns follow
constexpr float kTwo63 = 9.223372036854775808e18f;
static_assert(kAccCol0 + 2 * kBN <= kTmemCols, "tensor memory budget");
static_assert(kBStage % 1024 == 0, "swizzle atoms of B stages must stay 1024-byte aligned");
static_assert(kNB == kNumA, "A slots and B stages share one ring index and one release barrier");

template <int FMT>
struct SmemLayout {
  static constexpr int kScaleStage = scale_bytes_per_stage(FMT);
  static constexpr size_t b = 0;  // offset from the 1024-aligned base
  static constexpr size_t codes = b + (size_t)kNB * kBStage;
  static constexpr size_t scales = codes + (size_t)kNW * kCodeBytesPerStage;
  static constexpr size_t bars = round_up((int)(scales + (size_t)kNW * kScaleStage), 8);
  static constexpr int kNumBars = 2 * kNW + 3 * kNumA + 4 + 1;
  static constexpr size_t misc = bars + 8 * kNumBars;
  static constexpr size_t rows = misc + 16;
  static constexpr size_t total = rows + 8 * kBN + 1024;  // + alignment slack
};

struct Unit {
  int expert, tile, slot0, rows;
};

__device__ __forceinline__ int num_units(const GemmParams& p) {
  int c = *(volatile const int32_t*)p.chunk_count;
  c = c < 0 ? 0 : (c > p.max_chunks ? p.max_chunks : c);
  return c * p.n_tiles;
}

__device__ __forceinline__ bool get_unit(const GemmParams& p, int u, Unit& U) {
  const int c = u / p.n_tiles;
  U.tile = u - c * p.n_tiles;
  const int4 ch = p.chunks[c];
  U.expert = ch.x;
  U.slot0 = ch.y;
  U.rows = ch.z;
  return U.rows > 0;
}

// Timeline hook: CTA 0 records clock64() of event `kind` number `idx`.  It
// sits in the pipelines' per-stage loops, so it is compiled in only when the
// library is built with B4_TRACE defined (a profiling build).
__device__ __forceinline__ void trace_mark(const GemmParams& p, int kind, uint32_t idx) {
#ifdef B4_TRACE
  if (p.trace && blockIdx.x == 0 && idx < (uint32_t)kTraceLen) p.trace[kind * kTraceLen + idx] = clock64();
#else
  (void)p, (void)kind, (void)idx;
#endif
}

// One stage of four MMAs (A slices in tensor memory, B by descriptor), with
// two non-blocking tests of the next stage's barriers issued first and read
// only after the MMAs: a barrier test takes ~130 cycles, which the MMA issue
// then hides.  *na / *nb: the next stage's A / B barriers were seen complete
// (false when test is 0).
__device__ __forceinline__ void mma_stage_test_next(uint32_t d_tmem, const uint32_t (&a)[4], const uint64_t (&b)[4],
                                                    uint32_t idesc, uint32_t accumulate, uint64_t* bar_a,
                                                    uint32_t par_a, uint64_t* bar_b, uint32_t par_b, uint32_t test,
                                                    bool* na, bool* nb) {
  uint32_t ra, rb;
  asm volatile(
      "{\n\t.reg .pred pa, pb, g, q, t;\n\t"
      "setp.ne.b32 g, %9, 0;\n\t"
      "setp.ne.b32 pa, %9, %9;\n\t"
      "setp.ne.b32 pb, %9, %9;\n\t"
      "@g mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 pa, [%5], %6;\n\t"
      "@g mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 pb, [%7], %8;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "setp.eq.b32 t, %9, %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], [%3], %10, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], [%12], %13, %11, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], [%14], %15, %11, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%2], [%16], %17, %11, t;\n\t"
      "selp.u32 %0, 1, 0, pa;\n\t"
      "selp.u32 %1, 1, 0, pb;\n\t}"
      : "=r"(ra), "=r"(rb)
      : "r"(d_tmem), "r"(a[0]), "r"(accumulate), "r"(smem_u32(bar_a)), "r"(par_a), "r"(smem_u32(bar_b)),
        "r"(par_b), "r"(test), "l"(b[0]), "r"(idesc), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]),
        "l"(b[3])
      : "memory");
  *na = ra != 0;
  *nb = rb != 0;
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Abort& ab, uint32_t where) {
  const bool ok = mbar_wait(bar, parity, ab, where);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------------ kernel
template <int MODE, int FMT>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using L = SmemLayout<FMT>;
  constexpr int NW = kNW, NB = kNB;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int kScaleStage = L::kScaleStage;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled B stages need 1024-byte alignment of the shared address
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* s_b = smem + L::b;
  uint8_t* s_codes = smem + L::codes;
  uint8_t* s_scales = smem + L::scales;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + NW;
  uint64_t* full_a = empty_w + NW;
  uint64_t* stage_free = full_a + kNumA;  // A slot and B stage of a ring index, freed by one commit
  uint64_t* full_b = stage_free + kNumA;
  uint64_t* full_acc = full_b + NB;
  uint64_t* empty_acc = full_acc + 2;
  uint64_t* drain = empty_acc + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc + 4);
  int32_t* s_rows = reinterpret_cast<int32_t*>(smem + L::rows);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Abort ab{p.status, s_abort};

  if (threadIdx.x == 0) {
    *s_abort = 0;
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&empty_w[i], 4);
    }
    for (int i = 0; i < kNumA; ++i) {
      mbar_init(&full_a[i], 4);
      mbar_init(&stage_free[i], 1);
      mbar_init(&full_b[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_acc[i], 1);
      mbar_init(&empty_acc[i], 4);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (p.pdl_wait_first) pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int n_units = num_units(p);
  const size_t wtile_codes = (size_t)p.k_stages * kCodeBytesPerStage;
  const size_t wtile_scales = (size_t)p.k_stages * kScaleStage;

  if (warp == 0) {
    // ------------------------------------------------ weight producer
    uint32_t ws = 0;
    if (lane == 0) {
      for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
        Unit U;
        if (!get_unit(p, u, U)) continue;
        const size_t tile_id = (size_t)U.expert * p.n_tiles + U.tile;
        const uint8_t* gc = p.wcodes + tile_id * wtile_codes;
        const uint8_t* gsc = p.wscales + tile_id * wtile_scales;
        for (int s = 0; s < p.k_stages; ++s, ++ws) {
          const uint32_t slot = ws % NW;
          if (!mbar_wait(&empty_w[slot], ((ws / NW) & 1) ^ 1, ab, 1)) break;
          mbar_arrive_expect_tx(&full_w[slot], kCodeBytesPerStage + kScaleStage);
          bulk_g2s(s_codes + slot * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage, kCodeBytesPerStage,
                   &full_w[slot]);
          bulk_g2s(s_scales + slot * kScaleStage, gsc + (size_t)s * kScaleStage, kScaleStage, &full_w[slot]);
          trace_mark(p, 0, ws);
        }
      }
      if (ab.raised()) {
        // let copies already issued land before the CTA's shared memory goes away
        const uint32_t n = ws < (uint32_t)NW ? ws : (uint32_t)NW;
        for (uint32_t i = ws - n; i < ws; ++i) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full_w[i % NW], (i / NW) & 1) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t as = 0, bs = 0, acc_i = 0;
      const uint32_t b_base = smem_u32(s_b);
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        Unit U;
        if (!get_unit(p, u, U)) continue;
        const uint32_t abuf = acc_i & 1;
        if (!mbar_wait(&empty_acc[abuf], ((acc_i >> 1) & 1) ^ 1, ab, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + kAccCol0 + abuf * kBN;
        const uint32_t idesc = idesc_bf16_m128((uint32_t)round_up(U.rows, 16));
        bool ok = true;
        bool pre_a = false, pre_b = false;  // this stage's operands were seen ready during the previous stage
        for (int s = 0; s < p.k_stages; ++s, ++as, ++bs) {
          const uint32_t aslot = as % kNumA, bslot = bs % NB;
          if ((!pre_a && !mbar_wait(&full_a[aslot], (as / kNumA) & 1, ab, 3)) ||
              (!pre_b && !mbar_wait(&full_b[bslot], (bs / NB) & 1, ab, 4))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t a_tm[4];
          uint64_t b_desc[4];
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            a_tm[kk] = tmem_base + aslot * kAColsPerSlot + kk * 8;
            b_desc[kk] = smem_desc_sw128(b_base + bslot * kBStage + kk * 32);
          }
          const uint32_t nas = as + 1, nbs = bs + 1;
          mma_stage_test_next(d_tmem, a_tm, b_desc, idesc, s > 0 ? 1u : 0u, &full_a[nas % kNumA],
                              (nas / kNumA) & 1, &full_b[nbs % NB], (nbs / NB) & 1, s + 1 < p.k_stages ? 1u : 0u,
                              &pre_a, &pre_b);
          mma_commit(&stage_free[aslot]);
          trace_mark(p, 2, as);
        }
        if (!ok) break;
        mma_commit(&full_acc[abuf]);
        ++acc_i;
      }
      // drain: wait until every MMA issued by this thread has completed
      mma_commit(drain);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // --------------------------------------------------------- B producer
    if (MODE == kFc2Grouped) pdl_wait();  // h comes from FC1 (FC1 waited for its inputs at entry)
    uint32_t bs = 0;
    for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
      Unit U;
      if (!get_unit(p, u, U)) continue;
      const int nload = cdiv(U.rows, 80);
      const uint32_t bytes = (uint32_t)nload * 10240u;
      bool ok = true;
      for (int s = 0; s < p.k_stages; ++s, ++bs) {
        const uint32_t slot = bs % NB;
        if (!warp_wait(&stage_free[slot], ((bs / NB) & 1) ^ 1, ab, 5)) {
          ok = false;
          break;
        }
        uint8_t* stage = s_b + slot * kBStage;
        if (lane == 0) mbar_arrive_expect_tx(&full_b[slot], bytes);
        __syncwarp();
        for (int i = lane; i < nload; i += 32)
          tma_load_2d(stage + i * 10240, &p.tmap_b, s * kBK, U.slot0 + 80 * i, &full_b[slot]);
        if (lane == 0) trace_mark(p, 3, bs);
      }
      if (!ok) break;
    }
    if (ab.raised() && lane == 0) {
      // let issued loads land before the CTA exits
      const uint32_t n = bs < (uint32_t)NB ? bs : (uint32_t)NB;
      for (uint32_t i = bs - n; i < bs; ++i) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&full_b[i % NB], (i / NB) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------ dequantisers
    // two groups of four warps take alternate stages, so one group's tensor
    // memory store drains while the other group computes
    const int half = (warp - 4) >> 2;
    const int row = 32 * (warp & 3) + lane;  // TMEM lane == weight row in the tile
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t ws = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit(p, u, U)) continue;
      bool ok = true;
      for (int s = 0; s < p.k_stages; ++s, ++ws) {
        if ((ws & 1) != (uint32_t)half) continue;
        const uint32_t wslot = ws % NW;
        if (!warp_wait(&full_w[wslot], (ws / NW) & 1, ab, 6)) {
          ok = false;
          break;
        }
        const uint8_t* cs = s_codes + wslot * kCodeBytesPerStage;
        const uint4 c0 = *reinterpret_cast<const uint4*>(cs + row * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(cs + 2048 + row * 16);
        uint32_t sc;
        if constexpr (SB == 4) sc = *reinterpret_cast<const uint32_t*>(s_scales + wslot * kScaleStage + row * 4);
        else sc = *reinterpret_cast<const uint16_t*>(s_scales + wslot * kScaleStage + row * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_w[wslot]);
        uint32_t r[32];
        dequant_stage<FMT>(c0, c1, sc, r);
        const uint32_t aslot = ws % kNumA;
        if (!warp_wait(&stage_free[aslot], ((ws / kNumA) & 1) ^ 1, ab, 7)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st32(tmem_base + lane_base + aslot * kAColsPerSlot, r);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full_a[aslot]);
          trace_mark(p, 1, ws);
        }
      }
      if (!ok) break;
    }
  } else if (warp >= 12) {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int er = 32 * q4 + lane;  // TMEM lane == weight row in the tile
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int et = threadIdx.x - 384;  // 0..127
    int32_t* s_tok = s_rows;                                   // FC2: token of each column
    float* s_wt = reinterpret_cast<float*>(s_rows + kBN);     // FC2: router weight of each column
    if constexpr (MODE == kFc1Grouped) {
      // clear the FC2 accumulator (FC2 waits for this grid before adding)
      float4* z = reinterpret_cast<float4*>(p.acc_out);
      const size_t n4 = p.acc_zero_floats / 4;
      for (size_t i = (size_t)blockIdx.x * 128 + et; i < n4; i += (size_t)gridDim.x * 128)
        z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if constexpr (MODE == kFc2Grouped) pdl_wait();  // acc_out cleared by FC1
    uint32_t acc_i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit(p, u, U)) continue;
      const uint32_t abuf = acc_i & 1;
      if constexpr (MODE == kFc2Grouped) {
        // the unit's routes: token and router weight, resolved before the wait
        for (int i = et; i < U.rows; i += 128) {
          const int route = __ldg(p.sorted_routes + U.slot0 + i);
          s_tok[i] = route / p.top_k;
          s_wt[i] = p.topk_weights ? __ldg(p.topk_weights + route) : 1.0f;
        }
        named_bar_sync(2, 128);
      }
      if (!warp_wait(&full_acc[abuf], (acc_i >> 1) & 1, ab, 8)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_base + kAccCol0 + abuf * kBN;
      const float gsv = (p.gs ? __ldg(p.gs + U.expert) : 1.0f) * kTwo63;
      const int ncols = round_up(U.rows, 16);
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
        if constexpr (MODE == kFc1Grouped) {
          if (p.act == 0) {
            // rows: lanes 0-15 gate, 16-31 up, for i = tile*64 + q4*16 + lane%16
            const bool is_up = lane >= 16;
            const int i = U.tile * 64 + q4 * 16 + (lane & 15);
            float mine[8], other[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float send = __uint_as_float(is_up ? v[j] : v[j + 8]) * gsv;
              other[j] = __shfl_xor_sync(0xffffffffu, send, 16);
              mine[j] = __uint_as_float(is_up ? v[j + 8] : v[j]) * gsv;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int col = c0 + (is_up ? 8 : 0) + j;
              const float g = is_up ? other[j] : mine[j];
              const float upv = is_up ? mine[j] : other[j];
              if (col < U.rows && i < p.inter_pad)
                p.h_out[(size_t)(U.slot0 + col) * p.inter_pad + i] = float_to_bf16_bits(gated_act(g, upv, p.glu));
            }
          } else {
            const int i = U.tile * kTileRows + er;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c0 + j;
              const float a = __uint_as_float(v[j]) * gsv;
              if (col < U.rows && i < p.inter_pad)
                p.h_out[(size_t)(U.slot0 + col) * p.inter_pad + i] =
                    float_to_bf16_bits(p.act == 2 ? a : (a > 0.f ? a * a : 0.f));
            }
          }
        } else {
          const int n = U.tile * kTileRows + er;
          if (n < p.hidden) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c0 + j;
              if (col < U.rows)
                red_add_f32(p.acc_out + (size_t)s_tok[col] * p.hidden + n, __uint_as_float(v[j]) * gsv * s_wt[col]);
            }
          }
        }
      }
      tc_fence_before();
      if constexpr (MODE == kFc2Grouped) named_bar_sync(2, 128);  // route table free for the next unit
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty_acc[abuf]);
        if (warp == 12) trace_mark(p, 4, acc_i);
      }
      ++acc_i;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ----------------------------------------------------- host-side launchers
template <int MODE, int FMT>
cudaError_t launch_gemm(const GemmParams& p, int grid, bool pdl, cudaStream_t stream) {
  auto kern = moe_gemm_kernel<MODE, FMT>;
  const size_t smem = SmemLayout<FMT>::total;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template cudaError_t launch_gemm<kFc1Grouped, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc2Grouped, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc1Grouped, 1>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc2Grouped, 1>(const GemmParams&, int, bool, cudaStream_t);

}  // namespace b4
