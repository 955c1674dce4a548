// Grouped W4A16 GEMMs of the fused MoE layer on tcgen05 (sm_103a), weights on
// the N side: the form used when experts receive few routes (see the
// dispatch in api.cu; moe_gemm.cu is the form for many routes per expert).
//
// One persistent, warp-specialised kernel serves the two route-packed GEMMs
// (flashinfer PR #4255, Description: "Cooperative persistent launches for the
// fused FC1/FC2 kernel", "folding the top-k sum into the FC2 store
// epilogue"):
//
//   FC1  activations = x rows of the routes of one expert chunk, copied into
//        packed-route order by the route pack; the epilogue applies
//        SiLU-SwiGLU or ReLU^2 (none for the dense linear layer) and
//        stores bf16 h in the same order.
//   FC2  activations = h rows of the chunk; the epilogue multiplies by gs2 and
//        the router weight and adds into an fp32 [tokens, H] accumulator (the
//        top-k sum), which finalize_grouped_kernel rounds to bf16.
//
// A work unit is (expert chunk of <= 128 routes, pair of 128-row weight
// tiles).  The tensor-core operation: M = the chunk's routes (A, K-major in
// shared memory, loaded by TMA in 32-row 2-D boxes with the 128-byte
// swizzle), N = 256 weight rows (B, K-major in shared memory, 128-byte
// swizzle), fp32 accumulators in tensor memory.  With few routes per expert,
// putting 256 weight rows on N does the work of two weights-on-M
// instructions (whose N would be the few routes, padded to 16) in one, and
// the expert's weights are dequantised once per 128 routes.  Weights are dequantised from E2M1 codes and E4M3 / E8M0 block scales
// to bf16 by sixteen dequant warps and stored in the swizzled B layout.
// Roles, one CTA of 24 warps:
//   warp 0       bulk-copy (TMA engine) producer of packed codes and scales
//   warp 1       TMEM allocator and the single MMA-issuing thread
//   warp 2       activation producer (TMA tile loads)
//   warps 4-19   dequantisers (two threads per weight row, 32 K each)
//   warps 20-23  epilogue: tensor-memory accumulators -> outputs (one
//                thread per route, 16 contiguous outputs per load)
// Rings: weights (6 stages); activation and weight operand stages (3, one
// index, one release commit per stage); two accumulators of 256 columns, so
// the epilogue of one unit overlaps the next mainloop.
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
namespace wn {

constexpr int kThreads = 768;
constexpr int kDqWarps = 16;                    // dequantisers: two threads per weight row
constexpr int kNW = 6;                          // weight code/scale stages in flight
constexpr int kNS = 3;                          // operand stages (activations + weights)
constexpr int kBM = kChunkRowsN;                // 128 routes
constexpr int kBN = 2 * kTileRows;              // 256 weight rows
constexpr int kAStage = kBM * kBK * 2;          // 16 KB, swizzled
constexpr int kBStage = kBN * kBK * 2;          // 32 KB, swizzled
constexpr uint32_t kTmemCols = 512;             // two accumulators of kBN columns
constexpr float kTwo63 = 9.223372036854775808e18f;
static_assert(2 * kBN <= (int)kTmemCols, "tensor memory budget");
static_assert(kAStage % 1024 == 0 && kBStage % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");

template <int FMT>
struct SmemLayout {
  static constexpr int kScaleStage = scale_bytes_per_stage(FMT);
  static constexpr size_t a = 0;  // offset from the 1024-aligned base
  static constexpr size_t b = a + (size_t)kNS * kAStage;
  static constexpr size_t codes = b + (size_t)kNS * kBStage;
  static constexpr size_t scales = codes + (size_t)kNW * 2 * kCodeBytesPerStage;
  static constexpr size_t bars = round_up((int)(scales + (size_t)kNW * 2 * kScaleStage), 8);
  static constexpr int kNumBars = 2 * kNW + 3 * kNS + 4 + 1;
  static constexpr size_t misc = bars + 8 * kNumBars;
  static constexpr size_t total = misc + 16 + 1024;  // + alignment slack
};

struct Unit {
  int expert, pair, slot0, rows, ntiles;
  int kbeg, kend;  // K stages of the unit (a K split of FC2 adds its partial like any other)
};

__device__ __forceinline__ int num_pairs(const GemmParams& p) { return (p.n_tiles + 1) >> 1; }

__device__ __forceinline__ int num_chunks(const GemmParams& p) {
  const int c = *(volatile const int32_t*)p.chunk_count;
  return c < 0 ? 0 : (c > p.max_chunks ? p.max_chunks : c);
}

// K splits of every unit: p.k_splits when above 1; when negative (automatic,
// FC2 only), enough for about two units per CTA, at most 4 and with at least
// 4 stages each; otherwise none.  Every thread computes the same value from
// the chunk count.
__device__ __forceinline__ int num_ksplits(const GemmParams& p, int chunks) {
  if (p.k_splits > 1) return p.k_splits;
  if (p.k_splits < 0 && chunks > 0) {
    const int base = chunks * num_pairs(p);
    const int most = p.k_stages / 4 < 4 ? p.k_stages / 4 : 4;
    int ns = (2 * (int)gridDim.x + base - 1) / base;
    ns = ns < most ? ns : most;
    return ns > 1 ? ns : 1;
  }
  return 1;
}

// Unit u = ((chunk * pairs) + pair) * splits + split.
__device__ __forceinline__ bool get_unit(const GemmParams& p, int u, int ns, Unit& U) {
  const int np = num_pairs(p);
  if (ns > 1) {
    const int ks = u % ns;
    u /= ns;
    U.kbeg = ks * p.k_stages / ns;  // k_stages * splits stays far below 2^31
    U.kend = (ks + 1) * p.k_stages / ns;
  } else {
    U.kbeg = 0;
    U.kend = p.k_stages;
  }
  const int c = u / np;
  U.pair = u - c * np;
  U.ntiles = min(2, p.n_tiles - 2 * U.pair);
  const int4 ch = p.chunks[c];
  U.expert = ch.x;
  U.slot0 = ch.y;
  U.rows = ch.z;
  return U.rows > 0 && U.kend > U.kbeg;
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

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Abort& ab, uint32_t where) {
  const bool ok = mbar_wait(bar, parity, ab, where);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// ------------------------------------------------------------------ kernel
template <int MODE, int FMT>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using L = SmemLayout<FMT>;
  constexpr int NW = kNW, NS = kNS;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int kScaleStage = L::kScaleStage;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled operand stages need 1024-byte alignment of the shared address
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* s_a = smem + L::a;
  uint8_t* s_b = smem + L::b;
  uint8_t* s_codes = smem + L::codes;
  uint8_t* s_scales = smem + L::scales;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + NW;
  uint64_t* full_a = empty_w + NW;
  uint64_t* full_b = full_a + NS;
  uint64_t* stage_free = full_b + NS;  // activation and weight stage of a ring index, freed by one commit
  uint64_t* full_acc = stage_free + NS;
  uint64_t* empty_acc = full_acc + 2;
  uint64_t* drain = empty_acc + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Abort ab{p.status, s_abort};

  if (threadIdx.x == 0) {
    *s_abort = 0;
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&empty_w[i], kDqWarps);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full_a[i], 1);
      mbar_init(&full_b[i], kDqWarps);
      mbar_init(&stage_free[i], 1);
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

  const int n_chunks = num_chunks(p);
  const int n_split = num_ksplits(p, n_chunks);
  const int n_units = n_chunks * num_pairs(p) * n_split;
  const size_t wtile_codes = (size_t)p.k_stages * kCodeBytesPerStage;
  const size_t wtile_scales = (size_t)p.k_stages * kScaleStage;

  if (warp == 0) {
    // ------------------------------------------------ weight producer
    uint32_t ws = 0;
    if (lane == 0) {
      for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
        Unit U;
        if (!get_unit(p, u, n_split, U)) continue;
        const size_t tile0 = (size_t)U.expert * p.n_tiles + 2 * U.pair;
        for (int s = U.kbeg; s < U.kend; ++s, ++ws) {
          const uint32_t slot = ws % NW;
          if (!mbar_wait(&empty_w[slot], ((ws / NW) & 1) ^ 1, ab, 1)) break;
          mbar_arrive_expect_tx(&full_w[slot], U.ntiles * (kCodeBytesPerStage + kScaleStage));
          for (int t = 0; t < U.ntiles; ++t) {
            bulk_g2s(s_codes + (slot * 2 + t) * kCodeBytesPerStage,
                     p.wcodes + (tile0 + t) * wtile_codes + (size_t)s * kCodeBytesPerStage, kCodeBytesPerStage,
                     &full_w[slot]);
            bulk_g2s(s_scales + (slot * 2 + t) * kScaleStage,
                     p.wscales + (tile0 + t) * wtile_scales + (size_t)s * kScaleStage, kScaleStage, &full_w[slot]);
          }
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
      uint32_t ss = 0, acc_i = 0;
      const uint32_t a_base = smem_u32(s_a), b_base = smem_u32(s_b);
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        Unit U;
        if (!get_unit(p, u, n_split, U)) continue;
        const uint32_t abuf = acc_i & 1;
        if (!mbar_wait(&empty_acc[abuf], ((acc_i >> 1) & 1) ^ 1, ab, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + abuf * kBN;
        const uint32_t idesc = idesc_bf16_m128((uint32_t)(U.ntiles * kTileRows));
        bool ok = true;
        for (int s = U.kbeg; s < U.kend; ++s, ++ss) {
          const uint32_t slot = ss % NS;
          if (!mbar_wait(&full_a[slot], (ss / NS) & 1, ab, 3) || !mbar_wait(&full_b[slot], (ss / NS) & 1, ab, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + slot * kAStage + kk * 32);
            const uint64_t bdesc = smem_desc_sw128(b_base + slot * kBStage + kk * 32);
            mma_bf16_ss(d_tmem, adesc, bdesc, idesc, (s > U.kbeg || kk > 0) ? 1u : 0u);
          }
          mma_commit(&stage_free[slot]);
          trace_mark(p, 2, ss);
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
    // ---------------------------------------------- activation producer
    if (MODE == kFc2Grouped) pdl_wait();  // h comes from FC1 (FC1 waited for its inputs at entry)
    uint32_t ss = 0;
    for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
      Unit U;
      if (!get_unit(p, u, n_split, U)) continue;
      const int nload = cdiv(U.rows, 32);
      const uint32_t bytes = (uint32_t)nload * 4096u;
      bool ok = true;
      for (int s = U.kbeg; s < U.kend; ++s, ++ss) {
        const uint32_t slot = ss % NS;
        if (!warp_wait(&stage_free[slot], ((ss / NS) & 1) ^ 1, ab, 5)) {
          ok = false;
          break;
        }
        uint8_t* stage = s_a + slot * kAStage;
        if (lane == 0) mbar_arrive_expect_tx(&full_a[slot], bytes);
        __syncwarp();
        for (int i = lane; i < nload; i += 32)
          tma_load_2d(stage + i * 4096, &p.tmap_b, s * kBK, U.slot0 + 32 * i, &full_a[slot]);
        if (lane == 0) trace_mark(p, 3, ss);
      }
      if (!ok) break;
    }
    if (ab.raised() && lane == 0) {
      // let issued loads land before the CTA exits
      const uint32_t n = ss < (uint32_t)NS ? ss : (uint32_t)NS;
      for (uint32_t i = ss - n; i < ss; ++i) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&full_a[i % NS], (i / NS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + kDqWarps) {
    // ------------------------------------------------------ dequantisers
    // two threads per weight row of the tile pair, one per 32-element half of
    // the stage; 16-byte chunk c of a row is stored at position c ^ (row % 8)
    // of its 128-byte row (the 128-byte swizzle the MMA descriptor expects)
    const int dq = threadIdx.x - 128;  // 0..511
    const int row = dq & (kBN - 1), half = dq >> 8;
    const int tl = row >> 7, trow = row & (kTileRows - 1);
    uint32_t ws = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit(p, u, n_split, U)) continue;
      const bool active = tl < U.ntiles;
      bool ok = true;
      for (int s = U.kbeg; s < U.kend; ++s, ++ws) {
        const uint32_t wslot = ws % NW, slot = ws % NS;
        if (!warp_wait(&full_w[wslot], (ws / NW) & 1, ab, 6)) {
          ok = false;
          break;
        }
        uint4 c = make_uint4(0, 0, 0, 0);
        uint32_t sc = 0;
        if (active) {
          const uint8_t* cs = s_codes + (wslot * 2 + tl) * kCodeBytesPerStage;
          c = *reinterpret_cast<const uint4*>(cs + half * 2048 + trow * 16);
          const uint8_t* scp = s_scales + (wslot * 2 + tl) * kScaleStage + trow * SB;
          if constexpr (SB == 4) sc = *reinterpret_cast<const uint32_t*>(scp);
          else sc = *reinterpret_cast<const uint16_t*>(scp);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_w[wslot]);
        uint32_t r[16];
        dequant_half<FMT>(c, sc, half, r);
        if (!warp_wait(&stage_free[slot], ((ws / NS) & 1) ^ 1, ab, 7)) {
          ok = false;
          break;
        }
        if (active) {
          uint8_t* dst = s_b + slot * kBStage + row * 128;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int cch = 4 * half + j;
            *reinterpret_cast<uint4*>(dst + ((cch ^ (row & 7)) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();  // generic stores -> the tensor core's async-proxy reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full_b[slot]);
          if (warp == 4) trace_mark(p, 1, ws);
        }
      }
      if (!ok) break;
    }
  } else if (warp >= 4 + kDqWarps) {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int er = 32 * q4 + lane;  // TMEM lane == route row of the chunk
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    if constexpr (MODE == kFc1Grouped) {
      // clear the FC2 accumulator (FC2 waits for this grid before adding)
      float4* z = reinterpret_cast<float4*>(p.acc_out);
      const size_t n4 = p.acc_zero_floats / 4;
      for (size_t i = (size_t)blockIdx.x * 128 + er; i < n4; i += (size_t)gridDim.x * 128)
        z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if constexpr (MODE == kFc2Grouped) pdl_wait();  // acc_out cleared by FC1
    uint32_t acc_i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit(p, u, n_split, U)) continue;
      const uint32_t abuf = acc_i & 1;
      const bool live = er < U.rows;
      // per-route constants, resolved before the wait
      float gsv = (p.gs ? __ldg(p.gs + U.expert) : 1.0f) * kTwo63;
      int token = 0;
      if (MODE == kFc2Grouped && live) {
        const int route = __ldg(p.sorted_routes + U.slot0 + er);
        token = route / p.top_k;
        if (p.topk_weights) gsv *= __ldg(p.topk_weights + route);  // null: weight 1 (the dense linear layer)
      }
      if (!warp_wait(&full_acc[abuf], (acc_i >> 1) & 1, ab, 8)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_base + abuf * kBN;
      for (int t = 0; t < U.ntiles; ++t) {
        const int tile = 2 * U.pair + t;
        if constexpr (MODE == kFc1Grouped) {
          if (p.act == 0) {
            // columns 32q..32q+15 of a tile: gate of h[64 tile + 16q + l]; +16: up
            for (int q = 0; q < 4; ++q) {
              uint32_t g[16], v[16];
              tmem_ld16(taddr + t * kTileRows + 32 * q, g);
              tmem_ld16(taddr + t * kTileRows + 32 * q + 16, v);
              tmem_ld_wait();
              const int i0 = tile * 64 + q * 16;
              if (live && i0 < p.inter_pad) {
                uint32_t o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float a0 = __uint_as_float(g[2 * j]) * gsv, a1 = __uint_as_float(g[2 * j + 1]) * gsv;
                  const float b0 = __uint_as_float(v[2 * j]) * gsv, b1 = __uint_as_float(v[2 * j + 1]) * gsv;
                  o[j] = pack_bf16x2(gated_act(a0, b0, p.glu), gated_act(a1, b1, p.glu));
                }
                uint4* dst = reinterpret_cast<uint4*>(p.h_out + (size_t)(U.slot0 + er) * p.inter_pad + i0);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
              }
            }
          } else {
            for (int q = 0; q < kTileRows / 16; ++q) {
              uint32_t v[16];
              tmem_ld16(taddr + t * kTileRows + 16 * q, v);
              tmem_ld_wait();
              const int i0 = tile * kTileRows + q * 16;
              if (live && i0 < p.inter_pad) {
                uint32_t o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float a0 = __uint_as_float(v[2 * j]) * gsv, a1 = __uint_as_float(v[2 * j + 1]) * gsv;
                  o[j] = p.act == 2 ? pack_bf16x2(a0, a1)
                                    : pack_bf16x2(a0 > 0.f ? a0 * a0 : 0.f, a1 > 0.f ? a1 * a1 : 0.f);
                }
                uint4* dst = reinterpret_cast<uint4*>(p.h_out + (size_t)(U.slot0 + er) * p.inter_pad + i0);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
              }
            }
          }
        } else {
          for (int q = 0; q < kTileRows / 16; ++q) {
            uint32_t v[16];
            tmem_ld16(taddr + t * kTileRows + 16 * q, v);
            tmem_ld_wait();
            const int n0 = tile * kTileRows + q * 16;
            if (live && n0 < p.hidden) {  // H is a multiple of 16: all 16 are in range
              float* dst = p.acc_out + (size_t)token * p.hidden + n0;
#pragma unroll
              for (int j = 0; j < 16; j += 4)
                red_add_f32x4(dst + j, __uint_as_float(v[j]) * gsv, __uint_as_float(v[j + 1]) * gsv,
                              __uint_as_float(v[j + 2]) * gsv, __uint_as_float(v[j + 3]) * gsv);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty_acc[abuf]);
        if (warp == 4 + kDqWarps) trace_mark(p, 4, acc_i);
      }
      ++acc_i;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace wn

// ----------------------------------------------------- host-side launchers
template <int MODE, int FMT>
cudaError_t launch_gemm_wn(const GemmParams& p, int grid, bool pdl, cudaStream_t stream) {
  using namespace wn;
  auto kern = wn::moe_gemm_kernel<MODE, FMT>;
  const size_t smem = wn::SmemLayout<FMT>::total;
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

template cudaError_t launch_gemm_wn<kFc1Grouped, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm_wn<kFc2Grouped, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm_wn<kFc1Grouped, 1>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm_wn<kFc2Grouped, 1>(const GemmParams&, int, bool, cudaStream_t);

}  // namespace b4
