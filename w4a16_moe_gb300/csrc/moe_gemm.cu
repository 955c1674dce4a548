// Grouped W4A16 GEMMs of the fused MoE layer on tcgen05 (sm_103a).
//
// One persistent, warp-specialised kernel serves the four GEMMs of the layer
// (flashinfer PR #4255, Description: "Cooperative persistent launches for the
// fused FC1/FC2 kernel", "A tensor-core decode path for small batches ...
// folding the top-k sum into the FC2 store epilogue"):
//
//   FC1 grouped  routes packed by expert; B = gathered x rows; epilogue applies
//                the SiLU-SwiGLU or ReLU^2 activation and stores bf16 h.
//   FC2 grouped  B = h rows; epilogue multiplies by gs2 and the router weight
//                and adds into an fp32 [tokens, H] accumulator (the top-k sum).
//   FC1 decode   one route per work unit, K split across units; epilogue
//                stores fp32 partial sums.
//   FC2 decode   B = activation of the summed FC1 partials (computed while
//                loading); epilogue stores gs2 * w * y partials.
//
// The tensor-core operation is swapped: the 128 weight rows of a tile are the
// M operand, the routes are N.  Weights are dequantised from E2M1 codes and
// E4M3 / E8M0 block scales to bf16 by four dequant warps (one thread per
// weight row) and written straight into tensor memory with tcgen05.st, where
// tcgen05.mma reads them as its A operand; B (activations) is staged in
// shared memory.  Roles, one CTA of 12 warps:
//   warp 0       bulk-copy (TMA engine) producer of packed codes and scales
//   warp 1       TMEM allocator and the single MMA-issuing thread
//   warps 2-3    B loaders (cp.async gathers, or computed rows in FC2 decode)
//   warps 4-7    dequantisers: shared memory codes -> bf16 -> tensor memory
//   warps 8-11   epilogue: tensor memory accumulators -> outputs
// Four mbarrier rings connect them (weights, A slots in TMEM, B stages,
// double-buffered accumulators); every wait is bounded (ptx.cuh).
//
// Dequantised weights carry a factor 2^-63 so that every product of an E2M1
// code and a block scale is a normal bf16; the epilogue multiplies by 2^63.

#include <cuda_bf16.h>

#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

constexpr int kNumA = 4;          // A slots (K stages) held in tensor memory
constexpr int kThreads = 384;
constexpr int kAColsPerSlot = kBK / 2;  // 32 columns of packed bf16 pairs
constexpr float kTwo63 = 9.223372036854775808e18f;

template <int MODE>
struct ModeTraits {
  static constexpr bool kGrouped = MODE == kFc1Grouped || MODE == kFc2Grouped;
  static constexpr bool kFc1 = MODE == kFc1Grouped || MODE == kFc1Decode;
  static constexpr int kNW = kGrouped ? 8 : 16;       // weight stages
  static constexpr int kNB = 4;                        // B stages
  static constexpr int kBN = kGrouped ? kChunkRows : 16;  // max tcgen05 N
  static constexpr uint32_t kTmemCols = kGrouped ? 512 : 256;
  static constexpr uint32_t kAccCol0 = kNumA * kAColsPerSlot;  // 128
  static constexpr int kLag = kGrouped ? 2 : 1;       // cp.async stages in flight per loader
};

template <int MODE, int FMT>
struct SmemLayout {
  using T = ModeTraits<MODE>;
  static constexpr int kScaleStage = scale_bytes_per_stage(FMT);
  static constexpr int kBStage = T::kBN * kBK * 2;
  static constexpr size_t codes = 0;
  static constexpr size_t scales = codes + (size_t)T::kNW * kCodeBytesPerStage;
  static constexpr size_t b = round_up((int)(scales + (size_t)T::kNW * kScaleStage), 128);
  static constexpr size_t bars = b + (size_t)T::kNB * kBStage;
  static constexpr int kNumBars = 2 * T::kNW + 2 * kNumA + 2 * T::kNB + 4 + 1;
  static constexpr size_t misc = bars + 8 * kNumBars;
  static constexpr size_t rows = misc + 16;
  static constexpr size_t total = rows + 4 * T::kBN + 64;
};

struct Unit {
  int expert, tile, kbeg, kend, slot0, rows, route, split;
};

__device__ __forceinline__ int local_expert_of(const GemmParams& p, int route) {
  const int id = __ldg(p.topk_ids + route);
  if (id < 0 || id >= p.num_global_experts) return -1;
  const int l = p.expert_map ? __ldg(p.expert_map + id) : id;
  return (l >= 0 && l < p.num_local_experts) ? l : -1;
}

template <int MODE>
__device__ __forceinline__ int num_units(const GemmParams& p) {
  if constexpr (ModeTraits<MODE>::kGrouped) {
    int c = *(volatile const int32_t*)p.chunk_count;
    c = c < 0 ? 0 : (c > p.max_chunks ? p.max_chunks : c);
    return c * p.n_tiles;
  } else {
    return p.m * p.top_k * p.n_tiles * p.splits;
  }
}

// Returns false for a unit with nothing to do (a dropped route in decode).
template <int MODE>
__device__ __forceinline__ bool get_unit(const GemmParams& p, int u, Unit& U) {
  if constexpr (ModeTraits<MODE>::kGrouped) {
    const int c = u / p.n_tiles;
    U.tile = u - c * p.n_tiles;
    const int4 ch = p.chunks[c];
    U.expert = ch.x;
    U.slot0 = ch.y;
    U.rows = ch.z;
    U.kbeg = 0;
    U.kend = p.k_stages;
    U.route = -1;
    U.split = 0;
    return U.rows > 0;
  } else {
    const int per_route = p.n_tiles * p.splits;
    U.route = u / per_route;
    const int rem = u - U.route * per_route;
    U.tile = rem / p.splits;
    U.split = rem - U.tile * p.splits;
    U.kbeg = (int)((long long)U.split * p.k_stages / p.splits);
    U.kend = (int)((long long)(U.split + 1) * p.k_stages / p.splits);
    U.slot0 = U.route;
    U.rows = 1;
    U.expert = local_expert_of(p, U.route);
    return U.expert >= 0 && U.kend > U.kbeg;
  }
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Abort& ab, uint32_t where) {
  const bool ok = mbar_wait(bar, parity, ab, where);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// ------------------------------------------------------------------ kernel
template <int MODE, int FMT>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using T = ModeTraits<MODE>;
  using L = SmemLayout<MODE, FMT>;
  constexpr int NW = T::kNW, NB = T::kNB, BN = T::kBN;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int kScaleStage = L::kScaleStage;

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_codes = smem + L::codes;
  uint8_t* s_scales = smem + L::scales;
  uint8_t* s_b = smem + L::b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + NW;
  uint64_t* full_a = empty_w + NW;
  uint64_t* empty_a = full_a + kNumA;
  uint64_t* full_b = empty_a + kNumA;
  uint64_t* empty_b = full_b + NB;
  uint64_t* full_acc = empty_b + NB;
  uint64_t* empty_acc = full_acc + 2;
  uint64_t* drain = empty_acc + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc + 4);
  int32_t* s_rows = reinterpret_cast<int32_t*>(smem + L::rows);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Abort ab{p.status, s_abort};

  if (threadIdx.x == 0) {
    if (p.clear_status && blockIdx.x == 0 && p.status) {
      p.status[0] = 0;
      p.status[1] = 0;
    }
    *s_abort = 0;
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&empty_w[i], 4);
    }
    for (int i = 0; i < kNumA; ++i) {
      mbar_init(&full_a[i], 4);
      mbar_init(&empty_a[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&full_b[i], 64);
      mbar_init(&empty_b[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_acc[i], 1);
      mbar_init(&empty_acc[i], 4);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, T::kTmemCols);
    tmem_relinquish();
  }
  // B stages start as zeros: rows beyond a unit's routes then stay finite.
  if (warp == 2 || warp == 3) {
    uint4* z = reinterpret_cast<uint4*>(s_b);
    for (int i = threadIdx.x - 64; i < NB * L::kBStage / 16; i += 64) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (p.pdl_wait_first) pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int n_units = num_units<MODE>(p);
  const size_t wtile_codes = (size_t)p.k_stages * kCodeBytesPerStage;
  const size_t wtile_scales = (size_t)p.k_stages * kScaleStage;

  if (warp == 0) {
    // ------------------------------------------------ weight producer
    uint32_t ws = 0;
    if (lane == 0) {
      for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
        Unit U;
        if (!get_unit<MODE>(p, u, U)) continue;
        const size_t tile_id = (size_t)U.expert * p.n_tiles + U.tile;
        const uint8_t* gc = p.wcodes + tile_id * wtile_codes;
        const uint8_t* gsc = p.wscales + tile_id * wtile_scales;
        for (int s = U.kbeg; s < U.kend; ++s, ++ws) {
          const uint32_t slot = ws % NW;
          if (!mbar_wait(&empty_w[slot], ((ws / NW) & 1) ^ 1, ab, 1)) break;
          mbar_arrive_expect_tx(&full_w[slot], kCodeBytesPerStage + kScaleStage);
          bulk_g2s(s_codes + slot * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage, kCodeBytesPerStage,
                   &full_w[slot]);
          bulk_g2s(s_scales + slot * kScaleStage, gsc + (size_t)s * kScaleStage, kScaleStage, &full_w[slot]);
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
        if (!get_unit<MODE>(p, u, U)) continue;
        const uint32_t abuf = acc_i & 1;
        if (!mbar_wait(&empty_acc[abuf], ((acc_i >> 1) & 1) ^ 1, ab, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + T::kAccCol0 + abuf * BN;
        const uint32_t n16 = T::kGrouped ? (uint32_t)round_up(U.rows, 16) : 16u;
        const uint32_t idesc = idesc_bf16_m128(n16);
        bool ok = true;
        for (int s = U.kbeg; s < U.kend; ++s, ++as, ++bs) {
          const uint32_t aslot = as % kNumA, bslot = bs % NB;
          if (!mbar_wait(&full_a[aslot], (as / kNumA) & 1, ab, 3) ||
              !mbar_wait(&full_b[bslot], (bs / NB) & 1, ab, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t a_tmem = tmem_base + aslot * kAColsPerSlot + kk * 8;
            const uint64_t bdesc = smem_desc_noswizzle(b_base + bslot * L::kBStage + kk * 256, 128, 1024);
            mma_bf16_ts(d_tmem, a_tmem, bdesc, idesc, (s > U.kbeg || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty_a[aslot]);
          mma_commit(&empty_b[bslot]);
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
  } else if (warp == 2 || warp == 3) {
    // -------------------------------------------------------- B loaders
    const int lt = threadIdx.x - 64;
    const uint32_t b_base = smem_u32(s_b);
    uint32_t bs = 0, arrived = 0;
    if (MODE == kFc2Grouped || MODE == kFc2Decode) pdl_wait();  // h / FC1 partials come from FC1
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit<MODE>(p, u, U)) continue;
      if constexpr (T::kGrouped) {
        named_bar_sync(1, 64);  // previous unit's row table no longer read
        for (int i = lt; i < U.rows; i += 64) {
          const int slot = U.slot0 + i;
          s_rows[i] = MODE == kFc1Grouped ? __ldg(p.sorted_routes + slot) / p.top_k : slot;
        }
        named_bar_sync(1, 64);
      }
      bool ok = true;
      for (int s = U.kbeg; s < U.kend; ++s, ++bs) {
        const uint32_t slot = bs % NB;
        if (!warp_wait(&empty_b[slot], ((bs / NB) & 1) ^ 1, ab, 5)) {
          ok = false;
          break;
        }
        const uint32_t stage = b_base + slot * L::kBStage;
        const int k0 = s * kBK;
        if constexpr (MODE == kFc2Decode) {
          // h[i] = act(gs13 * 2^63 * sum of FC1 partials) for i = k0 + lt
          const int i = k0 + lt;
          const int R = p.m * p.top_k;
          const int wnat = fc1_natural_width(p.act, p.inter_pad);
          const float* pr = p.p_in + (size_t)U.route * wnat;
          float g = 0.f, up = 0.f;
          for (int sp = 0; sp < p.splits_in; ++sp) {
            const float* q = pr + (size_t)sp * R * wnat;
            g += q[i];
            if (p.act == 0) up += q[p.inter_pad + i];
          }
          // gs13 travels in p_in's companion: p.gs here is the FC2 scale, so
          // the FC1 scale was folded into the partials by the FC1 epilogue.
          const float hv = p.act == 0 ? silu_f(g) * up : (g > 0.f ? g * g : 0.f);
          const uint16_t hb = float_to_bf16_bits(hv);
          const uint32_t off = (uint32_t)(lt >> 3) * 128 + (lt & 7) * 2;
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(stage + off), "h"(hb) : "memory");
          fence_proxy_async_smem();
          mbar_arrive(&full_b[slot]);
          ++arrived;
        } else {
          const int kc = lt >> 3;    // 16-byte chunk along K: 0..7
          const int nlo = lt & 7;    // row within an 8-row group
          const int ke = k0 + kc * 8;
          const int kvalid = MODE == kFc1Grouped || MODE == kFc1Decode ? p.hidden : p.inter_pad;
          const uint32_t src_bytes = ke < kvalid ? 16u : 0u;
          const int nrows = T::kGrouped ? U.rows : 1;
          const int ngroups = cdiv(nrows, 8);
          for (int gi = 0; gi < ngroups; ++gi) {
            const int n = gi * 8 + nlo;
            if (n >= nrows) break;
            const uint16_t* row;
            if constexpr (MODE == kFc1Grouped) row = p.x + (size_t)s_rows[n] * p.hidden;
            else if constexpr (MODE == kFc2Grouped) row = p.h + (size_t)s_rows[n] * p.inter_pad;
            else row = p.x + (size_t)(U.route / p.top_k) * p.hidden;
            const uint16_t* src = src_bytes ? row + ke : p.x;
            cp_async16(stage + gi * 1024 + kc * 128 + nlo * 16, src, src_bytes);
          }
          if constexpr (T::kGrouped) {
            // zero-fill rows [rows, roundup16(rows)) so the padded columns stay finite
            const int n16 = round_up(U.rows, 16);
            for (int n = U.rows + nlo - (U.rows & 7); n < n16; n += 8) {
              if (n >= U.rows) cp_async16(stage + (n >> 3) * 1024 + kc * 128 + (n & 7) * 16, p.x, 0);
            }
          }
          cp_async_commit();
          // delayed arrival: stage bs - kLag has landed once <= kLag groups remain
          if (bs + 1 - arrived > (uint32_t)T::kLag) {
            cp_async_wait<T::kLag>();
            fence_proxy_async_smem();
            mbar_arrive(&full_b[arrived % NB]);
            ++arrived;
          }
        }
      }
      if (!ok) break;
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    while (arrived < bs && !ab.raised()) {
      mbar_arrive(&full_b[arrived % NB]);
      ++arrived;
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------ dequantisers
    const int row = threadIdx.x - 128;  // == 32 * (warp % 4) + lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t ws = 0, as = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit<MODE>(p, u, U)) continue;
      bool ok = true;
      for (int s = U.kbeg; s < U.kend; ++s, ++ws, ++as) {
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
        const uint32_t aslot = as % kNumA;
        if (!warp_wait(&empty_a[aslot], ((as / kNumA) & 1) ^ 1, ab, 7)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st32(tmem_base + lane_base + aslot * kAColsPerSlot, r);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_a[aslot]);
      }
      if (!ok) break;
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int er = 32 * q4 + lane;  // TMEM lane == weight row in the tile
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    if constexpr (MODE == kFc1Grouped) {
      // clear the FC2 accumulator (FC2 waits for this grid before adding)
      float4* z = reinterpret_cast<float4*>(p.acc_out);
      const size_t n4 = p.acc_zero_floats / 4;
      for (size_t i = (size_t)blockIdx.x * 128 + (threadIdx.x - 256); i < n4; i += (size_t)gridDim.x * 128)
        z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if constexpr (MODE == kFc2Grouped) pdl_wait();  // acc_out cleared by FC1
    uint32_t acc_i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit U;
      if (!get_unit<MODE>(p, u, U)) continue;
      const uint32_t abuf = acc_i & 1;
      if (!warp_wait(&full_acc[abuf], (acc_i >> 1) & 1, ab, 8)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_base + T::kAccCol0 + abuf * BN;
      const float gsv = (p.gs ? __ldg(p.gs + U.expert) : 1.0f) * kTwo63;
      const int ncols = T::kGrouped ? round_up(U.rows, 16) : 16;
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
                p.h_out[(size_t)(U.slot0 + col) * p.inter_pad + i] = float_to_bf16_bits(silu_f(g) * upv);
            }
          } else {
            const int i = U.tile * kTileRows + er;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c0 + j;
              const float a = __uint_as_float(v[j]) * gsv;
              if (col < U.rows && i < p.inter_pad)
                p.h_out[(size_t)(U.slot0 + col) * p.inter_pad + i] = float_to_bf16_bits(a > 0.f ? a * a : 0.f);
            }
          }
        } else if constexpr (MODE == kFc2Grouped) {
          const int n = U.tile * kTileRows + er;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col < U.rows) {
              const int route = __ldg(p.sorted_routes + U.slot0 + col);
              const float wt = __ldg(p.topk_weights + route);
              if (n < p.hidden)
                red_add_f32(p.acc_out + (size_t)(route / p.top_k) * p.hidden + n,
                            __uint_as_float(v[j]) * gsv * wt);
            }
          }
        } else if constexpr (MODE == kFc1Decode) {
          // natural index of this prepared row; partials carry gs13 * 2^63
          const int R = p.m * p.top_k;
          const int wnat = fc1_natural_width(p.act, p.inter_pad);
          int nat;
          if (p.act == 0) {
            const int i = U.tile * 64 + q4 * 16 + (lane & 15);
            nat = lane >= 16 ? p.inter_pad + i : i;
          } else {
            nat = U.tile * kTileRows + er;
            if (nat >= p.inter_pad) nat = -1;
          }
          if (nat >= 0)
            p.part_out[((size_t)U.split * R + U.route) * wnat + nat] = __uint_as_float(v[0]) * gsv;
        } else {
          const int R = p.m * p.top_k;
          const int n = U.tile * kTileRows + er;
          const float wt = __ldg(p.topk_weights + U.route);
          if (n < p.hidden)
            p.part_out[((size_t)U.split * R + U.route) * p.hidden + n] = __uint_as_float(v[0]) * gsv * wt;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_acc[abuf]);
      ++acc_i;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, T::kTmemCols);
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
  pdl_wait();
  const int R = p.m * p.top_k;
  const size_t total = (size_t)p.m * p.hidden;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / p.hidden);
    const int n = (int)(i - (size_t)t * p.hidden);
    float acc = 0.f;
    for (int j = 0; j < p.top_k; ++j) {
      const int route = t * p.top_k + j;
      const int id = p.topk_ids[route];
      if (id < 0 || id >= p.num_global_experts) continue;
      const int l = p.expert_map ? p.expert_map[id] : id;
      if (l < 0 || l >= p.num_local_experts) continue;
      for (int sp = 0; sp < p.splits; ++sp) acc += p.q[((size_t)sp * R + route) * p.hidden + n];
    }
    p.out[i] = float_to_bf16_bits(acc);
  }
}

// ----------------------------------------------------- host-side launchers
template <int MODE, int FMT>
size_t gemm_smem_bytes() {
  return SmemLayout<MODE, FMT>::total;
}

template <int MODE, int FMT>
cudaError_t launch_gemm(const GemmParams& p, int grid, bool pdl, cudaStream_t stream) {
  auto kern = moe_gemm_kernel<MODE, FMT>;
  const size_t smem = SmemLayout<MODE, FMT>::total;
  static bool configured = false;  // attribute set once per process (idempotent)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
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

cudaError_t launch_finalize(const FinalizeParams& p, bool grouped, int num_sms, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  const size_t total = grouped ? (size_t)p.m * p.hidden / 4 : (size_t)p.m * p.hidden;
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

template cudaError_t launch_gemm<kFc1Grouped, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc2Grouped, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc1Decode, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc2Decode, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc1Grouped, 1>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc2Grouped, 1>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc1Decode, 1>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_gemm<kFc2Decode, 1>(const GemmParams&, int, bool, cudaStream_t);
template size_t gemm_smem_bytes<kFc1Grouped, 0>();
template size_t gemm_smem_bytes<kFc1Decode, 0>();

}  // namespace b4
