// Small-m decode path of the fused W4A16 MoE layer (flashinfer PR #4255,
// Description: "A tensor-core decode path for small batches on the packed
// serving weights").
//
// With one route per unit, each GEMM is a matrix-vector product over the
// expert's weights: HBM-bound, 4 bits per weight.  The work unit is (route,
// 128-row tile, K split).  Warp 0 streams the tile's packed codes and scales
// stage by stage (64 K elements, one 4 KB + 512 B bulk copy each) through a
// 16-deep shared-memory ring; for FC1 it also loads the unit's slice of the
// x row with one more bulk copy, while FC2's compute warps build their h
// slice themselves (sum of the FC1 split-K partials, activation, bf16) at the
// start of the unit.  Warps 1..8 each own 16
// weight rows: they dequantise with the same register PRMT dequantiser as the
// grouped path and feed warp-level m16n8k16 bf16 MMAs with fp32 accumulators,
// whose eight columns hold the activation in column 0 and zeros elsewhere.
// The 5th-generation tensor core (tcgen05) is not used here: one tcgen05.mma
// covers 128 x 16 weights and costs ~165 cycles to issue whatever its N, which
// caps a GEMV near 2 TB/s; m16n8k16 costs a few cycles, so the dequantiser's
// ALU work is what remains.
//
// K order inside an MMA: thread t of a quad feeds fragment pairs
// (k = 2t, 2t+1) and (2t+8, 2t+9) of each 16-wide K block.  For weights and
// activations alike, block b's pair (2t, 2t+1) is physical pair 2b and pair
// (2t+8, 2t+9) physical pair 2b+1 of the thread's two code words (word t of
// chunk 0, elements 8t..8t+7; word t of chunk 1, elements 32+8t..39+8t).
// Being the same permutation on both operands, it leaves every dot product
// unchanged and lets each thread read one 32-bit word per row and chunk.

#include <cuda_bf16.h>

#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

constexpr int kDecThreads = 288;     // warp 0 producer + 8 compute warps
constexpr int kDecNW = 16;           // weight stages in flight
constexpr int kDecMaxStages = 128;   // K stages of one unit (its activation slice lives in shared memory)
constexpr int kDecRowBytes = kDecMaxStages * kBK * 2;
constexpr float kDecTwo63 = 9.223372036854775808e18f;
constexpr int kMaxDecSplits = 8;       // FC1 partials summed by the FC2 kernel

template <int FMT>
struct DecSmem {
  static constexpr int kScaleStage = scale_bytes_per_stage(FMT);
  static constexpr size_t codes = 0;
  static constexpr size_t scales = (size_t)kDecNW * kCodeBytesPerStage;
  static constexpr size_t rows = round_up((int)(scales + (size_t)kDecNW * kScaleStage), 128);
  static constexpr size_t bars = rows + 2 * (size_t)kDecRowBytes;
  static constexpr size_t misc = bars + 8 * (2 * kDecNW + 4);
  static constexpr size_t total = misc + 16;
};

__device__ __forceinline__ int dec_local_expert(const GemmParams& p, int route) {
  const int id = __ldg(p.topk_ids + route);
  if (id < 0 || id >= p.num_global_experts) return -1;
  const int l = p.expert_map ? __ldg(p.expert_map + id) : id;
  return (l >= 0 && l < p.num_local_experts) ? l : -1;
}

struct DecUnit {
  int route, tile, split, kbeg, kend, expert;
};

__device__ __forceinline__ bool dec_unit(const GemmParams& p, int u, DecUnit& U) {
  const int per_route = p.n_tiles * p.splits;
  U.route = u / per_route;
  const int rem = u - U.route * per_route;
  U.tile = rem / p.splits;
  U.split = rem - U.tile * p.splits;
  U.kbeg = (int)((long long)U.split * p.k_stages / p.splits);
  U.kend = (int)((long long)(U.split + 1) * p.k_stages / p.splits);
  U.expert = dec_local_expert(p, U.route);
  return U.expert >= 0 && U.kend > U.kbeg;
}

__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Block-scale multiplier (bf16x2 broadcast) of the serving scale byte.
template <int FMT>
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t byte) {
  const uint32_t bits = FMT == 0 ? (byte << 4) + 0x5800u : (byte + 63u) << 7;
  return bits * 0x10001u;
}

// Four packed bf16 pairs of one code word (pairs 0..3 at shifts 0, 2, 16, 18).
__device__ __forceinline__ void dequant_word(uint32_t v, uint32_t s, uint32_t (&o)[4]) {
  o[0] = bf16x2_mul(fp4x2_lookup(v), s);
  o[1] = bf16x2_mul(fp4x2_lookup(v >> 2), s);
  o[2] = bf16x2_mul(fp4x2_lookup(v >> 16), s);
  o[3] = bf16x2_mul(fp4x2_lookup(v >> 18), s);
}

// Timeline hook: CTA 0 records clock64() of event `kind` number `idx`
// (0 weight stage issued, 1 stage consumed by compute warp 1, 2 kernel start,
// 3 activation slice ready, 4 unit done).
__device__ __forceinline__ void dec_trace(const GemmParams& p, int kind, uint32_t idx) {
  if (p.trace && blockIdx.x == 0 && idx < (uint32_t)kTraceLen) p.trace[kind * kTraceLen + idx] = clock64();
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(kDecThreads, 2) decode_gemv_kernel(const __grid_constant__ GemmParams p) {
  using L = DecSmem<FMT>;
  constexpr int NW = kDecNW;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int kScaleStage = L::kScaleStage;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_codes = smem + L::codes;
  uint8_t* s_scales = smem + L::scales;
  uint8_t* s_rows = smem + L::rows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + NW;
  uint64_t* full_b = empty_w + NW;
  uint64_t* empty_b = full_b + 2;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{p.status, s_abort};
  if (threadIdx.x == 0) dec_trace(p, 2, 0);
  const int n_units = p.m * p.top_k * p.n_tiles * p.splits;
  // every thread resolves its first unit now: the routing loads overlap the setup
  DecUnit U0;
  const bool u0_ok = (int)blockIdx.x < n_units && dec_unit(p, blockIdx.x, U0);
  if (threadIdx.x == 0) {
    if (p.clear_status && blockIdx.x == 0 && p.status) {
      p.status[0] = 0;
      p.status[1] = 0;
    }
    *s_abort = 0;
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&empty_w[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_b[i], 1);
      mbar_init(&empty_b[i], 8);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const size_t wtile_codes = (size_t)p.k_stages * kCodeBytesPerStage;
  const size_t wtile_scales = (size_t)p.k_stages * kScaleStage;

  if (warp == 0) {
    // -------------------------------------------------------- producers
    // lane 0 streams weight stages, lane 1 the activation slices; the weight
    // stream does not depend on the previous kernel, so it starts at once
    if (lane == 0) {
      uint32_t ws = 0;
      for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
        DecUnit U = U0;
        if (u == (int)blockIdx.x ? !u0_ok : !dec_unit(p, u, U)) continue;
        const size_t tile_id = (size_t)U.expert * p.n_tiles + U.tile;
        const uint8_t* gc = p.wcodes + tile_id * wtile_codes;
        const uint8_t* gsc = p.wscales + tile_id * wtile_scales;
        for (int s = U.kbeg; s < U.kend; ++s, ++ws) {
          const uint32_t slot = ws % NW;
          if (!mbar_wait(&empty_w[slot], ((ws / NW) & 1) ^ 1, ab, 22)) break;
          mbar_arrive_expect_tx(&full_w[slot], kCodeBytesPerStage + kScaleStage);
          bulk_g2s(s_codes + slot * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage, kCodeBytesPerStage,
                   &full_w[slot]);
          bulk_g2s(s_scales + slot * kScaleStage, gsc + (size_t)s * kScaleStage, kScaleStage, &full_w[slot]);
          dec_trace(p, 0, ws);
        }
      }
      if (ab.raised()) {  // let issued copies land before the CTA exits
        const uint32_t n = ws < (uint32_t)NW ? ws : (uint32_t)NW;
        for (uint32_t i = ws - n; i < ws; ++i) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full_w[i % NW], (i / NW) & 1) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    } else if (lane == 1 && MODE == kFc1Decode) {
      // FC1: the unit's slice of x[token] by one bulk copy (FC2 builds its
      // h slice in the compute warps)
      uint32_t bs = 0;
      for (int u = blockIdx.x; u < n_units && !ab.raised(); u += gridDim.x) {
        DecUnit U = U0;
        if (u == (int)blockIdx.x ? !u0_ok : !dec_unit(p, u, U)) continue;
        const uint32_t rb = bs & 1;
        if (!mbar_wait(&empty_b[rb], ((bs >> 1) & 1) ^ 1, ab, 21)) break;
        uint8_t* row = s_rows + rb * kDecRowBytes;
        const int k0 = U.kbeg * kBK, nk = (U.kend - U.kbeg) * kBK;
        const int kv = min(nk, p.hidden - k0);
        for (int i = kv * 2; i < nk * 2; i += 16) *reinterpret_cast<uint4*>(row + i) = make_uint4(0, 0, 0, 0);
        const uint16_t* src = p.x + (size_t)(U.route / p.top_k) * p.hidden;
        mbar_arrive_expect_tx(&full_b[rb], (uint32_t)kv * 2);
        bulk_g2s(row, src + k0, (uint32_t)kv * 2, &full_b[rb]);
        ++bs;
      }
      if (ab.raised()) {
        for (uint32_t i = bs > 2 ? bs - 2 : 0; i < bs; ++i) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full_b[i & 1], (i >> 1) & 1) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- compute warps
    const int cw = warp - 1;          // 16 weight rows each
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * cw + g, r1 = r0 + 8;
    uint32_t ws = 0, bs = 0;
    if (MODE == kFc2Decode) pdl_wait();  // the FC1 partials come from the previous grid
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      DecUnit U = U0;
      if (u == (int)blockIdx.x ? !u0_ok : !dec_unit(p, u, U)) continue;
      const uint32_t rb = bs & 1;
      uint8_t* row = s_rows + rb * kDecRowBytes;
      if constexpr (MODE == kFc1Decode) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full_b[rb], (bs >> 1) & 1, ab, 23))) break;
      } else {
        // h[k] = act(sum over splits of the FC1 partials, which carry gs13 * 2^63)
        // for the unit's K slice, written into the row buffer by all 256 threads;
        // every partial load of a pass is issued before the first add
        named_bar_sync(1, 256);  // the previous unit's slice is no longer read
        const int R = p.m * p.top_k;
        const int wnat = fc1_natural_width(p.act, p.inter_pad);
        const size_t sstride = (size_t)R * wnat;
        const int k0 = U.kbeg * kBK, nk = (U.kend - U.kbeg) * kBK;
        const float* pr = p.p_in + (size_t)U.route * wnat + k0;
        const int tid = threadIdx.x - 32;
        for (int i0 = 0; i0 < nk; i0 += 512) {
          float gv[2][kMaxDecSplits], uv[2][kMaxDecSplits];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = i0 + e * 256 + tid;
#pragma unroll
            for (int sp = 0; sp < kMaxDecSplits; ++sp) {
              const bool live = i < nk && sp < p.splits_in;
              gv[e][sp] = live ? pr[sp * sstride + i] : 0.f;
              uv[e][sp] = (live && p.act == 0) ? pr[sp * sstride + p.inter_pad + i] : 0.f;
            }
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = i0 + e * 256 + tid;
            float g = 0.f, up = 0.f;
#pragma unroll
            for (int sp = 0; sp < kMaxDecSplits; ++sp) {
              g += gv[e][sp];
              up += uv[e][sp];
            }
            const float hv = p.act == 0 ? g / (1.0f + __expf(-g)) * up : (g > 0.f ? g * g : 0.f);
            if (i < nk) reinterpret_cast<__nv_bfloat16*>(row)[i] = __float2bfloat16_rn(hv);
          }
        }
        named_bar_sync(1, 256);  // the slice is complete
      }
      if (warp == 1 && lane == 0) dec_trace(p, 3, bs);
      float d[4] = {0.f, 0.f, 0.f, 0.f}, e4[4] = {0.f, 0.f, 0.f, 0.f};
      bool ok = true;
      for (int s = U.kbeg; s < U.kend; ++s, ++ws) {
        const uint32_t slot = ws % NW;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_w[slot], (ws / NW) & 1, ab, 24))) {
          ok = false;
          break;
        }
        const uint8_t* cs = s_codes + slot * kCodeBytesPerStage;
        const uint32_t w00 = *reinterpret_cast<const uint32_t*>(cs + r0 * 16 + t * 4);
        const uint32_t w01 = *reinterpret_cast<const uint32_t*>(cs + 2048 + r0 * 16 + t * 4);
        const uint32_t w10 = *reinterpret_cast<const uint32_t*>(cs + r1 * 16 + t * 4);
        const uint32_t w11 = *reinterpret_cast<const uint32_t*>(cs + 2048 + r1 * 16 + t * 4);
        const uint8_t* ss = s_scales + slot * kScaleStage;
        uint32_t sc0, sc1;
        if constexpr (SB == 4) {
          sc0 = *reinterpret_cast<const uint32_t*>(ss + r0 * 4);
          sc1 = *reinterpret_cast<const uint32_t*>(ss + r1 * 4);
        } else {
          sc0 = *reinterpret_cast<const uint16_t*>(ss + r0 * 2);
          sc1 = *reinterpret_cast<const uint16_t*>(ss + r1 * 2);
        }
        // activation pairs of the thread's physical elements (column 0 only)
        uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
        if (g == 0) {
          const uint8_t* xs = row + (s - U.kbeg) * (kBK * 2);
          x0 = *reinterpret_cast<const uint4*>(xs + t * 16);
          x1 = *reinterpret_cast<const uint4*>(xs + 64 + t * 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_w[slot]);
        // scale blocks: NVFP4 chunk 0 word t -> block t/2, chunk 1 -> 2 + t/2; MXFP4 -> 0, 1
        const int blo = FMT == 0 ? (t >> 1) : 0, bhi = FMT == 0 ? 2 + (t >> 1) : 1;
        const uint32_t s0lo = scale_bf16x2<FMT>((sc0 >> (8 * blo)) & 0xFF);
        const uint32_t s0hi = scale_bf16x2<FMT>((sc0 >> (8 * bhi)) & 0xFF);
        const uint32_t s1lo = scale_bf16x2<FMT>((sc1 >> (8 * blo)) & 0xFF);
        const uint32_t s1hi = scale_bf16x2<FMT>((sc1 >> (8 * bhi)) & 0xFF);
        uint32_t a0[8], a1[8];  // physical pairs 0..7 of rows r0 and r1
        {
          uint32_t q[4];
          dequant_word(w00, s0lo, q);
          a0[0] = q[0]; a0[1] = q[1]; a0[2] = q[2]; a0[3] = q[3];
          dequant_word(w01, s0hi, q);
          a0[4] = q[0]; a0[5] = q[1]; a0[6] = q[2]; a0[7] = q[3];
          dequant_word(w10, s1lo, q);
          a1[0] = q[0]; a1[1] = q[1]; a1[2] = q[2]; a1[3] = q[3];
          dequant_word(w11, s1hi, q);
          a1[4] = q[0]; a1[5] = q[1]; a1[6] = q[2]; a1[7] = q[3];
        }
        const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        // two accumulators halve the dependent MMA chain
        mma_m16n8k16_bf16(d, a0[0], a1[0], a0[1], a1[1], xb[0], xb[1]);
        mma_m16n8k16_bf16(e4, a0[2], a1[2], a0[3], a1[3], xb[2], xb[3]);
        mma_m16n8k16_bf16(d, a0[4], a1[4], a0[5], a1[5], xb[4], xb[5]);
        mma_m16n8k16_bf16(e4, a0[6], a1[6], a0[7], a1[7], xb[6], xb[7]);
        if (warp == 1 && lane == 0) dec_trace(p, 1, ws);
      }
      __syncwarp();
      if (MODE == kFc1Decode && lane == 0) mbar_arrive(&empty_b[rb]);
      if (warp == 1 && lane == 0) dec_trace(p, 4, bs);
      ++bs;
      if (!ok) break;
#pragma unroll
      for (int j = 0; j < 4; ++j) d[j] += e4[j];
      // column 0 of D: d[0] is row r0, d[2] row r1 (threads with t == 0)
      if (t == 0) {
        const float gsv = (p.gs ? __ldg(p.gs + U.expert) : 1.0f) * kDecTwo63;
        const int R = p.m * p.top_k;
        if constexpr (MODE == kFc1Decode) {
          const int wnat = fc1_natural_width(p.act, p.inter_pad);
          float* out = p.part_out + ((size_t)U.split * R + U.route) * wnat;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = h ? r1 : r0;
            int nat;
            if (p.act == 0) {
              const int i = U.tile * 64 + (r >> 5) * 16 + (r & 15);
              nat = (r & 31) >= 16 ? p.inter_pad + i : i;
            } else {
              nat = U.tile * kTileRows + r;
              if (nat >= p.inter_pad) nat = -1;
            }
            if (nat >= 0) out[nat] = d[2 * h] * gsv;
          }
        } else {
          const float wt = __ldg(p.topk_weights + U.route);
          float* out = p.part_out + ((size_t)U.split * R + U.route) * p.hidden;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int n = U.tile * kTileRows + (h ? r1 : r0);
            if (n < p.hidden) out[n] = d[2 * h] * gsv * wt;
          }
        }
      }
    }
  }
}

template <int MODE, int FMT>
cudaError_t launch_decode_gemv(const GemmParams& p, int grid, bool pdl, cudaStream_t stream) {
  auto kern = decode_gemv_kernel<MODE, FMT>;
  const size_t smem = DecSmem<FMT>::total;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template cudaError_t launch_decode_gemv<kFc1Decode, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_decode_gemv<kFc2Decode, 0>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_decode_gemv<kFc1Decode, 1>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_decode_gemv<kFc2Decode, 1>(const GemmParams&, int, bool, cudaStream_t);

}  // namespace b4
