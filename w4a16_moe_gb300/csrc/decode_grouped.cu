// Small-m path of the fused W4A16 MoE layer (flashinfer PR #4255, Description:
// "A tensor-core decode path for small batches on the packed serving
// weights"): ONE cooperative persistent kernel for FC1, the activation, FC2
// and the top-k combine, with the routes of each expert grouped so that an
// expert's weights stream once per call however many tokens picked it.
//
// Groups.  Every CTA sorts the m*top_k expert ids itself at launch (a stable
// counting sort in shared memory, no route-pack launch): the valid routes of
// local expert e, in ascending flat route index, are cut into groups of at
// most 8*SETS routes.  A group's routes are the B columns of warp-level
// m16n8k16 MMAs (8 routes per column set, SETS sets), its expert's weights the
// A rows; a dequantised weight fragment feeds every column set.
//
// Work and its partition.  FC1 is the list of (group, 128-row tile) pairs, each
// k_stages1 stages of 64 K; FC2 the list of (group, 128-row tile of H) pairs
// over k_stages2 stages.  A stage of a group costs w0 + (its column sets).  The
// CTAs split each list into contiguous ranges of equal cost (static, no
// claiming), so every CTA streams about the same weight bytes; a CTA's share
// of one tile is a unit (a K range), and the CTAs sharing a tile number their
// units 0, 1, ... ("pieces").  A CTA runs its FC1 units, then its FC2 units.
//
// Hand-offs, with no counters and no fences: before a grid barrier at launch
// the CTAs fill both partial buffers with a signalling-NaN bit pattern that no
// arithmetic produces, and a reader polls the values it needs until none of
// them holds it (a 4-byte store is seen whole or not at all).  A unit stores
// an fp32 partial per (route, row) and piece.  Each tile has a builder fixed
// by the partition: the CTA of its piece 0, whose share of the tile is the end
// of that CTA's range, so the other pieces (the starts of later CTAs' ranges)
// are done first.  The FC1 builder sums the tile's pieces (piece order) into
// bf16 h, activation applied, and then sets the tile's ready flag; an FC2
// unit's activation loads wait for the flags of the FC1 tiles holding its h
// columns.  Each (token, 128 output columns) has a fixed owner CTA, which,
// after its own FC2 units, sums the token's routes (ascending top-k slot) and
// their pieces (piece order) and rounds once to bf16.  Every sum has a fixed
// order, so the output is bitwise reproducible.  A wait only ever depends on
// CTAs of higher index (FC1 builders) or on FC2 units, which depend on FC1
// only; the cooperative launch keeps every CTA resident, so every wait ends,
// and each is bounded as well.
//
// Roles (one CTA per SM, 19 warps, so a thread may hold 96 registers):
//   warp 0        builds the group table; then one thread publishes unit
//                 descriptors and streams each unit's weights: bulk copies of
//                 four 64-wide stages of codes and scales per slot of a
//                 shared-memory ring;
//   warp 1        activation rows: x (FC1) or h (FC2) of the group's routes
//                 per stage, by cp.async;
//   warps 2..17   compute: warp w handles rows 16*(w%8)..+15 of the tile for
//                 stages 2*(w/8) and 2*(w/8)+1 of each four-stage slot;
//                 register dequantisation (E2M1 table lookup by PRMT, one
//                 bf16x2 multiply by the block scale) feeding m16n8k16 MMAs;
//                 the two halves add their fp32 results in shared memory at
//                 unit end;
//                 at a unit's end they store its partials and, where the CTA
//                 builds the tile, its h; after the last unit, the CTA's
//                 share of the output;
//   warp 18       waits for the grid barrier.
//
// The dense W4A16 linear layer (one weight matrix, top-1, no activation) runs
// the FC1 phase alone: the last piece of a tile writes out directly.
//
// Why warp-level MMAs and not tcgen05 here: the register dequantiser feeds
// m16n8k16 fragments directly, while a tcgen05.mma reads its weight operand
// from shared or tensor memory, so every dequantised weight would make a
// round trip there first; with at most 16 routes per group the MMA work is
// small either way and the dequantiser's integer work is the limit (per code
// word of 8 weights: two LOP3, three shifts and four PRMT on the half-rate
// integer pipe, four bf16x2 multiplies on the half-rate FMA pipe).
//
// K order inside an MMA: thread t of a quad owns physical 16-element block t
// of the 64-wide stage (one NVFP4 scale block); MMA j takes its pairs 2j and
// 2j+1 as the fragment's logical K pairs t and t + 4.  Weights and
// activations use the same permutation, so every dot product is unchanged.

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "coop_launch.cuh"
#include "decode_stage.cuh"
#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

cudaError_t ensure_smem_limit(const void* func, size_t bytes);

namespace dg {

namespace cg = cooperative_groups;

constexpr int kWarps = 19;
constexpr int kThreads = 32 * kWarps;
constexpr int kCompute = 16;          // compute warps
constexpr int kCT = 32 * kCompute;    // compute threads
constexpr int kWarpW = 0, kWarpAct = 1, kWarpC0 = 2, kWarpSync = 18;
constexpr int kDesc = 8;              // unit descriptor ring
constexpr int kSlotSt = 4;            // K stages per ring slot: each half of the compute warps takes two
constexpr int kActRow = 144;          // activation row stride (bytes): 128 + 16 keeps LDS.128 conflict-free
constexpr uint32_t kNotWritten = 0x7F800001u;  // signalling NaN: never an arithmetic result
constexpr float kTwo63 = 9.223372036854775808e18f;

template <int SETS>
struct Cfg {
  static constexpr int kRows = 8 * SETS;               // routes per group
  static constexpr int kSlots = SETS == 1 ? 8 : 6;     // ring slots of kSlotSt stages
  static constexpr int kActSlot = kSlotSt * kRows * kActRow;
  static constexpr int kChains = SETS == 1 ? 4 : 2;    // accumulator chains per column set
};

// A unit: one CTA's K range of one tile.  phase 0 ends the sequence.
struct GDesc {
  int phase;    // 1 FC1, 2 FC2, 0 none
  int g;        // group
  int tile;
  int s_lo, s_hi;
  int piece, npieces;
  int pad;
};
static_assert(sizeof(GDesc) == 32, "descriptor size");

struct Phase {
  unsigned long long T;  // total cost
  int G;                 // CTAs taking part
  int NT, KS;
};

// Shared-memory layout: fixed part, then the run-time tables.
template <int FMT, int SETS>
struct Smem {
  using C = Cfg<SETS>;
  static constexpr int kSS = scale_bytes_per_stage(FMT);
  static constexpr size_t codes = 0;
  static constexpr size_t scales = codes + (size_t)C::kSlots * kSlotSt * kCodeBytesPerStage;
  static constexpr size_t act = scales + (size_t)C::kSlots * kSlotSt * kSS;
  static constexpr size_t xchg = round_up((int)(act + (size_t)C::kSlots * C::kActSlot), 16);
  static constexpr size_t bars = xchg + (size_t)8 * SETS * 4 * 32 * 4;
  static constexpr int kNumBars = 3 * C::kSlots + 2 * kDesc + 2;
  static constexpr size_t desc = bars + 8 * kNumBars;
  // misc: abort flag, grid word, [NG, pad...], two phases
  static constexpr size_t misc = desc + sizeof(GDesc) * kDesc;
  static constexpr size_t tables = round_up((int)(misc + 32 + 2 * sizeof(Phase)), 16);
  // tables: routes[R] i16, rgroup[R] i16, gexp[R] i16, gfirst[R] i16, gcnt[R] i16,
  // tvalid[m] i16 (m <= R), Cg[R + 1] u32
  static size_t total(int R) { return tables + (size_t)R * 2 * 6 + (size_t)(R + 1) * 4 + 16; }
};

__device__ __forceinline__ int local_expert(const SmallGroupParams& p, int route) {
  if (!p.topk_ids) return 0;  // dense linear layer: one expert, every route valid
  const int id = __ldg(p.topk_ids + route);
  if (id < 0 || id >= p.num_global_experts) return -1;
  const int l = p.expert_map ? __ldg(p.expert_map + id) : id;
  return (l >= 0 && l < p.num_local_experts) ? l : -1;
}

// a / b with a 32-bit division whenever both fit (the usual sizes): a 64-bit
// division is a long instruction sequence, and these run on the critical
// path of the first unit.
__device__ __forceinline__ unsigned long long udiv(unsigned long long a, unsigned long long b) {
  if (((a | b) >> 32) == 0) return (uint32_t)a / (uint32_t)b;
  return a / b;
}
__device__ __forceinline__ unsigned long long ceil_div_u64(unsigned long long a, unsigned long long b) {
  return udiv(a + b - 1, b);
}

// CTA owning cost position P: max{b : floor(b*T/G) <= P}.
__device__ __forceinline__ int owner(const Phase& ph, unsigned long long P) {
  return (int)udiv((P + 1) * (unsigned long long)ph.G - 1, ph.T);
}

// Number of CTAs (pieces) that tile `tile` of group g is split over.
__device__ __forceinline__ int npieces_of(const Phase& ph, const uint32_t* Cg, int g, int tile) {
  const unsigned long long w = Cg[g + 1] - Cg[g];
  const unsigned long long P0 = (unsigned long long)Cg[g] * ph.NT * ph.KS + (unsigned long long)tile * ph.KS * w;
  return owner(ph, P0 + (unsigned long long)(ph.KS - 1) * w) - owner(ph, P0) + 1;
}

// Split grid barrier on the word a cooperative launch provides for
// grid.sync(), with grid.sync()'s arithmetic: every CTA adds 1 once, except
// CTA 0, which adds 2^31 - (G - 1), so the top bit flips exactly when all G
// CTAs have arrived.  The add releases the CTA's earlier writes (ordered
// before it by a CTA barrier); the polling load acquires every CTA's.
__device__ __forceinline__ uint32_t grid_arrive(uint32_t* word) {
  const uint32_t add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1) : 1u;
  uint32_t old;
  asm volatile("atom.add.release.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(word), "r"(add) : "memory");
  return old;
}
__device__ __forceinline__ bool grid_wait(const uint32_t* word, uint32_t old, const Abort& ab) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    uint32_t cur;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(cur) : "l"(word) : "memory");
    if ((cur ^ old) & 0x80000000u) return true;
    if (ab.raised()) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      ab.raise(50);
      return false;
    }
    __nanosleep(128);  // one word polled by every CTA: keep the traffic on it low
  }
}

__device__ __forceinline__ void st_release(int* addr, int v) {
  asm volatile("st.release.gpu.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* addr) {
  int v;
  asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Walks one CTA's units of one phase, in order.
struct UnitIter {
  Phase ph;
  int phase, NG;
  const uint32_t* Cg;     // cost prefix of the groups (per stage)
  unsigned long long pos, hi;
  int g;

  __device__ void init(const Phase& phs, int phase_, int NG_, const uint32_t* Cg_) {
    ph = phs;
    phase = phase_;
    NG = NG_;
    Cg = Cg_;
    g = NG;
    pos = hi = 0;
    if (ph.T == 0 || (int)blockIdx.x >= ph.G) return;
    const unsigned long long b = blockIdx.x;
    pos = udiv(b * ph.T, (unsigned long long)ph.G);
    hi = udiv((b + 1) * ph.T, (unsigned long long)ph.G);
    // the group holding cost position pos: last g with Cg[g]*NT*KS <= pos
    const unsigned long long ntks = (unsigned long long)ph.NT * ph.KS;
    int lo_g = 0, hi_g = NG - 1;
    while (lo_g < hi_g) {
      const int mid = (lo_g + hi_g + 1) >> 1;
      if ((unsigned long long)Cg[mid] * ntks <= pos) lo_g = mid;
      else hi_g = mid - 1;
    }
    g = lo_g;
  }

  __device__ bool next(GDesc& d) {
    const unsigned long long total = (unsigned long long)ph.NT * ph.KS;
    while (pos < hi && g < NG) {
      const unsigned long long base = (unsigned long long)Cg[g] * total;
      const unsigned long long w = Cg[g + 1] - Cg[g];
      const unsigned long long sidx = pos > base ? ceil_div_u64(pos - base, w) : 0;
      if (sidx >= total) {
        ++g;
        continue;
      }
      unsigned long long eidx = ceil_div_u64(hi - base, w);
      if (eidx > total) eidx = total;
      if (eidx <= sidx) {
        pos = hi;
        break;
      }
      const int t = (int)((uint32_t)sidx / (uint32_t)ph.KS);  // sidx < NT * KS
      const unsigned long long tile_end = (unsigned long long)(t + 1) * ph.KS;
      const unsigned long long uend = eidx < tile_end ? eidx : tile_end;
      const unsigned long long P0 = base + (unsigned long long)t * ph.KS * w;
      const unsigned long long P1 = P0 + (unsigned long long)(ph.KS - 1) * w;
      const int b0 = owner(ph, P0);
      d.phase = phase;
      d.g = g;
      d.tile = t;
      d.s_lo = (int)(sidx - (unsigned long long)t * ph.KS);
      d.s_hi = (int)(uend - (unsigned long long)t * ph.KS);
      d.piece = (int)blockIdx.x - b0;
      d.npieces = owner(ph, P1) - b0 + 1;
      d.pad = 0;
      pos = base + uend * w;
      if (uend == total) ++g;
      return true;
    }
    return false;
  }
};

// Piece cap and cost of a stage decide how many CTAs take part in a phase:
// every CTA's range holds at least one stage of the dearest group (so every
// CTA a tile spans owns a stage of it), and a tile spans at most pmax CTAs.
__device__ inline Phase make_phase(unsigned long long cost_total, int NT, int KS, int maxw, int pmax) {
  Phase ph;
  ph.NT = NT;
  ph.KS = KS;
  ph.T = cost_total * (unsigned long long)NT * KS;
  if (ph.T == 0) {
    ph.G = 0;
    return ph;
  }
  unsigned long long G = gridDim.x;
  const unsigned long long a = udiv(ph.T, (unsigned long long)maxw);
  const unsigned long long c = udiv(ph.T, ceil_div_u64((unsigned long long)KS * maxw, (unsigned long long)(pmax - 1)));
  if (a < G) G = a;
  if (c < G) G = c;
  ph.G = G < 1 ? 1 : (int)G;
  return ph;
}

// Timeline stamp (b4_set_trace): kinds 0 start, 1 group table built, 2 first
// descriptor published, 3 first weight copy issued, 4 first slot computed,
// 5 last FC1 unit stored, 6 first FC2 slot computed, 7 compute done,
// 8 epilogue done, 9 first FC2 unit's FC1 tiles ready, 10 grid barrier seen,
// 11 weight stream done, 12 last FC1 h tile built, 13 last output written,
// 14 buffers filled (CTA barrier passed), 15 route ids read.
__device__ __forceinline__ void stamp(const SmallGroupParams& p, int kind) {
  if (p.trace && blockIdx.x < (unsigned)kTraceLen) p.trace[kind * kTraceLen + blockIdx.x] = (long long)globaltimer();
}

// Loads of values another CTA may still be writing (polled until they no
// longer hold the marker): relaxed loads at GPU scope, volatile and with a
// memory clobber so that every poll iteration really reads memory.
__device__ __forceinline__ float ld_poll(const float* src) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(src) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_poll4(const float* src) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(src)
               : "memory");
  return v;
}

// The S consecutive piece partials of one (route, row), loaded together as
// float4s, and the first np of them summed in piece order.
template <int S>
__device__ __forceinline__ void load_pieces(float (&v)[S], const float* src) {
#pragma unroll
  for (int i = 0; i < S; i += 4) {
    const float4 a = ld_poll4(src + i);
    v[i] = a.x, v[i + 1] = a.y, v[i + 2] = a.z, v[i + 3] = a.w;
  }
}
template <int S>
__device__ __forceinline__ float sum_first(const float (&v)[S], int np) {
  float a = v[0];
#pragma unroll
  for (int i = 1; i < S; ++i)
    if (i < np) a += v[i];
  return a;
}

__device__ __forceinline__ bool is_marker(float v) { return __float_as_uint(v) == kNotWritten; }

// The FC1 builder's work: h (or, for the dense linear layer, out) of the
// tile's rows for the group's c routes, from its pieces' partials summed in
// piece order; an item is read again while any value it needs still holds the
// marker.  Returns false if a wait ran out.
template <int S>
__device__ __forceinline__ bool build_tile(const SmallGroupParams& p, const GDesc& u, int c, int first,
                                           const int16_t* s_routes, int tid, int wnat, const Abort& ab) {
  const int rows = p.act == 0 ? 64 : kTileRows;
  const int row0 = u.tile * rows;
  const int lim = p.act == 2 ? p.n_out : p.inter_pad;
  const int total = c * rows;
  constexpr int B = 1;
  for (int base = tid; base < total; base += B * kCT) {
    float va[B][S], vb[B][S];
    int rr[B], row[B];
    bool live[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int it = base + b * kCT;
      const int i = it / rows;
      row[b] = row0 + (it - i * rows);
      live[b] = it < total && row[b] < lim;
      rr[b] = live[b] ? s_routes[first + i] : 0;
    }
    const unsigned long long t0 = globaltimer();
    while (true) {
      bool ready = true;
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (!live[b]) continue;
        const float* pa = p.p + ((size_t)rr[b] * wnat + row[b]) * S;
        load_pieces<S>(va[b], pa);
        if (p.act == 0) load_pieces<S>(vb[b], pa + (size_t)p.inter_pad * S);
#pragma unroll
        for (int k = 0; k < S; ++k)
          if (k < u.npieces && (is_marker(va[b][k]) || (p.act == 0 && is_marker(vb[b][k])))) ready = false;
      }
      if (ready) break;
      if (ab.raised() || globaltimer() - t0 > kWaitLimitNs) {
        if (!ab.raised()) ab.raise(70);
        return false;
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (!live[b]) continue;
      const float a = sum_first<S>(va[b], u.npieces);
      if (p.act == 2) {
        p.out[(size_t)rr[b] * p.n_out + row[b]] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
      } else {
        const float hv = p.act == 0 ? gated_act(a, sum_first<S>(vb[b], u.npieces), p.glu) : (a > 0.f ? a * a : 0.f);
        p.h[(size_t)rr[b] * p.inter_pad + row[b]] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
      }
    }
  }
  return true;
}

// An output owner's work for one column n of a token: the sum over the
// token's valid routes (ascending top-k slot) of their pieces' FC2 partials
// (piece order), in bf16; four routes' loads go out together and are read
// again while any holds the marker.  Returns false if a wait ran out.
template <int PM>
__device__ __forceinline__ bool token_out(const SmallGroupParams& p, const Phase& ph2, const uint32_t* Cg,
                                          const int16_t* s_rgroup, int token, int tile, int n, int R,
                                          const Abort& ab) {
  const size_t stride = (size_t)R * p.hidden;
  float acc = 0.f;
  for (int j0 = 0; j0 < p.top_k; j0 += 4) {
    int np[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = j0 + jj;
      const int gj = j < p.top_k ? s_rgroup[token * p.top_k + j] : -1;
      np[jj] = gj >= 0 ? npieces_of(ph2, Cg, gj, tile) : 0;
    }
    float v[4][PM];
    const unsigned long long t0 = globaltimer();
    while (true) {
      bool ready = true;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const size_t at = (size_t)(token * p.top_k + j0 + jj) * p.hidden + n;
#pragma unroll
        for (int k = 0; k < PM; ++k) {
          v[jj][k] = k < np[jj] ? ld_poll(p.q + k * stride + at) : 0.f;
          if (k < np[jj] && is_marker(v[jj][k])) ready = false;
        }
      }
      if (ready) break;
      if (ab.raised() || globaltimer() - t0 > kWaitLimitNs) {
        if (!ab.raised()) ab.raise(71);
        return false;
      }
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int k = 0; k < PM; ++k)
        if (k < np[jj]) acc += v[jj][k];
  }
  p.out[(size_t)token * p.hidden + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  return true;
}

// One 64-wide stage of this thread's two weight rows: register dequantisation
// (E2M1 lookup, bf16x2 block-scale multiply) and, per column set, the
// activation rows and four m16n8k16 MMAs into chains ch0 and ch0 + 1.
template <int FMT, int SETS, int CH>
__device__ __forceinline__ void stage_mma(uint2 c0, uint2 c1, uint32_t b0, uint32_t b1, const uint8_t* xs,
                                          const uint32_t (&arow)[SETS], int sets, float (&acc)[SETS][CH][4],
                                          int ch0) {
  const uint32_t sa = d_scale<FMT>(b0), sb = d_scale<FMT>(b1);
  uint32_t a0[8], a1[8];
  fp4x8_lookup(c0.x, a0[0], a0[1], a0[2], a0[3]);
  fp4x8_lookup(c0.y, a0[4], a0[5], a0[6], a0[7]);
  fp4x8_lookup(c1.x, a1[0], a1[1], a1[2], a1[3]);
  fp4x8_lookup(c1.y, a1[4], a1[5], a1[6], a1[7]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a0[i] = bf16x2_mul(a0[i], sa);
    a1[i] = bf16x2_mul(a1[i], sb);
  }
#pragma unroll
  for (int q = 0; q < SETS; ++q) {
    if (q < sets) {
      const uint4 xa = *reinterpret_cast<const uint4*>(xs + arow[q]);
      const uint4 xb = *reinterpret_cast<const uint4*>(xs + arow[q] + 16);
      mma_16816(acc[q][ch0], a0[0], a1[0], a0[1], a1[1], xa.x, xa.y);
      mma_16816(acc[q][ch0 + 1], a0[2], a1[2], a0[3], a1[3], xa.z, xa.w);
      mma_16816(acc[q][ch0], a0[4], a1[4], a0[5], a1[5], xb.x, xb.y);
      mma_16816(acc[q][ch0 + 1], a0[6], a1[6], a0[7], a1[7], xb.z, xb.w);
    }
  }
}
template <int CH>
__device__ __forceinline__ float chain_sum(const float (&a)[CH][4], int i) {
  float v = a[0][i];
#pragma unroll
  for (int h = 1; h < CH; ++h) v += a[h][i];
  return v;
}

// ------------------------------------------------------------------ kernel
template <int FMT, int SETS>
__global__ void __launch_bounds__(kThreads, 1) decode_grouped_kernel(const __grid_constant__ SmallGroupParams p) {
  using C = Cfg<SETS>;
  using L = Smem<FMT, SETS>;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int kSS = L::kSS;
  constexpr int NS = C::kSlots;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_codes = smem + L::codes;
  uint8_t* s_scales = smem + L::scales;
  uint8_t* s_act = smem + L::act;
  float* s_xchg = reinterpret_cast<float*>(smem + L::xchg);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* full_w = bars;                 // weights of a slot landed (tx)
  uint64_t* full_a = full_w + NS;          // activations of a slot landed (32 cp.async arrivals)
  uint64_t* empty_s = full_a + NS;         // compute warps released the slot (16)
  uint64_t* dfull = empty_s + NS;          // descriptor published (1)
  uint64_t* dempty = dfull + kDesc;        // compute warps finished the unit (16)
  uint64_t* setup_bar = dempty + kDesc;    // group table ready (1)
  uint64_t* grid_bar = setup_bar + 1;      // every CTA's buffers filled (1)
  GDesc* s_desc = reinterpret_cast<GDesc*>(smem + L::desc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc);
  volatile int* s_misc = reinterpret_cast<volatile int*>(smem + L::misc + 8);  // [0] NG
  Phase* s_ph = reinterpret_cast<Phase*>(smem + L::misc + 32);
  const int R = p.m * p.top_k;
  int16_t* s_routes = reinterpret_cast<int16_t*>(smem + L::tables);
  int16_t* s_rgroup = s_routes + R;
  int16_t* s_gexp = s_rgroup + R;
  int16_t* s_gfirst = s_gexp + R;
  int16_t* s_gcnt = s_gfirst + R;
  int16_t* s_tvalid = s_gcnt + R;
  uint32_t* s_Cg = reinterpret_cast<uint32_t*>(smem + L::tables + (size_t)R * 2 * 6);
  // setup scratch [3][E_l] int32, aliasing the activation ring (unused until the table is built)
  int* s_ecnt = reinterpret_cast<int*>(s_act);
  int* s_eoff = s_ecnt + p.num_local_experts;
  int* s_goff = s_eoff + p.num_local_experts;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{p.status, s_abort};

  if (threadIdx.x == 0) {
    stamp(p, 0);
    *s_abort = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&full_a[i], 32);
      mbar_init(&empty_s[i], kCompute);
    }
    for (int i = 0; i < kDesc; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], kCompute);
    }
    mbar_init(setup_bar, 1);
    mbar_init(grid_bar, 1);
    fence_mbar_init();
    pdl_launch_dependents();  // the next kernel may launch and set up meanwhile
  }
  pdl_wait();  // launched with PDL: nothing of this call is read or written before the kernel before it is done

  // Before the grid barrier: fill both partial buffers with the not-written
  // marker, clear the FC1 tile flags and the status word, and zero the output
  // rows of tokens without a valid route (no unit writes them).
  {
    const size_t gt = (size_t)blockIdx.x * kThreads + threadIdx.x, gs = (size_t)gridDim.x * kThreads;
    const uint4 mark = make_uint4(kNotWritten, kNotWritten, kNotWritten, kNotWritten);
    for (size_t i = gt; i < p.p_floats / 4; i += gs) reinterpret_cast<uint4*>(p.p)[i] = mark;
    for (size_t i = gt; i < p.q_floats / 4; i += gs) reinterpret_cast<uint4*>(p.q)[i] = mark;
    for (size_t i = gt; i < p.n_flags; i += gs) p.hflag[i] = 0;
    if (gt == 0 && p.status) {
      p.status[0] = 0;
      p.status[1] = 0;
    }
    if (p.topk_ids) {
      const int gw = (int)(gt >> 5), nw = (int)(gs >> 5);
      for (int tk = gw; tk < p.m; tk += nw) {
        bool v = false;
        for (int j = lane; j < p.top_k; j += 32) v |= local_expert(p, tk * p.top_k + j) >= 0;
        if (__ballot_sync(0xffffffffu, v) == 0) {
          uint4* o = reinterpret_cast<uint4*>(p.out + (size_t)tk * p.hidden);
          for (int i = lane; i < p.hidden / 8; i += 32) o[i] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  cg::grid_group grid = cg::this_grid();
  if (!grid.is_valid()) {  // not a cooperative launch: there is no grid barrier to wait on
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0u, 4u);  // B4_ERR_CUDA
    return;
  }
  __syncthreads();

  if (threadIdx.x == 0) stamp(p, 14);
  if (warp == kWarpSync) {
    // ------------------------------------------------------- grid barrier
    // Every thread's fill precedes the CTA's arrival (a release at GPU scope);
    // the first partial store or read of the compute warps waits for grid_bar.
    if (lane == 0) {
      uint32_t* word = &cg::details::get_grid_workspace()->barrier;
      const uint32_t old = grid_arrive(word);
      // polling starts once the group table is built, off its critical path
      if (mbar_wait(setup_bar, 0, ab, 69) && grid_wait(word, old, ab)) mbar_arrive(grid_bar);
      stamp(p, 10);
    }
    __syncwarp();
    return;
  }

  if (warp == kWarpW) {
    // ------------------------------------------------------------ group table
    const int E = p.num_local_experts;
    for (int e = lane; e < E; e += 32) s_ecnt[e] = 0;
    __syncwarp();
    for (int r = lane; r < R; r += 32) {
      const int l = local_expert(p, r);
      s_rgroup[r] = (int16_t)l;
      if (l >= 0) atomicAdd(&s_ecnt[l], 1);
    }
    __syncwarp();
    if (lane == 0) stamp(p, 15);
    // exclusive scans of the counts and of the groups per expert
    int run_e = 0, run_g = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? s_ecnt[e] : 0;
      const int ng = (c + C::kRows - 1) / C::kRows;
      int ic = c, ig = ng;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int yc = __shfl_up_sync(0xffffffffu, ic, d), yg = __shfl_up_sync(0xffffffffu, ig, d);
        if (lane >= d) ic += yc, ig += yg;
      }
      if (e < E) {
        s_eoff[e] = run_e + ic - c;
        s_goff[e] = run_g + ig - ng;
        for (int i = 0; i < ng; ++i) {
          const int gi = run_g + ig - ng + i;
          s_gexp[gi] = (int16_t)e;
          s_gfirst[gi] = (int16_t)(run_e + ic - c + i * C::kRows);
          s_gcnt[gi] = (int16_t)min(C::kRows, c - i * C::kRows);
        }
        s_ecnt[e] = 0;  // now the placement cursor
      }
      run_e += __shfl_sync(0xffffffffu, ic, 31);
      run_g += __shfl_sync(0xffffffffu, ig, 31);
    }
    const int NG = run_g;
    __syncwarp();
    // stable placement: routes of an expert in ascending flat index
    for (int base = 0; base < R; base += 32) {
      const int r = base + lane;
      const int l = r < R ? s_rgroup[r] : -2;
      const unsigned peers = __match_any_sync(0xffffffffu, l);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (l >= 0) {
        const int within = s_ecnt[l] + rank;
        s_routes[s_eoff[l] + within] = (int16_t)r;
        s_rgroup[r] = (int16_t)(s_goff[l] + within / C::kRows);
      } else if (r < R) {
        s_rgroup[r] = -1;
      }
      __syncwarp();
      if (l >= 0 && lane == 31 - __clz(peers)) s_ecnt[l] += __popc(peers);
      __syncwarp();
    }
    // valid routes per token
    for (int t = lane; t < p.m; t += 32) {
      int c = 0;
      for (int j = 0; j < p.top_k; ++j) c += s_rgroup[t * p.top_k + j] >= 0;
      s_tvalid[t] = (int16_t)c;
    }
    // cost prefix: a stage of group g costs w0 + its column sets
    int run = 0, maxw = 0;
    for (int base = 0; base < NG; base += 32) {
      const int gi = base + lane;
      const int w = gi < NG ? p.w0 + (s_gcnt[gi] + 7) / 8 : 0;
      int iw = w;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, iw, d);
        if (lane >= d) iw += y;
      }
      if (gi < NG) s_Cg[gi] = (uint32_t)(run + iw - w);
      run += __shfl_sync(0xffffffffu, iw, 31);
      maxw = max(maxw, w);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) maxw = max(maxw, __shfl_xor_sync(0xffffffffu, maxw, d));
    if (lane == 0) {
      s_Cg[NG] = (uint32_t)run;
      s_misc[0] = NG;
      s_ph[0] = make_phase(NG ? run : 0, p.n_tiles1, p.k_stages1, maxw, p.pmax);
      s_ph[1] = make_phase(NG && p.n_tiles2 ? run : 0, p.n_tiles2 > 0 ? p.n_tiles2 : 1,
                           p.k_stages2 > 0 ? p.k_stages2 : 1, maxw, p.pmax);
      stamp(p, 1);
      mbar_arrive(setup_bar);
    }
    __syncwarp();

    // ---------------------------------- unit descriptors and weight stream
    // One thread walks the CTA's units (FC1, then FC2); it publishes each one
    // (at most kDesc ahead of the epilogue) and streams its weights.
    if (lane == 0) {
      UnitIter it;
      it.init(s_ph[0], 1, NG, s_Cg);
      int phase = 1;
      uint32_t d = 0, ws = 0;
      while (!ab.raised()) {
        GDesc u;
        bool have = it.next(u);
        if (!have && phase == 1) {
          it.init(s_ph[1], 2, NG, s_Cg);
          phase = 2;
          have = it.next(u);
        }
        if (!have) u.phase = 0;
        const uint32_t slot_d = d % kDesc;
        if (!mbar_wait(&dempty[slot_d], ((d / kDesc) & 1) ^ 1, ab, 51)) break;
        s_desc[slot_d] = u;
        mbar_arrive(&dfull[slot_d]);
        if (d == 0) stamp(p, 2);
        ++d;
        if (!have) break;
        const bool fc2 = u.phase == 2;
        const int nt = fc2 ? p.n_tiles2 : p.n_tiles1, ks = fc2 ? p.k_stages2 : p.k_stages1;
        const size_t tile_id = (size_t)s_gexp[u.g] * nt + u.tile;
        const uint8_t* gc = (fc2 ? p.w2_codes : p.w1_codes) + tile_id * ks * kCodeBytesPerStage;
        const uint8_t* gsc = (fc2 ? p.w2_scales : p.w1_scales) + tile_id * ks * kSS;
        bool ok = true;
        for (int s = u.s_lo; s < u.s_hi; s += kSlotSt, ++ws) {
          const uint32_t slot = ws % NS;
          if (!mbar_wait(&empty_s[slot], ((ws / NS) & 1) ^ 1, ab, 54)) {
            ok = false;
            break;
          }
          const int n = min(kSlotSt, u.s_hi - s);
          mbar_arrive_expect_tx(&full_w[slot], n * (kCodeBytesPerStage + kSS));
          bulk_g2s(s_codes + slot * kSlotSt * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage,
                   n * kCodeBytesPerStage, &full_w[slot]);
          bulk_g2s(s_scales + slot * kSlotSt * kSS, gsc + (size_t)s * kSS, n * kSS, &full_w[slot]);
          if (ws == 0) stamp(p, 3);
        }
        if (!ok) break;
      }
      stamp(p, 11);
      if (ab.raised()) {  // let issued copies land before the CTA exits
        const uint32_t n = ws < (uint32_t)NS ? ws : (uint32_t)NS;
        for (uint32_t i = ws - n; i < ws; ++i) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full_w[i % NS], (i / NS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
    return;
  }

  if (warp == kWarpAct) {
    // ------------------------------------------------- activation rows
    // Rows of the group's routes for each stage of a slot: x of the route's
    // token (FC1) or h of the route (FC2), 16 bytes per cp.async; x columns
    // past H are zero-filled.
    bool synced = false, stamped9 = false;
    uint32_t ws = 0;
    if (__all_sync(0xffffffffu, mbar_wait(setup_bar, 0, ab, 55))) {
      for (uint32_t d = 0; !ab.raised(); ++d) {
        const uint32_t slot_d = d % kDesc;
        if (!__all_sync(0xffffffffu, mbar_wait(&dfull[slot_d], (d / kDesc) & 1, ab, 56))) break;
        const GDesc u = s_desc[slot_d];
        if (u.phase == 0) break;
        const bool fc2 = u.phase == 2;
        const int c = s_gcnt[u.g], first = s_gfirst[u.g];
        // the row each of this lane's routes reads: x of its token (FC1) or h of the route (FC2)
        const uint16_t* rsrc[2 * SETS];
#pragma unroll
        for (int q = 0; q < 2 * SETS; ++q) {
          const int i = (lane >> 3) + 4 * q;
          const int r = i < c ? s_routes[first + i] : 0;
          rsrc[q] = fc2 ? p.h + (size_t)r * p.inter_pad : p.x + (size_t)(r / p.top_k) * p.hidden;
        }
        if (fc2) {
          if (!synced) {
            if (!__all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 57))) break;
            synced = true;
          }
          // the FC1 tiles holding this unit's h columns must be ready: one
          // flag per lane, polled together
          const int t_lo = p.act == 0 ? u.s_lo : u.s_lo >> 1;
          const int t_hi = p.act == 0 ? u.s_hi - 1 : (u.s_hi - 1) >> 1;
          bool ready = true;
          for (int t0 = t_lo; t0 <= t_hi; t0 += 32) {
            const int t1 = t0 + lane;
            if (t1 > t_hi) continue;
            const int* flag = p.hflag + (size_t)u.g * p.n_tiles1 + t1;
            const unsigned long long tb = globaltimer();
            while (ld_acquire(flag) == 0) {
              if (ab.raised() || globaltimer() - tb > kWaitLimitNs) {
                if (!ab.raised()) ab.raise(59);
                ready = false;
                break;
              }
            }
          }
          if (!__all_sync(0xffffffffu, ready)) break;
          if (!stamped9 && lane == 0) stamp(p, 9);
          stamped9 = true;
        }
        bool ok = true;
        for (int s = u.s_lo; s < u.s_hi; s += kSlotSt, ++ws) {
          const uint32_t slot = ws % NS;
          if (!__all_sync(0xffffffffu, mbar_wait(&empty_s[slot], ((ws / NS) & 1) ^ 1, ab, 58))) {
            ok = false;
            break;
          }
          const int n = min(kSlotSt, u.s_hi - s);
          uint8_t* dst0 = s_act + slot * C::kActSlot + (lane >> 3) * kActRow + (lane & 7) * 16;
          // lane l copies 16-byte chunk l % 8 of routes l / 8, l / 8 + 4, ...
          for (int st = 0; st < n; ++st) {
            const int k = (s + st) * kBK + (lane & 7) * 8;
            const int valid = (p.hidden - k) * 2;
            const uint32_t bytes = fc2 || valid >= 16 ? 16u : (valid > 0 ? (uint32_t)valid : 0u);
#pragma unroll
            for (int q = 0; q < 2 * SETS; ++q) {
              const int i = (lane >> 3) + 4 * q;
              if (i < c) {
                const uint32_t dst = smem_u32(dst0 + (st * C::kRows + 4 * q) * kActRow);
                cp_async16(dst, bytes ? rsrc[q] + k : p.x, bytes);
              }
            }
          }
          cp_async_arrive(&full_a[slot]);
        }
        if (!ok) break;
      }
    }
    cp_async_wait_all();
    __syncwarp();
    return;
  }

  // ---------------------------------------------------------- compute warps
  const int cw = warp - kWarpC0;
  const int rw = cw & 7, half = cw >> 3;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = 16 * rw + g, r1 = r0 + 8;
  const uint32_t code_off = (t >> 1) * (kCodeBytesPerStage / 2) + r0 * 16 + (t & 1) * 8;
  const uint32_t sc_off = FMT == 0 ? r0 * SB + t : r0 * SB + (t >> 1);
  const int wnat = fc1_natural_width(p.act == 0 ? 0 : 1, p.inter_pad);
  // every exit decision is agreed on by all 16 warps (named_bar_or) before
  // any named barrier, so they always leave the loop together
  const bool oks = __all_sync(0xffffffffu, mbar_wait(setup_bar, 0, ab, 64));
  if (named_bar_or(1, kCT, !oks)) return;
  const int tid = threadIdx.x - 32 * kWarpC0;  // 0 .. kCT - 1
  uint32_t ws = 0;
  bool fc2_seen = false, synced = false, failed = false;
  for (uint32_t d = 0;; ++d) {
    const uint32_t slot_d = d % kDesc;
    const bool okf = __all_sync(0xffffffffu, mbar_wait(&dfull[slot_d], (d / kDesc) & 1, ab, 65));
    if (named_bar_or(1, kCT, !okf)) break;
    const GDesc u = s_desc[slot_d];
    if (u.phase == 0) break;
    const bool fc2 = u.phase == 2;
    const int c = s_gcnt[u.g], first = s_gfirst[u.g];
    const int sets = (c + 7) >> 3;
    constexpr int CH = C::kChains;
    float acc[SETS][CH][4];
#pragma unroll
    for (int q = 0; q < SETS; ++q)
#pragma unroll
      for (int h = 0; h < CH; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[q][h][i] = 0.f;
    // activation row of each column set for this thread (route 8q + g, or the
    // group's last route where the set is not full: its columns are unused)
    uint32_t arow[SETS];
#pragma unroll
    for (int q = 0; q < SETS; ++q) arow[q] = (uint32_t)min(8 * q + g, c - 1) * kActRow + t * 32;
    bool ok = true;
    for (int s = u.s_lo; s < u.s_hi; s += kSlotSt, ++ws) {
      const uint32_t slot = ws % NS;
      const uint32_t par = (ws / NS) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&full_w[slot], par, ab, 66) && mbar_wait(&full_a[slot], par, ab, 67))) {
        ok = false;
        break;
      }
      // this half's two stages of the slot: both stages' codes and scales are
      // loaded before any arithmetic
      const int st0 = 2 * half;
      const int nst = min(2, min(kSlotSt, u.s_hi - s) - st0);
      if (nst > 0) {
        const uint8_t* cs = s_codes + (slot * kSlotSt + st0) * kCodeBytesPerStage + code_off;
        const uint8_t* ss = s_scales + (slot * kSlotSt + st0) * kSS + sc_off;
        const uint8_t* xs = s_act + slot * C::kActSlot + st0 * C::kRows * kActRow;
        const uint2 ca0 = *reinterpret_cast<const uint2*>(cs);
        const uint2 ca1 = *reinterpret_cast<const uint2*>(cs + 8 * 16);
        const uint32_t ba0 = ss[0], ba1 = ss[8 * SB];
        uint2 cb0 = make_uint2(0, 0), cb1 = make_uint2(0, 0);
        uint32_t bb0 = 0, bb1 = 0;
        if (nst > 1) {
          cb0 = *reinterpret_cast<const uint2*>(cs + kCodeBytesPerStage);
          cb1 = *reinterpret_cast<const uint2*>(cs + kCodeBytesPerStage + 8 * 16);
          bb0 = ss[kSS];
          bb1 = ss[kSS + 8 * SB];
        }
        stage_mma<FMT, SETS, CH>(ca0, ca1, ba0, ba1, xs, arow, sets, acc, 0);
        if (nst > 1)
          stage_mma<FMT, SETS, CH>(cb0, cb1, bb0, bb1, xs + C::kRows * kActRow, arow, sets, acc, CH == 4 ? 2 : 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_s[slot]);
      if (cw == 0 && lane == 0 && (ws == 0 || (fc2 && !fc2_seen))) {
        stamp(p, ws == 0 ? 4 : 6);
        if (fc2) fc2_seen = true;
      }
    }
    if (named_bar_or(1, kCT, !ok)) {
      failed = true;
      break;
    }
    if (!synced) {  // the first partial store waits for every CTA's marker fill
      const bool okg = __all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 68));
      if (named_bar_or(1, kCT, !okg)) {
        failed = true;
        break;
      }
      synced = true;
    }
    // the two halves' sums meet in shared memory; half 0 stores the partials
    float* xw = s_xchg + (size_t)rw * SETS * 4 * 32 + lane;
    if (half == 1) {
#pragma unroll
      for (int q = 0; q < SETS; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (q < sets) xw[(q * 4 + i) * 32] = chain_sum<CH>(acc[q], i);
    }
    named_bar_sync(1, kCT);
    if (half == 0) {
      const int e = s_gexp[u.g];
      const float gsv = ((fc2 ? p.gs2 : p.gs1) ? __ldg((fc2 ? p.gs2 : p.gs1) + e) : 1.0f) * kTwo63;
#pragma unroll
      for (int q = 0; q < SETS; ++q) {
        if (q >= sets) continue;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = chain_sum<CH>(acc[q], i) + xw[(q * 4 + i) * 32];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int i = 8 * q + 2 * t + j;
          if (i >= c) continue;
          const int r = s_routes[first + i];
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int row = hr ? r1 : r0;
            const float val = v[2 * hr + j];
            if (!fc2) {
              int nat;
              if (p.act == 0) {
                const int i2 = u.tile * 64 + (row >> 5) * 16 + (row & 15);
                nat = (row & 31) >= 16 ? p.inter_pad + i2 : i2;
              } else {
                nat = u.tile * kTileRows + row;
                if (nat >= p.inter_pad) continue;
              }
              p.p[((size_t)r * wnat + nat) * p.p_stride + u.piece] = val * gsv;
            } else {
              const int n = u.tile * kTileRows + row;
              if (n < p.hidden)
                p.q[((size_t)u.piece * R + r) * p.hidden + n] = val * gsv * __ldg(p.topk_weights + r);
            }
          }
        }
      }
    }
    named_bar_sync(1, kCT);  // the exchange buffer is free again
    if (!fc2 && u.piece == 0) {
      // this CTA builds the FC1 tile: h (or out) from all its pieces
      const bool okb = p.p_stride == 8 ? build_tile<8>(p, u, c, first, s_routes, tid, wnat, ab)
                                       : build_tile<4>(p, u, c, first, s_routes, tid, wnat, ab);
      if (named_bar_or(1, kCT, !okb)) {
        failed = true;
        break;
      }
      if (tid == 0 && p.act != 2) st_release(p.hflag + (size_t)u.g * p.n_tiles1 + u.tile, 1);
      if (tid == 0) stamp(p, 12);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&dempty[slot_d]);
    if (cw == 0 && lane == 0 && !fc2) stamp(p, 5);
  }
  if (cw == 0 && lane == 0) stamp(p, 7);
  // This CTA's share of the output: (token, 128 columns) pairs o = b, b + G2,
  // ... of the FC2 partition's G2 CTAs, four at a time (one column per
  // thread).
  const Phase ph2 = s_ph[1];
  if (!failed && p.n_tiles2 > 0 && ph2.G > 0 && (int)blockIdx.x < ph2.G) {
    const int total = p.m * p.n_tiles2;
    for (int o0 = blockIdx.x; o0 < total; o0 += 4 * ph2.G) {
      const int o = o0 + (tid >> 7) * ph2.G;
      bool okt = true;
      if (o < total) {
        const int token = o / p.n_tiles2, tile = o - token * p.n_tiles2;
        const int n = tile * kTileRows + (tid & (kTileRows - 1));
        if (s_tvalid[token] > 0 && n < p.hidden)
          okt = p.q_pieces == 8 ? token_out<8>(p, ph2, s_Cg, s_rgroup, token, tile, n, R, ab)
                                : token_out<4>(p, ph2, s_Cg, s_rgroup, token, tile, n, R, ab);
      }
      if (named_bar_or(1, kCT, !okt)) break;
    }
    if (tid == 0) stamp(p, 13);
  }
}

}  // namespace dg

size_t decode_grouped_smem(int fmt, int sets, int routes) {
  if (fmt == 0) return sets == 1 ? dg::Smem<0, 1>::total(routes) : dg::Smem<0, 2>::total(routes);
  return sets == 1 ? dg::Smem<1, 1>::total(routes) : dg::Smem<1, 2>::total(routes);
}

template <int FMT, int SETS>
static cudaError_t launch_dg(const SmallGroupParams& p, int grid, cudaStream_t stream) {
  auto kern = dg::decode_grouped_kernel<FMT, SETS>;
  const size_t smem = dg::Smem<FMT, SETS>::total(p.m * p.top_k);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_cooperative(kern, grid, dg::kThreads, smem, stream, p);
}

// Resident CTAs per SM of the kernel with `smem` bytes (the cooperative launch
// takes one CTA per SM, which must fit).
cudaError_t decode_grouped_occupancy(int fmt, int sets, size_t smem, int* blocks_per_sm) {
  const void* k = fmt == 0 ? (sets == 1 ? reinterpret_cast<const void*>(dg::decode_grouped_kernel<0, 1>)
                                        : reinterpret_cast<const void*>(dg::decode_grouped_kernel<0, 2>))
                           : (sets == 1 ? reinterpret_cast<const void*>(dg::decode_grouped_kernel<1, 1>)
                                        : reinterpret_cast<const void*>(dg::decode_grouped_kernel<1, 2>));
  cudaError_t e = ensure_smem_limit(k, smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, dg::kThreads, smem);
}

cudaError_t launch_decode_grouped(const SmallGroupParams& p, int fmt, int sets, int grid, cudaStream_t stream) {
  if (fmt == 0) return sets == 1 ? launch_dg<0, 1>(p, grid, stream) : launch_dg<0, 2>(p, grid, stream);
  return sets == 1 ? launch_dg<1, 1>(p, grid, stream) : launch_dg<1, 2>(p, grid, stream);
}

}  // namespace b4
