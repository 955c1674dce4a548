// Small-m decode path of the fused W4A16 MoE layer (flashinfer PR #4255,
// Description: "A tensor-core decode path for small batches on the packed
// serving weights"): ONE cooperative persistent kernel for FC1, the
// activation, FC2 and the top-k combine.  Two CTAs per SM, 11 warps each.
//
// With one route per work unit both GEMMs are matrix-vector products over the
// expert's weights: HBM-bound at 4 bits per weight.  The kernel is built so
// the weight stream runs from launch to exit and nothing on the path between
// FC1 and FC2 waits for a memory fence.
//
// Work units, in this order: FC1 units (route, 128-row tile, K split), then FC2
// units (route, 128-row tile of H, K split).  CTA b's first two units are b and
// b + G (G CTAs); later ones are claimed from a counter in unit order.  In the
// grouped instantiation (routes that repeat experts) a unit's "route" is a
// group of up to four routes of one expert, which share its weight stream.
//
//   warp 0        streams the unit's packed codes and scales, four 64-wide K
//                 stages per slot of a shared-memory ring (two copies of
//                 16 KB + 2 KB: the bulk-copy engine streams large copies
//                 faster); weights depend on nothing, so the next unit's
//                 stream (FC2 included) starts while this one computes.  It
//                 also issues the CTA's first x slice, ahead of its weights.
//   warp 1        resolves each unit once (expert, scale factors, the token's
//                 valid top-k slots, a group's routes), copies an FC1 unit's
//                 bf16 x slices into a row buffer (one bulk copy per route)
//                 and converts them there to the f16 slots the compute warps
//                 read.
//   warps 2..9    compute warps, 16 weight rows each of the unit's 128:
//                 hardware E2M1 -> f16 conversion feeding warp-level m16n8k16
//                 f16 MMAs whose activation operand is block diagonal, block
//                 scales applied to the fp32 block sums (decode_stage.cuh);
//                 each unit ends with an fp32 split partial store per route.
//                 An FC2 unit first builds its h slices, bf16(act(sum of the
//                 FC1 partials)), as f16 slots.
//   warp 10       makes the CTA's grid-barrier arrival and wait (below), then
//                 stores the bf16 output of a token's 128-column tile: it sums
//                 the FC2 partials of the token's valid routes (ascending
//                 top-k slot, then split) after the tile's last unit in unit
//                 order.  Fixed orders: the output is bitwise reproducible.
//
// Hand-offs between CTAs without counters or fences: before one grid barrier
// at launch, the CTAs fill both partial buffers with a signalling-NaN bit
// pattern that no arithmetic produces; a reader polls the values it needs
// until none of them holds the marker (a 4-byte store is seen whole or not at
// all).  The barrier is split: a CTA arrives as soon as its share of the fill
// is done, and only its first partial store or read waits for the other
// CTAs, so the first two units' weight streams and the first unit's
// arithmetic run meanwhile.  A reader only ever waits for units earlier in
// unit order, each CTA runs its units in increasing order, and a cooperative
// launch keeps every CTA resident, so every wait ends; every wait is bounded
// as well.  Before the barrier the
// CTAs also clear the status word and zero the output rows of tokens without
// a valid route.
//
// The dense W4A16 linear layer (one weight matrix, top-1, no activation, no
// FC2) runs in the same kernel: its FC1 units are the layer's K-split GEMV
// units, and each "FC2" unit is an output tile (token, 128 columns) that sums
// the FC1 split partials straight into out; those units stream no weights.
//
// Why warp-level MMAs and not tcgen05 here: with one token per unit the MMA
// work is tiny and the limit is turning 4-bit codes into MMA operands.  The
// register path reaches its fragments straight from the converted codes; a
// tcgen05.mma would need every weight written to shared or tensor memory
// first.  Measured on GB300 with the data in shared memory: the PRMT table
// lookup + bf16x2 scale multiply of the grouped kernels ran near 4.7 TB/s of
// weights at two CTAs per SM; the conversion instruction with f16 MMAs and
// block-diagonal activations near 11 TB/s.  The prepared layout stores plain
// E2M1 nibbles in the conversion's pairing, so the kernel converts code words
// as loaded (a bit-pair exchange per word, which the table lookup needs
// instead, cost this kernel 10-15 % of its time when it paid it).
//
// K order inside an MMA: thread t of a quad owns physical 16-element block t
// of each 64-wide stage; its bytes pair elements (0,2), (1,3), (4,6), (5,7)
// of every code word (decode_stage.cuh), and the activation slots are stored
// in the same pairing, so every dot product is unchanged.  MMA column c of a
// 128-wide chunk is the chunk's block c: only the thread that owns that block
// in that stage loads nonzero activations for it, so column c accumulates the
// block's unscaled sum.  Activations are prescaled per 128-wide slot by a
// power of two (exact) so that they fit f16; the scale and the prescale are
// applied to the fp32 block sum.
//
// Control flow of the compute warps: they share named barriers, so a failed
// bounded wait never makes one warp leave alone; the loop ends on an OR taken
// over all of them (bar.red.or), and every wait stays bounded.

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <mutex>

#include "coop_launch.cuh"
#include "decode_stage.cuh"
#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

cudaError_t ensure_smem_limit(const void* func, size_t bytes);

namespace cg = cooperative_groups;

constexpr int kDComputeWarps = 8;    // 16 weight rows each: a unit's 128-row tile
constexpr int kDThreads = 32 * (3 + kDComputeWarps);  // weights, schedule, compute, output
constexpr int kDMinBlocks = 2;       // resident CTAs per SM
constexpr int kDSlots = 4;           // weight ring slots
constexpr int kDSlotStages = 4;      // 64-wide K stages per slot (two copies of 16 KB + 2 KB: large copies stream faster)
constexpr int kDMaxStages = kDecodeMaxStages;  // K stages of one route's activation row (a row buffer)
constexpr int kDMaxSlots = kDMaxStages / 2;  // 128-wide slots of one route's activation row
constexpr int kDRowBytes = kDMaxStages * kBK * 2;
// Grouped units: up to four routes of one local expert share a unit (and its
// weight stream); each route's activation row takes a quarter of a row
// buffer, so a grouped unit spans at most 32 K stages.
constexpr int kDGroupMax = kDecodeGroupMax;
constexpr int kDGroupRowBytes = kDRowBytes / kDGroupMax;
constexpr int kDGroupSlots = kDMaxSlots / kDGroupMax;
constexpr int kDGroupMaxRoutes = kDecodeGroupRoutes;  // grouping takes m * top_k <= this: its tables are in shared memory
constexpr uint32_t kNotWritten = 0x7F800001u;  // signalling NaN: never an arithmetic result
static_assert(kDGroupMaxRoutes <= kDThreads, "the group table is built with one thread per route");

// A unit as passed between the warps of a CTA through shared memory.
struct DDesc {
  int u;          // unit index, or -1: no more units
  int expert;     // local expert
  float scale;    // FC1: gs; FC2 of a one-route unit: gs * router weight
  uint32_t mask;  // FC2 of a one-route unit: the token's valid top-k slots
  int nr;         // routes in the unit: 1, or 1 .. 4 for a grouped unit
  uint32_t outs;  // grouped FC2 unit: bit i set when route i's token tile is summed after this unit
  short route[kDGroupMax];  // grouped unit: its routes (-1 past nr)
  float rw[kDGroupMax];     // grouped FC2 unit: gs * router weight of each route
};
static_assert(sizeof(DDesc) == 48, "unit descriptors are 48 bytes");

// A token's 128-column output tile for the output warp.
struct EDesc {
  int tile, token;
  uint32_t mask;  // the token's valid top-k slots
  int end;        // nonzero: no more tiles
};
static_assert(sizeof(EDesc) == 16, "output descriptors are 16 bytes");

template <int FMT>
struct DSmem {
  static constexpr int kScaleStage = scale_bytes_per_stage(FMT);
  static constexpr size_t codes = 0;
  static constexpr size_t scales = (size_t)kDSlots * kDSlotStages * kCodeBytesPerStage;
  static constexpr size_t rows = scales + (size_t)kDSlots * kDSlotStages * kScaleStage;
  static constexpr size_t bars = rows + 2 * (size_t)kDRowBytes;
  static constexpr size_t misc = bars + 8 * (2 * kDSlots + 14);  // 13 barriers besides the ring, one spare
  static constexpr size_t desc = misc + 16;                      // abort flag, group count
  static constexpr size_t edesc = desc + 2 * sizeof(DDesc);      // two unit descriptors (with the rows)
  static constexpr size_t xexp = edesc + 2 * sizeof(EDesc);      // two output descriptors
  static constexpr size_t zero = xexp + 2 * kDMaxSlots * 4;      // per row buffer: prescale exponent of each slot
  static constexpr size_t gexp = zero + 32;                      // 32 zero bytes: inactive activation columns
  static constexpr size_t grp = gexp + 2 * kDGroupMaxRoutes;     // [R] local expert of each route (-1: none)
  static constexpr size_t gtab = grp + 2 * kDGroupMaxRoutes;     // [R] group of each valid route
  static constexpr size_t lastg = gtab + 8 * kDGroupMaxRoutes;   // [groups] the group's routes (-1 past its size)
  static constexpr size_t tmask = lastg + 2 * kDGroupMaxRoutes;  // [m] last group (in unit order) of a token's routes
  static constexpr size_t total = tmask + 4 * kDGroupMaxRoutes;  // [m] valid top-k slots of each token
  static_assert(gexp % 16 == 0, "the route experts are read 16 bytes at a time");
};

__device__ __forceinline__ int d_local_expert(const DecodeParams& p, int route) {
  if (!p.topk_ids) return 0;  // dense linear layer: one expert, every route valid
  const int id = __ldg(p.topk_ids + route);
  if (id < 0 || id >= p.num_global_experts) return -1;
  const int l = p.expert_map ? __ldg(p.expert_map + id) : id;
  return (l >= 0 && l < p.num_local_experts) ? l : -1;
}

struct DUnit {
  int fc2;
  int route;  // the route, or the group of a grouped unit
  int tile, split, kbeg, kend, expert;
};

// The routes of the call grouped by local expert (grouped units only): up to
// four routes of one expert, in ascending route order, per group; groups in
// the order of their first route.
struct DGroups {
  bool on;
  int ng;              // groups
  const short* gexp;   // [R] local expert of each route (-1: none)
  const short* grp;    // [R] group of each valid route
  const short* gtab;   // [ng][4] routes of each group (-1 past its size)
  const short* lastg;  // [m] a token's last group
  const uint32_t* tmask;  // [m] a token's valid top-k slots
};

// The arithmetic part of d_unit: route (or group), tile, split and K range of
// unit u; units [0, units1) are FC1 units.
__device__ __forceinline__ void d_unit_shape(const DecodeParams& p, int units1, int u, DUnit& U) {
  int nt, ns, ks;
  if (u < units1) {
    U.fc2 = 0, nt = p.n_tiles1, ns = p.s1, ks = p.k_stages1;
  } else {
    u -= units1;
    U.fc2 = 1, nt = p.n_tiles2, ns = p.s2, ks = p.k_stages2;
  }
  const int per_route = nt * ns;
  U.route = u / per_route;
  const int rem = u - U.route * per_route;
  U.tile = rem / ns;
  U.split = rem - U.tile * ns;
  U.kbeg = U.split * ks / ns;  // ks <= 1024 stages, ns <= 8 splits: no overflow
  U.kend = (U.split + 1) * ks / ns;
  U.expert = -1;
}

__device__ __forceinline__ bool d_unit(const DecodeParams& p, const DGroups& G, int units1, int u, DUnit& U) {
  d_unit_shape(p, units1, u, U);
  // a dense linear layer's output units stay one per route
  U.expert = G.on && !(U.fc2 && p.linear) ? G.gexp[G.gtab[4 * U.route]] : d_local_expert(p, U.route);
  return U.expert >= 0 && U.kend > U.kbeg;
}

__device__ __forceinline__ void d_trace(const DecodeParams& p, int kind, uint32_t idx) {
  if (p.trace && blockIdx.x == 0 && idx < (uint32_t)kTraceLen) p.trace[kind * kTraceLen + idx] = clock64();
}
// Per-CTA global timestamps (ns), indexed by CTA: kinds 5 start, 6 last FC2
// partial stored, 7 last FC1 partial stored, 8 compute warps done, 9 output
// warp done, 11 first weight slot computed, 12 first x row converted, 13 grid
// barrier complete; kind 10 holds the CTA's SM.
__device__ __forceinline__ void d_trace_cta(const DecodeParams& p, int kind) {
  if (p.trace && blockIdx.x < (uint32_t)kTraceLen) p.trace[kind * kTraceLen + blockIdx.x] = (long long)globaltimer();
}

// Split grid barrier on the word a cooperative launch provides for
// grid.sync(), with grid.sync()'s arithmetic: every CTA adds 1 once, except
// CTA 0, which adds 2^31 - (G - 1), so the top bit flips exactly when all G
// CTAs have arrived and the low bits end where they started.  The add
// releases the CTA's earlier writes; the polling load acquires every CTA's.
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
      ab.raise(30);
      return false;
    }
  }
}

// The split partials of one element, stored contiguously with stride S
// (s1 <= S of them written), summed in ascending split order.
template <int S>
__device__ __forceinline__ void load_splits(float (&v)[S], const float* src) {
  if (!src) {
#pragma unroll
    for (int i = 0; i < S; ++i) v[i] = 0.f;
  } else if constexpr (S == 1) {
    v[0] = __ldcg(src);
  } else if constexpr (S == 2) {
    const float2 a = __ldcg(reinterpret_cast<const float2*>(src));
    v[0] = a.x, v[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < S; i += 4) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(src + i));
      v[i] = a.x, v[i + 1] = a.y, v[i + 2] = a.z, v[i + 3] = a.w;
    }
  }
}
template <int S>
__device__ __forceinline__ float sum_splits(const float (&v)[S], int s1) {
  float a = v[0];
#pragma unroll
  for (int i = 1; i < S; ++i)
    if (i < s1) a += v[i];
  return a;
}

// Grouped units (m * top_k <= 256): every CTA builds the same group table,
// one thread per route.  A valid route's rank is the number of earlier routes
// of its local expert (counted eight routes per shared-memory load, with the
// last such route kept as its predecessor); ranks 0, 4, 8, ... open a group,
// which the next three routes of that expert join (a member finds its group's
// first route in at most three predecessor steps).  Groups are ordered by
// expert, then by rank, so that an expert's groups are neighbours in unit
// order and its weights are re-read from L2: a group's index is the number of
// groups of lower-numbered experts plus its rank / 4.  Then each token's last
// group (the largest index among its valid routes) and its valid top-k slots.
// Returns the number of groups; scan[] takes one int per warp, and lastg[]
// and tmask[] serve as scratch (predecessors, openers, group of each opener)
// first.
__device__ int build_groups(const DecodeParams& p, int R, short* gexp, short* grp, short* gtab, short* lastg,
                            uint32_t* tmask, int* scan) {
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  short* prev = reinterpret_cast<short*>(tmask);  // [R] the route's predecessor of its expert (-1: none)
  short* opens = prev + kDGroupMaxRoutes;          // [256] 0xFFFF where the route opens a group, else 0
  short* opener_group = lastg;                    // [R] group of a route that opens one
  int e = -1;
  if (i < R) {
    e = d_local_expert(p, i);
    gexp[i] = (short)e;
  }
  if (i < kDGroupMaxRoutes && i >= R) gexp[i] = -2;  // past the routes: matches no expert
  __syncthreads();
  int rank = 0, last = -1;
  if (e >= 0) {
    const uint32_t key = (uint32_t)(uint16_t)e * 0x10001u;
    for (int j = 0; j < i; j += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(gexp + j);
      const uint32_t m[4] = {__vcmpeq2(w.x, key), __vcmpeq2(w.y, key), __vcmpeq2(w.z, key), __vcmpeq2(w.w, key)};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int jj = j + 2 * q + hh;
          if (jj < i && ((m[q] >> (16 * hh)) & 1u)) {
            ++rank;
            last = jj;
          }
        }
      }
    }
    prev[i] = (short)last;
  }
  const bool lead = e >= 0 && (rank & (kDGroupMax - 1)) == 0;
  if (i < kDGroupMaxRoutes) opens[i] = lead ? (short)-1 : (short)0;
  const uint32_t b = __ballot_sync(0xffffffffu, lead);
  if (lane == 0) scan[warp] = __popc(b);
  __syncthreads();
  int ng = 0;
  for (int w = 0; w < kDThreads / 32; ++w) ng += scan[w];
  if (lead) {
    // groups of lower-numbered experts: openers with a smaller expert index
    const uint32_t key = (uint32_t)(uint16_t)e * 0x10001u;
    int bits = 0;  // 16 per opener
    for (int j = 0; j < R; j += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(gexp + j);
      const uint4 o = *reinterpret_cast<const uint4*>(opens + j);
      bits += __popc(__vcmpltu2(w.x, key) & o.x) + __popc(__vcmpltu2(w.y, key) & o.y) +
              __popc(__vcmpltu2(w.z, key) & o.z) + __popc(__vcmpltu2(w.w, key) & o.w);
    }
    const int g = (bits >> 4) + rank / kDGroupMax;
    opener_group[i] = (short)g;
    grp[i] = (short)g;
    gtab[kDGroupMax * g] = (short)i;
#pragma unroll
    for (int k = 1; k < kDGroupMax; ++k) gtab[kDGroupMax * g + k] = -1;
  }
  __syncthreads();
  if (e >= 0 && !lead) {
    int o = i;
    for (int k = 0; k < (rank & (kDGroupMax - 1)); ++k) o = prev[o];
    const int g = opener_group[o];
    grp[i] = (short)g;
    gtab[kDGroupMax * g + (rank & (kDGroupMax - 1))] = (short)i;
  }
  __syncthreads();
  if (i < p.m) {
    int lg = -1;
    uint32_t mask = 0;
    for (int k = 0; k < p.top_k; ++k) {
      const int r = i * p.top_k + k;
      if (gexp[r] >= 0) {
        lg = max(lg, (int)grp[r]);
        mask |= 1u << k;
      }
    }
    lastg[i] = (short)lg;
    tmask[i] = mask;
  }
  __syncthreads();
  return ng;
}

__device__ __forceinline__ int group_size(const DGroups& G, int g) {
  int n = 1;
  while (n < kDGroupMax && G.gtab[kDGroupMax * g + n] >= 0) ++n;
  return n;
}

// FC1 activation rows of one unit: lane 0 copies each route's bf16 x[k0 ..
// k0 + kv) (its token's row) into the row buffer, one bulk copy per route
// completing on xbar (a grouped unit's route i at i * kDGroupRowBytes);
// positions past the hidden size are zeroed by convert_x_rows.
__device__ __forceinline__ void issue_x_rows(const DecodeParams& p, const DGroups& G, const DUnit& U, uint8_t* row,
                                             uint64_t* xbar) {
  const int k0 = U.kbeg * kBK, nk = (U.kend - U.kbeg) * kBK;
  const uint32_t bytes = (uint32_t)min(nk, p.hidden - k0) * 2;  // hidden is a multiple of 16: whole 32-byte pieces
  const int nr = G.on ? group_size(G, U.route) : 1;
  mbar_arrive_expect_tx(xbar, bytes * nr);
  for (int i = 0; i < nr; ++i) {
    const int route = G.on ? G.gtab[kDGroupMax * U.route + i] : U.route;
    bulk_g2s(row + i * kDGroupRowBytes, p.x + (size_t)(route / p.top_k) * p.hidden + k0, bytes, xbar);
  }
}

// The warp converts an x row in place to 128-wide f16 slots, each prescaled
// by a power of two (exps[j]).  Lane l owns K positions 4l .. 4l+3 of a slot
// (block l / 4, quarter l % 4), whose eight bytes are the same in the bf16 and
// the f16 row.  Four slots at a time, so their max-reductions overlap.
__device__ __forceinline__ void convert_x_row(const DecodeParams& p, const DUnit& U, uint8_t* row, int* exps,
                                              int lane) {
  const int k0 = U.kbeg * kBK, nk = (U.kend - U.kbeg) * kBK;
  const int ns = (nk + 127) / 128;
  for (int j0 = 0; j0 < ns; j0 += 4) {
    float v[4][4], a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 128 * (j0 + q) + 4 * lane;  // four positions: all below the hidden size or all past it
      v[q][0] = v[q][1] = v[q][2] = v[q][3] = 0.f;
      if (j0 + q < ns && i < nk && k0 + i < p.hidden) {
        const uint2 w = *reinterpret_cast<const uint2*>(row + 256 * (j0 + q) + 8 * lane);
        v[q][0] = __uint_as_float(w.x << 16), v[q][1] = __uint_as_float(w.x & 0xFFFF0000u);
        v[q][2] = __uint_as_float(w.y << 16), v[q][3] = __uint_as_float(w.y & 0xFFFF0000u);
      }
      a[q] = fmaxf(fmaxf(fabsf(v[q][0]), fabsf(v[q][1])), fmaxf(fabsf(v[q][2]), fabsf(v[q][3])));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int q = 0; q < 4; ++q) a[q] = fmaxf(a[q], __shfl_xor_sync(0xffffffffu, a[q], o));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (j0 + q >= ns) break;
      const int e = slot_prescale(a[q]);
      store_x4_f16(row + 256 * (j0 + q) + 8 * lane, v[q][0], v[q][1], v[q][2], v[q][3], e);
      if (lane == 0) exps[j0 + q] = e;
    }
  }
}
// Waits for a unit's x copies, then converts every route's row (a grouped
// unit's route i: exps at i * kDGroupSlots).  False on timeout.
__device__ __forceinline__ bool convert_x_rows(const DecodeParams& p, const DGroups& G, const DUnit& U, uint8_t* row,
                                               int* exps, uint64_t* xbar, uint32_t parity, int lane,
                                               const Abort& ab) {
  if (!__all_sync(0xffffffffu, mbar_wait(xbar, parity, ab, 34))) return false;
  const int nr = G.on ? group_size(G, U.route) : 1;
  for (int i = 0; i < nr; ++i) convert_x_row(p, U, row + i * kDGroupRowBytes, exps + i * kDGroupSlots, lane);
  return true;
}

// Sums (ascending split order) of the split partials of four consecutive
// elements at each of N sources (splits innermost, stride S; s1 <= S
// written), read again by the whole warp while any written one still holds the
// not-written marker: the N sources share every round trip.  Sources with
// valid[q] == false take zeros and are not read.  False on timeout (abort
// raised).
template <int S, int N>
__device__ __forceinline__ bool poll_sum4(float (&sum)[N][4], const float* const (&src)[N], const bool (&valid)[N],
                                          int s1, const Abort& ab) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    float v[N][4 * S];
    bool ready = true;
#pragma unroll
    for (int q = 0; q < N; ++q) {
      if (valid[q]) {
#pragma unroll
        for (int c = 0; c < 4 * S; c += 4) {
          const float4 a = __ldcg(reinterpret_cast<const float4*>(src[q] + c));
          v[q][c] = a.x, v[q][c + 1] = a.y, v[q][c + 2] = a.z, v[q][c + 3] = a.w;
        }
#pragma unroll
        for (int c = 0; c < 4 * S; ++c)
          if (c % S < s1 && __float_as_uint(v[q][c]) == kNotWritten) ready = false;
      } else {
#pragma unroll
        for (int c = 0; c < 4 * S; ++c) v[q][c] = 0.f;
      }
    }
    if (__all_sync(0xffffffffu, ready)) {
#pragma unroll
      for (int q = 0; q < N; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a = v[q][e * S];
#pragma unroll
          for (int sp = 1; sp < S; ++sp)
            if (sp < s1) a += v[q][e * S + sp];
          sum[q][e] = a;
        }
      return true;
    }
    if (ab.raised() || globaltimer() - t0 > kWaitLimitNs) {
      if (!ab.raised()) ab.raise(40);
      return false;
    }
    __nanosleep(64);
  }
}

// One 128-wide slot j of an FC2 activation row from this lane's four h values
// (already act()-ed; lanes past the unit's K range pass valid == false):
// rounded to bf16, then the slot's power-of-two prescale and f16 as in
// convert_x_row.
__device__ __forceinline__ void store_h_slot(uint8_t* row, int* exps, int j, int lane, bool valid, float (&h)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) h[c] = valid ? __bfloat162float(__float2bfloat16_rn(h[c])) : 0.f;
  float a = fmaxf(fmaxf(fabsf(h[0]), fabsf(h[1])), fmaxf(fabsf(h[2]), fabsf(h[3])));
#pragma unroll
  for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const int e = slot_prescale(a);
  store_x4_f16(row + 256 * j + 8 * lane, h[0], h[1], h[2], h[3], e);
  if (lane == 0) exps[j] = e;
}

// FC2 activation rows of one unit (one per route; a grouped unit's route i at
// i * kDGroupRowBytes, exps at i * kDGroupSlots), built by the eight compute
// warps: h[i] = bf16(act(sum of the FC1 split partials, ascending split
// order)), then the slot's power-of-two prescale and f16 as in convert_x_row.
// Warp w takes items w, w + 8, ... of the (route, 128-wide slot) list; one
// poll reads NS partial sources at once (4 for a split stride of 1,
// else 2): the gate and up partials of NS / 2 SwiGLU items, or NS ReLU^2
// items (w + 8 q for q < NS).  Returns false on timeout (the abort flag is
// raised).
template <int S>
__device__ __forceinline__ bool build_h_f16(const DecodeParams& p, const DGroups& G, const DUnit& U, uint8_t* row,
                                            int* exps, int cw, int lane, int wnat, const Abort& ab) {
  constexpr int NS = S == 1 ? 4 : 2;  // partial sources per poll (4 S floats each in registers)
  const int k0 = U.kbeg * kBK, nk = (U.kend - U.kbeg) * kBK;
  const int ns = (nk + 127) / 128;  // activation slots per route
  const int nr = G.on ? group_size(G, U.route) : 1;
  const int items = nr * ns;
  // item f: route f / ns, slot f % ns; the start of its partials, and whether
  // this lane's four positions of it are inside the K range
  auto item = [&](int f, bool& valid) {
    const int i = f / ns, j = f - i * ns;
    const int e = 128 * j + 4 * lane;
    valid = f < items && e < nk;
    if (!valid) return p.p;
    const int route = G.on ? (int)G.gtab[kDGroupMax * U.route + i] : U.route;
    return p.p + ((size_t)route * wnat + k0 + e) * S;
  };
  auto store = [&](int f, bool valid, float (&h)[4]) {
    const int i = f / ns, j = f - i * ns;
    store_h_slot(row + i * kDGroupRowBytes, exps + i * kDGroupSlots, j, lane, valid, h);
  };
  if (p.act == 0) {
    constexpr int NI = NS / 2;  // items per poll: gate and up of each
    for (int f = cw; f < items; f += NI * kDComputeWarps) {
      const float* src[NS];
      bool vv[NS];
#pragma unroll
      for (int q = 0; q < NI; ++q) {
        const float* gate = item(f + q * kDComputeWarps, vv[2 * q]);
        vv[2 * q + 1] = vv[2 * q];
        src[2 * q] = gate;
        src[2 * q + 1] = vv[2 * q] ? gate + (size_t)p.inter_pad * S : p.p;
      }
      float gu[NS][4];
      if (!poll_sum4<S, NS>(gu, src, vv, p.s1, ab)) return false;
#pragma unroll
      for (int q = 0; q < NI; ++q) {
        if (f + q * kDComputeWarps >= items) break;
        float h[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) h[c] = gated_act(gu[2 * q][c], gu[2 * q + 1][c], p.glu);
        store(f + q * kDComputeWarps, vv[2 * q], h);
      }
    }
  } else {
    for (int f = cw; f < items; f += NS * kDComputeWarps) {
      const float* src[NS];
      bool vv[NS];
#pragma unroll
      for (int q = 0; q < NS; ++q) src[q] = item(f + q * kDComputeWarps, vv[q]);
      float hh[NS][4];
      if (!poll_sum4<S, NS>(hh, src, vv, p.s1, ab)) return false;
#pragma unroll
      for (int q = 0; q < NS; ++q) {
        if (f + q * kDComputeWarps >= items) break;
#pragma unroll
        for (int c = 0; c < 4; ++c) hh[q][c] = hh[q][c] > 0.f ? hh[q][c] * hh[q][c] : 0.f;
        store(f + q * kDComputeWarps, vv[q], hh[q]);
      }
    }
  }
  return true;
}

// Lane 0 of warp 1: a unit's routes into its descriptor (one, or a group's
// up to four), and for a grouped FC2 unit each route's output weight (gs *
// router weight) and whether it triggers its token's output tile: the route
// is its token's first in the token's last group.
__device__ __forceinline__ void fill_routes(const DecodeParams& p, const DGroups& G, const DUnit& U, DDesc* d) {
  int nr = 0;
  uint32_t outs = 0;
  const float gs = U.fc2 && G.on && p.gs2 ? __ldg(p.gs2 + U.expert) : 1.0f;
  for (int i = 0; i < kDGroupMax; ++i) {
    const int r = G.on ? (int)G.gtab[kDGroupMax * U.route + i] : (i == 0 ? U.route : -1);
    d->route[i] = (short)r;
    if (r < 0) continue;
    nr = i + 1;
    if (U.fc2 && G.on) {
      d->rw[i] = gs * __ldg(p.topk_weights + r);
      const int tk = r / p.top_k;
      bool first = G.lastg[tk] == U.route;
      for (int j = 0; j < i; ++j)
        if (d->route[j] / p.top_k == tk) first = false;
      if (first) outs |= 1u << i;
    }
  }
  d->nr = nr;
  d->outs = outs;
}

// Dense linear layer: out[token][n] = bf16(sum of the FC1 split partials of
// column n, ascending split order) for the unit's 128 columns, one compute
// thread per column; a partial still holding the not-written marker is read
// again.  Returns false on timeout (the abort flag is raised).
template <int S>
__device__ __forceinline__ bool linear_out(const DecodeParams& p, const DUnit& U, int tid, const Abort& ab) {
  const int n = U.tile * kTileRows + tid;
  if (tid >= kTileRows || n >= p.n_out) return true;
  const float* src = p.p + ((size_t)U.route * p.inter_pad + n) * S;
  const unsigned long long t0 = globaltimer();
  float v[S];
  while (true) {
    load_splits<S>(v, src);
    bool ready = true;
#pragma unroll
    for (int sp = 0; sp < S; ++sp)
      if (sp < p.s1 && __float_as_uint(v[sp]) == kNotWritten) ready = false;
    if (ready) break;
    if (ab.raised() || globaltimer() - t0 > kWaitLimitNs) {
      if (!ab.raised()) ab.raise(45);
      return false;
    }
    __nanosleep(64);
  }
  p.out[(size_t)(U.route / p.top_k) * p.n_out + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum_splits<S>(v, p.s1)));
  return true;
}

// ------------------------------------------------------------------ fused
// GRP: grouped units (p.group_max > 1); the one-route kernel carries none of
// their code.
template <int FMT, bool GRP>
__global__ void __launch_bounds__(kDThreads, kDMinBlocks) decode_moe_kernel(const __grid_constant__ DecodeParams p) {
  using L = DSmem<FMT>;
  constexpr int SB = scale_bytes_per_row(FMT);
  constexpr int kSS = L::kScaleStage;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_codes = smem + L::codes;
  uint8_t* s_scales = smem + L::scales;
  uint8_t* s_rows = smem + L::rows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + kDSlots;
  uint64_t* full_b = empty_w + kDSlots;
  uint64_t* empty_b = full_b + 2;
  uint64_t* epi_full = empty_b + 2;
  uint64_t* epi_empty = epi_full + 2;
  uint64_t* desc_full = epi_empty + 2;  // a unit descriptor is ready (for the weight stream)
  uint64_t* grid_bar = desc_full + 2;   // completes once every CTA has arrived at the grid barrier
  uint64_t* xbar = grid_bar + 1;        // [2] the bf16 x slices of an FC1 unit have landed
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc);
  DDesc* s_desc = reinterpret_cast<DDesc*>(smem + L::desc);    // [2] with the rows
  EDesc* s_edesc = reinterpret_cast<EDesc*>(smem + L::edesc);  // [2] for the output warp
  int* s_xexp = reinterpret_cast<int*>(smem + L::xexp);        // [2][kDMaxSlots]
  uint8_t* s_zero = smem + L::zero;
  short* s_gexp = reinterpret_cast<short*>(smem + L::gexp);
  short* s_grp = reinterpret_cast<short*>(smem + L::grp);
  short* s_gtab = reinterpret_cast<short*>(smem + L::gtab);
  short* s_lastg = reinterpret_cast<short*>(smem + L::lastg);
  uint32_t* s_tmask = reinterpret_cast<uint32_t*>(smem + L::tmask);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{p.status, s_abort};
  const int R = p.m * p.top_k;
  if (threadIdx.x == 0) {
    d_trace(p, 2, 0);
    d_trace_cta(p, 5);
    if (p.trace && blockIdx.x < (uint32_t)kTraceLen) p.trace[10 * kTraceLen + blockIdx.x] = smid();
    *s_abort = 0;
    for (int i = 0; i < kDSlots; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&empty_w[i], kDComputeWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_b[i], 1);
      mbar_init(&empty_b[i], kDComputeWarps);
      mbar_init(&epi_full[i], kDComputeWarps);
      mbar_init(&epi_empty[i], 1);
      mbar_init(&desc_full[i], 1);
    }
    mbar_init(grid_bar, 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 8) reinterpret_cast<uint32_t*>(s_zero)[threadIdx.x] = 0u;
  if (threadIdx.x == 0) pdl_launch_dependents();  // the next kernel may launch and set up meanwhile
  __syncthreads();
  pdl_wait();  // launched with PDL: nothing of this call is read or written before the kernel before it is done
  if (!cg::this_grid().is_valid()) {  // not a cooperative launch: there is no grid barrier to wait on
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0u, 4u);  // B4_ERR_CUDA
    return;
  }

  // Units are per route, or per group of up to four routes of one expert
  // (the group table is built here, by every CTA alike; the exponent area is
  // free scratch until the first x row is converted).
  DGroups G{GRP, 0, s_gexp, s_grp, s_gtab, s_lastg, s_tmask};
  if (G.on) G.ng = build_groups(p, R, s_gexp, s_grp, s_gtab, s_lastg, s_tmask, s_xexp);
  const int base = G.on ? G.ng : R;
  const int units1 = G.on ? base * p.n_tiles1 * p.s1 : p.units1;
  const int n_units = units1 + (G.on && !p.linear ? base * p.n_tiles2 * p.s2 : p.units2);

  // The producers resolve the CTA's first unit and start its weight stream
  // and (FC1) x slices before the grid barrier: neither touches the partial
  // buffers.
  DUnit U0;
  const bool u0_ok = warp < 2 && (int)blockIdx.x < n_units && d_unit(p, G, units1, blockIdx.x, U0);
  const bool x_pre = u0_ok && !U0.fc2;  // warp 0 issues the first unit's x slices
  uint32_t pre_slots = 0;
  if (warp == 0 && lane == 0 && x_pre) issue_x_rows(p, G, U0, s_rows, &xbar[0]);  // ahead of the weights
  if (warp == 0 && lane == 0 && u0_ok && !(U0.fc2 && p.linear)) {
    const size_t tile_id = (size_t)U0.expert * (U0.fc2 ? p.n_tiles2 : p.n_tiles1) + U0.tile;
    const int ks = U0.fc2 ? p.k_stages2 : p.k_stages1;
    const uint8_t* gc = (U0.fc2 ? p.w2_codes : p.w1_codes) + tile_id * ks * kCodeBytesPerStage;
    const uint8_t* gsc = (U0.fc2 ? p.w2_scales : p.w1_scales) + tile_id * ks * kSS;
    for (int s = U0.kbeg; s < U0.kend && pre_slots < (uint32_t)kDSlots; s += kDSlotStages, ++pre_slots) {
      const int n = min(kDSlotStages, U0.kend - s);
      mbar_arrive_expect_tx(&full_w[pre_slots], n * (kCodeBytesPerStage + kSS));
      bulk_g2s(s_codes + pre_slots * kDSlotStages * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage,
               n * kCodeBytesPerStage, &full_w[pre_slots]);
      bulk_g2s(s_scales + pre_slots * kDSlotStages * kSS, gsc + (size_t)s * kSS, n * kSS, &full_w[pre_slots]);
      d_trace(p, 0, pre_slots);
    }
    d_trace_cta(p, 14);
  }
  // Warp 1 publishes the first unit and converts its x slices before the
  // CTA's grid-barrier arrival: the arriving atomic (a release at GPU scope)
  // made while the first copies are in flight delays them.
  if (warp == 1 && x_pre) {
    if (lane == 0) {
      s_desc[0].u = blockIdx.x;
      s_desc[0].expert = U0.expert;
      mbar_arrive(&desc_full[0]);
      s_desc[0].scale = p.gs1 ? __ldg(p.gs1 + U0.expert) : 1.0f;
      fill_routes(p, G, U0, &s_desc[0]);
    }
    convert_x_rows(p, G, U0, s_rows, s_xexp, &xbar[0], 0, lane, ab);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&full_b[0]);
      d_trace_cta(p, 12);
    }
  }

  // Before the grid barrier: fill both partial buffers with the not-written
  // marker, clear the status word, and zero the output rows of tokens without
  // a valid route (no unit writes them).
  {
    const size_t gt = (size_t)blockIdx.x * kDThreads + threadIdx.x, gstride = (size_t)gridDim.x * kDThreads;
    const uint4 mark = make_uint4(kNotWritten, kNotWritten, kNotWritten, kNotWritten);
    for (size_t i = gt; i < p.p_floats / 4; i += gstride) reinterpret_cast<uint4*>(p.p)[i] = mark;
    for (size_t i = gt; i < p.q_floats / 4; i += gstride) reinterpret_cast<uint4*>(p.q)[i] = mark;
    if (gt == 0) {
      *p.ticket = 0;
      if (p.status) {
        p.status[0] = 0;
        p.status[1] = 0;
      }
    }
    const int gw = (int)(gt >> 5), nw = (int)(gstride >> 5);
    for (int tk = gw; tk < p.m; tk += nw) {
      const bool v = lane < p.top_k && d_local_expert(p, tk * p.top_k + lane) >= 0;
      if (__ballot_sync(0xffffffffu, v) == 0) {
        uint4* o = reinterpret_cast<uint4*>(p.out + (size_t)tk * p.hidden);
        for (int i = lane; i < p.hidden / 8; i += 32) o[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  // Every thread's fill precedes the CTA's arrival (a release at GPU scope),
  // which the output warp makes: the arriving atomic can hold its warp for
  // microseconds, and that warp has nothing to do before the first partials
  // exist, while warp 1 goes on to publish the CTA's second unit.  It then
  // waits for the other CTAs and completes grid_bar, which the first partial
  // store or read of each warp and the first claimed unit wait on (acquire).
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------ weight stream
    // follows the unit sequence that warp 1 publishes in the descriptors
    if (lane == 0) {
      uint32_t ws = 0;
      for (uint32_t ds = 0; !ab.raised(); ++ds) {
        const uint32_t rb = ds & 1;
        if (!mbar_wait(&desc_full[rb], (ds >> 1) & 1, ab, 31)) break;
        const int u = s_desc[rb].u;
        if (u < 0) break;
        DUnit U;
        d_unit_shape(p, units1, u, U);
        if (U.fc2 && p.linear) continue;  // an output unit of the dense linear layer streams no weights
        U.expert = s_desc[rb].expert;
        const size_t tile_id = (size_t)U.expert * (U.fc2 ? p.n_tiles2 : p.n_tiles1) + U.tile;
        const int ks = U.fc2 ? p.k_stages2 : p.k_stages1;
        const uint8_t* gc = (U.fc2 ? p.w2_codes : p.w1_codes) + tile_id * ks * kCodeBytesPerStage;
        const uint8_t* gsc = (U.fc2 ? p.w2_scales : p.w1_scales) + tile_id * ks * kSS;
        for (int s = U.kbeg; s < U.kend; s += kDSlotStages, ++ws) {
          if (ws < pre_slots) continue;  // issued before the grid barrier
          const uint32_t slot = ws % kDSlots;
          if (!mbar_wait(&empty_w[slot], ((ws / kDSlots) & 1) ^ 1, ab, 32)) break;
          const int n = min(kDSlotStages, U.kend - s);
          mbar_arrive_expect_tx(&full_w[slot], n * (kCodeBytesPerStage + kSS));
          bulk_g2s(s_codes + slot * kDSlotStages * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage,
                   n * kCodeBytesPerStage, &full_w[slot]);
          bulk_g2s(s_scales + slot * kDSlotStages * kSS, gsc + (size_t)s * kSS, n * kSS, &full_w[slot]);
          d_trace(p, 0, ws);
        }
      }
      if (ab.raised()) {  // let issued copies land before the CTA exits
        const uint32_t n = ws < (uint32_t)kDSlots ? ws : (uint32_t)kDSlots;
        for (uint32_t i = ws - n; i < ws; ++i) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full_w[i % kDSlots], (i / kDSlots) & 1) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
    return;
  }

  if (warp == 1) {
    // ------------------------------------- unit schedule and activation rows
    // The CTA's first two units are units blockIdx.x and blockIdx.x + G, so
    // the second one's weights stream while the first computes, whatever the
    // grid barrier is doing; later ones are claimed from a counter in unit
    // order (a CTA that runs faster takes more), after the grid barrier (the
    // counter is reset before it).  Each unit is resolved once and published
    // with the FC1 x slices in one of two descriptor/row slots; a unit index
    // of -1 ends the sequence.
    uint32_t bs = x_pre ? 1 : 0;                // the first unit went out before the grid barrier
    uint32_t xuse0 = x_pre ? 1 : 0, xuse1 = 0;  // FC1 x copies per row buffer (phase of xbar)
    int taken = x_pre ? 1 : 0;                  // static units taken
    bool synced = false;                        // grid_bar seen complete
    DUnit U;
    int u = 0;
    while (!ab.raised()) {
      // next valid unit: claims are issued one unit ahead of their use
      bool have = false;
      while (!have) {
        if (taken < 2) {
          u = (int)blockIdx.x + taken * (int)gridDim.x;
          ++taken;
        } else {
          if (!synced) {
            if (!__all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 46))) break;
            synced = true;
          }
          int t = 0;
          if (lane == 0) t = atomicAdd(p.ticket, 1);
          u = 2 * (int)gridDim.x + __shfl_sync(0xffffffffu, t, 0);
        }
        if (u >= n_units) break;
        have = d_unit(p, G, units1, u, U);
      }
      if (ab.raised()) break;
      const uint32_t rb = bs & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&empty_b[rb], ((bs >> 1) & 1) ^ 1, ab, 33))) break;
      DDesc* dsc = s_desc + rb;
      if (!have) {
        if (lane == 0) {
          dsc->u = -1;
          mbar_arrive(&full_b[rb]);
          mbar_arrive(&desc_full[rb]);
        }
        break;
      }
      if (!U.fc2) {
        uint8_t* row = s_rows + rb * kDRowBytes;
        if (lane == 0) {
          dsc->u = u;
          dsc->expert = U.expert;
          mbar_arrive(&desc_full[rb]);  // the weight stream needs only the unit
          issue_x_rows(p, G, U, row, &xbar[rb]);
          dsc->scale = p.gs1 ? __ldg(p.gs1 + U.expert) : 1.0f;
          fill_routes(p, G, U, dsc);
        }
        const uint32_t xu = rb ? xuse1 : xuse0;
        convert_x_rows(p, G, U, row, s_xexp + rb * kDMaxSlots, &xbar[rb], xu & 1, lane, ab);
        if (rb) ++xuse1;
        else ++xuse0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_b[rb]);
      } else if (p.linear || G.on) {
        // an output unit of the dense linear layer (one route), or a grouped FC2 unit
        if (lane == 0) {
          dsc->u = u;
          dsc->expert = U.expert;
          mbar_arrive(&desc_full[rb]);
          dsc->scale = 1.0f;
          dsc->mask = 1u;
          if (p.linear) dsc->nr = 1;
          else fill_routes(p, G, U, dsc);
          mbar_arrive(&full_b[rb]);
        }
      } else {
        if (lane == 0) {
          dsc->u = u;
          dsc->expert = U.expert;
          mbar_arrive(&desc_full[rb]);
        }
        const int token = U.route / p.top_k;
        const bool v = lane < p.top_k && d_local_expert(p, token * p.top_k + lane) >= 0;
        const uint32_t mask = __ballot_sync(0xffffffffu, v);
        if (lane == 0) {
          dsc->scale = (p.gs2 ? __ldg(p.gs2 + U.expert) : 1.0f) * __ldg(p.topk_weights + U.route);
          dsc->mask = mask;
          fill_routes(p, G, U, dsc);
          mbar_arrive(&full_b[rb]);
        }
      }
      ++bs;
    }
    if (ab.raised() && lane == 0) {  // let issued x copies land before the CTA exits
      for (int i = 0; i < 2; ++i) {
        const uint32_t n = i ? xuse1 : xuse0;
        if (n == 0) continue;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&xbar[i], (n - 1) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
    return;
  }

  if (warp == 2 + kDComputeWarps) {
    // ------------------------------------------------------ output tiles
    if (lane == 0) {
      uint32_t* word = &cg::details::get_grid_workspace()->barrier;
      if (grid_wait(word, grid_arrive(word), ab)) {
        mbar_arrive(grid_bar);
        d_trace_cta(p, 13);
      }
    }
    if (!__all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 42))) return;
    for (uint32_t es = 0;; ++es) {
      const uint32_t eb = es & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&epi_full[eb], (es >> 1) & 1, ab, 37))) break;
      const EDesc ed = s_edesc[eb];
      if (ed.end) break;
      const int token = ed.token;
      const uint32_t mask = ed.mask;
      // out = bf16(sum over valid routes and splits); each lane has 4 outputs
      // and 8 routes' partial loads are in flight at once.  Order: ascending
      // top-k slot within groups of 8, splits outer within a group.
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const int nb = ed.tile * kTileRows + lane;
      for (int jb = 0; jb < p.top_k; jb += 8) {
        for (int sp = 0; sp < p.s2; ++sp) {
          float v[8][4];
          const unsigned long long t0 = globaltimer();
          while (true) {
            bool ready = true;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = jb + jj;
              const bool valid = j < p.top_k && ((mask >> j) & 1u);
              const float* qr = p.q + ((size_t)sp * R + token * p.top_k + j) * p.hidden + nb;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                v[jj][c] = valid && nb + 32 * c < p.hidden ? __ldcg(qr + 32 * c) : 0.f;
                if (__float_as_uint(v[jj][c]) == kNotWritten) ready = false;
              }
            }
            if (__all_sync(0xffffffffu, ready)) break;
            if (ab.raised() || globaltimer() - t0 > kWaitLimitNs) {
              if (!ab.raised()) ab.raise(41);
              break;
            }
            __nanosleep(64);
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] += v[jj][c];
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (nb + 32 * c < p.hidden)
          p.out[(size_t)token * p.hidden + nb + 32 * c] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[c]));
      __syncwarp();
      if (lane == 0) mbar_arrive(&epi_empty[eb]);
    }
    if (lane == 0) d_trace_cta(p, 9);
    return;
  }

  // --------------------------------------------------------- compute warps
  // The eight compute warps share named barriers, so none of them leaves the
  // unit loop alone: a failed (bounded) wait sets `bad`, the warp skips the
  // work but still passes every barrier, and the loop ends only by an OR
  // taken over all of them.
  const int cw = warp - 2;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = 16 * cw + g, r1 = r0 + 8;
  const int tid = threadIdx.x - 64;
  constexpr uint32_t kNC = 32 * kDComputeWarps;
  // this thread's 8 code bytes of row r0 (block t of the stage) and of row r1
  const uint32_t code_off = (t >> 1) * (kCodeBytesPerStage / 2) + r0 * 16 + (t & 1) * 8;
  // Accumulator columns 2t, 2t+1 hold, in a one-route unit, the sums of blocks
  // 2t, 2t+1 of a 128-wide chunk (stage t >> 1 of it); in a grouped unit, the
  // sums of blocks 2(t&1), 2(t&1)+1 of every stage for route t >> 1 of the MMA
  // half.  Their scale bytes:
  const uint32_t scg_off = FMT == 0 ? r0 * SB + 2 * (t & 1) : r0 * SB + (t & 1);
  const uint32_t sc_off = (t >> 1) * kSS + scg_off;
  // One-route unit: MMA column g is block g of a chunk, so this thread's
  // activation operand is nonzero in the chunk's first stage when g == t and
  // in its second when g == t + 4.  Grouped unit: in every stage, columns 0-3
  // of MMA half h are route 2h (this thread supplies it when g == t) and
  // columns 4-7 route 2h + 1 (when g == t + 4).
  const bool col0 = g == t, col1 = g == t + 4;
  const int wnat = fc1_natural_width(p.act, p.inter_pad);
  uint32_t ws = 0, bs = 0, es = 0;
  bool synced = false;  // grid_bar seen complete
  bool bad = false;     // a wait of this warp failed (the abort flag is raised)
  while (true) {
    const uint32_t rb = bs & 1;
    if (!bad && !__all_sync(0xffffffffu, mbar_wait(&full_b[rb], (bs >> 1) & 1, ab, 35))) bad = true;
    if (named_bar_or(3, kNC, bad || ab.raised())) break;
    const DDesc* dp = s_desc + rb;
    const int du = dp->u;
    if (du < 0) break;
    DUnit U;
    d_unit_shape(p, units1, du, U);
    if (U.fc2 && !synced) {  // an FC2 or output unit reads other CTAs' partials
      if (!__all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 43))) bad = true;
      synced = true;
    }
    if (U.fc2 && p.linear) {
      // dense linear layer: this unit writes 128 columns of out
      if (!bad) {
        switch (p.s1_stride) {
          case 1: linear_out<1>(p, U, tid, ab); break;
          case 2: linear_out<2>(p, U, tid, ab); break;
          case 4: linear_out<4>(p, U, tid, ab); break;
          default: linear_out<8>(p, U, tid, ab); break;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_b[rb]);
      ++bs;
      continue;
    }
    uint8_t* row = s_rows + rb * kDRowBytes;
    int* xexp = s_xexp + rb * kDMaxSlots;
    const int nr = dp->nr;
    if (U.fc2) {
      // h = act(sum over FC1 splits) for this unit's K range, as f16 slots
      if (!bad) {
        bool built;
        switch (p.s1_stride) {
          case 1: built = build_h_f16<1>(p, G, U, row, xexp, cw, lane, wnat, ab); break;
          case 2: built = build_h_f16<2>(p, G, U, row, xexp, cw, lane, wnat, ab); break;
          default: built = build_h_f16<4>(p, G, U, row, xexp, cw, lane, wnat, ab); break;
        }
        bad = !built;
      }
      bad = named_bar_or(1, kNC, bad);
    }
    if (tid == 0) d_trace(p, 3, bs);
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [MMA half][row r0, r1]
    if (!GRP || nr == 1) {
      const uint8_t* xb0 = col0 ? row + g * 32 : s_zero;
      const uint8_t* xb1 = col1 ? row + g * 32 : s_zero;
      const int xstep0 = col0 ? 256 : 0, xstep1 = col1 ? 256 : 0;
      for (int s = U.kbeg, k = 0; !bad && s < U.kend; s += kDSlotStages, ++ws, ++k) {
        const uint32_t slot = ws % kDSlots;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_w[slot], (ws / kDSlots) & 1, ab, 36))) {
          bad = true;
          break;
        }
        if (tid == 0 && ws == 0) d_trace_cta(p, 15);
        const int ns = min(kDSlotStages, U.kend - s);
#pragma unroll
        for (int c = 0; c < kDSlotStages; c += 2) {  // the slot's 128-wide chunks
          if (c >= ns) break;
          const int j = 2 * k + c / 2;  // its activation slot
          const bool two = ns - c >= 2;
          const uint8_t* cs = s_codes + (slot * kDSlotStages + c) * kCodeBytesPerStage + code_off;
          const uint8_t* ss = s_scales + (slot * kDSlotStages + c) * kSS + sc_off;
          const int xe = xexp[j];
          float de[4] = {0.f, 0.f, 0.f, 0.f}, dq[4] = {0.f, 0.f, 0.f, 0.f};
          {
            const uint2 w0 = *reinterpret_cast<const uint2*>(cs);
            const uint2 w1 = *reinterpret_cast<const uint2*>(cs + 8 * 16);
            stage_mma_f16(w0, w1, xb0 + j * xstep0, de, dq);
          }
          if (two) {
            const uint2 w0 = *reinterpret_cast<const uint2*>(cs + kCodeBytesPerStage);
            const uint2 w1 = *reinterpret_cast<const uint2*>(cs + kCodeBytesPerStage + 8 * 16);
            stage_mma_f16(w0, w1, xb1 + j * xstep1, de, dq);
          }
          // columns of a missing second stage are zero and their scale bytes were not loaded
          if (two || t < 2) {
            if constexpr (FMT == 0) {
              const uint32_t u0 = *reinterpret_cast<const uint16_t*>(ss);
              const uint32_t u1 = *reinterpret_cast<const uint16_t*>(ss + 8 * SB);
              acc[0][0] = fmaf(de[0] + dq[0], f32_scale<0>(u0 & 0xFFu, xe), acc[0][0]);
              acc[0][0] = fmaf(de[1] + dq[1], f32_scale<0>(u0 >> 8, xe), acc[0][0]);
              acc[0][1] = fmaf(de[2] + dq[2], f32_scale<0>(u1 & 0xFFu, xe), acc[0][1]);
              acc[0][1] = fmaf(de[3] + dq[3], f32_scale<0>(u1 >> 8, xe), acc[0][1]);
            } else {
              acc[0][0] = fmaf((de[0] + dq[0]) + (de[1] + dq[1]), f32_scale<1>(ss[0], xe), acc[0][0]);
              acc[0][1] = fmaf((de[2] + dq[2]) + (de[3] + dq[3]), f32_scale<1>(ss[8 * SB], xe), acc[0][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_w[slot]);
        if (tid == 0) {
          d_trace(p, 1, ws);
          if (ws == 0) d_trace_cta(p, 11);
        }
      }
      // row totals: the quad's four threads hold two blocks of each chunk each
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        acc[0][0] += __shfl_xor_sync(0xffffffffu, acc[0][0], o);
        acc[0][1] += __shfl_xor_sync(0xffffffffu, acc[0][1], o);
      }
    } else {
      // grouped unit: the stage's codes are converted once and feed one MMA
      // half (routes 0, 1) or two (routes 2, 3 as well); block scales and
      // each route's activation prescale apply to every stage's sums
      const int nh = nr > 2 ? 2 : 1;
      const uint8_t* xh[2];
      int xo_on[2], xeb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ri = 2 * h + (col0 ? 0 : 1);  // the route this thread supplies activations of
        const bool live = (col0 || col1) && ri < nr;
        xh[h] = live ? row + ri * kDGroupRowBytes + t * 32 : s_zero;
        xo_on[h] = live ? 1 : 0;
        const int ra = 2 * h + (t >> 1);  // the route of this thread's accumulator columns
        xeb[h] = ra < nr ? ra * kDGroupSlots : -1;
      }
      for (int s = U.kbeg, k = 0; !bad && s < U.kend; s += kDSlotStages, ++ws, ++k) {
        const uint32_t slot = ws % kDSlots;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_w[slot], (ws / kDSlots) & 1, ab, 36))) {
          bad = true;
          break;
        }
        if (tid == 0 && ws == 0) d_trace_cta(p, 15);
        const int ns = min(kDSlotStages, U.kend - s);
#pragma unroll
        for (int c = 0; c < kDSlotStages; ++c) {  // the slot's stages
          if (c >= ns) break;
          const int j = 2 * k + (c >> 1);          // activation slot
          const int xo = j * 256 + (c & 1) * 128;  // this stage's half of it
          const uint8_t* cs = s_codes + (slot * kDSlotStages + c) * kCodeBytesPerStage + code_off;
          const uint8_t* ss = s_scales + (slot * kDSlotStages + c) * kSS + scg_off;
          F16Stage f;
          dequant_stage_f16(*reinterpret_cast<const uint2*>(cs), *reinterpret_cast<const uint2*>(cs + 8 * 16), f);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h >= nh) break;
            float de[4] = {0.f, 0.f, 0.f, 0.f}, dq[4] = {0.f, 0.f, 0.f, 0.f};
            mma_stage_f16(f, xh[h] + (xo_on[h] ? xo : 0), de, dq);
            const int xe = xeb[h] >= 0 ? xexp[xeb[h] + j] : 0;  // columns of a missing route are zero
            if constexpr (FMT == 0) {
              const uint32_t u0 = *reinterpret_cast<const uint16_t*>(ss);
              const uint32_t u1 = *reinterpret_cast<const uint16_t*>(ss + 8 * SB);
              acc[h][0] = fmaf(de[0] + dq[0], f32_scale<0>(u0 & 0xFFu, xe), acc[h][0]);
              acc[h][0] = fmaf(de[1] + dq[1], f32_scale<0>(u0 >> 8, xe), acc[h][0]);
              acc[h][1] = fmaf(de[2] + dq[2], f32_scale<0>(u1 & 0xFFu, xe), acc[h][1]);
              acc[h][1] = fmaf(de[3] + dq[3], f32_scale<0>(u1 >> 8, xe), acc[h][1]);
            } else {
              acc[h][0] = fmaf((de[0] + dq[0]) + (de[1] + dq[1]), f32_scale<1>(ss[0], xe), acc[h][0]);
              acc[h][1] = fmaf((de[2] + dq[2]) + (de[3] + dq[3]), f32_scale<1>(ss[8 * SB], xe), acc[h][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_w[slot]);
        if (tid == 0) {
          d_trace(p, 1, ws);
          if (ws == 0) d_trace_cta(p, 11);
        }
      }
      // row totals: threads t and t ^ 1 hold the two halves of a route's blocks
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        acc[h][0] += __shfl_xor_sync(0xffffffffu, acc[h][0], 1);
        acc[h][1] += __shfl_xor_sync(0xffffffffu, acc[h][1], 1);
      }
    }
    bad = named_bar_or(2, kNC, bad);
    // what the stores and output triggers need, before the descriptor slot is released
    const float dscale = dp->scale;
    const uint32_t dmask = dp->mask, douts = dp->outs;
    int droute[kDGroupMax];
#pragma unroll
    for (int i = 0; i < kDGroupMax; ++i) droute[i] = dp->route[i];
    const float drw0 = dp->rw[t >> 1], drw1 = dp->rw[2 + (t >> 1)];  // this thread's routes of halves 0 and 1
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_b[rb]);
    ++bs;
    if (bad) continue;  // the loop ends at the next agreement
    if (!synced) {
      if (!__all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 44))) bad = true;
      synced = true;
      if (bad) continue;
    }
    // partial stores: FC1 in natural row order (splits innermost), times gs;
    // FC2 times gs and the route's router weight
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int route, r;
      float v;
      if (!GRP || nr == 1) {
        if (h > 0 || t >= 2) continue;
        route = droute[0], r = t ? r1 : r0;
        v = (t ? acc[0][1] : acc[0][0]) * (U.fc2 && G.on ? drw0 : dscale);
      } else {
        const int ri = 2 * h + (t >> 1);
        if (ri >= nr) continue;
        route = (t >> 1) ? droute[2 * h + 1] : droute[2 * h], r = (t & 1) ? r1 : r0;
        v = ((t & 1) ? acc[h][1] : acc[h][0]) * (U.fc2 ? (h ? drw1 : drw0) : dscale);
      }
      if (!U.fc2) {
        int nat;
        if (p.act == 0) {
          const int i = U.tile * 64 + (r >> 5) * 16 + (r & 15);
          nat = (r & 31) >= 16 ? p.inter_pad + i : i;
        } else {
          nat = U.tile * kTileRows + r;
          if (nat >= p.inter_pad) nat = -1;
        }
        if (nat >= 0) p.p[((size_t)route * wnat + nat) * p.s1_stride + U.split] = v;
      } else {
        const int n = U.tile * kTileRows + r;
        if (n < p.hidden) p.q[((size_t)U.split * R + route) * p.hidden + n] = v;
      }
    }
    if (tid == 0) d_trace_cta(p, U.fc2 ? 6 : 7);
    if (U.fc2 && U.split == p.s2 - 1) {
      // the output tiles this unit completes (in unit order): a one-route
      // unit when its route is its token's last valid top-k slot, a grouped
      // unit for the routes its descriptor marks
      const int ntrig = G.on ? nr : 1;
#pragma unroll
      for (int i = 0; i < kDGroupMax; ++i) {
        if (i >= ntrig) break;
        int token;
        uint32_t mask;
        if (G.on) {
          if (!((douts >> i) & 1u)) continue;
          token = droute[i] / p.top_k;
          mask = G.tmask[token];
        } else {
          if ((U.route % p.top_k) != 31 - __clz(dmask)) continue;
          token = U.route / p.top_k;
          mask = dmask;
        }
        const uint32_t eb = es & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&epi_empty[eb], ((es >> 1) & 1) ^ 1, ab, 38))) {
          bad = true;
          break;
        }
        if (tid == 0) s_edesc[eb] = EDesc{U.tile, token, mask, 0};
        __syncwarp();
        if (lane == 0) mbar_arrive(&epi_full[eb]);
        ++es;
      }
      if (bad) continue;
    }
    if (tid == 0) d_trace(p, 4, bs - 1);
  }
  // end of the output-tile sequence
  const uint32_t eb = es & 1;
  if (__all_sync(0xffffffffu, mbar_wait(&epi_empty[eb], ((es >> 1) & 1) ^ 1, ab, 39))) {
    if (tid == 0) s_edesc[eb].end = 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&epi_full[eb]);
  }
  if (tid == 0) d_trace_cta(p, 8);
}

template <int FMT, bool GRP>
cudaError_t launch_decode_fmt(const DecodeParams& p, int grid, cudaStream_t stream) {
  auto kern = decode_moe_kernel<FMT, GRP>;
  const size_t smem = DSmem<FMT>::total;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_cooperative(kern, grid, kDThreads, smem, stream, p);
}

const void* decode_kernel_ptr(int fmt, bool grouped) {
  if (fmt == 0) return grouped ? reinterpret_cast<const void*>(decode_moe_kernel<0, true>)
                               : reinterpret_cast<const void*>(decode_moe_kernel<0, false>);
  return grouped ? reinterpret_cast<const void*>(decode_moe_kernel<1, true>)
                 : reinterpret_cast<const void*>(decode_moe_kernel<1, false>);
}

// Resident CTAs per SM of the fused decode kernel on the current device: a
// cooperative launch never exceeds the resident count, so every CTA runs at
// once and a wait on another CTA's unit always ends (each wait is bounded as
// well).  Kept per device and kernel, under a lock.
cudaError_t decode_occupancy(int fmt, bool grouped, int* blocks_per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static int cached[64][2][2] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev][fmt][grouped]) {
    *blocks_per_sm = cached[dev][fmt][grouped];
    return cudaSuccess;
  }
  const void* k = decode_kernel_ptr(fmt, grouped);
  const size_t smem = fmt == 0 ? DSmem<0>::total : DSmem<1>::total;
  e = ensure_smem_limit(k, smem);
  int occ = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kDThreads, smem);
  if (e != cudaSuccess) return e;
  if (dev < 64) cached[dev][fmt][grouped] = occ;
  *blocks_per_sm = occ;
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, int fmt, int grid, cudaStream_t stream) {
  const bool grouped = p.group_max > 1;
  if (fmt == 0) return grouped ? launch_decode_fmt<0, true>(p, grid, stream) : launch_decode_fmt<0, false>(p, grid, stream);
  return grouped ? launch_decode_fmt<1, true>(p, grid, stream) : launch_decode_fmt<1, false>(p, grid, stream);
}

}  // namespace b4
