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
// Hand-offs.  A unit stores an fp32 partial per (route, row) and piece.  The
// epilogue warps count finished pieces per tile (acquire-release atomics); the
// CTA that finishes a tile's last piece sums its pieces in piece order: FC1
// tiles into bf16 h (activation applied) -- then it marks the tile ready --
// and FC2 tiles into per-token completion counts, whose last route sums the
// token's 128 output columns over its routes (ascending top-k slot) and their
// pieces and rounds once to bf16.  Every sum has a fixed order, so the output
// is bitwise reproducible.  The FC2 activation loads wait per stage for the
// FC1 tile that holds those h columns.  Counters are zeroed at launch before a
// grid barrier that nothing waits on until its first counter access.  FC1
// never waits for other CTAs, the cooperative launch keeps every CTA
// resident, so every wait ends; each is bounded as well.
//
// Roles (one CTA per SM, 23 warps):
//   warp 0        weight stream: bulk copies of two 64-wide stages of codes and
//                 scales per slot of a shared-memory ring;
//   warp 1        builds the group table, publishes unit descriptors and
//                 prefetches the CTA's FC2 weights into L2 at launch;
//   warps 2..17   compute: warp w handles rows 16*(w%8)..+15 of the tile for
//                 the stages of one parity (w/8) of each slot; register
//                 dequantisation (E2M1 table lookup by PRMT, one bf16x2
//                 multiply by the block scale) feeding m16n8k16 MMAs; the two
//                 halves add their fp32 results in shared memory at unit end;
//   warps 18..21  epilogue: piece counting, h, output;
//   warp 22       activation rows: x (FC1) or h (FC2) of the group's routes
//                 per stage, by cp.async.
//
// The dense W4A16 linear layer (one weight matrix, top-1, no activation) runs
// the FC1 phase alone: the last piece of a tile writes out directly.
//
// Why warp-level MMAs and not tcgen05 here: the register dequantiser feeds
// m16n8k16 fragments directly, while a tcgen05.mma reads its weight operand
// from shared or tensor memory, so every dequantised weight would make a
// round trip there first; with at most 32 routes per group the MMA work is
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

#include "decode_stage.cuh"
#include "dequant.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

cudaError_t ensure_smem_limit(const void* func, size_t bytes);

namespace dg {

namespace cg = cooperative_groups;

constexpr int kWarps = 23;
constexpr int kThreads = 32 * kWarps;
constexpr int kCompute = 16;          // compute warps
constexpr int kEpiWarps = 4;
constexpr int kWarpW = 0, kWarpSched = 1, kWarpC0 = 2, kWarpE0 = 18, kWarpAct = 22;
constexpr int kDesc = 8;              // unit descriptor ring
constexpr int kActRow = 144;          // activation row stride (bytes): 128 + 16 keeps LDS.128 conflict-free
constexpr int kReady = 1 << 20;       // added to an FC1 tile's piece count once its h is stored
constexpr float kTwo63 = 9.223372036854775808e18f;

template <int SETS>
struct Cfg {
  static constexpr int kRows = 8 * SETS;              // routes per group
  static constexpr int kSlots = SETS == 1 ? 12 : 8;   // ring slots of two stages
  static constexpr int kActSlot = 2 * kRows * kActRow;
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
  static constexpr size_t scales = codes + (size_t)C::kSlots * 2 * kCodeBytesPerStage;
  static constexpr size_t act = scales + (size_t)C::kSlots * 2 * kSS;
  static constexpr size_t xchg = round_up((int)(act + (size_t)C::kSlots * C::kActSlot), 16);
  static constexpr size_t bars = xchg + (size_t)8 * SETS * 4 * 32 * 4;
  static constexpr int kNumBars = 3 * C::kSlots + 3 * kDesc + 2;
  static constexpr size_t desc = bars + 8 * kNumBars;
  static constexpr size_t misc = desc + sizeof(GDesc) * kDesc;  // abort, grid word, phases, tasks
  static constexpr size_t tables = misc + 16 + 2 * sizeof(Phase) + 4 * 64;
  // tables: routes[R] i16, rgroup[R] i16, gexp[R] i16, gfirst[R] i16, gcnt[R] i16,
  // tvalid[m] i16 (m <= R), Cg[R + 1] u32
  static size_t total(int R) { return tables + (size_t)R * 2 * 6 + (size_t)(R + 1) * 4 + 16; }
};

__device__ __forceinline__ int local_expert(const DecodeParams& p, int route) {
  if (!p.topk_ids) return 0;  // dense linear layer: one expert, every route valid
  const int id = __ldg(p.topk_ids + route);
  if (id < 0 || id >= p.num_global_experts) return -1;
  const int l = p.expert_map ? __ldg(p.expert_map + id) : id;
  return (l >= 0 && l < p.num_local_experts) ? l : -1;
}

__device__ __forceinline__ unsigned long long ceil_div_u64(unsigned long long a, unsigned long long b) {
  return (a + b - 1) / b;
}

// CTA owning cost position P: max{b : floor(b*T/G) <= P}.
__device__ __forceinline__ int owner(const Phase& ph, unsigned long long P) {
  return (int)(((P + 1) * (unsigned long long)ph.G - 1) / ph.T);
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
  }
}

__device__ __forceinline__ int atom_add_acq_rel(int* addr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release(int* addr, int v) {
  asm volatile("red.add.release.gpu.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* addr) {
  int v;
  asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_relaxed(const int* addr) {
  int v;
  asm volatile("ld.relaxed.gpu.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Hint: bring `bytes` of global memory into L2 (no destination, no completion).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Walks one CTA's units of one phase, in order.
struct UnitIter {
  Phase ph;
  int phase, NG, w0;
  const uint32_t* Cg;     // cost prefix of the groups (per stage)
  unsigned long long pos, hi;
  int g;

  __device__ void init(const Phase& phs, int phase_, int NG_, int w0_, const uint32_t* Cg_) {
    ph = phs;
    phase = phase_;
    NG = NG_;
    w0 = w0_;
    Cg = Cg_;
    g = NG;
    pos = hi = 0;
    if (ph.T == 0 || (int)blockIdx.x >= ph.G) return;
    const unsigned long long b = blockIdx.x;
    pos = b * ph.T / (unsigned long long)ph.G;
    hi = (b + 1) * ph.T / (unsigned long long)ph.G;
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
    const unsigned long long ntks = (unsigned long long)ph.NT * ph.KS;
    const unsigned long long total = ntks;
    while (pos < hi && g < NG) {
      const unsigned long long base = (unsigned long long)Cg[g] * ntks;
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
      const int t = (int)(sidx / ph.KS);
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
  const unsigned long long a = ph.T / (unsigned long long)maxw;
  const unsigned long long c = ph.T / ceil_div_u64((unsigned long long)KS * maxw, (unsigned long long)(pmax - 1));
  if (a < G) G = a;
  if (c < G) G = c;
  ph.G = G < 1 ? 1 : (int)G;
  return ph;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// ------------------------------------------------------------------ kernel
template <int FMT, int SETS>
__global__ void __launch_bounds__(kThreads, 1) decode_grouped_kernel(const __grid_constant__ DecodeParams p) {
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
  uint64_t* ddone = dfull + kDesc;         // compute warps stored the unit's partials (16)
  uint64_t* dempty = ddone + kDesc;        // epilogue finished the unit (1)
  uint64_t* setup_bar = dempty + kDesc;    // group table ready (1)
  uint64_t* grid_bar = setup_bar + 1;      // every CTA's counters zeroed (1)
  GDesc* s_desc = reinterpret_cast<GDesc*>(smem + L::desc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::misc);
  uint32_t* s_grid_old = reinterpret_cast<uint32_t*>(smem + L::misc + 4);
  int* s_misc = reinterpret_cast<int*>(smem + L::misc + 8);  // [0] NG, [1] last flag
  Phase* s_ph = reinterpret_cast<Phase*>(smem + L::misc + 16);
  int* s_tasks = reinterpret_cast<int*>(smem + L::misc + 16 + 2 * sizeof(Phase));  // [64]
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
    *s_abort = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full_w[i], 1);
      mbar_init(&full_a[i], 32);
      mbar_init(&empty_s[i], kCompute);
    }
    for (int i = 0; i < kDesc; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&ddone[i], kCompute);
      mbar_init(&dempty[i], 1);
    }
    mbar_init(setup_bar, 1);
    mbar_init(grid_bar, 1);
    fence_mbar_init();
  }

  // Before the grid barrier: zero the completion counters, clear the status
  // word, and zero the output rows of tokens without a valid route (no unit
  // writes them).
  {
    const size_t gt = (size_t)blockIdx.x * kThreads + threadIdx.x, gs = (size_t)gridDim.x * kThreads;
    for (size_t i = gt; i < p.n_counters; i += gs) p.hcount[i] = 0;
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

  if (warp == kWarpSched) {
    // ------------------------------------------------ grid arrival, group table
    if (lane == 0) *s_grid_old = grid_arrive(&cg::details::get_grid_workspace()->barrier);
    const int E = p.num_local_experts;
    for (int e = lane; e < E; e += 32) s_ecnt[e] = 0;
    __syncwarp();
    for (int r = lane; r < R; r += 32) {
      const int l = local_expert(p, r);
      s_rgroup[r] = (int16_t)l;
      if (l >= 0) atomicAdd(&s_ecnt[l], 1);
    }
    __syncwarp();
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
      s_ph[1] = make_phase(NG && p.n_tiles2 ? run : 0, p.n_tiles2 > 0 ? p.n_tiles2 : 1, p.k_stages2 > 0 ? p.k_stages2 : 1,
                           maxw, p.pmax);
      mbar_arrive(setup_bar);
    }
    __syncwarp();

    // --------------------------------------------------- unit descriptors
    if (lane == 0) {
      UnitIter it;
      it.init(s_ph[0], 1, NG, p.w0, s_Cg);
      uint32_t d = 0;
      bool ok = true;
      GDesc u;
      // the first descriptors go out before the L2 prefetch of FC2 weights
      while (d < (uint32_t)kDesc && it.next(u)) {
        s_desc[d] = u;
        mbar_arrive(&dfull[d]);
        ++d;
      }
      const bool fc1_left = d == (uint32_t)kDesc;
      {
        UnitIter pf;
        pf.init(s_ph[1], 2, NG, p.w0, s_Cg);
        long long budget = p.l2_prefetch_bytes;
        GDesc v;
        while (budget > 0 && pf.next(v)) {
          const size_t tile_id = (size_t)s_gexp[v.g] * p.n_tiles2 + v.tile;
          for (int s0 = v.s_lo; s0 < v.s_hi; s0 += 8) {  // at most 8 stages (32 KB of codes) per prefetch
            const int ns = min(8, v.s_hi - s0);
            prefetch_l2(p.w2_codes + (tile_id * p.k_stages2 + s0) * kCodeBytesPerStage, ns * kCodeBytesPerStage);
            prefetch_l2(p.w2_scales + (tile_id * p.k_stages2 + s0) * kSS, ns * kSS);
          }
          budget -= (long long)(v.s_hi - v.s_lo) * kCodeBytesPerStage;
        }
      }
      auto publish = [&](const GDesc& v) {
        const uint32_t slot = d % kDesc;
        if (!mbar_wait(&dempty[slot], ((d / kDesc) & 1) ^ 1, ab, 51)) return false;
        s_desc[slot] = v;
        mbar_arrive(&dfull[slot]);
        ++d;
        return true;
      };
      if (fc1_left)
        while (ok && it.next(u)) ok = publish(u);
      it.init(s_ph[1], 2, NG, p.w0, s_Cg);
      while (ok && it.next(u)) ok = publish(u);
      if (ok) {
        u.phase = 0;
        publish(u);
      }
    }
    __syncwarp();
    return;
  }

  if (warp == kWarpW) {
    // ------------------------------------------------------ weight stream
    if (lane == 0 && mbar_wait(setup_bar, 0, ab, 52)) {
      uint32_t ws = 0;
      for (uint32_t d = 0; !ab.raised(); ++d) {
        const uint32_t slot_d = d % kDesc;
        if (!mbar_wait(&dfull[slot_d], (d / kDesc) & 1, ab, 53)) break;
        const GDesc u = s_desc[slot_d];
        if (u.phase == 0) break;
        const bool fc2 = u.phase == 2;
        const int nt = fc2 ? p.n_tiles2 : p.n_tiles1, ks = fc2 ? p.k_stages2 : p.k_stages1;
        const size_t tile_id = (size_t)s_gexp[u.g] * nt + u.tile;
        const uint8_t* gc = (fc2 ? p.w2_codes : p.w1_codes) + tile_id * ks * kCodeBytesPerStage;
        const uint8_t* gsc = (fc2 ? p.w2_scales : p.w1_scales) + tile_id * ks * kSS;
        bool ok = true;
        for (int s = u.s_lo; s < u.s_hi; s += 2, ++ws) {
          const uint32_t slot = ws % NS;
          if (!mbar_wait(&empty_s[slot], ((ws / NS) & 1) ^ 1, ab, 54)) {
            ok = false;
            break;
          }
          const int n = min(2, u.s_hi - s);
          mbar_arrive_expect_tx(&full_w[slot], n * (kCodeBytesPerStage + kSS));
          bulk_g2s(s_codes + slot * 2 * kCodeBytesPerStage, gc + (size_t)s * kCodeBytesPerStage,
                   n * kCodeBytesPerStage, &full_w[slot]);
          bulk_g2s(s_scales + slot * 2 * kSS, gsc + (size_t)s * kSS, n * kSS, &full_w[slot]);
        }
        if (!ok) break;
      }
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
    bool synced = false;
    uint32_t ws = 0;
    if (__all_sync(0xffffffffu, mbar_wait(setup_bar, 0, ab, 55))) {
      for (uint32_t d = 0; !ab.raised(); ++d) {
        const uint32_t slot_d = d % kDesc;
        if (!__all_sync(0xffffffffu, mbar_wait(&dfull[slot_d], (d / kDesc) & 1, ab, 56))) break;
        const GDesc u = s_desc[slot_d];
        if (u.phase == 0) break;
        const bool fc2 = u.phase == 2;
        const int c = s_gcnt[u.g], first = s_gfirst[u.g];
        if (fc2 && !synced) {
          if (!__all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 57))) break;
          synced = true;
        }
        bool ok = true;
        for (int s = u.s_lo; s < u.s_hi; s += 2, ++ws) {
          const uint32_t slot = ws % NS;
          if (!__all_sync(0xffffffffu, mbar_wait(&empty_s[slot], ((ws / NS) & 1) ^ 1, ab, 58))) {
            ok = false;
            break;
          }
          const int n = min(2, u.s_hi - s);
          if (fc2) {
            // the FC1 tiles holding these h columns must be ready
            if (lane < n) {
              const int st = s + lane;
              const int t1 = p.act == 0 ? st : st >> 1;
              const int* flag = p.hcount + (size_t)u.g * p.n_tiles1 + t1;
              const unsigned long long t0 = globaltimer();
              while (ld_acquire(flag) < kReady) {
                if (ab.raised() || globaltimer() - t0 > kWaitLimitNs) {
                  if (!ab.raised()) ab.raise(59);
                  break;
                }
                __nanosleep(32);
              }
            }
            __syncwarp();
            if (ab.raised()) {
              ok = false;
              cp_async_arrive(&full_a[slot]);
              break;
            }
          }
          uint8_t* dst0 = s_act + slot * C::kActSlot;
          const int chunks = n * c * 8;
          for (int ci = lane; ci < chunks; ci += 32) {
            const int st = ci / (c * 8), rem = ci - st * c * 8;
            const int i = rem >> 3, ch = rem & 7;
            const int r = s_routes[first + i];
            const int k = (s + st) * kBK + ch * 8;
            const uint32_t dst = smem_u32(dst0 + (st * C::kRows + i) * kActRow + ch * 16);
            if (fc2) {
              cp_async16(dst, p.h + (size_t)r * p.inter_pad + k, 16);
            } else {
              const int valid = (p.hidden - k) * 2;
              const uint32_t bytes = valid >= 16 ? 16u : (valid > 0 ? (uint32_t)valid : 0u);
              cp_async16(dst, bytes ? p.x + (size_t)(r / p.top_k) * p.hidden + k : p.x, bytes);
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

  if (warp >= kWarpE0 && warp < kWarpE0 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 32 * kWarpE0;  // 0..127
    volatile int* s_last = s_misc + 1;
    volatile int* s_ntask = s_misc + 2;
    const bool oks = __all_sync(0xffffffffu, mbar_wait(setup_bar, 0, ab, 60));
    if (named_bar_or(2, 32 * kEpiWarps, !oks)) return;
    if (warp == kWarpE0 && lane == 0) {
      if (grid_wait(&cg::details::get_grid_workspace()->barrier, *s_grid_old, ab)) mbar_arrive(grid_bar);
    }
    const bool okg = __all_sync(0xffffffffu, mbar_wait(grid_bar, 0, ab, 61));
    if (named_bar_or(2, 32 * kEpiWarps, !okg)) return;
    const int wnat = fc1_natural_width(p.act == 0 ? 0 : 1, p.inter_pad);
    for (uint32_t d = 0;; ++d) {
      // every wait's outcome is agreed on by all four warps before any
      // named barrier, so they always leave the loop together
      const uint32_t slot_d = d % kDesc;
      const bool okf = __all_sync(0xffffffffu, mbar_wait(&dfull[slot_d], (d / kDesc) & 1, ab, 62));
      if (named_bar_or(2, 32 * kEpiWarps, !okf)) break;
      const GDesc u = s_desc[slot_d];
      if (u.phase == 0) break;
      const bool okd = __all_sync(0xffffffffu, mbar_wait(&ddone[slot_d], (d / kDesc) & 1, ab, 63));
      if (named_bar_or(2, 32 * kEpiWarps, !okd)) break;
      const int c = s_gcnt[u.g], first = s_gfirst[u.g];
      if (u.phase == 1) {
        int* cnt = p.hcount + (size_t)u.g * p.n_tiles1 + u.tile;
        if (et == 0) *s_last = atom_add_acq_rel(cnt, 1) == u.npieces - 1;
        named_bar_sync(2, 32 * kEpiWarps);
        if (*s_last) {
          // the tile's pieces are all stored: sum them (piece order) into h
          const int rows = p.act == 0 ? 64 : kTileRows;
          const int row0 = u.tile * rows;
          const int lim = p.act == 2 ? p.n_out : p.inter_pad;
          for (int it = et; it < c * rows; it += 32 * kEpiWarps) {
            const int i = it / rows, row = row0 + (it - i * rows);
            if (row >= lim) continue;
            const int r = s_routes[first + i];
            const float* pa = p.p + ((size_t)r * wnat + row) * p.p_stride;
            float a = 0.f, b = 0.f;
            for (int k = 0; k < u.npieces; ++k) a += __ldcg(pa + k);
            if (p.act == 0) {
              const float* pb = pa + (size_t)p.inter_pad * p.p_stride;
              for (int k = 0; k < u.npieces; ++k) b += __ldcg(pb + k);
            }
            if (p.act == 2) {
              p.out[(size_t)r * p.n_out + row] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
            } else {
              const float hv = p.act == 0 ? silu_f(a) * b : (a > 0.f ? a * a : 0.f);
              p.h[(size_t)r * p.inter_pad + row] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
          named_bar_sync(2, 32 * kEpiWarps);
          if (et == 0 && p.act != 2) red_add_release(cnt, kReady);
        }
      } else {
        int* pc = p.pcount + (size_t)u.g * p.n_tiles2 + u.tile;
        if (et == 0) *s_last = atom_add_acq_rel(pc, 1) == u.npieces - 1;
        named_bar_sync(2, 32 * kEpiWarps);
        if (*s_last) {
          // every piece of this tile is in: count the routes' tokens; the
          // token's last route sums its output columns
          if (warp == kWarpE0) {
            bool last = false;
            int token = 0;
            if (lane < c) {
              const int r = s_routes[first + lane];
              token = r / p.top_k;
              last = atom_add_acq_rel(p.ocount + (size_t)token * p.n_tiles2 + u.tile, 1) == s_tvalid[token] - 1;
            }
            const unsigned m = __ballot_sync(0xffffffffu, last);
            if (last) s_tasks[__popc(m & ((1u << lane) - 1u))] = token;
            if (lane == 0) *s_ntask = __popc(m);
          }
          named_bar_sync(2, 32 * kEpiWarps);
          const int ntask = *s_ntask;
          const int n = u.tile * kTileRows + et;
          for (int ti = 0; ti < ntask; ++ti) {
            const int token = s_tasks[ti];
            if (n < p.hidden) {
              float acc = 0.f;
              for (int j = 0; j < p.top_k; ++j) {
                const int r = token * p.top_k + j;
                const int gj = s_rgroup[r];
                if (gj < 0) continue;
                const int np = ld_relaxed(p.pcount + (size_t)gj * p.n_tiles2 + u.tile);
                for (int k = 0; k < np; ++k) acc += __ldcg(p.q + ((size_t)k * R + r) * p.hidden + n);
              }
              p.out[(size_t)token * p.hidden + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
            }
          }
        }
      }
      named_bar_sync(2, 32 * kEpiWarps);
      if (et == 0) mbar_arrive(&dempty[slot_d]);
    }
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
  if (named_bar_or(1, 32 * kCompute, !oks)) return;
  uint32_t ws = 0;
  for (uint32_t d = 0;; ++d) {
    const uint32_t slot_d = d % kDesc;
    const bool okf = __all_sync(0xffffffffu, mbar_wait(&dfull[slot_d], (d / kDesc) & 1, ab, 65));
    if (named_bar_or(1, 32 * kCompute, !okf)) break;
    const GDesc u = s_desc[slot_d];
    if (u.phase == 0) break;
    const bool fc2 = u.phase == 2;
    const int c = s_gcnt[u.g], first = s_gfirst[u.g];
    const int sets = (c + 7) >> 3;
    float acc[SETS][2][4];
#pragma unroll
    for (int q = 0; q < SETS; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[q][0][i] = acc[q][1][i] = 0.f;
    // activation row of each column set for this thread (route 8q + g, or the
    // group's last route where the set is not full: its columns are unused)
    uint32_t arow[SETS];
#pragma unroll
    for (int q = 0; q < SETS; ++q) arow[q] = (uint32_t)min(8 * q + g, c - 1) * kActRow + t * 32;
    bool ok = true;
    for (int s = u.s_lo; s < u.s_hi; s += 2, ++ws) {
      const uint32_t slot = ws % NS;
      const uint32_t par = (ws / NS) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&full_w[slot], par, ab, 66) && mbar_wait(&full_a[slot], par, ab, 67))) {
        ok = false;
        break;
      }
      if (s + half < u.s_hi) {
        const uint8_t* cs = s_codes + (slot * 2 + half) * kCodeBytesPerStage + code_off;
        const uint8_t* ss = s_scales + (slot * 2 + half) * kSS + sc_off;
        const uint2 c0 = *reinterpret_cast<const uint2*>(cs);
        const uint2 c1 = *reinterpret_cast<const uint2*>(cs + 8 * 16);
        const uint32_t sa = d_scale<FMT>(ss[0]), sb = d_scale<FMT>(ss[8 * SB]);
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
        const uint8_t* xs = s_act + slot * C::kActSlot + half * C::kRows * kActRow;
#pragma unroll
        for (int q = 0; q < SETS; ++q) {
          if (q < sets) {
            const uint4 xa = *reinterpret_cast<const uint4*>(xs + arow[q]);
            const uint4 xb = *reinterpret_cast<const uint4*>(xs + arow[q] + 16);
            mma_16816(acc[q][0], a0[0], a1[0], a0[1], a1[1], xa.x, xa.y);
            mma_16816(acc[q][1], a0[2], a1[2], a0[3], a1[3], xa.z, xa.w);
            mma_16816(acc[q][0], a0[4], a1[4], a0[5], a1[5], xb.x, xb.y);
            mma_16816(acc[q][1], a0[6], a1[6], a0[7], a1[7], xb.z, xb.w);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_s[slot]);
    }
    if (named_bar_or(1, 32 * kCompute, !ok)) break;
    // the two halves' sums meet in shared memory; half 0 stores the partials
    float* xw = s_xchg + (size_t)rw * SETS * 4 * 32 + lane;
    if (half == 1) {
#pragma unroll
      for (int q = 0; q < SETS; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (q < sets) xw[(q * 4 + i) * 32] = acc[q][0][i] + acc[q][1][i];
    }
    named_bar_sync(1, 32 * kCompute);
    if (half == 0) {
      const int e = s_gexp[u.g];
      const float gsv = ((fc2 ? p.gs2 : p.gs1) ? __ldg((fc2 ? p.gs2 : p.gs1) + e) : 1.0f) * kTwo63;
#pragma unroll
      for (int q = 0; q < SETS; ++q) {
        if (q >= sets) continue;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = acc[q][0][i] + acc[q][1][i] + xw[(q * 4 + i) * 32];
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
    named_bar_sync(1, 32 * kCompute);  // the exchange buffer is free again
    __syncwarp();
    if (lane == 0) mbar_arrive(&ddone[slot_d]);
  }
}

}  // namespace dg

size_t decode_grouped_smem(int fmt, int sets, int routes) {
  if (fmt == 0) return sets == 1 ? dg::Smem<0, 1>::total(routes) : dg::Smem<0, 4>::total(routes);
  return sets == 1 ? dg::Smem<1, 1>::total(routes) : dg::Smem<1, 4>::total(routes);
}

template <int FMT, int SETS>
static cudaError_t launch_dg(const DecodeParams& p, int grid, cudaStream_t stream) {
  auto kern = dg::decode_grouped_kernel<FMT, SETS>;
  const size_t smem = dg::Smem<FMT, SETS>::total(p.m * p.top_k);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(dg::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Resident CTAs per SM of the kernel with `smem` bytes (the cooperative launch
// takes one CTA per SM, which must fit).
cudaError_t decode_grouped_occupancy(int fmt, int sets, size_t smem, int* blocks_per_sm) {
  const void* k = fmt == 0 ? (sets == 1 ? reinterpret_cast<const void*>(dg::decode_grouped_kernel<0, 1>)
                                        : reinterpret_cast<const void*>(dg::decode_grouped_kernel<0, 4>))
                           : (sets == 1 ? reinterpret_cast<const void*>(dg::decode_grouped_kernel<1, 1>)
                                        : reinterpret_cast<const void*>(dg::decode_grouped_kernel<1, 4>));
  cudaError_t e = ensure_smem_limit(k, smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, dg::kThreads, smem);
}

cudaError_t launch_decode_grouped(const DecodeParams& p, int fmt, int sets, int grid, cudaStream_t stream) {
  if (fmt == 0) return sets == 1 ? launch_dg<0, 1>(p, grid, stream) : launch_dg<0, 4>(p, grid, stream);
  return sets == 1 ? launch_dg<1, 1>(p, grid, stream) : launch_dg<1, 4>(p, grid, stream);
}

}  // namespace b4
