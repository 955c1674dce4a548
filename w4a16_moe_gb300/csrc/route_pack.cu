// Route packing: top-k expert ids -> per-expert contiguous route lists.
//
// flashinfer PR #4255, Description ("Shape-stable route packing ... specialize
// on a power-of-two capacity instead of the exact token count") and Tests
// ("covering expert_map, invalid expert ids, preallocated buffers, and the
// workspace capacity contract").
//
// A stable counting sort without global atomics, so the result is bit-exact
// and the launch is capture-safe.  Every CTA (512 threads) builds the full
// histogram of local experts in shared memory, one row per warp over the
// warp's contiguous segment of routes (the ids of eight 32-route groups are
// loaded before any is used), and scans it into expert offsets and, per
// expert, each warp's base (the same numbers in every CTA).  CTA b then owns
// experts b, b + G, ...: each warp walks its segment again and a route of the
// expert lands at offsets[l] + warp base + running count + its rank in the
// group's ballot, so routes keep ascending flat index r = t*top_k + j.
// CTA 0 also writes counts, offsets, the grouped-GEMM chunk schedule (each
// expert's routes cut into chunks of at most `chunk_rows`), the -1 tail of
// the capacity and the cleared status word.  The ids are read a few times per
// CTA; they stay in L2.  For the grouped path each CTA then copies the x rows
// of its experts' routes into packed-route order (the FC1 B operand): it
// knows those slots already, so no other launch or grid-wide wait is needed.
// That launch has two CTAs per SM whatever the expert count: with fewer
// experts than CTAs, Q = G / E replicas take each expert, every one of them
// places the expert's routes (the same values into the same slots) and
// copies every Q-th of its rows.

#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

cudaError_t ensure_smem_limit(const void* func, size_t bytes);

// Optional copy of x rows into packed-route order (the grouped FC1's B
// operand): xp[slot] = x[token of the route at slot]; xp = null: none.
struct PackCopy {
  const uint16_t* x;
  uint16_t* xp;
  int hidden;
};

constexpr int kPackThreads = 512;
constexpr int kPackWarps = kPackThreads / 32;
constexpr int kBatch = 8;  // 32-route groups whose keys a warp loads before using any

// Local experts of the routes b0 + 32 i + lane (i < kBatch; -1 past `end` or
// invalid).  The id loads, then the expert_map loads, are issued as one batch
// each at clamped addresses, with the range checks applied afterwards: a
// per-route branch around each load keeps the loads from overlapping (the
// kernel then waits one L2 round trip per 32 routes).
__device__ __forceinline__ void load_keys(const RoutePackParams& p, int b0, int end, int lane, int (&keys)[kBatch]) {
  if (!p.topk_ids) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) keys[i] = b0 + 32 * i + lane < end ? 0 : -1;
    return;
  }
  int id[kBatch];
#pragma unroll
  for (int i = 0; i < kBatch; ++i) {
    const int r = b0 + 32 * i + lane;
    id[i] = __ldg(p.topk_ids + (r < end ? r : b0));  // b0 < end: a valid address
  }
#pragma unroll
  for (int i = 0; i < kBatch; ++i) {
    const bool ok = b0 + 32 * i + lane < end && id[i] >= 0 && id[i] < p.num_global_experts;
    id[i] = ok ? id[i] : -1;
  }
  if (p.expert_map) {
    int l[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) l[i] = __ldg(p.expert_map + (id[i] >= 0 ? id[i] : 0));
#pragma unroll
    for (int i = 0; i < kBatch; ++i) keys[i] = id[i] >= 0 && l[i] >= 0 && l[i] < p.num_local_experts ? l[i] : -1;
  } else {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) keys[i] = id[i] >= 0 && id[i] < p.num_local_experts ? id[i] : -1;
  }
}

// In-place exclusive scan of s[0..n) (n <= 2 * kPackThreads) by the block;
// returns the total.
__device__ __forceinline__ int block_scan(int* s, int n, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i0 = 2 * threadIdx.x;
  const int a = i0 < n ? s[i0] : 0, b = i0 + 1 < n ? s[i0 + 1] : 0;
  int incl = a + b;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < kPackWarps ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += y;
    }
    if (lane < kPackWarps) s_warp[lane] = wi - w;
    if (lane == 31) s_warp[kPackWarps] = wi;
  }
  __syncthreads();
  const int base = incl - (a + b) + s_warp[warp];
  if (i0 < n) s[i0] = base;
  if (i0 + 1 < n) s[i0 + 1] = base + a;
  const int total = s_warp[kPackWarps];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kPackThreads) route_pack_kernel(const __grid_constant__ RoutePackParams p,
                                                                 const __grid_constant__ PackCopy cp) {
  // The grouped FC1 (launched with programmatic dependent launch) may start
  // its set-up now; it waits for this grid to finish before it reads anything.
  pdl_launch_dependents();
  extern __shared__ int s_mem[];
  const int E = p.num_local_experts;
  int* s_whist = s_mem;                   // [warps][E]: counts, then each warp's base within the expert
  int* s_cnt = s_mem + kPackWarps * E;    // [E]: counts, then offsets; CTA 0 also [E] chunk starts, [E] scratch
  __shared__ int s_warp[kPackWarps + 1];
  const int R = p.m * p.top_k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  // each warp owns a contiguous segment of routes (the same in every pass)
  const int seg = round_up(cdiv(R, kPackWarps), 32);
  const int beg = warp * seg, end = min(R, beg + seg);

  // per-warp histograms of local experts
  for (int i = threadIdx.x; i < kPackWarps * E; i += kPackThreads) s_whist[i] = 0;
  __syncthreads();
  int* my_hist = s_whist + warp * E;
  for (int b0 = beg; b0 < end; b0 += 32 * kBatch) {
    int keys[kBatch];
    load_keys(p, b0, end, lane, keys);
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (keys[i] >= 0) atomicAdd(&my_hist[keys[i]], 1);
  }
  __syncthreads();
  // expert counts, and each warp's base among the expert's routes
  for (int e = threadIdx.x; e < E; e += kPackThreads) {
    int c = 0;
    for (int w = 0; w < kPackWarps; ++w) {
      const int h = s_whist[w * E + e];
      s_whist[w * E + e] = c;
      c += h;
    }
    s_cnt[e] = c;
  }
  __syncthreads();

  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += kPackThreads) p.counts[e] = s_cnt[e];
    if (p.chunks) {
      // chunk schedule: each expert's routes in chunks of <= chunk_rows, in
      // expert order (computed from the counts before they become offsets)
      int* s_nch = s_cnt + E;
      int* s_off = s_nch + E;
      for (int e = threadIdx.x; e < E; e += kPackThreads) {
        s_nch[e] = cdiv(s_cnt[e], p.chunk_rows);
        s_off[e] = s_cnt[e];
      }
      __syncthreads();
      const int tot_ch = block_scan(s_nch, E, s_warp);
      block_scan(s_off, E, s_warp);
      for (int e = threadIdx.x; e < E; e += kPackThreads) {
        const int cnt = s_cnt[e], off = s_off[e], ch0 = s_nch[e];
        for (int c = 0; c * p.chunk_rows < cnt; ++c)
          p.chunks[ch0 + c] = make_int4(e, off + c * p.chunk_rows, min(p.chunk_rows, cnt - c * p.chunk_rows), 0);
      }
      if (threadIdx.x == 0) *p.chunk_count = tot_ch;
      __syncthreads();
    }
    if (threadIdx.x == 0 && p.status) {
      p.status[0] = 0;
      p.status[1] = 0;
    }
  }
  const int valid = block_scan(s_cnt, E, s_warp);  // s_cnt now holds the offsets
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += kPackThreads) p.offsets[e] = s_cnt[e];
    if (threadIdx.x == 0) p.offsets[E] = valid;
    for (int i = valid + threadIdx.x; i < p.route_cap; i += kPackThreads) p.sorted_routes[i] = -1;
  }

  // this CTA's experts: b, b + G, ...; or, copying with fewer experts than
  // CTAs, expert b % E as replica b / E of Q (CTAs from Q * E on take none)
  int e0 = blockIdx.x, estep = gridDim.x, q = 0, Q = 1;
  if (cp.xp && (int)gridDim.x > E) {
    Q = (int)gridDim.x / E;
    q = (int)blockIdx.x / E;
    e0 = (int)blockIdx.x < Q * E ? (int)blockIdx.x % E : E;
    estep = E;
  }
  // the routes of this CTA's experts, in ascending flat index
  for (int e = e0; e < E; e += estep) {
    int pos = s_cnt[e] + my_hist[e];
    for (int b0 = beg; b0 < end; b0 += 32 * kBatch) {
      int keys[kBatch];
      load_keys(p, b0, end, lane, keys);
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const bool hit = keys[i] == e;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit) p.sorted_routes[pos + __popc(m & lt_mask)] = b0 + 32 * i + lane;
        pos += __popc(m);
      }
    }
  }
  if (!cp.xp) return;

  // xp[slot] = x[token of the route at slot] for this CTA's experts, one warp
  // per row, four 16-byte loads in flight per lane before their stores.  The
  // slots' routes were stored by this CTA: plain loads after the barrier.
  constexpr int kLoads = 4;
  __syncthreads();
  const int chunks = cp.hidden / 8;  // 16-byte pieces of a row
  for (int e = e0; e < E; e += estep) {
    const int off = s_cnt[e], cnt = (e + 1 < E ? s_cnt[e + 1] : valid) - off;
    for (int i = q * kPackWarps + warp; i < cnt; i += Q * kPackWarps) {
      const int tok = p.sorted_routes[off + i] / p.top_k;
      const uint4* src = reinterpret_cast<const uint4*>(cp.x + (size_t)tok * cp.hidden);
      uint4* dst = reinterpret_cast<uint4*>(cp.xp + (size_t)(off + i) * cp.hidden);
      for (int c = lane; c < chunks; c += 32 * kLoads) {
        uint4 v[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; ++k)
          if (c + 32 * k < chunks) v[k] = __ldg(src + c + 32 * k);
#pragma unroll
        for (int k = 0; k < kLoads; ++k)
          if (c + 32 * k < chunks) dst[c + 32 * k] = v[k];
      }
    }
  }
}

size_t route_pack_smem_bytes(int num_local_experts) {
  return (size_t)(kPackWarps + 3) * num_local_experts * sizeof(int);
}

cudaError_t launch_route_pack(const RoutePackParams& p, int num_sms, cudaStream_t stream, const uint16_t* x,
                              uint16_t* xp, int hidden) {
  const size_t smem = route_pack_smem_bytes(p.num_local_experts);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(route_pack_kernel), smem);
  if (e != cudaSuccess) return e;
  // one CTA per expert up to two per SM; copying x rows, always two per SM
  int grid = p.num_local_experts < 2 * num_sms && !xp ? p.num_local_experts : 2 * num_sms;
  if (grid < 1) grid = 1;
  route_pack_kernel<<<grid, kPackThreads, smem, stream>>>(p, PackCopy{x, xp, hidden});
  return cudaGetLastError();
}

}  // namespace b4
