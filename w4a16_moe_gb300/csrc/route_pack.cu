// Route packing: top-k expert ids -> per-expert contiguous route lists.
//
// flashinfer PR #4255, Description ("Shape-stable route packing ... specialize
// on a power-of-two capacity instead of the exact token count") and Tests
// ("covering expert_map, invalid expert ids, preallocated buffers, and the
// workspace capacity contract").
//
// One CTA of 1024 threads performs a stable counting sort with no global
// atomics and no allocation, so the result is bit-exact and the launch is
// capture-safe:
//   pass 1  each warp walks its contiguous segment of routes 32 at a time;
//           lanes with the same local expert are grouped (one ballot per key
//           bit) and the group leader adds the group size to the warp's
//           histogram row;
//   pass 2  per expert, an exclusive scan over the 32 warp rows gives each
//           warp its base, and a warp-shuffle scan over experts gives offsets;
//   pass 3  the segments are walked again; a route lands at
//           offsets[l] + warp base + running count + rank among equal lanes.
// Routes of one expert therefore keep ascending flat index r = t*top_k + j.
// The same kernel also emits the grouped-GEMM schedule: each expert's routes
// cut into chunks of at most `chunk_rows`.

#include "kernels.cuh"
#include "ptx.cuh"

namespace b4 {

constexpr int kPackThreads = 1024;
constexpr int kPackWarps = kPackThreads / 32;
constexpr int kKeys = 16;  // 32-route batches whose keys a warp loads together

__device__ __forceinline__ int pack_local_expert(const RoutePackParams& p, int r) {
  const int id = p.topk_ids[r];
  if (id < 0 || id >= p.num_global_experts) return -1;
  const int l = p.expert_map ? p.expert_map[id] : id;
  return (l >= 0 && l < p.num_local_experts) ? l : -1;
}

// Lanes of the warp holding the same key as this lane (keys in [-1, 2^nbits)),
// from one ballot per key bit plus one for validity: the result equals
// __match_any_sync, which issues far slower on this GPU.
__device__ __forceinline__ unsigned key_peers(int key, int nbits) {
  const unsigned valid = __ballot_sync(0xffffffffu, key >= 0);
  unsigned m = key >= 0 ? valid : ~valid;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = key >= 0 && ((key >> b) & 1);
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bb : ~bb;
  }
  return m;
}

// Exclusive block-wide scan of one value per thread (1024 threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += y;
    }
    s_warp[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  total = s_warp[32];
  const int out = incl - v + s_warp[warp];
  __syncthreads();
  return out;
}

__global__ void __launch_bounds__(kPackThreads, 1) route_pack_kernel(const __grid_constant__ RoutePackParams p) {
  extern __shared__ int s_hist[];  // [32][E_l], then [E_l] offsets
  __shared__ int s_warp[33];
  __shared__ int s_valid;
  const int E = p.num_local_experts;
  int* s_off = s_hist + kPackWarps * E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.m * p.top_k;
  const int seg = round_up(cdiv(R, kPackWarps), 32);
  const int beg = warp * seg;
  const int end = min(R, beg + seg);
  const unsigned lt_mask = (1u << lane) - 1u;
  int nbits = 0;
  while ((1 << nbits) < E) ++nbits;

  if (threadIdx.x == 0 && p.status) {
    p.status[0] = 0;
    p.status[1] = 0;
  }
  for (int i = threadIdx.x; i < kPackWarps * E; i += kPackThreads) s_hist[i] = 0;
  __syncthreads();

  // pass 1: per-warp histograms.  Keys of kKeys batches are loaded before
  // any is used, so the id and expert_map loads of a warp overlap.
  int* my_hist = s_hist + warp * E;
  for (int b0 = beg; b0 < end; b0 += 32 * kKeys) {
    int keys[kKeys];
#pragma unroll
    for (int i = 0; i < kKeys; ++i) {
      const int r = b0 + 32 * i + lane;
      keys[i] = r < end ? pack_local_expert(p, r) : -1;
    }
#pragma unroll
    for (int i = 0; i < kKeys; ++i) {
      if (b0 + 32 * i >= end) break;
      const int key = keys[i];
      const unsigned peers = key_peers(key, nbits);
      if (key >= 0 && lane == __ffs(peers) - 1) my_hist[key] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // pass 2: warp bases per expert, expert counts, offsets, chunk schedule
  for (int e0 = 0; e0 < E; e0 += kPackThreads) {
    // E <= 1024 is enforced by the host, so one iteration
    const int e = e0 + threadIdx.x;
    int cnt = 0;
    if (e < E) {
      for (int w = 0; w < kPackWarps; ++w) {
        const int c = s_hist[w * E + e];
        s_hist[w * E + e] = cnt;
        cnt += c;
      }
    }
    int total = 0;
    const int off = block_exclusive_scan(cnt, s_warp, total);
    if (e < E) {
      s_off[e] = off;
      p.counts[e] = cnt;
      p.offsets[e] = off;
    }
    if (threadIdx.x == 0) {
      p.offsets[E] = total;
      s_valid = total;
    }
    if (p.chunks) {
      const int nch = e < E ? cdiv(cnt, p.chunk_rows) : 0;
      int tot_ch = 0;
      const int ch0 = block_exclusive_scan(nch, s_warp, tot_ch);
      for (int c = 0; c < nch; ++c) {
        const int rows = min(p.chunk_rows, cnt - c * p.chunk_rows);
        p.chunks[ch0 + c] = make_int4(e, off + c * p.chunk_rows, rows, 0);
      }
      if (threadIdx.x == 0) *p.chunk_count = tot_ch;
    }
  }
  __syncthreads();

  // pass 3: scatter
  for (int b0 = beg; b0 < end; b0 += 32 * kKeys) {
    int keys[kKeys];
#pragma unroll
    for (int i = 0; i < kKeys; ++i) {
      const int r = b0 + 32 * i + lane;
      keys[i] = r < end ? pack_local_expert(p, r) : -1;
    }
#pragma unroll
    for (int i = 0; i < kKeys; ++i) {
      if (b0 + 32 * i >= end) break;
      const int r = b0 + 32 * i + lane;
      const int key = keys[i];
      const unsigned peers = key_peers(key, nbits);
      if (key >= 0) {
        const int pos = s_off[key] + my_hist[key] + __popc(peers & lt_mask);
        p.sorted_routes[pos] = r;
      }
      __syncwarp();
      if (key >= 0 && lane == __ffs(peers) - 1) my_hist[key] += __popc(peers);
      __syncwarp();
    }
  }
  // tail of the capacity: -1
  const int valid = s_valid;
  for (int i = valid + threadIdx.x; i < p.route_cap; i += kPackThreads) p.sorted_routes[i] = -1;
}

size_t route_pack_smem_bytes(int num_local_experts) {
  return (size_t)(kPackWarps + 1) * num_local_experts * sizeof(int);
}

cudaError_t launch_route_pack(const RoutePackParams& p, cudaStream_t stream) {
  const size_t smem = route_pack_smem_bytes(p.num_local_experts);
  static size_t configured = 0;
  if (smem > 48 * 1024 && smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(route_pack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  route_pack_kernel<<<1, kPackThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace b4
