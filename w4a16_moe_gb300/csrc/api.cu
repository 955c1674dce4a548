// extern "C" entry points of libb4moe (declared in include/b4moe.h):
// argument validation, workspace carve-up, path choice and kernel launches.
// Every launch goes to the caller's stream; nothing here allocates device
// memory or synchronises, except b4_prepare_weights and b4_check_status,
// which are documented as synchronous.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "b4moe.h"
#include "kernels.cuh"
#include "tma.cuh"

namespace b4 {
template <int MODE, int FMT>
cudaError_t launch_gemm(const GemmParams& p, int grid, bool pdl, cudaStream_t stream);
template <int MODE, int FMT>
cudaError_t launch_gemm_wn(const GemmParams& p, int grid, bool pdl, cudaStream_t stream);
cudaError_t launch_finalize(const FinalizeParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int fmt, int grid, cudaStream_t stream);
cudaError_t decode_occupancy(int fmt, bool grouped, int* blocks_per_sm);
cudaError_t launch_decode_grouped(const SmallGroupParams& p, int fmt, int sets, int grid, cudaStream_t stream);
cudaError_t decode_grouped_occupancy(int fmt, int sets, size_t smem, int* blocks_per_sm);
size_t decode_grouped_smem(int fmt, int sets, int routes);
// xp != null: the route pack also copies x rows into packed-route order
cudaError_t launch_route_pack(const RoutePackParams& p, int num_sms, cudaStream_t stream,
                              const uint16_t* x = nullptr, uint16_t* xp = nullptr, int hidden = 0);
size_t route_pack_smem_bytes(int num_local_experts);
cudaError_t launch_prepare(const PrepareParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_wait_self_test(uint32_t* status, unsigned long long limit_ns, cudaStream_t stream);
}  // namespace b4

using namespace b4;

namespace {

thread_local std::string g_last_error;
thread_local void* const* g_events = nullptr;  // b4_set_timing_events
thread_local int g_num_events = 0;
thread_local long long* g_trace = nullptr;     // b4_set_trace

// Records timing event i (if timing is on).
// Under stream capture a plain record only orders streams inside the graph;
// an external record becomes an event-record node that replays can time.
cudaError_t mark(int i, cudaStream_t s) {
  if (!g_events || i >= g_num_events) return cudaSuccess;
  cudaEvent_t ev = reinterpret_cast<cudaEvent_t>(g_events[i]);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

b4_status fail(b4_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

b4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(B4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Path choice.  flashinfer PR #4255 (Reviewer Notes) caps its decode path at
// m = 4 and notes that the crossover varies by card; on GB300 the small-m
// kernels were measured against the grouped tcgen05 GEMMs (K back-to-back
// calls, weights L2-cold): the small-m kernels beat the grouped GEMMs up to
// m = 16 (decode E128 k8 m = 16: 195 vs 289 us; small-batch E64 k6 m = 16:
// 91 vs 101 us), the grouped GEMMs win from m = 32 (small-batch m = 32).
// Inside the small-m path the per-route kernel streams about twice as fast as
// the route-grouped one (4.6 against 2.1 TB/s); one route per unit it re-reads
// an expert's weights for each route that selects it, which wins while there
// are fewer routes than local experts (small-batch m = 8, 48 routes on 64
// experts: 60 vs 66 us).  From m * top_k >= E_local its units take up to four
// routes of one expert (decode m = 16, 128 routes on 128 experts: 163 us
// grouped, 195 one route per unit, 271 route-grouped; m = 32, 256 routes: 266
// against 373 route-grouped and 382 for the grouped GEMMs; small-batch m = 16,
// 96 routes on 64 experts: 87 against 92 and 100).  At three routes per expert
// the route-grouped kernel wins again (small-batch m = 32: 139 against 145).
constexpr int kDecodeAutoMaxM = 16;  // AUTO takes a small-m kernel up to here
constexpr int kPerRouteMaxM = 4;     // the per-route kernel up to here, and while m top_k <= 2 E_local (grouped units)
// b4_linear (N = K = 4096, back-to-back calls): the per-route kernel reads W
// once per token at m = 1 and once per four tokens from m = 2 (grouped units;
// m = 1 / 2 / 3 / 4: 9.3 / 11.4 / 12.9 / 13.7 us), the route-grouped kernel once
// per 8 tokens (15.2 - 15.4 us for m = 3..4, 15.9 at m = 8, 20.0 at m = 16;
// the per-route kernel 18.7 / 27.2 there) against the K-split grouped GEMM
// (21.9 us at m = 8 and 16, on par from m = 32).
constexpr int kLinearSmallMaxM = 16;    // b4_linear's AUTO takes the small-m kernels up to here
constexpr int kLinearPerRouteMaxM = 4;  // b4_linear's small-m path: the per-route kernel up to here
constexpr int kDecodeW0 = 4;        // small-m partition: a stage costs kDecodeW0 + its route column sets
constexpr int kMaxSplits = 8;

int32_t next_pow2(int64_t n) {
  int64_t p = 1;
  while (p < n) p <<= 1;
  return (int32_t)p;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The kernels' FC1 activation of a b4_activation: 0 gated (SwiGLU and the
// clamped swiglu share the W13 layout and the kernels' gated epilogue), 1
// ReLU^2.
int kernel_act(int32_t activation) { return activation == B4_ACT_RELU2 ? 1 : 0; }

// Parameters of the gated epilogue: plain SwiGLU is alpha 1, beta 0, no clamp;
// the clamped swiglu takes the config's three values, checked here.
b4_status glu_params(const b4_moe_config* cfg, int32_t activation, GluParams* g) {
  if (activation != B4_ACT_SWIGLU_OAI) {
    *g = GluParams{1.0f, 0.0f, INFINITY};
    return B4_OK;
  }
  if (!std::isfinite(cfg->swiglu_alpha) || !std::isfinite(cfg->swiglu_beta) || !(cfg->swiglu_limit > 0.0f))
    return fail(B4_ERR_INVALID_ARGUMENT,
                "swiglu_alpha = %g and swiglu_beta = %g must be finite and swiglu_limit = %g positive",
                (double)cfg->swiglu_alpha, (double)cfg->swiglu_beta, (double)cfg->swiglu_limit);
  *g = GluParams{cfg->swiglu_alpha, cfg->swiglu_beta, cfg->swiglu_limit};
  return B4_OK;
}

// ------------------------------------------------------------ validation
b4_status check_config(const b4_moe_config* cfg, int32_t act) {
  if (!cfg) return fail(B4_ERR_INVALID_ARGUMENT, "cfg is NULL");
  if (cfg->m < 0) return fail(B4_ERR_INVALID_ARGUMENT, "m = %d < 0", cfg->m);
  if (cfg->m > (1 << 20)) return fail(B4_ERR_INVALID_ARGUMENT, "m = %d exceeds 2^20", cfg->m);
  if (cfg->top_k < 1 || cfg->top_k > 32) return fail(B4_ERR_INVALID_ARGUMENT, "top_k = %d not in [1, 32]", cfg->top_k);
  if (cfg->num_local_experts < 1 || cfg->num_local_experts > B4_MAX_LOCAL_EXPERTS)
    return fail(B4_ERR_INVALID_ARGUMENT, "num_local_experts = %d not in [1, %d]", cfg->num_local_experts,
                B4_MAX_LOCAL_EXPERTS);
  if (cfg->num_global_experts < 1 || cfg->num_global_experts > (1 << 20))
    return fail(B4_ERR_INVALID_ARGUMENT, "num_global_experts = %d out of range", cfg->num_global_experts);
  if (!cfg->expert_map && cfg->num_global_experts != cfg->num_local_experts)
    return fail(B4_ERR_INVALID_ARGUMENT, "without expert_map, num_global_experts must equal num_local_experts");
  if (cfg->format != B4_NVFP4_E4M3_K16 && cfg->format != B4_MXFP4_E8M0_K32)
    return fail(B4_ERR_INVALID_ARGUMENT, "format = %d unknown", cfg->format);
  if (cfg->path < B4_PATH_AUTO || cfg->path > B4_PATH_GROUPED)
    return fail(B4_ERR_INVALID_ARGUMENT, "path = %d unknown", cfg->path);
  if (act != B4_ACT_SILU_SWIGLU && act != B4_ACT_RELU2 && act != B4_ACT_SWIGLU_OAI)
    return fail(B4_ERR_INVALID_ARGUMENT, "activation = %d unknown", act);
  const int g = cfg->format == B4_NVFP4_E4M3_K16 ? 16 : 32;
  if (cfg->hidden < g || cfg->hidden % g || cfg->hidden > (1 << 16))
    return fail(B4_ERR_INVALID_ARGUMENT, "hidden = %d must be a positive multiple of %d (<= 65536)", cfg->hidden, g);
  if (cfg->inter < g || cfg->inter % g || cfg->inter > (1 << 16))
    return fail(B4_ERR_INVALID_ARGUMENT, "inter = %d must be a positive multiple of %d (<= 65536)", cfg->inter, g);
  if (cfg->path == B4_PATH_DECODE && cfg->m > B4_DECODE_MAX_M)
    return fail(B4_ERR_INVALID_ARGUMENT, "decode path takes m <= %d, got %d", B4_DECODE_MAX_M, cfg->m);
  return B4_OK;
}

// ------------------------------------------------------------- workspace
// Common pieces (status word, route pack, chunk schedule), then one region
// that the grouped path and the small-m path each lay out for themselves
// (a call runs one of them): its size is the larger of the two.  Every size
// depends on m only through T_cap, and monotonically.
struct WsLayout {
  size_t status, counts, offsets, sorted, chunks, chunk_count;
  size_t h, acc, xp;                     // grouped path
  size_t dp, dq, dh, dcnt;               // route-grouped small-m path
  size_t op, oq;                         // per-route decode path
  size_t total;
  int t_cap, r_cap, max_chunks, inter_pad, wnat;
  int dec_tcap, dec_rcap, dec_pmax;      // small-m path sizes (tokens capped at B4_DECODE_MAX_M)
  int dec_splits;                        // per-route decode path: most K splits
  bool decode_ok;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

WsLayout ws_layout(const b4_moe_config* cfg, int32_t act) {
  WsLayout L{};
  L.t_cap = next_pow2(cfg->m > 0 ? cfg->m : 1);
  L.r_cap = L.t_cap * cfg->top_k;
  L.max_chunks = L.r_cap / kChunkRowsN + cfg->num_local_experts + 1;  // the smaller chunk size
  L.inter_pad = round_up(cfg->inter, kBK);
  L.wnat = fc1_natural_width(kernel_act(act), L.inter_pad);
  L.decode_ok = L.t_cap <= B4_DECODE_MAX_M;
  L.dec_tcap = L.t_cap < B4_DECODE_MAX_M ? L.t_cap : B4_DECODE_MAX_M;
  L.dec_rcap = L.dec_tcap * cfg->top_k;
  // at most this many CTAs share one tile of the small-m partition: fewer at
  // larger capacity, so the partial buffers stay monotone and bounded
  L.dec_pmax = L.dec_rcap <= 64 ? 8 : 4;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.status = take(256);
  L.counts = take(sizeof(int32_t) * cfg->num_local_experts);
  L.offsets = take(sizeof(int32_t) * (cfg->num_local_experts + 1));
  L.sorted = take(sizeof(int32_t) * L.r_cap);
  L.chunks = take(sizeof(int4) * L.max_chunks);
  L.chunk_count = take(sizeof(int32_t));
  const size_t region = off;
  L.h = take(sizeof(uint16_t) * (size_t)L.r_cap * L.inter_pad);
  L.acc = take(sizeof(float) * (size_t)L.t_cap * cfg->hidden);
  L.xp = take(sizeof(uint16_t) * (size_t)L.r_cap * cfg->hidden);
  const size_t grouped_end = off;
  off = region;
  const int nt1 = cdiv(L.wnat, kTileRows) + 1;
  L.dp = take(sizeof(float) * (size_t)L.dec_rcap * L.wnat * L.dec_pmax);
  L.dq = take(sizeof(float) * (size_t)L.dec_pmax * L.dec_rcap * cfg->hidden);
  L.dh = take(sizeof(uint16_t) * (size_t)L.dec_rcap * L.inter_pad);
  L.dcnt = take(sizeof(int32_t) * (size_t)L.dec_rcap * nt1);
  const size_t small_end = off;
  // per-route decode path: K splits of about 256 units over the routes (a
  // unit covers at most 128 K stages, a grouped unit 32), FC1 partials with
  // the splits innermost padded to a power of two, FC2 partials per split
  off = region;
  int sp = 256 / L.dec_rcap;
  sp = sp < 1 ? 1 : (sp > kMaxSplits ? kMaxSplits : sp);
  const int kst = cdiv(cfg->hidden > L.inter_pad ? cfg->hidden : L.inter_pad, kBK);
  const int need = (kst * kDecodeGroupMax + kDecodeMaxStages - 1) / kDecodeMaxStages;  // grouped units' length cap
  L.dec_splits = sp > need ? sp : need;
  int p_splits = 1;
  while (p_splits < L.dec_splits) p_splits <<= 1;
  L.op = take(sizeof(float) * (size_t)p_splits * L.dec_rcap * L.wnat);
  L.oq = take(sizeof(float) * (size_t)L.dec_splits * L.dec_rcap * cfg->hidden);
  size_t end = off > grouped_end ? off : grouped_end;
  L.total = end > small_end ? end : small_end;
  return L;
}

// ---------------------------------------------------------------- device
struct DevInfo {
  bool ok = false;
  int sms = 0;
};

b4_status device_info(DevInfo& info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(B4_ERR_UNSUPPORTED_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  static std::mutex mu;
  static DevInfo cache[64];
  static bool known[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && known[dev]) {
    info = cache[dev];
  } else {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    info.ok = major == 10 && minor == 3;
    info.sms = sms;
    if (dev < 64) {
      cache[dev] = info;
      known[dev] = true;
    }
  }
  if (!info.ok) return fail(B4_ERR_UNSUPPORTED_DEVICE, "device is not sm_103 (GB300); no fallback path exists");
  return B4_OK;
}

// Decode schedule: K splits of FC1 and FC2 and the grid.  CTAs take their
// first unit statically and claim the rest in unit order, so load balance is
// dynamic; the splits aim at about two units per CTA of each GEMM with at
// least 12 (or 20, below) K stages per unit (a unit holds at most 128, a
// grouped unit of up to group_max routes 128 / group_max; FC1 needs at most 4
// splits below 512 K stages).  The planner counts routes, not groups: the
// kernel has at most as many units.  The FC1 partials are stored with a
// power-of-two split stride of at most max_splits rounded up.
struct DecodePlan {
  int s1, s2, grid;
};

DecodePlan plan_decode(int routes, const TensorGeom& g1, const TensorGeom& g2, int grid_cap, int max_splits,
                       int group_max) {
  int stride_cap = 1;
  while (stride_cap < max_splits) stride_cap <<= 1;
  // When FC1 has at most half as many (route, tile) pairs as CTAs (m = 1 on
  // the decode workload), units of >= 20 stages measured faster than >= 12:
  // every unit adds about a microsecond of hand-over.
  const int min_stages = 2LL * routes * g1.n_tiles <= grid_cap ? 20 : 12;
  auto pick = [&](const TensorGeom& g, int cap) {
    const long long base = (long long)routes * g.n_tiles;
    int s = (int)((2LL * grid_cap + base - 1) / base);
    const int most = g.k_stages / min_stages > 1 ? g.k_stages / min_stages : 1;
    if (s > most) s = most;
    if (s > cap) s = cap;
    const int least = (g.k_stages * group_max + kDecodeMaxStages - 1) / kDecodeMaxStages;  // unit length cap
    return s < least ? least : s;
  };
  DecodePlan plan;
  // at most 4 FC1 splits: an FC2 unit sums that many partials per h element,
  // and with a stride of 8 its loads take more round trips
  plan.s1 = pick(g1, stride_cap < 4 ? stride_cap : 4);
  plan.s2 = pick(g2, max_splits);
  const long long U = (long long)routes * (g1.n_tiles * plan.s1 + g2.n_tiles * plan.s2);
  plan.grid = (int)(U < grid_cap ? U : grid_cap);
  return plan;
}

template <int MODE>
cudaError_t launch_mode(int fmt, bool weights_on_n, const GemmParams& p, int grid, bool pdl, cudaStream_t st) {
  if (weights_on_n)
    return fmt == 0 ? launch_gemm_wn<MODE, 0>(p, grid, pdl, st) : launch_gemm_wn<MODE, 1>(p, grid, pdl, st);
  return fmt == 0 ? launch_gemm<MODE, 0>(p, grid, pdl, st) : launch_gemm<MODE, 1>(p, grid, pdl, st);
}

}  // namespace

namespace b4 {
// Raises the dynamic shared-memory limit of kernel `func` to `bytes` on the
// current device.  The limit is a per-device setting, so it is set once per
// (device, kernel) and raised again if a larger size is asked for; the table
// is shared by every host thread under one lock.
cudaError_t ensure_smem_limit(const void* func, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  struct Entry {
    int dev;
    const void* func;
    size_t bytes;
  };
  static std::mutex mu;
  static Entry table[256];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  int i = 0;
  for (; i < used; ++i)
    if (table[i].dev == dev && table[i].func == func) break;
  if (i < used && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (i < used) table[i].bytes = bytes;
  else if (used < 256) table[used++] = Entry{dev, func, bytes};
  return cudaSuccess;
}

// Sets the message b4_last_error returns on this thread (for entry points
// defined in other translation units).
void set_last_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}
}  // namespace b4

// device-side counter of invalid scale codes found by b4_prepare_weights
static __device__ int g_prepare_bad;

extern "C" {

int32_t b4_route_capacity_tokens(int32_t m) { return next_pow2(m > 0 ? m : 1); }

size_t b4_workspace_bytes(const b4_moe_config* cfg, int32_t activation) {
  if (check_config(cfg, activation) != B4_OK) return 0;
  return ws_layout(cfg, activation).total;
}

b4_status b4_prepared_sizes(const b4_moe_config* cfg, int32_t which, int32_t activation, size_t* code_bytes,
                            size_t* scale_bytes) {
  b4_status st = check_config(cfg, activation);
  if (st != B4_OK) return st;
  if (which != 0 && which != 1) return fail(B4_ERR_INVALID_ARGUMENT, "which = %d must be 0 (W13) or 1 (W2)", which);
  if (!code_bytes || !scale_bytes) return fail(B4_ERR_INVALID_ARGUMENT, "null output pointer");
  const TensorGeom g = tensor_geom(which, kernel_act(activation), cfg->hidden, cfg->inter);
  const size_t stages = (size_t)cfg->num_local_experts * g.n_tiles * g.k_stages;
  *code_bytes = stages * kCodeBytesPerStage;
  *scale_bytes = stages * scale_bytes_per_stage(cfg->format);
  return B4_OK;
}

b4_status b4_prepare_weights(const b4_moe_config* cfg, int32_t which, int32_t activation, const uint8_t* src_codes,
                             const uint8_t* src_scales, uint8_t* dst_codes, uint8_t* dst_scales, b4_stream_t stream) {
  size_t cb = 0, sb = 0;
  b4_status st = b4_prepared_sizes(cfg, which, activation, &cb, &sb);
  if (st != B4_OK) return st;
  if (!src_codes || !src_scales || !dst_codes || !dst_scales)
    return fail(B4_ERR_INVALID_ARGUMENT, "null weight pointer");
  if (!aligned(dst_codes, 16) || !aligned(dst_scales, 16))
    return fail(B4_ERR_INVALID_ARGUMENT, "prepared buffers must be 16-byte aligned");
  DevInfo dev;
  if ((st = device_info(dev)) != B4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int zero = 0;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_prepare_bad, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "prepare: reset");
  int* bad = nullptr;
  e = cudaGetSymbolAddress(reinterpret_cast<void**>(&bad), g_prepare_bad);
  if (e != cudaSuccess) return cuda_fail(e, "prepare: symbol");
  PrepareParams p{};
  p.src_codes = src_codes;
  p.src_scales = src_scales;
  p.dst_codes = dst_codes;
  p.dst_scales = dst_scales;
  p.num_experts = cfg->num_local_experts;
  p.which = which;
  p.act = kernel_act(activation);
  p.fmt = cfg->format;
  p.hidden = cfg->hidden;
  p.inter = cfg->inter;
  p.bad = bad;
  if ((e = launch_prepare(p, dev.sms, s)) != cudaSuccess) return cuda_fail(e, "prepare: launch");
  int nbad = 0;
  e = cudaMemcpyFromSymbolAsync(&nbad, g_prepare_bad, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "prepare: readback");
  if (nbad)
    return fail(B4_ERR_INVALID_ARGUMENT,
                "%d block scale(s) are NaN or outside the supported range (E8M0: 65..191 for nonzero blocks)", nbad);
  return B4_OK;
}

b4_status b4_route_pack(const b4_moe_config* cfg, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                        int32_t* sorted_routes, b4_stream_t stream) {
  b4_status st = check_config(cfg, B4_ACT_SILU_SWIGLU);
  if (st != B4_OK) return st;
  if ((cfg->m > 0 && !topk_ids) || !counts || !offsets || !sorted_routes)
    return fail(B4_ERR_INVALID_ARGUMENT, "null pointer argument");
  DevInfo dev;
  if ((st = device_info(dev)) != B4_OK) return st;
  RoutePackParams p{};
  p.topk_ids = topk_ids;
  p.expert_map = cfg->expert_map;
  p.m = cfg->m;
  p.top_k = cfg->top_k;
  p.num_global_experts = cfg->num_global_experts;
  p.num_local_experts = cfg->num_local_experts;
  p.route_cap = b4_route_capacity_tokens(cfg->m) * cfg->top_k;
  p.counts = counts;
  p.offsets = offsets;
  p.sorted_routes = sorted_routes;
  cudaError_t e = launch_route_pack(p, dev.sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? B4_OK : cuda_fail(e, "route_pack");
}

b4_status b4_fused_moe(const b4_moe_config* cfg, const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                       const float* gs13, const uint8_t* w2, const uint8_t* s2, const float* gs2,
                       const int32_t* topk_ids, const float* topk_weights, int32_t activation, uint16_t* out,
                       void* workspace, size_t workspace_bytes, b4_stream_t stream) {
  b4_status st = check_config(cfg, activation);
  if (st != B4_OK) return st;
  GluParams glu;
  if ((st = glu_params(cfg, activation, &glu)) != B4_OK) return st;
  if (cfg->m == 0) return B4_OK;  // nothing to compute, nothing launched
  if (!x || !w13 || !s13 || !w2 || !s2 || !topk_ids || !topk_weights || !out || !workspace)
    return fail(B4_ERR_INVALID_ARGUMENT, "null pointer argument");
  const bool nv = cfg->format == B4_NVFP4_E4M3_K16;
  if (nv && (!gs13 || !gs2)) return fail(B4_ERR_INVALID_ARGUMENT, "NVFP4 needs gs13 and gs2");
  if (!nv && (gs13 || gs2)) return fail(B4_ERR_INVALID_ARGUMENT, "MXFP4 takes no global scales (pass NULL)");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(w13, 16) || !aligned(s13, 16) || !aligned(w2, 16) ||
      !aligned(s2, 16))
    return fail(B4_ERR_INVALID_ARGUMENT, "x, out and the weight buffers must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(B4_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (!aligned(topk_ids, 4) || !aligned(topk_weights, 4) || (gs13 && !aligned(gs13, 4)) || (gs2 && !aligned(gs2, 4)))
    return fail(B4_ERR_INVALID_ARGUMENT, "misaligned 32-bit array");
  const WsLayout L = ws_layout(cfg, activation);
  if (workspace_bytes < L.total)
    return fail(B4_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes, %zu needed", workspace_bytes, L.total);
  DevInfo dev;
  if ((st = device_info(dev)) != B4_OK) return st;

  const int act = kernel_act(activation);
  const int fmt = cfg->format;
  // AUTO: the small-m path up to m = 16, and up to B4_DECODE_MAX_M while an
  // expert receives at most two routes on average (decode E128 k8 m = 32:
  // 334 vs 368 us on the grouped GEMMs; small-batch E64 k6 m = 32, three per
  // expert: the grouped GEMMs win)
  bool decode = cfg->path == B4_PATH_DECODE ||
                (cfg->path == B4_PATH_AUTO &&
                 (cfg->m <= kDecodeAutoMaxM ||
                  (cfg->m <= B4_DECODE_MAX_M && (long long)cfg->m * cfg->top_k <= 2LL * cfg->num_local_experts)));
  if (decode && !L.decode_ok) decode = false;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const TensorGeom g1 = tensor_geom(0, act, cfg->hidden, cfg->inter);
  const TensorGeom g2 = tensor_geom(1, act, cfg->hidden, cfg->inter);

  GemmParams base{};
  base.m = cfg->m;
  base.top_k = cfg->top_k;
  base.num_global_experts = cfg->num_global_experts;
  base.num_local_experts = cfg->num_local_experts;
  base.hidden = cfg->hidden;
  base.inter = cfg->inter;
  base.inter_pad = L.inter_pad;
  base.act = act;
  base.glu = glu;
  base.topk_ids = topk_ids;
  base.topk_weights = topk_weights;
  base.expert_map = cfg->expert_map;
  base.x = x;
  base.status = status;
  base.max_chunks = L.max_chunks;

  GemmParams p1 = base, p2 = base;
  p1.trace = g_trace;
  p2.trace = g_trace ? g_trace + 5 * kTraceLen : nullptr;
  p1.wcodes = w13;
  p1.wscales = s13;
  p1.gs = gs13;
  p1.n_tiles = g1.n_tiles;
  p1.k_stages = g1.k_stages;
  p2.wcodes = w2;
  p2.wscales = s2;
  p2.gs = gs2;
  p2.n_tiles = g2.n_tiles;
  p2.k_stages = g2.k_stages;

  FinalizeParams fp{};
  fp.m = cfg->m;
  fp.hidden = cfg->hidden;
  fp.out = out;

  cudaError_t e;
  const long long routes = (long long)cfg->m * cfg->top_k;
  const bool per_route = cfg->m <= kPerRouteMaxM || routes <= cfg->num_local_experts ||
                         (routes <= 2LL * cfg->num_local_experts && routes <= kDecodeGroupRoutes);
  if (decode && per_route) {
    // the per-route kernel: one unit per (route, tile, K split)
    const int R = cfg->m * cfg->top_k;
    // grouped units once routes repeat experts (m * top_k >= E_local), while
    // the group table fits and a grouped FC1 unit needs at most 4 K splits (an
    // FC2 unit sums up to 4 per h element)
    const int group_max = cfg->m >= 2 && R >= cfg->num_local_experts && R <= kDecodeGroupRoutes &&
                                  g1.k_stages <= kDecodeMaxStages
                              ? kDecodeGroupMax
                              : 1;
    int occ = 0;
    if ((e = decode_occupancy(fmt, group_max > 1, &occ)) != cudaSuccess) return cuda_fail(e, "decode occupancy");
    if (occ < 1) return fail(B4_ERR_CUDA, "the decode kernel does not fit on an SM");
    const DecodePlan plan = plan_decode(R, g1, g2, occ * dev.sms, L.dec_splits, group_max);
    DecodeParams dp{};
    dp.w1_codes = w13;
    dp.w1_scales = s13;
    dp.gs1 = gs13;
    dp.w2_codes = w2;
    dp.w2_scales = s2;
    dp.gs2 = gs2;
    dp.n_tiles1 = g1.n_tiles;
    dp.k_stages1 = g1.k_stages;
    dp.n_tiles2 = g2.n_tiles;
    dp.k_stages2 = g2.k_stages;
    dp.m = cfg->m;
    dp.top_k = cfg->top_k;
    dp.num_global_experts = cfg->num_global_experts;
    dp.num_local_experts = cfg->num_local_experts;
    dp.hidden = cfg->hidden;
    dp.inter_pad = L.inter_pad;
    dp.act = act;
    dp.glu = glu;
    dp.topk_ids = topk_ids;
    dp.topk_weights = topk_weights;
    dp.expert_map = cfg->expert_map;
    dp.x = x;
    dp.out = out;
    dp.s1 = plan.s1;
    dp.s2 = plan.s2;
    dp.s1_stride = 1;
    while (dp.s1_stride < plan.s1) dp.s1_stride <<= 1;
    dp.units1 = R * g1.n_tiles * plan.s1;
    dp.units2 = R * g2.n_tiles * plan.s2;
    dp.group_max = group_max;
    dp.p = reinterpret_cast<float*>(ws + L.op);
    dp.q = reinterpret_cast<float*>(ws + L.oq);
    dp.p_floats = (size_t)R * fc1_natural_width(act, L.inter_pad) * dp.s1_stride;
    dp.ticket = reinterpret_cast<int*>(ws + L.status + 64);
    dp.q_floats = (size_t)plan.s2 * R * cfg->hidden;
    dp.status = status;
    dp.trace = g_trace;
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = launch_decode(dp, fmt, plan.grid, s)) != cudaSuccess) return cuda_fail(e, "decode");
    if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    return B4_OK;
  }

  if (decode) {
    // the route-grouped kernel: an expert's weights stream once per group of routes
    const int R = cfg->m * cfg->top_k;
    const int sets = R <= 8 ? 1 : 2;  // groups of at most 8 or 16 routes
    const size_t smem = decode_grouped_smem(fmt, sets, R);
    int occ = 0;
    if ((e = decode_grouped_occupancy(fmt, sets, smem, &occ)) != cudaSuccess) return cuda_fail(e, "decode occupancy");
    if (occ < 1) return fail(B4_ERR_CUDA, "the small-m kernel does not fit on an SM");
    SmallGroupParams dp{};
    dp.w1_codes = w13;
    dp.w1_scales = s13;
    dp.gs1 = gs13;
    dp.w2_codes = w2;
    dp.w2_scales = s2;
    dp.gs2 = gs2;
    dp.n_tiles1 = g1.n_tiles;
    dp.k_stages1 = g1.k_stages;
    dp.n_tiles2 = g2.n_tiles;
    dp.k_stages2 = g2.k_stages;
    dp.m = cfg->m;
    dp.top_k = cfg->top_k;
    dp.num_global_experts = cfg->num_global_experts;
    dp.num_local_experts = cfg->num_local_experts;
    dp.hidden = cfg->hidden;
    dp.inter_pad = L.inter_pad;
    dp.act = act;
    dp.glu = glu;
    dp.topk_ids = topk_ids;
    dp.topk_weights = topk_weights;
    dp.expert_map = cfg->expert_map;
    dp.x = x;
    dp.out = out;
    dp.p = reinterpret_cast<float*>(ws + L.dp);
    dp.p_stride = L.dec_pmax;
    dp.q = reinterpret_cast<float*>(ws + L.dq);
    dp.q_pieces = L.dec_pmax;
    dp.p_floats = (size_t)R * L.wnat * L.dec_pmax;
    dp.q_floats = (size_t)L.dec_pmax * R * cfg->hidden;
    dp.h = reinterpret_cast<uint16_t*>(ws + L.dh);
    dp.hflag = reinterpret_cast<int*>(ws + L.dcnt);
    dp.n_flags = (size_t)R * g1.n_tiles;
    dp.pmax = L.dec_pmax;
    dp.w0 = kDecodeW0;
    dp.status = status;
    dp.trace = g_trace;
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = launch_decode_grouped(dp, fmt, sets, dev.sms, s)) != cudaSuccess) return cuda_fail(e, "decode");
    if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    return B4_OK;
  }

  RoutePackParams rp{};
  rp.topk_ids = topk_ids;
  rp.expert_map = cfg->expert_map;
  rp.m = cfg->m;
  rp.top_k = cfg->top_k;
  rp.num_global_experts = cfg->num_global_experts;
  rp.num_local_experts = cfg->num_local_experts;
  rp.route_cap = L.r_cap;
  rp.counts = reinterpret_cast<int32_t*>(ws + L.counts);
  rp.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  rp.sorted_routes = reinterpret_cast<int32_t*>(ws + L.sorted);
  rp.chunks = reinterpret_cast<int4*>(ws + L.chunks);
  rp.chunk_count = reinterpret_cast<int32_t*>(ws + L.chunk_count);
  // Weights on the MMA's N side (256 rows per instruction, chunks of <= 128
  // routes on M) issue half the MMAs when experts receive few routes; with
  // ~128 routes per expert (prefill) both issue about as many, and the weights-
  // on-M kernel keeps the weights in tensor memory and measured faster.
  const bool weights_on_n = (long long)cfg->m * cfg->top_k < 96LL * cfg->num_local_experts;
  rp.chunk_rows = weights_on_n ? kChunkRowsN : kChunkRowsM;
  rp.status = status;
  uint16_t* xp = reinterpret_cast<uint16_t*>(ws + L.xp);  // x rows in packed-route order, copied by the route pack
  if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  if ((e = launch_route_pack(rp, dev.sms, s, x, xp, cfg->hidden)) != cudaSuccess) return cuda_fail(e, "route pack");
  if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");

  uint16_t* hbuf = reinterpret_cast<uint16_t*>(ws + L.h);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  for (GemmParams* pp : {&p1, &p2}) {
    pp->sorted_routes = rp.sorted_routes;
    pp->chunk_count = rp.chunk_count;
    pp->chunks = rp.chunks;
  }
  // B boxes: 32 rows for the weights-on-N kernel's operand stages, 80 for the
  // weights-on-M kernel (two per 160-row stage)
  if (!make_tmap_bf16_2d(&p1.tmap_b, xp, (uint64_t)L.r_cap, (uint64_t)cfg->hidden, weights_on_n ? 32 : 80))
    return fail(B4_ERR_CUDA, "cuTensorMapEncodeTiled rejected the packed-x map");
  if (!make_tmap_bf16_2d(&p2.tmap_b, hbuf, (uint64_t)L.r_cap, (uint64_t)L.inter_pad, weights_on_n ? 32 : 80))
    return fail(B4_ERR_CUDA, "cuTensorMapEncodeTiled rejected the h map");
  p1.h_out = hbuf;
  p1.acc_out = acc;
  p1.acc_zero_floats = (size_t)cfg->m * cfg->hidden;
  p1.pdl_wait_first = 1;
  p2.h = hbuf;
  p2.acc_out = acc;
  if (weights_on_n) p2.k_splits = -1;  // few units: split FC2's K (its epilogue adds fp32 partials)
  if ((e = launch_mode<kFc1Grouped>(fmt, weights_on_n, p1, dev.sms, true, s)) != cudaSuccess) return cuda_fail(e, "fc1 grouped");
  if ((e = mark(2, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  if ((e = launch_mode<kFc2Grouped>(fmt, weights_on_n, p2, dev.sms, true, s)) != cudaSuccess) return cuda_fail(e, "fc2 grouped");
  if ((e = mark(3, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  fp.acc = acc;
  if ((e = launch_finalize(fp, dev.sms, s)) != cudaSuccess) return cuda_fail(e, "finalize grouped");
  if ((e = mark(4, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  return B4_OK;
}

// ------------------------------------------------------------ dense linear
namespace {
b4_status check_linear(const b4_moe_config* cfg) {
  b4_status st = check_config(cfg, B4_ACT_RELU2);
  if (st != B4_OK) return st;
  if (cfg->top_k != 1 || cfg->num_local_experts != 1 || cfg->num_global_experts != 1 || cfg->expert_map)
    return fail(B4_ERR_INVALID_ARGUMENT, "the linear layer takes top_k = 1, one expert and no expert_map");
  return B4_OK;
}

// The linear layer's workspace: the fused layer's pieces with the fp32
// accumulator rows widened to max(K, N) (a K-split GEMM adds into [m, N]).
WsLayout linear_layout(const b4_moe_config* cfg) {
  b4_moe_config c = *cfg;
  if (c.inter > c.hidden) c.hidden = c.inter;
  return ws_layout(&c, B4_ACT_RELU2);
}
}  // namespace

size_t b4_linear_workspace_bytes(const b4_moe_config* cfg) {
  if (check_linear(cfg) != B4_OK) return 0;
  return linear_layout(cfg).total;
}

b4_status b4_linear(const b4_moe_config* cfg, const uint16_t* x, const uint8_t* w, const uint8_t* sc,
                    const float* gs, uint16_t* out, void* workspace, size_t workspace_bytes, b4_stream_t stream) {
  b4_status st = check_linear(cfg);
  if (st != B4_OK) return st;
  if (cfg->m == 0) return B4_OK;  // nothing to compute, nothing launched
  if (!x || !w || !sc || !out || !workspace) return fail(B4_ERR_INVALID_ARGUMENT, "null pointer argument");
  const bool nv = cfg->format == B4_NVFP4_E4M3_K16;
  if (nv && !gs) return fail(B4_ERR_INVALID_ARGUMENT, "NVFP4 needs gs");
  if (!nv && gs) return fail(B4_ERR_INVALID_ARGUMENT, "MXFP4 takes no global scale (pass NULL)");
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(w, 16) || !aligned(sc, 16))
    return fail(B4_ERR_INVALID_ARGUMENT, "x, out and the weight buffers must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(B4_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (gs && !aligned(gs, 4)) return fail(B4_ERR_INVALID_ARGUMENT, "misaligned gs");
  const WsLayout L = linear_layout(cfg);
  if (workspace_bytes < L.total)
    return fail(B4_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes, %zu needed", workspace_bytes, L.total);
  DevInfo dev;
  if ((st = device_info(dev)) != B4_OK) return st;

  const int fmt = cfg->format;
  const int m = cfg->m, N = cfg->inter, K = cfg->hidden;
  bool small = cfg->path == B4_PATH_DECODE || (cfg->path == B4_PATH_AUTO && m <= kLinearSmallMaxM);
  if (small && !L.decode_ok) small = false;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const TensorGeom g1 = tensor_geom(0, 1, K, N);
  cudaError_t e;

  if (small && m <= kLinearPerRouteMaxM) {
    // The fused small-m kernel: K-split GEMV units, then one output unit per
    // (token, 128 columns) that sums the split partials into out.  From m = 2
    // its FC1 units take up to four tokens each (grouped units: every token
    // goes to the one weight matrix, so there are ceil(m / 4) groups).
    const int group_max = m >= 2 && g1.k_stages <= kDecodeMaxStages ? kDecodeGroupMax : 1;
    const int groups = (m + group_max - 1) / group_max;
    int occ = 0;
    if ((e = decode_occupancy(fmt, group_max > 1, &occ)) != cudaSuccess) return cuda_fail(e, "decode occupancy");
    if (occ < 1) return fail(B4_ERR_CUDA, "the decode kernel does not fit on an SM");
    // K splits: about two GEMV units per CTA, at least 8 stages each, at
    // most the partial buffer's split count (summing up to 8 partials per
    // output is cheap here: no activation row is built from them).
    const int cap = occ * dev.sms;
    const long long base = (long long)groups * g1.n_tiles;
    int s1 = (int)((2LL * cap + base - 1) / base);
    const int most = g1.k_stages / 8 > 1 ? g1.k_stages / 8 : 1;
    if (s1 > most) s1 = most;
    if (s1 > L.dec_splits) s1 = L.dec_splits;
    const int least = (g1.k_stages * group_max + kDecodeMaxStages - 1) / kDecodeMaxStages;
    if (s1 < least) s1 = least;
    const DecodePlan plan{s1, 1, 0};
    DecodeParams dp{};
    dp.group_max = group_max;
    dp.w1_codes = w;
    dp.w1_scales = sc;
    dp.gs1 = gs;
    dp.n_tiles1 = g1.n_tiles;
    dp.k_stages1 = g1.k_stages;
    dp.n_tiles2 = g1.n_tiles;
    dp.k_stages2 = 1;
    dp.m = m;
    dp.top_k = 1;
    dp.num_global_experts = 1;
    dp.num_local_experts = 1;
    dp.hidden = K;
    dp.inter_pad = L.inter_pad;
    dp.act = 1;  // the non-gated FC1 partial layout; no activation is applied
    dp.linear = 1;
    dp.n_out = N;
    dp.x = x;
    dp.out = out;
    dp.s1 = plan.s1;
    dp.s2 = 1;
    dp.s1_stride = 1;
    while (dp.s1_stride < plan.s1) dp.s1_stride <<= 1;
    dp.units1 = m * g1.n_tiles * plan.s1;
    dp.units2 = m * g1.n_tiles;
    dp.p = reinterpret_cast<float*>(ws + L.op);
    dp.p_floats = (size_t)m * L.inter_pad * dp.s1_stride;
    dp.ticket = reinterpret_cast<int*>(ws + L.status + 64);
    dp.status = status;
    dp.trace = g_trace;
    const long long U = (long long)dp.units1 + dp.units2;
    const int grid = (int)(U < cap ? U : cap);
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = launch_decode(dp, fmt, grid, s)) != cudaSuccess) return cuda_fail(e, "linear (fused small-m)");
    if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    return B4_OK;
  }

  if (small) {
    // The small-m kernel's FC1 phase alone: the routes are the tokens (every
    // one to the single expert), and the last piece of each 128-column tile
    // writes out.
    const int sets = m <= 8 ? 1 : 2;
    const size_t smem = decode_grouped_smem(fmt, sets, m);
    int occ = 0;
    if ((e = decode_grouped_occupancy(fmt, sets, smem, &occ)) != cudaSuccess) return cuda_fail(e, "decode occupancy");
    if (occ < 1) return fail(B4_ERR_CUDA, "the small-m kernel does not fit on an SM");
    SmallGroupParams dp{};
    dp.w1_codes = w;
    dp.w1_scales = sc;
    dp.gs1 = gs;
    dp.n_tiles1 = g1.n_tiles;
    dp.k_stages1 = g1.k_stages;
    dp.m = m;
    dp.top_k = 1;
    dp.num_global_experts = 1;
    dp.num_local_experts = 1;
    dp.hidden = K;
    dp.inter_pad = L.inter_pad;
    dp.act = 2;
    dp.n_out = N;
    dp.x = x;
    dp.out = out;
    dp.p = reinterpret_cast<float*>(ws + L.dp);
    dp.p_stride = L.dec_pmax;
    dp.q_pieces = L.dec_pmax;
    dp.p_floats = (size_t)m * L.wnat * L.dec_pmax;
    dp.hflag = reinterpret_cast<int*>(ws + L.dcnt);
    dp.n_flags = 0;
    dp.pmax = L.dec_pmax;
    dp.w0 = kDecodeW0;
    dp.status = status;
    dp.trace = g_trace;
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = launch_decode_grouped(dp, fmt, sets, dev.sms, s)) != cudaSuccess)
      return cuda_fail(e, "linear (fused small-m)");
    if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    return B4_OK;
  }

  // The grouped tcgen05 GEMM over one "expert" whose routes are the tokens in
  // order: the route pack of the trivial routing writes the chunk schedule
  // and the GEMM reads x rows directly (slot i is token i).  With enough
  // (chunk, tile) units for the GPU, its FC1 epilogue stores the scaled
  // accumulator as bf16; with few (small m: one chunk, N / 256 tile pairs),
  // the weights-on-N kernel runs in its FC2 mode with K split across units,
  // adding fp32 partials into [m, N], and the finalize kernel rounds them.
  RoutePackParams rp{};
  rp.topk_ids = nullptr;
  rp.m = m;
  rp.top_k = 1;
  rp.num_global_experts = 1;
  rp.num_local_experts = 1;
  rp.route_cap = L.r_cap;
  rp.counts = reinterpret_cast<int32_t*>(ws + L.counts);
  rp.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  rp.sorted_routes = reinterpret_cast<int32_t*>(ws + L.sorted);
  rp.chunks = reinterpret_cast<int4*>(ws + L.chunks);
  rp.chunk_count = reinterpret_cast<int32_t*>(ws + L.chunk_count);
  const bool weights_on_n = m < 96;  // the fused-MoE rule m * top_k < 96 * E_l with E_l = top_k = 1
  rp.chunk_rows = weights_on_n ? kChunkRowsN : kChunkRowsM;
  rp.status = status;
  const int base_units = cdiv(m, kChunkRowsN) * ((g1.n_tiles + 1) / 2);
  if (weights_on_n && base_units < dev.sms) {
    int ks = cdiv(dev.sms, base_units);
    const int most = g1.k_stages / 4 > 1 ? g1.k_stages / 4 : 1;  // >= 4 K stages per split
    if (ks > most) ks = most;
    GemmParams p2{};
    p2.m = m;
    p2.top_k = 1;
    p2.num_global_experts = 1;
    p2.num_local_experts = 1;
    p2.hidden = N;  // FC2 mode: output columns
    p2.inter = K;   // ... and its K
    p2.inter_pad = round_up(K, kBK);
    p2.act = 1;
    p2.x = x;
    p2.status = status;
    p2.max_chunks = L.max_chunks;
    p2.trace = g_trace;
    p2.wcodes = w;
    p2.wscales = sc;
    p2.gs = gs;
    p2.n_tiles = g1.n_tiles;
    p2.k_stages = g1.k_stages;
    p2.k_splits = ks;
    p2.sorted_routes = rp.sorted_routes;
    p2.chunk_count = rp.chunk_count;
    p2.chunks = rp.chunks;
    if (!make_tmap_bf16_2d(&p2.tmap_b, x, (uint64_t)m, (uint64_t)K, 32))
      return fail(B4_ERR_CUDA, "cuTensorMapEncodeTiled rejected the x map");
    float* acc = reinterpret_cast<float*>(ws + L.acc);
    p2.acc_out = acc;
    p2.pdl_wait_first = 1;
    FinalizeParams fp{};
    fp.m = m;
    fp.hidden = N;
    fp.acc = acc;
    fp.out = out;
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = cudaMemsetAsync(acc, 0, (size_t)m * N * sizeof(float), s)) != cudaSuccess)
      return cuda_fail(e, "linear: clear the accumulator");
    if ((e = launch_route_pack(rp, dev.sms, s)) != cudaSuccess) return cuda_fail(e, "route pack");
    if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = launch_mode<kFc2Grouped>(fmt, true, p2, dev.sms, true, s)) != cudaSuccess)
      return cuda_fail(e, "linear (K-split grouped)");
    if ((e = mark(2, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    if ((e = launch_finalize(fp, dev.sms, s)) != cudaSuccess) return cuda_fail(e, "linear: finalize");
    if ((e = mark(3, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
    return B4_OK;
  }
  GemmParams p1{};
  p1.m = m;
  p1.top_k = 1;
  p1.num_global_experts = 1;
  p1.num_local_experts = 1;
  p1.hidden = K;
  p1.inter = N;
  p1.inter_pad = L.inter_pad;
  p1.act = 2;
  p1.x = x;
  p1.status = status;
  p1.max_chunks = L.max_chunks;
  p1.trace = g_trace;
  p1.wcodes = w;
  p1.wscales = sc;
  p1.gs = gs;
  p1.n_tiles = g1.n_tiles;
  p1.k_stages = g1.k_stages;
  p1.sorted_routes = rp.sorted_routes;
  p1.chunk_count = rp.chunk_count;
  p1.chunks = rp.chunks;
  if (!make_tmap_bf16_2d(&p1.tmap_b, x, (uint64_t)m, (uint64_t)K, weights_on_n ? 32 : 80))
    return fail(B4_ERR_CUDA, "cuTensorMapEncodeTiled rejected the x map");
  const bool direct = N == L.inter_pad;  // rows of h are rows of out
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(ws + L.h);
  p1.h_out = direct ? out : hbuf;
  p1.pdl_wait_first = 1;
  if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  if ((e = launch_route_pack(rp, dev.sms, s)) != cudaSuccess) return cuda_fail(e, "route pack");
  if ((e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  if ((e = launch_mode<kFc1Grouped>(fmt, weights_on_n, p1, dev.sms, true, s)) != cudaSuccess)
    return cuda_fail(e, "linear (grouped)");
  if (!direct &&
      (e = cudaMemcpy2DAsync(out, (size_t)N * 2, hbuf, (size_t)L.inter_pad * 2, (size_t)N * 2, (size_t)m,
                             cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "linear: copy to out");
  if ((e = mark(2, s)) != cudaSuccess) return cuda_fail(e, "timing event record");
  return B4_OK;
}

b4_status b4_set_trace(void* device_buffer, size_t bytes) {
  if (device_buffer && bytes < 16 * kTraceLen * sizeof(long long))
    return fail(B4_ERR_INVALID_ARGUMENT, "trace buffer needs %zu bytes", 16 * kTraceLen * sizeof(long long));
  g_trace = static_cast<long long*>(device_buffer);
  return B4_OK;
}

b4_status b4_set_timing_events(void* const* events, int32_t n) {
  if (n > 0 && (!events || n < 2)) return fail(B4_ERR_INVALID_ARGUMENT, "need NULL or at least 2 events");
  g_events = n > 0 ? events : nullptr;
  g_num_events = n > 0 ? n : 0;
  return B4_OK;
}

b4_status b4_wait_self_test(void* workspace, size_t workspace_bytes, uint32_t limit_us, b4_stream_t stream) {
  if (!workspace || workspace_bytes < 8) return fail(B4_ERR_INVALID_ARGUMENT, "workspace needs >= 8 bytes");
  if (limit_us < 1 || limit_us > 1000000) return fail(B4_ERR_INVALID_ARGUMENT, "limit_us must be in 1 .. 1000000");
  const cudaError_t e = b4::launch_wait_self_test(reinterpret_cast<uint32_t*>(workspace),
                                                  1000ull * limit_us, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  return B4_OK;
}

b4_status b4_check_status(void* workspace, b4_stream_t stream) {
  if (!workspace) return fail(B4_ERR_INVALID_ARGUMENT, "workspace is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "check_status");
  if (word[0] != 0) {
    const uint32_t zero[2] = {0, 0};
    e = cudaMemcpyAsync(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "check_status reset");
    return fail(static_cast<b4_status>(word[0]), "device reported status %u at wait site %u", word[0], word[1]);
  }
  return B4_OK;
}

const char* b4_status_string(int32_t status) {
  switch (status) {
    case B4_OK: return "B4_OK";
    case B4_ERR_INVALID_ARGUMENT: return "B4_ERR_INVALID_ARGUMENT";
    case B4_ERR_UNSUPPORTED_DEVICE: return "B4_ERR_UNSUPPORTED_DEVICE";
    case B4_ERR_WORKSPACE_TOO_SMALL: return "B4_ERR_WORKSPACE_TOO_SMALL";
    case B4_ERR_CUDA: return "B4_ERR_CUDA";
    case B4_ERR_TIMEOUT: return "B4_ERR_TIMEOUT";
    default: return "B4_UNKNOWN_STATUS";
  }
}

const char* b4_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
