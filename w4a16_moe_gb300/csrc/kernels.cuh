// Kernel parameter blocks and layout constants shared by the host dispatch
// and the CUDA kernels of the fused W4A16 MoE layer.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

namespace b4 {

// ---------------------------------------------------------------- tiling
constexpr int kTileRows = 128;   // weight rows per tile (tcgen05 M)
constexpr int kBK = 64;          // K elements per pipeline stage
constexpr int kCodeBytesPerStage = kTileRows * kBK / 2;  // 4096: [2 chunks][128 rows][16 B]
// max routes of one expert per grouped work unit: tcgen05 N when the weights
// are on M (many routes per expert), tcgen05 M when the weights are on N
constexpr int kChunkRowsM = 160;
constexpr int kChunkRowsN = 128;

__host__ __device__ constexpr int scale_bytes_per_row(int fmt) { return fmt == 0 ? kBK / 16 : kBK / 32; }
__host__ __device__ constexpr int scale_bytes_per_stage(int fmt) { return kTileRows * scale_bytes_per_row(fmt); }
__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int round_up(int a, int b) { return cdiv(a, b) * b; }

// Serving-layout geometry of one tensor.
struct TensorGeom {
  int rows_valid;  // N of the source tensor
  int k_valid;     // K of the source tensor
  int n_tiles;     // 128-row tiles
  int k_stages;    // 64-element stages
};

// which: 0 = W13/W1, 1 = W2.  act: 0 = SwiGLU (gated W13), otherwise a
// non-gated W1 (1 = ReLU^2, 2 = none: the dense linear layer).
__host__ __device__ inline TensorGeom tensor_geom(int which, int act, int hidden, int inter) {
  TensorGeom g;
  const int inter_pad = round_up(inter, kBK);
  if (which == 0) {
    g.rows_valid = act == 0 ? 2 * inter : inter;
    g.k_valid = hidden;
    g.n_tiles = act == 0 ? inter_pad / 64 : cdiv(inter, kTileRows);
    g.k_stages = cdiv(hidden, kBK);
  } else {
    g.rows_valid = hidden;
    g.k_valid = inter;
    g.n_tiles = cdiv(hidden, kTileRows);
    g.k_stages = inter_pad / kBK;
  }
  return g;
}

// Parameters of the gated FC1 activation (act 0):
//   h = g' * sigmoid(alpha * g') * (u' + beta),
//   g' = min(g, limit), u' = u clamped to [-limit, limit]
// for the gate g and up u of one intermediate column.  Plain SwiGLU is
// alpha = 1, beta = 0, limit = +inf (g' = g, u' = u, g sigmoid(g) = silu(g));
// the clamped swiglu of the gpt-oss models is alpha 1.702, beta 1, limit 7.
struct GluParams {
  float alpha, beta, limit;
};

#ifdef __CUDACC__
// The comparisons (not fminf/fmaxf) keep a NaN input a NaN.  The sigmoid's
// division is the approximate one (__fdividef, 2 ulp; 0 once 1 + e^-x passes
// 2^126, where the exact quotient is below 2^-126 |g'| anyway): h is rounded
// to bf16 next, and the pages' kernels take the same trade (flashinfer PR
// #4255, review comments on moe_w4a16_fp4_helpers.py: silu_mul_32 forms the
// sigmoid with an approximate reciprocal).
__device__ __forceinline__ float gated_act(float g, float u, const GluParams& a) {
  const float gc = g > a.limit ? a.limit : g;
  const float uc = u > a.limit ? a.limit : (u < -a.limit ? -a.limit : u);
  return __fdividef(gc, 1.0f + __expf(-a.alpha * gc)) * (uc + a.beta);
}
#endif

enum GemmMode : int { kFc1Grouped = 0, kFc2Grouped = 1 };

struct GemmParams {
  // TMA map of the grouped activation operand: packed x rows (FC1) or h rows
  // (FC2), box 64 columns x 32 rows, 128-byte swizzle
  CUtensorMap tmap_b;
  // prepared weights of this GEMM
  const uint8_t* wcodes;
  const uint8_t* wscales;
  const float* gs;      // [E_l] or null (MXFP4)
  int n_tiles, k_stages;
  // layer shape
  int m, top_k, num_global_experts, num_local_experts, hidden, inter, inter_pad;
  int act;              // 0 gated (SwiGLU family), 1 ReLU^2, 2 none (dense linear: h = the scaled accumulator)
  GluParams glu;        // act 0
  // routing inputs
  const int32_t* topk_ids;
  const float* topk_weights;  // or null (FC2: router weight 1, the dense linear layer)
  const int32_t* expert_map;  // or null
  // grouped schedule (from the route-pack kernel)
  const int32_t* sorted_routes;
  const int32_t* chunk_count;
  const int4* chunks;   // (expert, first slot, rows, 0)
  int max_chunks;
  // K splits of each (chunk, tile pair) unit: weights-on-N kernel, FC2 mode
  // only (its epilogue adds partials); 0 or 1 = none, negative = chosen in
  // the kernel from the chunk count (about two units per CTA)
  int k_splits;
  // B operand sources
  const uint16_t* x;    // [m, H] bf16 (FC1)
  uint16_t* xp;         // unused (the route pack copies x rows into packed-route order)
  const int32_t* valid_count;  // unused
  const uint16_t* h;    // [R_cap, I_pad] bf16 (FC2 grouped)
  // outputs
  uint16_t* h_out;      // FC1 grouped
  float* acc_out;       // FC2 grouped: [T_cap, H] fp32, zeroed by FC1 grouped
  size_t acc_zero_floats;  // FC1 grouped: floats of acc_out to clear
  uint32_t* status;     // device status word(s)
  int pdl_wait_first;   // all threads wait on the previous grid before starting
  // Optional timeline of CTA 0 (clock64 cycles), or null: [kind][index] with
  // kinds 0 weight stage issued, 1 A stage stored to tensor memory, 2 MMA
  // stage issued, 3 B stage (grouped) or row (decode) ready, 4 epilogue of a
  // unit done; kTraceLen entries per kind.
  long long* trace;
};

constexpr int kTraceLen = 2048;

// The per-route decode path: one cooperative kernel (decode_moe.cu).
// The per-route small-m kernel's grouped units: up to kDecodeGroupMax routes
// of one local expert share a unit (and its weight stream) when m >= 2 and
// m * top_k <= kDecodeGroupRoutes (the group table is in shared memory); a
// grouped unit spans at most kDecodeMaxStages / kDecodeGroupMax K stages.
constexpr int kDecodeGroupMax = 4;
constexpr int kDecodeGroupRoutes = 256;
constexpr int kDecodeMaxStages = 128;

struct DecodeParams {
  const uint8_t* w1_codes;   // prepared W13 / W1
  const uint8_t* w1_scales;
  const float* gs1;          // [E_l] or null (MXFP4)
  const uint8_t* w2_codes;   // prepared W2
  const uint8_t* w2_scales;
  const float* gs2;
  int n_tiles1, k_stages1, n_tiles2, k_stages2;
  int m, top_k, num_global_experts, num_local_experts, hidden, inter_pad;
  int act;                   // 0 gated (SwiGLU family), 1 ReLU^2
  GluParams glu;             // act 0
  // Dense linear layer (E = 1, top-1, no activation, no FC2): the FC2 units
  // become output units (route, 128-column tile of N) that sum the FC1 split
  // partials into out [m, n_out] bf16; topk_ids, topk_weights, w2 and q are
  // unused.
  int linear, n_out;
  const int32_t* topk_ids;   // [m, top_k], or null: every route goes to local expert 0
  const float* topk_weights;
  const int32_t* expert_map;  // or null
  const uint16_t* x;         // [m, H] bf16
  uint16_t* out;             // [m, H] bf16
  int s1, s2;                // K splits of FC1 and FC2
  int s1_stride;             // split stride of the FC1 partials: s1 rounded up to 1, 2, 4 or 8
  int units1, units2;        // R * n_tiles1 * s1 and R * n_tiles2 * s2 (one route per unit)
  int group_max;             // 1: one route per unit; kDecodeGroupMax: units of up to that many routes of one expert
  float* p;                  // FC1 split partials [R][N1 natural][s1_stride]
  float* q;                  // FC2 split partials [s2][R][H]
  size_t p_floats, q_floats; // sizes of p and q (filled with the not-yet-written marker)
  int* ticket;               // units [grid, units1 + units2) are claimed from this counter
  uint32_t* status;
  long long* trace;          // optional timeline (see b4_set_trace)
};

// The route-grouped small-m path: one cooperative kernel (decode_grouped.cu).
struct SmallGroupParams {
  const uint8_t* w1_codes;   // prepared W13 / W1
  const uint8_t* w1_scales;
  const float* gs1;          // [E_l] or null (MXFP4)
  const uint8_t* w2_codes;   // prepared W2
  const uint8_t* w2_scales;
  const float* gs2;
  int n_tiles1, k_stages1;
  int n_tiles2, k_stages2;   // n_tiles2 = 0: no FC2 phase (the dense linear layer)
  int m, top_k, num_global_experts, num_local_experts, hidden, inter_pad;
  int act;                   // 0 gated (SwiGLU family), 1 ReLU^2, 2 none (the dense linear layer: FC1 writes out)
  GluParams glu;             // act 0
  int n_out;                 // the dense linear layer's N (out is [m, n_out])
  const int32_t* topk_ids;   // [m, top_k], or null: every route goes to local expert 0
  const float* topk_weights;
  const int32_t* expert_map;  // or null
  const uint16_t* x;         // [m, H] bf16
  uint16_t* out;             // [m, H] bf16 ([m, n_out] for the linear layer)
  float* p;                  // FC1 partials [R][N1 natural][p_stride] (piece innermost)
  int p_stride;
  float* q;                  // FC2 partials [q_pieces][R][H]
  int q_pieces;
  size_t p_floats, q_floats;  // sizes of p and q (filled with the not-written marker)
  uint16_t* h;               // [R][inter_pad] bf16
  int* hflag;                // [R][n_tiles1] FC1 tile's h built (zeroed at launch)
  size_t n_flags;
  int pmax;                  // most CTAs sharing one tile (<= p_stride, <= q_pieces)
  int w0;                    // partition cost of a stage: w0 + the group's column sets
  uint32_t* status;
  // Optional timeline (b4_set_trace), or null: %globaltimer ns per CTA at
  // phase boundaries, trace[kind * kTraceLen + blockIdx.x].
  long long* trace;
};

struct RoutePackParams {
  const int32_t* topk_ids;   // or null: every route goes to local expert 0 (the dense linear layer)
  const int32_t* expert_map;
  int m, top_k, num_global_experts, num_local_experts;
  int route_cap;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_routes;
  // optional grouped-GEMM schedule
  int4* chunks;
  int32_t* chunk_count;
  int chunk_rows;
  uint32_t* status;     // reset to 0 (first kernel of a grouped call), or null
};

struct FinalizeParams {
  int m, hidden;
  const float* acc;     // [m, H] fp32 top-k sums of the grouped path
  uint16_t* out;
};

struct PrepareParams {
  const uint8_t* src_codes;
  const uint8_t* src_scales;
  uint8_t* dst_codes;
  uint8_t* dst_scales;
  int num_experts, which, act, fmt, hidden, inter;
  int* bad;             // device counter of invalid scale codes
};

// width of the FC1 partial rows of the decode path (gate then up for SwiGLU)
__host__ __device__ inline int fc1_natural_width(int act, int inter_pad) {
  return act == 0 ? 2 * inter_pad : inter_pad;
}

}  // namespace b4
