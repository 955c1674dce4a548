/*
 * b4moe.h -- C ABI of the GB300 (sm_103a) fused W4A16 mixture-of-experts layer.
 *
 * The layer: 4-bit FP4 weights (NVFP4 or MXFP4), bf16 activations, route
 * packing, a grouped FC1 GEMM with in-kernel dequantisation and a fused
 * SiLU-SwiGLU, clamped swiglu or ReLU^2 epilogue, and a grouped FC2 GEMM whose store folds in
 * the top-k weighted sum, plus a separate small-m decode path.  It is the
 * layer described by flashinfer PR #4255, "feat(moe): sync SM12x W4A16 fused
 * MoE family to b12x HEAD" (Description), restated for GB300.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers are DEVICE pointers unless a parameter says "host".  The caller
 *   owns every buffer; the library never allocates or frees device memory.
 * - All GPU work is enqueued on the caller's `stream` (flashinfer PR #4255,
 *   review comment "Propagate the stream into route packing").  b4_route_pack
 *   and b4_fused_moe neither allocate nor synchronise, so both may be captured
 *   into a CUDA graph (b12x PR #136, Summary: caller-owned buffers so decode
 *   graph capture needs no library scratch arena).
 * - Argument problems are reported before anything is launched, as a
 *   b4_status; b4_last_error() then returns a thread-local message.
 * - Device-side failures (a bounded wait that ran out) are written to a
 *   status word at the start of the workspace; read it with b4_check_status.
 * - Only sm_103 devices are accepted (B4_ERR_UNSUPPORTED_DEVICE otherwise);
 *   there is no fallback path.
 *
 * Data types: token ids int32, router weights fp32, activations and output
 * bf16 (raw 16-bit patterns, row-major), packed FP4 codes uint8 (two codes per
 * byte, element 2j in the low nibble), block scales uint8 (E4M3 or E8M0 bit
 * patterns), global scales fp32.
 */
#ifndef B4MOE_H
#define B4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* b4_stream_t;

typedef enum b4_status {
  B4_OK = 0,
  B4_ERR_INVALID_ARGUMENT = 1,   /* bad shape, null or misaligned pointer, bad enum */
  B4_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not sm_103 */
  B4_ERR_WORKSPACE_TOO_SMALL = 3,
  B4_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
  B4_ERR_TIMEOUT = 5             /* a device-side bounded wait ran out */
} b4_status;

/* Weight source formats (flashinfer PR #4255, Description: NVFP4 weights and
 * "a new fp4_e8m0_k32 (MXFP4 K/32) weight source format").
 * NVFP4: E2M1 codes, one FP8-E4M3 block scale per 16 elements along K, and
 *        one fp32 global scale per expert (ModelOpt layout).
 * MXFP4: E2M1 codes, one E8M0 power-of-two scale 2^(e-127) per 32 elements
 *        along K, no global scale.  K need not be a multiple of 128 (the
 *        "scale tail" of tensor-parallel shards). */
typedef enum b4_format { B4_NVFP4_E4M3_K16 = 0, B4_MXFP4_E8M0_K32 = 1 } b4_format;

/* FC1 epilogue activations (flashinfer PR #4255, Performance: relu2, silu).
 * SILU_SWIGLU: W13 has 2*inter rows, rows [0, inter) gate and [inter, 2*inter)
 *              up; h = silu(gate) * up.
 * RELU2:       W1 has inter rows; h = max(a, 0)^2.
 * SWIGLU_OAI:  the clamped swiglu of the gpt-oss models, which the pages name
 *              (flashinfer PR #4255, Description: "swiglu-oai"; b12x PR, CodeRabbit
 *              summary: "SwiGLU parameters") without defining it.  W13 as for
 *              SILU_SWIGLU (gate rows first: a checkpoint that interleaves gate
 *              and up rows is de-interleaved before b4_prepare_weights);
 *              g' = min(gate, limit), u' = up clamped to [-limit, limit],
 *              h = g' * sigmoid(alpha * g') * (u' + beta), with alpha, beta and
 *              limit from b4_moe_config (gpt-oss: 1.702, 1, 7).  Prepared
 *              weights are shared with SILU_SWIGLU. */
typedef enum b4_activation { B4_ACT_SILU_SWIGLU = 0, B4_ACT_RELU2 = 1, B4_ACT_SWIGLU_OAI = 2 } b4_activation;

/* Execution path of b4_fused_moe.  DECODE is the small-m path (accepted for
 * m <= B4_DECODE_MAX_M): one cooperative launch, a per-route kernel for
 * m <= 4 or m * top_k <= num_local_experts (few routes per expert; from m = 2
 * with m * top_k >= num_local_experts its units take up to 4 routes of one
 * expert), also up to m * top_k <= 2 * num_local_experts while that is at
 * most 256 routes, and a route-grouped kernel (an expert's weights streamed
 * once per group of up to 16 of its routes) otherwise.  GROUPED is the route-packed
 * tcgen05 path.  AUTO takes DECODE for m <= 16, and for m <= 64 while
 * m * top_k <= 2 * num_local_experts (at most two routes per expert on
 * average), GROUPED otherwise: the crossover flashinfer PR #4255 (Reviewer
 * Notes) leaves to each card, as measured on GB300; b4_linear's AUTO takes the
 * small-m kernels for m <= 16 (the per-route kernel for m <= 4, the
 * route-grouped one above). */
typedef enum b4_path { B4_PATH_AUTO = 0, B4_PATH_DECODE = 1, B4_PATH_GROUPED = 2 } b4_path;

#define B4_DECODE_MAX_M 64
#define B4_MAX_LOCAL_EXPERTS 1024

/* Problem shape.  All fields are plain values except expert_map. */
typedef struct b4_moe_config {
  int32_t m;                  /* tokens, >= 0 */
  int32_t top_k;              /* routes per token, 1..32 */
  int32_t num_global_experts; /* E_g: valid ids are [0, E_g) */
  int32_t num_local_experts;  /* E_l: experts whose weights are passed, 1..B4_MAX_LOCAL_EXPERTS */
  int32_t hidden;             /* H: multiple of 64 */
  int32_t inter;              /* I: multiple of 32 (NVFP4: 16 suffices for K, 32 for tiling) */
  int32_t format;             /* b4_format */
  int32_t path;               /* b4_path */
  /* Device int32 [E_g] mapping a global expert id to a local expert, or -1;
   * NULL means the identity (then E_g must equal E_l).  flashinfer PR #4255,
   * Tests: "covering expert_map, invalid expert ids". */
  const int32_t* expert_map;
  /* B4_ACT_SWIGLU_OAI only (b4_fused_moe reads them for that activation and
   * ignores them otherwise): alpha and beta finite, limit > 0 (+inf: no
   * clamp); anything else is B4_ERR_INVALID_ARGUMENT. */
  float swiglu_alpha;
  float swiglu_beta;
  float swiglu_limit;
} b4_moe_config;

/* Token capacity the packing and workspace are sized to: next_pow2(max(m, 1))
 * (flashinfer PR #4255, Description: "specialize on a power-of-two capacity
 * instead of the exact token count").  Never fails. */
int32_t b4_route_capacity_tokens(int32_t m);

/* Bytes of workspace b4_fused_moe needs for this configuration and
 * activation.  Depends on m only through b4_route_capacity_tokens(m), so one
 * workspace serves every m up to the next power of two (flashinfer PR #4255,
 * Description: "The W4A16 workspaces are sized to the same capacity").
 * Returns 0 for an invalid configuration (see b4_last_error). */
size_t b4_workspace_bytes(const b4_moe_config* cfg, int32_t activation);

/* Sizes of the prepared (serving-layout) weights of one tensor:
 * which = 0: W13 (SwiGLU) or W1 (ReLU^2), [E_l, N1, H];  which = 1: W2, [E_l, H, I].
 * Writes the code and scale byte counts to *code_bytes and *scale_bytes (host). */
b4_status b4_prepared_sizes(const b4_moe_config* cfg, int32_t which, int32_t activation,
                            size_t* code_bytes, size_t* scale_bytes);

/* Converts checkpoint-layout weights of one tensor into the serving layout
 * b4_fused_moe reads (flashinfer PR #4255, CodeRabbit walkthrough: weight
 * preparation "with layout normalization, ... scale packing, and W13
 * rotation").
 *
 * src_codes  [E_l, N, K/2] uint8, two E2M1 codes per byte, element 2j low nibble.
 * src_scales [E_l, N, K/g] uint8 (E4M3 for NVFP4, g = 16; E8M0 for MXFP4, g = 32).
 * dst_codes, dst_scales: b4_prepared_sizes bytes each, 16-byte aligned.
 * The serving layout tiles rows by 128 and K by 64, pads both with zeros,
 * interleaves gate/up rows in groups of 16 for SwiGLU, reorders the E2M1
 * nibbles of every 8 codes into the pairing of the hardware FP4 conversion,
 * and re-encodes the block scales.
 * Blocks whose scale decodes to zero are stored with zero codes (the product
 * is zero either way); a negative E4M3 scale is folded into the code signs.
 *
 * Offline: this call synchronises `stream` to report invalid scale codes
 * (E4M3 NaN; E8M0 codes of 192 and above, or below 65 in a block with a
 * nonzero code -- scales outside 2^-62 .. 2^64 are outside the range the
 * bf16 dequantiser reproduces exactly) as B4_ERR_INVALID_ARGUMENT.
 * Not capture-safe. */
b4_status b4_prepare_weights(const b4_moe_config* cfg, int32_t which, int32_t activation,
                             const uint8_t* src_codes, const uint8_t* src_scales, uint8_t* dst_codes,
                             uint8_t* dst_scales, b4_stream_t stream);

/* Route packing (flashinfer PR #4255, Description: shape-stable route
 * packing; Tests: expert_map, invalid ids, preallocated buffers).
 *
 * topk_ids [m, top_k] int32.  A route r = t*top_k + j is valid iff
 * 0 <= id < E_g and the local expert l = expert_map[id] (or id) lies in
 * [0, E_l); invalid routes are dropped, never an error.
 * Outputs (caller-allocated):
 *   counts        [E_l]     int32: valid routes per local expert;
 *   offsets       [E_l + 1] int32: exclusive scan of counts, offsets[E_l] = valid routes;
 *   sorted_routes [R_cap]   int32, R_cap = b4_route_capacity_tokens(m) * top_k:
 *                 sorted_routes[offsets[l] + i] = i-th valid route of expert l in
 *                 ascending r (stable); entries past offsets[E_l] are -1.
 * One launch on `stream`; no allocation, no synchronisation (capture-safe).
 * The kernel lets a next kernel launched with programmatic dependent launch
 * start early; such a kernel must wait for it (griddepcontrol.wait) before
 * it reads the outputs. */
b4_status b4_route_pack(const b4_moe_config* cfg, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                        int32_t* sorted_routes, b4_stream_t stream);

/* The fused layer: out = sum_j w[t,j] * FC2_e(act(FC1_e(x[t]))) for the valid
 * routes (t, j), e = local expert of route (t, j), rounded to bf16 once.
 *
 * x             [m, H] bf16.
 * w13, s13      prepared FC1 weights (b4_prepare_weights, which = 0).
 * gs13          [E_l] fp32 global scales of FC1 (NVFP4); must be NULL for MXFP4.
 * w2, s2, gs2   the same for FC2 (which = 1).
 * topk_ids      [m, top_k] int32; topk_weights [m, top_k] fp32.
 * activation    b4_activation (of the layout the weights were prepared for:
 *               SILU_SWIGLU and SWIGLU_OAI share one).
 * out           [m, H] bf16, written in full (tokens without a valid route get 0).
 * workspace     >= b4_workspace_bytes(cfg, activation) bytes, 256-byte aligned;
 *               its contents on entry do not matter.  It holds the status word
 *               read by b4_check_status.
 * FC1 accumulates gs13 * (x . w13) in fp32, applies the activation in fp32 and
 * rounds h to bf16; FC2 accumulates in fp32, multiplies by gs2 and the router
 * weight and sums the routes of a token in fp32 before one bf16 rounding.
 * Enqueues 1 (the small-m path: one cooperative launch of one CTA per SM
 * for m > 4, grid no larger than the resident CTA count for m <= 4) or 4
 * (grouped: route pack with the copy of x rows into packed-route order, FC1,
 * FC2, finalize; the last three chained by programmatic dependent launch)
 * launches on `stream`; no allocation, no
 * synchronisation.  The small-m path's output is bitwise reproducible (every
 * sum in a fixed order); the grouped path's top-k sum uses fp32 atomics. */
b4_status b4_fused_moe(const b4_moe_config* cfg, const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                       const float* gs13, const uint8_t* w2, const uint8_t* s2, const float* gs2,
                       const int32_t* topk_ids, const float* topk_weights, int32_t activation, uint16_t* out,
                       void* workspace, size_t workspace_bytes, b4_stream_t stream);

/* Optional per-kernel timing.  events: host array of n cudaEvent_t handles
 * (created by the caller), or NULL to turn timing off.  While set, each
 * b4_fused_moe call on this thread records events[0] on its stream before its
 * first kernel and events[i+1] after kernel i, as far as n reaches: the
 * decode path launches 1 kernel (FC1, FC2 and the top-k combine fused); the
 * grouped path records 5 (before route pack, after it, after FC1, after
 * FC2, after finalize), so 2 and 5 events cover them.  b4_linear records 2 (small m), 4 (K-split GEMM: before the memset,
 * after the route pack, after the GEMM, after the rounding pass) or 3.  An event recorded between two kernels removes their programmatic
 * overlap, so timed calls can be slightly slower than untimed ones; use this
 * for measurement.
 * Returns B4_ERR_INVALID_ARGUMENT when n == 1 or events is NULL with n > 0. */
b4_status b4_set_timing_events(void* const* events, int32_t n);

/* Optional kernel timeline for profiling: while `device_buffer` is set
 * (>= 262144 bytes = [16][2048] int64, or NULL to turn it off), the kernels
 * of each b4_fused_moe / b4_linear call on this thread write timestamps into
 * it.  Grouped path (built with B4_TRACE defined only; otherwise nothing is
 * written): clock64() of CTA 0 as [5][2048] per GEMM, indexed by the CTA's
 * running counters, FC1 at int64 offset 0 and FC2 at 10240; kinds: weight
 * stage issued, A stage written to tensor memory (weights on M) or B stage
 * dequantised (weights on N), MMA stage issued, activation stage ready, unit
 * epilogue done.  Small-m path (one kernel), route-grouped kernel:
 * %globaltimer nanoseconds of each CTA at phase boundaries, entry [kind][CTA]:
 * 0 start, 1 group table built, 2 first unit published, 3 first weight copy
 * issued, 4 first slot computed, 5 last FC1 unit stored, 6 first FC2 slot
 * computed, 7 compute done, 8 epilogue done, 9 first FC2 unit's FC1 tiles
 * ready, 10 grid barrier seen, 11 weight stream done, 12 last FC1 tile's h
 * built, 13 last output row written, 14 buffers filled, 15 route ids read.
 * Per-route kernel: clock64() of CTA 0 as [kind][index] for kinds 0 (weight
 * slot issued), 1 (slot computed), 2 (start), 3 (unit begun), 4 (unit
 * done); %globaltimer of each CTA for kinds 5 (start), 6 (last FC2 partial
 * stored), 7 (last FC1 partial stored), 8 (compute done), 9 (output warp
 * done), 11 (first slot computed), 12 (first x row converted), 13 (grid
 * barrier complete), 14 (first unit's weights issued), 15 (first slot
 * landed); kind 10 holds each CTA's SM.  Entries not reached are left
 * untouched. */
b4_status b4_set_trace(void* device_buffer, size_t bytes);

/* Synchronises `stream`, then reads the device status word of `workspace`
 * (written by b4_fused_moe's kernels): B4_OK, or B4_ERR_TIMEOUT if a bounded
 * device wait ran out.  Resets the word to B4_OK.  Not capture-safe. */
b4_status b4_check_status(void* workspace, b4_stream_t stream);

/* Diagnostic of the device failure path (no passage of the pages defines it:
 * it exercises the bounded waits every kernel above relies on).  Enqueues on
 * `stream` one CTA that waits, through the same bounded-wait routine the
 * kernels use, on an mbarrier phase that no thread completes, with a limit of
 * `limit_us` microseconds.  When the limit runs out the kernel writes
 * B4_ERR_TIMEOUT and wait site 90 into the status word at the start of
 * `workspace` (device memory, at least 8 bytes, caller-owned) and exits
 * normally: it never traps and never waits longer than the limit.  Read the
 * result with b4_check_status.  Returns B4_ERR_INVALID_ARGUMENT for a NULL or
 * short workspace or a limit outside 1 .. 1000000 us, otherwise B4_OK once
 * launched (B4_ERR_CUDA if the launch fails).  Capture-safe. */
b4_status b4_wait_self_test(void* workspace, size_t workspace_bytes, uint32_t limit_us, b4_stream_t stream);

/* Allocation-free variant of b4_fused_moe.  The paper has no counterpart:
 * the layer it describes always takes its scratch from the caller.
 *
 * Who needs it: code that runs as a plugin hook of an inference runtime or as
 * a custom-op slot of a framework receives only its input and output buffers.
 * The host's allocator owns all device memory there; a cudaMalloc from inside
 * the hook would stall the whole device on the serving path and bypass the
 * host's memory accounting, so such code must not allocate and has no
 * workspace to give to b4_fused_moe.
 *
 * What it does: the same kernels and results as b4_fused_moe, with the
 * scratch taken from one array of B4_NOALLOC_SCRATCH_BYTES (64 MiB) that the
 * library declares in device memory.  The CUDA runtime places that array on
 * every GPU where it loads this library's device code, and it stays there
 * until the process exits.  This call never calls cudaMalloc, cudaFree or any
 * allocating library routine.
 *
 * Arguments: as b4_fused_moe, without workspace and workspace_bytes, plus
 * device_status: NULL, or 2 uint32 of device memory (4-byte aligned) that
 * receive this call's device status word in stream order -- status
 * (B4_OK or B4_ERR_TIMEOUT) and the wait site -- which b4_check_status would
 * otherwise read from a workspace.
 *
 * Limit: a shape whose b4_workspace_bytes exceeds B4_NOALLOC_SCRATCH_BYTES is
 * refused with B4_ERR_WORKSPACE_TOO_SMALL before anything is launched, and
 * b4_last_error gives both sizes; use b4_fused_moe for it.  With H = 4096,
 * I = 1536 and top_k = 8, 64 MiB holds the decode path (m <= 64) and the
 * grouped path up to m = 256.
 *
 * Set-up: the first call on each device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress, which may load the
 * library's device code onto that device) and keeps it with the id of the
 * context it was found in.  Make that first call before any stream capture
 * begins on the device.  A call in a different context on that device (after
 * cudaDeviceReset, or a teardown and re-creation of the primary context,
 * which may place the array elsewhere) looks the address up again, so a
 * stale address is never used; make that call, too, outside stream capture.
 *
 * Sharing: all calls on a device use the same array, and each call leaves its
 * contents behind.  Every part of it that a call reads is written earlier in
 * the same call (the status word by the first kernel, the fp32 top-k
 * accumulator by FC1 before FC2 adds into it), so calls ordered on one stream
 * do not see each other's data.  Calls that can run at the same time on the
 * GPU -- on two streams with no event between them, or from two host threads
 * -- race on the array and produce wrong results: keep them on one stream or
 * order them. */
#define B4_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
b4_status b4_fused_moe_noalloc(const b4_moe_config* cfg, const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                               const float* gs13, const uint8_t* w2, const uint8_t* s2, const float* gs2,
                               const int32_t* topk_ids, const float* topk_weights, int32_t activation,
                               uint16_t* out, uint32_t* device_status, b4_stream_t stream);

/* Dense W4A16 linear layer: one FP4 weight matrix W [N, K], bf16 x, no
 * routing and no activation -- the dense W4A16 GEMM with a capture-safe
 * small-M dispatch and caller-owned buffers of b12x PR #136, "fix(gemm):
 * restore capture-safe K6 small-M dispatch" (Summary), here on this
 * library's FP4 weights: the E = 1, top-1 case of the FC1 GEMM with the
 * activation left out.
 *   out[t][n] = bf16( gs * sum_k x[t][k] * W[n][k] ),  t < m, n < N,
 * W[n][k] = e2m1(code) * block scale (E4M3 per 16 or E8M0 per 32 along K),
 * accumulated in fp32 and rounded to bf16 once.
 *
 * cfg           m = tokens, hidden = K, inter = N, top_k = 1,
 *               num_global_experts = num_local_experts = 1, expert_map NULL,
 *               format, path (AUTO: the fused small-m kernels for m <= 16 --
 *               per-route for m <= 4, route-grouped above -- and the grouped
 *               tcgen05 GEMM beyond; DECODE is accepted for m <= B4_DECODE_MAX_M).
 * w, s          W prepared by b4_prepare_weights(cfg, which = 0,
 *               B4_ACT_RELU2, ...) -- the non-gated FC1 layout of one expert.
 * gs            [1] fp32 global scale (NVFP4); NULL for MXFP4.
 * x             [m, K] bf16; out [m, N] bf16, written in full.
 * workspace     >= b4_linear_workspace_bytes(cfg) bytes, 256-byte aligned;
 *               contents on entry do not matter; holds the status word.
 * Enqueues on `stream`: 1 cooperative launch (small m); or, when the GEMM
 * has fewer (token chunk, 256-row tile pair) units than SMs, 4 operations
 * (a memset of an fp32 accumulator, the route pack of the trivial routing,
 * the GEMM with K split across units adding fp32 partials, and a rounding
 * pass); otherwise 2-3 (route pack, the GEMM storing bf16, and a strided
 * device copy when N is not a multiple of 64).  No allocation, no
 * synchronisation (capture-safe).  Shape errors: B4_ERR_INVALID_ARGUMENT
 * before any launch. */
size_t b4_linear_workspace_bytes(const b4_moe_config* cfg);
b4_status b4_linear(const b4_moe_config* cfg, const uint16_t* x, const uint8_t* w, const uint8_t* s,
                    const float* gs, uint16_t* out, void* workspace, size_t workspace_bytes, b4_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* b4_status_string(int32_t status);

/* Thread-local message describing the last error returned on this thread. */
const char* b4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* B4MOE_H */
