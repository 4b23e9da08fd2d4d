/*
 * moe.h -- C ABI of the single-GPU MoE-layer forward for GB300 (sm_103a).
 *
 * The operation (from "Mixture-of-Kittens: MoE Megakernel for NVL72s",
 * Sec. 2.1, Eq. "MoE", and the vendor blog's E_i(x) with SiLU):
 *
 *   MoE(x) = f_shared(x) + sum_{i in E(x)} g_i f_i(x),   g_i = s_i / sum_{j in E(x)} s_j,
 *   f_i(x) = W_down^(i) ( SiLU(W_gate^(i) x) * W_up^(i) x ),
 *
 * E(x) = the k routed experts with the highest router score s = score(W_r x + b)
 * (score = sigmoid, or softmax over all experts).  All experts are on this GPU:
 * the paper's cross-GPU dispatch/combine become an on-device gather into a
 * fixed-size ring of minibatches and a scatter back to token order.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers on the plan's device;
 *     the caller owns all memory (inputs, outputs, workspace) and the stream.
 *   - Matrices are row-major; every weight is K-major (its contraction
 *     dimension contiguous), exactly the shapes of Sec. 2.1: W_up, W_gate in
 *     R^{I x D}, W_down in R^{D x I}; expert e's matrix is block e of the
 *     stacked [E, ...] array.
 *   - bf16 = IEEE bfloat16 bit patterns (2 bytes).
 *   - Calls are asynchronous on `stream`, allocate nothing on the device, do
 *     not synchronise the host, and never read device memory on the host;
 *     device-side failures are reported through moe_get_status().
 *   - Return value: MOE_OK (0) or a negative moe_error; no C++ exception
 *     crosses this interface.
 *   - Plans are immutable after creation and may be shared by threads; one
 *     workspace must not be used by two forwards that overlap on the GPU.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum moe_error {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* null pointer, T > T_max, bad enum value */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* shape outside the limits listed at moe_config */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3,
  MOE_ERR_CUDA = -4,               /* a CUDA runtime call failed (launch, copy, attribute) */
  MOE_ERR_UNSUPPORTED_DEVICE = -5, /* the current device is not sm_103 */
  MOE_ERR_STATIC_SCRATCH_TOO_SMALL = -6 /* moe_route_static: request exceeds its fixed scratch */
} moe_error;

typedef enum moe_device_status {
  MOE_STATUS_OK = 0,
  MOE_STATUS_TIMEOUT = 1,          /* a device-side wait exceeded its limit; outputs are invalid */
  MOE_STATUS_SCHEDULE_INVALID = 2, /* an expert index out of range or route counts inconsistent */
  MOE_STATUS_STAGING_OVERFLOW = 3  /* the forward completed, but an expert output left the fp16 range of
                                      the staging rows (|v| > 65504, or NaN) and was saturated: the
                                      output is finite but not the layer's value */
} moe_device_status;

typedef enum moe_score_fn { MOE_SCORE_SIGMOID = 0, MOE_SCORE_SOFTMAX = 1 } moe_score_fn;
typedef enum moe_precision { MOE_PREC_BF16 = 0, MOE_PREC_MXFP8 = 1 } moe_precision;
typedef enum moe_dispatch { MOE_DISPATCH_RING = 0, MOE_DISPATCH_DIRECT = 1, MOE_DISPATCH_SPREAD = 2 } moe_dispatch;

/*
 * Layer shape and execution knobs.
 *   T_max  largest token count a forward will be called with (>= 1)
 *   D      hidden size, multiple of 256
 *   I      routed-expert intermediate size, multiple of 128
 *   E      routed experts, 1..512
 *   k      experts per token, 1..min(16, E)
 *   I_s    shared-expert intermediate size, multiple of 128, or 0 (no shared expert)
 *   score_fn   moe_score_fn
 *   precision  moe_precision of the routed experts (the router and the shared
 *              expert always run in bf16, Sec. 3.4 "MXFP8 Support")
 *   minibatch  b: routes per minibatch of the dispatch ring, multiple of 128,
 *              128..32768 (Sec. 3.2 sweeps 512..32768)
 *   ring_slots minibatch slots in the ring (>= lag + 1); ring_slots * minibatch
 *              >= T*k gives the over-allocated (no wrap) buffer of Sec. 3.3
 *   dispatch   MOE_DISPATCH_RING: gather CTAs copy the routed tokens into the
 *              ring of minibatches (the pages' communication SMs);
 *              MOE_DISPATCH_DIRECT: the GEMM CTAs' TMA producers fetch each
 *              tile's token rows straight from x (tile::gather4), no gather
 *              CTAs and no x ring (MXFP8: from the router pass's x codes);
 *              MOE_DISPATCH_SPREAD: the same ring as MOE_DISPATCH_RING, filled
 *              by two otherwise idle warps of every GEMM CTA (each takes the
 *              minibatch's M-tiles c, c + gemm CTAs, ...), so every SM runs
 *              expert tiles; gather_ctas is ignored
 *   gather_ctas  ring dispatch: CTAs (one per SM) that only gather tokens, >= 1
 *              (Sec. 3.4 "Computation-Communication SM Tuning"); ignored for
 *              direct dispatch
 *   gemm_ctas  CTAs that run expert GEMMs; 0 = all remaining SMs
 *   lag        0: down projections of minibatch m follow its up/gate tiles;
 *              1: they follow the up/gate tiles of minibatch m + 1
 *   timeout_ms limit of every device-side wait (0 = 2000 ms)
 *   l2_prefetch  K steps ahead that the GEMM producers prefetch operand tiles
 *              into L2 (0 = off, the default: on DSV3 it measured slower)
 *   mma_pair   1: the GEMM CTAs run as pairs (clusters of 2) and each expert
 *              tile is one tcgen05.mma.cta_group::2 of 256 rows, the pair's
 *              two 128-row M-tiles sharing the weight tile, each CTA loading
 *              half of it (half the operand bytes per SM of the one-CTA tile);
 *              a segment with an odd number of M-tiles pads its last pair.
 *              With mxfp8 the scale blocks of both CTAs' rows travel with the
 *              pair's loads and every CTA holds the weight tile's scales for
 *              all 256 columns.  Ring or spread dispatch (direct gives
 *              MOE_ERR_INVALID_ARG); gather_ctas must be even.  Results are
 *              bitwise those of the one-CTA tiles.  0: one CTA per tile.
 *   clc        1: the GEMM CTAs take their work tokens from cluster launch
 *              control (MoK Sec. 3.4 "RDMA Overlap via Cluster Launch
 *              Control"): the kernel is launched with one CTA per task beyond
 *              the gather CTAs, not cooperatively; each running CTA cancels
 *              the launch of a CTA that has not started and takes its token,
 *              so when the hardware declines (a higher-priority stream wants
 *              the SM) the CTA finishes its unit and leaves, and CTAs launched
 *              later take the remaining units.  Which unit a token buys still
 *              comes from the global counter in task order, so results are
 *              bitwise those of the default scheduling.  One CTA per tile only
 *              (mma_pair = 1 gives MOE_ERR_INVALID_ARG).  0: the persistent
 *              cooperative grid claims units from the counter alone.
 *   test_unfilled_minibatch  test hook for the bounded waits, 0 in normal
 *              use: n >= 1 makes the ring fill never mark minibatch n - 1 as
 *              gathered, so the expert tiles waiting for it give up after
 *              timeout_ms and the forward ends with MOE_STATUS_TIMEOUT (the
 *              kernels return normally, the stream stays usable).  Ring or
 *              spread dispatch only (direct gives MOE_ERR_INVALID_ARG).
 *   pad_odd_tiles  CTA pairs: 1 pairs an expert segment's odd last M-tile with
 *              an empty partner (one M = 256 MMA, 128 of its rows zero); 0 =
 *              the default: with bf16 precision the tile is split over the
 *              pair instead (one M = 128 MMA, 64 rows per CTA: half the A
 *              bytes and half the tensor time of the padded form).  MXFP8
 *              pairs always pad.  Results are bitwise the same either way.
 *   plain_launch  profiling aid, 0 in normal use: 1 launches the persistent
 *              kernel without the cooperative attribute (profilers that replay
 *              kernels cannot launch a cooperative cluster kernel).  Its CTAs
 *              still wait on each other, so the grid (sized to what fits on
 *              the GPU at once) must all be resident, which it is when nothing
 *              else runs on the GPU; every wait is bounded, so a grid that
 *              did not fit ends the forward with MOE_STATUS_TIMEOUT.  Ignored
 *              with clc (never cooperative).
 *   raster     order of an expert segment's up/gate tiles: groups of `raster`
 *              M-tiles, each group sweeping all I/128 column tiles (so a
 *              group's token rows are re-read from L2 while its weight
 *              slices stream); 0 = the library default, >= the segment's
 *              M-tile count = column-tile major over the whole segment.  With
 *              mma_pair it is rounded up to even.  Results do not depend on it.
 * Zero for minibatch / ring_slots / gather_ctas / lag picks the defaults
 * (8192 / 4 / 8 / 1).
 */
typedef struct moe_config {
  int64_t T_max;
  int64_t D;
  int64_t I;
  int64_t E;
  int64_t k;
  int64_t I_s;
  int32_t score_fn;
  int32_t precision;
  int32_t minibatch;
  int32_t ring_slots;
  int32_t gather_ctas;
  int32_t gemm_ctas;
  int32_t lag;
  int32_t timeout_ms;
  int32_t dispatch;
  int32_t l2_prefetch;
  int32_t mma_pair;
  int32_t raster;
  int32_t test_unfilled_minibatch;
  int32_t clc;
  int32_t plain_launch;
  int32_t pad_odd_tiles;
} moe_config;

/*
 * Layer parameters (device pointers).
 *   W_router [E, D] bf16;  b_router [E] fp32 or NULL (no bias; the bias is
 *   added to the logits before the score function)
 *   bf16 precision:  W_up, W_gate [E, I, D] bf16;  W_down [E, D, I] bf16;
 *                    the *_scale pointers are ignored
 *   MXFP8 precision: W_up, W_gate [E, I, D] and W_down [E, D, I] E4M3 codes
 *                    (1 byte), and *_scale the E8M0 block scales written by
 *                    moe_quantize_mxfp8 for the same matrices
 *   Ws_up, Ws_gate [I_s, D] bf16; Ws_down [D, I_s] bf16; all three NULL = no
 *   shared expert in this call (required when I_s = 0)
 */
typedef struct moe_weights {
  const void* W_router;
  const float* b_router;
  const void* W_up;
  const void* W_gate;
  const void* W_down;
  const uint8_t* W_up_scale;
  const uint8_t* W_gate_scale;
  const uint8_t* W_down_scale;
  const void* Ws_up;
  const void* Ws_gate;
  const void* Ws_down;
} moe_weights;

/*
 * Outputs (device pointers).  `out` is required; every other field may be
 * NULL (not exported).
 *   out            [T, D] bf16: MoE(x)
 *   topk_idx       [T, k] int32: selected experts, ascending id per token
 *   topk_w         [T, k] fp32: g, same order
 *   expert_counts  [E] int32: M_e, routes per expert (Algorithm 1)
 *   expert_offsets [E + 1] int32: S_e, exclusive prefix of M (S_E = T*k)
 *   sched          [T*k, 3] int32: schedule table row P = {src_index t,
 *                  expert e, dst_index j = t*k + slot}, rows sorted by expert
 *                  then token (Algorithm 1 with one rank)
 *   route_row      [T*k] int32: inverse of sched, route j -> row P
 */
typedef struct moe_outputs {
  void* out;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* expert_counts;
  int32_t* expert_offsets;
  int32_t* sched;
  int32_t* route_row;
} moe_outputs;

typedef struct moe_plan moe_plan;

/*
 * Validate `cfg` for the current CUDA device and create a plan.
 * Errors: MOE_ERR_INVALID_ARG (null), MOE_ERR_UNSUPPORTED_SHAPE,
 * MOE_ERR_UNSUPPORTED_DEVICE, MOE_ERR_CUDA.  *out is NULL on failure.
 * Host memory only; the caller releases it with moe_plan_destroy.
 */
int moe_plan_create(const moe_config* cfg, moe_plan** out);

/* Release a plan (NULL is accepted).  Returns MOE_OK. */
int moe_plan_destroy(moe_plan* plan);

/* Bytes of device workspace a forward of T tokens needs (0 on bad input).
 * The workspace holds the routing results, the schedule, the task list, the
 * dispatch ring, the gated activations and the token-order staging rows. */
size_t moe_workspace_bytes(const moe_plan* plan, int64_t T);

/*
 * MXFP8 weight pre-quantisation (Sec. 3.4 "MXFP8 Support", OCP MX v1.0):
 * W [rows, K] bf16 (device), rows and K multiples of 128 -> q [rows, K] E4M3
 * codes and scales (E8M0, one per 32 consecutive K elements),
 * moe_mxfp8_scale_bytes(rows, K) = rows * K / 32 bytes.  Block scale
 * X = 2^(floor(log2 amax) - 8), elements rounded to nearest-even and saturated
 * at +-448; an all-zero block gets X = 2^-127.  Scale layout: 512-byte blocks
 * ordered [rows/128][K/128], each holding 128 rows x 4 blocks of 32 with the
 * scale of (row r, block kb) at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + kb
 * (the layout the block-scaled tensor-core MMA reads).  A stacked [E, I, D]
 * weight is quantised as rows = E * I.  Asynchronous on `stream`.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_CUDA.
 */
int moe_quantize_mxfp8(const moe_plan* plan, const void* W, int64_t rows, int64_t K, uint8_t* q,
                       uint8_t* scales, moe_stream_t stream);
size_t moe_mxfp8_scale_bytes(int64_t rows, int64_t K);

/*
 * The forward pass for T tokens (0 <= T <= T_max; T = 0 does nothing).
 *   x          [T, D] bf16 (device)
 *   w          layer parameters, see moe_weights
 *   o          outputs, see moe_outputs
 *   workspace  device memory of at least moe_workspace_bytes(plan, T) bytes,
 *              256-byte aligned; its contents need no initialisation
 * Launches, in order on `stream`: router + top-k (for MXFP8 it also
 * quantises x per token), schedule, persistent forward kernel -- three
 * kernels, no host synchronisation.  Two calls on identical
 * inputs give bitwise-identical outputs, also across minibatch, ring_slots,
 * gather_ctas, gemm_ctas and lag settings.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA.
 */
int moe_fwd(const moe_plan* plan, int64_t T, const void* x, const moe_weights* w, const moe_outputs* o,
            void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Read the device status of the last forward that used `workspace` (a
 * moe_device_status: a failure if one was recorded, else
 * MOE_STATUS_STAGING_OVERFLOW if that warning was raised, else MOE_STATUS_OK).
 * This call waits for `stream` to finish: it is the one host synchronisation
 * point, taken only when the caller asks.
 */
int moe_get_status(const moe_plan* plan, const void* workspace, int* device_status, moe_stream_t stream);

/*
 * Optional per-launch timing for profiling harnesses: with events != NULL,
 * every later moe_fwd with this plan records events[0] (cudaEvent_t) on its
 * stream before the router launch, events[1] after it, events[2] after the
 * schedule launch and events[3] after the persistent kernel; events == NULL
 * turns it off.  The caller owns the events.  Not to be called while another
 * thread runs moe_fwd with the same plan.
 */
int moe_plan_set_timing_events(moe_plan* plan, void* const* events);

/*
 * Optional phase timing for profiling harnesses: the persistent kernel of the
 * last forward that used `workspace` stamps, with the GPU's global timer, when
 * its first CTA started, when the last minibatch was marked gathered (ring or
 * spread dispatch), and when the final combine pass began (the first CTA to
 * start it) and ended (the last CTA to finish it).  times_ms[0..2] receive the
 * last three as milliseconds after the start (-1 where a phase did not
 * happen).  Like moe_get_status, this call waits for `stream` to finish.
 */
int moe_get_phase_times(const moe_plan* plan, const void* workspace, double* times_ms, moe_stream_t stream);

/*
 * Routing stage without any device allocation -- no counterpart in the paper.
 *
 * For callers that cannot call cudaMalloc themselves and cannot hand over a
 * workspace: code embedded in a framework whose allocator owns all device
 * memory, or latency-critical loops where an allocation (which can
 * synchronise the device) is not allowed.  It runs the same router + top-k
 * and schedule kernels as moe_fwd, but their scratch (per-chunk expert
 * histograms, counters, status word, schedule-builder lists) lives in one
 * fixed array inside the library, moe_route_static_scratch_bytes() bytes
 * (512 KiB), that every GPU which loads the library keeps until the process
 * exits.  Limits: T <= MOE_ROUTE_STATIC_MAX_TOKENS (and <= the plan's T_max);
 * larger requests return MOE_ERR_STATIC_SCRATCH_TOO_SMALL and launch nothing.
 *   x [T, D] bf16, W_router [E, D] bf16, b_router [E] fp32 or NULL (device)
 *   outputs (device, all required): topk_idx [T, k] int32, topk_w [T, k] fp32,
 *   expert_counts [E], expert_offsets [E + 1], sched [T*k, 3], route_row [T*k]
 *   (int32, same meaning as in moe_outputs); device_status: optional device
 *   int32 that receives the call's moe_device_status.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array, which keeps the previous call's
 * contents (the kernels clear what must start at zero): calls that overlap on
 * the GPU -- on two streams, or from two threads -- race with each other.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_STATIC_SCRATCH_TOO_SMALL, MOE_ERR_CUDA.
 */
#define MOE_ROUTE_STATIC_MAX_TOKENS 16384
int moe_route_static(const moe_plan* plan, int64_t T, const void* x, const void* W_router, const float* b_router,
                     int32_t* topk_idx, float* topk_w, int32_t* expert_counts, int32_t* expert_offsets,
                     int32_t* sched, int32_t* route_row, int32_t* device_status, moe_stream_t stream);
size_t moe_route_static_scratch_bytes(void);

/*
 * Gradients of the layer (device pointers), written by moe_bwd.
 *   dx        [T, D] bf16: dL/dx (required)
 *   dW_router [E, D] fp32: dL/dW_r (required)
 *   db_router [E] fp32: dL/db, or NULL (not exported)
 *   dW_up, dW_gate [E, I, D] bf16; dW_down [E, D, I] bf16 (required)
 *   dWs_up, dWs_gate [I_s, D] bf16; dWs_down [D, I_s] bf16: the shared
 *   expert's, required when the forward had a shared expert, else NULL
 */
typedef struct moe_grads {
  void* dx;
  float* dW_router;
  float* db_router;
  void* dW_up;
  void* dW_gate;
  void* dW_down;
  void* dWs_up;
  void* dWs_gate;
  void* dWs_down;
} moe_grads;

/* Bytes of device workspace moe_bwd needs for T tokens (0 on bad input or a
 * shape the backward does not support: I and I_s must be multiples of 256). */
size_t moe_bwd_workspace_bytes(const moe_plan* plan, int64_t T);

/*
 * The backward pass ("Mixture-of-Kittens: MoE Megakernel for NVL72s",
 * Sec. 3.3 "Ring-Aware Forward Replay" and Sec. 3.4 "Router Weight Gradient
 * Computation"): given dO = dL/d out for the forward that moe_fwd computed on
 * the same x and weights with `fwd_workspace` (its routing and schedule are
 * reused, unmodified, from that workspace), writes every gradient of
 * moe_grads by the chain rule on Eq. MoE:
 *   dy_j = g_j dO;  dg_j = <W_down[e]^T dO, h>  (the SonicMoE form: the
 *   expert output is never materialised);  dh = g_j W_down[e]^T dO;
 *   da_u = dh * SiLU(a_g);  da_g = dh * a_u * SiLU'(a_g);
 *   dW_down[e] = sum dy h^T;  dW_up[e] = sum da_u x^T;  dW_gate[e] = sum da_g x^T;
 *   dx = sum_j (W_up[e]^T da_u + W_gate[e]^T da_g) + shared expert + W_r^T dl,
 *   with dl from g = s_sel / sum s_sel through the score function.
 * The gated activations are recomputed (the forward replay): every route's
 * up/gate projections run again from the gathered x rows.  BF16 routed
 * experts only (MOE_ERR_UNSUPPORTED_SHAPE for an MXFP8 plan).  No
 * floating-point atomics: every gradient element is produced by one tile with
 * a fixed K order or by a fixed-order sum, so two calls give the same bits.
 *   dO         [T, D] bf16 (device)
 *   workspace  at least moe_bwd_workspace_bytes(plan, T) bytes, 256-byte aligned
 * Launches eight kernels on `stream`; no host synchronisation; device-side
 * failures are reported through moe_get_status on `workspace`.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE,
 * MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA.
 */
int moe_bwd(const moe_plan* plan, int64_t T, const void* x, const moe_weights* w, const void* dO,
            const void* fwd_workspace, const moe_grads* grads, void* workspace, size_t workspace_bytes,
            moe_stream_t stream);

/*
 * Optional per-phase timing of moe_bwd for profiling harnesses: with events
 * != NULL, every later moe_bwd with this plan records events[0] before its
 * first launch, events[1] after the gather of the routes' x and dO rows,
 * events[2] after the replay + activation-gradient GEMMs, events[3] after the
 * input- and weight-gradient GEMMs and events[4] after its last launch;
 * NULL turns it off.  The caller owns the events (cudaEvent_t).
 */
int moe_plan_set_bwd_timing_events(moe_plan* plan, void* const* events);

/* Static description of an error code. */
const char* moe_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
