// Shared definitions of the MoE forward kernels: launch parameters, the task
// record the schedule kernel writes for the persistent kernel, workspace
// sections and bounded device-side waits.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace moe {

typedef __nv_bfloat16 bf16;

// GEMM tiling shared by all tcgen05 kernels
constexpr int BM = 128;          // rows (tokens) per tile = UMMA M
constexpr int BK = 64;           // K per stage = one 128-byte swizzle atom of bf16
constexpr int UMMA_K = 16;       // K per tcgen05.mma for 16-bit inputs
constexpr int BN_UP = 128;       // intermediate columns per GEMM1 tile (x2: up and gate)
constexpr int BN_DOWN = 256;     // output columns per GEMM2 tile
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;        // 16 KB (= 128 rows x 128 B, also in MXFP8)
constexpr int B_STAGE_BYTES = 256 * BK * 2;       // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
// MXFP8: a K step is 128 E4M3 codes (one 128-byte swizzle atom per row) plus
// the E8M0 scale blocks of A (512 B) and of B's two 128-row halves (1 KB)
constexpr int BK_MX = 128;
constexpr int SF_BLOCK_BYTES = 512;               // 128 rows x 4 K-blocks of 32
constexpr int SF_STAGE_BYTES = 3 * SF_BLOCK_BYTES;
constexpr int MX_STAGE_TX = STAGE_BYTES + SF_STAGE_BYTES;
constexpr int STAGE_STRIDE = 51200;               // 1024-aligned stage pitch (BF16 and MXFP8)
static_assert(STAGE_BYTES + SF_STAGE_BYTES <= STAGE_STRIDE && STAGE_STRIDE % 1024 == 0, "stage pitch");
// CTA pairs (cta_group::2): each CTA stages its 128 A rows and half of the
// 256 B rows (up or gate for GEMM1, one half of the output columns for GEMM2)
constexpr int PAIR_B_STAGE_BYTES = 128 * BK * 2;  // 16 KB
constexpr int PAIR_STAGE_BYTES = A_STAGE_BYTES + PAIR_B_STAGE_BYTES;  // 32 KB per CTA
constexpr int PAIR_STAGES = 7;  // BF16 pairs: the epilogue stores rows from registers, no staging blocks
// CTA pairs, MXFP8 routed tiles: per CTA and stage its A codes and its half
// of B's codes in the 32 KB stage, and in a separate array of 1.5 KB slots
// (one per stage, after the stages) the A scale block of its rows and B's two
// scale blocks (each CTA needs the scales of all 256 B rows).  Keeping the
// scales out of the 1024-aligned stages leaves room for six stages.
constexpr int PAIR_MX_STAGE_TX = PAIR_STAGE_BYTES + SF_STAGE_BYTES;  // 33.5 KB
constexpr int PAIR_MX_STAGES = 6;
constexpr int ACC_COLS = 256;    // fp32 accumulator columns per tile
constexpr int MEGA_THREADS = 256;  // 8 warps
constexpr int ROUTER_THREADS = 256;
constexpr int SCHED_THREADS = 512;
constexpr int TOPK_MAX = 16;
constexpr int E_MAX = 512;

// device status codes (written to the workspace status word)
enum : int { STATUS_OK = 0, STATUS_TIMEOUT = 1, STATUS_SCHEDULE_INVALID = 2 };
// sticky warning bits in the word after the status word: they do not stop the
// forward (the status word does), they only qualify its result
enum : int { FLAG_STAGING_OVERFLOW = 1 };

// phase stamps of one persistent-kernel launch (ns of %globaltimer), for
// per-phase bandwidth figures: the first CTA's start, the last ring fill, the
// first CTA to start the combine and the last to finish it
enum : int { STAMP_START = 0, STAMP_LAST_FILL = 1, STAMP_COMBINE_START = 2, STAMP_COMBINE_END = 3, N_STAMPS = 4 };
constexpr int STATUS_AREA_BYTES = 256;  // status word, warning bits (8 B), then the stamps (8-byte aligned)

// task kinds of the persistent kernel
enum : int { TASK_R1 = 0, TASK_R2 = 1, TASK_S1 = 2, TASK_S2 = 3 };

struct __align__(16) Task {  // 64 bytes
  int kind;        // TASK_*
  int n;           // output column tile
  int e;           // routed expert (0 for the shared expert)
  int a_row;       // row coordinate of the A operand in its tensor map
  int rows;        // valid rows of the tile (<= BM)
  int p0;          // first schedule row (routed) / first token (shared)
  int out_row;     // first output row (R1: ring_h row, S1/S2: token)
  int dep0, need0; // wait until counters[dep0] >= need0 (dep < 0: none)
  int dep1, need1;
  int done0, done1;  // counters incremented when the tile is stored (-1: none)
  int mt;            // global M-tile index (routed) / token tile (shared)
  int half;          // 1: one 64-row half of a routed M-tile that the pair runs as one M = 128 MMA
  int pad;
};
static_assert(sizeof(Task) == 64, "task record is 64 bytes");

// meta block written by the schedule kernel (int32 offsets)
enum : int { META_N_TASKS = 0, META_N_MTILES = 1, META_TOTAL_Y = 2 /* real R2 and S2 tasks */, META_MB = 4 };
// per minibatch m, META_MB + 4 m + {0: R1 task count, 1: R2 task count,
// 2: first M-tile, 3: M-tile count}

struct FwdParams {
  int T, D, I, E, k, I_s;
  int kY;               // staging slots per token: k routed, plus 1 for the shared expert's output
  int score_fn;
  int mx;               // routed experts in MXFP8 (1) or BF16 (0)
  int direct;           // 1: GEMM producers gather A rows from x themselves (no gather CTAs, no x ring)
  int pair;             // 1: GEMM CTAs run as pairs, tasks 2i and 2i + 1 share one cta_group::2 MMA
  int plain_launch;     // 1: the persistent kernel is launched without the cooperative attribute (profiling)
  int half_tiles;       // 1: a segment's odd last M-tile is split over the pair (BF16 CTA pairs)
  int spread;           // 1: two spare warps of every GEMM CTA fill the ring (no gather CTAs)
  int gparts;           // parts the ring fill of a minibatch is split into (gather CTAs or GEMM CTAs)
  int raster;           // M-tiles per group of a segment's up/gate tiles (column tiles swept per group)
  int b, slots, G, n_gemm, lag;
  int n_mb, R;          // minibatches, routes (T*k)
  int N1, N2, N1s, N2s; // column tiles: I/128, D/256, I_s/128, D/256
  int n_chunks;         // router tiles = ceil(T/128)
  int n_router_cols;    // E rounded up (MMA N of the router)
  int n_mtiles_max, n_smtiles, n_tasks_max;
  int n_counters;
  int l2_prefetch;      // K steps ahead that the producer prefetches into L2 (0 = off)
  int test_unfilled;    // test hook: 0 off; m + 1 = minibatch m is never marked gathered
  int clc;              // 1: GEMM CTAs get their work tokens from cluster launch control (one-CTA kernel)
  long long timeout_ns;
  // inputs
  const bf16* x;
  const float* b_router;
  // workspace sections
  int* status;        // [0] moe_device_status, [1] FLAG_* warning bits; both zeroed by the router kernel
  unsigned long long* stamps;  // [STAMP_*] %globaltimer phase stamps of the persistent kernel (reset by the router)
  int* counters;      // zeroed by the router kernel
  int* meta;
  int* topk_idx;      // [T,k]
  float* topk_w;      // [T,k]
  float* topk_logit;  // [T,k] the selected experts' biased fp32 logits (kept for the backward pass), or null
  int* chunk_counts;  // [n_chunks, E]
  int* M;             // [E]
  int* S;             // [E+1]
  int* sched;         // [R,3] {src_index t, expert e, dst_index j}
  int* route_row;     // [R]
  int* mtiles;        // [n_mtiles_max, 4] {e, p0, rows, m}, row order
  int* segs;          // scratch for the task builder
  Task* tasks;        // [n_tasks_max]
  bf16* ring_x;       // [slots*b, D] (MXFP8: E4M3 codes, 1 byte each)
  bf16* ring_h;       // [slots*b, I] (MXFP8: E4M3 codes)
  uint8_t* sfx;       // MXFP8 ring dispatch: scale blocks of the gathered x, [n_mtiles_max][D/128][512 B]
  uint8_t* xq;        // MXFP8: x quantised once per token, [T, D] E4M3 (gathered into the ring, or read directly)
  uint8_t* xs;        // ... and its E8M0 scales, [T, D/32] row-major
  uint8_t* sfh;       // MXFP8: scale blocks of h, [n_mtiles_max][I/128][512 B]
  const uint8_t* w_up_sf;    // MXFP8 weight scale blocks (moe_quantize_mxfp8 layout)
  const uint8_t* w_gate_sf;
  const uint8_t* w_down_sf;
  bf16* h_s;          // [T, I_s]
  __half* Y;          // fp16 staging rows of the expert outputs, blocked: for token tile tt = t / 128 and
                      // column tile n (256 columns), block (tt, n) holds [128 tokens][kY slots][256 columns]
                      // contiguously (slots 0..k-1 routed, slot k the shared expert), so the combine reads
                      // one kY x 512-byte block per token and column tile
  bf16* out;          // [T, D]
  unsigned long long* trace;  // [grid, TRACE_SLOTS] when built with MOE_TRACE, else null
  int* dbg;           // MOE_DEBUG_LOG builds: [grid, DBG_SLOTS] progress records in host memory, else null
};

// Optional per-CTA timing of the persistent kernel (build with -DMOE_TRACE):
// SM cycles spent in each kind of wait, plus start/end %globaltimer stamps.
enum : int {
  TR_START_NS = 0, TR_END_NS, TR_PROD_DEP, TR_PROD_EMPTY, TR_MMA_FULL, TR_MMA_TEMPTY, TR_EPI_TFULL, TR_EPI_BUSY,
  TR_GATHER_WAIT, TR_GATHER_BUSY, TR_FINAL_WAIT, TR_TASKS, TR_EPI_R1, TR_EPI_R2, TR_EPI_S1, TR_EPI_S2,
  TR_TMA_LAT_NS /* stage issue -> full barrier seen by the MMA issuer, summed */, TR_TMA_STAGES,
  TR_GATHER_LOADWAIT /* bulk gather: waiting for a row load */, TR_GATHER_STOREWAIT /* ... for stores to drain */,
  TR_START_CLK /* clock64 at TR_START_NS */, TR_END_CLK /* ... at TR_END_NS: the SM clock over the run */,
  TR_COMBINE /* the final combine pass */,
  TRACE_SLOTS = 23
};
// Each thread that times anything keeps its sums in registers (TRACE_LOCALS)
// and adds them to the CTA's slots once, at the end (TRACE_FLUSH), so the
// timers stay off the paths they measure.
#ifdef MOE_TRACE
#define TRACE_LOCALS() unsigned long long _trv[TRACE_SLOTS] = {0}
#define TRACE_T0() const long long _tr0 = clock64()
#define TRACE_ADD(p, slot) (_trv[(slot)] += (unsigned long long)(clock64() - _tr0))
#define TRACE_FLUSH(p)                                                                       \
  do {                                                                                       \
    if ((p).trace && blockIdx.x < 1024)                                                      \
      for (int _i = 2; _i < TRACE_SLOTS; ++_i)                                               \
        if (_trv[_i]) atomicAdd((p).trace + (size_t)blockIdx.x * TRACE_SLOTS + _i, _trv[_i]); \
  } while (0)
#define TRACE_SET(p, slot, v)                                                                  \
  do {                                                                                         \
    if ((p).trace && blockIdx.x < 1024)                                                        \
      (p).trace[(size_t)blockIdx.x * TRACE_SLOTS + (slot)] = (unsigned long long)(v);          \
  } while (0)
#else
#define TRACE_LOCALS() do {} while (0)
#define TRACE_T0() do {} while (0)
#define TRACE_ADD(p, slot) do {} while (0)
#define TRACE_FLUSH(p) do {} while (0)
#define TRACE_SET(p, slot, v) do {} while (0)
#endif

// Debug builds (-DMOE_DEBUG_LOG): each CTA records its progress and the first
// failed bounds check in host memory (mapped pinned memory, readable by the
// host even after the context is lost), one store + system fence per record.
enum : int {
  DBG_PHASE = 0, DBG_RANK, DBG_TMEM, DBG_PROD_UNIT, DBG_PROD_ISSUED, DBG_MMA_UNIT, DBG_MMA_STAGES, DBG_MMA_ACC,
  DBG_EPI_UNIT, DBG_EPI_DONE, DBG_FAIL_SITE, DBG_FAIL_V0, DBG_FAIL_V1, DBG_FAIL_V2, DBG_PROD_WAIT, DBG_MMA_WAIT,
  DBG_EPI_WAIT, DBG_EPI_TASK, DBG_SLOTS = 32
};
#ifdef MOE_DEBUG_LOG
__device__ __forceinline__ void dbg_set(const FwdParams& p, int slot, int v) {
  if (p.dbg) {
    *reinterpret_cast<volatile int*>(p.dbg + (size_t)blockIdx.x * DBG_SLOTS + slot) = v;
    __threadfence_system();
  }
}
// false (and the first failure recorded) when cond does not hold: the caller skips the access
__device__ __forceinline__ bool dbg_check(const FwdParams& p, bool cond, int site, int v0, int v1, int v2) {
  if (cond) return true;
  if (p.dbg) {
    volatile int* d = p.dbg + (size_t)blockIdx.x * DBG_SLOTS;
    if (d[DBG_FAIL_SITE] == 0) {
      d[DBG_FAIL_V0] = v0;
      d[DBG_FAIL_V1] = v1;
      d[DBG_FAIL_V2] = v2;
      d[DBG_FAIL_SITE] = site;
      __threadfence_system();
    }
  }
  return false;
}
#define DBG_SET(p, slot, v) dbg_set((p), (slot), (int)(v))
#define DBG_CHECK(p, cond, site, v0, v1, v2) dbg_check((p), (cond), (site), (int)(v0), (int)(v1), (int)(v2))
#else
#define DBG_SET(p, slot, v) do {} while (0)
#define DBG_CHECK(p, cond, site, v0, v1, v2) (true)
#endif

// counter indices
__host__ __device__ inline int ctr_ydone() { return 0; }
__host__ __device__ inline int ctr_filled(const FwdParams& p, int m) { return 1 + m; }
__host__ __device__ inline int ctr_r1(const FwdParams& p, int m) { return 1 + p.n_mb + m; }
__host__ __device__ inline int ctr_r2(const FwdParams& p, int m) { return 1 + 2 * p.n_mb + m; }
__host__ __device__ inline int ctr_hready(const FwdParams& p, int mt) { return 1 + 3 * p.n_mb + mt; }
__host__ __device__ inline int ctr_shready(const FwdParams& p, int mt) {
  return 1 + 3 * p.n_mb + p.n_mtiles_max + mt;
}
// the 256 staging columns of column tile n for route (token t, slot s)
__host__ __device__ inline size_t y_offset(const FwdParams& p, int t, int s, int n) {
  return ((((size_t)(t / BM) * p.N2 + n) * BM + (size_t)(t % BM)) * p.kY + s) * BN_DOWN;
}
// the GEMM CTAs' unit claims (persistent kernel)
__host__ __device__ inline int ctr_claim(const FwdParams& p) { return 1 + 3 * p.n_mb + p.n_mtiles_max + p.n_smtiles; }
// the combine's claims of round chunks (cluster-launch-control scheduling)
__host__ __device__ inline int ctr_combine(const FwdParams& p) { return 2 + 3 * p.n_mb + p.n_mtiles_max + p.n_smtiles; }
__host__ __device__ inline int n_counters(const FwdParams& p) { return 3 + 3 * p.n_mb + p.n_mtiles_max + p.n_smtiles; }

struct TensorMaps {
  CUtensorMap x;        // [T, D]            box {64, 128}
  CUtensorMap x_rows;   // direct dispatch: [T, D] bf16 box {64, 1} or E4M3 box {128, 1} (tile::gather4)
  CUtensorMap ring_x;   // [slots*b, D]      box {64, 128}
  CUtensorMap w_up;     // [E*I, D]          box {64, 128}
  CUtensorMap w_gate;   // [E*I, D]          box {64, 128}
  CUtensorMap ring_h;   // [slots*b, I]      box {64, 128}
  CUtensorMap ring_x64; // BF16 pairs, split M-tiles: [slots*b, D] box {64, 64}
  CUtensorMap ring_h64; // ... [slots*b, I] box {64, 64}
  CUtensorMap w_up64;   // ... [E*I, D] box {64, 64}: 64 up rows and
  CUtensorMap w_gate64; //     64 gate rows per CTA
  CUtensorMap w_down;   // [E*D, I]          box {64, 256}
  CUtensorMap ws_up;    // [I_s, D]          box {64, 128}
  CUtensorMap ws_gate;  // [I_s, D]          box {64, 128}
  CUtensorMap h_s;      // [T, I_s]          box {64, 128}
  CUtensorMap ws_down;  // [D, I_s]          box {64, 256}
  // CTA pairs with MXFP8 routed tiles: the 512-byte scale blocks as rows of
  // 128 bytes (box {128, 4} = one block), so that both CTAs' loads can be
  // counted on the even CTA's barrier
  CUtensorMap sf_x, sf_h, sf_up, sf_gate, sf_down;
};

struct RouterMaps {
  CUtensorMap x;   // [T, D] box {64, 128}
  CUtensorMap wr;  // [E, D] box {64, n_router_cols} (or half of it when E > 256)
};

// ------------------------------------------------------------------ bounded waits
// Every wait gives up after timeout_ns (or as soon as another thread has set a
// non-zero status), records STATUS_TIMEOUT and returns false; callers then
// stop issuing work and leave cleanly.
__device__ __forceinline__ void raise_status(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ bool wait_counter_ge(const int* ctr, int need, int* status, long long timeout_ns) {
  if (ld_acquire_gpu(ctr) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (ld_acquire_gpu(ctr) >= need) return true;
    if ((++it & 31u) == 0) {
      if (ld_relaxed_gpu(status) != 0) return false;
      if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) {
        raise_status(status, STATUS_TIMEOUT);
        return false;
      }
    }
    __nanosleep(32);
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (ld_relaxed_gpu(status) != 0) return false;
      if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) {
        raise_status(status, STATUS_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// Waiting for this CTA's own asynchronous copies or MMAs before it frees
// their resources or exits: the status word is not consulted (work already
// issued always completes), only the time limit.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > (uint64_t)limit_ns) return false;
  return true;
}
// after an abort (status raised), a bounded pause so that copies other CTAs of
// a pair issued into this CTA's shared memory have landed before it exits
__device__ __forceinline__ void settle_after_abort(const int* status) {
  if (ld_relaxed_gpu(status) == 0) return;
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
}

// the same for a phase completed with the help of the other CTA of a pair
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status, long long timeout_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (ld_relaxed_gpu(status) != 0) return false;
      if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) {
        raise_status(status, STATUS_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// SiLU(v) = v / (1 + e^-v) with the fast exponential and reciprocal intrinsics
// (for v -> -inf the reciprocal of +inf is 0, so the result tends to -0)
__device__ __forceinline__ float silu_f32(float v) { return v * __fdividef(1.0f, 1.0f + __expf(-v)); }

// OCP MX v1.0, MXFP8 E4M3 block of 32: X = 2^(floor(log2 amax) - 8), codes =
// E4M3(v / X) rounded to nearest-even and saturated at +-448; an all-zero block
// gets the code 0 (X = 2^-127).  Returns the E8M0 code; q receives the codes.
__device__ __forceinline__ uint32_t mx_quantize32(const float* v, uint32_t* q) {
  // max |v| as a pairwise tree (exact in any order; five dependent steps, not 32)
  float m[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) m[j] = fmaxf(fabsf(v[j]), fabsf(v[j + 16]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
  const float amax = m[0];
  if (amax == 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0;
    return 0;
  }
  // floor(log2 amax) from the exponent field (a subnormal amax has none)
  const uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;
  int se = (eb != 0u ? (int)eb - 127 : ilogbf(amax)) - 8;
  se = max(-127, min(127, se));
  // v * 2^-se, exact (|result| < 2^9) when 2^-se is a normal float, as ldexpf
  const bool pow2 = se >= -126 && se <= 126;
  const float scale = __uint_as_float((uint32_t)(127 - se) << 23);
  float a[32];
  if (pow2) {
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = v[j] * scale;
  } else {  // 2^-se is not a normal float (a block of huge or tiny values)
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = ldexpf(v[j], -se);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // two codes per conversion; element 4i + j lands in byte j of the word
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a[4 * i], a[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a[4 * i + 2], a[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
    q[i] = lo | (hi << 16);
  }
  return (uint32_t)(se + 127);
}

// 32 bf16 values (64 bytes, 16-byte aligned) -> fp32
__device__ __forceinline__ void load_bf16x32(const bf16* src, float* v) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = __ldg(s4 + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[8 * i + 2 * j] = f.x;
      v[8 * i + 2 * j + 1] = f.y;
    }
  }
}

}  // namespace moe
