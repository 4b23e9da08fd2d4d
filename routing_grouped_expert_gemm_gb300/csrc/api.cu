// C ABI of the MoE forward (declared in include/moe.h): plan validation,
// workspace layout, TMA tensor-map encoding and the three launches.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/moe.h"
#include "common.cuh"
#include "plan.cuh"

namespace moe {
cudaError_t launch_router(const RouterMaps& maps, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_schedule(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_megakernel(const TensorMaps& maps, const FwdParams& p, int grid, cudaStream_t stream);
int megakernel_smem_bytes();
int megakernel_pair_max_ctas(bool mx);
cudaError_t launch_mx_quantize(const bf16* W, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, cudaStream_t st);
size_t mx_scale_bytes(int64_t rows, int64_t K);
}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Layout {
  size_t status, counters, meta, topk_idx, topk_w, topk_logit, chunk_counts, M, S, sched, route_row, mtiles, segs, tasks;
  size_t ring_x, ring_h, sfx, sfh, xq, xs, h_s, Y, trace, total;
  int64_t n_mb, n_mtiles_max, n_smtiles, n_tasks_max, n_counters, n_chunks, max_segs, R;
};

Layout make_layout(const moe_plan* pl, int64_t T) {
  const moe_config& c = pl->cfg;
  Layout L{};
  L.R = T * c.k;
  L.n_mb = ceil_div(L.R, c.minibatch);
  L.n_chunks = ceil_div(T, BM);
  L.max_segs = L.n_mb + c.E;
  L.n_mtiles_max = ceil_div(L.R, BM) + L.n_mb + c.E;
  L.n_smtiles = c.I_s > 0 ? L.n_chunks : 0;
  // CTA pairs pad every expert segment and the shared token tiles to an even count
  const int64_t pad_seg = c.mma_pair ? L.max_segs : 0, pad_sh = c.mma_pair ? 1 : 0;
  L.n_tasks_max = (L.n_mtiles_max + pad_seg) * (c.I / BN_UP + c.D / BN_DOWN) +
                  (c.I_s > 0 ? (L.n_smtiles + pad_sh) * (c.I_s / BN_UP + c.D / BN_DOWN) : 0);
  L.n_counters = 3 + 3 * L.n_mb + L.n_mtiles_max + L.n_smtiles;  // see ctr_claim, ctr_combine
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  };
  L.status = take(STATUS_AREA_BYTES);  // status word, warning bits, phase stamps
  L.counters = take(sizeof(int) * L.n_counters);
  L.meta = take(sizeof(int) * (META_MB + 4 * L.n_mb));
  L.topk_idx = take(sizeof(int) * L.R);
  L.topk_w = take(sizeof(float) * L.R);
  L.topk_logit = take(sizeof(float) * L.R);
  L.chunk_counts = take(sizeof(int) * L.n_chunks * c.E);
  L.M = take(sizeof(int) * c.E);
  L.S = take(sizeof(int) * (c.E + 1));
  L.sched = take(sizeof(int) * 3 * L.R);
  L.route_row = take(sizeof(int) * L.R);
  L.mtiles = take(sizeof(int) * 4 * L.n_mtiles_max);
  L.segs = take(sizeof(int) * (4 * L.max_segs + 4 * (2 * L.max_segs + 2) + L.n_mb + 1));
  L.tasks = take(sizeof(Task) * L.n_tasks_max);
  const int64_t ring_rows = (int64_t)c.ring_slots * c.minibatch;
  const bool mx = c.precision == MOE_PREC_MXFP8;
  const bool direct = c.dispatch == MOE_DISPATCH_DIRECT;
  const size_t elem = mx ? 1 : 2;  // E4M3 codes or bf16 in the rings
  L.ring_x = take(direct ? 0 : (size_t)ring_rows * c.D * elem);
  L.ring_h = take((size_t)ring_rows * c.I * elem);
  L.sfx = take(mx && !direct ? (size_t)L.n_mtiles_max * (c.D / BK_MX) * SF_BLOCK_BYTES : 0);
  // MXFP8: x quantised once per token by the router pass (it reads every row)
  L.xq = take(mx ? (size_t)T * c.D : 0);
  L.xs = take(mx ? (size_t)T * (c.D / 32) : 0);
  L.sfh = take(mx ? (size_t)L.n_mtiles_max * (c.I / BK_MX) * SF_BLOCK_BYTES : 0);
  L.h_s = take((size_t)T * c.I_s * 2);
  L.Y = take((size_t)L.n_chunks * BM * (c.k + (c.I_s > 0 ? 1 : 0)) * c.D * 2);  // blocked by token tile, see FwdParams::Y
#ifdef MOE_TRACE
  L.trace = take(sizeof(unsigned long long) * TRACE_SLOTS * 1024);
#endif
  L.total = off;
  return L;
}

// E4M3 codes, one byte each: 128-byte rows of the box like the bf16 maps
int encode_u8_2d(const moe_plan* pl, CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {BK_MX, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = pl->encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int encode_bf16_2d(const moe_plan* pl, CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = pl->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// 512-byte MX scale blocks seen as rows of 128 bytes: box {128, 4} is one block
int encode_sf_blocks(const moe_plan* pl, CUtensorMap* m, const void* ptr, size_t bytes) {
  cuuint64_t dims[2] = {128, bytes / 128};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 4};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = pl->encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace moe {
// Where a forward of T tokens keeps its routing and schedule in its workspace
// (read by the backward pass, which reuses them).
int fwd_routing_views(const moe_plan* pl, int64_t T, const void* workspace, FwdRoutingViews* v) {
  if (!pl || !workspace || !v || T < 1 || T > pl->cfg.T_max) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(pl, T);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  v->topk_idx = reinterpret_cast<const int*>(ws + L.topk_idx);
  v->topk_w = reinterpret_cast<const float*>(ws + L.topk_w);
  v->topk_logit = reinterpret_cast<const float*>(ws + L.topk_logit);
  v->M = reinterpret_cast<const int*>(ws + L.M);
  v->S = reinterpret_cast<const int*>(ws + L.S);
  v->sched = reinterpret_cast<const int*>(ws + L.sched);
  return MOE_OK;
}
}  // namespace moe

extern "C" {

const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case MOE_ERR_STATIC_SCRATCH_TOO_SMALL:
      return "request exceeds the library's fixed routing scratch (T > MOE_ROUTE_STATIC_MAX_TOKENS)";
    default: return "unknown error";
  }
}

int moe_plan_create(const moe_config* cfg_in, moe_plan** out) {
  if (!cfg_in || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_config c = *cfg_in;
  if (c.dispatch != MOE_DISPATCH_RING && c.dispatch != MOE_DISPATCH_DIRECT && c.dispatch != MOE_DISPATCH_SPREAD)
    return MOE_ERR_INVALID_ARG;
  if (c.minibatch == 0) c.minibatch = 8192;
  if (c.ring_slots == 0) c.ring_slots = 4;
  if (c.gather_ctas == 0 && c.dispatch == MOE_DISPATCH_RING) c.gather_ctas = 8;
  if (c.timeout_ms <= 0) c.timeout_ms = 2000;
  if (c.l2_prefetch < 0 || c.l2_prefetch > 64) return MOE_ERR_INVALID_ARG;
  if (c.lag < 0 || c.lag > 1) return MOE_ERR_INVALID_ARG;
  if (c.score_fn != MOE_SCORE_SIGMOID && c.score_fn != MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
  if (c.precision != MOE_PREC_BF16 && c.precision != MOE_PREC_MXFP8) return MOE_ERR_INVALID_ARG;
  if (c.T_max < 1 || c.D < 256 || c.D % 256 || c.I < 128 || c.I % 128 || c.E < 1 || c.E > E_MAX || c.k < 1 ||
      c.k > TOPK_MAX || c.k > c.E || c.I_s < 0 || c.I_s % 128)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.D > 65536 || c.I > 65536 || c.I_s > 65536 || c.T_max * c.k > (int64_t)1 << 30 ||
      c.E * c.I > (int64_t)1 << 30 || c.E * c.D > (int64_t)1 << 30)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.minibatch < BM || c.minibatch > 32768 || c.minibatch % BM) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.ring_slots < c.lag + 1 || c.ring_slots > 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((c.T_max * c.k + c.minibatch - 1) / c.minibatch > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;  // schedule smem
  if (c.raster < 0) return MOE_ERR_INVALID_ARG;
  if (c.raster == 0) c.raster = 1 << 20;  // default: column-tile major over the whole segment
  if (c.mma_pair != 0 && c.mma_pair != 1) return MOE_ERR_INVALID_ARG;
  // cluster launch control schedules the one-CTA kernel
  if (c.clc != 0 && c.clc != 1) return MOE_ERR_INVALID_ARG;
  if (c.plain_launch != 0 && c.plain_launch != 1) return MOE_ERR_INVALID_ARG;
  if (c.pad_odd_tiles != 0 && c.pad_odd_tiles != 1) return MOE_ERR_INVALID_ARG;
  if (c.clc && c.mma_pair) return MOE_ERR_INVALID_ARG;
#ifdef MOE_DEBUG_LOG
  if (c.clc) return MOE_ERR_INVALID_ARG;  // the progress records are sized for the persistent grid
#endif
  // the test hook needs a ring whose fill is signalled (ring or spread dispatch)
  if (c.test_unfilled_minibatch < 0 || (c.test_unfilled_minibatch > 0 && c.dispatch == MOE_DISPATCH_DIRECT))
    return MOE_ERR_INVALID_ARG;
  if (c.mma_pair) c.raster = (c.raster + 1) & ~1;  // a pair's two tasks share a column tile
  if (c.dispatch == MOE_DISPATCH_SPREAD) c.gather_ctas = 0;  // the GEMM CTAs' spare warps gather
  if (c.mma_pair && (c.dispatch == MOE_DISPATCH_DIRECT || (c.gather_ctas & 1) ||
                     (c.gemm_ctas & 1)))
    return MOE_ERR_INVALID_ARG;
  if (c.dispatch == MOE_DISPATCH_DIRECT) c.gather_ctas = 0;  // the GEMM producers gather
  if ((c.dispatch == MOE_DISPATCH_RING && c.gather_ctas < 1) || c.gemm_ctas < 0) return MOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED_DEVICE;
  // CTAs resident at once: one per SM, or for CTA pairs as many as whole
  // clusters of 2 can be placed
  const int resident =
      c.mma_pair ? megakernel_pair_max_ctas(c.precision == MOE_PREC_MXFP8) : prop.multiProcessorCount;
  if (resident < 2) return MOE_ERR_CUDA;
  const int gemm = c.gemm_ctas > 0 ? c.gemm_ctas : resident - c.gather_ctas;
  if (gemm < (c.mma_pair ? 2 : 1) || c.gather_ctas + gemm > resident) return MOE_ERR_INVALID_ARG;

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return MOE_ERR_CUDA;

  moe_plan* pl = new (std::nothrow) moe_plan;
  if (!pl) return MOE_ERR_INVALID_ARG;
  pl->cfg = c;
  pl->device = dev;
  pl->num_sms = prop.multiProcessorCount;
  pl->grid = c.gather_ctas + gemm;
  pl->encode = reinterpret_cast<encode_tiled_fn>(fn);
  pl->timed = false;
  pl->bwd_timed = false;
  *out = pl;
  return MOE_OK;
}

int moe_plan_set_timing_events(moe_plan* plan, void* const* events) {
  if (!plan) return MOE_ERR_INVALID_ARG;
  if (!events) {
    plan->timed = false;
    return MOE_OK;
  }
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return MOE_ERR_INVALID_ARG;
    plan->timing[i] = static_cast<cudaEvent_t>(events[i]);
  }
  plan->timed = true;
  return MOE_OK;
}

int moe_get_phase_times(const moe_plan* plan, const void* workspace, double* times_ms, moe_stream_t stream) {
  if (!plan || !workspace || !times_ms) return MOE_ERR_INVALID_ARG;
  unsigned long long st[N_STAMPS];
  const uint8_t* area = static_cast<const uint8_t*>(workspace) + 8;
  if (cudaMemcpyAsync(st, area, sizeof(st), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  const unsigned long long t0 = st[STAMP_START];
  auto rel = [&](unsigned long long v) {
    return (v == 0ull || v == ~0ull || t0 == ~0ull || v < t0) ? -1.0 : (double)(v - t0) * 1e-6;
  };
  times_ms[0] = rel(st[STAMP_LAST_FILL]);
  times_ms[1] = rel(st[STAMP_COMBINE_START]);
  times_ms[2] = rel(st[STAMP_COMBINE_END]);
  return MOE_OK;
}

int moe_plan_set_bwd_timing_events(moe_plan* plan, void* const* events) {
  if (!plan) return MOE_ERR_INVALID_ARG;
  if (!events) {
    plan->bwd_timed = false;
    return MOE_OK;
  }
  for (int i = 0; i < 5; ++i) {
    if (!events[i]) return MOE_ERR_INVALID_ARG;
    plan->bwd_timing[i] = static_cast<cudaEvent_t>(events[i]);
  }
  plan->bwd_timed = true;
  return MOE_OK;
}

int moe_plan_destroy(moe_plan* plan) {
  delete plan;
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_plan* plan, int64_t T) {
  if (!plan || T < 0 || T > plan->cfg.T_max) return 0;
  if (T == 0) return kAlign;
  return make_layout(plan, T).total;
}

size_t moe_mxfp8_scale_bytes(int64_t rows, int64_t K) { return mx_scale_bytes(rows, K); }

int moe_quantize_mxfp8(const moe_plan* plan, const void* W, int64_t rows, int64_t K, uint8_t* q, uint8_t* scales,
                       moe_stream_t stream) {
  if (!plan || !W || !q || !scales || rows < 1 || K < 128) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || K % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  return launch_mx_quantize(static_cast<const bf16*>(W), rows, K, q, scales, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_fwd(const moe_plan* pl, int64_t T, const void* x, const moe_weights* w, const moe_outputs* o,
            void* workspace, size_t workspace_bytes, moe_stream_t stream_) {
  if (!pl || !w || !o || T < 0 || T > pl->cfg.T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const moe_config& c = pl->cfg;
  if (!x || !w->W_router || !w->W_up || !w->W_gate || !w->W_down || !o->out || !workspace)
    return MOE_ERR_INVALID_ARG;
  const bool shared = w->Ws_up || w->Ws_gate || w->Ws_down;
  if (shared && (!w->Ws_up || !w->Ws_gate || !w->Ws_down || c.I_s == 0)) return MOE_ERR_INVALID_ARG;
  const bool mx = c.precision == MOE_PREC_MXFP8;
  if (mx && (!w->W_up_scale || !w->W_gate_scale || !w->W_down_scale)) return MOE_ERR_INVALID_ARG;
  if (mx && (!aligned16(w->W_up_scale) || !aligned16(w->W_gate_scale) || !aligned16(w->W_down_scale)))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w->W_router, w->W_up, w->W_gate, w->W_down, o->out, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (shared && (!aligned16(w->Ws_up) || !aligned16(w->Ws_gate) || !aligned16(w->Ws_down))) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(pl, T);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = (cudaStream_t)stream_;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != pl->device) return MOE_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FwdParams p{};
  p.T = (int)T;
  p.D = (int)c.D;
  p.I = (int)c.I;
  p.E = (int)c.E;
  p.k = (int)c.k;
  p.kY = (int)c.k + (shared ? 1 : 0);  // a call without the shared weights has no slot k
  p.I_s = shared ? (int)c.I_s : 0;
  p.score_fn = c.score_fn;
  p.mx = mx ? 1 : 0;
  p.direct = c.dispatch == MOE_DISPATCH_DIRECT ? 1 : 0;
  p.spread = c.dispatch == MOE_DISPATCH_SPREAD ? 1 : 0;
  p.pair = c.mma_pair;
  p.raster = c.raster;
  p.b = c.minibatch;
  p.slots = c.ring_slots;
  p.G = c.gather_ctas;
  p.n_gemm = pl->grid - c.gather_ctas;
  p.gparts = p.spread ? p.n_gemm : c.gather_ctas;
  p.lag = c.lag;
  p.n_mb = (int)L.n_mb;
  p.R = (int)L.R;
  p.N1 = p.I / BN_UP;
  p.N2 = p.D / BN_DOWN;
  p.N1s = shared ? p.I_s / BN_UP : 0;
  p.N2s = shared ? p.D / BN_DOWN : 0;
  p.n_chunks = (int)L.n_chunks;
  p.n_router_cols = c.E <= 256 ? (int)(ceil_div(c.E, 32) * 32) : (int)(ceil_div(c.E, 64) * 64);
  p.n_mtiles_max = (int)L.n_mtiles_max;
  p.n_smtiles = shared ? (int)L.n_smtiles : 0;
  p.n_tasks_max = (int)L.n_tasks_max;
  p.n_counters = (int)L.n_counters;
  p.timeout_ns = (long long)c.timeout_ms * 1000000LL;
  p.l2_prefetch = c.l2_prefetch;
  p.test_unfilled = c.test_unfilled_minibatch;
  p.clc = c.clc;
  p.plain_launch = c.plain_launch;
  p.half_tiles = c.mma_pair && c.precision == MOE_PREC_BF16 && !c.pad_odd_tiles ? 1 : 0;
  p.x = static_cast<const bf16*>(x);
  p.b_router = w->b_router;
  p.status = reinterpret_cast<int*>(ws + L.status);
  p.stamps = reinterpret_cast<unsigned long long*>(ws + L.status + 8);
  p.counters = reinterpret_cast<int*>(ws + L.counters);
  p.meta = reinterpret_cast<int*>(ws + L.meta);
  p.topk_idx = reinterpret_cast<int*>(ws + L.topk_idx);
  p.topk_w = reinterpret_cast<float*>(ws + L.topk_w);
  p.topk_logit = reinterpret_cast<float*>(ws + L.topk_logit);
  p.chunk_counts = reinterpret_cast<int*>(ws + L.chunk_counts);
  p.M = reinterpret_cast<int*>(ws + L.M);
  p.S = reinterpret_cast<int*>(ws + L.S);
  p.sched = reinterpret_cast<int*>(ws + L.sched);
  p.route_row = reinterpret_cast<int*>(ws + L.route_row);
  p.mtiles = reinterpret_cast<int*>(ws + L.mtiles);
  p.segs = reinterpret_cast<int*>(ws + L.segs);
  p.tasks = reinterpret_cast<Task*>(ws + L.tasks);
  p.ring_x = reinterpret_cast<bf16*>(ws + L.ring_x);
  p.ring_h = reinterpret_cast<bf16*>(ws + L.ring_h);
  p.xq = mx ? ws + L.xq : nullptr;
  p.xs = mx ? ws + L.xs : nullptr;
  p.sfx = mx && !p.direct ? ws + L.sfx : nullptr;
  p.sfh = mx ? ws + L.sfh : nullptr;
  p.w_up_sf = mx ? w->W_up_scale : nullptr;
  p.w_gate_sf = mx ? w->W_gate_scale : nullptr;
  p.w_down_sf = mx ? w->W_down_scale : nullptr;
  p.h_s = reinterpret_cast<bf16*>(ws + L.h_s);
  p.Y = reinterpret_cast<__half*>(ws + L.Y);
  p.out = static_cast<bf16*>(o->out);
#ifdef MOE_TRACE
  p.trace = reinterpret_cast<unsigned long long*>(ws + L.trace);
  cudaMemsetAsync(p.trace, 0, sizeof(unsigned long long) * TRACE_SLOTS * 1024, stream);
#endif

#ifdef MOE_DEBUG_LOG
  // debugging builds only: the address of mapped pinned host memory for the
  // progress records, [grid, DBG_SLOTS] int32, given by the environment
  if (const char* dbg = std::getenv("MOE_DEBUG_LOG_PTR")) p.dbg = reinterpret_cast<int*>(std::strtoull(dbg, nullptr, 0));
#endif
  // tensor maps (raw pointers are baked in, so they are encoded per call)
  RouterMaps rm;
  TensorMaps tm;
  std::memset(&rm, 0, sizeof(rm));
  std::memset(&tm, 0, sizeof(tm));
  const int64_t ring_rows = (int64_t)c.ring_slots * c.minibatch;
  const uint32_t wr_box = (uint32_t)(p.n_router_cols > 256 ? p.n_router_cols / 4 : p.n_router_cols / 2);  // per CTA of a pair
  const uint32_t down_box = c.mma_pair ? 128u : (uint32_t)BN_DOWN;  // pairs: each CTA loads half the columns
  int rc = MOE_OK;
  rc |= encode_bf16_2d(pl, &rm.x, x, T, c.D, BM);
  rc |= encode_bf16_2d(pl, &rm.wr, w->W_router, c.E, c.D, wr_box);
  rc |= encode_bf16_2d(pl, &tm.x, x, T, c.D, BM);
  if (p.direct) {  // one-row boxes for tile::gather4 from x (bf16) or its E4M3 copy
    if (mx)
      rc |= encode_u8_2d(pl, &tm.x_rows, p.xq, T, c.D, 1);
    else
      rc |= encode_bf16_2d(pl, &tm.x_rows, x, T, c.D, 1);
  }
  if (mx) {  // routed operands as E4M3 codes
    if (!p.direct) rc |= encode_u8_2d(pl, &tm.ring_x, p.ring_x, ring_rows, c.D, BM);
    rc |= encode_u8_2d(pl, &tm.w_up, w->W_up, c.E * c.I, c.D, BN_UP);
    rc |= encode_u8_2d(pl, &tm.w_gate, w->W_gate, c.E * c.I, c.D, BN_UP);
    rc |= encode_u8_2d(pl, &tm.ring_h, p.ring_h, ring_rows, c.I, BM);
    rc |= encode_u8_2d(pl, &tm.w_down, w->W_down, c.E * c.D, c.I, down_box);
    if (c.mma_pair) {  // scale blocks through tensor maps (loads counted on the even CTA's barrier)
      rc |= encode_sf_blocks(pl, &tm.sf_x, p.sfx, (size_t)L.n_mtiles_max * (c.D / BK_MX) * SF_BLOCK_BYTES);
      rc |= encode_sf_blocks(pl, &tm.sf_h, p.sfh, (size_t)L.n_mtiles_max * (c.I / BK_MX) * SF_BLOCK_BYTES);
      rc |= encode_sf_blocks(pl, &tm.sf_up, w->W_up_scale, mx_scale_bytes(c.E * c.I, c.D));
      rc |= encode_sf_blocks(pl, &tm.sf_gate, w->W_gate_scale, mx_scale_bytes(c.E * c.I, c.D));
      rc |= encode_sf_blocks(pl, &tm.sf_down, w->W_down_scale, mx_scale_bytes(c.E * c.D, c.I));
    }
  } else {
    if (!p.direct) rc |= encode_bf16_2d(pl, &tm.ring_x, p.ring_x, ring_rows, c.D, BM);
    rc |= encode_bf16_2d(pl, &tm.w_up, w->W_up, c.E * c.I, c.D, BN_UP);
    rc |= encode_bf16_2d(pl, &tm.w_gate, w->W_gate, c.E * c.I, c.D, BN_UP);
    rc |= encode_bf16_2d(pl, &tm.ring_h, p.ring_h, ring_rows, c.I, BM);
    rc |= encode_bf16_2d(pl, &tm.w_down, w->W_down, c.E * c.D, c.I, down_box);
    if (p.half_tiles) {  // a split M-tile's 64 rows per CTA
      rc |= encode_bf16_2d(pl, &tm.ring_x64, p.ring_x, ring_rows, c.D, BM / 2);
      rc |= encode_bf16_2d(pl, &tm.ring_h64, p.ring_h, ring_rows, c.I, BM / 2);
      rc |= encode_bf16_2d(pl, &tm.w_up64, w->W_up, c.E * c.I, c.D, BM / 2);
      rc |= encode_bf16_2d(pl, &tm.w_gate64, w->W_gate, c.E * c.I, c.D, BM / 2);
    }
  }
  if (shared) {
    rc |= encode_bf16_2d(pl, &tm.ws_up, w->Ws_up, c.I_s, c.D, BN_UP);
    rc |= encode_bf16_2d(pl, &tm.ws_gate, w->Ws_gate, c.I_s, c.D, BN_UP);
    rc |= encode_bf16_2d(pl, &tm.h_s, p.h_s, T, c.I_s, BM);
    rc |= encode_bf16_2d(pl, &tm.ws_down, w->Ws_down, c.D, c.I_s, down_box);
  }
  if (rc != MOE_OK) return MOE_ERR_INVALID_ARG;

  if (pl->timed && cudaEventRecord(pl->timing[0], stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_router(rm, p, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (pl->timed && cudaEventRecord(pl->timing[1], stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_schedule(p, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (pl->timed && cudaEventRecord(pl->timing[2], stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_megakernel(tm, p, pl->grid, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (pl->timed && cudaEventRecord(pl->timing[3], stream) != cudaSuccess) return MOE_ERR_CUDA;

  const size_t R = (size_t)L.R;
  struct Copy { void* dst; const void* src; size_t bytes; } copies[] = {
      {o->topk_idx, p.topk_idx, R * 4}, {o->topk_w, p.topk_w, R * 4},
      {o->expert_counts, p.M, (size_t)c.E * 4}, {o->expert_offsets, p.S, (size_t)(c.E + 1) * 4},
      {o->sched, p.sched, 3 * R * 4}, {o->route_row, p.route_row, R * 4}};
  for (const Copy& cp : copies)
    if (cp.dst && cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_get_status(const moe_plan* plan, const void* workspace, int* device_status, moe_stream_t stream) {
  if (!plan || !workspace || !device_status) return MOE_ERR_INVALID_ARG;
  int v[2] = {0, 0};  // the status word and the warning bits after it
  if (cudaMemcpyAsync(v, workspace, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  *device_status = v[0] != STATUS_OK ? v[0] : ((v[1] & FLAG_STAGING_OVERFLOW) ? MOE_STATUS_STAGING_OVERFLOW : MOE_STATUS_OK);
  return MOE_OK;
}

}  // extern "C"
