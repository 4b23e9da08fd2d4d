// moe_route_static: the routing stage (router projection + top-k + g, then
// the per-expert counts, offsets and schedule table) for callers that cannot
// allocate device memory.  The paper has no counterpart to this entry point.
//
// Who needs it: code that must not call cudaMalloc/cudaFree itself, for
// example a plugin living inside a host framework that owns every device
// byte through its own pool, or a latency-critical loop where an allocation
// (which may synchronise the device) is not allowed.  moe_fwd needs a
// caller-allocated workspace; this entry point needs none.
//
// The kernels' scratch (per-chunk expert histograms, counters, status word,
// schedule-builder lists) lives in one file-scope device array of
// kRouteScratchBytes that every GPU which loads this library holds until the
// process exits.  The router and schedule kernels are the same ones moe_fwd
// launches; only where their scratch lives differs.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "plan.cuh"

namespace moe {
cudaError_t launch_router(const RouterMaps& maps, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_schedule(const FwdParams& p, cudaStream_t stream);
}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kRouteScratchBytes = 512u * 1024u;  // fits T <= MOE_ROUTE_STATIC_MAX_TOKENS, E <= 512, k <= 16
constexpr int kRouteMinibatch = 32768;                // largest minibatch: fewest schedule-builder segments
constexpr int kMaxDevices = 64;

// The array every call shares.  In host code this name is only a stand-in:
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on `dev` (which is the current device);
// looked up once per device.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct RouteLayout {
  size_t status, counters, meta, chunk_counts, mtiles, segs, total;
  int n_mb, n_chunks, max_segs, n_mtiles_max, n_counters;
};

// Scratch layout of one call; the counter block has the size the kernels
// index (n_counters() of the persistent kernel's layout, no shared tiles).
constexpr RouteLayout route_layout(int64_t T, int64_t E, int64_t k) {
  RouteLayout L{};
  const int64_t R = T * k;
  L.n_mb = (int)((R + kRouteMinibatch - 1) / kRouteMinibatch);
  L.n_chunks = (int)((T + BM - 1) / BM);
  L.max_segs = L.n_mb + (int)E;
  L.n_mtiles_max = (int)((R + BM - 1) / BM) + L.n_mb + (int)E;
  L.n_counters = 3 + 3 * L.n_mb + L.n_mtiles_max;
  size_t off = 0;
  L.status = off;  // status word, warning bits, phase stamps
  off = align256(off + STATUS_AREA_BYTES);
  L.counters = off;
  off = align256(off + sizeof(int) * (size_t)L.n_counters);
  L.meta = off;
  off = align256(off + sizeof(int) * (size_t)(META_MB + 4 * L.n_mb));
  L.chunk_counts = off;
  off = align256(off + sizeof(int) * (size_t)L.n_chunks * (size_t)E);
  L.mtiles = off;
  off = align256(off + sizeof(int) * 4 * (size_t)L.n_mtiles_max);
  L.segs = off;
  off = align256(off + sizeof(int) * (size_t)(4 * L.max_segs + 4 * (2 * L.max_segs + 2) + L.n_mb + 1));
  L.total = off;
  return L;
}
// the documented limits fit the fixed array
static_assert(route_layout(MOE_ROUTE_STATIC_MAX_TOKENS, E_MAX, TOPK_MAX).total <= kRouteScratchBytes,
              "routing scratch too small for T = MOE_ROUTE_STATIC_MAX_TOKENS, E = 512, k = 16");

int encode_rows(const moe_plan* pl, CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = pl->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" size_t moe_route_static_scratch_bytes(void) { return kRouteScratchBytes; }

extern "C" int moe_route_static(const moe_plan* pl, int64_t T, const void* x, const void* W_router,
                                const float* b_router, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                                int32_t* expert_offsets, int32_t* sched, int32_t* route_row, int32_t* device_status,
                                moe_stream_t stream_) {
  if (!pl || T < 0 || T > pl->cfg.T_max) return MOE_ERR_INVALID_ARG;
  if (T > MOE_ROUTE_STATIC_MAX_TOKENS) return MOE_ERR_STATIC_SCRATCH_TOO_SMALL;
  if (T == 0) return MOE_OK;
  if (!x || !W_router || !topk_idx || !topk_w || !expert_counts || !expert_offsets || !sched || !route_row)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_router)) return MOE_ERR_INVALID_ARG;
  const moe_config& c = pl->cfg;
  const RouteLayout L = route_layout(T, c.E, c.k);
  if (L.total > kRouteScratchBytes) return MOE_ERR_STATIC_SCRATCH_TOO_SMALL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != pl->device) return MOE_ERR_INVALID_ARG;
  void* base = nullptr;
  const int rc = scratch_address(cur, &base);
  if (rc != MOE_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(base);
  cudaStream_t stream = (cudaStream_t)stream_;

  FwdParams p{};
  p.T = (int)T;
  p.D = (int)c.D;
  p.I = (int)c.I;
  p.E = (int)c.E;
  p.k = (int)c.k;
  p.I_s = 0;
  p.score_fn = c.score_fn;
  p.b = kRouteMinibatch;
  p.slots = 1;
  p.G = 1;
  p.n_gemm = 1;
  p.lag = 0;
  p.n_mb = L.n_mb;
  p.R = (int)(T * c.k);
  p.N1 = p.N2 = p.N1s = p.N2s = 0;  // routing only: the schedule kernel lays out no expert tasks
  p.n_chunks = L.n_chunks;
  p.n_router_cols = c.E <= 256 ? (int)((c.E + 31) / 32 * 32) : (int)((c.E + 63) / 64 * 64);
  p.n_mtiles_max = L.n_mtiles_max;
  p.n_smtiles = 0;
  p.n_tasks_max = 0;
  p.n_counters = L.n_counters;
  p.timeout_ns = (long long)c.timeout_ms * 1000000LL;
  p.x = static_cast<const bf16*>(x);
  p.b_router = b_router;
  p.status = reinterpret_cast<int*>(ws + L.status);
  p.stamps = nullptr;  // no persistent kernel
  p.counters = reinterpret_cast<int*>(ws + L.counters);
  p.meta = reinterpret_cast<int*>(ws + L.meta);
  p.chunk_counts = reinterpret_cast<int*>(ws + L.chunk_counts);
  p.mtiles = reinterpret_cast<int*>(ws + L.mtiles);
  p.segs = reinterpret_cast<int*>(ws + L.segs);
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.M = expert_counts;
  p.S = expert_offsets;
  p.sched = sched;
  p.route_row = route_row;

  RouterMaps rm;
  std::memset(&rm, 0, sizeof(rm));
  const uint32_t wr_box = (uint32_t)(p.n_router_cols > 256 ? p.n_router_cols / 4 : p.n_router_cols / 2);  // per CTA of a pair
  if (encode_rows(pl, &rm.x, x, T, c.D, BM) != MOE_OK || encode_rows(pl, &rm.wr, W_router, c.E, c.D, wr_box) != MOE_OK)
    return MOE_ERR_INVALID_ARG;
  // the router kernel zeroes the status word and the counters; every other
  // scratch word is written before it is read
  if (launch_router(rm, p, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_schedule(p, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (device_status &&
      cudaMemcpyAsync(device_status, p.status, sizeof(int), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
