// Persistent MoE forward kernel: dispatch (gather), routed and shared expert
// FFNs on tcgen05 tensor cores, and the fixed-order weighted combine.
//
// "Mixture-of-Kittens: MoE Megakernel for NVL72s":
//  * Sec. 3.2 "Kernel Fusion": one persistent kernel; some SMs only move
//    tokens (here: gather CTAs), the others only run expert FFNs (GEMM CTAs);
//    they signal each other through GPU-local counters.
//  * Sec. 3.2 "Maximally Deferred Synchronization": the gather walks
//    minibatches breadth-first, as far ahead as the ring allows; the GEMM CTAs
//    walk them depth-first (all up/gate tiles of a minibatch, then its down
//    tiles); the only meeting points are "minibatch m gathered" and "ring slot
//    free again".
//  * Sec. 3.3: the tokens of minibatch m (b consecutive schedule rows) go to
//    ring slot m mod slots of a fixed-size device ring; nothing is sized on
//    the host and no token is dropped.
//  * Sec. 3.4 "Shared Expert": the shared expert's up/gate tiles come first,
//    while the first minibatch is being gathered; its down-projection tiles
//    come last and store the shared output as one more staging slot per
//    token.
//  * Sec. 3.4 "Determinism": no floating-point atomics; every output element
//    is produced by one tile with a fixed K order, and the weighted sum runs
//    in a fixed slot order from a token-order fp16 staging buffer (10
//    mantissa bits: the sum's error stays below the bf16 output rounding),
//    once every staging row is stored, on all CTAs at once (a pass bound by
//    HBM bandwidth, with many loads in flight per warp).
// The expert FFN is the one of Sec. 2.1 / the blog's E_i(x) with SiLU:
// h = SiLU(x W_gate^T) * (x W_up^T) in fp32 from TMEM, stored bf16; y = h W_down^T.
//
// GEMM CTA roles (256 threads): warp 0 issues TMA loads, warp 1 issues
// tcgen05.mma (128 x 256 x 16, fp32 accumulators in TMEM, two accumulator
// buffers), warps 2-5 drain TMEM (tcgen05.ld), apply the epilogue and store.
// A GEMM1 tile is 128 rows x (128 up + 128 gate) columns; a GEMM2 tile is
// 128 rows x 256 output columns.
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint8_t* align_1024_mk(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int TMEM_COLS = 2 * ACC_COLS;  // 512: two accumulator buffers
constexpr int GATHER_BUFS = 32;          // row buffers of a gather CTA (at most)
constexpr int GATHER_STORES = 4;         // row stores a gather CTA keeps in flight
constexpr int GATHER_TOK_CHUNK = 4096;   // rows whose tokens a gather CTA stages in shared memory at a time
constexpr int EPI_STAGE_BYTES = 4 * 4224;  // 4 epilogue warps x sizeof(EpiStage)

// ------------------------------------------------------------------ MXFP8 helpers
// byte offset of (row r of a 128-row block, K-block kb of a 128-wide K step)
// inside its 512-byte scale block
__device__ __forceinline__ int sf_offset(int r, int kb) { return (r & 31) * 16 + ((r >> 5) & 3) * 4 + kb; }

// ------------------------------------------------------------------ gather (dispatch)
// Ring slot m % slots receives schedule rows [m b, min((m+1) b, R)) of x, at
// ring row (row - m b).  Gather CTA g takes the minibatch's M-tiles g, g + G,
// ...; its warps take the tile's rows.  MXFP8: the per-token E4M3 codes go to
// the ring and their E8M0 scales into the tile's scale blocks.
__device__ void gather_copy_row(const FwdParams& p, const bf16* src_row, bf16* dst_row) {
  const int lane = threadIdx.x & 31;
  const int nv = p.D / 8;  // 16-byte vectors per row
  // a whole row in flight per warp (D <= 8192 in one pass), loads before stores
  constexpr int UNR = 32;
  const uint4* src = reinterpret_cast<const uint4*>(src_row);
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
  for (int base = 0; base < nv; base += 32 * UNR) {
    uint4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nv) v[u] = __ldg(src + i);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nv) dst[i] = v[u];
    }
  }
}

// MXFP8: a token's E4M3 codes into a ring row (the warp's lanes copy 16-byte
// vectors, the whole row in flight) and its E8M0 words into the M-tile's
// scale blocks (one word per 128-wide K step, row r_in_tile of the tile)
__device__ void gather_copy_row_mx(const FwdParams& p, int t, uint8_t* dst_row, uint8_t* sf_tile, int r_in_tile) {
  const int lane = threadIdx.x & 31;
  const int nv = p.D / 16;
  constexpr int UNR = 16;  // D <= 8192 in one pass
  const uint4* src = reinterpret_cast<const uint4*>(p.xq + (size_t)t * p.D);
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
  for (int base = 0; base < nv; base += 32 * UNR) {
    uint4 v[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nv) v[u] = __ldg(src + i);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nv) dst[i] = v[u];
    }
  }
  const int nkg = p.D / BK_MX;
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(p.xs + (size_t)t * (p.D / 32));
  for (int kg = lane; kg < nkg; kg += 32)
    *reinterpret_cast<uint32_t*>(sf_tile + (size_t)kg * SF_BLOCK_BYTES + sf_offset(r_in_tile, 0)) = __ldg(sw + kg);
}

// Ring fill spread over the GEMM CTAs (MOE_DISPATCH_SPREAD): warps 6 and 7
// of GEMM CTA `part` (of `parts`) copy the rows of the M-tiles mt with
// mt % parts == part through registers, while the CTA's other warps run
// expert tiles; every part adds 1 to the minibatch's fill counter.  They sync
// among themselves with named barrier 2 (64 threads).
__device__ void gather_role_spread(const FwdParams& p, int part, int parts, volatile int* s_gflag) {
  const int w = (threadIdx.x >> 5) - 6;  // 0 or 1
  const bool lead = threadIdx.x == 6 * 32;
  constexpr int CH = BM / 32;  // 32-row chunks per M-tile
  for (int m = 0; m < p.n_mb; ++m) {
    const int mt0 = p.meta[META_MB + 4 * m + 2], ntile = p.meta[META_MB + 4 * m + 3];
    // The minibatch's M-tiles are filled in 32-row chunks: chunk c of the run
    // (M-tile c / CH) goes to part c % parts, so that a small minibatch (few
    // M-tiles) still spreads over many parts and the chunks rotate over every
    // part.  A part with no chunk in this minibatch only reports it done: it
    // neither waits for the ring slot nor writes to it (waiting would make
    // every minibatch a grid-wide step)
    const int nch = ntile * CH;
    const int i0 = ((part - mt0 * CH) % parts + parts) % parts;  // this part's first chunk of the minibatch
    const bool mine = i0 < nch;
    if (mine && m >= p.slots) {  // ring slot m % slots free again: minibatch m - slots' up/gate tiles are done
      if (lead)
        *s_gflag = wait_counter_ge(p.counters + ctr_r1(p, m - p.slots), p.meta[META_MB + 4 * (m - p.slots)],
                                   p.status, p.timeout_ns) ? 1 : 0;
      named_bar_sync(2, 64);
      if (*s_gflag == 0) break;
    }
    const int lo = m * p.b;
    const size_t slot_base = (size_t)(m % p.slots) * p.b;
    for (int i = i0; i < nch; i += parts) {
      const int mt = mt0 + i / CH;
      const int p0 = p.mtiles[4 * mt + 1], rows = p.mtiles[4 * mt + 2];
      const int r1 = min(rows, (i % CH + 1) * 32);
      for (int r = (i % CH) * 32 + w; r < r1; r += 2) {
        const int t = p.sched[(size_t)(p0 + r) * 3];
        const size_t ring_row = slot_base + (size_t)(p0 + r - lo);
        if (p.mx)
          gather_copy_row_mx(p, t, reinterpret_cast<uint8_t*>(p.ring_x) + ring_row * p.D,
                             p.sfx + (size_t)mt * (p.D / BK_MX) * SF_BLOCK_BYTES, r);
        else
          gather_copy_row(p, p.x + (size_t)t * p.D, p.ring_x + ring_row * p.D);
      }
    }
    fence_proxy_async_global();  // the ring rows are read by TMA
    named_bar_sync(2, 64);
    if (lead && m + 1 != p.test_unfilled) {
      red_release_add_gpu(p.counters + ctr_filled(p, m), 1);
      if (m == p.n_mb - 1) atomicMax(p.stamps + STAMP_LAST_FILL, (unsigned long long)globaltimer_ns());
    }
  }
}

// The ring through the TMA engine: one thread streams the CTA's rows of a
// minibatch (bf16 x rows, or MXFP8 E4M3 code rows of the per-token quantised
// x) through nbuf shared-memory row buffers (bulk load -> buffer -> bulk store
// to the ring), keeping nbuf - GATHER_STORES loads and
// up to GATHER_STORES stores in flight: the buffer of row i + ahead is the one
// row i - GATHER_STORES used, refilled once that row's store has finished
// reading it.  row_seq counts rows over the whole kernel (buffer = row_seq %
// nbuf, its mbarrier phase = (row_seq / nbuf) & 1).  Returns false if a load
// did not land within the time limit.
__device__ bool gather_rows_bulk(const FwdParams& p, const uint8_t* src, uint8_t* dst, uint32_t row_bytes, int lo,
                                 int r0, int r1, const int* tok, size_t slot_base, uint8_t* buf, uint64_t* gbar,
                                 int nbuf, uint32_t& row_seq) {
  const int n = r1 - r0;
  const int ahead = nbuf - GATHER_STORES;
  auto load = [&](int i) {
    const uint32_t q = row_seq + (uint32_t)i;
    const int b = (int)(q % (uint32_t)nbuf);
    const int t = tok[i];  // row r0 + i's token, from the shared table
    mbar_arrive_expect_tx(&gbar[b], row_bytes);
    bulk_load(buf + (size_t)b * row_bytes, src + (size_t)t * row_bytes, row_bytes, &gbar[b]);
  };
  TRACE_LOCALS();
  int loaded = min(ahead, n);
  for (int i = 0; i < loaded; ++i) load(i);
  bool ok = true;
  int i = 0;
  for (; i < n; ++i) {
    const uint32_t q = row_seq + (uint32_t)i;
    const int b = (int)(q % (uint32_t)nbuf);
    TRACE_T0();
    const bool landed = mbar_wait(&gbar[b], (q / (uint32_t)nbuf) & 1u, p.status, p.timeout_ns);
    TRACE_ADD(p, TR_GATHER_LOADWAIT);
    if (!landed) {
      ok = false;
      break;
    }
    bulk_store(dst + (slot_base + (size_t)(r0 + i - lo)) * row_bytes, buf + (size_t)b * row_bytes, row_bytes);
    bulk_commit_group();
    if (i + ahead < n) {
      {
        TRACE_T0();
        bulk_wait_group_read<GATHER_STORES>();  // rows <= i - GATHER_STORES are done reading their buffers
        TRACE_ADD(p, TR_GATHER_STOREWAIT);
      }
      load(i + ahead);
      ++loaded;
    }
  }
  // aborted: the loads issued but not yet consumed land before the buffers are left
  for (; i < loaded; ++i) {
    const uint32_t q = row_seq + (uint32_t)i;
    mbar_wait_drain(&gbar[q % (uint32_t)nbuf], (q / (uint32_t)nbuf) & 1u, p.timeout_ns);
  }
  {
    TRACE_T0();
    bulk_wait_group_all();
    TRACE_ADD(p, TR_GATHER_STOREWAIT);
  }
  TRACE_FLUSH(p);
  row_seq += (uint32_t)loaded;
  return ok;
}

__device__ void gather_role(const FwdParams& p, volatile int* s_flag, uint8_t* buf, int buf_bytes, uint64_t* gbar,
                            int* tok) {
  TRACE_LOCALS();
  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5, lane = threadIdx.x & 31;
  // a ring row: D bf16, or D E4M3 codes
  const uint32_t row_bytes = (uint32_t)p.D * (p.mx ? 1u : 2u);
  const uint8_t* src = p.mx ? p.xq : reinterpret_cast<const uint8_t*>(p.x);
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.ring_x);
  const int nbuf = min(GATHER_BUFS, buf_bytes / (int)row_bytes);  // >= 12 for D <= 8192
  uint32_t row_seq = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nbuf; ++i) mbar_init(&gbar[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  for (int m = 0; m < p.n_mb; ++m) {
    if (threadIdx.x == 0) *s_flag = 1;
    if (m >= p.slots) {
      if (threadIdx.x == 0) {
        const int need = p.meta[META_MB + 4 * (m - p.slots)];
        TRACE_T0();
        *s_flag = wait_counter_ge(p.counters + ctr_r1(p, m - p.slots), need, p.status, p.timeout_ns) ? 1 : 0;
        TRACE_ADD(p, TR_GATHER_WAIT);
      }
      __syncthreads();
      if (*s_flag == 0) break;
    }
    const int lo = m * p.b;
    const size_t slot_base = (size_t)(m % p.slots) * p.b;
    TRACE_T0();
    // contiguous row ranges per CTA for the rows themselves
    const int hi = min(p.R, lo + p.b);
    const int per = (hi - lo + p.G - 1) / p.G;
    const int r0 = lo + g * per, r1 = min(hi, r0 + per);
    if (warp == 0) {
      // the rows' tokens go to a shared table first (32 lanes, independent
      // loads), so the issuing lane never waits on a global load per row
      bool ok = true;
      for (int c0 = r0; c0 < r1 && ok; c0 += GATHER_TOK_CHUNK) {
        const int c1 = min(r1, c0 + GATHER_TOK_CHUNK);
        for (int i = lane; i < c1 - c0; i += 32) tok[i] = p.sched[(size_t)(c0 + i) * 3];
        __syncwarp();
        int okl = 1;
        if (lane == 0)
          okl = gather_rows_bulk(p, src, dst, row_bytes, lo, c0, c1, tok, slot_base, buf, gbar, nbuf, row_seq) ? 1
                                                                                                               : 0;
        ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
        __syncwarp();
      }
      if (lane == 0 && !ok) *s_flag = 0;
    } else if (p.mx) {
      // MXFP8: the other warps put the tokens' E8M0 words into the scale
      // blocks of the minibatch's M-tiles g, g + G, ... (one word per row and
      // 128-wide K step)
      const int mt0 = p.meta[META_MB + 4 * m + 2], ntile = p.meta[META_MB + 4 * m + 3];
      const int nkg = p.D / BK_MX;
      for (int i = g; i < ntile; i += p.G) {
        const int mt = mt0 + i;
        const int p0 = p.mtiles[4 * mt + 1], rows = p.mtiles[4 * mt + 2];
        uint8_t* sf_tile = p.sfx + (size_t)mt * nkg * SF_BLOCK_BYTES;
        for (int r = warp - 1; r < rows; r += nwarps - 1) {
          const int t = p.sched[(size_t)(p0 + r) * 3];
          const uint32_t* sw = reinterpret_cast<const uint32_t*>(p.xs + (size_t)t * (p.D / 32));
          for (int kg = lane; kg < nkg; kg += 32)
            *reinterpret_cast<uint32_t*>(sf_tile + (size_t)kg * SF_BLOCK_BYTES + sf_offset(r, 0)) = __ldg(sw + kg);
        }
      }
    }
    fence_proxy_async_global();
    __syncthreads();
    if (*s_flag == 0) break;  // a bulk load gave up: the minibatch is not complete
    if (threadIdx.x == 0) {
      TRACE_ADD(p, TR_GATHER_BUSY);
      if (m + 1 != p.test_unfilled) {
        red_release_add_gpu(p.counters + ctr_filled(p, m), 1);
        if (m == p.n_mb - 1) atomicMax(p.stamps + STAMP_LAST_FILL, (unsigned long long)globaltimer_ns());
      }
    }
  }
  TRACE_FLUSH(p);
}

// ------------------------------------------------------------------ operand selection
struct Operands {
  const CUtensorMap* a;
  const CUtensorMap* a64;  // routed BF16 pair tiles split over the pair: 64-row A boxes
  const CUtensorMap* b0;
  const CUtensorMap* b1;  // null: one 256-row B box
  int b_row;
  int nk;
};

__device__ __forceinline__ bool task_is_mx(const FwdParams& p, int kind) {
  return p.mx && (kind == TASK_R1 || kind == TASK_R2);
}

__device__ __forceinline__ Operands task_operands(const TensorMaps& maps, const FwdParams& p, const Task& t) {
  Operands o;
  const int kstep = p.mx ? BK_MX : BK;  // routed tensor maps are E4M3 (MXFP8) or bf16
  switch (t.kind) {
    case TASK_R1:
      o.a = &maps.ring_x; o.a64 = &maps.ring_x64; o.b0 = &maps.w_up; o.b1 = &maps.w_gate;
      o.b_row = t.e * p.I + t.n * BN_UP; o.nk = p.D / kstep;
      break;
    case TASK_R2:
      o.a = &maps.ring_h; o.a64 = &maps.ring_h64; o.b0 = &maps.w_down; o.b1 = nullptr;
      o.b_row = t.e * p.D + t.n * BN_DOWN; o.nk = p.I / kstep;
      break;
    case TASK_S1:
      o.a = &maps.x; o.a64 = nullptr; o.b0 = &maps.ws_up; o.b1 = &maps.ws_gate;
      o.b_row = t.n * BN_UP; o.nk = p.D / BK;
      break;
    default:  // TASK_S2
      o.a = &maps.h_s; o.a64 = nullptr; o.b0 = &maps.ws_down; o.b1 = nullptr;
      o.b_row = t.n * BN_DOWN; o.nk = p.I_s / BK;
      break;
  }
  return o;
}

__device__ __forceinline__ int task_nk(const FwdParams& p, int kind) {
  const int kstep = task_is_mx(p, kind) ? BK_MX : BK;
  return (kind == TASK_R1 || kind == TASK_S1) ? p.D / kstep : (kind == TASK_R2 ? p.I / kstep : p.I_s / BK);
}

// MXFP8 scale blocks of a K step: A (the tile's rows), then B's two 128-row halves
__device__ __forceinline__ void mx_scale_sources(const FwdParams& p, const Task& t, int kb, const uint8_t** src) {
  if (t.kind == TASK_R1) {  // direct dispatch: src[0] unused (the producer lanes write the A block)
    const int nkg = p.D / BK_MX;
    src[0] = p.sfx ? p.sfx + ((size_t)t.mt * nkg + kb) * SF_BLOCK_BYTES : nullptr;
    const size_t wb = ((size_t)(t.e * p.I + t.n * BN_UP) / BM * nkg + kb) * SF_BLOCK_BYTES;
    src[1] = p.w_up_sf + wb;
    src[2] = p.w_gate_sf + wb;
  } else {
    const int nkg = p.I / BK_MX;
    src[0] = p.sfh + ((size_t)t.mt * nkg + kb) * SF_BLOCK_BYTES;
    const size_t rb = (size_t)(t.e * p.D + t.n * BN_DOWN) / BM;
    src[1] = p.w_down_sf + (rb * nkg + kb) * SF_BLOCK_BYTES;
    src[2] = p.w_down_sf + ((rb + 1) * nkg + kb) * SF_BLOCK_BYTES;
  }
}

// ------------------------------------------------------------------ epilogues
// Handing an accumulator buffer back to the MMA issuer after its last TMEM
// read: every epilogue thread arrives on the local barrier (one CTA per tile),
// or one lane per warp arrives on the even CTA's barrier (CTA pairs).
// An epilogue hands its accumulator buffer back twice: the first columns once
// they are read (an MXFP8 tile in the other buffer puts its block scales
// there), the whole buffer after the last read.
struct AccRelease {
  uint64_t* local;
  uint32_t remote;  // cluster address of the even CTA's barrier
  uint64_t* head_local;
  uint32_t head_remote;
  bool pair;
};
__device__ __forceinline__ void release_bar(uint64_t* local, uint32_t remote, bool pair) {
  tc_fence_before();
  if (pair) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_remote(remote);
  } else {
    mbar_arrive(local);
  }
}
__device__ __forceinline__ void release_acc(const AccRelease& r) { release_bar(r.local, r.remote, r.pair); }
__device__ __forceinline__ void release_head(const AccRelease& r) { release_bar(r.head_local, r.head_remote, r.pair); }

// Epilogue data movement: each warp owns 32 tile rows (TMEM lanes).  A
// tcgen05.ld gives lane r the 32 columns of row r; the warp stages that 32x32
// block in shared memory (row stride 33 floats: conflict-free both ways) and
// re-reads it so that lane l handles row 4i + l/8, columns 4 (l%8) .. +3:
// every warp store then covers 4 rows x a contiguous 32-column segment.
struct EpiStage {
  float v[32][33];
};
static_assert(sizeof(EpiStage) == 4224, "epilogue staging size");

__device__ __forceinline__ void stage_block(EpiStage& st, const float* v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 32; ++j) st.v[lane][j] = v[j];
  __syncwarp();
}

__device__ __forceinline__ float4 staged4(const EpiStage& st, int rr, int cc) {
  return make_float4(st.v[rr][cc], st.v[rr][cc + 1], st.v[rr][cc + 2], st.v[rr][cc + 3]);
}

__device__ __forceinline__ uint2 pack_bf16x4(float4 f) {
  return make_uint2(pack_bf16x2(f.x, f.y), pack_bf16x2(f.z, f.w));
}

// staging rows are fp16: 10 mantissa bits keep the weighted sum's error below
// the bf16 output rounding; values saturate at the fp16 maximum (no infinities)
__device__ __forceinline__ uint32_t pack_f16x2_sat(float a, float b) {
  const float m = 65504.0f;
  __half2 h = __floats2half2_rn(fminf(fmaxf(a, -m), m), fminf(fmaxf(b, -m), m));
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float4 load_f16x4(const __half* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// up/gate tile -> h = SiLU(gate) * up (bf16): TMEM columns [0,128) up, [128,256) gate.
// dst: row 0 of the warp's rows, column 0 of the tile; ld: row stride (elements).
__device__ void epilogue_swiglu(uint32_t taddr, EpiStage& st, bf16* dst, size_t ld, int nrows, const AccRelease& rel) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int c = 0; c < BN_UP; c += 32) {
    uint32_t u[32], g[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, u);
    tmem_ld_32x32b_x32(taddr + (uint32_t)(BN_UP + c), g);
    tmem_ld_wait();
    if (c == 0) release_head(rel);
    if (c + 32 == BN_UP) {  // last TMEM read of this tile: hand the accumulator back
      release_acc(rel);
    }
    float h[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) h[j] = silu_f32(__uint_as_float(g[j])) * __uint_as_float(u[j]);
    stage_block(st, h);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3), cc = 4 * (lane & 7);
      if (rr < nrows) *reinterpret_cast<uint2*>(dst + (size_t)rr * ld + c + cc) = pack_bf16x4(staged4(st, rr, cc));
    }
    __syncwarp();
  }
}

// MXFP8 up/gate tile -> h quantised per 32 columns: E4M3 codes into the h ring
// (thread = row, 128 bytes) and one 32-bit word of four E8M0 codes into the
// tile's scale block (this tile's 128 columns are one 128-wide K step of the
// down projection).  The accumulator is handed back after the last TMEM read.
__device__ void epilogue_swiglu_mx(uint32_t taddr, uint8_t* dst_row, uint8_t* sf_block, int row, bool valid,
                                   const AccRelease& rel) {
  uint32_t q[4][8];
  uint32_t scales = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t u[32], g[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)(32 * c), u);
    tmem_ld_32x32b_x32(taddr + (uint32_t)(BN_UP + 32 * c), g);
    tmem_ld_wait();
    if (c == 0) release_head(rel);
    if (c == 3) {
      release_acc(rel);
    }
    float h[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) h[j] = silu_f32(__uint_as_float(g[j])) * __uint_as_float(u[j]);
    scales |= mx_quantize32(h, q[c]) << (8 * c);
  }
  if (valid) {
    uint4* d = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      d[2 * c] = make_uint4(q[c][0], q[c][1], q[c][2], q[c][3]);
      d[2 * c + 1] = make_uint4(q[c][4], q[c][5], q[c][6], q[c][7]);
    }
    *reinterpret_cast<uint32_t*>(sf_block + sf_offset(row, 0)) = scales;
  }
}

// routed down-projection tile -> fp16 staging rows (route j = t k + slot from
// the schedule table), restaged through shared memory so that every warp
// store covers 4 rows x 64 contiguous bytes; y_mine: offset of this thread's
// row's 256-column segment.  The buffer is handed back after the last TMEM
// read (with two accumulator buffers the MMA issuer rarely waits for it).
// A value outside the fp16 range (or NaN) is saturated and raises
// FLAG_STAGING_OVERFLOW in flags (the forward goes on; its status says so).
// ncols of the warp's 32 TMEM lanes (from taddr) are output columns col0 .. col0 + ncols - 1 of
// its rows: all 256 columns, or (a split tile: lanes 0-63 columns 0-127, lanes 64-127 columns
// 128-255 of the same 64 rows) 128 of them
__device__ void epilogue_copy_f16_staged(uint32_t taddr, EpiStage& st, __half* Y, long long y_mine, int nrows,
                                         const AccRelease& rel, int* flags, int ncols = BN_DOWN, int col0 = 0) {
  const int lane = threadIdx.x & 31;
  bool ovf = false;
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
    tmem_ld_wait();
    if (c == 0) release_head(rel);
    if (c + 32 == ncols) release_acc(rel);
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    stage_block(st, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3), cc = 4 * (lane & 7);
      const long long yr = __shfl_sync(0xffffffffu, y_mine, rr);
      if (rr < nrows) {
        const float4 f = staged4(st, rr, cc);
        const float a = fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w)));
        ovf |= !(a <= 65504.0f) || f.x != f.x || f.y != f.y || f.z != f.z || f.w != f.w;
        *reinterpret_cast<uint2*>(Y + yr + col0 + c + cc) =
            make_uint2(pack_f16x2_sat(f.x, f.y), pack_f16x2_sat(f.z, f.w));
      }
    }
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, ovf) && lane == 0) atomicOr(flags, FLAG_STAGING_OVERFLOW);
}

// BF16 CTA pairs store their epilogue rows from registers: lane l holds 32
// columns of its row per TMEM load and writes them as two 32-byte vectors
// (full L2 sectors), so the kernel keeps no staging blocks and has room for a
// seventh operand stage.  live: the row is a real tile row.
//
// Up/gate tile -> h = SiLU(gate) * up (bf16): up columns at taddr + c, gate
// columns at taddr + gate_off + c, c < ncols (a whole tile: 128 and 128; a tile
// split over the pair: this lane's 64 h columns, up then gate); dst: the row's
// first h column.
__device__ void epilogue_swiglu_direct(uint32_t taddr, bf16* dst, bool live, const AccRelease& rel, int gate_off,
                                       int ncols) {
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint32_t u[32], g[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, u);
    tmem_ld_32x32b_x32(taddr + (uint32_t)(gate_off + c), g);
    tmem_ld_wait();
    if (c == 0) release_head(rel);
    if (c + 32 == ncols) release_acc(rel);  // last TMEM read of this tile
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = pack_bf16x2(silu_f32(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]),
                         silu_f32(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]));
    if (live) {
      st_global_v8(dst + c, w);
      st_global_v8(dst + c + 16, w + 8);
    }
  }
}

// Down-projection tile -> fp16 staging row: ncols TMEM columns from taddr are
// output columns 0 .. ncols - 1 from yrow (all 256, or 128 for a split tile);
// saturation at the fp16 maximum and NaN are flagged as in the staged form.
__device__ void epilogue_copy_f16_direct(uint32_t taddr, __half* yrow, bool live, const AccRelease& rel, int* flags,
                                         int ncols) {
  bool ovf = false;
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
    tmem_ld_wait();
    if (c == 0) release_head(rel);
    if (c + 32 == ncols) release_acc(rel);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
      ovf |= !(fmaxf(fabsf(a), fabsf(b)) <= 65504.0f) || a != a || b != b;
      w[j] = pack_f16x2_sat(a, b);
    }
    if (live) {
      st_global_v8(yrow + c, w);
      st_global_v8(yrow + c + 16, w + 8);
    }
  }
  if (__any_sync(0xffffffffu, ovf && live) && (threadIdx.x & 31) == 0) atomicOr(flags, FLAG_STAGING_OVERFLOW);
}

// ------------------------------------------------------------------ combine
// Weighted sum back in token order (Eq. MoE), in fp32 with one rounding to
// bf16 at the end: out[t] = y_s[t] + g[t,0] Y[t,0] + ... + g[t,k-1] Y[t,k-1],
// the shared expert's output (staging slot k; absent without a shared expert)
// first, then the routed slots in slot order, whatever order the tiles ran in.
// It runs on every CTA once every staging row is stored, as a stream bound by
// HBM bandwidth.  A unit is one token and one 256-column tile; its kY staging
// rows are one contiguous block of kY x 512 bytes, and units in staging order
// are consecutive blocks.  A round is 8 consecutive units, one per warp; each
// CTA takes a contiguous range of rounds and streams them into its (idle)
// stage buffers with one bulk copy per round, up to CMB_BUFS rounds ahead;
// lane l of a warp sums columns 8l .. 8l + 7 of its unit from shared memory.
constexpr int CMB_BUFS = 8;
constexpr int CMB_BAR_OFFSET = 1024;  // barriers in the epilogue staging area, past the gather's

__device__ __forceinline__ void fma_f16x8(float* acc, float g, uint4 w) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
    acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
  }
}

// buf: buf_bytes of shared memory free for the pass; bars: CMB_BUFS free
// mbarrier slots; ok: a shared flag.  Every thread of the CTA calls it.  The
// rounds are split statically over the grid's CTAs, or (cluster launch
// control: the grid is far larger than the CTAs that run) claimed in chunks of
// CMB_CHUNK rounds from a global counter.  Which CTA sums a unit does not
// change its arithmetic.
constexpr int CMB_CHUNK = 16;
__device__ void combine_role(const FwdParams& p, uint8_t* buf, int buf_bytes, uint64_t* bars, volatile int* ok) {
  const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
  const int warps = (int)(blockDim.x >> 5);  // units per round
  const int k = p.k, kY = p.kY;
  const bool shared = kY > k;
  const uint32_t unit_bytes = (uint32_t)kY * BN_DOWN * 2;
  const uint32_t round_bytes = (uint32_t)warps * unit_bytes;
  const int nb = min(CMB_BUFS, buf_bytes / (int)round_bytes);  // >= 2: kY <= 17 and >= 192 KB of buffers
  const long long per_tt = (long long)p.N2 * BM;              // units of one token tile
  const long long n_units = (long long)((p.T + BM - 1) / BM) * per_tt;
  const long long n_rounds = (n_units + warps - 1) / warps;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nb; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  volatile long long* s_r0 = reinterpret_cast<volatile long long*>(bars + CMB_BUFS);
  uint32_t seq = 0;  // rounds this CTA has streamed so far (buffer = seq % nb, phase = (seq / nb) & 1)
  for (int range = 0;; ++range) {
    long long r0;
    int nr;
    if (p.clc) {
      if (threadIdx.x == 0) *s_r0 = (long long)atomicAdd(p.counters + ctr_combine(p), 1) * CMB_CHUNK;
      __syncthreads();
      r0 = *s_r0;
      nr = (int)max(0ll, min(n_rounds, r0 + CMB_CHUNK) - r0);
    } else {
      if (range > 0) break;
      const long long per_cta = (n_rounds + gridDim.x - 1) / gridDim.x;
      r0 = (long long)blockIdx.x * per_cta;
      nr = (int)max(0ll, min(n_rounds, r0 + per_cta) - r0);
    }
    if (nr == 0) break;
    auto issue = [&](int i) {  // this range's round i into buffer (seq + i) % nb
      const uint32_t q = seq + (uint32_t)i;
      const long long u = (r0 + i) * warps;
      const uint32_t bytes = (uint32_t)min((long long)warps, n_units - u) * unit_bytes;
      mbar_arrive_expect_tx(&bars[q % nb], bytes);
      bulk_load(buf + (size_t)(q % nb) * round_bytes, p.Y + (size_t)u * kY * BN_DOWN, bytes, &bars[q % nb]);
    };
    __syncthreads();  // every warp is done with the previous range's buffers
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();
      for (int i = 0; i < min(nb, nr); ++i) issue(i);
    }
    int issued = min(nb, nr);  // thread 0: rounds whose copies were issued
    // router weights of the warp's next unit, loaded a round ahead: lane s holds slot s
    auto unit_tok = [&](int i) {
      const long long u = (r0 + i) * warps + warp;
      const int t = (int)(u / per_tt) * BM + (int)(u % BM);
      return (i < nr && u < n_units && t < p.T) ? t : -1;
    };
    int tok = unit_tok(0);
    float g = tok >= 0 && lane < k ? p.topk_w[(size_t)tok * k + lane] : 0.0f;
    int i = 0;
    for (; i < nr; ++i) {
      const uint32_t q = seq + (uint32_t)i;
      if (threadIdx.x == 0) *ok = mbar_wait(&bars[q % nb], (q / nb) & 1u, p.status, p.timeout_ns) ? 1 : 0;
      __syncthreads();  // also: every warp is done with round i - 1
      if (*ok == 0) break;
      if (threadIdx.x == 0 && i >= 1 && i - 1 + nb < nr) {  // refill the buffer round i - 1 used
        fence_proxy_async_smem();
        issue(i - 1 + nb);
        ++issued;
      }
      const int tok_next = unit_tok(i + 1);
      const float g_next = tok_next >= 0 && lane < k ? p.topk_w[(size_t)tok_next * k + lane] : 0.0f;
      if (tok >= 0) {
        const __half* y = reinterpret_cast<const __half*>(buf + (size_t)(q % nb) * round_bytes +
                                                          (size_t)warp * unit_bytes) + 8 * lane;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        if (shared) fma_f16x8(acc, 1.0f, *reinterpret_cast<const uint4*>(y + (size_t)k * BN_DOWN));  // exact
#pragma unroll 4
        for (int s = 0; s < k; ++s)
          fma_f16x8(acc, __shfl_sync(0xffffffffu, g, s), *reinterpret_cast<const uint4*>(y + (size_t)s * BN_DOWN));
        const long long u = (r0 + i) * warps + warp;
        const int n = (int)((u / BM) % p.N2);
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(p.out + (size_t)tok * p.D + n * BN_DOWN + 8 * lane) = o;
      }  // (tok is the same for the whole warp: all lanes or none take part in the shuffles)
      tok = tok_next;
      g = g_next;
    }
    // copies still in flight (an abort) land before the CTA leaves
    if (threadIdx.x == 0)
      for (int j = i; j < issued; ++j) {
        const uint32_t q = seq + (uint32_t)j;
        mbar_wait_drain(&bars[q % nb], (q / nb) & 1u, p.timeout_ns);
      }
    __syncthreads();
    if (*ok == 0) break;
    seq += (uint32_t)nr;  // every round of the range was streamed (only thread 0 counts `issued`)
  }
}

// ------------------------------------------------------------------ the kernel
// Stage geometry of the two kernel flavours: one CTA per tile (A 128 rows + B
// 256 rows per stage, MXFP8 scale blocks after them) or CTA pairs (A 128 rows
// + B 128 rows per CTA and stage).
// kMx (pairs only): the routed tiles are MXFP8; their scale blocks take one
// slot per stage after the stages.  Then the barriers and small shared
// variables (BAR_BYTES) and the epilogue staging.
constexpr int BAR_BYTES = 512;
constexpr int QN = 8;  // unit queue slots (the producer runs at most a few units ahead)
// kDirectEpi (BF16 pairs): the epilogue stores rows straight from registers,
// so the area after the barriers only holds the combine's and the gather's
// barriers (1.5 KB) and the stages take a seventh slot.
template <bool kPair, bool kMx = false>
struct MegaGeom {
  static constexpr bool kDirectEpi = kPair && !kMx;
  static constexpr int stages = kPair ? (kMx ? PAIR_MX_STAGES : PAIR_STAGES) : STAGES;
  static constexpr int stride = kPair ? PAIR_STAGE_BYTES : STAGE_STRIDE;
  static constexpr int sf_bytes = kMx ? stages * SF_STAGE_BYTES : 0;
  static constexpr int epi_bytes = kDirectEpi ? 1536 : EPI_STAGE_BYTES;
  static constexpr int smem_bytes = stages * stride + sf_bytes + 1024 /*align*/ + BAR_BYTES + epi_bytes;
};
static_assert(MegaGeom<true>::smem_bytes <= 232448 && MegaGeom<false>::smem_bytes <= 232448 &&
                  MegaGeom<true, true>::smem_bytes <= 232448,
              "shared memory");
// the small area (BF16 pairs) holds the gather's barriers and, past them, the
// combine's barriers and claim word; the gather's token table goes to the
// stage buffers there, which keep room for at least 12 rows of D <= 8192
static_assert(CMB_BAR_OFFSET + (CMB_BUFS + 1) * 8 <= MegaGeom<true>::epi_bytes && GATHER_BUFS * 8 <= CMB_BAR_OFFSET &&
                  EPI_STAGE_BYTES >= GATHER_BUFS * 8 + GATHER_TOK_CHUNK * 4 &&
                  MegaGeom<true>::stages * PAIR_STAGE_BYTES - GATHER_TOK_CHUNK * 4 >= 12 * 8192 * 2,
              "shared areas of the gather and the combine");

template <bool kPair>
__device__ __forceinline__ void tmem_alloc_all(uint32_t* slot) {
  if constexpr (kPair) {
    tmem_alloc_pair<TMEM_COLS>(slot);
    tmem_relinquish_pair();
  } else {
    tmem_alloc<TMEM_COLS>(slot);
    tmem_relinquish();
  }
}

// Accumulator buffer of each task: the two TMEM buffers alternate.  A routed
// MXFP8 task puts its block scales in the first 12 columns of the other
// buffer, which the previous task's epilogue hands back after its first TMEM
// read.  Per-buffer use counts give the mbarrier parities; the MMA issuer and
// the epilogue walk the same tasks, so they pick the same buffers.
struct AccSeq {
  uint32_t uses0 = 0u, uses1 = 0u;  // scalars, not an array: no local memory
  uint32_t alt = 0u;
  __device__ __forceinline__ uint32_t next() {
    const uint32_t b = alt;
    alt ^= 1u;
    return b;
  }
  __device__ __forceinline__ uint32_t uses(uint32_t b) const { return b ? uses1 : uses0; }
  __device__ __forceinline__ void used(uint32_t b) {
    if (b) ++uses1;
    else ++uses0;
  }
};

// Units of work: a unit is one task, or with CTA pairs two consecutive tasks
// (2u: even CTA, 2u + 1: odd CTA) that share one weight tile.  The producer of
// each GEMM CTA (of the even CTA of a pair) claims units from a global counter
// in increasing order, one ahead of the unit it is loading, and hands each to
// the MMA issuer, the epilogue and (pairs) the odd CTA through a queue of QN
// slots in shared memory.  Every dependency of a unit points to an earlier
// unit, and every unit below the highest claimed one has been claimed, so the
// smallest unfinished unit can always proceed.
struct TaskWalk {
  int n_units, rank;
  bool pair;
  __device__ __forceinline__ int task(int u) const { return pair ? 2 * u + rank : u; }
};

template <bool kPair, bool kMxPair = false>
__device__ __forceinline__ void mega_body(const TensorMaps& maps, const FwdParams& p) {
  using G = MegaGeom<kPair, kMxPair>;
  constexpr int NST = G::stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024_mk(smem_raw);
  uint8_t* sf_slots = smem + NST * G::stride;  // pairs with MXFP8 tiles: scale blocks per stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_slots + G::sf_bytes);
  static_assert(2 * NST + 7 <= 24 && 48 * 8 + QN * 4 <= 52 * 8 && 56 * 8 <= BAR_BYTES, "barrier area");
  uint64_t* full = bars;
  uint64_t* empty = bars + NST;
  uint64_t* tfull = bars + 2 * NST;
  uint64_t* tempty = tfull + 2;
  uint64_t* thead = tempty + 2;  // first columns of a buffer read by its epilogue
  uint64_t* drain = thead + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = s_flag + 1;  // s_ok + 1: the spread ring fill's flag, s_ok + 2: the epilogue's unit
  uint64_t* qfull = bars + 32;       // unit queue: slot written
  uint64_t* qempty = bars + 40;      // ... slot read by every reader
  volatile int* qslot = reinterpret_cast<volatile int*>(bars + 48);
  uint64_t* clc_bar = bars + 52;     // cluster launch control: the response's barrier ...
  void* clc_resp = bars + 54;        // ... and the 16-byte response (16-byte aligned)
  EpiStage* epi = reinterpret_cast<EpiStage*>(sf_slots + G::sf_bytes + BAR_BYTES);
#ifdef MOE_TRACE
  volatile uint64_t* s_issue_ns = bars + 24;  // per stage: when its loads were issued (trace builds)
#endif

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_gather = (int)blockIdx.x < p.G;
  // cluster launch control: the grid has one CTA per task of the largest
  // possible task list; a CTA launched past the actual list only starts once
  // every real task's token is spent (launches go in index order, and the
  // running CTAs cancel in that order), so it has nothing to do
  // (the first n_gemm GEMM CTAs also fill the ring in spread dispatch: they stay)
  if (!kPair && p.clc && !is_gather && (int)blockIdx.x - p.G >= max(p.meta[META_N_TASKS], p.n_gemm)) return;
  if (threadIdx.x == 0) {
    atomicMin(p.stamps + STAMP_START, (unsigned long long)globaltimer_ns());
    TRACE_SET(p, TR_START_NS, globaltimer_ns());
    TRACE_SET(p, TR_START_CLK, clock64());
  }
  if (threadIdx.x == 0) DBG_SET(p, DBG_PHASE, 1);

  if (is_gather) {
    // the stage buffers hold rows in flight; the barriers live in the (unused) epilogue staging area
    if constexpr (G::kDirectEpi) {
      // the small area after the barriers holds the gather's barriers only; its token
      // table (GATHER_TOK_CHUNK ints) takes the end of the stage buffers
      constexpr int rows_bytes = NST * G::stride - GATHER_TOK_CHUNK * 4;
      gather_role(p, s_flag, smem, rows_bytes, reinterpret_cast<uint64_t*>(epi),
                  reinterpret_cast<int*>(smem + rows_bytes));
    } else {
      gather_role(p, s_flag, smem, NST * G::stride, reinterpret_cast<uint64_t*>(epi),
                  reinterpret_cast<int*>(reinterpret_cast<uint64_t*>(epi) + GATHER_BUFS));
    }
    __syncthreads();
  } else {
    const int cta = blockIdx.x - p.G;
    const int n_tasks = p.meta[META_N_TASKS];
    TaskWalk walk;
    walk.pair = kPair;
    walk.rank = kPair ? (int)(cluster_ctarank() & 1u) : 0;
    walk.n_units = kPair ? n_tasks >> 1 : n_tasks;
    const bool leader = walk.rank == 0;  // the CTA that issues the MMAs
    if (threadIdx.x == 0) {
      for (int s = 0; s < NST; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&tfull[a], 1);
        mbar_init(&tempty[a], kPair ? 8 : 128);  // pairs: one arrival per epilogue warp of both CTAs
        mbar_init(&thead[a], kPair ? 8 : 128);
      }
      mbar_init(drain, 1);
      mbar_init(clc_bar, 1);
      for (int i = 0; i < QN; ++i) {
        mbar_init(&qfull[i], 1);
        mbar_init(&qempty[i], kPair ? 4 : 2);  // MMA issuer + epilogue (pairs: + the odd CTA's producer and epilogue)
      }
      fence_barrier_init();
    }
    if (warp == 1) tmem_alloc_all<kPair>(tmem_slot);
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // the other CTA's barriers exist before anything targets them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
      DBG_SET(p, DBG_RANK, walk.rank);
      DBG_SET(p, DBG_TMEM, tmem);
      DBG_SET(p, DBG_PHASE, 2);
    }
    // waits on barriers that the other CTA of a pair helps complete
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
      if constexpr (kPair) return mbar_wait_cluster(bar, parity, p.status, p.timeout_ns);
      else return mbar_wait(bar, parity, p.status, p.timeout_ns);
    };

    if (warp == 0) {
      // ---------------- TMA producer (whole warp: lane 0 waits, loads B and
      // arrives; with direct dispatch every lane also gathers 4 of the tile's
      // 128 token rows per K step, and for MXFP8 writes their scale words)
      const bool lead_lane = lane == 0;
      TRACE_LOCALS();
      if (lead_lane) {
        prefetch_tensormap(&maps.x);
        prefetch_tensormap(&maps.ring_x);
        prefetch_tensormap(&maps.w_up);
        prefetch_tensormap(&maps.w_gate);
        prefetch_tensormap(&maps.ring_h);
        prefetch_tensormap(&maps.w_down);
        if (p.direct) prefetch_tensormap(&maps.x_rows);
      }
      // pairs: every load of both CTAs is counted on the even CTA's full barrier
      const uint32_t full_even = kPair ? mapa_shared(full, 0) : 0u;
      const uint32_t q_odd = kPair ? mapa_shared(const_cast<int*>(qslot), 1) : 0u;
      const uint32_t qfull_odd = kPair ? mapa_shared(qfull, 1) : 0u;
      const uint32_t qempty_even = kPair ? mapa_shared(qempty, 0) : 0u;
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      // even / only CTA: the unit claimed for the next queue slot.  Every
      // claim takes the next unit from the global counter, so the claimed
      // units are always a prefix of the task order.  With cluster launch
      // control a claim also needs a work token: this CTA's own launch, then
      // one launch of this grid cancelled before it started (requested while
      // the previous unit loads); no token, no further claim.
      int claim = 0;
      bool clc_pending = false;
      uint32_t clc_phase = 0;
      if (lead_lane && leader) claim = atomicAdd(p.counters + ctr_claim(p), 1);
      for (int i = 0; ok; ++i) {
        const int slot = i % QN;
        const uint32_t qpar = (uint32_t)(i / QN) & 1u;
        int u = -2;  // -2: a wait ran out; -1: no units left
        if (lead_lane) {
          if (leader) {  // publish the claimed unit, then claim the one after it
            if (clc_pending) {
              clc_pending = false;
              uint32_t cx = 0;
              if (!mbar_wait(clc_bar, clc_phase, p.status, p.timeout_ns)) {
                claim = INT_MAX;
              } else {
                clc_phase ^= 1u;
                claim = (clc_query(clc_resp, &cx) && (int)cx >= p.G) ? atomicAdd(p.counters + ctr_claim(p), 1)
                                                                    : INT_MAX;
              }
            }
            if (wait_bar(&qempty[slot], qpar ^ 1u)) {
              u = claim < walk.n_units ? claim : -1;
              qslot[slot] = u;
              if constexpr (kPair) {
                st_shared_cluster_u32(q_odd + 4u * slot, (uint32_t)u);
                mbar_arrive_remote_cluster(qfull_odd + 8u * slot);
              }
              mbar_arrive(&qfull[slot]);
              if (u >= 0) {
                if (!kPair && p.clc) {
                  mbar_arrive_expect_tx(clc_bar, 16u);
                  clc_try_cancel(clc_resp, clc_bar);
                  clc_pending = true;
                } else {
                  claim = atomicAdd(p.counters + ctr_claim(p), 1);
                }
              }
            }
          } else if (wait_bar(&qfull[slot], qpar)) {  // odd CTA: the even CTA's unit
            u = qslot[slot];
          }
        }
        u = __shfl_sync(0xffffffffu, u, 0);
        if (kPair && lead_lane && !leader && u != -2) mbar_arrive_remote(qempty_even + 8u * slot);
        if (u < 0) {
          ok = u == -1;
          break;
        }
        if (!DBG_CHECK(p, walk.task(u) < p.n_tasks_max, 1, u, walk.task(u), p.n_tasks_max)) break;
        const Task t = p.tasks[walk.task(u)];
        int good = 1;
        if (lead_lane) {
          DBG_SET(p, DBG_PROD_UNIT, u);
          DBG_SET(p, DBG_PROD_WAIT, 2);
          TRACE_T0();
          if (t.dep0 >= 0 && !wait_counter_ge(p.counters + t.dep0, t.need0, p.status, p.timeout_ns)) good = 0;
          if (good && t.dep1 >= 0 && !wait_counter_ge(p.counters + t.dep1, t.need1, p.status, p.timeout_ns)) good = 0;
          TRACE_ADD(p, TR_PROD_DEP);
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
        fence_proxy_async_global();
        const Operands o = task_operands(maps, p, t);
        const bool mx = task_is_mx(p, t.kind);
        const bool gather_a = p.direct && t.kind == TASK_R1;
        // MXFP8 direct dispatch: the lanes write the A scale block (the tile's
        // 128 tokens' E8M0 words of this K step) into shared memory themselves
        const bool sf_lanes = gather_a && mx;
        // pairs: this CTA's half of B -- up (even) or gate (odd) rows for
        // GEMM1, the first or second 128 output columns for GEMM2
        const CUtensorMap* bmap_pair = o.b1 ? (walk.rank ? o.b1 : o.b0) : o.b0;
        const int brow_pair = o.b1 ? o.b_row : o.b_row + 128 * walk.rank;
        // lane l handles tile rows 4l .. 4l+3 (rows past the tile's end repeat
        // its first token: discarded rows, in-bounds reads)
        int tok[4] = {0, 0, 0, 0};
        uint32_t sfw[4][4];  // MXFP8: scale words of the 4 rows, 4 K steps ahead
        const int nkg = p.D / BK_MX;
        if (gather_a || sf_lanes) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 4 * lane + j;
            tok[j] = p.sched[(size_t)(t.p0 + (r < t.rows ? r : 0)) * 3];
          }
          if (mx) {
#pragma unroll
            for (int d = 0; d < 4; ++d)
#pragma unroll
              for (int j = 0; j < 4; ++j)
                sfw[d][j] = d < o.nk ? *reinterpret_cast<const uint32_t*>(p.xs + (size_t)tok[j] * (nkg * 4) + d * 4) : 0u;
          }
        }
        // pairs: one K step's loads into `stage` (lane 0 only), counted on the even CTA's full barrier
        auto issue_pair = [&](uint32_t stage, int kb) {
          uint8_t* sa = smem + stage * G::stride;
          uint8_t* sb = sa + A_STAGE_BYTES;
          const int kc = kb * (mx ? BK_MX : BK);
          // a split tile: 64 A rows per CTA (8 KB)
          const bool half = !kMxPair && t.half;
          if (leader)
            mbar_arrive_expect_tx(&full[stage], 2u * (uint32_t)(mx ? PAIR_MX_STAGE_TX
                                                                   : (half ? PAIR_STAGE_BYTES - A_STAGE_BYTES / 2
                                                                           : PAIR_STAGE_BYTES)));
          const uint32_t fb = full_even + stage * 8u;
          tma_load_2d_pair(sa, half ? o.a64 : o.a, fb, kc, t.a_row);
          if (half && t.kind == TASK_R1) {
            // a split up/gate tile: this CTA's 128 weight rows are up rows 64 r .. 64 r + 63
            // of the column tile, then the same gate rows, so each TMEM lane holds the up and
            // the gate values of the same h columns
            tma_load_2d_pair(sb, &maps.w_up64, fb, kc, o.b_row + 64 * walk.rank);
            tma_load_2d_pair(sb + PAIR_B_STAGE_BYTES / 2, &maps.w_gate64, fb, kc, o.b_row + 64 * walk.rank);
          } else {
            tma_load_2d_pair(sb, bmap_pair, fb, kc, brow_pair);
          }
          if constexpr (kMxPair) {
            if (mx) {  // scale blocks: this CTA's A rows, then all 256 B rows (two blocks)
              uint8_t* ssf2 = sf_slots + stage * SF_STAGE_BYTES;
              if (t.kind == TASK_R1) {
                const int nkg1 = p.D / BK_MX;
                const int ub = (t.e * p.I + t.n * BN_UP) / BM;
                tma_load_2d_pair(ssf2, &maps.sf_x, fb, 0, 4 * (t.mt * nkg1 + kb));
                tma_load_2d_pair(ssf2 + SF_BLOCK_BYTES, &maps.sf_up, fb, 0, 4 * (ub * nkg1 + kb));
                tma_load_2d_pair(ssf2 + 2 * SF_BLOCK_BYTES, &maps.sf_gate, fb, 0, 4 * (ub * nkg1 + kb));
              } else {
                const int nkg2 = p.I / BK_MX;
                const int rb = (t.e * p.D + t.n * BN_DOWN) / BM;
                tma_load_2d_pair(ssf2, &maps.sf_h, fb, 0, 4 * (t.mt * nkg2 + kb));
                tma_load_2d_pair(ssf2 + SF_BLOCK_BYTES, &maps.sf_down, fb, 0, 4 * (rb * nkg2 + kb));
                tma_load_2d_pair(ssf2 + 2 * SF_BLOCK_BYTES, &maps.sf_down, fb, 0, 4 * ((rb + 1) * nkg2 + kb));
              }
            }
          }
        };
        if constexpr (kPair) {
          // pairs gather no rows in the producer: lane 0 alone runs the K steps,
          // with no warp-wide exchange per step (the single issuing thread's
          // loop is on the critical path)
          if (lead_lane) {
            for (int kb = 0; kb < o.nk; ++kb) {
              TRACE_T0();
              if (!wait_bar(&empty[stage], phase ^ 1u)) { ok = false; break; }
              TRACE_ADD(p, TR_PROD_EMPTY);
#ifdef MOE_TRACE
              s_issue_ns[stage] = globaltimer_ns();
#endif
              issue_pair(stage, kb);
              ++issued;
              if (++stage == NST) { stage = 0; phase ^= 1u; }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        } else {
        for (int kb = 0; kb < o.nk; ++kb) {
          int free = 1;
          if (lead_lane) {
            DBG_SET(p, DBG_PROD_WAIT, 1);
            TRACE_T0();
            free = wait_bar(&empty[stage], phase ^ 1u) ? 1 : 0;
            TRACE_ADD(p, TR_PROD_EMPTY);
            DBG_SET(p, DBG_PROD_WAIT, 0);
            if (!DBG_CHECK(p, stage < (uint32_t)NST, 2, stage, phase, u)) free = 0;
          }
          if (!__shfl_sync(0xffffffffu, free, 0)) { ok = false; break; }
          uint8_t* sa = smem + stage * G::stride;
          uint8_t* sb = sa + A_STAGE_BYTES;
          uint8_t* ssf = sa + STAGE_BYTES;
          // a K step is 64 bf16 or 128 E4M3 elements: 128 bytes per row either way
          const int kc = kb * (mx ? BK_MX : BK);
#ifdef MOE_TRACE
          if (lead_lane) s_issue_ns[stage] = globaltimer_ns();
#endif
          if constexpr (kPair) {
            if (lead_lane) issue_pair(stage, kb);
          } else {
            if (gather_a)
              tma_gather4(sa + lane * 4 * 128, &maps.x_rows, &full[stage], kc, tok[0], tok[1], tok[2], tok[3]);
            {
              if (sf_lanes) {  // the tile's A scale block, written here rather than copied
                const int d = kb & 3;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t w = 0;
#pragma unroll
                  for (int dd = 0; dd < 4; ++dd)
                    if (dd == d) w = sfw[dd][j];
                  *reinterpret_cast<uint32_t*>(ssf + sf_offset(4 * lane + j, 0)) = w;
                }
                if (kb + 4 < o.nk) {  // refill this slot with K step kb + 4
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const uint32_t w =
                        *reinterpret_cast<const uint32_t*>(p.xs + (size_t)tok[j] * (nkg * 4) + (kb + 4) * 4);
#pragma unroll
                    for (int dd = 0; dd < 4; ++dd)
                      if (dd == d) sfw[dd][j] = w;
                  }
                }
                fence_proxy_async_smem();
              }
            }
            __syncwarp();
            if (lead_lane) {
              // bytes the TMA engine delivers (the scale block written above is not counted)
              const uint32_t tx = (mx ? (uint32_t)MX_STAGE_TX : (uint32_t)STAGE_BYTES) -
                                  (sf_lanes ? (uint32_t)SF_BLOCK_BYTES : 0u);
              mbar_arrive_expect_tx(&full[stage], tx);
              if (!gather_a) tma_load_2d(sa, o.a, &full[stage], kc, t.a_row);
              if (o.b1) {
                tma_load_2d(sb, o.b0, &full[stage], kc, o.b_row);
                tma_load_2d(sb + B_STAGE_BYTES / 2, o.b1, &full[stage], kc, o.b_row);
              } else {
                tma_load_2d(sb, o.b0, &full[stage], kc, o.b_row);
              }
              if (mx) {
                const uint8_t* src[3];
                mx_scale_sources(p, t, kb, src);
                for (int i = sf_lanes ? 1 : 0; i < 3; ++i)
                  bulk_load(ssf + i * SF_BLOCK_BYTES, src[i], SF_BLOCK_BYTES, &full[stage]);
              }
              // L2 prefetch of the tiles p.l2_prefetch K steps ahead: the loads that
              // follow then wait for L2, not for HBM
              const int kp = kb + p.l2_prefetch;
              if (p.l2_prefetch > 0 && kp < o.nk) {
                const int kcp = kp * (mx ? BK_MX : BK);
                if (!gather_a) tma_prefetch_2d(o.a, kcp, t.a_row);
                tma_prefetch_2d(o.b0, kcp, o.b_row);
                if (o.b1) tma_prefetch_2d(o.b1, kcp, o.b_row);
              }
            }
          }
          ++issued;
          if (lead_lane) DBG_SET(p, DBG_PROD_ISSUED, issued);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        }  // one CTA per tile
      }
      // a cancellation request still in flight is answered before the CTA leaves
      if (lead_lane && clc_pending) mbar_wait_drain(clc_bar, clc_phase, p.timeout_ns);
      // the last loads issued have landed before the CTA may leave (pairs: the
      // even CTA's full barriers count both CTAs' loads, and the odd CTA waits
      // for the even one at the cluster barrier below)
      if (lead_lane && leader)
        for (int i = (issued > NST ? issued - NST : 0); i < issued; ++i)
          mbar_wait_drain(&full[i % NST], (uint32_t)(i / NST) & 1u, p.timeout_ns);
      if (lead_lane) TRACE_FLUSH(p);
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer (pairs: the even CTA issues for both)
      if (leader && elect_one()) {
        TRACE_LOCALS();
        const uint32_t idesc = idesc_bf16_f32(kPair ? 2 * BM : BM, 256);
        const uint32_t idesc_mx = idesc_mxf8_e4m3(kPair ? 2 * BM : BM, 256);
        uint32_t stage = 0, phase = 0;
        AccSeq accs;
        bool ok = true;
#ifdef MOE_DEBUG_LOG
        int mma_stages = 0;
#endif
        for (int i = 0; ok; ++i) {
          const int slot = i % QN;
          if (!wait_bar(&qfull[slot], (uint32_t)(i / QN) & 1u)) break;
          const int u = qslot[slot];
          if (u < 0) {  // (the branch has the value: the slot may be reused after the arrive)
            mbar_arrive(&qempty[slot]);
            break;
          }
          mbar_arrive(&qempty[slot]);
          const int kind = p.tasks[walk.task(u)].kind;
          const bool mx = task_is_mx(p, kind);
          const int nk = task_nk(p, kind);
          // a split tile (BF16 pairs): one M = 128 MMA, 64 rows per CTA
          const uint32_t idesc_u = (kPair && !kMxPair && p.tasks[walk.task(u)].half) ? idesc_bf16_f32(BM, 256) : idesc;
          const uint32_t acc = accs.next();
          DBG_SET(p, DBG_MMA_UNIT, u);
          DBG_SET(p, DBG_MMA_ACC, acc);
#ifdef MOE_DEBUG_LOG
          if (kPair) {
            const Task& t0 = p.tasks[2 * u];
            const Task& t1 = p.tasks[2 * u + 1];
            if (!DBG_CHECK(p, t0.kind == t1.kind && t0.n == t1.n && t0.e == t1.e, 10, u, t0.kind * 16 + t1.kind,
                           t0.n * 4096 + t1.n))
              break;
          }
#endif
          if (!DBG_CHECK(p, (tmem & 0xFFFFu) + acc * ACC_COLS + ACC_COLS <= (uint32_t)TMEM_COLS && (tmem >> 16) == 0,
                         11, tmem, acc, u))
            break;
          {
            DBG_SET(p, DBG_MMA_WAIT, 1);
            TRACE_T0();
            if (!wait_bar(&tempty[acc], (accs.uses(acc) & 1u) ^ 1u)) break;
            // MXFP8: the block scales go to the other buffer's first columns, which its latest user must have read
            const uint32_t o = acc ^ 1u;
            if (mx && accs.uses(o) > 0 && !wait_bar(&thead[o], (accs.uses(o) & 1u) ^ 1u)) break;
            TRACE_ADD(p, TR_MMA_TEMPTY);
            DBG_SET(p, DBG_MMA_WAIT, 0);
          }
          tc_fence_after();
          const uint32_t d = tmem + acc * ACC_COLS;
          const uint32_t sfc = tmem + (acc ^ 1u) * ACC_COLS;  // MXFP8 scale columns: A, B rows 0-127, B rows 128-255
          for (int kb = 0; kb < nk; ++kb) {
            {
              DBG_SET(p, DBG_MMA_WAIT, 2);
              TRACE_T0();
              if (!wait_bar(&full[stage], phase)) { ok = false; break; }
              TRACE_ADD(p, TR_MMA_FULL);
#ifdef MOE_TRACE
              _trv[TR_TMA_LAT_NS] += globaltimer_ns() - s_issue_ns[stage];
              _trv[TR_TMA_STAGES] += 1;
#endif
              DBG_SET(p, DBG_MMA_WAIT, 0);
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + stage * G::stride);
            const uint32_t b_addr = a_addr + A_STAGE_BYTES;
            if constexpr (kPair) {
              bool mx_step = false;
              if constexpr (kMxPair) mx_step = mx;
              if (mx_step) {
                if constexpr (kMxPair) {
                  // both CTAs' scale blocks -> their TMEM, then four 32-wide K blocks
                  const uint32_t sf = smem_u32(sf_slots) + stage * SF_STAGE_BYTES;
                  tmem_cp_32x128b_warpx4_pair(sfc, sdesc_sf_block(sf));
                  tmem_cp_32x128b_warpx4_pair(sfc + 4, sdesc_sf_block(sf + SF_BLOCK_BYTES));
                  tmem_cp_32x128b_warpx4_pair(sfc + 8, sdesc_sf_block(sf + 2 * SF_BLOCK_BYTES));
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    mma_mxf8_pair(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32),
                                  idesc_mx | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), sfc, sfc + 4,
                                  (kb | kk) != 0 ? 1u : 0u);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                  mma_bf16_pair(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32), idesc_u,
                                (kb | kk) != 0 ? 1u : 0u);
              }
              mma_commit_pair(&empty[stage], 0x3);
            } else {
              if (mx) {
                // scales -> TMEM (in order with the MMAs below), then four 32-wide K blocks
                const uint32_t sf = a_addr + STAGE_BYTES;
                tmem_cp_32x128b_warpx4(sfc, sdesc_sf_block(sf));
                tmem_cp_32x128b_warpx4(sfc + 4, sdesc_sf_block(sf + SF_BLOCK_BYTES));
                tmem_cp_32x128b_warpx4(sfc + 8, sdesc_sf_block(sf + 2 * SF_BLOCK_BYTES));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_mxf8_ss(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32),
                              idesc_mx | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), sfc, sfc + 4,
                              (kb | kk) != 0 ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                  mma_bf16_ss(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                              (kb | kk) != 0 ? 1u : 0u);
              }
              mma_commit(&empty[stage]);
            }
#ifdef MOE_DEBUG_LOG
            DBG_SET(p, DBG_MMA_STAGES, ++mma_stages);
#endif
            if (++stage == NST) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          if constexpr (kPair) mma_commit_pair(&tfull[acc], 0x3);
          else mma_commit(&tfull[acc]);
          accs.used(acc);
        }
        if constexpr (kPair) mma_commit_pair(drain, 0x1);
        else mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);  // every MMA issued has completed before TMEM is freed
        TRACE_FLUSH(p);
      }
      __syncwarp();
    } else if (warp >= 6) {
      // ---------------- ring fill spread over the GEMM CTAs
      if (p.spread && cta < p.n_gemm) gather_role_spread(p, cta, p.n_gemm, s_ok + 1);
    } else if (warp >= 2 && warp < 6) {
      // ---------------- epilogue
      const int q = warp & 3;
      const int row = q * 32 + lane;
      AccSeq accs;
      const uint32_t tempty_even = kPair ? mapa_shared(tempty, 0) : 0u;
      const uint32_t thead_even = kPair ? mapa_shared(thead, 0) : 0u;
      TRACE_LOCALS();
      const uint32_t qempty_even = kPair ? mapa_shared(qempty, 0) : 0u;
      volatile int* s_unit = s_ok + 2;
      for (int i = 0;; ++i) {
        // one thread waits and decides for all four warps, so that they agree
        // on stopping and never strand each other at the named barrier
        if (threadIdx.x == 64) {
          const int slot = i % QN;
          if (wait_bar(&qfull[slot], (uint32_t)(i / QN) & 1u)) {
            *s_unit = qslot[slot];  // (the store has the value before the arrive)
            if (kPair && !leader) mbar_arrive_remote(qempty_even + 8u * slot);
            else mbar_arrive(&qempty[slot]);
          } else {
            *s_unit = -2;
          }
        }
        named_bar_sync(1, 128);
        const int u = *s_unit;
        if (u < 0) break;
        const int ti = walk.task(u);
        const Task t = p.tasks[ti];
        const uint32_t acc = accs.next();
        if (threadIdx.x == 64) {
          DBG_SET(p, DBG_EPI_UNIT, u);
          DBG_SET(p, DBG_EPI_TASK, ti);
          DBG_SET(p, DBG_EPI_WAIT, 1);
          TRACE_T0();
          const int ok = wait_bar(&tfull[acc], accs.uses(acc) & 1u) ? 1 : 0;
          DBG_SET(p, DBG_EPI_WAIT, 0);
          *s_ok = ok;
          TRACE_ADD(p, TR_EPI_TFULL);
        }
        named_bar_sync(1, 128);
        if (*s_ok == 0) break;
        TRACE_T0();
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS;
        const int r0 = q * 32;                        // the warp's first tile row
        int nrows = min(32, max(0, t.rows - r0));  // its valid rows
        bool store_ok = true;                      // (debug builds: false when a bounds check failed)
#ifdef MOE_DEBUG_LOG
        {
          const bool col_ok = (tmem & 0xFFFFu) + acc * ACC_COLS + ACC_COLS <= (uint32_t)TMEM_COLS;
          bool rows_ok = true;
          if (t.kind == TASK_R1) rows_ok = t.out_row + r0 + nrows <= p.slots * p.b;
          else if (t.kind == TASK_S1 || t.kind == TASK_S2) rows_ok = t.out_row + r0 + nrows <= p.T;
          else {
            const int jj = row < t.rows ? p.sched[(size_t)(t.p0 + row) * 3 + 2] : 0;
            rows_ok = t.p0 + t.rows <= p.R && jj >= 0 && jj < p.R &&
                      y_offset(p, jj / p.k, jj % p.k, t.n) + BN_DOWN <= (size_t)p.n_chunks * BM * p.kY * p.D;
          }
          if (!DBG_CHECK(p, col_ok, 20, tmem, acc, ti) || !DBG_CHECK(p, rows_ok, 21 + t.kind, t.out_row, r0, ti))
            nrows = 0, store_ok = false;
        }
#endif
        const AccRelease rel{&tempty[acc], tempty_even + acc * 8u, &thead[acc], thead_even + acc * 8u, kPair};
        if constexpr (G::kDirectEpi) {
          // a routed tile split over the pair (one M = 128 MMA): each CTA's 64 rows sit in
          // TMEM lanes 0-63 and again in lanes 64-127; lanes 0-63 hold output columns 0-127
          // (split up/gate tiles: h columns 0-63, up then gate), lanes 64-127 the rest
          const int hq = q & 1, hrow = 32 * hq + lane;
          if (t.kind == TASK_R1 && t.half) {
            epilogue_swiglu_direct(taddr, p.ring_h + (size_t)(t.out_row + hrow) * p.I + t.n * BN_UP + (q >> 1) * 64,
                                   store_ok && hrow < t.rows, rel, 64, 64);
          } else if (t.kind == TASK_R1) {
            epilogue_swiglu_direct(taddr, p.ring_h + (size_t)(t.out_row + row) * p.I + t.n * BN_UP,
                                   store_ok && row < t.rows, rel, BN_UP, BN_UP);
          } else if (t.kind == TASK_S1) {
            epilogue_swiglu_direct(taddr, p.h_s + (size_t)(t.out_row + row) * p.I_s + t.n * BN_UP,
                                   store_ok && row < t.rows, rel, BN_UP, BN_UP);
          } else if (t.kind == TASK_R2 && t.half) {
            const int j = hrow < t.rows ? p.sched[(size_t)(t.p0 + hrow) * 3 + 2] : 0;
            epilogue_copy_f16_direct(taddr, p.Y + y_offset(p, j / p.k, j % p.k, t.n) + (q >> 1) * (BN_DOWN / 2),
                                     store_ok && hrow < t.rows, rel, p.status + 1, BN_DOWN / 2);
          } else if (t.kind == TASK_R2) {
            const int j = row < t.rows ? p.sched[(size_t)(t.p0 + row) * 3 + 2] : 0;
            epilogue_copy_f16_direct(taddr, p.Y + y_offset(p, j / p.k, j % p.k, t.n), store_ok && row < t.rows, rel,
                                     p.status + 1, BN_DOWN);
          } else {  // the shared expert's output: staging slot k of its tokens
            epilogue_copy_f16_direct(taddr, p.Y + y_offset(p, t.out_row + row, p.k, t.n), store_ok && row < t.rows,
                                     rel, p.status + 1, BN_DOWN);
          }
        } else {
        EpiStage& st = epi[q];
        if (t.kind == TASK_R1 && p.mx) {
          epilogue_swiglu_mx(taddr, reinterpret_cast<uint8_t*>(p.ring_h) + (size_t)(t.out_row + row) * p.I + t.n * BN_UP,
                             p.sfh + ((size_t)t.mt * (p.I / BK_MX) + t.n) * SF_BLOCK_BYTES, row, row < t.rows, rel);
        } else if (t.kind == TASK_R1) {
          epilogue_swiglu(taddr, st, p.ring_h + (size_t)(t.out_row + r0) * p.I + t.n * BN_UP, p.I, nrows, rel);
        } else if (t.kind == TASK_S1) {
          epilogue_swiglu(taddr, st, p.h_s + (size_t)(t.out_row + r0) * p.I_s + t.n * BN_UP, p.I_s, nrows, rel);
        } else if (t.kind == TASK_R2) {
          const int j = row < t.rows ? p.sched[(size_t)(t.p0 + row) * 3 + 2] : 0;
          epilogue_copy_f16_staged(taddr, st, p.Y, (long long)y_offset(p, j / p.k, j % p.k, t.n), nrows, rel,
                                   p.status + 1);
        } else {  // the shared expert's output: staging slot k of its tokens
          epilogue_copy_f16_staged(taddr, st, p.Y, (long long)y_offset(p, t.out_row + row, p.k, t.n), nrows, rel,
                                   p.status + 1);
        }
        }
        // h tiles are read back by TMA (async proxy); Y and out only by plain loads
        if (t.kind == TASK_R1 || t.kind == TASK_S1) fence_proxy_async_global();
        named_bar_sync(1, 128);
        if (threadIdx.x == 64) {
          TRACE_ADD(p, TR_EPI_BUSY);
          TRACE_ADD(p, TR_EPI_R1 + t.kind);
          TRACE_SET(p, TR_TASKS, ti);
          if (t.done0 >= 0) red_release_add_gpu(p.counters + t.done0, 1);
          if (t.done1 >= 0) red_release_add_gpu(p.counters + t.done1, 1);
          DBG_SET(p, DBG_EPI_DONE, u);
        }
        accs.used(acc);
      }
      if (threadIdx.x == 64) TRACE_FLUSH(p);
    }
    if constexpr (kPair) settle_after_abort(p.status);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) DBG_SET(p, DBG_PHASE, 3);
    // pairs: neither CTA frees TMEM or leaves while the other may still issue
    // into its TMEM, arrive on its barriers or load into its shared memory
    if constexpr (kPair) cluster_sync_all();
    if (threadIdx.x == 0) DBG_SET(p, DBG_PHASE, 4);
    if (warp == 1) {
      tc_fence_after();
      if constexpr (kPair) tmem_dealloc_pair(tmem, TMEM_COLS);
      else tmem_dealloc(tmem, TMEM_COLS);
    }
  }

  // ---------------- combine: every CTA, once every staging row is stored.
  // Cluster launch control: a GEMM CTA whose cancellation request was declined
  // while units were still unclaimed yields its SM at once (CTAs of this grid
  // launched later take the rest, and the combine is claimed in chunks).
  if (threadIdx.x == 0) {
    TRACE_LOCALS();
    TRACE_T0();
    const bool yield = p.clc && !is_gather && ld_relaxed_gpu(p.counters + ctr_claim(p)) < p.meta[META_N_TASKS];
    *s_flag = !yield && wait_counter_ge(p.counters + ctr_ydone(), p.meta[META_TOTAL_Y], p.status, p.timeout_ns)
                  ? 1 : 0;
    if (*s_flag) atomicMin(p.stamps + STAMP_COMBINE_START, (unsigned long long)globaltimer_ns());
    TRACE_ADD(p, TR_FINAL_WAIT);
    TRACE_FLUSH(p);
  }
  __syncthreads();
  if (*s_flag) {
#ifdef MOE_TRACE
    const long long c0 = clock64();
#endif
    combine_role(p, smem, NST * G::stride,
                 reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(epi) + CMB_BAR_OFFSET), s_ok);
    if (threadIdx.x == 0) atomicMax(p.stamps + STAMP_COMBINE_END, (unsigned long long)globaltimer_ns());
#ifdef MOE_TRACE
    if (threadIdx.x == 0 && p.trace && blockIdx.x < 1024) p.trace[(size_t)blockIdx.x * TRACE_SLOTS + TR_COMBINE] = clock64() - c0;
#endif
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    TRACE_SET(p, TR_END_NS, globaltimer_ns());
    TRACE_SET(p, TR_END_CLK, clock64());
  }
  if (threadIdx.x == 0) DBG_SET(p, DBG_PHASE, 5);
}

__global__ void __launch_bounds__(MEGA_THREADS, 1)
    moe_megakernel(const __grid_constant__ TensorMaps maps, const FwdParams p) {
  mega_body<false>(maps, p);
}

// CTA pairs: launched with a cluster of 2 (ranks 0/1 of a cluster form a pair)
__global__ void __launch_bounds__(MEGA_THREADS, 1)
    moe_megakernel_pair(const __grid_constant__ TensorMaps maps, const FwdParams p) {
  mega_body<true>(maps, p);
}

// CTA pairs with MXFP8 routed tiles
__global__ void __launch_bounds__(MEGA_THREADS, 1)
    moe_megakernel_pair_mx(const __grid_constant__ TensorMaps maps, const FwdParams p) {
  mega_body<true, true>(maps, p);
}

cudaError_t launch_megakernel(const TensorMaps& maps, const FwdParams& p, int grid, cudaStream_t stream) {
  const bool pair = p.pair != 0, pair_mx = pair && p.mx;
  // cluster launch control: one CTA per task beyond the gather CTAs; the CTAs
  // that run cancel the launches of the others and take their tokens
  if (p.clc && !pair) grid = p.G + p.n_tasks_max;
  const void* fn = pair_mx ? reinterpret_cast<const void*>(moe_megakernel_pair_mx)
                   : pair  ? reinterpret_cast<const void*>(moe_megakernel_pair)
                           : reinterpret_cast<const void*>(moe_megakernel);
  const int smem = pair_mx ? MegaGeom<true, true>::smem_bytes
                   : pair  ? MegaGeom<true>::smem_bytes
                           : MegaGeom<false>::smem_bytes;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(MEGA_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident (they wait on each other)
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  // cluster launch control: not cooperative (the grid exceeds the SMs); the
  // profiling launch: not cooperative either (the grid still fits the GPU)
  const bool coop = !p.clc && !p.plain_launch;
  cfg.attrs = coop ? attr : attr + 1;
  cfg.numAttrs = (coop ? 1 : 0) + (pair ? 1 : 0);
  if (pair_mx) return cudaLaunchKernelEx(&cfg, moe_megakernel_pair_mx, maps, p);
  if (pair) return cudaLaunchKernelEx(&cfg, moe_megakernel_pair, maps, p);
  return cudaLaunchKernelEx(&cfg, moe_megakernel, maps, p);
}

int megakernel_smem_bytes() { return MegaGeom<false>::smem_bytes; }

// CTAs of the pair kernel that can be resident at once (clusters of 2, one CTA per SM)
int megakernel_pair_max_ctas(bool mx) {
  const int smem = mx ? MegaGeom<true, true>::smem_bytes : MegaGeom<true>::smem_bytes;
  const void* fn = mx ? reinterpret_cast<const void*>(moe_megakernel_pair_mx)
                      : reinterpret_cast<const void*>(moe_megakernel_pair);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms & ~1));
  cfg.blockDim = dim3(MEGA_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) return -1;
  return 2 * clusters;
}

}  // namespace moe
