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
//    come last and carry the weighted sum in their epilogue (the shared
//    output never leaves TMEM in fp32 before it is added).
//  * Sec. 3.4 "Determinism": no floating-point atomics; every output element
//    is produced by one tile with a fixed K order, and the weighted sum runs
//    in a fixed slot order from a token-order fp32 staging buffer (fp32 so
//    that the sum rounds once, at the bf16 output).
// The expert FFN is the one of Sec. 2.1 / the blog's E_i(x) with SiLU:
// h = SiLU(x W_gate^T) * (x W_up^T) in fp32 from TMEM, stored bf16; y = h W_down^T.
//
// GEMM CTA roles (256 threads): warp 0 issues TMA loads, warp 1 issues
// tcgen05.mma (128 x 256 x 16, fp32 accumulators in TMEM, two accumulator
// buffers), warps 2-5 drain TMEM (tcgen05.ld), apply the epilogue and store.
// A GEMM1 tile is 128 rows x (128 up + 128 gate) columns; a GEMM2 tile is
// 128 rows x 256 output columns.
#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint8_t* align_1024_mk(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int TMEM_COLS = 2 * ACC_COLS;  // 512: two accumulator buffers
constexpr int EPI_STAGE_BYTES = 4 * 6272;  // 4 epilogue warps x sizeof(EpiStage)
constexpr int MEGA_SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + EPI_STAGE_BYTES;

// ------------------------------------------------------------------ gather (dispatch)
// Ring slot m % slots receives schedule rows [m b, min((m+1) b, R)) of x.
__device__ void gather_role(const FwdParams& p, volatile int* s_flag) {
  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int nv = p.D / 8;  // 16-byte vectors per row
  // a whole row in flight per warp (D <= 8192 in one pass), loads before stores
  constexpr int UNR = 32;
  for (int m = 0; m < p.n_mb; ++m) {
    if (m >= p.slots) {
      if (threadIdx.x == 0) {
        const int need = p.meta[META_MB + 2 * (m - p.slots)];
        TRACE_T0();
        *s_flag = wait_counter_ge(p.counters + ctr_r1(p, m - p.slots), need, p.status, p.timeout_ns) ? 1 : 0;
        TRACE_ADD(p, TR_GATHER_WAIT);
      }
      __syncthreads();
      if (*s_flag == 0) return;
    }
    const int lo = m * p.b, hi = min(p.R, lo + p.b);
    const int per = (hi - lo + p.G - 1) / p.G;
    const int r0 = lo + g * per, r1 = min(hi, r0 + per);
    const size_t slot_base = (size_t)(m % p.slots) * p.b;
    TRACE_T0();
    for (int r = r0 + warp; r < r1; r += nwarps) {
      const int t = p.sched[(size_t)r * 3];
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D);
      uint4* dst = reinterpret_cast<uint4*>(p.ring_x + (slot_base + (size_t)(r - lo)) * p.D);
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
    fence_proxy_async_global();
    __syncthreads();
    if (threadIdx.x == 0) {
      TRACE_ADD(p, TR_GATHER_BUSY);
      red_release_add_gpu(p.counters + ctr_filled(p, m), 1);
    }
  }
}

// ------------------------------------------------------------------ operand selection
struct Operands {
  const CUtensorMap* a;
  const CUtensorMap* b0;
  const CUtensorMap* b1;  // null: one 256-row B box
  int b_row;
  int nk;
};

__device__ __forceinline__ Operands task_operands(const TensorMaps& maps, const FwdParams& p, const Task& t) {
  Operands o;
  switch (t.kind) {
    case TASK_R1:
      o.a = &maps.ring_x; o.b0 = &maps.w_up; o.b1 = &maps.w_gate;
      o.b_row = t.e * p.I + t.n * BN_UP; o.nk = p.D / BK;
      break;
    case TASK_R2:
      o.a = &maps.ring_h; o.b0 = &maps.w_down; o.b1 = nullptr;
      o.b_row = t.e * p.D + t.n * BN_DOWN; o.nk = p.I / BK;
      break;
    case TASK_S1:
      o.a = &maps.x; o.b0 = &maps.ws_up; o.b1 = &maps.ws_gate;
      o.b_row = t.n * BN_UP; o.nk = p.D / BK;
      break;
    default:  // TASK_S2
      o.a = &maps.h_s; o.b0 = &maps.ws_down; o.b1 = nullptr;
      o.b_row = t.n * BN_DOWN; o.nk = p.I_s / BK;
      break;
  }
  return o;
}

__device__ __forceinline__ int task_nk(const FwdParams& p, int kind) {
  return (kind == TASK_R1 || kind == TASK_S1) ? p.D / BK : (kind == TASK_R2 ? p.I / BK : p.I_s / BK);
}

// ------------------------------------------------------------------ epilogues
// 128 threads, thread r owns tile row r (TMEM lane r).
__device__ __forceinline__ void store_row_bf16x32(bf16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    d[i] = w;
  }
}

// Epilogue data movement: each warp owns 32 tile rows (TMEM lanes).  A
// tcgen05.ld gives lane r the 32 columns of row r; the warp stages that 32x32
// block in shared memory (row stride 33 floats: conflict-free both ways) and
// re-reads it so that lane l handles row 4i + l/8, columns 4 (l%8) .. +3:
// every warp store then covers 4 rows x a contiguous 32-column segment.
struct EpiStage {
  float v[32][33];
  float g[32][TOPK_MAX];  // router weights of the warp's 32 tokens (combine)
};
static_assert(sizeof(EpiStage) == 6272, "epilogue staging size");

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

// up/gate tile -> h = SiLU(gate) * up (bf16): TMEM columns [0,128) up, [128,256) gate.
// dst: row 0 of the warp's rows, column 0 of the tile; ld: row stride (elements).
__device__ void epilogue_swiglu(uint32_t taddr, EpiStage& st, bf16* dst, size_t ld, int nrows, uint64_t* tempty) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int c = 0; c < BN_UP; c += 32) {
    uint32_t u[32], g[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, u);
    tmem_ld_32x32b_x32(taddr + (uint32_t)(BN_UP + c), g);
    tmem_ld_wait();
    if (c + 32 == BN_UP) {  // last TMEM read of this tile: hand the accumulator back
      tc_fence_before();
      mbar_arrive(tempty);
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

// routed down-projection tile -> fp32 staging rows Y[j] (j from the schedule table)
__device__ void epilogue_copy_f32(uint32_t taddr, EpiStage& st, float* Y, size_t D, int col0, int j_mine, int nrows,
                                  uint64_t* tempty) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int c = 0; c < BN_DOWN; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
    tmem_ld_wait();
    if (c + 32 == BN_DOWN) {
      tc_fence_before();
      mbar_arrive(tempty);
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    stage_block(st, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3), cc = 4 * (lane & 7);
      const int jr = __shfl_sync(0xffffffffu, j_mine, rr);
      if (rr < nrows) *reinterpret_cast<float4*>(Y + (size_t)jr * D + col0 + c + cc) = staged4(st, rr, cc);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ combine
// Weighted sum back in token order (Eq. MoE), fp32, slot order 0..k-1, one
// rounding to bf16 at the end.  With a shared expert the sum is fused into the
// shared expert's down-projection epilogue and starts from its fp32 output;
// without one, this pass runs once every routed output row is stored.
__device__ __forceinline__ void accumulate_routed(const FwdParams& p, int t, int col, const float* g, float* acc) {
  const float* y = p.Y + (size_t)t * p.k * p.D + col;
#pragma unroll
  for (int s = 0; s < TOPK_MAX; ++s) {
    if (s < p.k) {
      const float4* src = reinterpret_cast<const float4*>(y + (size_t)s * p.D);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = src[i];
        acc[4 * i + 0] = fmaf(g[s], f.x, acc[4 * i + 0]);
        acc[4 * i + 1] = fmaf(g[s], f.y, acc[4 * i + 1]);
        acc[4 * i + 2] = fmaf(g[s], f.z, acc[4 * i + 2]);
        acc[4 * i + 3] = fmaf(g[s], f.w, acc[4 * i + 3]);
      }
    }
  }
}

__device__ __forceinline__ void load_g(const FwdParams& p, int t, bool valid, float* g) {
#pragma unroll
  for (int s = 0; s < TOPK_MAX; ++s) g[s] = (valid && s < p.k) ? p.topk_w[(size_t)t * p.k + s] : 0.0f;
}

// shared-expert down projection + combine: out = bf16(y_s + sum_slot g * Y[t k + slot]),
// y_s in fp32 straight from TMEM; t0 = token of the warp's first row
__device__ void epilogue_shared_combine(uint32_t taddr, EpiStage& st, const FwdParams& p, int t0, int col0,
                                        int nrows, uint64_t* tempty) {
  const int lane = threadIdx.x & 31;
  const int k = p.k;
#pragma unroll
  for (int s = 0; s < TOPK_MAX; ++s) st.g[lane][s] = (lane < nrows && s < k) ? p.topk_w[(size_t)(t0 + lane) * k + s] : 0.0f;
  // the k staging rows of a token are read once: ask L2 for them two chunks
  // ahead (lane = row; one 128-byte line per slot and chunk)
  const float* yrow = p.Y + (size_t)(t0 + lane) * k * p.D + col0;
  auto prefetch_chunk = [&](int c) {
    if (lane < nrows && c < BN_DOWN)
      for (int s = 0; s < k; ++s) prefetch_l2(yrow + (size_t)s * p.D + c);
  };
  prefetch_chunk(0);
  prefetch_chunk(32);
#pragma unroll 1
  for (int c = 0; c < BN_DOWN; c += 32) {
    prefetch_chunk(c + 64);
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
    tmem_ld_wait();
    if (c + 32 == BN_DOWN) {
      tc_fence_before();
      mbar_arrive(tempty);
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    stage_block(st, v);
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3), cc = 4 * (lane & 7);
      if (rr < nrows) {
        const int t = t0 + rr;
        float4 acc = staged4(st, rr, cc);
        const float* y = p.Y + (size_t)t * k * p.D + col0 + c + cc;
#pragma unroll
        for (int s = 0; s < TOPK_MAX; ++s) {
          if (s < k) {
            const float gs = st.g[rr][s];
            const float4 f = __ldcs(reinterpret_cast<const float4*>(y + (size_t)s * p.D));
            acc.x = fmaf(gs, f.x, acc.x);
            acc.y = fmaf(gs, f.y, acc.y);
            acc.z = fmaf(gs, f.z, acc.z);
            acc.w = fmaf(gs, f.w, acc.w);
          }
        }
        *reinterpret_cast<uint2*>(p.out + (size_t)t * p.D + col0 + c + cc) = pack_bf16x4(acc);
      }
    }
    __syncwarp();
  }
}

// no shared expert: every CTA takes tokens blockIdx.x, blockIdx.x + gridDim.x, ...
__device__ void combine_role(const FwdParams& p) {
  const int chunks = p.D / 32;
  for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
    float g[TOPK_MAX];
    load_g(p, t, true, g);
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
      accumulate_routed(p, t, c * 32, g, acc);
      store_row_bf16x32(p.out + (size_t)t * p.D + c * 32, acc);
    }
  }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(MEGA_THREADS, 1)
    moe_megakernel(const __grid_constant__ TensorMaps maps, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024_mk(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = s_flag + 1;
  EpiStage* epi = reinterpret_cast<EpiStage*>(smem + STAGES * STAGE_BYTES + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_gather = (int)blockIdx.x < p.G;
  if (threadIdx.x == 0) TRACE_SET(p, TR_START_NS, globaltimer_ns());
  const bool has_shared = p.N1s > 0;

  if (is_gather) {
    gather_role(p, s_flag);
    __syncthreads();
  } else {
    const int cta = blockIdx.x - p.G;
    const int n_tasks = p.meta[META_N_TASKS];
    if (threadIdx.x == 0) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&tfull[a], 1);
        mbar_init(&tempty[a], 128);
      }
      mbar_init(drain, 1);
      fence_barrier_init();
    }
    if (warp == 1) {
      tmem_alloc<TMEM_COLS>(tmem_slot);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
      // ---------------- TMA producer
      if (elect_one()) {
        prefetch_tensormap(&maps.x);
        prefetch_tensormap(&maps.ring_x);
        prefetch_tensormap(&maps.w_up);
        prefetch_tensormap(&maps.w_gate);
        prefetch_tensormap(&maps.ring_h);
        prefetch_tensormap(&maps.w_down);
        uint32_t stage = 0, phase = 0;
        int issued = 0;
        bool ok = true;
        for (int ti = cta; ti < n_tasks && ok; ti += p.n_gemm) {
          const Task t = p.tasks[ti];
          {
            TRACE_T0();
            if (t.dep0 >= 0 && !wait_counter_ge(p.counters + t.dep0, t.need0, p.status, p.timeout_ns)) break;
            if (t.dep1 >= 0 && !wait_counter_ge(p.counters + t.dep1, t.need1, p.status, p.timeout_ns)) break;
            TRACE_ADD(p, TR_PROD_DEP);
          }
          fence_proxy_async_global();
          const Operands o = task_operands(maps, p, t);
          for (int kb = 0; kb < o.nk; ++kb) {
            {
              TRACE_T0();
              if (!mbar_wait(&empty[stage], phase ^ 1u, p.status, p.timeout_ns)) { ok = false; break; }
              TRACE_ADD(p, TR_PROD_EMPTY);
            }
            uint8_t* sa = smem + stage * STAGE_BYTES;
            uint8_t* sb = sa + A_STAGE_BYTES;
            mbar_arrive_expect_tx(&full[stage], (uint32_t)STAGE_BYTES);
            tma_load_2d(sa, o.a, &full[stage], kb * BK, t.a_row);
            if (o.b1) {
              tma_load_2d(sb, o.b0, &full[stage], kb * BK, o.b_row);
              tma_load_2d(sb + B_STAGE_BYTES / 2, o.b1, &full[stage], kb * BK, o.b_row);
            } else {
              tma_load_2d(sb, o.b0, &full[stage], kb * BK, o.b_row);
            }
            ++issued;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        // the last STAGES loads this thread issued have landed before the CTA may exit
        for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
          mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u, p.status, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------- MMA issuer
      if (elect_one()) {
        const uint32_t idesc = idesc_bf16_f32(BM, 256);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        for (int ti = cta; ti < n_tasks && ok; ti += p.n_gemm) {
          const int nk = task_nk(p, p.tasks[ti].kind);
          {
            TRACE_T0();
            if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.status, p.timeout_ns)) break;
            TRACE_ADD(p, TR_MMA_TEMPTY);
          }
          tc_fence_after();
          const uint32_t d = tmem + acc * ACC_COLS;
          for (int kb = 0; kb < nk; ++kb) {
            {
              TRACE_T0();
              if (!mbar_wait(&full[stage], phase, p.status, p.timeout_ns)) { ok = false; break; }
              TRACE_ADD(p, TR_MMA_FULL);
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              mma_bf16_ss(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
            mma_commit(&empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          mma_commit(&tfull[acc]);
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        mma_commit(drain);
        mbar_wait(drain, 0, p.status, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp >= 2 && warp < 6) {
      // ---------------- epilogue
      const int q = warp & 3;
      const int row = q * 32 + lane;
      uint32_t acc = 0, acc_phase = 0;
      bool routed_done = false;
      for (int ti = cta; ti < n_tasks; ti += p.n_gemm) {
        const Task t = p.tasks[ti];
        // one thread waits and decides for all four warps, so that they agree
        // on stopping and never strand each other at the named barrier
        if (threadIdx.x == 64) {
          TRACE_T0();
          int ok = mbar_wait(&tfull[acc], acc_phase, p.status, p.timeout_ns) ? 1 : 0;
          if (ok && t.kind == TASK_S2 && !routed_done)  // the combine reads every routed output row
            ok = wait_counter_ge(p.counters + ctr_ydone(), p.meta[META_TOTAL_Y], p.status, p.timeout_ns) ? 1 : 0;
          routed_done = routed_done || (ok && t.kind == TASK_S2);
          *s_ok = ok;
          TRACE_ADD(p, TR_EPI_TFULL);
        }
        named_bar_sync(1, 128);
        if (*s_ok == 0) break;
        TRACE_T0();
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS;
        const int r0 = q * 32;                        // the warp's first tile row
        const int nrows = min(32, max(0, t.rows - r0));  // its valid rows
        EpiStage& st = epi[q];
        if (t.kind == TASK_R1) {
          epilogue_swiglu(taddr, st, p.ring_h + (size_t)(t.out_row + r0) * p.I + t.n * BN_UP, p.I, nrows, &tempty[acc]);
        } else if (t.kind == TASK_S1) {
          epilogue_swiglu(taddr, st, p.h_s + (size_t)(t.out_row + r0) * p.I_s + t.n * BN_UP, p.I_s, nrows,
                          &tempty[acc]);
        } else if (t.kind == TASK_R2) {
          const int j = row < t.rows ? p.sched[(size_t)(t.p0 + row) * 3 + 2] : 0;
          epilogue_copy_f32(taddr, st, p.Y, p.D, t.n * BN_DOWN, j, nrows, &tempty[acc]);
        } else {
          epilogue_shared_combine(taddr, st, p, t.out_row + r0, t.n * BN_DOWN, nrows, &tempty[acc]);
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
        }
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, TMEM_COLS);
    }
  }

  // ---------------- combine without a shared expert: every CTA, once all routed rows are stored
  if (!has_shared) {
    if (threadIdx.x == 0) {
      TRACE_T0();
      *s_flag = wait_counter_ge(p.counters + ctr_ydone(), p.meta[META_TOTAL_Y], p.status, p.timeout_ns) ? 1 : 0;
      TRACE_ADD(p, TR_FINAL_WAIT);
    }
    __syncthreads();
    if (*s_flag) combine_role(p);
  }
  __syncthreads();
  if (threadIdx.x == 0) TRACE_SET(p, TR_END_NS, globaltimer_ns());
}

cudaError_t launch_megakernel(const TensorMaps& maps, const FwdParams& p, int grid, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(moe_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MEGA_SMEM_BYTES);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(MEGA_THREADS);
  cfg.dynamicSmemBytes = MEGA_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident (they wait on each other)
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_megakernel, maps, p);
}

int megakernel_smem_bytes() { return MEGA_SMEM_BYTES; }

}  // namespace moe
