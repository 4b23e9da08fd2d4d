// Router projection + top-k + router-weight normalisation (one tcgen05 GEMM
// tile of 128 tokens per CTA, selection fused into the TMEM epilogue).
//
// "Mixture-of-Kittens: MoE Megakernel for NVL72s", Sec. 2.1: a router
// projection selects the top-k routed experts and gives each a router weight;
// Eq. MoE normalises them, g_i = s_i / sum_{j in E} s_j.  Readings: the bias is
// added to the logits; both score functions (sigmoid, softmax over all E) are
// increasing in the logit, so the selection is made on the biased fp32 logits
// (ties: lower expert id first); the k winners are listed in ascending expert
// id; for softmax the normaliser over all E cancels in g.
//
// The kernel also zeroes the persistent kernel's counters and the status word
// and writes each CTA's per-expert route histogram (input of the schedule).
//
// MXFP8 routed experts (Sec. 3.4 "MXFP8 Support": activation quantisation
// fused into the dispatch): this is the one pass that reads every token's x
// row, so it also quantises x for the expert GEMMs.  While the MMA consumes a
// stage, the four epilogue warps (idle until the logits are ready) read the
// same x tile from shared memory, one row per thread, and write its E4M3 codes
// and E8M0 scales (OCP MX, 32-element blocks along D) to the workspace; the
// stage is refilled only after the MMA and the four warps have released it.
// The dispatch then moves the codes into the ring.
#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__global__ void __launch_bounds__(ROUTER_THREADS, 1)
    router_topk_kernel(const __grid_constant__ RouterMaps maps, const FwdParams p, int stages, int tmem_cols) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  __shared__ int s_hist[E_MAX];
  __shared__ float s_beta[E_MAX];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_bar[2 * 8 + 2];

  const int ncols = p.n_router_cols;
  const int split = ncols > 256 ? 2 : 1;
  const int nb = ncols / split;
  const int stage_bytes = A_STAGE_BYTES + ncols * 128;
  uint64_t* full = s_bar;
  uint64_t* empty = s_bar + 8;
  const bool quant = p.mx && p.xq != nullptr;  // MXFP8: the epilogue warps quantise x on the way
  uint64_t* tfull = s_bar + 16;
  uint64_t* drain = s_bar + 17;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, k = p.k;

  // counters / status of this forward start at zero
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.n_counters; i += gridDim.x * blockDim.x)
    p.counters[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.status[0] = 0;
    p.status[1] = 0;
    if (p.stamps) {
      p.stamps[STAMP_START] = p.stamps[STAMP_COMBINE_START] = ~0ull;
      p.stamps[STAMP_LAST_FILL] = p.stamps[STAMP_COMBINE_END] = 0ull;
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_hist[e] = 0;
    s_beta[e] = p.b_router ? p.b_router[e] : 0.0f;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], quant ? 5 : 1);  // the MMA's commit (+ one arrival per quantising warp)
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
    prefetch_tensormap(&maps.x);
    prefetch_tensormap(&maps.wr);
  }
  if (warp == 1) {
    tmem_alloc_dyn(&s_tmem, (uint32_t)tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int t0 = blockIdx.x * BM;
  const int nk = p.D / BK;

  if (warp == 0) {
    if (elect_one()) {
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (uint32_t)(kb / stages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, p.status, p.timeout_ns)) break;
        uint8_t* a = smem + s * stage_bytes;
        uint8_t* b = a + A_STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
        tma_load_2d(a, &maps.x, &full[s], kb * BK, t0);
        tma_load_2d(b, &maps.wr, &full[s], kb * BK, 0);
        if (split == 2) tma_load_2d(b + nb * 128, &maps.wr, &full[s], kb * BK, nb);
        ++issued;
      }
      // let every copy this thread issued land before the CTA can exit
      for (int kb = (issued > stages ? issued - stages : 0); kb < issued; ++kb)
        mbar_wait(&full[kb % stages], (uint32_t)(kb / stages) & 1u, p.status, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (elect_one()) {
      const uint32_t idesc = idesc_bf16_f32(BM, (uint32_t)nb);
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (uint32_t)(kb / stages) & 1u;
        if (!mbar_wait(&full[s], ph, p.status, p.timeout_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + s * stage_bytes);
        const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t adesc = sdesc_kmajor_sw128(a_addr + kk * 32);
          for (int h = 0; h < split; ++h) {
            const uint64_t bdesc = sdesc_kmajor_sw128(b_addr + h * nb * 128 + kk * 32);
            mma_bf16_ss(tmem + (uint32_t)(h * nb), adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
      }
      if (ok) mma_commit(tfull);
      mma_commit(drain);
      mbar_wait(drain, 0, p.status, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 6) {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int t = t0 + row;
    if (quant) {
      // this thread's row of every x stage: 64 bf16 (one 128-byte swizzled
      // row, 16-byte chunk c at c ^ (row % 8)) -> two MX blocks of 32
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % stages;
        if (!mbar_wait(&full[s], (uint32_t)(kb / stages) & 1u, p.status, p.timeout_ns)) break;
        const uint8_t* a = smem + s * stage_bytes + row * 128;
        float v[64];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(a + ((c ^ (row & 7)) << 4));
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            v[8 * c + 2 * j] = f.x;
            v[8 * c + 2 * j + 1] = f.y;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage's x tile is read
        uint32_t c0[8], c1[8];
        const uint32_t s0 = mx_quantize32(v, c0), s1 = mx_quantize32(v + 32, c1);
        if (t < p.T) {
          uint4* d = reinterpret_cast<uint4*>(p.xq + (size_t)t * p.D + kb * BK);
          d[0] = make_uint4(c0[0], c0[1], c0[2], c0[3]);
          d[1] = make_uint4(c0[4], c0[5], c0[6], c0[7]);
          d[2] = make_uint4(c1[0], c1[1], c1[2], c1[3]);
          d[3] = make_uint4(c1[4], c1[5], c1[6], c1[7]);
          *reinterpret_cast<uint16_t*>(p.xs + (size_t)t * (p.D / 32) + 2 * kb) = (uint16_t)(s0 | (s1 << 8));
        }
      }
    }
    if (mbar_wait(tfull, 0, p.status, p.timeout_ns)) {
      tc_fence_after();
      float bv[TOPK_MAX];
      int bi[TOPK_MAX];
#pragma unroll
      for (int i = 0; i < TOPK_MAX; ++i) {
        bv[i] = -INFINITY;
        bi[i] = 0x7fffffff;
      }
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < ncols; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + (uint32_t)c, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int e = c + j;
          if (e < E) {
            const float l = __uint_as_float(r[j]) + s_beta[e];
            if (l > bv[TOPK_MAX - 1]) {
              // insert, keeping descending value order; an equal value never
              // passes an earlier (lower-id) entry
              bv[TOPK_MAX - 1] = l;
              bi[TOPK_MAX - 1] = e;
#pragma unroll
              for (int i = TOPK_MAX - 1; i > 0; --i) {
                if (bv[i] > bv[i - 1]) {
                  const float tv = bv[i]; bv[i] = bv[i - 1]; bv[i - 1] = tv;
                  const int ti = bi[i]; bi[i] = bi[i - 1]; bi[i - 1] = ti;
                }
              }
            }
          }
        }
      }
      // keep the first k, list them by ascending expert id
#pragma unroll
      for (int i = 0; i < TOPK_MAX; ++i)
        if (i >= k) bi[i] = 0x7fffffff;
#pragma unroll
      for (int pass = 0; pass < TOPK_MAX - 1; ++pass) {
#pragma unroll
        for (int i = 0; i < TOPK_MAX - 1; ++i) {
          if (bi[i] > bi[i + 1]) {
            const float tv = bv[i]; bv[i] = bv[i + 1]; bv[i + 1] = tv;
            const int ti = bi[i]; bi[i] = bi[i + 1]; bi[i + 1] = ti;
          }
        }
      }
      float s[TOPK_MAX];
      float sum = 0.0f;
      if (p.score_fn == 1) {  // softmax: g = exp(l_i - m) / sum_sel exp(l_j - m)
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < TOPK_MAX; ++i)
          if (i < k) m = fmaxf(m, bv[i]);
#pragma unroll
        for (int i = 0; i < TOPK_MAX; ++i) {
          s[i] = (i < k) ? expf(bv[i] - m) : 0.0f;
          sum += s[i];
        }
      } else {  // sigmoid
#pragma unroll
        for (int i = 0; i < TOPK_MAX; ++i) {
          s[i] = (i < k) ? 1.0f / (1.0f + expf(-bv[i])) : 0.0f;
          sum += s[i];
        }
      }
      if (t < p.T) {
        const float inv = 1.0f / sum;
#pragma unroll
        for (int i = 0; i < TOPK_MAX; ++i) {
          if (i < k) {
            p.topk_idx[(size_t)t * k + i] = bi[i];
            p.topk_w[(size_t)t * k + i] = s[i] * inv;
            if (p.topk_logit) p.topk_logit[(size_t)t * k + i] = bv[i];
            atomicAdd(&s_hist[bi[i]], 1);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) p.chunk_counts[(size_t)blockIdx.x * E + e] = s_hist[e];
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)tmem_cols);
  }
}

}  // namespace moe

// host-side launcher (called from api.cu)
namespace moe {
int router_smem_bytes(int ncols, int* stages_out) {
  const int stage_bytes = A_STAGE_BYTES + ncols * 128;
  int stages = (200 * 1024) / stage_bytes;
  if (stages > 4) stages = 4;
  if (stages < 2) stages = 2;
  *stages_out = stages;
  return stages * stage_bytes + 1024;
}

cudaError_t launch_router(const RouterMaps& maps, const FwdParams& p, cudaStream_t stream) {
  int stages = 0;
  const int smem = router_smem_bytes(p.n_router_cols, &stages);
  int tmem_cols = 32;
  while (tmem_cols < p.n_router_cols) tmem_cols <<= 1;
  cudaError_t err = cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  router_topk_kernel<<<p.n_chunks, ROUTER_THREADS, smem, stream>>>(maps, p, stages, tmem_cols);
  return cudaGetLastError();
}
}  // namespace moe
