// Router projection + top-k + router-weight normalisation (128 tokens per
// CTA, selection fused into the TMEM epilogue).  CTAs run in pairs: one
// tcgen05.mma.cta_group::2 per K step multiplies both CTAs' 256 token rows by
// W_r, each CTA staging its own 128 x rows and half of W_r's rows, so every
// SM loads a third fewer bytes than a CTA that stages all of W_r; each CTA's
// TMEM receives all logits of its own tokens.
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
// row, so it also quantises x for the expert GEMMs.  Once the MMA has consumed
// a stage (its commit reaches both CTAs of the pair), the four epilogue warps
// (idle until the logits are ready) read the stage's x tile from shared
// memory, one row per thread, and write its E4M3 codes and E8M0 scales (OCP
// MX, 32-element blocks along D) to the workspace; the stage is refilled only
// after the four warps have released it.
// The dispatch then moves the codes into the ring.
#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Insert (l, e) into a list of L (value, id) pairs kept in descending value
// order, dropping the last; an equal value never passes an entry already
// listed, so with ids inserted in increasing order ties keep the lower id.
// Every comparison reads the old list, so the L selects are independent of
// each other (no serial swap chain).
template <int L>
__device__ __forceinline__ void topk_insert(float* bv, int* bi, float l, int e) {
  bool gt[L];
#pragma unroll
  for (int i = 0; i < L; ++i) gt[i] = l > bv[i];
#pragma unroll
  for (int i = L - 1; i > 0; --i) {
    bv[i] = gt[i - 1] ? bv[i - 1] : (gt[i] ? l : bv[i]);
    bi[i] = gt[i - 1] ? bi[i - 1] : (gt[i] ? e : bi[i]);
  }
  bv[0] = gt[0] ? l : bv[0];
  bi[0] = gt[0] ? e : bi[0];
}

// One warp's part of the top-k for its 32 token rows: rank the biased logits
// of columns [c0, c1) (L >= k entries).  The second-half warp leaves its list
// in shared memory; the first-half warp merges it (its ids are all higher),
// keeps the first k, lists them by ascending expert id and writes g, the
// logits, the ids and the route histogram.
template <int L>
__device__ __forceinline__ void topk_epilogue(const FwdParams& p, uint32_t tbase, int c0, int c1, bool first,
                                              bool ready, int q, int lane, int t, const float* s_beta, int* s_hist,
                                              float (*s_pv)[TOPK_MAX][32], int (*s_pi)[TOPK_MAX][32]) {
  const int E = p.E, k = p.k;
  float bv[L];
  int bi[L];
#pragma unroll
  for (int i = 0; i < L; ++i) {
    bv[i] = -INFINITY;
    bi[i] = 0x7fffffff;
  }
  if (ready) {
    for (int c = c0; c < c1; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tbase + (uint32_t)c, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = c + j;
        const float l = e < E ? __uint_as_float(r[j]) + s_beta[e] : -INFINITY;
        if (__any_sync(0xffffffffu, l > bv[L - 1])) topk_insert<L>(bv, bi, l, e);
      }
    }
  }
  if (!first) {
#pragma unroll
    for (int i = 0; i < L; ++i) {
      s_pv[q][i][lane] = bv[i];
      s_pi[q][i][lane] = bi[i];
    }
    named_bar_sync(1 + q, 64);
    return;
  }
  named_bar_sync(1 + q, 64);
  if (!ready) return;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    const float l = s_pv[q][i][lane];
    if (__any_sync(0xffffffffu, l > bv[L - 1])) topk_insert<L>(bv, bi, l, s_pi[q][i][lane]);
  }
  // keep the first k, list them by ascending expert id
#pragma unroll
  for (int i = 0; i < L; ++i)
    if (i >= k) bi[i] = 0x7fffffff;
#pragma unroll
  for (int pass = 0; pass < L - 1; ++pass) {
#pragma unroll
    for (int i = 0; i < L - 1; ++i) {
      if (bi[i] > bi[i + 1]) {
        const float tv = bv[i]; bv[i] = bv[i + 1]; bv[i + 1] = tv;
        const int ti = bi[i]; bi[i] = bi[i + 1]; bi[i + 1] = ti;
      }
    }
  }
  float sc[L];
  float sum = 0.0f;
  if (p.score_fn == 1) {  // softmax: g = exp(l_i - m) / sum_sel exp(l_j - m)
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < L; ++i)
      if (i < k) m = fmaxf(m, bv[i]);
#pragma unroll
    for (int i = 0; i < L; ++i) {
      sc[i] = (i < k) ? expf(bv[i] - m) : 0.0f;
      sum += sc[i];
    }
  } else {  // sigmoid
#pragma unroll
    for (int i = 0; i < L; ++i) {
      sc[i] = (i < k) ? 1.0f / (1.0f + expf(-bv[i])) : 0.0f;
      sum += sc[i];
    }
  }
  if (t < p.T) {
    const float inv = 1.0f / sum;
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (i < k) {
        p.topk_idx[(size_t)t * k + i] = bi[i];
        p.topk_w[(size_t)t * k + i] = sc[i] * inv;
        if (p.topk_logit) p.topk_logit[(size_t)t * k + i] = bv[i];
        atomicAdd(&s_hist[bi[i]], 1);
      }
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(ROUTER_THREADS, 1)
    router_topk_kernel(const __grid_constant__ RouterMaps maps, const FwdParams p, int stages, int tmem_cols) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  __shared__ int s_hist[E_MAX];
  __shared__ float s_beta[E_MAX];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_bar[3 * 8 + 2];
  __shared__ float s_pv[4][TOPK_MAX][32];  // second-half lists, per lane quadrant, entry, lane
  __shared__ int s_pi[4][TOPK_MAX][32];

  const int ncols = p.n_router_cols;
  const int split = ncols > 256 ? 2 : 1;  // MMAs per K step, N = nb each
  const int nb = ncols / split;
  const int hb = nb / 2;                  // W_r rows of one MMA staged by this CTA
  const int stage_bytes = A_STAGE_BYTES + split * hb * 128;
  const uint32_t rank = cluster_ctarank() & 1u;
  const bool leader = rank == 0;
  uint64_t* full = s_bar;
  uint64_t* empty = s_bar + 8;
  const bool quant = p.mx && p.xq != nullptr;  // MXFP8: the epilogue warps quantise x on the way
  uint64_t* qfree = s_bar + 16;  // MXFP8: the quantising warps are done with the stage's x tile
  uint64_t* tfull = s_bar + 24;
  uint64_t* drain = s_bar + 25;

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
      mbar_init(&empty[s], 1);  // the MMA's commit (it reaches both CTAs)
      mbar_init(&qfree[s], 4);  // one arrival per quantising warp
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
    prefetch_tensormap(&maps.x);
    prefetch_tensormap(&maps.wr);
  }
  if (warp == 1) {
    tmem_alloc_pair_dyn(&s_tmem, (uint32_t)tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the other CTA's barriers exist before anything targets them
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int t0 = blockIdx.x * BM;
  const int nk = p.D / BK;

  if (warp == 0) {
    if (elect_one()) {
      // both CTAs' loads are counted on the even CTA's full barrier
      const uint32_t full_even = mapa_shared(full, 0);
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (uint32_t)(kb / stages) & 1u;
        if (!mbar_wait_cluster(&empty[s], ph ^ 1u, p.status, p.timeout_ns)) break;
        if (quant && !mbar_wait(&qfree[s], ph ^ 1u, p.status, p.timeout_ns)) break;
        uint8_t* a = smem + s * stage_bytes;
        uint8_t* b = a + A_STAGE_BYTES;
        if (leader) mbar_arrive_expect_tx(&full[s], 2u * (uint32_t)stage_bytes);
        const uint32_t fb = full_even + 8u * (uint32_t)s;
        tma_load_2d_pair(a, &maps.x, fb, kb * BK, t0);
        for (int h = 0; h < split; ++h)  // rows [h nb + rank hb, + hb) of W_r: this CTA's half of MMA h's N
          tma_load_2d_pair(b + h * hb * 128, &maps.wr, fb, kb * BK, h * nb + (int)rank * hb);
        ++issued;
      }
      // let every copy of both CTAs land before either can exit (the odd CTA
      // waits for the even one at the cluster barrier below)
      if (leader)
        for (int kb = (issued > stages ? issued - stages : 0); kb < issued; ++kb)
          mbar_wait_drain(&full[kb % stages], (uint32_t)(kb / stages) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader && elect_one()) {
      const uint32_t idesc = idesc_bf16_f32(2 * BM, (uint32_t)nb);
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (uint32_t)(kb / stages) & 1u;
        if (!mbar_wait_cluster(&full[s], ph, p.status, p.timeout_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + s * stage_bytes);
        const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t adesc = sdesc_kmajor_sw128(a_addr + kk * 32);
          for (int h = 0; h < split; ++h) {
            const uint64_t bdesc = sdesc_kmajor_sw128(b_addr + h * hb * 128 + kk * 32);
            mma_bf16_pair(tmem + (uint32_t)(h * nb), adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit_pair(&empty[s], 0x3);
      }
      if (ok) mma_commit_pair(tfull, 0x3);
      mma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0, p.timeout_ns);  // every MMA into both CTAs' TMEM has completed
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
        // the stage's loads complete on the even CTA's barrier; the MMA's
        // commit, which reaches both CTAs, says the tile has landed (and been
        // multiplied): the x tile stays until this warp releases it
        if (!mbar_wait_cluster(&empty[s], (uint32_t)(kb / stages) & 1u, p.status, p.timeout_ns)) break;
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
        if (lane == 0) mbar_arrive(&qfree[s]);  // the stage's x tile is read
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
  }

  // ---------------- top-k: every warp.  Warp w reads TMEM lanes 32 (w % 4) ..
  // +31 (its token rows); warps 2-5 rank the first half of the expert columns,
  // warps 0, 1, 6, 7 the second half, and the second list of each row is
  // merged into the first through shared memory.
  {
    const int q = warp & 3;
    const int t = t0 + q * 32 + lane;
    const bool first = warp >= 2 && warp < 6;
    const int csplit = ((ncols / 32 + 1) / 2) * 32;  // column blocks of 32: the first half gets the odd one
    // (warp-uniform: the ranking loop votes across the warp)
    const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull, 0, p.status, p.timeout_ns));
    tc_fence_after();
    if (k <= 8)
      topk_epilogue<8>(p, tmem + ((uint32_t)(q * 32) << 16), first ? 0 : csplit, first ? csplit : ncols, first, ready,
                       q, lane, t, s_beta, s_hist, s_pv, s_pi);
    else
      topk_epilogue<TOPK_MAX>(p, tmem + ((uint32_t)(q * 32) << 16), first ? 0 : csplit, first ? csplit : ncols, first,
                              ready, q, lane, t, s_beta, s_hist, s_pv, s_pi);
  }
  tc_fence_before();
  __syncthreads();
  // (a grid padded to whole pairs has one CTA past the last token tile)
  if (blockIdx.x < (unsigned)p.n_chunks)
    for (int e = threadIdx.x; e < E; e += blockDim.x) p.chunk_counts[(size_t)blockIdx.x * E + e] = s_hist[e];
  // neither CTA frees TMEM or leaves while the other may still load into its
  // shared memory or the MMA may still write its TMEM
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, (uint32_t)tmem_cols);
  }
}

}  // namespace moe

// host-side launcher (called from api.cu)
namespace moe {
int router_smem_bytes(int ncols, int* stages_out) {
  const int stage_bytes = A_STAGE_BYTES + (ncols / 2) * 128;  // x tile + this CTA's half of W_r
  int stages = (200 * 1024) / stage_bytes;
  if (stages > 8) stages = 8;
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
  router_topk_kernel<<<(p.n_chunks + 1) & ~1, ROUTER_THREADS, smem, stream>>>(maps, p, stages, tmem_cols);
  return cudaGetLastError();
}
}  // namespace moe
