// Device-side dispatch schedule: per-expert route counts, a deterministic
// prefix sum and the {src_index, expert, dst_index} table, with no host sync.
//
// "Mixture-of-Kittens: MoE Megakernel for NVL72s", Sec. 3.1, Algorithm 1
// (pull-based dispatch schedule construction) with one rank: M_l counts the
// routes to expert l, S_l = sum_{l'<l} M_l' starts expert l's region, and
// route j (= t*k + slot) lands at S_l + o, o being the number of earlier
// routes to the same expert.  Table row P holds {src_index = t, expert = l,
// dst_index = j}: the gather reads x[t] into ring position P, and the combine
// reuses the table the other way round, writing expert output row P to the
// token-order staging row j (Sec. 3.1, "Finally, the schedule can be built
// once and reused").
//
// One CTA per 128-token chunk (the router's tiles): each CTA sums the router's
// per-chunk histograms (its own prefix and the totals), scans them, and ranks
// its routes with per-warp lane masks, so every count and position is
// independent of thread timing.  CTA 0 also lays out the persistent kernel's
// task list (minibatches, expert segments, M-tiles, column tiles).
#include "common.cuh"

namespace moe {

__device__ void build_tasks(const FwdParams& p, const int* sS);

__global__ void __launch_bounds__(SCHED_THREADS, 1) schedule_kernel(const FwdParams p) {
  __shared__ int sM[E_MAX];
  __shared__ int sPre[E_MAX];
  __shared__ int sS[E_MAX + 1];
  __shared__ uint32_t sMask[4][E_MAX];
  __shared__ int sWarp[SCHED_THREADS / 32];

  const int c = blockIdx.x, E = p.E, k = p.k, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  for (int e = tid; e < E; e += blockDim.x) {
    int tot = 0, pre = 0;
    for (int cc = 0; cc < p.n_chunks; ++cc) {
      const int v = p.chunk_counts[(size_t)cc * E + e];
      tot += v;
      if (cc < c) pre += v;
    }
    sM[e] = tot;
    sPre[e] = pre;
  }
  for (int i = tid; i < 4 * E_MAX; i += blockDim.x) (&sMask[0][0])[i] = 0;
  __syncthreads();

  // exclusive scan of sM over experts (E <= blockDim)
  {
    const int v = tid < E ? sM[tid] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    if (lane == 31) sWarp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x / 32) ? sWarp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      if (lane < (int)(blockDim.x / 32)) sWarp[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const int before = warp > 0 ? sWarp[warp - 1] : 0;
    if (tid < E) sS[tid] = before + inc - v;
    if (tid == E - 1) sS[E] = before + inc;
  }
  __syncthreads();

  // ranks inside the chunk: lane masks per (warp, expert)
  const int t = c * BM + tid;
  const bool has_tok = tid < BM && t < p.T;
  if (has_tok) {
    for (int s = 0; s < k; ++s) {
      const int e = p.topk_idx[(size_t)t * k + s];
      if (e < 0 || e >= E) {
        raise_status(p.status, STATUS_SCHEDULE_INVALID);
        continue;
      }
      atomicOr(&sMask[warp][e], 1u << lane);
    }
  }
  __syncthreads();
  if (has_tok) {
    for (int s = 0; s < k; ++s) {
      const int e = p.topk_idx[(size_t)t * k + s];
      if (e < 0 || e >= E) continue;
      int rank = __popc(sMask[warp][e] & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) rank += __popc(sMask[w][e]);
      const int P = sS[e] + sPre[e] + rank;
      const int j = t * k + s;
      if (P < 0 || P >= p.R) {  // only reachable with inconsistent counts
        raise_status(p.status, STATUS_SCHEDULE_INVALID);
        continue;
      }
      p.sched[(size_t)P * 3 + 0] = t;
      p.sched[(size_t)P * 3 + 1] = e;
      p.sched[(size_t)P * 3 + 2] = j;
      p.route_row[j] = P;
    }
  }

  if (c == 0) {
    for (int e = tid; e < E; e += blockDim.x) p.M[e] = sM[e];
    for (int e = tid; e <= E; e += blockDim.x) p.S[e] = sS[e];
    if (tid == 0 && sS[E] != p.R) raise_status(p.status, STATUS_SCHEDULE_INVALID);
    build_tasks(p, sS);
  }
}

// ------------------------------------------------------------------ task list
// Work items, in execution order:
//   S1 (shared expert up/gate, all tokens) ;
//   for step s = 0 .. n_mb - 1 + lag:  R1(s) if s < n_mb ;  R2(s - lag) if s >= lag ;
//   S2 (shared expert down projection + combine, all tokens)
// R1(m) / R2(m): for each expert segment of minibatch m: for each column tile
// n: for each M-tile of the segment (M-tiles of one weight slice run side by
// side, so the slice is read from HBM once).
// A GEMM CTA takes tasks g, g + n_gemm, g + 2 n_gemm, ...; every dependency of
// a task points to an earlier task (or to the gather, whose own dependencies
// are earlier tasks), so the smallest unfinished task can always proceed.
//
// Workspace scratch (p.segs): [segments x 4] {e, mt_begin, mt_count, m},
// then [items x 4] {kind, seg (-1 = shared), task_begin, count},
// then [n_mb + 1] first segment of each minibatch.
__device__ void build_tasks(const FwdParams& p, const int* sS) {
  __shared__ int s_nitems;
  const int max_segs = p.n_mb + p.E;
  int* segs = p.segs;
  int* items = p.segs + 4 * max_segs;
  int* mb_seg = items + 4 * (2 * max_segs + 2);
  const int tid = threadIdx.x;

  if (tid == 0) {
    int nmt = 0, nseg = 0, e = 0;
    for (int m = 0; m < p.n_mb; ++m) {
      const int lo = m * p.b, hi = min(p.R, lo + p.b);
      while (e < p.E && sS[e + 1] <= lo) ++e;
      mb_seg[m] = nseg;
      const int mt0 = nmt;
      for (int ee = e; ee < p.E && sS[ee] < hi; ++ee) {
        const int s0 = max(sS[ee], lo), s1 = min(sS[ee + 1], hi);
        if (s1 <= s0) continue;
        const int beg = nmt;
        if (nseg >= max_segs || nmt + (s1 - s0 + BM - 1) / BM > p.n_mtiles_max) {
          raise_status(p.status, STATUS_SCHEDULE_INVALID);
          break;
        }
        for (int r0 = s0; r0 < s1; r0 += BM) {
          int* mt = p.mtiles + 4 * nmt;
          mt[0] = ee;
          mt[1] = r0;
          mt[2] = min(BM, s1 - r0);
          mt[3] = m;
          ++nmt;
        }
        int* sg = segs + 4 * nseg;
        sg[0] = ee;
        sg[1] = beg;
        sg[2] = nmt - beg;
        sg[3] = m;
        ++nseg;
      }
      p.meta[META_MB + 2 * m] = (nmt - mt0) * p.N1;
      p.meta[META_MB + 2 * m + 1] = (nmt - mt0) * p.N2;
    }
    mb_seg[p.n_mb] = nseg;

    int nit = 0, ntask = 0, total_y = 0;
    auto add = [&](int kind, int seg, int count) {
      int* it = items + 4 * nit;
      it[0] = kind;
      it[1] = seg;
      it[2] = ntask;
      it[3] = count;
      ++nit;
      ntask += count;
      if (kind == TASK_R2) total_y += count;
    };
    const bool shared = p.N1s > 0;
    if (shared) add(TASK_S1, -1, p.N1s * p.n_smtiles);
    for (int s = 0; s < p.n_mb + p.lag; ++s) {
      if (s < p.n_mb)
        for (int g = mb_seg[s]; g < mb_seg[s + 1]; ++g) add(TASK_R1, g, segs[4 * g + 2] * p.N1);
      const int m = s - p.lag;
      if (m >= 0)
        for (int g = mb_seg[m]; g < mb_seg[m + 1]; ++g) add(TASK_R2, g, segs[4 * g + 2] * p.N2);
    }
    // the shared expert's down projection carries the combine in its epilogue,
    // so it comes last: its epilogue needs every routed output row
    if (shared) add(TASK_S2, -1, p.N2s * p.n_smtiles);
    if (ntask > p.n_tasks_max) {  // cannot happen for consistent counts; run nothing
      raise_status(p.status, STATUS_SCHEDULE_INVALID);
      nit = 0;
      ntask = 0;
      total_y = 0;
    }
    p.meta[META_N_TASKS] = ntask;
    p.meta[META_N_MTILES] = nmt;
    p.meta[META_TOTAL_Y] = total_y;
    s_nitems = nit;
  }
  __syncthreads();

  const int nit = s_nitems;
  const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  for (int i = warp; i < nit; i += nwarps) {
    const int kind = items[4 * i], seg = items[4 * i + 1], base = items[4 * i + 2], count = items[4 * i + 3];
    for (int q = lane; q < count; q += 32) {
      Task tk;
      tk.kind = kind;
      tk.dep0 = tk.dep1 = tk.done0 = tk.done1 = -1;
      tk.need0 = tk.need1 = 0;
      tk.pad[0] = tk.pad[1] = tk.pad[2] = 0;
      if (seg < 0) {  // shared expert: tiles of 128 tokens
        const int mt = q % p.n_smtiles;
        tk.n = q / p.n_smtiles;
        tk.e = 0;
        tk.a_row = mt * BM;
        tk.rows = min(BM, p.T - mt * BM);
        tk.p0 = mt * BM;
        tk.out_row = mt * BM;
        if (kind == TASK_S1) {
          tk.done0 = ctr_shready(p, mt);
        } else {
          tk.dep0 = ctr_shready(p, mt);
          tk.need0 = p.N1s;
        }
      } else {
        const int* sg = segs + 4 * seg;
        const int cnt = sg[2];
        const int mt = sg[1] + q % cnt;
        tk.n = q / cnt;
        const int* mtr = p.mtiles + 4 * mt;
        const int m = mtr[3];
        tk.e = mtr[0];
        tk.p0 = mtr[1];
        tk.rows = mtr[2];
        tk.a_row = (m % p.slots) * p.b + (mtr[1] - m * p.b);
        tk.out_row = tk.a_row;
        if (kind == TASK_R1) {
          tk.dep0 = ctr_filled(p, m);
          tk.need0 = p.G;
          if (m >= p.slots) {
            tk.dep1 = ctr_r2(p, m - p.slots);
            tk.need1 = p.meta[META_MB + 2 * (m - p.slots) + 1];
          }
          tk.done0 = ctr_hready(p, mt);
          tk.done1 = ctr_r1(p, m);
        } else {
          tk.dep0 = ctr_hready(p, mt);
          tk.need0 = p.N1;
          tk.done0 = ctr_r2(p, m);
          tk.done1 = ctr_ydone();
        }
      }
      p.tasks[base + q] = tk;
    }
  }
}

cudaError_t launch_schedule(const FwdParams& p, cudaStream_t stream) {
  schedule_kernel<<<p.n_chunks, SCHED_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
