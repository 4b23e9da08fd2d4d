// Device-side dispatch schedule: per-expert route counts, a deterministic
// prefix sum and the {src_index, expert, dst_index} table, with no host sync.
//
// "Mixture-of-Kittens: MoE Megakernel for NVL72s", Sec. 3.1, Algorithm 1
// (pull-based dispatch schedule construction) with one rank: M_l counts the
// routes to expert l, S_l = sum_{l'<l} M_l' starts expert l's region, and
// route j (= t*k + slot) lands at S_l + o, o being the number of earlier
// routes to the same expert.  Table row P holds {src_index = t, expert = l,
// dst_index = j}: the gather reads x[t] into ring position P, and the combine
// reads the same table the other way round, writing expert output row P to the
// token-order staging row j (Sec. 3.1: one table, built once, serves the
// dispatch, the combine and the backward pass's counterparts).
//
// One CTA per 128-token chunk (the router's tiles): each CTA sums the router's
// per-chunk histograms (its own prefix and the totals), scans them, and ranks
// its routes with per-warp lane masks, so every count and position is
// independent of thread timing.  CTA 0 also lays out the persistent kernel's
// task list (minibatches, expert segments, M-tiles, column tiles).
#include "common.cuh"

namespace moe {

__device__ void build_tasks(const FwdParams& p, const int* sS, int* dsm);

__global__ void __launch_bounds__(SCHED_THREADS, 1) schedule_kernel(const FwdParams p) {
  __shared__ int sM[E_MAX];
  __shared__ int sPre[E_MAX];
  __shared__ int sS[E_MAX + 1];
  __shared__ uint32_t sMask[4][E_MAX];
  __shared__ int sWarp[SCHED_THREADS / 32];

  extern __shared__ int dyn_smem[];
  const int c = blockIdx.x, E = p.E, k = p.k, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  for (int e = tid; e < E; e += blockDim.x) {
    int tot = 0, pre = 0;
#pragma unroll 8
    for (int cc = 0; cc < p.n_chunks; ++cc) {  // independent loads: unrolled so they overlap
      const int v = p.chunk_counts[(size_t)cc * E + e];
      tot += v;
      pre += cc < c ? v : 0;
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
  }
  build_tasks(p, sS, dyn_smem);  // every CTA: CTA 0 writes the layout, all CTAs share the task fill
}

// ------------------------------------------------------------------ task list
// Order of execution:
//   S1 (shared expert up/gate, all tokens) ;
//   for step s = 0 .. n_mb - 1 + lag:  R1(s) if s < n_mb ;  R2(s - lag) if s >= lag ;
//   S2 (shared expert down projection into staging slot k, all tokens)
// and then, in every CTA once all staging rows are stored, the combine.
// R1(m) / R2(m): for each segment of minibatch m (an expert's rows inside m),
// for each column tile n, for each M-tile of the segment -- the M-tiles that
// share a weight slice run side by side (slice read from HBM once).
// S1 / S2: token-tile major -- the column tiles of one token tile run side by
// side.
// The GEMM CTAs claim tasks (pairs of tasks with CTA pairs) in increasing
// order from a global counter; every dependency of a task points to an earlier
// task (or to the gather, whose own dependencies are earlier tasks), so the
// smallest unfinished task can always proceed.
//
// Segments sorted by first row are in expert-major order and every
// minibatch's segments are contiguous, so the whole layout comes from
// per-expert counts and block-wide scans (no serial walk).
// p.segs holds [segments x 4] {e, mt_begin, mt_count, m}.
// Dynamic shared memory: see sched_dyn_ints.

// exclusive scan of v[0..n) in place (shared memory), returns the total; all threads call it
__device__ int block_exclusive_scan(int* v, int n, int* warp_tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + tid;
    const int x = i < n ? v[i] : 0;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) warp_tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nwarps ? warp_tmp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nwarps) warp_tmp[lane] = w;
    }
    __syncthreads();
    const int before = warp > 0 ? warp_tmp[warp - 1] : 0;
    const int total = warp_tmp[nwarps - 1];
    if (i < n) v[i] = carry + before + inc - x;
    carry += total;
    __syncthreads();
  }
  return carry;
}

// a task record as four 16-byte stores
__device__ __forceinline__ void store_task(Task* dst, const Task& t) {
  const int4* src = reinterpret_cast<const int4*>(&t);
  int4* d = reinterpret_cast<int4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = src[i];
}

__device__ __forceinline__ void piece_rows(const int* sS, int e, int m, int b, int& a, int& z) {
  a = max(sS[e], m * b);
  z = min(sS[e + 1], (m + 1) * b);
}

// A operand row of an empty partner task: the whole 128-row box lies before
// the tensor, so TMA fills it with zeros without reading memory (and the
// tensor cores multiply zeros, which draws less power than real rows).
constexpr int NO_ROWS = -BM;

__device__ void build_tasks(const FwdParams& p, const int* sS, int* dsm) {
  __shared__ int s_seg[E_MAX];  // per expert: segment count, then first segment
  __shared__ int s_mt[E_MAX];   // per expert: M-tile count, then first M-tile
  __shared__ int s_mtp[E_MAX];  // per expert: task slots per column tile (M-tiles, padded to pairs), then first
  __shared__ int s_tmp[SCHED_THREADS / 32];
  __shared__ int s_tot[4];
  const int E = p.E, b = p.b, n_mb = p.n_mb, tid = threadIdx.x;
  int* mb_tiles = dsm;             // per minibatch: M-tiles
  int* mt_first = dsm + n_mb;      // ... first M-tile
  int* mb_ptiles = dsm + 2 * n_mb;  // ... task slots per column tile (= mb_tiles without pairs)
  int* mtp_first = dsm + 3 * n_mb;  // ... first task slot
  int* step_off = dsm + 4 * n_mb;
  const int n_steps = n_mb + p.lag;
  // CTA pairs take two consecutive tasks on the same weight tile: a segment's
  // M-tile count is rounded up to even, the extra task being an empty partner
  auto padded = [&](int cnt) { return p.pair ? (cnt + 1) & ~1 : cnt; };

  for (int m = tid; m < n_mb; m += blockDim.x) mb_tiles[m] = mb_ptiles[m] = 0;
  if (tid < E) {
    int nseg = 0, ntile = 0, nptile = 0;
    if (sS[tid + 1] > sS[tid]) {
      const int m0 = sS[tid] / b, m1 = (sS[tid + 1] - 1) / b;
      nseg = m1 - m0 + 1;
      for (int m = m0; m <= m1; ++m) {
        int a, z;
        piece_rows(sS, tid, m, b, a, z);
        const int cnt = (z - a + BM - 1) / BM;
        ntile += cnt;
        nptile += padded(cnt);
      }
    }
    s_seg[tid] = nseg;
    s_mt[tid] = ntile;
    s_mtp[tid] = nptile;
  }
  __syncthreads();
  const int nseg_tot = block_exclusive_scan(s_seg, E, s_tmp);
  const int nmt_tot = block_exclusive_scan(s_mt, E, s_tmp);
  block_exclusive_scan(s_mtp, E, s_tmp);
  const bool fits = nseg_tot <= p.n_mb + E && nmt_tot <= p.n_mtiles_max;
  if (tid == 0 && !fits) raise_status(p.status, STATUS_SCHEDULE_INVALID);

  if (blockIdx.x == 0 && fits && tid < E && sS[tid + 1] > sS[tid]) {
    const int m0 = sS[tid] / b, m1 = (sS[tid + 1] - 1) / b;
    int g = s_seg[tid], mt = s_mt[tid];
    for (int m = m0; m <= m1; ++m, ++g) {
      int a, z;
      piece_rows(sS, tid, m, b, a, z);
      const int cnt = (z - a + BM - 1) / BM;
      int* sg = p.segs + 4 * g;
      sg[0] = tid;
      sg[1] = mt;
      sg[2] = cnt;
      sg[3] = m;
      mt += cnt;
    }
  }
  if (fits && tid < E && sS[tid + 1] > sS[tid]) {
    const int m0 = sS[tid] / b, m1 = (sS[tid + 1] - 1) / b;
    int mt = s_mt[tid], mtp = s_mtp[tid];
    for (int m = m0; m <= m1; ++m) {
      int a, z;
      piece_rows(sS, tid, m, b, a, z);
      const int cnt = (z - a + BM - 1) / BM;
      if (a == m * b) {  // exactly one segment opens each minibatch
        mt_first[m] = mt;
        mtp_first[m] = mtp;
      }
      atomicAdd(&mb_tiles[m], cnt);
      atomicAdd(&mb_ptiles[m], padded(cnt));
      mt += cnt;
      mtp += padded(cnt);
    }
  }
  __syncthreads();

  // per-minibatch task counts and the first task of every step
  if (blockIdx.x == 0) {
    for (int m = tid; m < n_mb; m += blockDim.x) {
      // tasks that complete per column tile: one per M-tile, and with split tail
      // tiles one per pair slot (both halves of a split tile complete)
      const int inc = p.half_tiles ? mb_ptiles[m] : mb_tiles[m];
      p.meta[META_MB + 4 * m] = fits ? inc * p.N1 : 0;
      p.meta[META_MB + 4 * m + 1] = fits ? inc * p.N2 : 0;
      p.meta[META_MB + 4 * m + 2] = fits ? mt_first[m] : 0;
      p.meta[META_MB + 4 * m + 3] = fits ? mb_tiles[m] : 0;
    }
  }
  for (int s = tid; s < n_steps; s += blockDim.x) {
    const int r1 = s < n_mb ? mb_ptiles[s] * p.N1 : 0;
    const int r2 = s - p.lag >= 0 ? mb_ptiles[s - p.lag] * p.N2 : 0;
    step_off[s] = r1 + r2;
  }
  __syncthreads();
  const int n_st = padded(p.n_smtiles);  // shared-expert token tiles, padded to pairs
  const int n_s1 = p.N1s * n_st, n_s2 = p.N2s * n_st;
  const int routed = block_exclusive_scan(step_off, n_steps, s_tmp);
  const long long total = (long long)n_s1 + routed + n_s2;
  if (tid == 0) {
    const bool ok = fits && total <= p.n_tasks_max;
    if (blockIdx.x == 0) {
      if (!ok) raise_status(p.status, STATUS_SCHEDULE_INVALID);
      p.meta[META_N_TASKS] = ok ? (int)total : 0;
      p.meta[META_N_MTILES] = nmt_tot;
      int y = 0;
      for (int m = 0; m < n_mb; ++m) y += (p.half_tiles ? mb_ptiles[m] : mb_tiles[m]) * p.N2;
      y += p.n_smtiles * p.N2s;
      p.meta[META_TOTAL_Y] = ok ? y : 0;
    }
    s_tot[0] = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s_tot[0]) return;

  // shared-expert tasks: tiles of 128 tokens, token-tile major (with pairs:
  // token-tile-pair major, the pair's two tiles side by side per column tile)
  for (int q = blockIdx.x * blockDim.x + tid; q < n_s1 + n_s2; q += gridDim.x * blockDim.x) {
    const bool down = q >= n_s1;
    const int qq = down ? q - n_s1 : q;
    const int nn = down ? p.N2s : p.N1s;
    const int mt = p.pair ? 2 * (qq / (2 * nn)) + (qq & 1) : qq / nn;
    const int n = p.pair ? (qq >> 1) % nn : qq % nn;
    const bool real = mt < p.n_smtiles;
    const int mtr = real ? mt : mt - 1;  // an empty partner takes its partner's rows (A: none)
    Task tk;
    tk.kind = down ? TASK_S2 : TASK_S1;
    tk.n = n;
    tk.e = 0;
    tk.a_row = real ? mtr * BM : NO_ROWS;
    tk.rows = real ? min(BM, p.T - mt * BM) : 0;
    tk.p0 = mtr * BM;
    tk.out_row = mtr * BM;
    tk.dep0 = down && real ? ctr_shready(p, mt) : -1;
    tk.need0 = down && real ? p.N1s : 0;
    tk.dep1 = -1;
    tk.need1 = 0;
    tk.done0 = !down && real ? ctr_shready(p, mt) : -1;
    tk.done1 = down && real ? ctr_ydone() : -1;  // the shared output is staging slot k
    tk.mt = mtr;
    tk.half = 0;
    tk.pad = 0;
    store_task(p.tasks + (down ? (int)total - n_s2 + qq : qq), tk);
  }
  // routed tasks: CTA c fills experts c, c + gridDim.x, ...; its threads stride
  // over the expert's tasks, segment by segment
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    if (sS[e + 1] <= sS[e]) continue;
    const int m0 = sS[e] / b, m1 = (sS[e + 1] - 1) / b;
    int mtb = s_mt[e], ptb = s_mtp[e];
    for (int m = m0; m <= m1; ++m) {
      int a, z;
      piece_rows(sS, e, m, b, a, z);
      const int cnt = (z - a + BM - 1) / BM;
      const int cntp = padded(cnt);
      const int slot_row = (m % p.slots) * b;
      const int r1_base = n_s1 + step_off[m] + p.N1 * (ptb - mtp_first[m]);
      const int sr2 = m + p.lag;
      const int r2_base =
          n_s1 + step_off[sr2] + (sr2 < n_mb ? mb_ptiles[sr2] * p.N1 : 0) + p.N2 * (ptb - mtp_first[m]);
      const int need_h = m >= p.slots ? (p.half_tiles ? mb_ptiles[m - p.slots] : mb_tiles[m - p.slots]) * p.N2 : 0;
      // BF16 pairs: an odd segment's last M-tile is split over the pair's two
      // tasks (rows 0-63 and 64-127, one M = 128 MMA) instead of padded
      const bool split_tail = p.half_tiles && (cnt & 1);
      for (int q = tid; q < cntp * (p.N1 + p.N2); q += blockDim.x) {
        const bool down = q >= cntp * p.N1;
        const int qq = down ? q - cntp * p.N1 : q;
        int i, n;
        if (down) {  // column-tile major: the segment's tiles share a weight slice
          i = qq % cntp;
          n = qq / cntp;
        } else {  // groups of p.raster M-tiles, each sweeping the column tiles
          const int grp = qq / (p.raster * p.N1), within = qq % (p.raster * p.N1);
          const int gc = min(p.raster, cntp - grp * p.raster);  // M-tiles in this group
          i = grp * p.raster + within % gc;
          n = within / gc;
        }
        const bool half = split_tail && i >= cnt - 1;  // half h = i - (cnt - 1) of the last tile
        const bool real = i < cnt || half;
        const int ir = half ? cnt - 1 : (real ? i : i - 1);  // an empty partner takes its partner's rows (A: none)
        const int hh = half ? i - (cnt - 1) : 0;
        const int r0 = a + ir * BM + (BM / 2) * hh;
        Task tk;
        tk.kind = down ? TASK_R2 : TASK_R1;
        tk.n = n;
        tk.e = e;
        tk.out_row = slot_row + (r0 - m * b);
        tk.a_row = real ? tk.out_row : NO_ROWS;
        tk.rows = half ? max(0, min(BM / 2, z - r0)) : (real ? min(BM, z - r0) : 0);
        tk.p0 = r0;
        tk.half = half ? 1 : 0;
        if (!real) {
          tk.dep0 = tk.dep1 = tk.done0 = tk.done1 = -1;
          tk.need0 = tk.need1 = 0;
        } else if (!down) {
          tk.dep0 = p.direct ? -1 : ctr_filled(p, m);  // direct dispatch: x itself is the A operand
          tk.need0 = p.gparts;
          tk.dep1 = m >= p.slots ? ctr_r2(p, m - p.slots) : -1;
          tk.need1 = need_h;
          tk.done0 = ctr_hready(p, mtb + ir);
          tk.done1 = ctr_r1(p, m);
        } else {
          tk.dep0 = ctr_hready(p, mtb + ir);
          tk.need0 = half ? 2 * p.N1 : p.N1;  // both halves of a split tile count on its counter
          tk.dep1 = -1;
          tk.need1 = 0;
          tk.done0 = ctr_r2(p, m);
          tk.done1 = ctr_ydone();
        }
        tk.mt = mtb + ir;
        tk.pad = 0;
        store_task(p.tasks + (down ? r2_base : r1_base) + qq, tk);
      }
      for (int i = tid; i < cnt; i += blockDim.x) {  // the M-tile table (the gather walks it)
        int* mr = p.mtiles + 4 * (mtb + i);
        mr[0] = e;
        mr[1] = a + i * BM;
        mr[2] = min(BM, z - (a + i * BM));
        mr[3] = m;
      }
      mtb += cnt;
      ptb += cntp;
    }
  }
}

// dynamic shared memory of build_tasks: mb_tiles, mt_first, mb_ptiles and
// mtp_first [n_mb] each, then step_off [n_mb + lag + 1]
__host__ __device__ inline int sched_dyn_ints(int n_mb, int lag) { return 4 * n_mb + (n_mb + lag + 1); }

int schedule_smem_bytes(const FwdParams& p) { return (int)sizeof(int) * sched_dyn_ints(p.n_mb, p.lag); }

cudaError_t launch_schedule(const FwdParams& p, cudaStream_t stream) {
  const int smem = schedule_smem_bytes(p);
  if (smem > 48 * 1024) {
    const cudaError_t err = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
  }
  schedule_kernel<<<p.n_chunks, SCHED_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
