// Backward pass of the MoE layer on tcgen05 tensor cores.
//
// "Mixture-of-Kittens: MoE Megakernel for NVL72s" trains the layer of Sec. 2.1
// (Eq. MoE); its backward reuses the forward's dispatch schedule (Sec. 3.1:
// one table serves every communication step, the backward's included),
// recomputes the forward's expert activations instead of keeping them
// (Sec. 3.3 "Ring-Aware Forward Replay") and takes the router-weight gradient
// from the inner product of the gated activation h with the down projection's
// input gradient W_down^T dO (Sec. 3.4 "Router Weight Gradient Computation",
// the SonicMoE form), so the routed experts' outputs are never materialised.
// With every expert on this GPU the replay recomputes the up/gate projections
// of every route: the forward keeps no pre-activation.
//
// Chain rule for route j = (token t, slot) with expert e and router weight g_j
// (a_u = W_up[e] x, a_g = W_gate[e] x, h = SiLU(a_g) a_u):
//   dh' = W_down[e]^T dO_t;  dg_j = <dh', h>;  dh = g_j dh'
//   da_u = dh SiLU(a_g);  da_g = dh a_u SiLU'(a_g),  SiLU'(z) = s(z)(1 + z(1 - s(z)))
//   dW_down[e] = sum_j dO_t (g_j h)^T;  dW_up[e] = sum_j da_u x_t^T;  dW_gate[e] = sum_j da_g x_t^T
//   dx_t += W_up[e]^T da_u + W_gate[e]^T da_g
// The shared expert is the same with g = 1 over all tokens.  Router: with
// c_t = sum_j g_j dg_j, sigmoid scores give dl_j = (dg_j - c_t) / S_t s_j (1 - s_j)
// (S_t = sum of the selected scores), softmax gives dl_j = g_j (dg_j - c_t);
// dW_r[e] = sum_j dl_j x_t, db_e = sum_j dl_j, dx_t += sum_j dl_j W_r[e].
//
// Kernels, in stream order:
//   bwd_prep        expert segments padded to 64 routes, M-tile list, expert order
//   bwd_gather      x and dO rows of every route into the padded expert-major buffers
//   bwd_gemm<0>     per (M-tile, 128 columns of I): replayed up/gate GEMM and the
//                   dh' GEMM (W_down[e] as an MN-major operand), epilogue -> g h,
//                   da_u, da_g (bf16) and dg partial sums
//   bwd_router_dl   dg (fixed-order sum of the partials), dl per route
//   bwd_gemm<1>     dx per route ([da_u da_g] x [W_up; W_gate], MN-major B, K = 2I),
//                   dW_down / dW_up / dW_gate per (expert, output tile) with both
//                   operands MN-major and K = the expert's padded routes, and the
//                   shared expert's
//   bwd_router_wr   dW_r / db partial sums over chunks of each expert's routes
//   bwd_router_fin  fixed-order sum of the chunk partials
//   bwd_dx_combine  dx_t = shared + sum over slots + router term, fixed order
// No floating-point atomics anywhere: every output element comes from one tile
// with a fixed K order or from a fixed-order sum.
#include "common.cuh"
#include "plan.cuh"

#include <cstring>

namespace moe {

constexpr int BWD_THREADS = 256;
constexpr int BWD_STAGES = 4;
constexpr int BWD_STAGE = 49152;   // A 16 KB + B 32 KB, 1024-aligned
constexpr int BWD_QN = 8;
constexpr int BOXB = 8192;         // one {64, 64} bf16 box: 64 rows x 128 B
constexpr int PADK = 64;           // an expert's routes padded to a multiple of 64 (one K step)
constexpr int WR_CHUNK = 256;      // routes per router-gradient partial sum
constexpr int BWD_BAR_BYTES = 512;
constexpr int BWD_SMEM = BWD_STAGES * BWD_STAGE + 1024 + BWD_BAR_BYTES;
// CTA pairs: per CTA and stage its A (16 KB) and its half of B (up to 16 KB)
constexpr int BWD_PAIR_STAGES = 6;
constexpr int BWD_PAIR_STAGE = 32768;
constexpr int BWD_PAIR_SMEM = BWD_PAIR_STAGES * BWD_PAIR_STAGE + 1024 + BWD_BAR_BYTES;

enum : int {
  BU_A_ROUTED = 0, BU_A_SHARED, BU_DX_ROUTED, BU_DX_SHARED, BU_DW_DOWN, BU_DW_UP, BU_DW_GATE, BU_DWS_DOWN,
  BU_DWS_UP, BU_DWS_GATE
};
enum : int { BM_NMT = 0, BM_RP = 1, BM_NWC = 2 };  // meta words

struct BwdMaps {  // every map: 2-D row-major bf16, box {64 columns, 64 rows}, 128-byte swizzle
  CUtensorMap xg, dOg, hg, dau, dag;     // [Rp, D], [Rp, D], [Rp, I] x 3
  CUtensorMap w_up, w_gate, w_down;      // [E*I, D], [E*I, D], [E*D, I]
  CUtensorMap x, dO;                     // [T, D]
  CUtensorMap hs, dasu, dasg;            // [T, I_s]
  CUtensorMap ws_up, ws_gate, ws_down;   // [I_s, D], [I_s, D], [D, I_s]
  // the same tensors read K-major, 128 rows per load: box {64 columns, 128 rows}
  CUtensorMap k_xg, k_dOg, k_dau, k_dag, k_w_up, k_w_gate, k_x, k_dO, k_dasu, k_dasg, k_ws_up, k_ws_gate;
  // ... and read MN-major, two 64-column blocks per load: a 3-D view (64 columns,
  // row, 64-column block; the block stride 128 bytes), box {64, 64, 2}
  CUtensorMap m_xg, m_dOg, m_hg, m_dau, m_dag, m_w_up, m_w_gate, m_w_down;
  CUtensorMap m_x, m_dO, m_hs, m_dasu, m_dasg, m_ws_up, m_ws_gate, m_ws_down;
};

struct BwdParams {
  int T, D, I, E, k, I_s, kY, score_fn;
  int N1, N1s, N2;        // I/128, I_s/128, D/256 column tiles
  int n_tt;               // token tiles ceil(T/128)
  int n_mt_max, Rp_max, n_wc_max;
  int pair;               // 1: CTA pairs (cta_group::2); M-tile entries are pairs of tiles
  int mn3d;               // 1: the 3-D MN-major maps are encoded (two 64-column blocks per load)
  long long timeout_ns;
  // the forward's routing and schedule (its workspace)
  const int* topk_idx;
  const float* topk_w;
  const float* topk_logit;
  const int* M;
  const int* S;
  const int* sched;
  // inputs
  const bf16* x;
  const bf16* dO;
  const bf16* w_router;
  // workspace
  int* status;
  int* counters;          // [0] phase-A claims, [1] phase-B claims
  int* meta;              // BM_*
  int* Sp;                // [E + 1] padded segment starts
  int* wc0;               // [E + 1] first router-gradient chunk of each expert
  int* eorder;            // [E] experts by descending route count
  int* mtiles;            // [n_mt_max, 4] {e, first padded row, rows, -}; pairs: {e, first row, rows of
                          // the first tile, rows of the second (0: an empty partner)}
  int* prow_route;        // [Rp_max] route of a padded row, -1 for padding
  int* route_prow;        // [T k] padded row of a route
  bf16* xg;               // [Rp_max, D]
  bf16* dOg;              // [Rp_max, D]
  bf16* hg;               // [Rp_max, I]  g h
  bf16* dau;              // [Rp_max, I]
  bf16* dag;              // [Rp_max, I]
  float* dgp;             // [Rp_max, N1] dg partial sums per 128 columns of I
  bf16* hs;               // [T, I_s]
  bf16* dasu;             // [T, I_s]
  bf16* dasg;             // [T, I_s]
  __half* dxs;            // [T, kY, D] dx per route (slot k: the shared expert)
  float* dl;              // [T k]
  float* wr_part;         // [n_wc_max, D]
  float* wb_part;         // [n_wc_max]
  // outputs
  bf16* dx;
  float* dW_r;
  float* db_r;
  bf16* dW_up;
  bf16* dW_gate;
  bf16* dW_down;
  bf16* dWs_up;
  bf16* dWs_gate;
  bf16* dWs_down;
};

// Shared-memory descriptor of an MN-major operand staged by {64, 64} TMA boxes
// with 128-byte swizzle: 64-wide MN blocks one box (8192 B) apart (leading
// byte offset), 8-row K groups 1024 B apart (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(BOXB >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
constexpr uint32_t IDESC_A_MN = 1u << 15, IDESC_B_MN = 1u << 16;

// ------------------------------------------------------------------ prep
// One CTA: padded segment starts Sp (each expert's routes rounded up to 64),
// the 128-row M-tiles over them, the experts by descending route count (ties:
// lower id first) and the router-gradient chunks; zeroes the claim counters
// and the status words.
__global__ void __launch_bounds__(512, 1) bwd_prep(BwdParams p) {
  __shared__ int sM[E_MAX], sPad[E_MAX + 1], sTiles[E_MAX + 1], sChunk[E_MAX + 1];
  const int E = p.E, tid = threadIdx.x;
  if (tid == 0) {
    p.status[0] = 0;
    p.status[1] = 0;
    p.counters[0] = 0;
    p.counters[1] = 0;
  }
  for (int e = tid; e < E; e += blockDim.x) sM[e] = p.M[e];
  __syncthreads();
  if (tid == 0) {  // E <= 512: serial scans in fixed order
    int sp = 0, mt = 0, wc = 0;
    const int tile_rows = p.pair ? 2 * BM : BM;  // rows of one M-tile entry
    for (int e = 0; e < E; ++e) {
      const int m64 = (sM[e] + PADK - 1) / PADK * PADK;
      sPad[e] = sp;
      sTiles[e] = mt;
      sChunk[e] = wc;
      sp += m64;
      mt += (m64 + tile_rows - 1) / tile_rows;
      wc += (sM[e] + WR_CHUNK - 1) / WR_CHUNK;
    }
    sPad[E] = sp;
    sTiles[E] = mt;
    sChunk[E] = wc;
    p.meta[BM_NMT] = mt;
    p.meta[BM_RP] = sp;
    p.meta[BM_NWC] = wc;
    if (sp > p.Rp_max || mt > p.n_mt_max || wc > p.n_wc_max) raise_status(p.status, STATUS_SCHEDULE_INVALID);
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {
    p.Sp[e] = sPad[e];
    p.wc0[e] = sChunk[e];
  }
  for (int e = tid; e < E; e += blockDim.x) {
    int rank = 0;
    for (int f = 0; f < E; ++f) rank += (sM[f] > sM[e] || (sM[f] == sM[e] && f < e)) ? 1 : 0;
    p.eorder[rank] = e;
    const int m64 = sPad[e + 1] - sPad[e];
    const int tile_rows = p.pair ? 2 * BM : BM;
    for (int i = 0; i * tile_rows < m64 && sTiles[e] + i < p.n_mt_max; ++i) {
      int* r = p.mtiles + 4 * (sTiles[e] + i);
      r[0] = e;
      r[1] = sPad[e] + i * tile_rows;
      r[2] = min(BM, m64 - i * tile_rows);
      r[3] = p.pair ? max(0, min(BM, m64 - i * tile_rows - BM)) : 0;
    }
  }
}

// ------------------------------------------------------------------ gather
// Padded row p of expert e (Sp[e] <= p < Sp[e+1]) holds route o = p - Sp[e] of
// e's schedule region (x and dO of its token), or zeros past the expert's
// routes.  One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) bwd_gather(BwdParams p) {
  __shared__ int sSp[E_MAX + 1];
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x) sSp[e] = p.Sp[e];
  __syncthreads();
  const int Rp = min(sSp[p.E], p.Rp_max);
  const int lane = threadIdx.x & 31;
  const int nv = p.D / 8;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < Rp; r += warps) {
    int lo = 0, hi = p.E;  // last e with Sp[e] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sSp[mid] <= r) lo = mid;
      else hi = mid;
    }
    const int e = lo, o = r - sSp[e];
    uint4* dx4 = reinterpret_cast<uint4*>(p.xg + (size_t)r * p.D);
    uint4* dd4 = reinterpret_cast<uint4*>(p.dOg + (size_t)r * p.D);
    if (o < p.M[e]) {
      const int P = p.S[e] + o;
      const int t = p.sched[3 * (size_t)P], j = p.sched[3 * (size_t)P + 2];
      const uint4* sx = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.D);
      const uint4* sd = reinterpret_cast<const uint4*>(p.dO + (size_t)t * p.D);
      for (int v = lane; v < nv; v += 32) {
        const uint4 a = __ldg(sx + v), b = __ldg(sd + v);
        dx4[v] = a;
        dd4[v] = b;
      }
      if (lane == 0) {
        p.prow_route[r] = j;
        p.route_prow[j] = r;
      }
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = lane; v < nv; v += 32) {
        dx4[v] = z;
        dd4[v] = z;
      }
      if (lane == 0) p.prow_route[r] = -1;
    }
  }
}

// ------------------------------------------------------------------ GEMM units
struct BUnit {
  int kind, e, m, n, a_row, rows, k0, nk1, nk2;
};

// Units: one per CTA, or with CTA pairs one per pair (the pair's two CTAs
// take two 128-row tiles that share the weight tile, each loading half of it).
__device__ __forceinline__ int bwd_units(const BwdParams& p, int phase) {
  const int n_mt = min(p.meta[BM_NMT], p.n_mt_max);
  const bool sh = p.I_s > 0;
  const int rt = p.pair ? 2 * BM : BM;  // output rows per unit of the weight gradients
  const int n_tt = p.pair ? (p.n_tt + 1) / 2 : p.n_tt;
  if (phase == 0) return n_mt * p.N1 + (sh ? n_tt * p.N1s : 0);
  const int c_e = (p.D / rt) * (p.I / 256) + 2 * (p.I / rt) * (p.D / 256);
  const int c_s = sh ? (p.D / rt) * (p.I_s / 256) + 2 * (p.I_s / rt) * (p.D / 256) : 0;
  return c_s + p.E * c_e + n_mt * p.N2 + (sh ? n_tt * p.N2 : 0);
}

// Phase 0: routed (M-tile, 128 columns of I) units, then the shared expert's
// (token tile, 128 columns of I_s).  Phase 1: the shared expert's weight
// gradients (K = T), the routed weight gradients expert by expert in
// descending route count (K = the expert's padded routes), then dx per route
// and the shared expert's dx (K = 2I and 2 I_s): longest units first.  With
// CTA pairs, `rank` picks this CTA's tile of the pair's two (rows = 0: an
// empty partner, whose A box lies outside its tensor and is zero-filled).
__device__ __forceinline__ BUnit bwd_decode(const BwdParams& p, int phase, int u, int rank) {
  BUnit b{};
  const int n_mt = min(p.meta[BM_NMT], p.n_mt_max);
  const int rt = p.pair ? 2 * BM : BM;
  auto routed_tile = [&](int mt) {
    b.e = p.mtiles[4 * mt];
    const int row0 = p.mtiles[4 * mt + 1];
    b.rows = rank ? p.mtiles[4 * mt + 3] : p.mtiles[4 * mt + 2];
    b.a_row = b.rows > 0 ? row0 + rank * BM : -2 * BM;
  };
  auto shared_tile = [&](int tp) {
    const int tt = p.pair ? 2 * tp + rank : tp;
    b.rows = max(0, min(BM, p.T - tt * BM));
    b.a_row = b.rows > 0 ? tt * BM : -2 * BM;
  };
  if (phase == 0) {
    const int nr = n_mt * p.N1;
    if (u < nr) {
      b.kind = BU_A_ROUTED;
      b.n = u % p.N1;
      routed_tile(u / p.N1);
    } else {
      const int v = u - nr;
      b.kind = BU_A_SHARED;
      b.n = v % p.N1s;
      shared_tile(v / p.N1s);
    }
    b.nk1 = b.nk2 = p.D / BK;
    return b;
  }
  const bool sh = p.I_s > 0;
  const int c_e = (p.D / rt) * (p.I / 256) + 2 * (p.I / rt) * (p.D / 256);
  const int c_s = sh ? (p.D / rt) * (p.I_s / 256) + 2 * (p.I_s / rt) * (p.D / 256) : 0;
  int v = u;
  if (v < c_s) {  // shared expert weight gradients, K = T
    const int nd = (p.D / rt) * (p.I_s / 256), nu = (p.I_s / rt) * (p.D / 256);
    b.nk1 = (p.T + BK - 1) / BK;
    if (v < nd) {
      b.kind = BU_DWS_DOWN;
      b.m = v / (p.I_s / 256);
      b.n = v % (p.I_s / 256);
    } else {
      v -= nd;
      b.kind = v < nu ? BU_DWS_UP : BU_DWS_GATE;
      v %= nu;
      b.m = v / (p.D / 256);
      b.n = v % (p.D / 256);
    }
    if (p.pair) b.m = 2 * b.m + rank;  // in 128-row tiles of the output
    return b;
  }
  v -= c_s;
  if (v < p.E * c_e) {  // routed weight gradients of expert eorder[v / c_e]
    b.e = p.eorder[v / c_e];
    v %= c_e;
    b.k0 = p.Sp[b.e];
    b.nk1 = (p.Sp[b.e + 1] - b.k0) / PADK;
    const int nd = (p.D / rt) * (p.I / 256), nu = (p.I / rt) * (p.D / 256);
    if (v < nd) {
      b.kind = BU_DW_DOWN;
      b.m = v / (p.I / 256);
      b.n = v % (p.I / 256);
    } else {
      v -= nd;
      b.kind = v < nu ? BU_DW_UP : BU_DW_GATE;
      v %= nu;
      b.m = v / (p.D / 256);
      b.n = v % (p.D / 256);
    }
    if (p.pair) b.m = 2 * b.m + rank;
    return b;
  }
  v -= p.E * c_e;
  if (v < n_mt * p.N2) {  // dx of the routes of one M-tile (pair)
    b.kind = BU_DX_ROUTED;
    b.n = v % p.N2;
    routed_tile(v / p.N2);
    b.nk1 = b.nk2 = p.I / BK;
    return b;
  }
  v -= n_mt * p.N2;
  b.kind = BU_DX_SHARED;  // the shared expert's dx
  b.n = v % p.N2;
  shared_tile(v / p.N2);
  b.nk1 = b.nk2 = p.I_s / BK;
  return b;
}

__device__ __forceinline__ int unit_steps(const BUnit& b) {
  return (b.kind == BU_A_ROUTED || b.kind == BU_A_SHARED || b.kind == BU_DX_ROUTED || b.kind == BU_DX_SHARED)
             ? b.nk1 + b.nk2
             : b.nk1;
}

// {64, 64} boxes one CTA loads for K step s of unit b: A is always two (128
// rows or columns); B is the whole weight tile for one CTA, or this CTA's half
// of it in a pair.
__device__ __forceinline__ uint32_t step_boxes(const BUnit& b, int s, bool pair) {
  const bool dh = (b.kind == BU_A_ROUTED || b.kind == BU_A_SHARED) && s >= b.nk1;  // B: 128 columns of W_down
  return 2u + (dh ? (pair ? 1u : 2u) : (pair ? 2u : 4u));
}

// TMA loads of K step s of unit b into stage (sa: A, 16 KB; sb: B, up to
// 32 KB).  One CTA: every box completes on `bar`.  CTA pairs: every box of
// both CTAs completes on the even CTA's barrier (`bar_pair`, a cluster
// address); this CTA loads its own A rows and its half of B -- for the
// replayed up/gate tile the even CTA the up rows and the odd CTA the gate
// rows, otherwise the first or second half of the N columns.
template <bool kPair>
__device__ __forceinline__ void bwd_issue(const BwdMaps& mp, const BwdParams& p, const BUnit& b, int s, uint8_t* sa,
                                          uint8_t* sb, uint64_t* bar, uint32_t bar_pair, int rank) {
  auto box = [&](uint8_t* dst, const CUtensorMap* m, int c0, int c1) {
    if constexpr (kPair) tma_load_2d_pair(dst, m, bar_pair, c0, c1);
    else tma_load_2d(dst, m, bar, c0, c1);
  };
  // MN-major columns [col, col + 128) of K rows [krow, krow + 64): one 3-D load,
  // or two {64, 64} boxes
  auto mn128 = [&](uint8_t* dst, const CUtensorMap* m2, const CUtensorMap* m3, int col, int krow) {
    if (p.mn3d) {
      if constexpr (kPair) tma_load_3d_pair(dst, m3, bar_pair, 0, krow, col / 64);
      else tma_load_3d(dst, m3, bar, 0, krow, col / 64);
    } else {
      box(dst, m2, col, krow);
      box(dst + BOXB, m2, col + 64, krow);
    }
  };
  switch (b.kind) {
    case BU_A_ROUTED:
    case BU_A_SHARED: {
      const bool r = b.kind == BU_A_ROUTED;
      if (s < b.nk1) {  // replayed up/gate: A = x rows (K-major), B = [W_up; W_gate] rows (K-major)
        const int kc = s * BK;
        box(sa, r ? &mp.k_xg : &mp.k_x, kc, b.a_row);  // 128 rows
        const int br = (r ? b.e * p.I : 0) + b.n * BN_UP;
        const CUtensorMap* up = r ? &mp.k_w_up : &mp.k_ws_up;
        const CUtensorMap* gt = r ? &mp.k_w_gate : &mp.k_ws_gate;
        if (kPair) {
          box(sb, rank ? gt : up, kc, br);
        } else {
          box(sb, up, kc, br);
          box(sb + 2 * BOXB, gt, kc, br);
        }
        return;
      }
      // dh' = dO W_down[e]: A = dO rows (K-major), B = W_down[e] [D, I] MN-major (N = I contiguous)
      const int kc = (s - b.nk1) * BK;
      box(sa, r ? &mp.k_dOg : &mp.k_dO, kc, b.a_row);
      const CUtensorMap* dn = r ? &mp.w_down : &mp.ws_down;
      const int krow = (r ? b.e * p.D : 0) + kc;
      if (kPair) {
        box(sb, dn, b.n * BN_UP + 64 * rank, krow);
      } else {
        mn128(sb, dn, r ? &mp.m_w_down : &mp.m_ws_down, b.n * BN_UP, krow);
      }
      return;
    }
    case BU_DX_ROUTED:
    case BU_DX_SHARED: {  // dx = [da_u da_g] [W_up; W_gate]: A K-major, B [I, D] MN-major (N = D contiguous)
      const bool r = b.kind == BU_DX_ROUTED;
      const bool second = s >= b.nk1;
      const int kc = (second ? s - b.nk1 : s) * BK;
      box(sa, r ? (second ? &mp.k_dag : &mp.k_dau) : (second ? &mp.k_dasg : &mp.k_dasu), kc, b.a_row);
      const CUtensorMap* w = r ? (second ? &mp.w_gate : &mp.w_up) : (second ? &mp.ws_gate : &mp.ws_up);
      const CUtensorMap* w3 = r ? (second ? &mp.m_w_gate : &mp.m_w_up) : (second ? &mp.m_ws_gate : &mp.m_ws_up);
      const int krow = (r ? b.e * p.I : 0) + kc;
      const int nq = kPair ? 1 : 2, q0 = kPair ? rank : 0;  // 128-column halves
      for (int q = 0; q < nq; ++q) mn128(sb + 2 * q * BOXB, w, w3, b.n * 256 + 128 * (q0 + q), krow);
      return;
    }
    default: {  // weight gradients: A and B MN-major, K = routes (or tokens)
      const CUtensorMap *a, *bm, *a3, *bm3;
      switch (b.kind) {
        case BU_DW_DOWN: a = &mp.dOg; bm = &mp.hg; a3 = &mp.m_dOg; bm3 = &mp.m_hg; break;
        case BU_DW_UP: a = &mp.dau; bm = &mp.xg; a3 = &mp.m_dau; bm3 = &mp.m_xg; break;
        case BU_DW_GATE: a = &mp.dag; bm = &mp.xg; a3 = &mp.m_dag; bm3 = &mp.m_xg; break;
        case BU_DWS_DOWN: a = &mp.dO; bm = &mp.hs; a3 = &mp.m_dO; bm3 = &mp.m_hs; break;
        case BU_DWS_UP: a = &mp.dasu; bm = &mp.x; a3 = &mp.m_dasu; bm3 = &mp.m_x; break;
        default: a = &mp.dasg; bm = &mp.x; a3 = &mp.m_dasg; bm3 = &mp.m_x; break;
      }
      const int krow = b.k0 + s * BK;
      mn128(sa, a, a3, b.m * BM, krow);
      const int nq = kPair ? 1 : 2, q0 = kPair ? rank : 0;  // 128-column halves
      for (int q = 0; q < nq; ++q) mn128(sb + 2 * q * BOXB, bm, bm3, b.n * 256 + 128 * (q0 + q), krow);
      return;
    }
  }
}

// ------------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ void store_bf16x32(bf16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}
// fp16 with saturation at +-65504; returns true if a value left that range (or is NaN)
__device__ __forceinline__ bool store_f16x32_sat(__half* dst, const float* v) {
  bool bad = false;
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float a = v[2 * i], b = v[2 * i + 1];
    bad |= !(fabsf(a) <= 65504.0f) || !(fabsf(b) <= 65504.0f);
    __half2 h = __floats2half2_rn(fminf(fmaxf(a, -65504.0f), 65504.0f), fminf(fmaxf(b, -65504.0f), 65504.0f));
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  return bad;
}

// Phase 0 epilogue of one row (TMEM lane): columns [0,128) up, [128,256) gate,
// [256,384) dh'.  Writes g h, da_u, da_g (bf16) for 128 columns of I and
// returns this row's part of dg = <dh', h> (fp32, columns in order).
__device__ __forceinline__ float epi_act_grad(uint32_t taddr, float g, bool store, bf16* hg_row, bf16* dau_row,
                                              bf16* dag_row) {
  float dg = 0.0f;
#pragma unroll 1
  for (int c = 0; c < BN_UP; c += 32) {
    uint32_t u[32], gt[32], d[32];
    tmem_ld_32x32b_x32(taddr + (uint32_t)c, u);
    tmem_ld_32x32b_x32(taddr + (uint32_t)(BN_UP + c), gt);
    tmem_ld_32x32b_x32(taddr + (uint32_t)(2 * BN_UP + c), d);
    tmem_ld_wait();
    float vh[32], vu[32], vg[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float au = __uint_as_float(u[j]), ag = __uint_as_float(gt[j]), dh1 = __uint_as_float(d[j]);
      const float sg = __fdividef(1.0f, 1.0f + __expf(-ag));
      const float si = ag * sg;
      const float h = si * au;
      dg = fmaf(dh1, h, dg);
      const float dh = g * dh1;
      vh[j] = g * h;
      vu[j] = dh * si;
      vg[j] = dh * au * sg * (1.0f + ag * (1.0f - sg));
    }
    if (store) {
      store_bf16x32(hg_row + c, vh);
      store_bf16x32(dau_row + c, vu);
      store_bf16x32(dag_row + c, vg);
    }
  }
  return dg;
}

// ------------------------------------------------------------------ the GEMM kernel
// Persistent, one CTA (or one CTA pair) per SM (pair), units claimed from a
// global counter.  Warp 0: TMA producer (the only or even CTA claims the units
// and hands them to its other warps, and to the odd CTA, through a queue in
// shared memory); warp 1: tcgen05.mma issuer (the even CTA issues for both CTAs
// of a pair, cta_group::2, M = 256); warps 2-5: epilogue of this CTA's 128 rows
// (TMEM lanes 32 (warp % 4) ...).  Phase 0 keeps one 384-column accumulator
// (up, gate, dh'); phase 1 alternates two 256-column accumulators.  The pair
// protocol (loads of both CTAs counted on the even CTA's full barrier, MMA
// commits multicast to both, accumulators handed back by remote arrivals) is
// the forward kernel's.
template <int PHASE, bool kPair>
__global__ void __launch_bounds__(BWD_THREADS, 1) bwd_gemm(const __grid_constant__ BwdMaps mp, const BwdParams p) {
  constexpr int NST = kPair ? BWD_PAIR_STAGES : BWD_STAGES;
  constexpr int STG = kPair ? BWD_PAIR_STAGE : BWD_STAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * STG);
  uint64_t* full = bars;                 // [NST]
  uint64_t* empty = bars + NST;          // [NST]
  uint64_t* tfull = bars + 2 * NST;      // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* qfull = tempty + 2;          // [BWD_QN]
  uint64_t* qempty = qfull + BWD_QN;     // [BWD_QN]
  uint64_t* drain = qempty + BWD_QN;
  volatile int* qslot = reinterpret_cast<volatile int*>(drain + 1);  // [BWD_QN]
  volatile int* s_unit = qslot + BWD_QN;
  volatile int* s_ok = s_unit + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(s_ok + 1));
  static_assert((2 * NST + 4 + 2 * BWD_QN + 1) * 8 + (BWD_QN + 3) * 4 <= BWD_BAR_BYTES, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = kPair ? (int)(cluster_ctarank() & 1u) : 0;
  const bool leader = rank == 0;
  const int n_units = bwd_units(p, PHASE);
  int* claim_ctr = p.counters + PHASE;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kPair ? 8 : 128);  // pairs: one arrival per epilogue warp of both CTAs
    }
    for (int i = 0; i < BWD_QN; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kPair ? 4 : 2);  // MMA issuer + epilogue (pairs: + the odd CTA's producer and epilogue)
    }
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair<512>(tmem_slot);
      tmem_relinquish_pair();
    } else {
      tmem_alloc<512>(tmem_slot);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the other CTA's barriers exist before anything targets them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // waits on barriers that the other CTA of a pair helps complete
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
    if constexpr (kPair) return mbar_wait_cluster(bar, parity, p.status, p.timeout_ns);
    else return mbar_wait(bar, parity, p.status, p.timeout_ns);
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full_even = kPair ? mapa_shared(full, 0) : 0u;
      const uint32_t q_odd = kPair ? mapa_shared(const_cast<int*>(qslot), 1) : 0u;
      const uint32_t qfull_odd = kPair ? mapa_shared(qfull, 1) : 0u;
      const uint32_t qempty_even = kPair ? mapa_shared(qempty, 0) : 0u;
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      int claim = leader ? atomicAdd(claim_ctr, 1) : 0;
      for (int i = 0;; ++i) {
        const int slot = i % BWD_QN;
        const uint32_t qpar = (uint32_t)(i / BWD_QN) & 1u;
        int u = -2;  // -2: a wait ran out; -1: no units left
        if (leader) {  // publish the claimed unit, then claim the one after it
          if (wait_bar(&qempty[slot], qpar ^ 1u)) {
            u = claim < n_units ? claim : -1;
            qslot[slot] = u;
            if constexpr (kPair) {
              st_shared_cluster_u32(q_odd + 4u * slot, (uint32_t)u);
              mbar_arrive_remote_cluster(qfull_odd + 8u * slot);
            }
            mbar_arrive(&qfull[slot]);
            if (u >= 0) claim = atomicAdd(claim_ctr, 1);
          }
        } else if (wait_bar(&qfull[slot], qpar)) {  // odd CTA: the even CTA's unit
          u = qslot[slot];
        }
        if (kPair && !leader && u != -2) mbar_arrive_remote(qempty_even + 8u * slot);
        if (u < 0) break;
        const BUnit b = bwd_decode(p, PHASE, u, rank);
        const int ns = unit_steps(b);
        bool ok = true;
        for (int s = 0; s < ns; ++s) {
          if (!wait_bar(&empty[stage], phase ^ 1u)) { ok = false; break; }
          uint8_t* sa = smem + stage * STG;
          // the byte count first (pairs: both CTAs' boxes, on the even CTA's barrier)
          if (leader) mbar_arrive_expect_tx(&full[stage], (kPair ? 2u : 1u) * step_boxes(b, s, kPair) * BOXB);
          bwd_issue<kPair>(mp, p, b, s, sa, sa + 2 * BOXB, &full[stage], full_even + stage * 8u, rank);
          ++issued;
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // the last loads issued have landed before the CTA may leave (pairs: the
      // even CTA's full barriers count both CTAs' loads, and the odd CTA waits
      // for the even one at the cluster barrier below)
      if (leader)
        for (int i = (issued > NST ? issued - NST : 0); i < issued; ++i)
          mbar_wait_drain(&full[i % NST], (uint32_t)(i / NST) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader && elect_one()) {
      const uint32_t M = kPair ? 2 * BM : BM;
      uint32_t stage = 0, phase = 0;
      uint32_t uses0 = 0u, uses1 = 0u;  // accumulator buffers' use counts (scalars: no local memory)
      uint32_t alt = 0;
      bool ok = true;
      auto mma = [&](uint32_t d, uint64_t a, uint64_t bd, uint32_t id, uint32_t acc_flag) {
        if constexpr (kPair) mma_bf16_pair(d, a, bd, id, acc_flag);
        else mma_bf16_ss(d, a, bd, id, acc_flag);
      };
      for (int i = 0; ok; ++i) {
        const int slot = i % BWD_QN;
        if (!wait_bar(&qfull[slot], (uint32_t)(i / BWD_QN) & 1u)) break;
        const int u = qslot[slot];
        mbar_arrive(&qempty[slot]);
        if (u < 0) break;
        const BUnit b = bwd_decode(p, PHASE, u, 0);
        const uint32_t acc = PHASE == 0 ? 0u : alt;
        alt ^= (PHASE == 0 ? 0u : 1u);
        if (!wait_bar(&tempty[acc], ((acc ? uses1 : uses0) & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256u;
        const int ns = unit_steps(b);
        for (int s = 0; s < ns; ++s) {
          if (!wait_bar(&full[stage], phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STG);
          const uint32_t b_addr = a_addr + 2 * BOXB;
          if (b.kind == BU_A_ROUTED || b.kind == BU_A_SHARED) {
            if (s < b.nk1) {  // up/gate into columns [0, 256)
              const uint32_t id = idesc_bf16_f32(M, 256);
#pragma unroll
              for (int kk = 0; kk < BK / UMMA_K; ++kk)
                mma(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32), id,
                    (s | kk) != 0 ? 1u : 0u);
            } else {  // dh' into columns [256, 384)
              const uint32_t id = idesc_bf16_f32(M, BN_UP) | IDESC_B_MN;
              const int s2 = s - b.nk1;
#pragma unroll
              for (int kk = 0; kk < BK / UMMA_K; ++kk)
                mma(d + 256u, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_mnmajor_sw128(b_addr + kk * 2048), id,
                    (s2 | kk) != 0 ? 1u : 0u);
            }
          } else if (b.kind == BU_DX_ROUTED || b.kind == BU_DX_SHARED) {
            const uint32_t id = idesc_bf16_f32(M, 256) | IDESC_B_MN;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              mma(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_mnmajor_sw128(b_addr + kk * 2048), id,
                  (s | kk) != 0 ? 1u : 0u);
          } else {
            const uint32_t id = idesc_bf16_f32(M, 256) | IDESC_A_MN | IDESC_B_MN;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              mma(d, sdesc_mnmajor_sw128(a_addr + kk * 2048), sdesc_mnmajor_sw128(b_addr + kk * 2048), id,
                  (s | kk) != 0 ? 1u : 0u);
          }
          if constexpr (kPair) mma_commit_pair(&empty[stage], 0x3);
          else mma_commit(&empty[stage]);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        // (a unit with no K steps only hands the buffer on)
        if constexpr (kPair) mma_commit_pair(&tfull[acc], 0x3);
        else mma_commit(&tfull[acc]);
        if (acc) ++uses1; else ++uses0;
      }
      if constexpr (kPair) mma_commit_pair(drain, 0x1);
      else mma_commit(drain);
      mbar_wait_drain(drain, 0, p.timeout_ns);  // every MMA issued has completed before TMEM is freed
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 6) {
    const int q = warp & 3;
    const int rloc = q * 32 + lane;  // this thread's tile row (TMEM lane)
    const uint32_t tempty_even = kPair ? mapa_shared(tempty, 0) : 0u;
    const uint32_t qempty_even = kPair ? mapa_shared(qempty, 0) : 0u;
    uint32_t uses0 = 0u, uses1 = 0u;
    uint32_t alt = 0;
    bool ovf = false;
    for (int i = 0;; ++i) {
      if (threadIdx.x == 64) {  // one thread decides for the four warps
        const int slot = i % BWD_QN;
        if (wait_bar(&qfull[slot], (uint32_t)(i / BWD_QN) & 1u)) {
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
      const BUnit b = bwd_decode(p, PHASE, u, rank);
      const uint32_t acc = PHASE == 0 ? 0u : alt;
      alt ^= (PHASE == 0 ? 0u : 1u);
      if (threadIdx.x == 64) *s_ok = wait_bar(&tfull[acc], (acc ? uses1 : uses0) & 1u) ? 1 : 0;
      named_bar_sync(1, 128);
      if (*s_ok == 0) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * 256u;
      if (b.kind == BU_A_ROUTED) {
        const bool valid = rloc < b.rows;
        const int prow = b.a_row + rloc;
        const int j = valid ? p.prow_route[prow] : -1;
        const float g = j >= 0 ? p.topk_w[j] : 0.0f;  // padding rows: all zero
        const size_t o = valid ? (size_t)prow * p.I + b.n * BN_UP : 0;
        const float dg = epi_act_grad(taddr, g, valid, p.hg + o, p.dau + o, p.dag + o);
        if (j >= 0) p.dgp[(size_t)prow * p.N1 + b.n] = dg;
      } else if (b.kind == BU_A_SHARED) {
        const int t = b.a_row + rloc;
        const bool valid = rloc < b.rows;
        const size_t o = (size_t)(valid ? t : 0) * p.I_s + b.n * BN_UP;
        epi_act_grad(taddr, 1.0f, valid, p.hs + o, p.dasu + o, p.dasg + o);
      } else if (b.kind == BU_DX_ROUTED || b.kind == BU_DX_SHARED) {
        int srow = -1;  // staging row t kY + slot
        if (rloc < b.rows) {
          if (b.kind == BU_DX_ROUTED) {
            const int j = p.prow_route[b.a_row + rloc];
            if (j >= 0) srow = (j / p.k) * p.kY + (j % p.k);
          } else {
            srow = (b.a_row + rloc) * p.kY + p.k;
          }
        }
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v[jj] = __uint_as_float(r[jj]);
          if (srow >= 0) ovf |= store_f16x32_sat(p.dxs + (size_t)srow * p.D + b.n * 256 + c, v);
        }
      } else {  // weight gradient tile: rows m*128 + rloc, columns n*256 ...
        bf16* out;
        int ld;
        switch (b.kind) {
          case BU_DW_DOWN: out = p.dW_down + (size_t)b.e * p.D * p.I; ld = p.I; break;
          case BU_DW_UP: out = p.dW_up + (size_t)b.e * p.I * p.D; ld = p.D; break;
          case BU_DW_GATE: out = p.dW_gate + (size_t)b.e * p.I * p.D; ld = p.D; break;
          case BU_DWS_DOWN: out = p.dWs_down; ld = p.I_s; break;
          case BU_DWS_UP: out = p.dWs_up; ld = p.D; break;
          default: out = p.dWs_gate; ld = p.D; break;
        }
        bf16* row = out + (size_t)(b.m * BM + rloc) * ld + b.n * 256;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          float v[32];
          if (b.nk1 > 0) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] = __uint_as_float(r[jj]);
          } else {  // an expert no route reached: its gradient is zero
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] = 0.0f;
          }
          store_bf16x32(row + c, v);
        }
      }
      // hand the accumulator back (pairs: one arrival per warp on the even CTA's barrier)
      tc_fence_before();
      if constexpr (kPair) {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_even + acc * 8u);
      } else {
        mbar_arrive(&tempty[acc]);
      }
      if (acc) ++uses1; else ++uses0;
    }
    if (__any_sync(0xffffffffu, ovf) && lane == 0) atomicOr(p.status + 1, FLAG_STAGING_OVERFLOW);
  }
  if constexpr (kPair) settle_after_abort(p.status);
  tc_fence_before();
  __syncthreads();
  // pairs: neither CTA frees TMEM or leaves while the other may still issue
  // into its TMEM, arrive on its barriers or load into its shared memory
  if constexpr (kPair) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ router
// One warp per token, lane = slot: dg_j (fixed-order sum of the per-128-column
// partials), c = sum_j g_j dg_j and (sigmoid) S = sum_j s_j by the same xor
// butterfly on every lane, then dl_j.
__device__ __forceinline__ float warp_sum_bfly(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256) bwd_router_dl(BwdParams p) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= p.T) return;
  const bool on = lane < p.k;
  const int j = t * p.k + lane;
  float dg = 0.0f, g = 0.0f, sv = 0.0f;
  if (on) {
    const int r = p.route_prow[j];
    for (int n = 0; n < p.N1; ++n) dg += p.dgp[(size_t)r * p.N1 + n];
    g = p.topk_w[j];
    if (p.score_fn == MOE_SCORE_SIGMOID) sv = 1.0f / (1.0f + expf(-p.topk_logit[j]));
  }
  const float c = warp_sum_bfly(on ? g * dg : 0.0f);
  float dl;
  if (p.score_fn == MOE_SCORE_SIGMOID) {
    const float S = warp_sum_bfly(sv);
    dl = (dg - c) / S * sv * (1.0f - sv);
  } else {
    dl = g * (dg - c);
  }
  if (on) p.dl[j] = dl;
}

// dW_r and db partial sums over chunks of WR_CHUNK consecutive routes of one
// expert (its padded rows, in schedule order); one CTA per chunk.
__global__ void __launch_bounds__(256) bwd_router_wr(BwdParams p) {
  __shared__ float s_dl[WR_CHUNK];
  __shared__ int s_e;
  const int c = blockIdx.x;
  if (c >= p.meta[BM_NWC]) return;
  if (threadIdx.x == 0) {
    int lo = 0, hi = p.E;  // last e with wc0[e] <= c
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.wc0[mid] <= c) lo = mid;
      else hi = mid;
    }
    s_e = lo;
  }
  __syncthreads();
  const int e = s_e;
  const int o0 = (c - p.wc0[e]) * WR_CHUNK;
  const int n = min(WR_CHUNK, p.M[e] - o0);
  const int r0 = p.Sp[e] + o0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s_dl[i] = p.dl[p.prow_route[r0 + i]];
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int i = 0; i < n; ++i) b += s_dl[i];
    p.wb_part[c] = b;
  }
  float* out = p.wr_part + (size_t)c * p.D;
  for (int v = threadIdx.x; v < p.D / 8; v += blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int i = 0; i < n; ++i) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.xg + (size_t)(r0 + i) * p.D) + v);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
      const float d = s_dl[i];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        acc[2 * q] = fmaf(d, f.x, acc[2 * q]);
        acc[2 * q + 1] = fmaf(d, f.y, acc[2 * q + 1]);
      }
    }
    float4* o4 = reinterpret_cast<float4*>(out + 8 * v);
    o4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// dW_r[e] and db[e]: the expert's chunk partials summed in chunk order.
__global__ void __launch_bounds__(256) bwd_router_fin(BwdParams p) {
  const int e = blockIdx.x;
  const int c0 = p.wc0[e], c1 = p.wc0[e + 1];
  for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
    float s = 0.0f;
    for (int c = c0; c < c1; ++c) s += p.wr_part[(size_t)c * p.D + d];
    p.dW_r[(size_t)e * p.D + d] = s;
  }
  if (threadIdx.x == 0 && p.db_r) {
    float b = 0.0f;
    for (int c = c0; c < c1; ++c) b += p.wb_part[c];
    p.db_r[e] = b;
  }
}

// dx_t = (shared expert's dx) + sum over slots of the routes' dx + sum over
// slots of dl_j W_r[e_j], in that order, fp32, one rounding to bf16.  One warp
// per token, 8 columns per lane and step.
__global__ void __launch_bounds__(256) bwd_dx_combine(BwdParams p) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= p.T) return;
  const bool sh = p.kY > p.k;
  float dl[TOPK_MAX];
  int ex[TOPK_MAX];
#pragma unroll
  for (int s = 0; s < TOPK_MAX; ++s) {
    dl[s] = s < p.k ? p.dl[(size_t)t * p.k + s] : 0.0f;
    ex[s] = s < p.k ? p.topk_idx[(size_t)t * p.k + s] : 0;
  }
  const __half* ys = p.dxs + (size_t)t * p.kY * p.D;
  for (int v = lane; v < p.D / 8; v += 32) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    auto add_f16 = [&](const __half* src) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + 8 * v);
      const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(h[q]);
        acc[2 * q] += f.x;
        acc[2 * q + 1] += f.y;
      }
    };
    if (sh) add_f16(ys + (size_t)p.k * p.D);
    for (int s = 0; s < p.k; ++s) add_f16(ys + (size_t)s * p.D);
    for (int s = 0; s < p.k; ++s) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.w_router + (size_t)ex[s] * p.D) + v);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        acc[2 * q] = fmaf(dl[s], f.x, acc[2 * q]);
        acc[2 * q + 1] = fmaf(dl[s], f.y, acc[2 * q + 1]);
      }
    }
    *reinterpret_cast<uint4*>(p.dx + (size_t)t * p.D + 8 * v) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

}  // namespace moe

// ------------------------------------------------------------------ host side
namespace {

using namespace moe;

size_t bwd_align(size_t v) { return (v + 255) & ~size_t(255); }

struct BwdLayout {
  size_t status, counters, meta, Sp, wc0, eorder, mtiles, prow_route, route_prow, xg, dOg, hg, dau, dag, dgp, hs,
      dasu, dasg, dxs, dl, wr_part, wb_part, total;
  int64_t Rp_max, n_mt_max, n_wc_max;
};

BwdLayout bwd_layout(const moe_config& c, int64_t T) {
  BwdLayout L{};
  const int64_t R = T * c.k;
  L.Rp_max = R + (int64_t)(PADK - 1) * c.E;
  L.n_mt_max = (L.Rp_max + BM - 1) / BM + c.E;
  L.n_wc_max = (R + WR_CHUNK - 1) / WR_CHUNK + c.E;
  const int64_t kY = c.k + (c.I_s > 0 ? 1 : 0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = bwd_align(off + bytes);
    return at;
  };
  L.status = take(STATUS_AREA_BYTES);  // at offset 0: moe_get_status reads it
  L.counters = take(2 * sizeof(int));
  L.meta = take(4 * sizeof(int));
  L.Sp = take(sizeof(int) * (c.E + 1));
  L.wc0 = take(sizeof(int) * (c.E + 1));
  L.eorder = take(sizeof(int) * c.E);
  L.mtiles = take(sizeof(int) * 4 * L.n_mt_max);
  L.prow_route = take(sizeof(int) * L.Rp_max);
  L.route_prow = take(sizeof(int) * R);
  L.xg = take((size_t)L.Rp_max * c.D * 2);
  L.dOg = take((size_t)L.Rp_max * c.D * 2);
  L.hg = take((size_t)L.Rp_max * c.I * 2);
  L.dau = take((size_t)L.Rp_max * c.I * 2);
  L.dag = take((size_t)L.Rp_max * c.I * 2);
  L.dgp = take((size_t)L.Rp_max * (c.I / BM) * 4);
  L.hs = take((size_t)T * c.I_s * 2);
  L.dasu = take((size_t)T * c.I_s * 2);
  L.dasg = take((size_t)T * c.I_s * 2);
  L.dxs = take((size_t)T * kY * c.D * 2);
  L.dl = take((size_t)R * 4);
  L.wr_part = take((size_t)L.n_wc_max * c.D * 4);
  L.wb_part = take((size_t)L.n_wc_max * 4);
  L.total = off;
  return L;
}

bool bwd_shape_ok(const moe_config& c) {
  return c.precision == MOE_PREC_BF16 && c.I % 256 == 0 && c.I_s % 256 == 0 && c.D % 256 == 0;
}

int encode_box64(const moe_plan* pl, CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                 uint32_t box_rows = 64) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = pl->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// 3-D view of a row-major bf16 [rows, cols] matrix for MN-major loads: (64
// columns, row, 64-column block), box {64, 64, 2}
int encode_mn3d(const moe_plan* pl, CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols) {
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = pl->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" size_t moe_bwd_workspace_bytes(const moe_plan* plan, int64_t T) {
  if (!plan || T < 1 || T > plan->cfg.T_max || !bwd_shape_ok(plan->cfg)) return 0;
  return bwd_layout(plan->cfg, T).total;
}

extern "C" int moe_bwd(const moe_plan* pl, int64_t T, const void* x, const moe_weights* w, const void* dO,
                       const void* fwd_workspace, const moe_grads* gr, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream_) {
  if (!pl || !w || !gr || T < 0 || T > pl->cfg.T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const moe_config& c = pl->cfg;
  if (!bwd_shape_ok(c)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const bool shared = w->Ws_up || w->Ws_gate || w->Ws_down;
  if (shared && (!w->Ws_up || !w->Ws_gate || !w->Ws_down || c.I_s == 0)) return MOE_ERR_INVALID_ARG;
  if (shared != (gr->dWs_up != nullptr) || (gr->dWs_up != nullptr) != (gr->dWs_gate != nullptr) ||
      (gr->dWs_up != nullptr) != (gr->dWs_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  const void* req[] = {x, dO, fwd_workspace, workspace, w->W_router, w->W_up, w->W_gate, w->W_down,
                       gr->dx, gr->dW_router, gr->dW_up, gr->dW_gate, gr->dW_down};
  for (const void* q : req)
    if (!q || !al16(q)) return MOE_ERR_INVALID_ARG;
  if (shared) {
    const void* sreq[] = {w->Ws_up, w->Ws_gate, w->Ws_down, gr->dWs_up, gr->dWs_gate, gr->dWs_down};
    for (const void* q : sreq)
      if (!al16(q)) return MOE_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const BwdLayout L = bwd_layout(c, T);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != pl->device) return MOE_ERR_INVALID_ARG;
  FwdRoutingViews fv;
  if (fwd_routing_views(pl, T, fwd_workspace, &fv) != MOE_OK) return MOE_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdParams p{};
  p.T = (int)T;
  p.D = (int)c.D;
  p.I = (int)c.I;
  p.E = (int)c.E;
  p.k = (int)c.k;
  p.I_s = shared ? (int)c.I_s : 0;
  p.kY = (int)c.k + (shared ? 1 : 0);
  p.score_fn = c.score_fn;
  p.N1 = p.I / BM;
  p.N1s = p.I_s / BM;
  p.N2 = p.D / 256;
  p.n_tt = (int)((T + BM - 1) / BM);
  p.n_mt_max = (int)L.n_mt_max;
  p.Rp_max = (int)L.Rp_max;
  p.n_wc_max = (int)L.n_wc_max;
  p.pair = c.mma_pair;  // the backward's GEMMs run as CTA pairs when the plan's forward does
  p.timeout_ns = (long long)c.timeout_ms * 1000000LL;
  p.topk_idx = fv.topk_idx;
  p.topk_w = fv.topk_w;
  p.topk_logit = fv.topk_logit;
  p.M = fv.M;
  p.S = fv.S;
  p.sched = fv.sched;
  p.x = static_cast<const bf16*>(x);
  p.dO = static_cast<const bf16*>(dO);
  p.w_router = static_cast<const bf16*>(w->W_router);
  p.status = reinterpret_cast<int*>(ws + L.status);
  p.counters = reinterpret_cast<int*>(ws + L.counters);
  p.meta = reinterpret_cast<int*>(ws + L.meta);
  p.Sp = reinterpret_cast<int*>(ws + L.Sp);
  p.wc0 = reinterpret_cast<int*>(ws + L.wc0);
  p.eorder = reinterpret_cast<int*>(ws + L.eorder);
  p.mtiles = reinterpret_cast<int*>(ws + L.mtiles);
  p.prow_route = reinterpret_cast<int*>(ws + L.prow_route);
  p.route_prow = reinterpret_cast<int*>(ws + L.route_prow);
  p.xg = reinterpret_cast<bf16*>(ws + L.xg);
  p.dOg = reinterpret_cast<bf16*>(ws + L.dOg);
  p.hg = reinterpret_cast<bf16*>(ws + L.hg);
  p.dau = reinterpret_cast<bf16*>(ws + L.dau);
  p.dag = reinterpret_cast<bf16*>(ws + L.dag);
  p.dgp = reinterpret_cast<float*>(ws + L.dgp);
  p.hs = reinterpret_cast<bf16*>(ws + L.hs);
  p.dasu = reinterpret_cast<bf16*>(ws + L.dasu);
  p.dasg = reinterpret_cast<bf16*>(ws + L.dasg);
  p.dxs = reinterpret_cast<__half*>(ws + L.dxs);
  p.dl = reinterpret_cast<float*>(ws + L.dl);
  p.wr_part = reinterpret_cast<float*>(ws + L.wr_part);
  p.wb_part = reinterpret_cast<float*>(ws + L.wb_part);
  p.dx = static_cast<bf16*>(gr->dx);
  p.dW_r = gr->dW_router;
  p.db_r = gr->db_router;
  p.dW_up = static_cast<bf16*>(gr->dW_up);
  p.dW_gate = static_cast<bf16*>(gr->dW_gate);
  p.dW_down = static_cast<bf16*>(gr->dW_down);
  p.dWs_up = static_cast<bf16*>(gr->dWs_up);
  p.dWs_gate = static_cast<bf16*>(gr->dWs_gate);
  p.dWs_down = static_cast<bf16*>(gr->dWs_down);

  BwdMaps mp;
  std::memset(&mp, 0, sizeof(mp));
  const uint64_t Rp = (uint64_t)L.Rp_max, E = c.E, D = c.D, I = c.I, Is = c.I_s;
  int rc = MOE_OK;
  rc |= encode_box64(pl, &mp.xg, p.xg, Rp, D);
  rc |= encode_box64(pl, &mp.dOg, p.dOg, Rp, D);
  rc |= encode_box64(pl, &mp.hg, p.hg, Rp, I);
  rc |= encode_box64(pl, &mp.dau, p.dau, Rp, I);
  rc |= encode_box64(pl, &mp.dag, p.dag, Rp, I);
  rc |= encode_box64(pl, &mp.w_up, w->W_up, E * I, D);
  rc |= encode_box64(pl, &mp.w_gate, w->W_gate, E * I, D);
  rc |= encode_box64(pl, &mp.w_down, w->W_down, E * D, I);
  rc |= encode_box64(pl, &mp.x, x, (uint64_t)T, D);
  rc |= encode_box64(pl, &mp.dO, dO, (uint64_t)T, D);
  rc |= encode_box64(pl, &mp.k_xg, p.xg, Rp, D, 128);
  rc |= encode_box64(pl, &mp.k_dOg, p.dOg, Rp, D, 128);
  rc |= encode_box64(pl, &mp.k_dau, p.dau, Rp, I, 128);
  rc |= encode_box64(pl, &mp.k_dag, p.dag, Rp, I, 128);
  rc |= encode_box64(pl, &mp.k_w_up, w->W_up, E * I, D, 128);
  rc |= encode_box64(pl, &mp.k_w_gate, w->W_gate, E * I, D, 128);
  rc |= encode_box64(pl, &mp.k_x, x, (uint64_t)T, D, 128);
  rc |= encode_box64(pl, &mp.k_dO, dO, (uint64_t)T, D, 128);
  if (shared) {
    rc |= encode_box64(pl, &mp.hs, p.hs, (uint64_t)T, Is);
    rc |= encode_box64(pl, &mp.dasu, p.dasu, (uint64_t)T, Is);
    rc |= encode_box64(pl, &mp.dasg, p.dasg, (uint64_t)T, Is);
    rc |= encode_box64(pl, &mp.ws_up, w->Ws_up, Is, D);
    rc |= encode_box64(pl, &mp.ws_gate, w->Ws_gate, Is, D);
    rc |= encode_box64(pl, &mp.ws_down, w->Ws_down, D, Is);
    rc |= encode_box64(pl, &mp.k_dasu, p.dasu, (uint64_t)T, Is, 128);
    rc |= encode_box64(pl, &mp.k_dasg, p.dasg, (uint64_t)T, Is, 128);
    rc |= encode_box64(pl, &mp.k_ws_up, w->Ws_up, Is, D, 128);
    rc |= encode_box64(pl, &mp.k_ws_gate, w->Ws_gate, Is, D, 128);
  }
  if (rc != MOE_OK) return MOE_ERR_INVALID_ARG;
  // the MN-major 3-D views (without them every MN-major tile is two 2-D loads)
  int rc3 = MOE_OK;
  rc3 |= encode_mn3d(pl, &mp.m_xg, p.xg, Rp, D);
  rc3 |= encode_mn3d(pl, &mp.m_dOg, p.dOg, Rp, D);
  rc3 |= encode_mn3d(pl, &mp.m_hg, p.hg, Rp, I);
  rc3 |= encode_mn3d(pl, &mp.m_dau, p.dau, Rp, I);
  rc3 |= encode_mn3d(pl, &mp.m_dag, p.dag, Rp, I);
  rc3 |= encode_mn3d(pl, &mp.m_w_up, w->W_up, E * I, D);
  rc3 |= encode_mn3d(pl, &mp.m_w_gate, w->W_gate, E * I, D);
  rc3 |= encode_mn3d(pl, &mp.m_w_down, w->W_down, E * D, I);
  rc3 |= encode_mn3d(pl, &mp.m_x, x, (uint64_t)T, D);
  rc3 |= encode_mn3d(pl, &mp.m_dO, dO, (uint64_t)T, D);
  if (shared) {
    rc3 |= encode_mn3d(pl, &mp.m_hs, p.hs, (uint64_t)T, Is);
    rc3 |= encode_mn3d(pl, &mp.m_dasu, p.dasu, (uint64_t)T, Is);
    rc3 |= encode_mn3d(pl, &mp.m_dasg, p.dasg, (uint64_t)T, Is);
    rc3 |= encode_mn3d(pl, &mp.m_ws_up, w->Ws_up, Is, D);
    rc3 |= encode_mn3d(pl, &mp.m_ws_gate, w->Ws_gate, Is, D);
    rc3 |= encode_mn3d(pl, &mp.m_ws_down, w->Ws_down, D, Is);
  }
  p.mn3d = rc3 == MOE_OK ? 1 : 0;

  cudaStream_t st = (cudaStream_t)stream_;
  const int sms = pl->num_sms;
  const bool pair = p.pair != 0;
  const void* g0 = pair ? reinterpret_cast<const void*>(bwd_gemm<0, true>) : reinterpret_cast<const void*>(bwd_gemm<0, false>);
  const void* g1 = pair ? reinterpret_cast<const void*>(bwd_gemm<1, true>) : reinterpret_cast<const void*>(bwd_gemm<1, false>);
  const int gsmem = pair ? BWD_PAIR_SMEM : BWD_SMEM;
  if (cudaFuncSetAttribute(g0, cudaFuncAttributeMaxDynamicSharedMemorySize, gsmem) != cudaSuccess ||
      cudaFuncSetAttribute(g1, cudaFuncAttributeMaxDynamicSharedMemorySize, gsmem) != cudaSuccess)
    return MOE_ERR_CUDA;
  // one CTA per SM; pairs: clusters of 2 (the even CTA of each issues the pair's MMAs)
  cudaLaunchConfig_t gcfg = {};
  gcfg.gridDim = dim3((unsigned)(pair ? (sms & ~1) : sms));
  gcfg.blockDim = dim3(BWD_THREADS);
  gcfg.dynamicSmemBytes = gsmem;
  gcfg.stream = st;
  cudaLaunchAttribute gattr[1];
  gattr[0].id = cudaLaunchAttributeClusterDimension;
  gattr[0].val.clusterDim.x = 2;
  gattr[0].val.clusterDim.y = 1;
  gattr[0].val.clusterDim.z = 1;
  gcfg.attrs = gattr;
  gcfg.numAttrs = pair ? 1 : 0;
  auto gemm = [&](int phase) {
    if (pair) return phase ? cudaLaunchKernelEx(&gcfg, bwd_gemm<1, true>, mp, p) : cudaLaunchKernelEx(&gcfg, bwd_gemm<0, true>, mp, p);
    return phase ? cudaLaunchKernelEx(&gcfg, bwd_gemm<1, false>, mp, p) : cudaLaunchKernelEx(&gcfg, bwd_gemm<0, false>, mp, p);
  };
  const int tok_blocks = (int)((T + 7) / 8);  // 8 warps per block, one token per warp
  auto mark = [&](int i) { return !pl->bwd_timed || cudaEventRecord(pl->bwd_timing[i], st) == cudaSuccess; };
  bool ok = mark(0);
  bwd_prep<<<1, 512, 0, st>>>(p);
  bwd_gather<<<4 * sms, 256, 0, st>>>(p);
  ok = ok && mark(1);
  ok = ok && gemm(0) == cudaSuccess;
  ok = ok && mark(2);
  bwd_router_dl<<<tok_blocks, 256, 0, st>>>(p);
  ok = ok && gemm(1) == cudaSuccess;
  ok = ok && mark(3);
  bwd_router_wr<<<(unsigned)L.n_wc_max, 256, 0, st>>>(p);
  bwd_router_fin<<<(unsigned)c.E, 256, 0, st>>>(p);
  bwd_dx_combine<<<tok_blocks, 256, 0, st>>>(p);
  ok = ok && mark(4);
  return ok && cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
