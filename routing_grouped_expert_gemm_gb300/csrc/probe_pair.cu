// Test hook: one tcgen05.mma.cta_group::2 tile on a CTA pair, used by the GPU
// tests to pin the pair encodings (TMEM allocation for two CTAs, TMA loads
// counted on the even CTA's mbarrier, M = 256 instruction descriptor, the
// split of A and B over the two shared memories, the multicast commit and the
// rows of D each CTA's TMEM receives) against a CPU reference.  Not part of
// the forward path.
//
// m = 256: D [256, 256] fp32 = A [256, 64] B [256, 64]^T, A and B bf16
// row-major (K contiguous).  CTA r of the pair loads A rows [128 r, 128 r +
// 128) and B rows [128 r, 128 r + 128); the even CTA issues four M = 256,
// N = 256, K = 16 MMAs.  m = 128: A [128, 64], CTA r loads A rows [64 r, 64 r
// + 64) (and the same B halves); the MMAs are M = 128.  Either way CTA r then
// writes all 128 TMEM lanes x 256 columns it holds to D_raw [2][128][256]
// (lanes the MMA did not write hold whatever was there).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

namespace {

constexpr uint64_t kProbeWaitNs = 2000000000ull;  // 2 s per wait

template <bool kCluster>
__device__ bool probe_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kProbeWaitNs) return false;
  }
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_probe_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB, float* D,
                      int* status, int m, int reps, unsigned long long* ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;          // 128 (m = 256) or 64 (m = 128) rows x 128 B (64 bf16), 128-byte swizzle
  uint8_t* sB = smem + 16384;  // 128 rows x 128 B
  __shared__ __align__(8) uint64_t full;
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    mbar_init(&full, 1);
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc_pair<256>(&tmem_slot);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (threadIdx.x == 0) {
    const uint32_t full_even = mapa_shared(&full, rank & ~1u);
    const uint32_t a_bytes = m == 256 ? 16384u : 8192u;
    if ((rank & 1u) == 0) mbar_arrive_expect_tx(&full, 2u * (a_bytes + 16384u));  // both CTAs' A and B halves
    tma_load_2d_pair(sA, &mA, full_even, 0, (int)((m / 2) * rank));
    tma_load_2d_pair(sB, &mB, full_even, 0, (int)(128 * rank));
    if ((rank & 1u) == 0) {
      if (probe_wait<true>(&full, 0)) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32((uint32_t)m, 256);
        const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
        const uint64_t t0 = globaltimer_ns();
        // reps > 1: the same four MMAs again, accumulating (timing only)
        for (int rep = 0; rep < reps; ++rep)
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_pair(tmem, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                          (rep | kk) > 0 ? 1u : 0u);
        mma_commit_pair(&done, 0x3);
        if (ns) {
          probe_wait<true>(&done, 0);
          *ns = globaltimer_ns() - t0;
        }
      } else {
        atomicExch(status, 1);
      }
    }
  }
  __syncwarp();
  const bool ok = probe_wait<true>(&done, 0);
  tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < 256; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + lane_base + c, r);
      tmem_ld_wait();
      for (int j = 0; j < 32; ++j) D[((size_t)rank * 128 + row) * 256 + c + j] = __uint_as_float(r[j]);
    }
  } else if (lane == 0) {
    atomicExch(status + 1 + rank, 1);
  }
  tc_fence_before();
  cluster_sync_all();  // no CTA frees TMEM or leaves while the other may still touch it
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 256);
  }
}

// Block-scaled MXFP8 pair tile: D [256, 256] = sum_kb A_kb B_kb^T sa(row, kb) sb(col, kb),
// A and B [256, 128] E4M3 codes; CTA r loads A rows [128 r, +128) and B rows [128 r, +128)
// with TMA (counted on the even CTA's barrier) and copies scale blocks from sf (four
// 512-byte blocks: A rows 0-127, A rows 128-255, B rows 0-127, B rows 128-255) into its
// shared memory.  mode 0: CTA r's TMEM gets (tcgen05.cp.cta_group::2) its A block at
// column 256 and its own B half's block at 260.  mode 1: its A block at 256 and both B
// blocks at 260 and 264.  The MMA reads A scales at 256, B scales at 260.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_mx_probe_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                         const uint8_t* __restrict__ sf, float* D, int* status, int mode) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;           // 128 rows x 128 B E4M3, 128-byte swizzle
  uint8_t* sB = smem + 16384;   // 128 rows x 128 B
  uint8_t* sSF = smem + 32768;  // A block, then one or two B blocks
  __shared__ __align__(8) uint64_t full;
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  // scale blocks into shared memory (generic stores, then made visible to the async proxy)
  for (int i = threadIdx.x; i < 512 / 16; i += blockDim.x) {
    reinterpret_cast<uint4*>(sSF)[i] = reinterpret_cast<const uint4*>(sf + rank * 512)[i];
    if (mode == 0) {
      reinterpret_cast<uint4*>(sSF + 512)[i] = reinterpret_cast<const uint4*>(sf + (2 + rank) * 512)[i];
    } else {
      reinterpret_cast<uint4*>(sSF + 512)[i] = reinterpret_cast<const uint4*>(sf + 2 * 512)[i];
      reinterpret_cast<uint4*>(sSF + 1024)[i] = reinterpret_cast<const uint4*>(sf + 3 * 512)[i];
    }
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&full, 1);
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc_pair<512>(&tmem_slot);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers, scale blocks and TMEM ready
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (threadIdx.x == 0) {
    const uint32_t full_even = mapa_shared(&full, rank & ~1u);
    if ((rank & 1u) == 0) mbar_arrive_expect_tx(&full, 2u * 32768u);
    tma_load_2d_pair(sA, &mA, full_even, 0, (int)(128 * rank));
    tma_load_2d_pair(sB, &mB, full_even, 0, (int)(128 * rank));
    if ((rank & 1u) == 0) {
      if (probe_wait<true>(&full, 0)) {
        tc_fence_after();
        const uint32_t sf_addr = smem_u32(sSF);
        tmem_cp_32x128b_warpx4_pair(tmem + 256, sdesc_sf_block(sf_addr));
        tmem_cp_32x128b_warpx4_pair(tmem + 260, sdesc_sf_block(sf_addr + 512));
        if (mode == 1) tmem_cp_32x128b_warpx4_pair(tmem + 264, sdesc_sf_block(sf_addr + 1024));
        const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
        for (int kb = 0; kb < 4; ++kb)
          mma_mxf8_pair(tmem, sdesc_kmajor_sw128(a_addr + kb * 32), sdesc_kmajor_sw128(b_addr + kb * 32),
                        idesc_mxf8_e4m3(256, 256) | ((uint32_t)kb << 4) | ((uint32_t)kb << 29), tmem + 256,
                        tmem + 260, kb > 0 ? 1u : 0u);
        mma_commit_pair(&done, 0x3);
      } else {
        atomicExch(status, 1);
      }
    }
  }
  __syncwarp();
  const bool ok = probe_wait<true>(&done, 0);
  tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < 256; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + lane_base + c, r);
      tmem_ld_wait();
      for (int j = 0; j < 32; ++j) D[((size_t)rank * 128 + row) * 256 + c + j] = __uint_as_float(r[j]);
    }
  } else if (lane == 0) {
    atomicExch(status + 1 + rank, 1);
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace moe

namespace {

typedef CUresult (*probe_encode_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode_probe_map(probe_encode_fn enc, CUtensorMap* m, const void* ptr, uint32_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -1;
}

}  // namespace

namespace moe {
int launch_pair_probe(const void* A, const void* B, float* D, int* status, int m, int reps, unsigned long long* ns,
                      void* stream);
}

extern "C" int moe_testing_pair_tile(const void* A, const void* B, float* D, int* status, int m, void* stream) {
  return moe::launch_pair_probe(A, B, D, status, m, 1, nullptr, stream);
}

int moe::launch_pair_probe(const void* A, const void* B, float* D, int* status, int m, int reps,
                           unsigned long long* ns, void* stream) {
  if (!A || !B || !D || !status || (m != 128 && m != 256) || reps < 1) return -1;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) return -1;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return -4;
  CUtensorMap mA, mB;
  if (encode_probe_map(reinterpret_cast<probe_encode_fn>(fn), &mA, A, (uint32_t)m, (uint32_t)m / 2) ||
      encode_probe_map(reinterpret_cast<probe_encode_fn>(fn), &mB, B, 256, 128))
    return -1;
  const int smem = 32 * 1024 + 1024;
  if (cudaFuncSetAttribute(moe::pair_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -4;
  moe::pair_probe_kernel<<<2, 128, smem, (cudaStream_t)stream>>>(mA, mB, D, status, m, reps, ns);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Time `reps` x 4 back-to-back pair MMAs (M = m, N = 256, K = 16) on one CTA pair: *ns (device
// memory) receives the even CTA's %globaltimer span from the first issue to the completion.
extern "C" int moe_testing_pair_mma_time(const void* A, const void* B, float* D, int* status, int m, int reps,
                                         unsigned long long* ns, void* stream) {
  if (!ns) return -1;
  return moe::launch_pair_probe(A, B, D, status, m, reps, ns, stream);
}

// One block-scaled MXFP8 cta_group::2 tile (see pair_mx_probe_kernel); A, B [256, 128] E4M3
// codes, sf four 512-byte scale blocks, D [256, 256] fp32; all device pointers.
extern "C" int moe_testing_pair_mx_tile(const void* A, const void* B, const void* sf, float* D, int* status, int mode,
                                        void* stream) {
  if (!A || !B || !sf || !D || !status || mode < 0 || mode > 1) return -1;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(sf)) & 15u)
    return -1;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return -4;
  auto enc = reinterpret_cast<probe_encode_fn>(fn);
  CUtensorMap mA, mB;
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[2] = {128, 256};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    if (enc(i ? &mB : &mA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(i ? B : A), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return -1;
  }
  const int smem = 32 * 1024 + 1536 + 1024;
  if (cudaFuncSetAttribute(moe::pair_mx_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -4;
  moe::pair_mx_probe_kernel<<<2, 128, smem, (cudaStream_t)stream>>>(mA, mB, static_cast<const uint8_t*>(sf), D,
                                                                    status, mode);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
