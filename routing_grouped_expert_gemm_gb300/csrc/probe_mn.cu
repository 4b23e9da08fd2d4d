// Test hook: one bf16 tcgen05 MMA tile whose operands may be staged MN-major
// (the M or N index contiguous in shared memory) instead of K-major.  The
// backward pass contracts over tokens and over the output dimension of the
// forward's weights, so several of its operands arrive MN-major; this probe
// pins that encoding against a CPU reference.  Not part of any product path.
//
// D[128, N] (fp32) = A[128, 64] B[N, 64]^T, A and B given row-major (K
// contiguous) in global memory; N = 128 or 256.  The kernel stages each operand
// in shared memory the way a TMA load with 128-byte swizzling leaves it:
//   K-major: row r (M or N index) is 128 bytes at r * 128, its 16-byte chunk c
//            at chunk c ^ (r % 8);
//   MN-major: 64-wide MN blocks, block q at q * 8192 holding 64 K rows of
//            128 bytes (64 MN elements), K row k at k * 128, its chunk c at
//            chunk c ^ (k % 8) -- what a {64 MN, 64 K} box of the transposed
//            matrix looks like.
// The descriptor of an MN-major operand takes lbo and sbo from the caller:
// (8192, 1024) reads the leading offset as the step between 64-wide MN blocks
// and the stride offset as the step between 8-row K groups; (1024, 8192) the
// other way round.  A test pins which reading the hardware takes.
#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint64_t sdesc_sw128_lbo_sbo(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// stage rows x 64 bf16 (row-major, K contiguous) at dst, K-major or MN-major
__device__ void probe_stage(uint8_t* dst, const uint16_t* src, int rows, bool mn) {
  for (int i = threadIdx.x; i < rows * 64; i += blockDim.x) {
    const int r = i / 64, k = i % 64;
    uint32_t off;
    if (!mn) {
      const int c = k / 8;
      off = r * 128 + ((c ^ (r & 7)) << 4) + (k % 8) * 2;
    } else {
      const int q = r / 64, rr = r % 64, c = rr / 8;
      off = q * 8192 + k * 128 + ((c ^ (k & 7)) << 4) + (rr % 8) * 2;
    }
    *reinterpret_cast<uint16_t*>(dst + off) = src[i];
  }
}

__global__ void __launch_bounds__(128, 1)
    mn_probe_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, float* __restrict__ D, int N,
                    int a_mn, int b_mn, uint32_t lbo, uint32_t sbo) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;          // 16 KB
  uint8_t* sB = smem + 16384;  // up to 32 KB
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  probe_stage(sA, A, 128, a_mn != 0);
  probe_stage(sB, B, N, b_mn != 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc<256>(&tmem_slot);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
    for (int kk = 0; kk < 4; ++kk) {  // four K = 16 steps
      const uint32_t a = smem_u32(sA) + (a_mn ? kk * 2048 : kk * 32);
      const uint32_t b = smem_u32(sB) + (b_mn ? kk * 2048 : kk * 32);
      const uint64_t ad = a_mn ? sdesc_sw128_lbo_sbo(a, lbo, sbo) : sdesc_kmajor_sw128(a);
      const uint64_t bd = b_mn ? sdesc_sw128_lbo_sbo(b, lbo, sbo) : sdesc_kmajor_sw128(b);
      mma_bf16_ss(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
    mma_commit(&bar);
  }
  __syncwarp();
  const uint64_t t0 = globaltimer_ns();  // one bounded wait (2 s) on the commit
  bool done = false;
  while (!(done = mbar_try_wait(&bar, 0)) && globaltimer_ns() - t0 < 2000000000ull) {
  }
  tc_fence_after();
  const int row = warp * 32 + lane;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (done) {
    for (int c = 0; c < N; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + lane_base + c, r);
      tmem_ld_wait();
      for (int j = 0; j < 32; ++j) D[row * N + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace moe

extern "C" int moe_testing_mn_tile(const void* A, const void* B, float* D, int N, int a_mn, int b_mn, int lbo,
                                   int sbo, void* stream) {
  // the two readings of the offsets; either keeps every read inside the staging
  // (the allocation has 16 KB to spare past B)
  const bool pair_ok = (lbo == 8192 && sbo == 1024) || (lbo == 1024 && sbo == 8192);
  if (!A || !B || !D || (N != 128 && N != 256) || !pair_ok) return -1;
  const int smem = 16384 + 32768 + 16384 + 1024;
  if (cudaFuncSetAttribute(moe::mn_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -4;
  moe::mn_probe_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(static_cast<const uint16_t*>(A),
                                                              static_cast<const uint16_t*>(B), D, N, a_mn, b_mn,
                                                              (uint32_t)lbo, (uint32_t)sbo);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
