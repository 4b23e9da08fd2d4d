// Test hook: one block-scaled MXFP8 tcgen05 MMA tile, used by the GPU tests to
// pin the instruction descriptor and the scale-factor placement in TMEM
// against a CPU reference.  Not part of the forward path.
//
// D[128, 256] (fp32) = sum over four 32-wide K blocks kb of
//   (A[:, 32kb : 32kb+32] B[:, 32kb : 32kb+32]^T) * scale_a(row, kb) * scale_b(col, kb)
// A [128, 128] and B [256, 128] are E4M3 codes, row-major (K contiguous).
// mode 0: sf_img [128 lanes][12 columns] (uint32) is written verbatim to TMEM
// columns 256..267 with tcgen05.st.  mode 1: sf_img holds three 512-byte scale
// blocks (A, B rows 0-127, B rows 128-255) copied to columns 256, 260, 264 with
// tcgen05.cp.  The MMA reads A scales from column 256 and B scales from column
// 260, with scale-factor id kb for the kb-th MMA.
#include "common.cuh"

namespace moe {

__global__ void __launch_bounds__(128, 1)
    mx_probe_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B, const uint32_t* __restrict__ sf_img,
                    float* __restrict__ D, int mode) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;          // 128 rows x 128 B
  uint8_t* sB = smem + 16384;  // 256 rows x 128 B
  uint8_t* sSF = smem + 49152;  // mode 1: A scale block (512 B), then two B blocks
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // K-major, 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int r = i >> 3, ch = i & 7;
    *reinterpret_cast<uint4*>(sA + r * 128 + ((ch ^ (r & 7)) << 4)) = reinterpret_cast<const uint4*>(A)[i];
  }
  for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) {
    const int r = i >> 3, ch = i & 7;
    *reinterpret_cast<uint4*>(sB + r * 128 + ((ch ^ (r & 7)) << 4)) = reinterpret_cast<const uint4*>(B)[i];
  }
  if (mode == 1)
    for (int i = threadIdx.x; i < 1536 / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(sSF)[i] = reinterpret_cast<const uint4*>(sf_img)[i];
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc<512>(&tmem_slot);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int row = warp * 32 + lane;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t* img = sf_img + row * 12;
  if (mode == 0) {
    for (int c = 0; c < 12; c += 4)
      tmem_st_32x32b_x4(tmem + lane_base + 256 + c, img[c], img[c + 1], img[c + 2], img[c + 3]);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
    if (mode == 1) {  // scales through the async copy path, in order with the MMAs below
      const uint32_t sf = smem_u32(sSF);
      tmem_cp_32x128b_warpx4(tmem + 256, sdesc_sf_block(sf));
      tmem_cp_32x128b_warpx4(tmem + 260, sdesc_sf_block(sf + 512));
      tmem_cp_32x128b_warpx4(tmem + 264, sdesc_sf_block(sf + 1024));
    }
    for (int kb = 0; kb < 4; ++kb) {
      const uint32_t idesc = idesc_mxf8_e4m3(128, 256) | ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
      mma_mxf8_ss(tmem, sdesc_kmajor_sw128(a_addr + kb * 32), sdesc_kmajor_sw128(b_addr + kb * 32), idesc,
                  tmem + 256, tmem + 260, kb > 0 ? 1u : 0u);
    }
    mma_commit(&bar);
  }
  __syncwarp();
  // one bounded wait (2 s) on the commit
  const uint64_t t0 = globaltimer_ns();
  bool done = false;
  while (!(done = mbar_try_wait(&bar, 0)) && globaltimer_ns() - t0 < 2000000000ull) {
  }
  tc_fence_after();
  if (done) {
    for (int c = 0; c < 256; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + lane_base + c, r);
      tmem_ld_wait();
      for (int j = 0; j < 32; ++j) D[row * 256 + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace moe

extern "C" int moe_testing_mx_tile(const void* A, const void* B, const void* sf_img, float* D, int mode,
                                   void* stream) {
  if (!A || !B || !sf_img || !D || mode < 0 || mode > 1) return -1;
  const int smem = 48 * 1024 + 1536 + 1024;
  if (cudaFuncSetAttribute(moe::mx_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -4;
  moe::mx_probe_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(static_cast<const uint8_t*>(A),
                                                              static_cast<const uint8_t*>(B),
                                                              static_cast<const uint32_t*>(sf_img), D, mode);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
