// Test hook: one TMA load through a 3-D view of a row-major bf16 matrix
// [rows, cols] whose dimensions are (64 columns, row, 64-column block): the
// block dimension has a stride of 128 bytes, smaller than the row stride.  A
// {64, 64, 2} box then brings two adjacent 64-column blocks of 64 rows into
// shared memory as two 8 KB tiles with 128-byte swizzling -- the layout of an
// MN-major operand of 128 MN elements -- in one instruction.  The test pins
// that the encoder accepts the view and what lands where.  Not part of any
// product path.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

__global__ void __launch_bounds__(128, 1)
    tma3d_probe_kernel(const __grid_constant__ CUtensorMap m3, uint8_t* out, int* status, int r0, int b0) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, 16384u);
    tma_load_3d(smem, &m3, &bar, 0, r0, b0);
    const uint64_t t0 = globaltimer_ns();
    bool ok = false;
    while (!(ok = mbar_try_wait(&bar, 0)) && globaltimer_ns() - t0 < 200000000ull) {
    }
    *status = ok ? 1 : 2;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16384 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(smem)[i];
}

}  // namespace moe

// src: device bf16 [rows, cols] row-major (cols a multiple of 128, rows >= 64,
// 16-byte aligned); loads rows [r0, r0 + 64) of column blocks b0 and b0 + 1
// into out (device, 16384 bytes) as laid out in shared memory; status (device
// int): 1 loaded, 2 the wait ran out (200 ms).  Returns 0, -1 (bad argument),
// -4 (CUDA error) or -5 (the encoder rejected the 3-D view).
extern "C" int moe_testing_tma3d_load(const void* src, int rows, int cols, int r0, int b0, void* out, int* status,
                                      void* stream) {
  if (!src || !out || !status || rows < 64 || cols < 128 || cols % 128 || r0 < 0 || r0 + 64 > rows || b0 < 0 ||
      64 * (b0 + 2) > cols || (reinterpret_cast<uintptr_t>(src) & 15u))
    return -1;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return -4;
  typedef CUresult (*enc_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  CUtensorMap m3;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)cols / 64};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  if (reinterpret_cast<enc_fn>(fn)(&m3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(src), dims, strides, box,
                                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -5;
  const int smem = 16384 + 1024;
  if (cudaFuncSetAttribute(moe::tma3d_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -4;
  moe::tma3d_probe_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(m3, static_cast<uint8_t*>(out), status, r0, b0);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
