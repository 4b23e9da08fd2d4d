// MXFP8 weight quantiser ("Mixture-of-Kittens: MoE Megakernel for NVL72s",
// Sec. 3.4 "MXFP8 Support": weights are quantised ahead of time).
// Format: OCP Microscaling (MX) v1.0, MXFP8 E4M3, one E8M0 scale per 32
// consecutive elements along K:  X = 2^(floor(log2 amax) - 8)  (8 = exponent of
// E4M3's largest normal, 448), q = E4M3_rne_satfinite(v / X); amax = 0 -> X = 2^-127.
// Scale layout (what the block-scaled MMA loads with tcgen05.cp): 512-byte
// blocks, one per 128 rows x 128 K-elements, ordered [rows/128][K/128]; inside
// a block the scale of row r (mod 128) and 32-wide K block kb (mod 4) is at
// byte (r % 32) * 16 + (r / 32) * 4 + kb.  rows and K are multiples of 128.
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

__global__ void mx_quantize_kernel(const bf16* __restrict__ W, int64_t rows, int64_t K, uint8_t* __restrict__ q,
                                   uint8_t* __restrict__ scales) {
  const int64_t nb = K / 32;
  const int64_t total = rows * nb;
  for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < total;
       blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = blk / nb, b = blk % nb;
    const uint4* src = reinterpret_cast<const uint4*>(W + r * K + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = src[i];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        v[8 * i + 2 * j] = f.x;
        v[8 * i + 2 * j + 1] = f.y;
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    uint8_t code = 0;
    uint32_t packed[8];
    if (amax == 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) packed[i] = 0;
    } else {
      int se = ilogbf(amax) - 8;
      se = max(-127, min(127, se));
      code = (uint8_t)(se + 127);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float s = ldexpf(v[4 * i + j], -se);
          const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
          word |= (uint32_t)c << (8 * j);
        }
        packed[i] = word;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(q + r * K + b * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    const int64_t sblk = (r / 128) * (K / 128) + b / 4;
    scales[sblk * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (b % 4)] = code;
  }
}

size_t mx_scale_bytes(int64_t rows, int64_t K) { return (size_t)(rows * (K / 32)); }

cudaError_t launch_mx_quantize(const bf16* W, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, cudaStream_t st) {
  const int64_t total = rows * (K / 32);
  int64_t grid = (total + 255) / 256;
  if (grid > 152 * 16) grid = 152 * 16;
  mx_quantize_kernel<<<(unsigned)grid, 256, 0, st>>>(W, rows, K, q, s);
  return cudaGetLastError();
}

}  // namespace moe
