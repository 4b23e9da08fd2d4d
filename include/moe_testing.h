/*
 * moe_testing.h -- test hooks of the MoE library (not part of the forward
 * path).  They exist so that the GPU tests can pin hardware encodings against
 * a CPU reference.
 */
#ifndef MOE_GB300_TESTING_H
#define MOE_GB300_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One block-scaled MXFP8 (E4M3 x E4M3, E8M0 scales per 32 K-elements)
 * tcgen05 MMA tile on one CTA:
 *   D [128, 256] fp32 = sum_{kb<4} A[:, 32kb:32kb+32] B[:, 32kb:32kb+32]^T * sa(row, kb) * sb(col, kb)
 * A [128, 128] and B [256, 128] E4M3 codes, row-major.  mode 0: sf_img
 * [128][12] uint32 copied verbatim into TMEM lanes 0..127, columns 256..267
 * (tcgen05.st); mode 1: sf_img = three 512-byte scale blocks (A; B rows 0-127;
 * B rows 128-255) copied with tcgen05.cp.32x128b.warpx4 to columns 256, 260,
 * 264.  A scales are read from column 256, B scales from column 260,
 * scale-factor id = kb.  All pointers are device pointers; asynchronous on
 * `stream` (a cudaStream_t).  Returns 0, -1 (bad argument) or -4 (CUDA error).
 */
int moe_testing_mx_tile(const void* A, const void* B, const void* sf_img, float* D, int mode, void* stream);

#ifdef __cplusplus
}
#endif

#endif
