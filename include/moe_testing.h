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

/*
 * One bf16 tcgen05.mma.cta_group::2 tile on a pair of CTAs (a cluster of 2).
 *   m = 256: D = A [256, 64] B [256, 64]^T; CTA r loads A rows [128r, 128r+128)
 *   m = 128: D = A [128, 64] B [256, 64]^T; CTA r loads A rows [64r, 64r+64)
 * and B rows [128r, 128r+128), with TMA into its own shared memory, both
 * CTAs' loads counted on the even CTA's mbarrier; the even CTA issues four
 * M=m N=256 K=16 MMAs and commits to a barrier in both CTAs; CTA r then copies
 * all 128 lanes x 256 columns of its TMEM to D [2][128][256] fp32 (lanes the
 * MMA did not write hold unspecified values).  A and B bf16 row-major (K
 * contiguous), device pointers, 16-byte aligned.  status (device, int[3],
 * zeroed by the caller): [0] set if the even CTA's wait for the loads ran out
 * (2 s), [1 + r] if CTA r's wait for the MMA did.  Asynchronous on `stream`.
 * Returns 0, -1 (bad argument) or -4 (CUDA error).
 */
int moe_testing_pair_tile(const void* A, const void* B, float* D, int* status, int m, void* stream);

/*
 * The same tile, with the four MMAs issued `reps` times back to back
 * (accumulating) and the even CTA's %globaltimer span from the first issue to
 * their completion written to *ns (device memory): the pair MMA's issue rate
 * for M = m.  Returns 0, -1 or -4 as above.
 */
int moe_testing_pair_mma_time(const void* A, const void* B, float* D, int* status, int m, int reps,
                              unsigned long long* ns, void* stream);

/*
 * One block-scaled MXFP8 tcgen05.mma.cta_group::2 tile (E4M3 x E4M3, E8M0
 * scales per 32 K-elements) on a CTA pair:
 *   D [256, 256] fp32 = sum_{kb<4} A[:, 32kb:+32] B[:, 32kb:+32]^T * sa(row, kb) * sb(col, kb)
 * A, B [256, 128] E4M3 codes row-major; sf = four 512-byte scale blocks (A
 * rows 0-127, A rows 128-255, B rows 0-127, B rows 128-255) in the layout of
 * moe_testing_mx_tile.  CTA r loads A and B rows [128r, 128r+128) and copies
 * (tcgen05.cp.cta_group::2) its A block to TMEM column 256 and, mode 0, its
 * own B half's block to column 260, or, mode 1, both B blocks to 260 and 264;
 * the MMA reads A scales at 256 and B scales at 260.  D and status as for
 * moe_testing_pair_tile.  Returns 0, -1 (bad argument) or -4 (CUDA error).
 */
int moe_testing_pair_mx_tile(const void* A, const void* B, const void* sf, float* D, int* status, int mode,
                             void* stream);

/*
 * One bf16 tcgen05 MMA tile with operands staged K-major or MN-major:
 *   D [128, N] fp32 = A [128, 64] B [N, 64]^T,  N = 128 or 256,
 * A and B row-major bf16 (K contiguous) in device memory.  a_mn / b_mn = 1
 * stage that operand MN-major in shared memory (64-wide MN blocks of 64 K rows
 * x 128 B, 128-byte swizzle, 8192 B apart) and set its major bit in the
 * instruction descriptor; its matrix descriptor gets leading byte offset lbo
 * and stride byte offset sbo, (lbo, sbo) = (8192, 1024) or (1024, 8192).
 * Asynchronous on `stream`.  Returns 0, -1 (bad argument) or -4 (CUDA error).
 */
int moe_testing_mn_tile(const void* A, const void* B, float* D, int N, int a_mn, int b_mn, int lbo, int sbo,
                        void* stream);

/*
 * One TMA load through a 3-D view (64 columns, row, 64-column block; the
 * block stride 128 bytes, below the row stride) of src, a device bf16
 * [rows, cols] row-major matrix (cols a multiple of 128): box {64, 64, 2} at
 * rows [r0, r0 + 64), column blocks b0 and b0 + 1, 128-byte swizzle, copied
 * from shared memory to out (device, 16384 bytes) as it landed.  status
 * (device int): 1 when the load completed, 2 when the wait ran out (200 ms).
 * Asynchronous on `stream`.  Returns 0, -1 (bad argument), -4 (CUDA error)
 * or -5 (the tensor-map encoder rejected the view).
 */
int moe_testing_tma3d_load(const void* src, int rows, int cols, int r0, int b0, void* out, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif
