/*
 * flamia_debug.h -- test-only entry points of the flamia library.
 *
 * They expose one tensor-core tile product so the tests can check, on a
 * single 128-row tile, every operand layout and scale-factor layout the
 * attention kernels rely on (the review page's sec. 3.1: one E4M3 payload read
 * both K-major and MN-major; block-scaled products with E8M0 scales per 32
 * elements; the mixed path's NVFP4 product with E4M3 scales per 16).
 * Not part of the attention API; same ownership and error rules as flamia.h.
 */
#ifndef FLAMIA_DEBUG_H
#define FLAMIA_DEBUG_H

#include <stdint.h>

#include "flamia.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * D[128][N] (float32, device) = A[128 x K] * B[K x N] for one tile.
 *  mode 0: E4M3 x E4M3, unscaled (K = 128).
 *  mode 1: E4M3 x E4M3 block-scaled, E8M0 scale per 32 along K (K = 128);
 *          sfa u8 [128][4], sfb u8 [N][4].
 *  mode 2: E2M1 x E2M1 block-scaled, E4M3 scale per 16 along K (K = 64,
 *          two codes per byte, element 2i in the low nibble); sfa u8 [128][4],
 *          sfb u8 [N][4]; both operands K-major.
 *  mode 3: as mode 1, with A read from tensor memory (row m in lane m, four
 *          E4M3 elements per 32-bit column along K); A must be K-major.
 *  mode 4: as mode 0, with A read from tensor memory as in mode 3.
 *  a: a_mn_major == 0 -> u8 [128][K bytes] (rows = M); 1 -> u8 [K][128].
 *  b: b_mn_major == 0 -> u8 [N][K bytes]   (rows = N); 1 -> u8 [K][N].
 *  N in {32, 64, 128}.  variant: bit 0 swaps the leading / stride byte offsets of
 *  MN-major descriptors; bits 1..2 select the scale-factor placement in
 *  tensor memory (0: column = row / 32, lane = row % 32, replicated in all
 *  lane quadrants; 1: lane = row; 2: as 0 for B, while each lane quadrant q
 *  holds only A's rows 32 q .. 32 q + 31, in column q, and zeros elsewhere).
 * All pointers are device pointers, 16-byte aligned.
 */
flamia_status flamia_debug_mma_tile(int mode, int N, int a_mn_major, int b_mn_major, int variant,
                                    const uint8_t* a, const uint8_t* b, const uint8_t* sfa,
                                    const uint8_t* sfb, float* d_out, int* dev_status,
                                    void* stream);

/*
 * The library's bounded waits running out on purpose: one thread waits on an
 * mbarrier that nothing arrives on, then on a dQ turn counter (device int,
 * zeroed by this call) that nothing passes, with the kernels' own wait
 * helpers; each gives up after its time limit (2 s) and ORs FLAMIA_DEV_TIMEOUT
 * into *dev_status.  Nothing hangs or faults, and the context stays usable.
 * turn: device int the call may write.
 */
flamia_status flamia_debug_bounded_waits(int* turn, int* dev_status, void* stream);

/*
 * The max-reducing tensor-memory load the forward uses on unmasked score
 * tiles: 128 rows of 32 floats (in, device, row-major [128][32]) are stored to
 * tensor memory and loaded back; vals receives the loaded values [128][32],
 * mx the largest value of each row [128] as the load reports it.
 */
flamia_status flamia_debug_tmem_ldred(const float* in, float* vals, float* mx, void* stream);

/*
 * One product of a CTA pair (a cluster of two CTAs whose tensor cores run it
 * together, tcgen05 .cta_group::2; review page sec. 3.4 "Backward pass": the
 * 2-CTA mode splits 256 keys between the pair), in the three shapes the pair
 * backward uses.  CTA r (0, 1) holds A's rows 128 r .. 128 r + 127 and half of
 * B's columns; D rows of CTA r are returned in d_out[r][128][N] (float32).
 *  shape 0: E4M3 unscaled, M 256, N 64, K 128 (S^T = K Q^T):
 *           a u8 [2][128][128] (rows = M, K-major); b u8 [2][32][128]
 *           (CTA r: columns 32 r .. 32 r + 31, rows = N, K-major).
 *  shape 1: E4M3 block-scaled, M 256, N 128, K 64 (dV = P^T dO):
 *           a u8 [2][128][64] (K-major); b u8 [2][64][64] (CTA r: columns
 *           64 r .. 64 r + 63, [K][N], MN-major); sfa u8 [2][128][2] (per row and
 *           K block); sfb u8 [2] (per K block, every column).
 *  shape 2: E4M3 block-scaled, M 256, N 64, K 256 (dQ^T = K^T dS^T):
 *           a u8 [2][256][128] ([K][M], MN-major); b u8 [2][256][32] ([K][N],
 *           MN-major); sfa u8 [2][8], sfb u8 [2][8] (per CTA, per K block,
 *           uniform over M / N).  Only the columns a CTA supplied itself
 *           (32 r .. 32 r + 31) are products of its own A and B.
 * variant (diagnostics, shape 1): bit 0 leaves out the copies of A's scales
 * at column + 4 + row / 32; bit 1 fills B's scales only in the columns of
 * this CTA's own half.  tmem_cols (device u32 [2]) receives each CTA's
 * allocated tensor-memory address.  All pointers are device pointers.
 */
flamia_status flamia_debug_pair_mma(int shape, int variant, const uint8_t* a, const uint8_t* b,
                                    const uint8_t* sfa, const uint8_t* sfb, float* d_out,
                                    uint32_t* tmem_cols, int* dev_status, void* stream);

/*
 * Number of kernel launches the library has enqueued since it was loaded, over
 * every entry point and host thread (memsets are not kernels and are not
 * counted).  Read it before and after a region to count that region's
 * launches.
 */
unsigned long long flamia_debug_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FLAMIA_DEBUG_H */
