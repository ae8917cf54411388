/*
 * kda_selftest.h — diagnostic entry point of the KDA GB300 library.
 *
 * Checks, on the GPU, the tensor-core building blocks the KDA kernels rely on:
 * a chain of tcgen05.mma (kind::f16, bf16 operands, fp32 accumulator in
 * TMEM) over shared-memory operands in the 128-byte-swizzled tile layout, read
 * back with tcgen05.ld, optionally with operand A brought in by a TMA tiled
 * load. Not part of the KDA computation; the pages have no counterpart.
 */
#ifndef KDA_GB300_SELFTEST_H
#define KDA_GB300_SELFTEST_H

#include <stdint.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * raw[lane][col] (fp32, 128 x N, device) receives TMEM lanes 0..127, columns
 * 0..N-1 after D = A x B^T with D of shape M x N and reduction depth Kd:
 *   mode bit 0 clear: A is given as M x Kd row-major (used K-major);
 *             set:    A is given as Kd x M row-major (used MN-major).
 *   mode bit 1: the same for B (N x Kd, or Kd x N).
 *   mode bit 2: load A with a TMA tiled load (only with bit 0 clear).
 * A, B: bf16 device arrays. M in {64, 128}; N in {64, 128, 256}; Kd in {64, 128}.
 * status: device int, set nonzero if a bounded wait gave up (caller zeroes it).
 * Errors: KDA_ERR_INVALID_ARG for other sizes / null pointers; KDA_ERR_CUDA.
 */
kda_status kda_selftest_umma(int32_t M, int32_t N, int32_t Kd, int32_t mode, const void* A, const void* B,
                             float* raw, int* status, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_SELFTEST_H */
