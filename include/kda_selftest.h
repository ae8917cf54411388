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
 *   mode bit 3: instead of the MMA, check the bounded device wait: the kernel
 *             waits on an mbarrier phase that nothing completes, gives up after
 *             about a millisecond, writes 7 to *status and exits normally.
 * A, B: bf16 device arrays. M in {64, 128}; N in {64, 128, 256}; Kd in {64, 128}.
 * status: device int, set nonzero if a bounded wait gave up (caller zeroes it).
 * Errors: KDA_ERR_INVALID_ARG for other sizes / null pointers; KDA_ERR_CUDA.
 */
kda_status kda_selftest_umma(int32_t M, int32_t N, int32_t Kd, int32_t mode, const void* A, const void* B,
                             float* raw, int* status, kda_stream_t stream);

/*
 * Stage-by-stage check of the tensor-core backward (bf16, K = V = 128 only):
 * runs its first `stages` kernels (1: intra-chunk, 2: + forward state pass,
 * 3: + reverse state-gradient pass, 4: + gradients, whose outputs are not
 * returned here) on `ws`, leaving their intermediates in the workspace.
 * Arguments as kda_chunk_bwd (dh0 nullable; needs h0). Errors:
 * KDA_ERR_UNSUPPORTED off the tensor-core path, else as kda_chunk_bwd.
 */
kda_status kda_debug_bwd_stages(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                                const void* beta, const float* h0, const int64_t* cu_seqlens,
                                const int32_t* chunk_idx, const int64_t* chunk_off, const void* d_o,
                                const float* dht, float* dh0, int32_t stages, void* ws, size_t ws_bytes,
                                kda_stream_t stream);

/*
 * Byte offset and size, inside the backward (pass = KDA_PASS_BWD) workspace,
 * of a tensor-core intermediate: "w", "u", "kh", "qs", "aqk", "inv", "egc",
 * "sin", "dso", "vn", "dvn" (bf16 tiles per chunk and value head, see the
 * library's tile layout; "egc" is fp32). KDA_ERR_UNSUPPORTED off that path.
 */
kda_status kda_debug_ws_region(const kda_dims* dims, int32_t pass, const char* name, size_t* offset, size_t* bytes);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_SELFTEST_H */
