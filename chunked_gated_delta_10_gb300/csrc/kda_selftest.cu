// Diagnostic: one tcgen05.mma chain over shared-memory operand tiles, read back
// raw from TMEM (declared in include/kda_selftest.h).
#include "../../include/kda_selftest.h"
#include "tc_util.cuh"
#include "tma_host.h"

namespace kda {
namespace {

constexpr int kSelftestSmem = 32768 + 65536 + 1024 + 64;

__global__ void __launch_bounds__(128) k_umma_selftest(int M, int N, int Kd, int mode,
                                                       const __nv_bfloat16* __restrict__ A,
                                                       const __nv_bfloat16* __restrict__ B, float* __restrict__ raw,
                                                       int* status, const __grid_constant__ CUtensorMap tmA) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* At = sm;
    uint8_t* Bt = sm + 32768;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 32768 + 65536);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool a_mn = mode & 1, b_mn = mode & 2, a_tma = (mode & 4) && !a_mn;
    const int Ar = a_mn ? Kd : M, Ac = a_mn ? M : Kd;
    const int Br = b_mn ? Kd : N, Bc = b_mn ? N : Kd;
    const uint32_t ncols = N < 32 ? 32 : N;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, ncols);
    for (int i = tid; i < Br * Bc; i += blockDim.x)
        *reinterpret_cast<__nv_bfloat16*>(Bt + tile_off(i / Bc, i % Bc, Br)) = B[i];
    if (!a_tma)
        for (int i = tid; i < Ar * Ac; i += blockDim.x)
            *reinterpret_cast<__nv_bfloat16*>(At + tile_off(i / Ac, i % Ac, Ar)) = A[i];
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;
    if (mode & 8) {
        // bounded-wait check: wait on a barrier phase that nothing completes, with a
        // short limit; the wait must give up, record status 7 and let the kernel finish.
        if (tid == 0) mbar_wait(&bars[0], 0, status, 7, 2000000LL);
        __syncthreads();
        tc_fence_before();
        if (warp == 0) tmem_dealloc(tmem, ncols);
        return;
    }
    if (tid == 0) {
        if (a_tma) {
            mbar_expect_tx(&bars[0], (uint32_t)(Ar * Ac * 2));
            for (int cb = 0; cb < Ac / 64; ++cb) tma_load_2d(At + cb * Ar * 128, &tmA, cb * 64, 0, &bars[0]);
            ok = mbar_wait(&bars[0], 0, status, 2);
        }
        if (ok) {
            const uint32_t id = idesc_bf16(M, N, a_mn, b_mn);
            const uint32_t a0 = smem_u32(At), b0 = smem_u32(Bt);
            for (int ks = 0; ks < Kd / 16; ++ks) {
                const uint64_t ad = a_mn ? desc_mnmajor(a0, Ar, ks) : desc_kmajor(a0, Ar, ks);
                const uint64_t bd = b_mn ? desc_mnmajor(b0, Br, ks) : desc_kmajor(b0, Br, ks);
                mma_bf16(tmem, ad, bd, id, ks > 0 ? 1u : 0u);
            }
            mma_commit(&bars[1]);
        }
    }
    __syncthreads();
    if (*(volatile int*)status == 0 && mbar_wait(&bars[1], 0, status, 3)) {
        tc_fence_after();
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
            tmem_ld_wait();
            for (int j = 0; j < 32; ++j) raw[(warp * 32 + lane) * N + c0 + j] = v[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_selftest_umma(int32_t M, int32_t N, int32_t Kd, int32_t mode, const void* A, const void* B,
                                        float* raw, int* status, kda_stream_t stream) {
    using namespace kda;
    if (!(M == 64 || M == 128) || !(N == 64 || N == 128 || N == 256) || !(Kd == 64 || Kd == 128) || mode < 0 ||
        mode > 15 || !A || !B || !raw || !status)
        return KDA_ERR_INVALID_ARG;
    CUtensorMap tm;
    memset(&tm, 0, sizeof(tm));
    if ((mode & 4) && !(mode & 1)) {
        if (!make_tmap_bf16_2d(&tm, A, (uint64_t)Kd, (uint64_t)M, (uint64_t)Kd * 2, 64, (uint32_t)M))
            return KDA_ERR_CUDA;
    }
    cudaError_t e = cudaFuncSetAttribute(k_umma_selftest, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelftestSmem);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    k_umma_selftest<<<1, 128, kSelftestSmem, (cudaStream_t)stream>>>(
        M, N, Kd, mode, (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, raw, status, tm);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
