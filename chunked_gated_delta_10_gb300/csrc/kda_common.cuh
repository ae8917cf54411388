// Shared device-side definitions of the KDA CUDA library (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kC = 64;                          // chunk size (rows per chunk)
constexpr float kLog2e = 1.4426950408889634f;   // gates are carried in log2 units on the device
constexpr float kLn2 = 0.6931471805599453f;

// Everything a kernel needs to locate a chunk or a sequence.
struct Prob {
    int B, T, H, HV, K, V, N;
    int64_t NT;          // total chunks
    int NTs;             // chunks per sequence when sequences have equal length
    float scale;
    const int64_t* cu;   // [N+1] packed offsets, or null (equal-length sequences)
    const int32_t* cidx; // [NT][2] (sequence, chunk in sequence), or null
    const int64_t* coff; // [N+1] first global chunk of a sequence, or null
};

// Rows [r0, r0 + c) of global chunk gc.
__device__ __forceinline__ void chunk_rows(const Prob& p, int64_t gc, int64_t& r0, int& c) {
    int64_t bos, eos;
    int it;
    if (p.cu) {
        const int n = p.cidx[2 * gc];
        it = p.cidx[2 * gc + 1];
        bos = p.cu[n];
        eos = p.cu[n + 1];
    } else {
        const int n = (int)(gc / p.NTs);
        it = (int)(gc % p.NTs);
        bos = (int64_t)n * p.T;
        eos = bos + p.T;
    }
    r0 = bos + (int64_t)it * kC;
    const int64_t rem = eos - r0;
    c = rem < kC ? (int)rem : kC;
}

// Row range and first global chunk of sequence n.
__device__ __forceinline__ void seq_range(const Prob& p, int n, int64_t& bos, int64_t& eos, int64_t& c0) {
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        c0 = p.coff[n];
    } else {
        bos = (int64_t)n * p.T;
        eos = bos + p.T;
        c0 = (int64_t)n * p.NTs;
    }
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace kda
