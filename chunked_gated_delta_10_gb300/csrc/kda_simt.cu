// FP32 FFMA (SIMT) kernels of the chunked KDA forward and backward.
//
// These are the exact-precision path of the library: every product runs in
// fp32 on the CUDA cores, operands staged in shared memory. The library uses
// them for fp32 inputs, where the tensor-core path (bf16 operands) would not
// meet fp32 accuracy. Stage by stage they compute what the bf16 tensor-core
// kernels compute, in the same order of steps:
//
//   intra      per (chunk, value head): gate cumsum (log2 units), the decayed
//              triangles Akk / Aqk, INV = (I + Akk)^-1 by forward
//              substitution, w = INV diag(beta) K~, u = INV diag(beta) V.
//   state_fwd  per (sequence, value head, 32-column slice of V): the chunk
//              loop delta = u - w S_in, S_out = Diag(e^Gamma_C) S_in + K^^T
//              delta, storing S_in of every chunk (and o, ht in the forward).
//   ds_rev     per (sequence, value head, V slice), chunks in reverse:
//              d_delta = Aqk^T dO + K^ dS_out,
//              dS_in = Diag(e^Gamma_C) dS_out + scale Q~^T dO - w^T d_delta.
//   grads_a    per (chunk, value head, 32-row slice of K): the products with
//              the states, dQ~ = scale dO S_in^T, dK^ = delta dS_out^T,
//              dw = -d_delta S_in^T and the Gamma_C term of dg.
//   grads_b    per (chunk, value head): dAqk, dINV, dAkk = -INV^T dINV INV^T,
//              dv, dbeta, the triangle backward, dq, dk, and dg by a reverse
//              in-chunk cumsum.
//   gva_reduce dq, dk summed over each key head's value heads in order.
//
// Notation (natural log Gamma_r = sum_{s<=r} g_s within the chunk; the device
// stores Gamma2 = Gamma * log2(e) and uses exp2):
//   K~ = k e^Gamma, Q~ = q e^Gamma, K^ = k e^(Gamma_C - Gamma),
//   Kr = k e^(Gamma - Gamma_ref), Kc = k e^(Gamma_ref - Gamma) (Gamma_ref is
//   the middle row of the chunk, so both factors stay within e^(span/2)),
//   Akk = tril_-1(diag(beta) Kr Kc^T), Aqk = scale tril_0(Qr Kc^T).
// The chunk formulas are those of the FlashKDA backward (K2) page ("Step 1:
// Recompute U", dU, dkr, dvcorr, dL, dMqk) and FLA's chunk_bwd.py page
// (chunk_kda_bwd, chunk_kda_bwd_kernel_dAv, chunk_kda_bwd_kernel_wy_dqkg_fused).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 32;  // V-slice width of the state kernels / K-slice of grads_a

// C(i,j) (+)= alpha * sum_k A(i,k) B(k,j) on shared-memory fp32 operands.
// A(i,k) = A[i*as0 + k*as1], B(k,j) = B[k*bs0 + j*bs1], C(i,j) = C[i*cs0 + j].
// Each thread owns 4x4 output tiles; every thread sums in the same k order.
__device__ void sgemm(int M, int N, int Kd, const float* A, int as0, int as1, const float* B, int bs0, int bs1,
                      float* Cm, int cs0, float alpha, bool accumulate) {
    const int tn = (N + 3) / 4;
    const int tiles = ((M + 3) / 4) * tn;
    for (int t = threadIdx.x; t < tiles; t += blockDim.x) {
        const int i0 = (t / tn) * 4, j0 = (t % tn) * 4;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        for (int kk = 0; kk < Kd; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = (i0 + i < M) ? A[(i0 + i) * as0 + kk * as1] : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = (j0 + j < N) ? B[kk * bs0 + (j0 + j) * bs1] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i0 + i < M && j0 + j < N) {
                    float* dst = Cm + (i0 + i) * cs0 + j0 + j;
                    *dst = accumulate ? fmaf(alpha, acc[i][j], *dst) : alpha * acc[i][j];
                }
    }
}

// --------------------------------------------------------------------------
// intra: gate cumsum, Akk, Aqk, INV, w, u for one (chunk, value head).
// --------------------------------------------------------------------------
template <typename TI>
__global__ void __launch_bounds__(kThreads) k_intra(Prob p, const TI* __restrict__ q, const TI* __restrict__ k,
                                                    const TI* __restrict__ v, const float* __restrict__ g,
                                                    const TI* __restrict__ beta, Ws ws) {
    extern __shared__ float sm[];
    const int K = p.K, V = p.V, HV = p.HV, H = p.H;
    const int64_t gc = blockIdx.x;
    const int hv = blockIdx.y, h = hv / (HV / H);
    int64_t r0;
    int c;
    chunk_rows(p, gc, r0, c);
    const int tid = threadIdx.x;
    const int KM = K > V ? K : V;
    float* gam = sm;               // [C][K]
    float* kr = gam + kC * K;      // [C][KM]
    float* kc = kr + kC * KM;      // [C][KM]
    float* qr = kc + kC * KM;      // [C][KM]
    float* Akk = qr + kC * KM;     // [C][C]
    float* Aqk = Akk + kC * kC;    // [C][C]
    float* INV = Aqk + kC * kC;    // [C][C]
    float* bet = INV + kC * kC;    // [C]
    float* ref = bet + kC;         // [K]

    for (int d = tid; d < K; d += blockDim.x) {
        float acc = 0.f;
        for (int r = 0; r < kC; ++r) {
            if (r < c) acc += g[((r0 + r) * HV + hv) * K + d];
            const float gm = acc * kLog2e;
            gam[r * K + d] = gm;
            if (r < c) ws.gam[((r0 + r) * HV + hv) * K + d] = gm;
        }
    }
    for (int r = tid; r < kC; r += blockDim.x) bet[r] = r < c ? to_f(beta[(r0 + r) * HV + hv]) : 0.f;
    __syncthreads();
    const int rmid = (c - 1) / 2;
    for (int d = tid; d < K; d += blockDim.x) ref[d] = gam[rmid * K + d];
    __syncthreads();
    for (int i = tid; i < kC * K; i += blockDim.x) {
        const int r = i / K, d = i % K;
        float kv = 0.f, qv = 0.f;
        if (r < c) {
            kv = to_f(k[((r0 + r) * H + h) * K + d]);
            qv = to_f(q[((r0 + r) * H + h) * K + d]);
        }
        const float ep = exp2f(gam[i] - ref[d]), em = exp2f(ref[d] - gam[i]);
        kr[i] = kv * ep;
        kc[i] = kv * em;
        qr[i] = qv * ep;
    }
    __syncthreads();
    sgemm(kC, kC, K, kr, K, 1, kc, 1, K, Akk, kC, 1.f, false);
    sgemm(kC, kC, K, qr, K, 1, kc, 1, K, Aqk, kC, 1.f, false);
    __syncthreads();
    float* aqk_out = ws.aqk + (gc * HV + hv) * kC * kC;
    for (int i = tid; i < kC * kC; i += blockDim.x) {
        const int r = i / kC, j = i % kC;
        Akk[i] = j < r ? bet[r] * Akk[i] : 0.f;
        Aqk[i] = j <= r ? p.scale * Aqk[i] : 0.f;
        aqk_out[i] = Aqk[i];
    }
    __syncthreads();
    // INV = (I + Akk)^-1: forward substitution, one column per thread.
    if (tid < kC) {
        const int j = tid;
        for (int r = 0; r < kC; ++r) INV[r * kC + j] = r == j ? 1.f : 0.f;
        for (int r = j + 1; r < kC; ++r) {
            float s = 0.f;
            for (int m = j; m < r; ++m) s = fmaf(Akk[r * kC + m], INV[m * kC + j], s);
            INV[r * kC + j] = -s;
        }
    }
    __syncthreads();
    float* inv_out = ws.inv + (gc * HV + hv) * kC * kC;
    for (int i = tid; i < kC * kC; i += blockDim.x) inv_out[i] = INV[i];
    // w = INV diag(beta) K~
    for (int i = tid; i < kC * K; i += blockDim.x) {
        const int r = i / K, d = i % K;
        const float kv = r < c ? to_f(k[((r0 + r) * H + h) * K + d]) : 0.f;
        kr[i] = bet[r] * kv * exp2f(gam[i]);
    }
    __syncthreads();
    sgemm(kC, K, kC, INV, kC, 1, kr, K, 1, qr, K, 1.f, false);
    __syncthreads();
    for (int i = tid; i < c * K; i += blockDim.x) ws.w[((r0 + i / K) * HV + hv) * K + i % K] = qr[i];
    // u = INV diag(beta) V
    for (int i = tid; i < kC * V; i += blockDim.x) {
        const int r = i / V, e = i % V;
        kr[i] = r < c ? bet[r] * to_f(v[((r0 + r) * HV + hv) * V + e]) : 0.f;
    }
    __syncthreads();
    sgemm(kC, V, kC, INV, kC, 1, kr, V, 1, kc, V, 1.f, false);
    __syncthreads();
    for (int i = tid; i < c * V; i += blockDim.x) ws.u[((r0 + i / V) * HV + hv) * V + i % V] = kc[i];
}

// --------------------------------------------------------------------------
// state_fwd: sequential chunk loop for one (sequence, value head, V slice).
// --------------------------------------------------------------------------
template <typename TI>
__global__ void __launch_bounds__(kThreads) k_state_fwd(Prob p, const TI* __restrict__ q, const TI* __restrict__ k,
                                                        const float* __restrict__ h0, TI* __restrict__ o,
                                                        float* __restrict__ ht, float* __restrict__ states, Ws ws) {
    extern __shared__ float sm[];
    const int K = p.K, V = p.V, HV = p.HV, H = p.H;
    const int n = blockIdx.x, hv = blockIdx.y, h = hv / (HV / H), v0 = blockIdx.z * kSlice;
    const int tid = threadIdx.x;
    float* S = sm;                  // [K][32]
    float* w = S + K * kSlice;      // [C][K]
    float* kh = w + kC * K;         // [C][K]
    float* dl = kh + kC * K;        // [C][32]
    float* tmp = dl + kC * kSlice;  // [C][32]
    float* gC = tmp + kC * kSlice;  // [K]
    float* qt = gC + K;             // [C][K]   (only with o)
    float* aqk = qt + kC * K;       // [C][C]   (only with o)
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    for (int i = tid; i < K * kSlice; i += blockDim.x) {
        const int d = i / kSlice, j = i % kSlice;
        S[i] = h0 ? h0[(((int64_t)n * HV + hv) * K + d) * V + v0 + j] : 0.f;
    }
    __syncthreads();
    for (int it = 0; it < nts; ++it) {
        const int64_t gc = c0 + it, r0 = bos + (int64_t)it * kC;
        const int c = (int)(eos - r0 < kC ? eos - r0 : kC);
        if (states)
            for (int i = tid; i < K * kSlice; i += blockDim.x)
                states[((gc * HV + hv) * K + i / kSlice) * V + v0 + i % kSlice] = S[i];
        for (int d = tid; d < K; d += blockDim.x) gC[d] = ws.gam[((r0 + c - 1) * HV + hv) * K + d];
        __syncthreads();
        for (int i = tid; i < kC * K; i += blockDim.x) {
            const int r = i / K, d = i % K;
            float wv = 0.f, khv = 0.f, qv = 0.f;
            if (r < c) {
                const int64_t gi = ((r0 + r) * HV + hv) * K + d;
                const int64_t ki = ((r0 + r) * H + h) * K + d;
                wv = ws.w[gi];
                const float gm = ws.gam[gi];
                khv = to_f(k[ki]) * exp2f(gC[d] - gm);
                if (o) qv = p.scale * to_f(q[ki]) * exp2f(gm);
            }
            w[i] = wv;
            kh[i] = khv;
            if (o) qt[i] = qv;
        }
        for (int i = tid; i < kC * kSlice; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice;
            dl[i] = r < c ? ws.u[((r0 + r) * HV + hv) * V + v0 + j] : 0.f;
        }
        if (o)
            for (int i = tid; i < kC * kC; i += blockDim.x) aqk[i] = ws.aqk[(gc * HV + hv) * kC * kC + i];
        __syncthreads();
        sgemm(kC, kSlice, K, w, K, 1, S, kSlice, 1, tmp, kSlice, 1.f, false);
        __syncthreads();
        for (int i = tid; i < kC * kSlice; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice;
            const float x = r < c ? dl[i] - tmp[i] : 0.f;
            dl[i] = x;
            if (r < c) ws.vn[((r0 + r) * HV + hv) * V + v0 + j] = x;
        }
        __syncthreads();
        if (o) {
            sgemm(kC, kSlice, K, qt, K, 1, S, kSlice, 1, tmp, kSlice, 1.f, false);
            __syncthreads();
            sgemm(kC, kSlice, kC, aqk, kC, 1, dl, kSlice, 1, tmp, kSlice, 1.f, true);
            __syncthreads();
            for (int i = tid; i < c * kSlice; i += blockDim.x)
                o[((r0 + i / kSlice) * HV + hv) * V + v0 + i % kSlice] = from_f<TI>(tmp[i]);
        }
        for (int i = tid; i < K * kSlice; i += blockDim.x) S[i] *= exp2f(gC[i / kSlice]);
        __syncthreads();
        sgemm(K, kSlice, kC, kh, 1, K, dl, kSlice, 1, S, kSlice, 1.f, true);
        __syncthreads();
    }
    if (ht)
        for (int i = tid; i < K * kSlice; i += blockDim.x)
            ht[(((int64_t)n * HV + hv) * K + i / kSlice) * V + v0 + i % kSlice] = S[i];
}

// --------------------------------------------------------------------------
// ds_rev: reverse chunk loop of the state gradient for one (seq, hv, V slice).
// --------------------------------------------------------------------------
template <typename TI>
__global__ void __launch_bounds__(kThreads) k_ds_rev(Prob p, const TI* __restrict__ q, const TI* __restrict__ k,
                                                     const TI* __restrict__ d_o, const float* __restrict__ dht,
                                                     float* __restrict__ dh0, Ws ws) {
    extern __shared__ float sm[];
    const int K = p.K, V = p.V, HV = p.HV, H = p.H;
    const int n = blockIdx.x, hv = blockIdx.y, h = hv / (HV / H), v0 = blockIdx.z * kSlice;
    const int tid = threadIdx.x;
    float* dS = sm;                 // [K][32]
    float* kh = dS + K * kSlice;    // [C][K]
    float* w = kh + kC * K;         // [C][K]
    float* qt = w + kC * K;         // [C][K]
    float* aqk = qt + kC * K;       // [C][C]
    float* dO = aqk + kC * kC;      // [C][32]
    float* dd = dO + kC * kSlice;   // [C][32]
    float* gC = dd + kC * kSlice;   // [K]
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    for (int i = tid; i < K * kSlice; i += blockDim.x)
        dS[i] = dht ? dht[(((int64_t)n * HV + hv) * K + i / kSlice) * V + v0 + i % kSlice] : 0.f;
    __syncthreads();
    for (int it = nts - 1; it >= 0; --it) {
        const int64_t gc = c0 + it, r0 = bos + (int64_t)it * kC;
        const int c = (int)(eos - r0 < kC ? eos - r0 : kC);
        for (int i = tid; i < K * kSlice; i += blockDim.x)
            ws.dso[((gc * HV + hv) * K + i / kSlice) * V + v0 + i % kSlice] = dS[i];
        for (int d = tid; d < K; d += blockDim.x) gC[d] = ws.gam[((r0 + c - 1) * HV + hv) * K + d];
        __syncthreads();
        for (int i = tid; i < kC * K; i += blockDim.x) {
            const int r = i / K, d = i % K;
            float wv = 0.f, khv = 0.f, qv = 0.f;
            if (r < c) {
                const int64_t gi = ((r0 + r) * HV + hv) * K + d;
                const int64_t ki = ((r0 + r) * H + h) * K + d;
                wv = ws.w[gi];
                const float gm = ws.gam[gi];
                khv = to_f(k[ki]) * exp2f(gC[d] - gm);
                qv = p.scale * to_f(q[ki]) * exp2f(gm);
            }
            w[i] = wv;
            kh[i] = khv;
            qt[i] = qv;
        }
        for (int i = tid; i < kC * kSlice; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice;
            dO[i] = r < c ? to_f(d_o[((r0 + r) * HV + hv) * V + v0 + j]) : 0.f;
        }
        for (int i = tid; i < kC * kC; i += blockDim.x) aqk[i] = ws.aqk[(gc * HV + hv) * kC * kC + i];
        __syncthreads();
        sgemm(kC, kSlice, kC, aqk, 1, kC, dO, kSlice, 1, dd, kSlice, 1.f, false);
        __syncthreads();
        sgemm(kC, kSlice, K, kh, K, 1, dS, kSlice, 1, dd, kSlice, 1.f, true);
        __syncthreads();
        for (int i = tid; i < c * kSlice; i += blockDim.x)
            ws.dvn[((r0 + i / kSlice) * HV + hv) * V + v0 + i % kSlice] = dd[i];
        for (int i = tid; i < K * kSlice; i += blockDim.x) dS[i] *= exp2f(gC[i / kSlice]);
        __syncthreads();
        sgemm(K, kSlice, kC, qt, 1, K, dO, kSlice, 1, dS, kSlice, 1.f, true);
        __syncthreads();
        sgemm(K, kSlice, kC, w, 1, K, dd, kSlice, 1, dS, kSlice, -1.f, true);
        __syncthreads();
    }
    if (dh0)
        for (int i = tid; i < K * kSlice; i += blockDim.x)
            dh0[(((int64_t)n * HV + hv) * K + i / kSlice) * V + v0 + i % kSlice] = dS[i];
}

// --------------------------------------------------------------------------
// grads_a: products with the chunk states for one (chunk, hv, K slice).
// --------------------------------------------------------------------------
template <typename TI>
__global__ void __launch_bounds__(kThreads) k_grads_a(Prob p, const TI* __restrict__ d_o, Ws ws) {
    extern __shared__ float sm[];
    const int K = p.K, V = p.V, HV = p.HV;
    const int64_t gc = blockIdx.x;
    const int hv = blockIdx.y, d0 = blockIdx.z * kSlice;
    int64_t r0;
    int c;
    chunk_rows(p, gc, r0, c);
    const int tid = threadIdx.x;
    float* dO = sm;                 // [C][V]
    float* dl = dO + kC * V;        // [C][V]
    float* dd = dl + kC * V;        // [C][V]
    float* Si = dd + kC * V;        // [32][V]
    float* dSo = Si + kSlice * V;   // [32][V]
    float* oq = dSo + kSlice * V;   // [C][32]
    float* ok = oq + kC * kSlice;   // [C][32]
    float* ow = ok + kC * kSlice;   // [C][32]
    for (int i = tid; i < kC * V; i += blockDim.x) {
        const int r = i / V, e = i % V;
        const bool in = r < c;
        const int64_t gi = ((r0 + r) * HV + hv) * V + e;
        dO[i] = in ? to_f(d_o[gi]) : 0.f;
        dl[i] = in ? ws.vn[gi] : 0.f;
        dd[i] = in ? ws.dvn[gi] : 0.f;
    }
    const float* si = ws.sin + ((gc * HV + hv) * K + d0) * V;
    const float* so = ws.dso + ((gc * HV + hv) * K + d0) * V;
    for (int i = tid; i < kSlice * V; i += blockDim.x) {
        Si[i] = si[i];
        dSo[i] = so[i];
    }
    __syncthreads();
    sgemm(kC, kSlice, V, dO, V, 1, Si, 1, V, oq, kSlice, p.scale, false);
    sgemm(kC, kSlice, V, dl, V, 1, dSo, 1, V, ok, kSlice, 1.f, false);
    sgemm(kC, kSlice, V, dd, V, 1, Si, 1, V, ow, kSlice, -1.f, false);
    __syncthreads();
    for (int i = tid; i < c * kSlice; i += blockDim.x) {
        const int r = i / kSlice, j = i % kSlice;
        const int64_t gi = ((r0 + r) * HV + hv) * K + d0 + j;
        ws.dqt[gi] = oq[i];
        ws.dkh[gi] = ok[i];
        ws.dw[gi] = ow[i];
    }
    if (tid < kSlice) {
        float acc = 0.f;
        for (int e = 0; e < V; ++e) acc = fmaf(Si[tid * V + e], dSo[tid * V + e], acc);
        const float gCd = ws.gam[((r0 + c - 1) * HV + hv) * K + d0 + tid];
        ws.dgc[(gc * HV + hv) * K + d0 + tid] = acc * exp2f(gCd);
    }
}

// --------------------------------------------------------------------------
// grads_b: everything else for one (chunk, value head).
// --------------------------------------------------------------------------
template <typename TI>
__global__ void __launch_bounds__(kThreads) k_grads_b(Prob p, const TI* __restrict__ q, const TI* __restrict__ k,
                                                      const TI* __restrict__ v, const TI* __restrict__ beta,
                                                      const TI* __restrict__ d_o, TI* __restrict__ dq_out,
                                                      TI* __restrict__ dk_out, TI* __restrict__ dv_out,
                                                      float* __restrict__ dg_out, TI* __restrict__ db_out, Ws ws) {
    extern __shared__ float sm[];
    const int K = p.K, V = p.V, HV = p.HV, H = p.H, G = HV / H;
    const int64_t gc = blockIdx.x;
    const int hv = blockIdx.y, h = hv / G;
    int64_t r0;
    int c;
    chunk_rows(p, gc, r0, c);
    const int tid = threadIdx.x;
    constexpr int CC = kC * kC, CS = kC * kSlice;
    float* INV = sm;            // [C][C]
    float* dN = INV + CC;       // dAqk -> scale * masked
    float* dX = dN + CC;        // dINV -> dAkk -> dM
    float* M = dX + CC;         // Kr Kc^T
    float* Tm = M + CC;         // temp
    float* t0 = Tm + CC;        // 10 slice buffers [C][32]
    float* t1 = t0 + CS;
    float* t2 = t1 + CS;
    float* t3 = t2 + CS;
    float* t4 = t3 + CS;
    float* t5 = t4 + CS;
    float* t6 = t5 + CS;
    float* t7 = t6 + CS;
    float* t8 = t7 + CS;
    float* t9 = t8 + CS;
    float* bet = t9 + CS;       // [C]
    float* db = bet + kC;       // [C]
    float* ref = db + kC;       // [K]
    float* gC = ref + K;        // [K]
    float* dgc = gC + K;        // [32]

    for (int i = tid; i < CC; i += blockDim.x) INV[i] = ws.inv[(gc * HV + hv) * CC + i];
    for (int r = tid; r < kC; r += blockDim.x) {
        bet[r] = r < c ? to_f(beta[(r0 + r) * HV + hv]) : 0.f;
        db[r] = 0.f;
    }
    const int rmid = (c - 1) / 2;
    for (int d = tid; d < K; d += blockDim.x) {
        ref[d] = ws.gam[((r0 + rmid) * HV + hv) * K + d];
        gC[d] = ws.gam[((r0 + c - 1) * HV + hv) * K + d];
    }
    __syncthreads();

    // Phase 1 (V slices): dAqk += dO delta^T, dINV += d_delta (beta V)^T,
    // dv = beta INV^T d_delta, dbeta += rowsum(INV^T d_delta * V).
    for (int e0 = 0; e0 < V; e0 += kSlice) {
        for (int i = tid; i < CS; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice;
            const bool in = r < c;
            const int64_t gi = ((r0 + r) * HV + hv) * V + e0 + j;
            t0[i] = in ? to_f(d_o[gi]) : 0.f;
            t1[i] = in ? ws.vn[gi] : 0.f;
            t2[i] = in ? ws.dvn[gi] : 0.f;
            const float vv = in ? to_f(v[gi]) : 0.f;
            t3[i] = vv;
            t4[i] = bet[r] * vv;
        }
        __syncthreads();
        sgemm(kC, kC, kSlice, t0, kSlice, 1, t1, 1, kSlice, dN, kC, 1.f, e0 > 0);
        sgemm(kC, kC, kSlice, t2, kSlice, 1, t4, 1, kSlice, dX, kC, 1.f, e0 > 0);
        sgemm(kC, kSlice, kC, INV, 1, kC, t2, kSlice, 1, t5, kSlice, 1.f, false);
        __syncthreads();
        for (int i = tid; i < c * kSlice; i += blockDim.x)
            dv_out[((r0 + i / kSlice) * HV + hv) * V + e0 + i % kSlice] = from_f<TI>(bet[i / kSlice] * t5[i]);
        if (tid < kC) {
            float acc = db[tid];
            for (int j = 0; j < kSlice; ++j) acc = fmaf(t5[tid * kSlice + j], t3[tid * kSlice + j], acc);
            db[tid] = acc;
        }
        __syncthreads();
    }
    // Phase 2 (K slices): dINV += dw (beta K~)^T, M += Kr Kc^T.
    for (int d0 = 0; d0 < K; d0 += kSlice) {
        for (int i = tid; i < CS; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice, d = d0 + j;
            const bool in = r < c;
            const int64_t gi = ((r0 + r) * HV + hv) * K + d;
            const float kv = in ? to_f(k[((r0 + r) * H + h) * K + d]) : 0.f;
            const float gm = in ? ws.gam[gi] : gC[d];
            t0[i] = in ? ws.dw[gi] : 0.f;
            t1[i] = bet[r] * kv * exp2f(gm);
            t2[i] = kv * exp2f(gm - ref[d]);
            t3[i] = kv * exp2f(ref[d] - gm);
        }
        __syncthreads();
        sgemm(kC, kC, kSlice, t0, kSlice, 1, t1, 1, kSlice, dX, kC, 1.f, true);
        sgemm(kC, kC, kSlice, t2, kSlice, 1, t3, 1, kSlice, M, kC, 1.f, d0 > 0);
        __syncthreads();
    }
    // Phase 3: dAkk = -INV^T dINV INV^T (strict lower), dbeta from Akk = beta M,
    // dM = beta dAkk, dN = scale dAqk (lower incl. diagonal).
    sgemm(kC, kC, kC, dX, kC, 1, INV, 1, kC, Tm, kC, 1.f, false);
    __syncthreads();
    sgemm(kC, kC, kC, INV, 1, kC, Tm, kC, 1, dX, kC, -1.f, false);
    __syncthreads();
    for (int i = tid; i < CC; i += blockDim.x) {
        const int r = i / kC, j = i % kC;
        const float dA = j < r ? dX[i] : 0.f;
        M[i] = j < r ? M[i] * dA : 0.f;  // dbeta terms, summed per row below
        dX[i] = bet[r] * dA;
        dN[i] = j <= r ? p.scale * dN[i] : 0.f;
    }
    __syncthreads();
    if (tid < kC) {
        float acc = db[tid];
        for (int j = 0; j < kC; ++j) acc += M[tid * kC + j];
        db[tid] = acc;
    }
    __syncthreads();
    // Phase 4 (K slices): triangle backward, exponential chain rule, dq, dk, dg.
    for (int d0 = 0; d0 < K; d0 += kSlice) {
        for (int i = tid; i < CS; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice, d = d0 + j;
            const bool in = r < c;
            const int64_t gi = ((r0 + r) * HV + hv) * K + d;
            const int64_t ki = ((r0 + r) * H + h) * K + d;
            const float kv = in ? to_f(k[ki]) : 0.f;
            const float qv = in ? to_f(q[ki]) : 0.f;
            const float gm = in ? ws.gam[gi] : gC[d];
            t0[i] = kv * exp2f(gm - ref[d]);   // Kr
            t1[i] = kv * exp2f(ref[d] - gm);   // Kc
            t2[i] = qv * exp2f(gm - ref[d]);   // Qr
            t3[i] = in ? ws.dw[gi] : 0.f;      // dw
        }
        if (tid < kSlice) dgc[tid] = ws.dgc[(gc * HV + hv) * K + d0 + tid];
        __syncthreads();
        sgemm(kC, kSlice, kC, INV, 1, kC, t3, kSlice, 1, t4, kSlice, 1.f, false);   // dXk = INV^T dw
        sgemm(kC, kSlice, kC, dN, kC, 1, t1, kSlice, 1, t5, kSlice, 1.f, false);    // dQr = dN Kc
        sgemm(kC, kSlice, kC, dX, kC, 1, t1, kSlice, 1, t6, kSlice, 1.f, false);    // dKr = dM Kc
        sgemm(kC, kSlice, kC, dX, 1, kC, t0, kSlice, 1, t7, kSlice, 1.f, false);    // dKc = dM^T Kr
        __syncthreads();
        sgemm(kC, kSlice, kC, dN, 1, kC, t2, kSlice, 1, t7, kSlice, 1.f, true);     //     + dN^T Qr
        __syncthreads();
        // Elementwise: t8 = dq, t9 = dk, t3 = dGamma (natural-log units).
        for (int i = tid; i < CS; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice, d = d0 + j;
            const bool in = r < c;
            const int64_t gi = ((r0 + r) * HV + hv) * K + d;
            const int64_t ki = ((r0 + r) * H + h) * K + d;
            const float kv = in ? to_f(k[ki]) : 0.f;
            const float qv = in ? to_f(q[ki]) : 0.f;
            const float gm = in ? ws.gam[gi] : gC[d];
            const float E = exp2f(gm), eh = exp2f(gC[d] - gm);
            const float ep = exp2f(gm - ref[d]), em = exp2f(ref[d] - gm);
            const float dQt = in ? ws.dqt[gi] : 0.f;
            const float dKh = in ? ws.dkh[gi] : 0.f;
            const float dXk = t4[i], dQr = t5[i], dKr = t6[i], dKc = t7[i];
            t8[i] = dQt * E + dQr * ep;
            t9[i] = dKh * eh + bet[r] * dXk * E + dKr * ep + dKc * em;
            t3[i] = dQt * qv * E - dKh * kv * eh + bet[r] * dXk * kv * E + dQr * t2[i] + dKr * t0[i] - dKc * t1[i];
            t4[i] = dXk * kv * E;   // dbeta term (rowsum below)
            t5[i] = dKh * kv * eh;  // Gamma_C term (colsum below)
        }
        __syncthreads();
        if (tid < kC) {
            float acc = db[tid];
            for (int j = 0; j < kSlice; ++j) acc += t4[tid * kSlice + j];
            db[tid] = acc;
        }
        if (tid >= 128 && tid < 128 + kSlice) {
            // per channel: add the Gamma_C terms to the last valid row, then
            // the reverse in-chunk cumsum gives dg.
            const int j = tid - 128;
            float acc = dgc[j];
            for (int r = 0; r < c; ++r) acc += t5[r * kSlice + j];
            t3[(c - 1) * kSlice + j] += acc;
            float run = 0.f;
            for (int r = c - 1; r >= 0; --r) {
                run += t3[r * kSlice + j];
                dg_out[((r0 + r) * HV + hv) * K + d0 + j] = run;
            }
        }
        for (int i = tid; i < c * kSlice; i += blockDim.x) {
            const int r = i / kSlice, j = i % kSlice;
            if (G == 1) {
                const int64_t oi = ((r0 + r) * H + h) * K + d0 + j;
                dq_out[oi] = from_f<TI>(t8[i]);
                dk_out[oi] = from_f<TI>(t9[i]);
            } else {
                const int64_t gi = ((r0 + r) * HV + hv) * K + d0 + j;
                ws.dqp[gi] = t8[i];
                ws.dkp[gi] = t9[i];
            }
        }
        __syncthreads();
    }
    for (int r = tid; r < c; r += blockDim.x) db_out[(r0 + r) * HV + hv] = from_f<TI>(db[r]);
}

// dq, dk of key head h = sum over its G value heads in ascending order.
template <typename TI>
__global__ void k_gva_reduce(int64_t rows, int H, int G, int K, const float* __restrict__ dqp,
                             const float* __restrict__ dkp, TI* __restrict__ dq, TI* __restrict__ dk) {
    const int64_t total = rows * H * K;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int d = (int)(i % K);
        const int64_t rh = i / K;
        const int h = (int)(rh % H);
        const int64_t r = rh / H;
        const int64_t base = (r * H * G + (int64_t)h * G) * K + d;
        float aq = 0.f, ak = 0.f;
        for (int j = 0; j < G; ++j) {
            aq += dqp[base + (int64_t)j * K];
            ak += dkp[base + (int64_t)j * K];
        }
        dq[i] = from_f<TI>(aq);
        dk[i] = from_f<TI>(ak);
    }
}

template <typename F>
cudaError_t set_smem(F* f, size_t bytes) {
    return cudaFuncSetAttribute(reinterpret_cast<const void*>(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)bytes);
}

size_t smem_intra(const Prob& p) {
    const int KM = p.K > p.V ? p.K : p.V;
    return sizeof(float) * ((size_t)kC * p.K + 3 * (size_t)kC * KM + 3 * kC * kC + kC + p.K);
}
size_t smem_state_fwd(const Prob& p, bool with_o) {
    size_t f = (size_t)p.K * kSlice + 2 * (size_t)kC * p.K + 2 * kC * kSlice + p.K;
    if (with_o) f += (size_t)kC * p.K + kC * kC;
    return sizeof(float) * f;
}
size_t smem_ds_rev(const Prob& p) {
    return sizeof(float) * ((size_t)p.K * kSlice + 3 * (size_t)kC * p.K + kC * kC + 2 * kC * kSlice + p.K);
}
size_t smem_grads_a(const Prob& p) {
    return sizeof(float) * (3 * (size_t)kC * p.V + 2 * (size_t)kSlice * p.V + 3 * kC * kSlice);
}
size_t smem_grads_b(const Prob& p) {
    return sizeof(float) * (5 * kC * kC + 10 * kC * kSlice + 2 * kC + 2 * (size_t)p.K + kSlice);
}

template <typename TI>
cudaError_t fwd_impl(const Prob& p, const IO& io, const Ws& ws, cudaStream_t st) {
    cudaError_t e;
    const size_t s1 = smem_intra(p), s2 = smem_state_fwd(p, true);
    if ((e = set_smem(k_intra<TI>, s1)) != cudaSuccess) return e;
    if ((e = set_smem(k_state_fwd<TI>, s2)) != cudaSuccess) return e;
    if (p.NT > 0)
        k_intra<TI><<<dim3((unsigned)p.NT, p.HV), kThreads, s1, st>>>(p, (const TI*)io.q, (const TI*)io.k,
                                                                       (const TI*)io.v, io.g, (const TI*)io.beta, ws),
            note_launch("simt_intra", st);
    k_state_fwd<TI><<<dim3(p.N, p.HV, p.V / kSlice), kThreads, s2, st>>>(
        p, (const TI*)io.q, (const TI*)io.k, io.h0, (TI*)io.o, io.ht, io.states_out, ws);
    note_launch("simt_state_fwd", st);
    return cudaGetLastError();
}

template <typename TI>
cudaError_t bwd_impl(const Prob& p, const IO& io, const Ws& ws, cudaStream_t st) {
    cudaError_t e;
    const size_t s1 = smem_intra(p), s2 = smem_state_fwd(p, false), s3 = smem_ds_rev(p), s4 = smem_grads_a(p),
                 s5 = smem_grads_b(p);
    if ((e = set_smem(k_intra<TI>, s1)) != cudaSuccess) return e;
    if ((e = set_smem(k_state_fwd<TI>, s2)) != cudaSuccess) return e;
    if ((e = set_smem(k_ds_rev<TI>, s3)) != cudaSuccess) return e;
    if ((e = set_smem(k_grads_a<TI>, s4)) != cudaSuccess) return e;
    if ((e = set_smem(k_grads_b<TI>, s5)) != cudaSuccess) return e;
    const TI *q = (const TI*)io.q, *k = (const TI*)io.k, *v = (const TI*)io.v, *beta = (const TI*)io.beta,
             *d_o = (const TI*)io.d_o;
    if (p.NT > 0) {
        k_intra<TI><<<dim3((unsigned)p.NT, p.HV), kThreads, s1, st>>>(p, q, k, v, io.g, beta, ws);
        note_launch("simt_intra", st);
    }
    k_state_fwd<TI><<<dim3(p.N, p.HV, p.V / kSlice), kThreads, s2, st>>>(p, q, k, io.h0, (TI*)nullptr, nullptr,
                                                                          ws.sin, ws);
    note_launch("simt_state_fwd", st);
    k_ds_rev<TI><<<dim3(p.N, p.HV, p.V / kSlice), kThreads, s3, st>>>(p, q, k, d_o, io.dht, io.dh0, ws);
    note_launch("simt_ds_rev", st);
    if (p.NT == 0) return cudaGetLastError();
    k_grads_a<TI><<<dim3((unsigned)p.NT, p.HV, p.K / kSlice), kThreads, s4, st>>>(p, d_o, ws);
    note_launch("simt_grads_a", st);
    k_grads_b<TI><<<dim3((unsigned)p.NT, p.HV), kThreads, s5, st>>>(p, q, k, v, beta, d_o, (TI*)io.dq, (TI*)io.dk,
                                                                     (TI*)io.dv, io.dg, (TI*)io.dbeta, ws);
    note_launch("simt_grads_b", st);
    if (p.HV != p.H) {
        const int64_t rows = (int64_t)p.B * p.T;
        k_gva_reduce<TI><<<1024, 256, 0, st>>>(rows, p.H, p.HV / p.H, p.K, ws.dqp, ws.dkp, (TI*)io.dq, (TI*)io.dk);
        note_launch("gva_reduce", st);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t simt_fwd(const Prob& p, bool bf16, const IO& io, const Ws& ws, cudaStream_t st) {
    return bf16 ? fwd_impl<__nv_bfloat16>(p, io, ws, st) : fwd_impl<float>(p, io, ws, st);
}

cudaError_t simt_bwd(const Prob& p, bool bf16, const IO& io, const Ws& ws, cudaStream_t st) {
    return bf16 ? bwd_impl<__nv_bfloat16>(p, io, ws, st) : bwd_impl<float>(p, io, ws, st);
}

}  // namespace kda
