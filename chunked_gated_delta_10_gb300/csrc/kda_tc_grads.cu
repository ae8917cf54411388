// Tensor-core per-chunk gradient kernel of the chunked KDA backward (bf16,
// K = V = 128, chunks of 64), and the grouped-value-head reduction.
//
// One CTA per (chunk, value head), 512 threads. Inputs: q, k, v, dO (TMA),
// and from the earlier stages delta, d_delta, S_in, dS_out, INV, e^Gamma_C
// (bulk copies of bf16 tiles). With Kr = k e^(G-Gref), Kc = k e^(Gref-G),
// Qr = q e^(G-Gref), K~ = k e^G, Q~ = q e^G, K^ = k e^(G_C-G) (natural-log
// Gamma, Gref = middle row), the kernel evaluates, in five dependent MMA
// phases (fp32 accumulators in TMEM, columns noted):
//
//  A  dQ~^T = S_in dO^T [0,64)     dK^^T = dS_out delta^T [64,128)
//     dw = -d_delta S_in^T [128,256) (M=64)   dAqk = dO delta^T [256,320)
//  B  PR^T = V d_delta^T + K~ dw^T [128,192)  Mkk = Kr Kc^T [192,256)
//     dQr^T = Kc^T dN^T [256,320)   dXv = INV^T d_delta [320,448)
//     dXk^T = dw^T INV [448,512)
//  C  T = dINV INV^T [128,192)     with dINV = (P + R) diag(beta)
//  D  dAkk = -INV^T T [320,384)
//  E  dKr^T = Kc^T dM^T [128,192)  dKc^T = Qr^T dN + Kr^T dM [192,256)
//
// where dN = scale tril0(dAqk) and dM = diag(beta) tril-1(dAkk). The
// epilogues give dv = beta dXv and dbeta = sum_j INV[j,r] PR[j,r] +
// sum_j dAkk[r,j] Mkk[r,j] per chunk row (row-per-thread layout), and per key
// channel (channel-per-thread layout) dq, dk and dGamma, whose reverse
// in-chunk cumsum is dg (the Gamma_C terms e^Gamma_C <S_in, dS_out> and
// sum_r dK^ K^ land on the last valid row first). These are the formulas of
// FLA's chunk_bwd.py page (kernel wy_dqkg_fused: dq, dk, dw, dA = -A^T dA A^T,
// dg = q dq - k dk + [last] dgk + kg dkgb beta; the triangle backward of
// chunk_kda_bwd_intra) and the FlashKDA K2 page (dvcorr = INV^T dU, dL).
#include <string.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"
#include "tma_host.h"

namespace kda {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int D = 128;
constexpr int TCD = kC * D * 2, TCC = kC * kC * 2, TDD = D * D * 2;

// Shared-memory map (offsets from a 1024-aligned base).
struct GS {
    static constexpr int Q = 0, K = TCD, V = 2 * TCD, DO = 3 * TCD, DL = 4 * TCD, DDL = 5 * TCD;
    static constexpr int SIN = 6 * TCD, DSO = SIN + TDD;
    // after phase A the S_in / dS_out area holds the decayed factor tiles
    static constexpr int KR = SIN, KC = SIN + TCD, QR = SIN + 2 * TCD, KT = SIN + 3 * TCD;
    static constexpr int DW = DSO + TDD;
    static constexpr int INV = DW + TCD, DN = INV + TCC, DM = DN + TCC, DINV = DM + TCC, TT = DINV + TCC;
    static constexpr int EGC = TT + TCC, BETA = EGC + 512, BARS = BETA + 256, END = BARS + 64;
    // exchange scratch: before phase C the TT tile area holds the gate-cumsum quarter totals
    // and the reference / last-row gates; after phase A the dead dO tile holds the fixed-order
    // partial sums of <S_in, dS_out>, the Gamma_C terms, the dg quarter totals and dbeta.
    static constexpr int XTOT = TT, XRG = TT + 2048;
    static constexpr int XRD = DO, XGC = DO + 2048, XT1 = DO + 4096, XDB = DO + 6144;
};
constexpr int kGradsSmem = 1024 + GS::END;

struct GradMaps {
    CUtensorMap q, k, v, d_o;
};

// 512 threads. Channel-oriented work: thread (d = tid % 128, quarter = tid / 128)
// owns key channel d for chunk rows 16 * quarter .. 16 * quarter + 15. Row-oriented
// work on M = 64 accumulators: row r = 16 * (warp % 4) + lane (lane < 16), column
// quarter warp / 4. Every cross-thread sum is combined in a fixed order.
__global__ void __launch_bounds__(512, 1)
    k_tc_grads(Prob p, const float* __restrict__ g, const bf16* __restrict__ beta, bf16* __restrict__ dq_out,
               bf16* __restrict__ dk_out, bf16* __restrict__ dv_out, float* __restrict__ dg_out,
               bf16* __restrict__ db_out, TcWs ws, const __grid_constant__ GradMaps maps) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = align1024(smraw);
    float* sbeta = reinterpret_cast<float*>(sm + GS::BETA);
    const float* segc = reinterpret_cast<const float*>(sm + GS::EGC);
    float* xtot = reinterpret_cast<float*>(sm + GS::XTOT);
    float* xrg = reinterpret_cast<float*>(sm + GS::XRG);
    float* xrd = reinterpret_cast<float*>(sm + GS::XRD);
    float* xgc = reinterpret_cast<float*>(sm + GS::XGC);
    float* xt1 = reinterpret_cast<float*>(sm + GS::XT1);
    float* xdb = reinterpret_cast<float*>(sm + GS::XDB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + GS::BARS);  // [0] loads, [1] mma
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
    int* fail = reinterpret_cast<int*>(tslot + 1);
    auto S = [&](int off) { return smem_u32(sm + off); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = tid & 127, qtr = tid >> 7, q4 = warp & 3, cq = warp >> 2;
    const int HV = p.HV, H = p.H, G = HV / H, hv = blockIdx.y, h = hv / G;
    const int64_t gc = blockIdx.x, ch = gc * HV + hv;
    int64_t r0;
    int c;
    chunk_rows(p, gc, r0, c);
    float G2[16];  // g of channel d, this thread's 16 rows; Gamma2 after the cumsum below
    load_g_quarters<1>(g, r0, c, HV, hv, d, qtr, G2);

    if (tid == 0) {  // all input copies start right after the g loads
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        *fail = 0;
        mbar_expect_tx(&bars[0], 6 * TCD + 2 * TDD + TCC + 512);
        const int row = (int)r0;
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(sm + GS::Q + b * (TCD / 2), &maps.q, 64 * b, h, row, &bars[0]);
            tma_load_3d(sm + GS::K + b * (TCD / 2), &maps.k, 64 * b, h, row, &bars[0]);
            tma_load_3d(sm + GS::V + b * (TCD / 2), &maps.v, 64 * b, hv, row, &bars[0]);
            tma_load_3d(sm + GS::DO + b * (TCD / 2), &maps.d_o, 64 * b, hv, row, &bars[0]);
        }
        bulk_load(sm + GS::DL, ws.vn + ch * TCD, TCD, &bars[0]);
        bulk_load(sm + GS::DDL, ws.dvn + ch * TCD, TCD, &bars[0]);
        bulk_load(sm + GS::SIN, ws.sin + ch * TDD, TDD, &bars[0]);
        bulk_load(sm + GS::DSO, ws.dso + ch * TDD, TDD, &bars[0]);
        bulk_load(sm + GS::INV, ws.inv + ch * TCC, TCC, &bars[0]);
        bulk_load(sm + GS::EGC, ws.egc + ch * D, 512, &bars[0]);
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    if (tid < kC) sbeta[tid] = tid < c ? __bfloat162float(beta[(r0 + tid) * HV + hv]) : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const ColAddr ad(d, kC);  // this thread's column in the 64-row tiles
    // Gamma2 of channel d for this thread's 16 rows (the canonical order of tc_intra)
    quarter_cumsum_log2<1>(G2, d, qtr, xtot, G2);
    const int rmid = (c - 1) >> 1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (16 * qtr + i == rmid) xrg[d] = G2[i];
        if (16 * qtr + i == c - 1) xrg[128 + d] = G2[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lb = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
    const int rrow = 16 * q4 + lane;                // row of an M = 64 accumulator (lane < 16)
    const bool rv = lane < 16;
    const float ref = xrg[d], gC = xrg[128 + d];
    // per element only ep = 2^(G-ref) and em = 2^(ref-G) are evaluated; E = 2^G and
    // K^'s factor 2^(G_C-G) follow from them (the same formulas in both passes below)
    const float e_ref = exp2f(ref), e_cr = exp2f(gC - ref);

    float rd = 0.f;
    if (!wait_all(&bars[0], 0, ws.status, 41, fail)) goto cleanup;
    if (tid == 0) {  // phase A
        tc_fence_after();
        const uint32_t i128 = idesc_bf16(128, 64, false, false), i64n = idesc_bf16(64, 128, false, false),
                       i64 = idesc_bf16(64, 64, false, false);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 0, desc_kmajor(S(GS::SIN), D, ks), desc_kmajor(S(GS::DO), kC, ks), i128, ks > 0);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 64, desc_kmajor(S(GS::DSO), D, ks), desc_kmajor(S(GS::DL), kC, ks), i128, ks > 0);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 128, desc_kmajor(S(GS::DDL), kC, ks), desc_kmajor(S(GS::SIN), D, ks), idesc_neg_a(i64n),
                     ks > 0);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 256, desc_kmajor(S(GS::DO), kC, ks), desc_kmajor(S(GS::DL), kC, ks), i64, ks > 0);
        mma_commit(&bars[1]);
    }
#pragma unroll
    for (int c8 = 32 * qtr; c8 < 32 * qtr + 32; c8 += 8) {  // <S_in[d, v], dS_out[d, v]> over 32 columns v
        const uint4 a = *reinterpret_cast<const uint4*>(sm + GS::SIN + tile_off(d, c8, D));
        const uint4 b = *reinterpret_cast<const uint4*>(sm + GS::DSO + tile_off(d, c8, D));
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 fa = __bfloat1622float2(pa[u]), fb = __bfloat1622float2(pb[u]);
            rd = fmaf(fa.x, fb.x, rd);
            rd = fmaf(fa.y, fb.y, rd);
        }
    }
    if (!wait_all(&bars[1], 0, ws.status, 42, fail)) goto cleanup;
    tc_fence_after();
    xrd[qtr * 128 + d] = rd;  // the dO tile is dead from here on
    {  // epilogue A: dw row segment (32 columns) and dN row segment (16 columns)
        float x[32];
        tmem_ld32(tmem + lb + 128 + 32 * cq, x);
        tmem_ld_wait();
        if (rv)
            for (int u = 0; u < 4; ++u) st_tile_row8(sm + GS::DW, rrow, 32 * cq + 8 * u, kC, x + 8 * u);
        tmem_ld16(tmem + lb + 256 + 16 * cq, x);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = (16 * cq + u <= rrow && rrow < c) ? p.scale * x[u] : 0.f;
        if (rv)
            for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::DN, rrow, 16 * cq + 8 * u, kC, x + 8 * u);
    }
    tc_fence_before();
    // decayed factor tiles, stored transposed (row = key channel, column = chunk row): channel d,
    // this thread's 16 rows as two 16-byte row segments per tile (rows >= c are zero)
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
        float kr[8], kc[8], qr[8], kt[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 16 * qtr + 8 * h8 + i;
            const bool in = r < c;
            const float kv = in ? ld_col(sm + GS::K, ad, r) : 0.f;
            const float qv = in ? ld_col(sm + GS::Q, ad, r) : 0.f;
            const float gm = G2[8 * h8 + i];
            const float ep = fast_exp2(gm - ref), em = fast_exp2(ref - gm), E = ep * e_ref;
            kr[i] = kv * ep;
            kc[i] = kv * em;
            qr[i] = qv * ep;
            kt[i] = kv * E;
        }
        const int c0 = 16 * qtr + 8 * h8;
        st_tile_row8(sm + GS::KR, d, c0, D, kr);
        st_tile_row8(sm + GS::KC, d, c0, D, kc);
        st_tile_row8(sm + GS::QR, d, c0, D, qr);
        st_tile_row8(sm + GS::KT, d, c0, D, kt);
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {  // phase B
        tc_fence_after();
        const uint32_t i64 = idesc_bf16(64, 64, false, false), i64t = idesc_bf16(64, 64, true, false),
                       i64tt = idesc_bf16(64, 64, true, true);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 128, desc_kmajor(S(GS::V), kC, ks), desc_kmajor(S(GS::DDL), kC, ks), i64, ks > 0);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 128, desc_mnmajor(S(GS::KT), D, ks), desc_kmajor(S(GS::DW), kC, ks), i64t, 1);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + 192, desc_mnmajor(S(GS::KR), D, ks), desc_mnmajor(S(GS::KC), D, ks), i64tt, ks > 0);
        const uint32_t imk = idesc_bf16(128, 64, false, false);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 256, desc_kmajor(S(GS::KC), D, ks), desc_kmajor(S(GS::DN), kC, ks), imk, ks > 0);
        const uint32_t ixv = idesc_bf16(64, 128, true, true);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 320, desc_mnmajor(S(GS::INV), kC, ks), desc_mnmajor(S(GS::DDL), kC, ks), ixv, ks > 0);
        const uint32_t ixk = idesc_bf16(128, 64, true, true);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 448, desc_mnmajor(S(GS::DW), kC, ks), desc_mnmajor(S(GS::INV), kC, ks), ixk, ks > 0);
        mma_commit(&bars[1]);
    }
    if (!wait_all(&bars[1], 1, ws.status, 43, fail)) goto cleanup;
    tc_fence_after();
    {  // epilogue B: dbeta (INV part), dINV columns, dv rows
        const float br = rv ? sbeta[rrow] : 0.f;
        float x[32];
        float db = 0.f;
        tmem_ld16(tmem + lb + 128 + 16 * cq, x);
        tmem_ld_wait();
        if (rv) {
            const ColAddr ar(rrow, kC);
#pragma unroll
            for (int u = 0; u < 16; ++u) db = fmaf(ld_col(sm + GS::INV, ar, 16 * cq + u), x[u], db);
#pragma unroll
            for (int u = 0; u < 16; u += 2) st_col_pair(sm + GS::DINV, ar, 16 * cq + u, br * x[u], br * x[u + 1]);
            xdb[cq * 64 + rrow] = db;
        }
        tmem_ld32(tmem + lb + 320 + 32 * cq, x);
        tmem_ld_wait();
        if (rv && rrow < c) {
            bf16* dvrow = dv_out + ((r0 + rrow) * HV + hv) * D + 32 * cq;
#pragma unroll
            for (int u = 0; u < 32; u += 8) {
                uint4 vv;
                vv.x = pack2(br * x[u], br * x[u + 1]);
                vv.y = pack2(br * x[u + 2], br * x[u + 3]);
                vv.z = pack2(br * x[u + 4], br * x[u + 5]);
                vv.w = pack2(br * x[u + 6], br * x[u + 7]);
                *reinterpret_cast<uint4*>(dvrow + u) = vv;
            }
        }
    }
    tc_fence_before();
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {  // phase C: T = dINV INV^T
        tc_fence_after();
        const uint32_t i64 = idesc_bf16(64, 64, false, false);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 128, desc_kmajor(S(GS::DINV), kC, ks), desc_kmajor(S(GS::INV), kC, ks), i64, ks > 0);
        mma_commit(&bars[1]);
    }
    if (!wait_all(&bars[1], 0, ws.status, 44, fail)) goto cleanup;
    tc_fence_after();
    {
        float x[16];
        tmem_ld16(tmem + lb + 128 + 16 * cq, x);
        tmem_ld_wait();
        if (rv)
            for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::TT, rrow, 16 * cq + 8 * u, kC, x + 8 * u);
    }
    tc_fence_before();
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {  // phase D: dAkk = -INV^T T
        tc_fence_after();
        const uint32_t id = idesc_neg_a(idesc_bf16(64, 64, true, true));
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 320, desc_mnmajor(S(GS::INV), kC, ks), desc_mnmajor(S(GS::TT), kC, ks), id, ks > 0);
        mma_commit(&bars[1]);
    }
    if (!wait_all(&bars[1], 1, ws.status, 45, fail)) goto cleanup;
    tc_fence_after();
    {  // epilogue D: dbeta (Akk part), dM row segments
        const float br = rv ? sbeta[rrow] : 0.f;
        float a[16], m[16];
        float db = 0.f;
        tmem_ld16(tmem + lb + 320 + 16 * cq, a);
        tmem_ld16(tmem + lb + 192 + 16 * cq, m);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int j = 16 * cq + u;
            const bool in = j < rrow && rrow < c;
            db = in ? fmaf(a[u], m[u], db) : db;
            a[u] = in ? br * a[u] : 0.f;
        }
        if (rv) {
            for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::DM, rrow, 16 * cq + 8 * u, kC, a + 8 * u);
            xdb[256 + cq * 64 + rrow] = db;
        }
    }
    tc_fence_before();
    fence_async_smem();
    __syncthreads();
    if (tid < kC && tid < c)
        db_out[(r0 + tid) * HV + hv] = __float2bfloat16_rn(((xdb[tid] + xdb[64 + tid]) + (xdb[128 + tid] + xdb[192 + tid])) +
                                                           ((xdb[256 + tid] + xdb[320 + tid]) +
                                                            (xdb[384 + tid] + xdb[448 + tid])));
    if (tid == 0) {  // phase E
        tc_fence_after();
        const uint32_t ik = idesc_bf16(128, 64, false, false), im = idesc_bf16(128, 64, false, true);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 128, desc_kmajor(S(GS::KC), D, ks), desc_kmajor(S(GS::DM), kC, ks), ik, ks > 0);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 192, desc_kmajor(S(GS::QR), D, ks), desc_mnmajor(S(GS::DN), kC, ks), im, ks > 0);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem + 192, desc_kmajor(S(GS::KR), D, ks), desc_mnmajor(S(GS::DM), kC, ks), im, 1);
        mma_commit(&bars[1]);
    }
    if (!wait_all(&bars[1], 0, ws.status, 46, fail)) goto cleanup;
    tc_fence_after();
    {  // final epilogue, channel d, rows 16 * quarter .. +15: dq, dk, dGamma -> dg
        float dG[16];
        float dGC = 0.f;
        const float sc = p.scale;
#pragma unroll
        for (int rb = 0; rb < 2; ++rb) {
            const uint32_t cb = (uint32_t)(16 * qtr + 8 * rb);
            float aQt[8], aKh[8], aKr[8], aKc[8], aQr[8], aXk[8];
            tmem_ld8(tmem + lb + 0 + cb, aQt);
            tmem_ld8(tmem + lb + 64 + cb, aKh);
            tmem_ld8(tmem + lb + 128 + cb, aKr);
            tmem_ld8(tmem + lb + 192 + cb, aKc);
            tmem_ld8(tmem + lb + 256 + cb, aQr);
            tmem_ld8(tmem + lb + 448 + cb, aXk);
            tmem_ld_wait();
            // the bf16 factor values the MMAs used (zero on rows >= c): row d of the transposed tiles
            const uint4 fkt = ld_raw16(sm + GS::KT, d, (int)cb, D), fqr = ld_raw16(sm + GS::QR, d, (int)cb, D);
            const uint4 fkr = ld_raw16(sm + GS::KR, d, (int)cb, D), fkc = ld_raw16(sm + GS::KC, d, (int)cb, D);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ii = 8 * rb + i, r = 16 * qtr + ii;
                const bool in = r < c;
                const float kv = in ? ld_col(sm + GS::K, ad, r) : 0.f;
                const float qv = in ? ld_col(sm + GS::Q, ad, r) : 0.f;
                const float kt_b = bf16_at(fkt, i), qr_b = bf16_at(fqr, i);
                const float kr_b = bf16_at(fkr, i), kc_b = bf16_at(fkc, i);
                const float gm = G2[ii];
                const float ep = fast_exp2(gm - ref), em = fast_exp2(ref - gm), E = ep * e_ref, eh = em * e_cr;
                const float b = sbeta[r];
                const float dQt = sc * aQt[i], bX = b * aXk[i];
                const float dqv = dQt * E + aQr[i] * ep;
                const float dkv = aKh[i] * eh + bX * E + aKr[i] * ep + aKc[i] * em;
                const float khk = aKh[i] * kv * eh;
                // The factor values of the dGamma pair terms are the bf16 values the MMAs used, so that each
                // in-chunk pair's contributions to its two rows cancel in the chunk sum as they do exactly.
                const float dgv = dQt * qv * E - khk + bX * kt_b + aQr[i] * qr_b + aKr[i] * kr_b - aKc[i] * kc_b;
                dG[ii] = in ? dgv : 0.f;
                if (in) {
                    dGC += khk;
                    if (G == 1) {
                        const int64_t o = ((r0 + r) * H + h) * D + d;
                        st_bf16_pair(reinterpret_cast<uint8_t*>(dq_out + o), reinterpret_cast<uint8_t*>(dk_out + o),
                                     dqv, dkv);
                    } else {
                        const int64_t o = ((r0 + r) * HV + hv) * D + d;
                        ws.dqp[o] = dqv;
                        ws.dkp[o] = dkv;
                    }
                }
            }
        }
        xgc[qtr * 128 + d] = dGC;
        __syncthreads();
        const float dGCt = segc[d] * ((xrd[d] + xrd[128 + d]) + (xrd[256 + d] + xrd[384 + d])) +
                           ((xgc[d] + xgc[128 + d]) + (xgc[256 + d] + xgc[384 + d]));
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (16 * qtr + i == c - 1) dG[i] += dGCt;
        float run = 0.f;
#pragma unroll
        for (int i = 15; i >= 0; --i) {
            run += dG[i];
            dG[i] = run;
        }
        xt1[qtr * 128 + d] = run;
        __syncthreads();
        float carry = 0.f;  // later quarters' totals, added in the order 3, 2, 1
        for (int qq = 3; qq > qtr; --qq) carry += xt1[qq * 128 + d];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * qtr + i;
            if (r < c) dg_out[((r0 + r) * HV + hv) * D + d] = dG[i] + carry;
        }
    }
cleanup:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// dq, dk of key head h = sum over its G value heads in ascending order.
__global__ void k_tc_gva_reduce(int64_t rows, int H, int G, const float* __restrict__ dqp,
                                const float* __restrict__ dkp, bf16* __restrict__ dq, bf16* __restrict__ dk) {
    const int64_t total = rows * H * D;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int dd = (int)(i % D);
        const int64_t rh = i / D;
        const int hh = (int)(rh % H);
        const int64_t r = rh / H;
        const int64_t base = (r * H * G + (int64_t)hh * G) * D + dd;
        float aq = 0.f, ak = 0.f;
        for (int j = 0; j < G; ++j) {
            aq += dqp[base + (int64_t)j * D];
            ak += dkp[base + (int64_t)j * D];
        }
        dq[i] = __float2bfloat16_rn(aq);
        dk[i] = __float2bfloat16_rn(ak);
    }
}

}  // namespace

cudaError_t tc_grads(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_grads, cudaFuncAttributeMaxDynamicSharedMemorySize, kGradsSmem);
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.B * p.T;
    if (p.NT == 0 || rows == 0) return cudaSuccess;
    GradMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rq = (uint64_t)p.H * D * 2, rv = (uint64_t)p.HV * D * 2;
    if (!make_tmap_bf16_3d(&m.q, io.q, D, p.H, rows, D * 2, rq, 64, 1, kC) ||
        !make_tmap_bf16_3d(&m.k, io.k, D, p.H, rows, D * 2, rq, 64, 1, kC) ||
        !make_tmap_bf16_3d(&m.v, io.v, D, p.HV, rows, D * 2, rv, 64, 1, kC) ||
        !make_tmap_bf16_3d(&m.d_o, io.d_o, D, p.HV, rows, D * 2, rv, 64, 1, kC))
        return cudaErrorInvalidValue;
    k_tc_grads<<<dim3((unsigned)p.NT, p.HV), 512, kGradsSmem, st>>>(
        p, io.g, (const bf16*)io.beta, (bf16*)io.dq, (bf16*)io.dk, (bf16*)io.dv, io.dg, (bf16*)io.dbeta, ws, m);
    note_launch("tc_grads", st);
    if (p.HV != p.H) {
        k_tc_gva_reduce<<<1024, 256, 0, st>>>(rows, p.H, p.HV / p.H, ws.dqp, ws.dkp, (bf16*)io.dq, (bf16*)io.dk);
        note_launch("tc_gva_reduce", st);
    }
    return cudaGetLastError();
}

}  // namespace kda
