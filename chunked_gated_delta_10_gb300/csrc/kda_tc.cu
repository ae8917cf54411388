// Tensor-core (tcgen05) kernels of the chunked KDA forward and backward for
// bf16 inputs with K = V = 128 and chunks of 64 tokens.
//
// Stages (the same steps as the fp32 kernels in kda_simt.cu, regrouped so
// that every dense product is a tcgen05.mma with bf16 operands and an fp32
// accumulator in TMEM):
//
//   tc_intra      persistent, per (chunk, value head): gate cumsum in log2
//                 units, the decayed factors Kr = k e^(G-Gref), Qr =
//                 q e^(G-Gref), Kc = k e^(Gref-G) (Gref = middle row of the
//                 chunk), one MMA group [Kr; Qr] Kc^T giving Akk and Aqk together
//                 (Kc as a bf16 pair hi + lo, so its rounding drops out),
//                 the inverse INV = (I + Akk)^-1 by blocked forward
//                 substitution in fp32, then INVb = INV diag(beta) and
//                 w = INVb K~. Writes w, K^, scale*Q~, Aqk, INV, INVb and
//                 e^(Gamma_C). u = INVb V is never formed on its own: the
//                 state passes take it into delta's accumulator (below), so
//                 it is not rounded to bf16 and makes no round trip.
//   tc_state_fwd  per (sequence, value head[, segment]): the chunk loop
//                 delta = INVb V - w S (one accumulator),
//                 S <- e^(Gamma_C) S + K^^T delta with S in registers (fp32)
//                 and a bf16 copy in shared memory; writes S_in and delta of
//                 every chunk (or, for segmented sweeps, the segment's end
//                 state and transition).
//   tc_ds_rev     per (sequence, value head[, segment]), chunks in reverse:
//                 dDelta = Aqk^T dO + K^ dS,
//                 dS <- e^(Gamma_C) dS + Q~s^T dO - w^T dDelta; writes dS_out,
//                 dDelta and dh0.
//   tc_state_both the two sweeps above in one launch (they are independent: the
//                 reverse pass reads neither S_in nor delta), used when each
//                 pass has at most one (sequence, value head) sweep per SM; with
//                 at most one per two SMs each sweep also splits by state
//                 columns over two CTAs (the columns evolve independently).
//   tc_seg_combine   chains segment start states (long sequences).
//   tc_state_load the backward's state pass from the forward's saved states.
//   tc_fwd_out    the forward: the state pass with o = (scale Q~) S + Aqk
//                 delta formed in the same MMA group.
//
// The columns of S and dS evolve independently (delta, dDelta and o take, per
// column, only that column of S or dS and of V or dO), so when a batch has at
// most one (sequence, value head) sweep per SM each whole sweep of the state,
// reverse and output passes runs as two CTAs of 64 columns (the _half kernels
// and the NH = 1 bodies): narrower MMAs and half the epilogue work per chunk
// step on a chain that is latency-bound there. With packed sequences the
// sweeps start longest first (k_seq_order; a sweep is as long as its sequence).
//
// Intermediates live in the workspace as bf16 tiles in exactly the
// shared-memory operand layout of tc_util.cuh (row-major, 64-column blocks,
// 128-byte swizzle), so each consumer fetches a tile with one bulk copy.
#include <string.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"
#include "tma_host.h"

namespace kda {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int D = 128;                 // K = V on this path
constexpr int TCD = kC * D * 2;        // bytes of a 64 x 128 bf16 tile
constexpr int TCC = kC * kC * 2;       // 64 x 64
constexpr int TDD = D * D * 2;         // 128 x 128

// ---------------------------------------------------------------------------
// (I + L)^-1 for a strictly lower triangular 64 x 64 L (fp32, shared), by
// blocked forward substitution: 16 x 16 diagonal blocks first, then the
// 2 x 2 block formula [[A,0],[C,B]]^-1 = [[A^-1,0],[-B^-1 C A^-1, B^-1]] at
// 32 and 64. 256 threads. Out (64 x 64) receives the lower block triangle
// only: its blocks above the diagonal 16 x 16 blocks are never written nor
// read (the bf16 conversion writes zeros there; see inv_zero_block). Scratch X
// holds 32 x 36 floats.
// ---------------------------------------------------------------------------
// The strictly lower L is stored skewed: element (r, m) at r * 64 + ((m + r) & 63),
// so a warp reading or writing one row per lane hits 32 different banks.
__device__ __forceinline__ int lsk(int r, int m) { return r * kC + ((m + r) & (kC - 1)); }

// Whether 8 columns c0 .. c0+7 (c0 % 8 == 0) of INV row r lie in a block that tri_inverse64 leaves unwritten.
__device__ __forceinline__ bool inv_zero_block(int r, int c0) {
    return (r < 32 && c0 >= 32) || ((r & 31) < 16 && (c0 & 31) >= 16 && (c0 >> 5) == (r >> 5));
}

__device__ void tri_inverse64(const float* L, float* Out, float* X) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp < 4 && lane < 16) {
        // diagonal 16 x 16 block `warp`, column j = lane, right-looking: once x[m] is
        // known, every later row's partial sum takes its term (independent FMAs).
        const int b = warp * 16, j = lane;
        float acc[16], x[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) acc[rr] = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            x[m] = m == j ? 1.f : (m > j ? -acc[m] : 0.f);
#pragma unroll
            for (int rr = m + 1; rr < 16; ++rr) acc[rr] = fmaf(L[lsk(b + rr, b + m)], x[m], acc[rr]);
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Out[(b + rr) * kC + b + j] = x[rr];
    }
    __syncthreads();
    // 16 -> 32: blocks (1,0) and (3,2). X = L21 D0 (D0 lower triangular, zeros included), then -D1 X.
    // Each thread forms a 1 x 2 strip (256 strips per product).
    {
        const int pr = tid >> 7, base = 32 * pr, a = (tid >> 3) & 15, c = 2 * (tid & 7);
        float2 s = bc2(0.f);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float l = L[lsk(base + 16 + a, base + m)];
            s = fma2(bc2(l), *reinterpret_cast<const float2*>(Out + (base + m) * kC + base + c), s);
        }
        *reinterpret_cast<float2*>(X + pr * 256 + a * 16 + c) = s;
    }
    __syncthreads();
    {
        const int pr = tid >> 7, base = 32 * pr, a = (tid >> 3) & 15, c = 2 * (tid & 7);
        float2 s = bc2(0.f);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float l = Out[(base + 16 + a) * kC + base + 16 + m];
            s = fma2(bc2(l), *reinterpret_cast<const float2*>(X + pr * 256 + m * 16 + c), s);
        }
        *reinterpret_cast<float2*>(Out + (base + 16 + a) * kC + base + c) = neg2(s);
    }
    __syncthreads();
    // 32 -> 64, rows 32..63, columns 0..31. X = L[32:64, 0:32] D0 with D0 the (block lower
    // triangular) top-left 32 x 32 inverse: row a = lane, columns 4 warp .. +3; the columns
    // of D0's upper-right zero block (16..31 for rows 0..15) only take rows 16..31.
    {
        const int a = lane, c0 = 4 * warp;
        float2 s01 = bc2(0.f), s23 = bc2(0.f);
        auto term = [&](int m) {
            const float l = L[lsk(32 + a, m)];
            const float4 o = *reinterpret_cast<const float4*>(Out + m * kC + c0);
            s01 = fma2(bc2(l), f2(o.x, o.y), s01);
            s23 = fma2(bc2(l), f2(o.z, o.w), s23);
        };
        if (c0 < 16) {
#pragma unroll
            for (int m = 0; m < 32; ++m) term(m);
        } else {
#pragma unroll
            for (int m = 16; m < 32; ++m) term(m);
        }
        *reinterpret_cast<float4*>(X + a * 36 + c0) = make_float4(s01.x, s01.y, s23.x, s23.y);
    }
    __syncthreads();
    // then -D1 X with D1 the bottom-right 32 x 32 inverse: row 32 + a, columns c0 .. c0+3,
    // a = 4 warp + lane / 8 (rows 0..15 of D1 end at its column 15)
    {
        const int a = tid >> 3, c0 = (tid & 7) * 4;
        float2 s01 = bc2(0.f), s23 = bc2(0.f);
        auto term = [&](int m) {
            const float l = Out[(32 + a) * kC + 32 + m];
            const float4 xv = *reinterpret_cast<const float4*>(X + m * 36 + c0);
            s01 = fma2(bc2(l), f2(xv.x, xv.y), s01);
            s23 = fma2(bc2(l), f2(xv.z, xv.w), s23);
        };
        if (a < 16) {
#pragma unroll
            for (int m = 0; m < 16; ++m) term(m);
        } else {
#pragma unroll
            for (int m = 0; m < 32; ++m) term(m);
        }
        *reinterpret_cast<float4*>(Out + (32 + a) * kC + c0) = make_float4(-s01.x, -s01.y, -s23.x, -s23.y);
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// tc_intra: persistent, two 256-thread CTAs per SM (two threads per key channel:
// rows 0..31 and 32..63), each walking its (chunk, value head) items round-robin.
// Inputs staged by TMA and transformed in place (q -> scale Q~, k -> K^). The
// next item's q and k are fetched once the K^ / Q~ copies have read their tiles,
// and its g (registers) and beta while the current item finishes. 112 KB of
// shared memory.
// ---------------------------------------------------------------------------
struct IS {
    static constexpr int Q = 0, K = TCD, XB = 2 * TCD, KQ = 3 * TCD, KC = 5 * TCD, XK = 6 * TCD, MISC = 7 * TCD;
    // XB holds the low part of Kc (Kc - bf16(Kc), rounded to bf16) for the first MMA.
    // aliases: after the first MMA, KQ holds Akk / INV in fp32; after the last, w staging.
    // after the first MMA, KC holds the bf16 INV tile and the inversion scratch; XB holds the bf16 INVb tile.
    static constexpr int AKK = KQ, FI = KQ + 16384, TINV = KC, XS = KC + TCC, TINVB = XB, WST = KQ;
    static constexpr int END = MISC + 512 + 64;  // beta (two item slots), barriers
};
constexpr int kIntraSmem = IS::END;

struct IntraMaps {
    CUtensorMap q, k;
};

__global__ void __launch_bounds__(256, 2) k_tc_intra(Prob p, const float* __restrict__ g,
                                                      const bf16* __restrict__ beta, TcWs ws,
                                                      const __grid_constant__ IntraMaps maps) {
    extern __shared__ __align__(1024) uint8_t sm[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + IS::MISC + 512);  // [0, 1] inputs (by item parity), [2] mma
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
    int* fail = reinterpret_cast<int*>(tslot + 1);
    float* Akk = reinterpret_cast<float*>(sm + IS::AKK);
    float* Fi = reinterpret_cast<float*>(sm + IS::FI);
    // item-start scratch (6 x 128 floats) in the K~ tile, dead from the second product of the previous item
    // to this item's factor pass
    float* tmp = reinterpret_cast<float*>(sm + IS::XK);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d0 = 2 * (tid & 63), qt = tid >> 6;  // key channels d0, d0 + 1; chunk rows 16 qt .. +15
    const int HV = p.HV, H = p.H, G = HV / H;
    const int64_t total = p.NT * HV;
    if (tid == 0) {
        *fail = (smem_u32(sm) & 1023u) ? 1 : 0;  // tiles need a 1024-byte aligned base
        if (*fail) *(volatile int*)ws.status = 10;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (*(volatile int*)fail) goto cleanup;
    {
        const ColAddr a64(d0, kC), a128(d0, 128);  // this thread's channel pair in the 64- and 128-row tiles
        auto issue_qk = [&](int64_t r0, int h, uint64_t* b) {
            mbar_expect_tx(b, 2 * TCD);
            for (int x = 0; x < 2; ++x) {
                tma_load_3d(sm + IS::Q + x * (TCD / 2), &maps.q, 64 * x, h, (int)r0, b);
                tma_load_3d(sm + IS::K + x * (TCD / 2), &maps.k, 64 * x, h, (int)r0, b);
            }
        };
        int64_t w = blockIdx.x;
        int64_t r0;
        int c;
        chunk_rows(p, w / HV, r0, c);
        float G2[32];  // g of channels d0 + ch, rows 16 qt + i at [16 ch + i] (the next item's during the last phase)
        load_g_pair(g, r0, c, HV, (int)(w % HV), d0, qt, G2);
        if (tid < kC) {
            float* sb0 = reinterpret_cast<float*>(sm + IS::MISC);
            sb0[tid] = tid < c ? __bfloat162float(beta[(r0 + tid) * HV + (int)(w % HV)]) : 0.f;
        }
        if (tid == 0) issue_qk(r0, (int)(w % HV) / G, &bars[0]);
        uint32_t mph = 0;
        for (int i = 0; w < total; ++i, w += gridDim.x) {
            const int slot = i & 1;
            const int64_t ch = w;
            // (r0, c: this item's rows, found while the previous item ran; with packed sequences a look-up in
            // the chunk table, two dependent global loads, that would otherwise stall the item's start)
            const int64_t wn = w + gridDim.x;
            const bool has_next = wn < total;
            const int hvn = (int)(wn % HV);
            int64_t r0n = r0;
            int cn = c;
            if (has_next) chunk_rows(p, wn / HV, r0n, cn);
            const float* sb = reinterpret_cast<const float*>(sm + IS::MISC + 256 * slot);

            pair_cumsum_log2(G2, d0, qt, tmp);
            // reference row (middle of the chunk) and last valid row
            const int rmid = (c - 1) >> 1;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                if (16 * qt + x == rmid) {
                    tmp[512 + d0] = G2[x];
                    tmp[512 + d0 + 1] = G2[16 + x];
                }
                if (16 * qt + x == c - 1) {
                    tmp[640 + d0] = G2[x];
                    tmp[640 + d0 + 1] = G2[16 + x];
                }
            }
            __syncthreads();
            const float ref0 = tmp[512 + d0], ref1 = tmp[512 + d0 + 1], gC0 = tmp[640 + d0], gC1 = tmp[640 + d0 + 1];
            if (qt == 0) *reinterpret_cast<float2*>(ws.egc + ch * D + d0) = make_float2(exp2f(gC0), exp2f(gC1));
            // per element only ep = 2^(G-ref) and em = 2^(ref-G) are evaluated; E = 2^G = ep 2^ref and K^'s
            // factor 2^(G_C-G) = em 2^(G_C-ref) follow from them (the formulas of the gradient kernel)
            const float2 er = f2(exp2f(ref0), exp2f(ref1)), ec = f2(exp2f(gC0 - ref0), exp2f(gC1 - ref1));
            const float2 nref = f2(-ref0, -ref1);
            // this item's q and k landed, and every thread has read the reference rows (the factor pass
            // overwrites the scratch)
            if (!wait_all(&bars[slot], (uint32_t)(i >> 1) & 1, ws.status, 11, fail)) break;
            // decayed factors, two key channels per 32-bit access; in place: q -> scale Q~, k -> K^
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int r = 16 * qt + x;
                const bool in = r < c;
                const uint32_t o = a64.at(r);
                const uint32_t k2 = in ? *reinterpret_cast<const uint32_t*>(sm + IS::K + o) : 0u;
                const uint32_t q2 = in ? *reinterpret_cast<const uint32_t*>(sm + IS::Q + o) : 0u;
                // channels d0 and d0 + 1 as packed fp32 pairs
                const float2 kk = f2(bf_lo(k2), bf_hi(k2)), qq = f2(bf_lo(q2), bf_hi(q2));
                const float2 gd = add2(f2(G2[x], G2[16 + x]), nref);  // G - Gref
                const float2 ep = f2(fast_exp2(gd.x), fast_exp2(gd.y)), em = f2(fast_exp2(-gd.x), fast_exp2(-gd.y));
                const float2 E = mul2(ep, er), eh = mul2(em, ec);
                const float2 kr = mul2(kk, ep), qr = mul2(qq, ep), kc = mul2(kk, em);
                const float2 kt = mul2(kk, E), kh = mul2(kk, eh), qs = mul2(mul2(bc2(p.scale), qq), E);
                *reinterpret_cast<uint32_t*>(sm + IS::KQ + a128.at(r)) = pack2(kr.x, kr.y);
                *reinterpret_cast<uint32_t*>(sm + IS::KQ + a128.at(kC + r)) = pack2(qr.x, qr.y);
                {  // Kc as a bf16 pair and the bf16 pair of its rounding remainder
                    const uint32_t hi = pack2(kc.x, kc.y);
                    *reinterpret_cast<uint32_t*>(sm + IS::KC + o) = hi;
                    const float2 lo = add2(kc, neg2(f2(bf_lo(hi), bf_hi(hi))));
                    *reinterpret_cast<uint32_t*>(sm + IS::XB + o) = pack2(lo.x, lo.y);
                }
                *reinterpret_cast<uint32_t*>(sm + IS::XK + o) = pack2(kt.x, kt.y);
                *reinterpret_cast<uint32_t*>(sm + IS::K + o) = pack2(kh.x, kh.y);
                *reinterpret_cast<uint32_t*>(sm + IS::Q + o) = pack2(qs.x, qs.y);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0) {
                // [Kr; Qr] (Kc_hi + Kc_lo)^T: the remainder of Kc's rounding is carried by a second product
                const uint32_t id = idesc_bf16(128, 64, false, false);
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_bf16(tmem, desc_kmajor(smem_u32(sm + IS::KQ), 128, ks),
                             desc_kmajor(smem_u32(sm + IS::KC), kC, ks), id, ks > 0);
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_bf16(tmem, desc_kmajor(smem_u32(sm + IS::KQ), 128, ks),
                             desc_kmajor(smem_u32(sm + IS::XB), kC, ks), id, 1);
                mma_commit(&bars[2]);
                bulk_store(ws.kh + ch * TCD, sm + IS::K, TCD);
                bulk_store(ws.qs + ch * TCD, sm + IS::Q, TCD);
                bulk_commit();
            }
            // beta of the next item: loaded now, stored to its shared slot at the end of this item
            const float nbeta =
                (has_next && tid < cn) ? __bfloat162float(beta[(r0n + tid) * HV + hvn]) : 0.f;
            warp_wait(&bars[2], mph, ws.status, 12, fail);  // per warp; a time-out leaves at the next barrier
            mph ^= 1;
            if (tid == 0 && has_next) {
                bulk_wait_read();  // the K^ and scale Q~ copies have read their tiles
                issue_qk(r0n, hvn / G, &bars[slot ^ 1]);
            }
            tc_fence_after();
            {  // Akk (rows 0..63) and Aqk (rows 64..127): lane row 32 * (warp % 4) + lane, 32 columns per warp half
                const int R = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);
                float row[32];
                tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + c0, row);
                tmem_ld_wait();
                if (R < kC) {
                    const int r = R;
                    const float2 br = bc2(sb[r]);
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 v = mul2(br, f2(row[j], row[j + 1]));
                        Akk[lsk(r, c0 + j)] = (c0 + j < r) ? v.x : 0.f;
                        Akk[lsk(r, c0 + j + 1)] = (c0 + j + 1 < r) ? v.y : 0.f;
                    }
                } else {
                    const int r = R - kC;
                    uint8_t* gA = ws.aqk + ch * TCC;
                    for (int u = 0; u < 32; u += 8) {
                        uint32_t pk[4];
#pragma unroll
                        for (int t = 0; t < 8; t += 2) {
                            const float2 v = mul2(bc2(p.scale), f2(row[u + t], row[u + t + 1]));
                            pk[t / 2] = pack2((c0 + u + t <= r) ? v.x : 0.f, (c0 + u + t + 1 <= r) ? v.y : 0.f);
                        }
                        *reinterpret_cast<uint4*>(gA + tile_off(r, c0 + u, kC)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
            tc_fence_before();
            __syncthreads();
            if (*(volatile int*)fail) break;
            tri_inverse64(Akk, Fi, reinterpret_cast<float*>(sm + IS::XS));
            // INV and INVb = INV diag(beta) (column j scaled by beta_j) as bf16 operand tiles
            for (int e = tid; e < kC * (kC / 8); e += blockDim.x) {
                const int r = e >> 3, c0 = (e & 7) * 8;
                if (inv_zero_block(r, c0)) {
                    *reinterpret_cast<uint4*>(sm + IS::TINV + tile_off(r, c0, kC)) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sm + IS::TINVB + tile_off(r, c0, kC)) = make_uint4(0u, 0u, 0u, 0u);
                } else {
                    const float* fr = Fi + r * kC + c0;
                    st_tile_row8(sm + IS::TINV, r, c0, kC, fr);
                    float xb[8];
#pragma unroll
                    for (int t = 0; t < 8; t += 2) {
                        const float2 v = mul2(*reinterpret_cast<const float2*>(fr + t),
                                              *reinterpret_cast<const float2*>(sb + c0 + t));
                        xb[t] = v.x, xb[t + 1] = v.y;
                    }
                    st_tile_row8(sm + IS::TINVB, r, c0, kC, xb);
                }
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                // w = INVb K~: chunk rows on TMEM lanes (M = 64, N = 128)
                const uint32_t id = idesc_bf16(64, 128, false, true);
                const uint32_t ti = smem_u32(sm + IS::TINVB);
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_bf16(tmem, desc_kmajor(ti, kC, ks), desc_mnmajor(smem_u32(sm + IS::XK), kC, ks), id, ks > 0);
                mma_commit(&bars[2]);
                bulk_store(ws.inv + ch * TCC, sm + IS::TINV, TCC);
                bulk_store(ws.invb + ch * TCC, sm + IS::TINVB, TCC);
                bulk_commit();
            }
            warp_wait(&bars[2], mph, ws.status, 13, fail);
            mph ^= 1;
            if (has_next) load_g_pair(g, r0n, cn, HV, hvn, d0, qt, G2);
            tc_fence_after();
            {  // w rows: row r = 16 (warp % 4) + lane (lane < 16), 64 columns per warp half
                const int r = 16 * (warp & 3) + lane, cb = 64 * (warp >> 2);
                const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int col = 32 * t + cb;
                    float x[32];
                    tmem_ld32(tmem + lb + col, x);
                    tmem_ld_wait();
                    if (lane < 16) {
#pragma unroll
                        for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(sm + IS::WST, r, col + c8, kC, x + c8);
                    }
                }
            }
            if (tid < kC) reinterpret_cast<float*>(sm + IS::MISC + 256 * (slot ^ 1))[tid] = nbeta;
            tc_fence_before();
            fence_async_smem();
            __syncthreads();
            if (*(volatile int*)fail) break;
            if (tid == 0) {
                bulk_store(ws.w + ch * TCD, sm + IS::WST, TCD);
                bulk_commit();
                bulk_wait_read();  // the w, INV and INV diag(beta) tiles are rewritten by the next item's factor pass
            }
            r0 = r0n;
            c = cn;
            // (no barrier here: before its first barrier the next item writes only the item-start scratch, in the
            // dead K~ tile, and thread 0 reaches that barrier only once the copies above have read their tiles)
        }
    }
cleanup:
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// Segment modes of the state passes (grid z = segment, or 2 x segments for
// mode kSegEnds: z < M the end state from a zero start, z >= M the transition).
//   kSegNone   one sweep over the sequence (len = 0), checkpoints written
//   kSegCkpt   checkpoints of one segment from its start state (seg_s0)
//   kSegEnds   per segment: the end state from a zero start (seg_e) and the
//              transition, i.e. the end state from the identity with the
//              chunk inputs that do not multiply the state set to zero (seg_p)
// ---------------------------------------------------------------------------
enum { kSegNone = 0, kSegCkpt = 1, kSegEnds = 2 };
struct SegArg {
    int len, M, mode;
};

// ---------------------------------------------------------------------------
// tc_state_fwd: one CTA per (value head, sequence[, segment]), 256 threads;
// thread t owns state row k = t % 128, columns 64 (t / 128) .. +63 in fp32
// registers (split by columns, tc_state_fwd_half: 64 columns per CTA, 32 per
// thread). A bf16 copy of S in shared memory feeds the MMAs and is the S_in
// checkpoint. Chunk inputs: V (TMA) and e^Gamma_C double-buffered; w with INVb,
// and K^, single-buffered, each refetched as soon as its MMA has consumed it.
// delta = INVb V - w S accumulates in one TMEM accumulator and overwrites V in
// place.
// ---------------------------------------------------------------------------
struct FwdSm {
    static constexpr int W = 0, IVB = TCD, KH = TCD + TCC, U = 2 * TCD + TCC;
    static constexpr int UBUF = TCD + 1024;  // V (then delta) tile, then e^Gamma_C (512 B)
    static constexpr int S = U + 2 * UBUF, BARS = S + TDD, END = BARS + 64;
};
constexpr int kFwdSmem = 1024 + FwdSm::END;

// (sequence n, value head hv, grid z: the segment, or for kSegEnds segment and mode.) The state's columns
// evolve independently (delta's column v takes only S's column v), so a sweep may be split by columns: NH
// = 2 runs all 128 on this CTA (thread = row k, 64 columns); NH = 1 runs the 64 columns of half h (thread
// = row k, 32 columns), with narrower MMAs, for batches whose sweeps leave SMs idle.
template <int NH>
__device__ __forceinline__ void state_fwd_body(const Prob& p, const float* __restrict__ h0, const TcWs& ws,
                                               const SegArg& sg, const CUtensorMap& tm_v, uint8_t* sm, int hv, int n,
                                               int z, int h) {
    constexpr int CW = 64 * NH, TW = CW / 2;  // state columns of this CTA and of each thread
    uint8_t* tS = sm + FwdSm::S;              // bf16 copy of S (128 x CW)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + FwdSm::BARS);  // u[2], w, K^, mma
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 5);
    int* fail = reinterpret_cast<int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = tid & 127, vq = tid >> 7;
    const int cbase = 64 * h + TW * vq;  // this thread's first state column
    const int HV = p.HV;
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    // segment and mode: 0 checkpoints, 1 end state from zero, 2 transition
    const int m = sg.mode == kSegEnds ? z % sg.M : z;
    const int mode = sg.mode == kSegEnds ? 1 + z / sg.M : 0;
    const int lo = sg.len ? m * sg.len : 0, hi = sg.len ? min(lo + sg.len, nts) : nts;
    if (sg.len && lo >= hi) return;
    const bool ckpt = mode == 0, with_u = mode != 2;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tslot, 2 * CW);  // delta [0, CW), state [CW, 2 CW)
    float S[TW];
    const int64_t seg_at = (((int64_t)n * HV + hv) * sg.M + m) * D * D + (int64_t)k * D + cbase;
    {
        const float* src = nullptr;
        if (mode == 0) src = (lo == 0) ? (h0 ? h0 + (((int64_t)n * HV + hv) * D + k) * D + cbase : nullptr)
                                       : ws.seg_s0 + seg_at;
#pragma unroll
        for (int j = 0; j < TW; ++j) S[j] = src ? src[j] : (mode == 2 && cbase + j == k ? 1.f : 0.f);
    }
    auto chunk = [&](int it) { return (c0 + it) * HV + hv; };
    auto issue_u = [&](int it) {  // V rows of chunk it (TMA; this CTA's columns) and e^Gamma_C
        const int b = (it - lo) & 1;
        uint8_t* buf = sm + FwdSm::U + b * FwdSm::UBUF;
        mbar_expect_tx(&bars[b], (with_u ? NH * (TCD / 2) : 0) + 512);
        if (with_u) {
            const int row = (int)(bos + (int64_t)it * kC);
            for (int x = 0; x < NH; ++x) tma_load_3d(buf + x * (TCD / 2), &tm_v, 64 * (h + x), hv, row, &bars[b]);
        }
        bulk_load(buf + TCD, ws.egc + chunk(it) * D, 512, &bars[b]);
    };
    auto issue_w = [&](int it) {  // w and INVb
        mbar_expect_tx(&bars[2], TCD + (with_u ? TCC : 0));
        bulk_load(sm + FwdSm::W, ws.w + chunk(it) * TCD, TCD, &bars[2]);
        if (with_u) bulk_load(sm + FwdSm::IVB, ws.invb + chunk(it) * TCC, TCC, &bars[2]);
    };
    auto issue_kh = [&](int it) {
        mbar_expect_tx(&bars[3], TCD);
        bulk_load(sm + FwdSm::KH, ws.kh + chunk(it) * TCD, TCD, &bars[3]);
    };
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter
    if (tid == 0 && lo < hi) {
        issue_w(lo);
        issue_kh(lo);
        issue_u(lo);
        if (lo + 1 < hi) issue_u(lo + 1);
    }
    uint32_t mph = 0;
    for (int it = lo; it < hi; ++it) {
        const int64_t ch = chunk(it);
        const int rel = it - lo;
        const uint32_t ph = (uint32_t)rel & 1;  // phase of the single-buffered w and K^ barriers
        uint8_t* tU = sm + FwdSm::U + (rel & 1) * FwdSm::UBUF;
        // bf16 copy of S (row k, this thread's columns) for the MMAs and the S_in checkpoint
#pragma unroll
        for (int c8 = 0; c8 < TW; c8 += 8) st_tile_row8(tS, k, TW * vq + c8, D, S + c8);
        fence_async_smem();
        // w, INVb and V (both prefetched) in one wait
        if (!wait_all2(&bars[2], ph, 21, &bars[rel & 1], (rel >> 1) & 1, 24, ws.status, fail)) break;
        const float e = reinterpret_cast<const float*>(tU + TCD)[k];  // e^Gamma_C of this thread's state row
        // delta accumulator = -w S + INVb V (chunk rows on TMEM lanes, M = 64, N = CW)
        const uint32_t idd = idesc_bf16(64, CW, false, true);
        if (tid == 0) {
            tc_fence_after();
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + FwdSm::W), kC, ks), desc_mnmajor(smem_u32(tS), D, ks),
                         idesc_neg_a(idd), ks > 0);
            if (with_u)
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_bf16(tmem, desc_kmajor(smem_u32(sm + FwdSm::IVB), kC, ks), desc_mnmajor(smem_u32(tU), kC, ks),
                             idd, 1);
            mma_commit(&bars[4]);
            if (ckpt) {  // (column block h of the 128-row tile)
                bulk_store(ws.sin + ch * TDD + h * (D * 128), tS, D * CW * 2);
                bulk_commit();
            }
        }
        // per warp (the next barrier reads *fail): after it a warp touches only what the finished MMAs have read
        warp_wait(&bars[4], mph, ws.status, 22, fail);
        mph ^= 1;
        if (tid == 0 && it + 1 < hi) issue_w(it + 1);  // w and INVb are consumed
        tc_fence_after();
        {  // delta (bf16) in place of V: row r = 16 (warp % 4) + lane (lane < 16), CW / 2 columns per warp half
            const int r = 16 * (warp & 3) + lane, cb = (CW / 2) * (warp >> 2);
#pragma unroll
            for (int x = 0; x < CW / 64; ++x) {
                float acc[32];
                tmem_ld32(tmem + lq + cb + 32 * x, acc);
                tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(tU, r, cb + 32 * x + c8, kC, acc + c8);
                }
            }
        }
        tc_fence_before();
        fence_async_smem();
        if (!wait_all(&bars[3], ph, ws.status, 25, fail)) break;
        if (tid == 0) {  // S accumulator = K^^T delta (M = 128, N = CW)
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, CW, true, true);
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem + CW, desc_mnmajor(smem_u32(sm + FwdSm::KH), kC, ks), desc_mnmajor(smem_u32(tU), kC, ks),
                         id, ks > 0);
            mma_commit(&bars[4]);
            if (ckpt) {  // (column block h of the 64-row tile)
                bulk_store(ws.vn + ch * TCD + h * (kC * 128), tU, kC * CW * 2);
                bulk_commit();
            }
        }
        if (tid == 0) bulk_wait_read();  // S_in and delta copies have read tS and the V / delta buffer
        // after this wait every thread has read e^Gamma_C and the state MMA has read delta: the buffer is free
        if (!wait_all(&bars[4], mph, ws.status, 23, fail)) break;
        mph ^= 1;
        if (tid == 0) {
            if (it + 1 < hi) issue_kh(it + 1);  // K^ is consumed
            if (it + 2 < hi) issue_u(it + 2);
        }
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < TW / 32; ++x) {
            float acc[32];
            tmem_ld32(tmem + lq + CW + TW * vq + 32 * x, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 v = fma2(bc2(e), f2(S[32 * x + j], S[32 * x + j + 1]), f2(acc[j], acc[j + 1]));
                S[32 * x + j] = v.x, S[32 * x + j + 1] = v.y;
            }
        }
        tc_fence_before();
    }
    if (mode != 0 && *(volatile int*)fail == 0) {
        float* dst = (mode == 1 ? ws.seg_e : ws.seg_p) + seg_at;
#pragma unroll
        for (int j = 0; j < TW; ++j) dst[j] = S[j];
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * CW);
}

__global__ void __launch_bounds__(256, 2) k_tc_state_fwd(Prob p, const float* __restrict__ h0, TcWs ws, SegArg sg,
                                                          const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smraw[];
    state_fwd_body<2>(p, h0, ws, sg, tm_v, align1024(smraw), blockIdx.x, sweep_seq(ws, blockIdx.y), blockIdx.z, 0);
}
// whole sweeps split by columns: grid x = 2 HV (value head x / 2, column half x % 2)
__global__ void __launch_bounds__(256, 2) k_tc_state_fwd_half(Prob p, const float* __restrict__ h0, TcWs ws,
                                                               const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smraw[];
    state_fwd_body<1>(p, h0, ws, SegArg{0, 1, kSegNone}, tm_v, align1024(smraw), blockIdx.x >> 1,
                      sweep_seq(ws, blockIdx.y), 0, blockIdx.x & 1);
}

// ---------------------------------------------------------------------------
// tc_seg_combine: start states of the segments of one (sequence, value head),
// fp32: S_start(first) = init (h0 or dht, or zero), S_start(next) = P S_start + E
// with P the segment's transition and E its end state from zero; forward
// segments in ascending order, reverse segments in descending order. One CTA
// per 16 state columns, 256 threads: thread t owns state row k = t % 128 and
// one half of the reduction index j. The transitions do not depend on the
// chain, so each thread holds its 64 values of P's row k in registers and
// loads the next segment's while it works on the current one; S_start's 16
// columns go through shared memory. Each thread forms 16 partial sums over its
// 64 j in order, and the two halves are added in a fixed order.
// ---------------------------------------------------------------------------
constexpr int kCombCols = 16;

__global__ void __launch_bounds__(256, 1) k_tc_seg_combine(Prob p, SegArg sg, int reverse,
                                                           const float* __restrict__ init, TcWs ws) {
    __shared__ float Cs[D * kCombCols];  // S_start[j][v], this CTA's 16 columns
    __shared__ float Hs[D * kCombCols];  // partial sums of the upper j half
    const int tid = threadIdx.x;
    const int k = tid & 127, jh = tid >> 7;  // this thread's row and its half of j
    const int hv = blockIdx.x, n = blockIdx.y, v0 = kCombCols * blockIdx.z, HV = p.HV;
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    const int nseg = (nts + sg.len - 1) / sg.len;
    float cur[16];  // S_start[k][v0 ..] (held by the lower half)
    {
        const float* src = (init && jh == 0) ? init + (((int64_t)n * HV + hv) * D + k) * D + v0 : nullptr;
#pragma unroll
        for (int v = 0; v < 16; ++v) cur[v] = src ? src[v] : 0.f;
    }
    const int64_t head = ((int64_t)n * HV + hv) * sg.M;
    auto seg_at = [&](int s) { return (head + (reverse ? nseg - 1 - s : s)) * D * D; };
    auto load_p = [&](int s, float4 (&dst)[16]) {  // P[k][64 jh .. 64 jh + 63] of step s
        const float4* src = reinterpret_cast<const float4*>(ws.seg_p + seg_at(s) + (int64_t)k * D + 64 * jh);
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = __ldg(src + i);
    };
    float4 pc[16], pn[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pn[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nseg > 1) load_p(0, pc);
    for (int s = 0; s < nseg; ++s) {
        const int64_t at = seg_at(s);
        if (jh == 0) {
            float* st = ws.seg_s0 + at + (int64_t)k * D + v0;
#pragma unroll
            for (int v = 0; v < 16; v += 4)
                *reinterpret_cast<float4*>(st + v) = make_float4(cur[v], cur[v + 1], cur[v + 2], cur[v + 3]);
        }
        if (s + 1 == nseg) break;
        if (s + 2 < nseg) load_p(s + 1, pn);
        float acc[16];
        if (jh == 0) {
            const float* erow = ws.seg_e + at + (int64_t)k * D + v0;
#pragma unroll
            for (int v = 0; v < 16; v += 4) {
                const float4 e4 = *reinterpret_cast<const float4*>(erow + v);
                acc[v] = e4.x;
                acc[v + 1] = e4.y;
                acc[v + 2] = e4.z;
                acc[v + 3] = e4.w;
            }
        } else {
#pragma unroll
            for (int v = 0; v < 16; ++v) acc[v] = 0.f;
        }
        __syncthreads();  // the previous step's reads of Cs and Hs are done
        if (jh == 0) {
#pragma unroll
            for (int v = 0; v < 16; ++v) Cs[k * kCombCols + v] = cur[v];
        }
        __syncthreads();
        const float* crow = Cs + 64 * jh * kCombCols;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            const float4 p4 = pc[j >> 2];
            const float pkj = (j & 3) == 0 ? p4.x : (j & 3) == 1 ? p4.y : (j & 3) == 2 ? p4.z : p4.w;
            const float4* cj = reinterpret_cast<const float4*>(crow + j * kCombCols);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
                const float4 c4 = cj[v4];
                const float2 lo = fma2(bc2(pkj), f2(c4.x, c4.y), f2(acc[4 * v4], acc[4 * v4 + 1]));
                const float2 hi = fma2(bc2(pkj), f2(c4.z, c4.w), f2(acc[4 * v4 + 2], acc[4 * v4 + 3]));
                acc[4 * v4] = lo.x, acc[4 * v4 + 1] = lo.y, acc[4 * v4 + 2] = hi.x, acc[4 * v4 + 3] = hi.y;
            }
        }
        if (jh == 1) {
#pragma unroll
            for (int v = 0; v < 16; ++v) Hs[k * kCombCols + v] = acc[v];
        }
        __syncthreads();
        if (jh == 0) {
#pragma unroll
            for (int v = 0; v < 16; ++v) cur[v] = acc[v] + Hs[k * kCombCols + v];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) pc[i] = pn[i];
    }
}

// ---------------------------------------------------------------------------
// tc_ds_rev: one CTA per (value head, sequence), chunks in reverse; 256
// threads, thread t owns dS row k = t % 128, columns 64 (t / 128) .. +63
// (tc_ds_rev_half: 64 columns per CTA, 32 per thread).
// Chunk inputs are single-buffered in two groups, each refetched for the next
// chunk as soon as its MMAs have consumed it: K^, Q~s, Aqk and dO after the
// first MMA group, w and e^Gamma_C after the second. dDelta is staged in the
// dS tile once the dS_out copy has read it.
// ---------------------------------------------------------------------------
struct RevSm {
    static constexpr int KH = 0, QS = TCD, AQK = 2 * TCD, DO = 2 * TCD + TCC, W = 3 * TCD + TCC, EGC = 4 * TCD + TCC;
    static constexpr int S = EGC + 1024, BARS = S + TDD, END = BARS + 64;
};
constexpr int kRevSmem = 1024 + RevSm::END;

// (sequence n, value head hv, grid z as in state_fwd_body.) The columns of dS evolve independently as well
// (dDelta's column v takes only dS's and dO's column v): NH as in state_fwd_body.
template <int NH>
__device__ __forceinline__ void ds_rev_body(const Prob& p, const float* __restrict__ dht, float* __restrict__ dh0,
                                            const TcWs& ws, const CUtensorMap& tm_do, const SegArg& sg, uint8_t* sm,
                                            int hv, int n, int z, int h) {
    constexpr int CW = 64 * NH, TW = CW / 2;  // dS columns of this CTA and of each thread
    uint8_t* tS = sm + RevSm::S;              // bf16 dS (128 x CW), later dDelta (64 x CW)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + RevSm::BARS);  // group 1, group 2, mma
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
    int* fail = reinterpret_cast<int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = tid & 127, vq = tid >> 7;
    const int cbase = 64 * h + TW * vq;  // this thread's first dS column
    const int HV = p.HV;
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    // segment and mode: 0 checkpoints, 1 end state from zero, 2 transition (dO taken as zero)
    const int m = sg.mode == kSegEnds ? z % sg.M : z;
    const int mode = sg.mode == kSegEnds ? 1 + z / sg.M : 0;
    const int lo = sg.len ? m * sg.len : 0, hi = sg.len ? min(lo + sg.len, nts) : nts;
    if (sg.len && lo >= hi) return;
    const bool ckpt = mode == 0, with_do = mode != 2;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tslot, 2 * CW);  // dDelta [0, CW), dS [CW, 2 CW)
    float S[TW];
    const int64_t seg_at = (((int64_t)n * HV + hv) * sg.M + m) * D * D + (int64_t)k * D + cbase;
    {
        const float* src = nullptr;
        if (mode == 0) src = (hi == nts) ? (dht ? dht + (((int64_t)n * HV + hv) * D + k) * D + cbase : nullptr)
                                         : ws.seg_s0 + seg_at;
#pragma unroll
        for (int j = 0; j < TW; ++j) S[j] = src ? src[j] : (mode == 2 && cbase + j == k ? 1.f : 0.f);
    }
    auto chunk = [&](int it) { return (c0 + it) * HV + hv; };
    auto issue1 = [&](int it) {  // operands of the first MMA group
        const int64_t ch = chunk(it);
        mbar_expect_tx(&bars[0], with_do ? 2 * TCD + TCC + NH * (TCD / 2) : TCD);
        bulk_load(sm + RevSm::KH, ws.kh + ch * TCD, TCD, &bars[0]);
        if (with_do) {
            bulk_load(sm + RevSm::QS, ws.qs + ch * TCD, TCD, &bars[0]);
            bulk_load(sm + RevSm::AQK, ws.aqk + ch * TCC, TCC, &bars[0]);
            const int row = (int)(bos + (int64_t)it * kC);
            for (int x = 0; x < NH; ++x)  // this CTA's columns of dO
                tma_load_3d(sm + RevSm::DO + x * (TCD / 2), &tm_do, 64 * (h + x), hv, row, &bars[0]);
        }
    };
    auto issue2 = [&](int it) {  // w (second MMA group) and e^Gamma_C (state update)
        const int64_t ch = chunk(it);
        mbar_expect_tx(&bars[1], TCD + 512);
        bulk_load(sm + RevSm::W, ws.w + ch * TCD, TCD, &bars[1]);
        bulk_load(sm + RevSm::EGC, ws.egc + ch * D, 512, &bars[1]);
    };
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
    if (tid == 0 && lo < hi) {
        issue1(hi - 1);
        issue2(hi - 1);
    }
    uint32_t mph = 0;
    for (int it = hi - 1; it >= lo; --it) {
        const int64_t ch = chunk(it);
        const uint32_t ph = (uint32_t)(hi - 1 - it) & 1;
        // bf16 copy of dS (row k, this thread's columns): MMA operand and the dS_out checkpoint
#pragma unroll
        for (int c8 = 0; c8 < TW; c8 += 8) st_tile_row8(tS, k, TW * vq + c8, D, S + c8);
        fence_async_smem();
        if (!wait_all(&bars[0], ph, ws.status, 31, fail)) break;
        if (tid == 0) {
            tc_fence_after();
            // dDelta = Aqk^T dO + K^ dS (chunk rows on TMEM lanes, M = 64, N = CW)
            const uint32_t ida = idesc_bf16(64, CW, true, true), idb = idesc_bf16(64, CW, false, true);
            if (with_do)
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_bf16(tmem, desc_mnmajor(smem_u32(sm + RevSm::AQK), kC, ks),
                             desc_mnmajor(smem_u32(sm + RevSm::DO), kC, ks), ida, ks > 0);
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + RevSm::KH), kC, ks), desc_mnmajor(smem_u32(tS), D, ks), idb,
                         with_do || ks > 0);
            // dS accumulator = Q~s^T dO (M = 128, N = CW)
            const uint32_t idc = idesc_bf16(128, CW, true, true);
            if (with_do)
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_bf16(tmem + CW, desc_mnmajor(smem_u32(sm + RevSm::QS), kC, ks),
                             desc_mnmajor(smem_u32(sm + RevSm::DO), kC, ks), idc, ks > 0);
            mma_commit(&bars[2]);
            if (ckpt) {  // (column block h of the 128-row tile)
                bulk_store(ws.dso + ch * TDD + h * (D * 128), tS, D * CW * 2);
                bulk_commit();
            }
        }
        if (tid == 0) bulk_wait_read();  // the dS_out copy has read tS
        if (!wait_all(&bars[2], mph, ws.status, 32, fail)) break;
        mph ^= 1;
        if (tid == 0 && it > lo) issue1(it - 1);  // the first group's operands are consumed
        tc_fence_after();
        {  // dDelta rows into tS: row r = 16 (warp % 4) + lane (lane < 16), CW / 2 columns per warp half
            const int r = 16 * (warp & 3) + lane, cb = (CW / 2) * (warp >> 2);
#pragma unroll
            for (int x = 0; x < CW / 64; ++x) {
                float acc[32];
                tmem_ld32(tmem + lq + cb + 32 * x, acc);
                tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(tS, r, cb + 32 * x + c8, kC, acc + c8);
                }
            }
        }
        tc_fence_before();
        fence_async_smem();
        if (!wait_all(&bars[1], ph, ws.status, 34, fail)) break;
        if (tid == 0) {  // dS accumulator -= w^T dDelta
            tc_fence_after();
            const uint32_t id = idesc_neg_a(idesc_bf16(128, CW, true, true));
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem + CW, desc_mnmajor(smem_u32(sm + RevSm::W), kC, ks), desc_mnmajor(smem_u32(tS), kC, ks),
                         id, with_do || ks > 0);
            mma_commit(&bars[2]);
            if (ckpt) {  // (column block h of the 64-row tile)
                bulk_store(ws.dvn + ch * TCD + h * (kC * 128), tS, kC * CW * 2);
                bulk_commit();
            }
        }
        const float e = reinterpret_cast<const float*>(sm + RevSm::EGC)[k];
        if (tid == 0) bulk_wait_read();  // the dDelta copy has read tS
        if (!wait_all(&bars[2], mph, ws.status, 33, fail)) break;
        mph ^= 1;
        if (tid == 0 && it > lo) issue2(it - 1);  // w and e^Gamma_C are consumed
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < TW / 32; ++x) {
            float acc[32];
            tmem_ld32(tmem + lq + CW + TW * vq + 32 * x, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 v = fma2(bc2(e), f2(S[32 * x + j], S[32 * x + j + 1]), f2(acc[j], acc[j + 1]));
                S[32 * x + j] = v.x, S[32 * x + j + 1] = v.y;
            }
        }
        tc_fence_before();
    }
    if (*(volatile int*)fail == 0) {
        float* dst = mode == 1 ? ws.seg_e + seg_at
                     : mode == 2 ? ws.seg_p + seg_at
                     : (dh0 && lo == 0) ? dh0 + (((int64_t)n * HV + hv) * D + k) * D + cbase
                                        : nullptr;
        if (dst)
#pragma unroll
            for (int j = 0; j < TW; ++j) dst[j] = S[j];
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * CW);
}

__global__ void __launch_bounds__(256, 2) k_tc_ds_rev(Prob p, const float* __restrict__ dht, float* __restrict__ dh0,
                                                       TcWs ws, const __grid_constant__ CUtensorMap tm_do, SegArg sg) {
    extern __shared__ uint8_t smraw[];
    ds_rev_body<2>(p, dht, dh0, ws, tm_do, sg, align1024(smraw), blockIdx.x, sweep_seq(ws, blockIdx.y), blockIdx.z,
                   0);
}
// whole sweeps split by columns: grid x = 2 HV (value head x / 2, column half x % 2)
__global__ void __launch_bounds__(256, 2) k_tc_ds_rev_half(Prob p, const float* __restrict__ dht,
                                                            float* __restrict__ dh0, TcWs ws,
                                                            const __grid_constant__ CUtensorMap tm_do) {
    extern __shared__ uint8_t smraw[];
    ds_rev_body<1>(p, dht, dh0, ws, tm_do, SegArg{0, 1, kSegNone}, align1024(smraw), blockIdx.x >> 1,
                   sweep_seq(ws, blockIdx.y), 0, blockIdx.x & 1);
}

// The forward state pass and the reverse state-gradient pass, whole sweeps, in one launch: grid z = 0 runs
// tc_state_fwd's sweep of (sequence, value head), z = 1 tc_ds_rev's. The reverse pass reads only the
// intra-chunk tiles and dO (not S_in nor delta), so the two sweeps are independent and, when all their
// CTAs are resident at once, run side by side instead of one after the other. NH = 1 splits each sweep
// by columns over two CTAs (grid x = 2 HV: value head x / 2, column half x % 2).
constexpr int kBothSmem = kFwdSmem > kRevSmem ? kFwdSmem : kRevSmem;
template <int NH>
__global__ void __launch_bounds__(256, 2)
    k_tc_state_both(Prob p, const float* __restrict__ h0, const float* __restrict__ dht, float* __restrict__ dh0,
                    TcWs ws, const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do) {
    extern __shared__ uint8_t smraw[];
    const SegArg whole{0, 1, kSegNone};
    const int hv = NH == 2 ? (int)blockIdx.x : (int)blockIdx.x >> 1, h = NH == 2 ? 0 : (int)blockIdx.x & 1;
    const int n = sweep_seq(ws, blockIdx.y);
    if (blockIdx.z == 0)
        state_fwd_body<NH>(p, h0, ws, whole, tm_v, align1024(smraw), hv, n, 0, h);
    else
        ds_rev_body<NH>(p, dht, dh0, ws, tm_do, whole, align1024(smraw), hv, n, 0, h);
}

// ---------------------------------------------------------------------------
// tc_state_load: the backward's replacement of tc_state_fwd when the forward's
// states are given. One CTA per (chunk, value head), 256 threads: S_in (fp32)
// becomes the bf16 checkpoint tile, and delta = INVb V - w S_in with chunk rows
// on TMEM lanes; the same arithmetic as tc_state_fwd on the same state values.
// ---------------------------------------------------------------------------
struct LoadSm {
    static constexpr int W = 0, U = TCD, S = 2 * TCD, IVB = S + TDD, BARS = IVB + TCC, END = BARS + 64;
};
constexpr int kLoadSmem = 1024 + LoadSm::END;

__global__ void __launch_bounds__(256, 3) k_tc_state_load(Prob p, const float* __restrict__ states, TcWs ws,
                                                           const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = align1024(smraw);
    uint8_t* tS = sm + LoadSm::S;
    uint8_t* tU = sm + LoadSm::U;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LoadSm::BARS);  // loads, mma
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
    int* fail = reinterpret_cast<int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ch = (int64_t)blockIdx.x * p.HV + blockIdx.y;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        *fail = 0;
        int64_t r0;
        int c;
        chunk_rows(p, (int64_t)blockIdx.x, r0, c);
        mbar_expect_tx(&bars[0], 2 * TCD + TCC);
        bulk_load(sm + LoadSm::W, ws.w + ch * TCD, TCD, &bars[0]);
        bulk_load(sm + LoadSm::IVB, ws.invb + ch * TCC, TCC, &bars[0]);
        tma_load_3d(tU, &tm_v, 0, (int)blockIdx.y, (int)r0, &bars[0]);
        tma_load_3d(tU + TCD / 2, &tm_v, 64, (int)blockIdx.y, (int)r0, &bars[0]);
    }
    if (warp == 0) tmem_alloc(tslot, 128);
    {  // S_in as bf16: warp w reads whole rows w, w + 8, ..., one 512-byte row per load instruction;
       // lane l converts columns 4l .. 4l + 3
        const float4* src = reinterpret_cast<const float4*>(states + ch * D * D) + lane;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float4 a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = __ldg(src + (warp + 8 * (8 * h + i)) * (D / 4));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = warp + 8 * (8 * h + i);
                *reinterpret_cast<uint2*>(tS + tile_off(r, 4 * lane, D)) =
                    make_uint2(pack2(a[i].x, a[i].y), pack2(a[i].z, a[i].w));
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (!wait_all(&bars[0], 0, ws.status, 51, fail)) goto cleanup;
    if (tid == 0) {  // delta accumulator = -w S_in + INVb V (M = 64, N = 128), the order of tc_state_fwd
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 128, false, true);
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem, desc_kmajor(smem_u32(sm + LoadSm::W), kC, ks), desc_mnmajor(smem_u32(tS), D, ks),
                     idesc_neg_a(id), ks > 0);
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tmem, desc_kmajor(smem_u32(sm + LoadSm::IVB), kC, ks), desc_mnmajor(smem_u32(tU), kC, ks), id,
                     1);
        mma_commit(&bars[1]);
        bulk_store(ws.sin + ch * TDD, tS, TDD);
        bulk_commit();
    }
    if (!wait_all(&bars[1], 0, ws.status, 52, fail)) goto cleanup;
    tc_fence_after();
    {  // delta (bf16) in place of V: row r = 16 (warp % 4) + lane (lane < 16), 64 columns per warp half
        const int r = 16 * (warp & 3) + lane, cb = 64 * (warp >> 2);
        const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float acc[32];
            tmem_ld32(tmem + lq + cb + 32 * h, acc);
            tmem_ld_wait();
            if (lane < 16) {
#pragma unroll
                for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(tU, r, cb + 32 * h + c8, kC, acc + c8);
            }
        }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
        bulk_store(ws.vn + ch * TCD, tU, TCD);
        bulk_commit();
    }
cleanup:
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// tc_fwd_out: the forward's state pass with the output fused in. One CTA per
// (value head, sequence), 256 threads, thread t owns state row k = t % 128,
// columns 64 (t / 128) .. +63. Per chunk: delta = INVb V - w S (chunk rows on
// TMEM lanes, in place of V), then S <- e^(Gamma_C) S + K^^T delta and
// o = (scale Q~) S + Aqk delta in one MMA group; o leaves as bf16 rows. Inputs
// are single-buffered in two groups: w and INVb are refetched once the delta
// MMA has consumed them, the rest once the state and output MMAs have. Two
// CTAs per SM: 112.6 KB of shared memory each, from a 1024-byte aligned base
// (no alignment slack). With a saved-context workspace (ws.sin, ws.vn set) it
// also stores every chunk's bf16 S_in and delta tiles, the ones the backward's
// state pass would recompute.
// ---------------------------------------------------------------------------
struct FoSm {
    static constexpr int W = 0, IVB = TCD, KH = TCD + TCC, QS = 2 * TCD + TCC, U = 3 * TCD + TCC;
    static constexpr int AQK = 4 * TCD + TCC, S = 4 * TCD + 2 * TCC, EGC = S + TDD, BARS = EGC + 512, END = BARS + 64;
};
constexpr int kFoSmem = FoSm::END;

// (sequence n, value head hv, segment z; NH and the column half h as in state_fwd_body: o's column v takes
// only S's and delta's column v)
template <int NH>
__device__ __forceinline__ void fwd_out_body(const Prob& p, const float* __restrict__ h0, float* __restrict__ ht,
                                             float* __restrict__ states, bf16* __restrict__ o, const TcWs& ws,
                                             const SegArg& sg, const CUtensorMap& tm_v, uint8_t* sm, int hv, int n,
                                             int z, int h) {
    constexpr int CW = 64 * NH, TW = CW / 2;  // state columns of this CTA and of each thread
    uint8_t* tS = sm + FoSm::S;
    uint8_t* tU = sm + FoSm::U;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + FoSm::BARS);  // w, group 2, mma
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
    int* fail = reinterpret_cast<int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = tid & 127, vq = tid >> 7;
    const int cbase = 64 * h + TW * vq;  // this thread's first state column
    const int HV = p.HV;
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    const int m = z;  // segment (kSegCkpt) or the whole sequence (kSegNone)
    const int lo = sg.len ? m * sg.len : 0, hi = sg.len ? min(lo + sg.len, nts) : nts;
    if (sg.len && lo >= hi) return;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *fail = (smem_u32(sm) & 1023u) ? 1 : 0;  // tiles need a 1024-byte aligned base
        if (*fail) *(volatile int*)ws.status = 70;
    }
    if (warp == 0) tmem_alloc(tslot, 2 * CW);  // delta and then o [0, CW), state [CW, 2 CW)
    float S[TW];
    {
        const float* src = lo == 0 ? (h0 ? h0 + (((int64_t)n * HV + hv) * D + k) * D + cbase : nullptr)
                                   : ws.seg_s0 + (((int64_t)n * HV + hv) * sg.M + m) * D * D + (int64_t)k * D + cbase;
#pragma unroll
        for (int j = 0; j < TW; ++j) S[j] = src ? src[j] : 0.f;
    }
    auto chunk = [&](int it) { return (c0 + it) * HV + hv; };
    auto issue_w = [&](int it) {  // w and INVb
        mbar_expect_tx(&bars[0], TCD + TCC);
        bulk_load(sm + FoSm::W, ws.w + chunk(it) * TCD, TCD, &bars[0]);
        bulk_load(sm + FoSm::IVB, ws.invb + chunk(it) * TCC, TCC, &bars[0]);
    };
    auto issue_g2 = [&](int it) {  // K^, scale Q~, V (TMA; this CTA's columns), Aqk, e^Gamma_C
        const int64_t ch = chunk(it);
        const int row = (int)(bos + (int64_t)it * kC);
        mbar_expect_tx(&bars[1], 2 * TCD + NH * (TCD / 2) + TCC + 512);
        bulk_load(sm + FoSm::KH, ws.kh + ch * TCD, TCD, &bars[1]);
        bulk_load(sm + FoSm::QS, ws.qs + ch * TCD, TCD, &bars[1]);
        for (int x = 0; x < NH; ++x) tma_load_3d(tU + x * (TCD / 2), &tm_v, 64 * (h + x), hv, row, &bars[1]);
        bulk_load(sm + FoSm::AQK, ws.aqk + ch * TCC, TCC, &bars[1]);
        bulk_load(sm + FoSm::EGC, ws.egc + ch * D, 512, &bars[1]);
    };
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
    const bool run = *(volatile int*)fail == 0;
    const bool save = ws.sin != nullptr && ws.vn != nullptr;
    if (tid == 0 && lo < hi && run) {
        issue_w(lo);
        issue_g2(lo);
    }
    uint32_t mph = 0;
    for (int it = lo; it < hi && run; ++it) {
        const int64_t ch = chunk(it);
        const uint32_t ph = (uint32_t)(it - lo) & 1;
        // bf16 copy of S (row k, this thread's columns): operand of the delta and output MMAs
#pragma unroll
        for (int c8 = 0; c8 < TW; c8 += 8) st_tile_row8(tS, k, TW * vq + c8, D, S + c8);
        fence_async_smem();
        if (states) {  // the fp32 state entering this chunk, [chunk, HV, K, V]
            float4* dst = reinterpret_cast<float4*>(states + (ch * D + k) * D + cbase);
#pragma unroll
            for (int j = 0; j < TW / 4; ++j) dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
        }
        if (!wait_all2(&bars[0], ph, 71, &bars[1], ph, 73, ws.status, fail)) break;
        // delta accumulator = -w S + INVb V (M = 64, N = CW)
        const uint32_t idd = idesc_bf16(64, CW, false, true);
        if (tid == 0) {
            tc_fence_after();
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + FoSm::W), kC, ks), desc_mnmajor(smem_u32(tS), D, ks),
                         idesc_neg_a(idd), ks > 0);
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + FoSm::IVB), kC, ks), desc_mnmajor(smem_u32(tU), kC, ks),
                         idd, 1);
            mma_commit(&bars[2]);
            if (save) {  // (column block h of the 128-row tile)
                bulk_store(ws.sin + ch * TDD + h * (D * 128), tS, D * CW * 2);
                bulk_commit();
            }
        }
        if (!wait_all(&bars[2], mph, ws.status, 72, fail)) break;
        mph ^= 1;
        if (tid == 0 && it + 1 < hi) issue_w(it + 1);  // w and INVb are consumed
        tc_fence_after();
        // M = 64 row of this lane, and this warp's half of the CTA's columns
        const int r = 16 * (warp & 3) + lane, cb = (CW / 2) * (warp >> 2);
        {  // delta (bf16) in place of V
#pragma unroll
            for (int x = 0; x < CW / 64; ++x) {
                float acc[32];
                tmem_ld32(tmem + lq + cb + 32 * x, acc);
                tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(tU, r, cb + 32 * x + c8, kC, acc + c8);
                }
            }
        }
        tc_fence_before();
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // S accumulator = K^^T delta (M = 128, N = CW)
            const uint32_t is = idesc_bf16(128, CW, true, true);
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem + CW, desc_mnmajor(smem_u32(sm + FoSm::KH), kC, ks), desc_mnmajor(smem_u32(tU), kC, ks),
                         is, ks > 0);
            // o accumulator (in the delta columns) = (scale Q~) S + Aqk delta (M = 64, N = CW)
            const uint32_t io = idesc_bf16(64, CW, false, true);
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + FoSm::QS), kC, ks), desc_mnmajor(smem_u32(tS), D, ks), io,
                         ks > 0);
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + FoSm::AQK), kC, ks), desc_mnmajor(smem_u32(tU), kC, ks), io,
                         1);
            mma_commit(&bars[2]);
            if (save) {  // (column block h of the 64-row tile)
                bulk_store(ws.vn + ch * TCD + h * (kC * 128), tU, kC * CW * 2);
                bulk_commit();
                bulk_wait_read();  // the S_in and delta copies have read tS and tU (both rewritten next)
            }
        }
        const float e = reinterpret_cast<const float*>(sm + FoSm::EGC)[k];
        if (!wait_all(&bars[2], mph, ws.status, 74, fail)) break;
        mph ^= 1;
        if (tid == 0 && it + 1 < hi) issue_g2(it + 1);  // K^, Q~s, u / delta, Aqk, e^Gamma_C are consumed
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < TW / 32; ++x) {  // state update
            float acc[32];
            tmem_ld32(tmem + lq + CW + TW * vq + 32 * x, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) S[32 * x + j] = fmaf(e, S[32 * x + j], acc[j]);
        }
        {  // o rows (bf16)
            const int64_t r0 = bos + (int64_t)it * kC;
            const int c = (int)((eos - r0) < kC ? (eos - r0) : kC);
#pragma unroll
            for (int y = 0; y < CW / 32; ++y) {  // 16 columns at a time (the state values stay in registers)
                float x[16];
                tmem_ld16(tmem + lq + cb + 16 * y, x);
                tmem_ld_wait();
                if (lane < 16 && r < c) {
                    bf16* dst = o + ((r0 + r) * HV + hv) * D + 64 * h + cb + 16 * y;
#pragma unroll
                    for (int u = 0; u < 16; u += 8) {
                        uint4 vv;
                        vv.x = pack2(x[u], x[u + 1]);
                        vv.y = pack2(x[u + 2], x[u + 3]);
                        vv.z = pack2(x[u + 4], x[u + 5]);
                        vv.w = pack2(x[u + 6], x[u + 7]);
                        *reinterpret_cast<uint4*>(dst + u) = vv;
                    }
                }
            }
        }
        tc_fence_before();
    }
    if (ht && hi == nts && *(volatile int*)fail == 0) {
        float* dst = ht + (((int64_t)n * HV + hv) * D + k) * D + cbase;
#pragma unroll
        for (int j = 0; j < TW; ++j) dst[j] = S[j];
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * CW);
}

__global__ void __launch_bounds__(256, 2) k_tc_fwd_out(Prob p, const float* __restrict__ h0, float* __restrict__ ht,
                                                        float* __restrict__ states, bf16* __restrict__ o, TcWs ws,
                                                        SegArg sg, const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ __align__(1024) uint8_t sm[];
    fwd_out_body<2>(p, h0, ht, states, o, ws, sg, tm_v, sm, blockIdx.x, sweep_seq(ws, blockIdx.y), blockIdx.z, 0);
}
// whole sweeps split by columns: grid x = 2 HV (value head x / 2, column half x % 2)
__global__ void __launch_bounds__(256, 2) k_tc_fwd_out_half(Prob p, const float* __restrict__ h0,
                                                             float* __restrict__ ht, float* __restrict__ states,
                                                             bf16* __restrict__ o, TcWs ws,
                                                             const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ __align__(1024) uint8_t sm[];
    fwd_out_body<1>(p, h0, ht, states, o, ws, SegArg{0, 1, kSegNone}, tm_v, sm, blockIdx.x >> 1,
                    sweep_seq(ws, blockIdx.y), 0, blockIdx.x & 1);
}

// Packed sequences: order[rank] = sequence, by decreasing chunk count (ties by index), so that the state
// passes launch the sweeps of the longest sequences first and the short ones fill in behind them. Thread i
// ranks sequence i against all others, N in tiles of 256 through shared memory.
__global__ void __launch_bounds__(256) k_seq_order(const int64_t* __restrict__ cu, int N, int* __restrict__ order) {
    __shared__ int tile[256];
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    auto chunks = [&](int j) { return (int)((cu[j + 1] - cu[j] + kC - 1) / kC); };
    const int ci = i < N ? chunks(i) : 0;
    int rank = 0;
    for (int j0 = 0; j0 < N; j0 += 256) {
        const int j = j0 + (int)threadIdx.x;
        tile[threadIdx.x] = j < N ? chunks(j) : -1;
        __syncthreads();
        const int m = N - j0 < 256 ? N - j0 : 256;
        for (int t = 0; t < m; ++t) {
            const int cj = tile[t];
            rank += (cj > ci || (cj == ci && j0 + t < i)) ? 1 : 0;
        }
        __syncthreads();
    }
    if (i < N) order[rank] = i;
}

template <typename F>
cudaError_t set_smem(F* f, int bytes) {
    return cudaFuncSetAttribute(reinterpret_cast<const void*>(f), cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

bool tc_path_ok(const Prob& p, bool bf16) { return bf16 && p.K == D && p.V == D; }

// Dense batches whose (sequence, value head) sweeps cannot fill the GPU and whose sequences are long
// run the state passes in segments of at least 32 chunks. (Shorter sequences gain nothing: a segment
// step of the chain costs about as much as the chunk steps it saves.) The segment count M minimises a
// pass's critical path in chunk steps: the "ends" launch (2 S M CTAs for S sweeps) and the checkpoint
// launch (S M CTAs) each take ceil(CTAs / slots) waves of ceil(chunks / M) steps, slots = two CTAs per
// SM; the combine chain adds about 2.5 chunk steps per segment.
SegPlan seg_plan(const Prob& p) {
    SegPlan sp{0, 1};
    const int64_t sweeps = (int64_t)p.B * p.HV;
    if (p.cu || p.K != D || p.V != D || sweeps > 64 || p.NTs < 128) return sp;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || nsm <= 0)
        nsm = 152;
    const int64_t slots = 2 * (int64_t)nsm;
    int M = 2;
    double best = 0.0;
    for (int m = 2; m <= p.NTs / 32; ++m) {
        const int64_t len = (p.NTs + m - 1) / m;
        const double cost = (double)(((2 * sweeps * m + slots - 1) / slots + (sweeps * m + slots - 1) / slots) * len) +
                            2.5 * m;
        if (m == 2 || cost < best) {
            best = cost;
            M = m;
        }
    }
    sp.len = (p.NTs + M - 1) / M;
    sp.M = (p.NTs + sp.len - 1) / sp.len;
    return sp;
}

namespace {

// Packed batches of up to kOrderMaxSeqs sequences get the longest-first sweep order (k_seq_order, one
// launch of a few microseconds); other batches keep the natural order (seq_order null).
constexpr int kOrderMaxSeqs = 4096;
TcWs order_sweeps(const Prob& p, TcWs ws, cudaStream_t st) {
    if (!p.cu || p.N < 2 || p.N > kOrderMaxSeqs || !ws.seq_order) {
        ws.seq_order = nullptr;
        return ws;
    }
    k_seq_order<<<(p.N + 255) / 256, 256, 0, st>>>(p.cu, p.N, ws.seq_order);
    note_launch("tc_seq_order", st);
    return ws;
}

cudaError_t launch_intra(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st) {
    cudaError_t e;
    if ((e = set_smem(k_tc_intra, kIntraSmem)) != cudaSuccess) return e;
    if (p.NT == 0) return cudaSuccess;
    const int64_t rows = (int64_t)p.B * p.T;
    IntraMaps im;
    memset(&im, 0, sizeof(im));
    const uint64_t rq = (uint64_t)p.H * D * 2;
    if (!make_tmap_bf16_3d(&im.q, io.q, D, p.H, rows, D * 2, rq, 64, 1, kC) ||
        !make_tmap_bf16_3d(&im.k, io.k, D, p.H, rows, D * 2, rq, 64, 1, kC))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t items = p.NT * p.HV;  // persistent: two CTAs per SM, items dealt round-robin
    const unsigned grid = (unsigned)(items < 2 * (int64_t)nsm ? items : 2 * (int64_t)nsm);
    k_tc_intra<<<grid, 256, kIntraSmem, st>>>(p, io.g, (const bf16*)io.beta, ws, im);
    note_launch("tc_intra", st);
    return cudaSuccess;
}

}  // namespace

// Tensor map of V [rows, HV, 128] bf16 in 64 x 64 boxes (one 64-column half of a chunk's rows).
static bool make_tmap_v(CUtensorMap* m, const Prob& p, const void* v) {
    memset(m, 0, sizeof(*m));
    const int64_t rows = (int64_t)p.B * p.T;
    return rows == 0 || make_tmap_bf16_3d(m, v, D, (uint64_t)p.HV, (uint64_t)rows, (uint64_t)D * 2,
                                          (uint64_t)p.HV * D * 2, 64, 1, kC);
}

cudaError_t tc_fwd(const Prob& p, const IO& io, const TcWs& ws_in, cudaStream_t st) {
    cudaError_t e;
    const TcWs ws = order_sweeps(p, ws_in, st);
    if ((e = set_smem(k_tc_fwd_out, kFoSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_fwd_out_half, kFoSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_state_fwd, kFwdSmem)) != cudaSuccess) return e;
    CUtensorMap tm_v;
    if (!make_tmap_v(&tm_v, p, io.v)) return cudaErrorInvalidValue;
    if ((e = launch_intra(p, io, ws, st)) != cudaSuccess) return e;
    const SegPlan sp = seg_plan(p);
    if (sp.len) {  // segment ends and transitions, their chain, then o per segment
        const SegArg ends{sp.len, sp.M, kSegEnds};
        k_tc_state_fwd<<<dim3(p.HV, p.N, 2 * sp.M), 256, kFwdSmem, st>>>(p, io.h0, ws, ends, tm_v);
        note_launch("tc_state_fwd_seg", st);
        k_tc_seg_combine<<<dim3(p.HV, p.N, D / kCombCols), 256, 0, st>>>(p, ends, 0, io.h0, ws);
        note_launch("tc_seg_combine", st);
    }
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (!sp.len && (int64_t)p.N * p.HV <= nsm) {  // few whole sweeps: each split by columns over two CTAs
        k_tc_fwd_out_half<<<dim3(2 * p.HV, p.N), 256, kFoSmem, st>>>(p, io.h0, io.ht, io.states_out, (bf16*)io.o, ws,
                                                                     tm_v);
        note_launch("tc_fwd_out_vhalf", st);
    } else {
        k_tc_fwd_out<<<dim3(p.HV, p.N, sp.M), 256, kFoSmem, st>>>(p, io.h0, io.ht, io.states_out, (bf16*)io.o, ws,
                                                                  SegArg{sp.len, sp.M, sp.len ? kSegCkpt : kSegNone},
                                                                  tm_v);
        note_launch("tc_fwd_out", st);
    }
    return cudaGetLastError();
}

cudaError_t tc_bwd(const Prob& p, const IO& io, const TcWs& ws_in, cudaStream_t st, int stages, bool from_saved,
                   bool fused) {
    cudaError_t e;
    const TcWs ws = stages >= 2 ? order_sweeps(p, ws_in, st) : ws_in;
    if ((e = set_smem(k_tc_state_fwd, kFwdSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_state_fwd_half, kFwdSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_state_load, kLoadSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_ds_rev, kRevSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_ds_rev_half, kRevSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_state_both<2>, kBothSmem)) != cudaSuccess) return e;
    if ((e = set_smem(k_tc_state_both<1>, kBothSmem)) != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.B * p.T;
    CUtensorMap tm_do;
    memset(&tm_do, 0, sizeof(tm_do));
    if (rows > 0 && !make_tmap_bf16_3d(&tm_do, io.d_o, D, (uint64_t)p.HV, (uint64_t)rows, (uint64_t)D * 2,
                                       (uint64_t)p.HV * D * 2, 64, 1, kC))
        return cudaErrorInvalidValue;
    CUtensorMap tm_v;
    if (!make_tmap_v(&tm_v, p, io.v)) return cudaErrorInvalidValue;
    if (stages >= 1 && !from_saved && (e = launch_intra(p, io, ws, st)) != cudaSuccess) return e;
    const SegPlan sp = seg_plan(p);
    const SegArg ends{sp.len, sp.M, kSegEnds}, ckpt{sp.len, sp.M, kSegCkpt}, whole{0, 1, kSegNone};
    // the two state passes side by side when each has at most one sweep per SM (both fit at two CTAs per SM),
    // and with each sweep split by columns over two CTAs when that still fits
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t sweeps = (int64_t)p.N * p.HV;
    const bool both = stages >= 3 && !fused && !from_saved && !io.states_in && !sp.len && sweeps <= nsm;
    if (both) {
        if (2 * sweeps <= nsm) {
            k_tc_state_both<1><<<dim3(2 * p.HV, p.N, 2), 256, kBothSmem, st>>>(p, io.h0, io.dht, io.dh0, ws, tm_v,
                                                                                tm_do);
            note_launch("tc_state_both_vhalf", st);
        } else {
            k_tc_state_both<2><<<dim3(p.HV, p.N, 2), 256, kBothSmem, st>>>(p, io.h0, io.dht, io.dh0, ws, tm_v, tm_do);
            note_launch("tc_state_both", st);
        }
        if (stages >= 4) {
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            return tc_grads(p, io, ws, st);
        }
        return cudaGetLastError();
    }
    if (stages >= 2 && !from_saved) {
        if (io.states_in) {  // the forward's saved states: no sequential recompute
            if (p.NT > 0) {
                k_tc_state_load<<<dim3((unsigned)p.NT, p.HV), 256, kLoadSmem, st>>>(p, io.states_in, ws, tm_v);
                note_launch("tc_state_load", st);
            }
        } else if (sp.len) {  // two-level: segment ends and transitions, their chain, then the checkpoints
            k_tc_state_fwd<<<dim3(p.HV, p.N, 2 * sp.M), 256, kFwdSmem, st>>>(p, io.h0, ws, ends, tm_v);
            note_launch("tc_state_fwd_seg", st);
            k_tc_seg_combine<<<dim3(p.HV, p.N, D / kCombCols), 256, 0, st>>>(p, ends, 0, io.h0, ws);
            note_launch("tc_seg_combine", st);
            k_tc_state_fwd<<<dim3(p.HV, p.N, sp.M), 256, kFwdSmem, st>>>(p, io.h0, ws, ckpt, tm_v);
            note_launch("tc_state_fwd", st);
        } else if (sweeps <= nsm) {  // a pass alone, each sweep split by columns (two CTAs per SM at most)
            k_tc_state_fwd_half<<<dim3(2 * p.HV, p.N), 256, kFwdSmem, st>>>(p, io.h0, ws, tm_v);
            note_launch("tc_state_fwd_vhalf", st);
        } else {
            k_tc_state_fwd<<<dim3(p.HV, p.N), 256, kFwdSmem, st>>>(p, io.h0, ws, whole, tm_v);
            note_launch("tc_state_fwd", st);
        }
    }
    if (fused) {  // the reverse pass and the gradients in one launch (whole sweeps)
        if (stages < 4) return cudaGetLastError();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return tc_rev_fused(p, io, ws, st);
    }
    if (stages >= 3) {
        if (sp.len) {
            k_tc_ds_rev<<<dim3(p.HV, p.N, 2 * sp.M), 256, kRevSmem, st>>>(p, io.dht, io.dh0, ws, tm_do, ends);
            note_launch("tc_ds_rev_seg", st);
            k_tc_seg_combine<<<dim3(p.HV, p.N, D / kCombCols), 256, 0, st>>>(p, ends, 1, io.dht, ws);
            note_launch("tc_seg_combine", st);
            k_tc_ds_rev<<<dim3(p.HV, p.N, sp.M), 256, kRevSmem, st>>>(p, io.dht, io.dh0, ws, tm_do, ckpt);
            note_launch("tc_ds_rev", st);
        } else if (sweeps <= nsm) {
            k_tc_ds_rev_half<<<dim3(2 * p.HV, p.N), 256, kRevSmem, st>>>(p, io.dht, io.dh0, ws, tm_do);
            note_launch("tc_ds_rev_vhalf", st);
        } else {
            k_tc_ds_rev<<<dim3(p.HV, p.N), 256, kRevSmem, st>>>(p, io.dht, io.dh0, ws, tm_do, whole);
            note_launch("tc_ds_rev", st);
        }
    }
    if (stages >= 4) {
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return tc_grads(p, io, ws, st);
    }
    return cudaGetLastError();
}

}  // namespace kda
