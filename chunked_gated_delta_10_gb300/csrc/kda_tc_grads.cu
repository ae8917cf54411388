// Tensor-core per-chunk gradient kernel of the chunked KDA backward (bf16,
// K = V = 128, chunks of 64), with the grouped-value-head sum of dq and dk.
//
// Persistent: one CTA per SM (512 SIMT threads and a producer warp) walks
// (chunk, value head) items and prefetches the next item's inputs. Inputs: q, k, v, dO, g (TMA),
// and from the earlier stages delta, d_delta, S_in, dS_out, INV, e^Gamma_C
// (bulk copies of bf16 tiles). With Kr = k e^(G-Gref), Kc = k e^(Gref-G),
// Qr = q e^(G-Gref), K~ = k e^G, Q~ = q e^G, K^ = k e^(G_C-G) (natural-log
// Gamma, Gref = middle row), the kernel evaluates, in three dependent MMA
// phases (fp32 accumulators in TMEM, columns noted):
//
//  A  [dQ~^T | -dw^T] = S_in [dO; d_delta]^T [0,128)
//     [V; delta] [dO; d_delta]^T [128,256): V d_delta^T (rows 0..63, columns 192..255),
//        dAqk^T = delta dO^T and T^T = delta d_delta^T (rows 64..127)
//     dK^^T = dS_out delta^T [256,320)   dXv = INV^T d_delta [320,448)   (Gamma2 [448,512))
//  B  PR^T = V d_delta^T + K~ dw^T [192,256)   dAkk = -INV^T T [64,128)
//     dXk^T = dw^T INV [128,192)   Mkk = Kr Kc^T [320,384)   dQr^T = Kc^T dN^T [384,448)
//  E  dKr^T = Kc^T dM^T [64,128)   dKc^T = Qr^T dN + Kr^T dM [320,384)
//
// T stands for dINV INV^T with dINV = (P + R) diag(beta) = (d_delta V^T +
// dw K~^T) diag(beta): since INV diag(beta) V = u, INV diag(beta) K~ = w,
// dw = -d_delta S_in^T and delta = u - w S_in, it equals d_delta delta^T and
// needs no dINV product of its own. Here dN = scale tril0(dAqk) and dM = diag(beta) tril-1(dAkk). The
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
    // v and delta, and dO and d_delta, interleave by 64-column half (v h0, delta h0, v h1, delta h1; half
    // stride 2 * 8 KB), so that each pair is one 128-row operand: [V; delta] and [dO; d_delta]
    static constexpr int Q = 0, K = TCD, V = 2 * TCD, DL = 2 * TCD + TCD / 2, DO = 4 * TCD, DDL = 4 * TCD + TCD / 2;
    static constexpr int SIN = 6 * TCD, DSO = SIN + TDD;
    // after phase A the S_in / dS_out area holds the decayed factor tiles, stored transposed
    static constexpr int KR = SIN, KC = SIN + TCD, QR = SIN + 2 * TCD, KT = SIN + 3 * TCD;
    static constexpr int DW = DSO + TDD;
    static constexpr int INV = DW + TCD, DN = INV + TCC, DM = DN + TCC, TT = DM + 2 * TCC;  // DM .. TT: g tile part
    // the g tile (64 x 128 fp32) of a chunk lands on DN .. TT, which the previous chunk no longer needs after phase E
    static constexpr int GT = DN;
    // dN = dN_hi + dN_lo as a bf16 pair (phases B and E take both); dM takes the first 8 KB of its region
    static constexpr int DNL = DM + TCC;
    static constexpr int EGC = TT + TCC, BETA = EGC + 1024, XRD = BETA + 512, BARS = XRD + 2048;
    // cumsum quarter totals and the reference / last-row gates (chunk start), in a region of their own: the
    // warps write the dw tile in epilogue A without waiting for each other to have read them
    static constexpr int XTOT = BARS + 128, XRG = XTOT + 2048;
    static constexpr int END = XRG + 1024;
    // scratch in the dw tile while that tile is dead: dbeta partials (epilogues B and D), Gamma_C terms and dg
    // quarter totals (final epilogue)
    static constexpr int XDB = DW + 4096, XGC = DW + 8192, XT1 = DW + 10240;
};
constexpr int kGradsSmem = 1024 + GS::END;

// Shared-memory map of the sweep CTA of a fused reverse cluster: the chunk inputs K^, scale Q~, Aqk, dO, w,
// e^Gamma_C, then up to three bf16 dS_out tiles and three d_delta tiles (item i in buffer i % (NG + 1) with
// NG gradient CTAs: tiles in flight to the gradient CTAs while the next is written). Barriers: [0] K^, Q~,
// Aqk, dO landed; [1] w, e^Gamma_C landed; [2] MMA; [kFree + g] an item of gradient CTA g finished (remote
// arrivals).
struct RevF {
    static constexpr int KH = 0, QS = TCD, AQK = 2 * TCD, DO = 2 * TCD + TCC, W = 3 * TCD + TCC, EGC = 4 * TCD + TCC;
    static constexpr int kBufs = 3;
    static constexpr int S0 = EGC + 1024, DD0 = S0 + kBufs * TDD, BARS = DD0 + kBufs * TCD, END = BARS + 64;
    static constexpr int kFree = 3;  // [3], [4]
};
static_assert(RevF::END <= GS::END, "the sweep CTA fits the gradient CTA's shared memory");

struct GradMaps {
    CUtensorMap q, k, v, d_o, g;
};

// One work item = one (chunk, value head), index w = chunk * HV + hv (the kernel says how items are dealt
// to its persistent CTAs).
struct Item {
    int64_t r0, ch;
    int hv, h, c, valid;
};
// An item whose rows were looked up earlier and left in shared memory (r0, c at xrows[0], xrows[1]).
__device__ __forceinline__ Item handed_item(const Prob& p, int64_t w, const int64_t* xrows) {
    Item it;
    it.hv = (int)(w % p.HV);
    it.h = it.hv / (p.HV / p.H);
    it.ch = w;
    it.valid = 1;
    it.r0 = xrows[0];
    it.c = (int)xrows[1];
    return it;
}
__device__ __forceinline__ Item make_item(const Prob& p, int64_t w, bool valid) {
    Item it;
    it.hv = (int)(w % p.HV);
    it.h = it.hv / (p.HV / p.H);
    it.ch = w;
    it.valid = valid ? 1 : 0;
    chunk_rows(p, w / p.HV, it.r0, it.c);
    return it;
}

// Persistent, one CTA per SM: 512 SIMT threads (warps 0..15) and one producer warp (warp 16).
// The producer's lane 0 issues every TMA copy and tensor-core MMA; an MMA's issue runs only a
// couple of instructions ahead of its execution, so the issuing thread is held for about the
// length of a phase, and in a warp of its own it holds nobody else. Mbarriers carry the hand-offs
// between the two: inputs of an item (by item parity) and MMA phases A / B / E complete, which each
// SIMT warp waits for on its own (phase A and, with grouped value heads, phase E as a group), and
// operands of phase B / phase E written and the accumulators of the final epilogue read (TMEM free),
// which each SIMT warp signals on its own once its part is done: phase A of the next item then runs
// while the SIMT threads finish the current one. The SIMT threads meet on barrier 1
// (group_sync<512>) three times per item: for the cumsum's quarter totals, with the phase-A wait (the
// reference rows, and S_in / dS_out no longer read before the factor pass overwrites them), and for
// dg's cross-quarter sums. A time-out of a per-warp wait sets the failure flag, which the next of
// these barriers reads.
// Channel-oriented work: thread (d = tid % 128, quarter = tid / 128) owns key channel d for chunk
// rows 16 * quarter .. 16 * quarter + 15. Row-oriented work on M = 64 accumulators: row r =
// 16 * (warp % 4) + lane (lane < 16), column quarter warp / 4. Every cross-thread sum is
// combined in a fixed order. The inputs of the next item are fetched in four groups, each as
// soon as the current item has consumed its regions: dO, delta, v and d_delta after phase A;
// INV after epilogue B/D; S_in, dS_out, g and e^Gamma_C after phase E; q and k once the final
// epilogue has read them.
constexpr int kSimt = 512, kProducerWarp = kSimt / 32, kGradsThreads = kSimt + 32;
// gradient CTAs per sweep CTA in the fused reverse kernel
constexpr int kFusedGradCtas = 2;

// GROUPED: HV = G H with G > 1 (the G value heads of a key head each add to its dq and dk).
// FUSED: a gradient CTA (cluster rank frank) of a fused reverse cluster (below): items fw0, fw0 - fstep, ...,
// down to wlo (its share of the chunks of one sweep, last first), with d_delta and dS_out pushed by the sweep
// CTA instead of loaded.
template <bool GROUPED, bool FUSED>
__device__ __forceinline__ void grads_body(const Prob& p, const bf16* __restrict__ beta, bf16* __restrict__ dq_out,
                                           bf16* __restrict__ dk_out, bf16* __restrict__ dv_out,
                                           float* __restrict__ dg_out, bf16* __restrict__ db_out, const TcWs& ws,
                                           const GradMaps& maps, uint8_t* sm, int64_t fw0, int64_t wlo,
                                           int64_t fstep = 0, int frank = 1) {
    // [0, 1] inputs (by item parity); [2] phase A, [3] phase B, [4] phase E complete; operands
    // written: [8] of phase B's first part, [5] of its second part, [6] of phase E; [7] accumulators read
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + GS::BARS);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 9);
    int* fail = reinterpret_cast<int*>(tslot + 1);  // written by SIMT warp 0 only
    auto S = [&](int off) { return smem_u32(sm + off); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HV = p.HV, H = p.H, G = GROUPED ? HV / H : 1;
    // this CTA's items, round-robin: items b, b + grid, ...; with grouped value heads (w = group * G + j)
    // groups b, b + grid, ..., each group's G items back to back, so that this CTA keeps their running
    // dq / dk sum
    auto next_w = [&](int64_t w) -> int64_t {
        if (FUSED) return w - fstep;
        return GROUPED ? ((w + 1) % G ? w + 1 : w + 1 + (int64_t)(gridDim.x - 1) * G) : w + gridDim.x;
    };
    const int64_t w0 = FUSED ? fw0 : GROUPED ? (int64_t)blockIdx.x * G : blockIdx.x;
    const int64_t total = p.NT * HV;
    auto live = [&](int64_t w) { return FUSED ? w >= wlo : w < total; };

    if (tid == 0) {
        mbar_init(&bars[0], 4);  // four input groups per item
        mbar_init(&bars[1], 4);
        // [2, 3, 4] by the producer's MMA commits; [5, 6, 7, 8] by each SIMT warp
        for (int x = 2; x < 9; ++x) mbar_init(&bars[x], x >= 5 ? kSimt / 32 : 1);
        fence_mbar_init();
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (FUSED) cluster_sync();  // the sweep CTA's barriers are initialised, and ours for its copies
    const uint32_t tmem = *tslot;

    if (warp == kProducerWarp) {
        if (lane == 0) {  // the producer thread; lanes 1 .. 31 wait at the warp barrier below
            auto pwait = [&](uint64_t* b, uint32_t parity, int code) { return mbar_wait(b, parity, ws.status, code); };
            // the four input groups of an item into input barrier `b`
            auto issue_a = [&](const Item& n, uint64_t* b) {  // dO, delta, v, d_delta
                mbar_expect_tx(b, 4 * TCD);
                for (int x = 0; x < 2; ++x) {
                    tma_load_3d(sm + GS::DO + x * TCD, &maps.d_o, 64 * x, n.hv, (int)n.r0, b);
                    tma_load_3d(sm + GS::V + x * TCD, &maps.v, 64 * x, n.hv, (int)n.r0, b);
                    bulk_load(sm + GS::DL + x * TCD, ws.vn + n.ch * TCD + x * (TCD / 2), TCD / 2, b);
                    if (!FUSED)  // (fused: pushed by the sweep CTA, counted on the same barrier)
                        bulk_load(sm + GS::DDL + x * TCD, ws.dvn + n.ch * TCD + x * (TCD / 2), TCD / 2, b);
                }
            };
            auto issue_qk = [&](const Item& n, uint64_t* b) {
                mbar_expect_tx(b, 2 * TCD);
                for (int x = 0; x < 2; ++x) {
                    tma_load_3d(sm + GS::Q + x * (TCD / 2), &maps.q, 64 * x, n.h, (int)n.r0, b);
                    tma_load_3d(sm + GS::K + x * (TCD / 2), &maps.k, 64 * x, n.h, (int)n.r0, b);
                }
            };
            auto issue_d = [&](const Item& n, uint64_t* b) {  // INV
                mbar_expect_tx(b, TCC);
                bulk_load(sm + GS::INV, ws.inv + n.ch * TCC, TCC, b);
            };
            auto issue_e = [&](const Item& n, uint64_t* b, int slot) {  // S_in, dS_out, g, e^Gamma_C
                mbar_expect_tx(b, 2 * TDD + kC * D * 4 + 512);
                bulk_load(sm + GS::SIN, ws.sin + n.ch * TDD, TDD, b);
                if (!FUSED) bulk_load(sm + GS::DSO, ws.dso + n.ch * TDD, TDD, b);
                tma_load_3d(sm + GS::GT, &maps.g, 0, n.hv, (int)n.r0, b);
                bulk_load(sm + GS::EGC + 512 * slot, ws.egc + n.ch * D, 512, b);
            };
            int64_t w = w0;
            // (fused) the sweep CTA's barrier on which each finished item frees dS_out's and d_delta's regions
            const uint32_t rev_free = FUSED ? peer_addr(S(RevF::BARS + 8 * (RevF::kFree + frank - 1)), 0) : 0u;
            if (!FUSED || live(w)) {
                const Item first = make_item(p, w, true);
                issue_a(first, &bars[0]);
                issue_qk(first, &bars[0]);
                issue_d(first, &bars[0]);
                issue_e(first, &bars[0], 0);
            }
            int i = 0;
            for (; live(w); ++i, w = next_w(w)) {
                const int slot = i & 1;
                const uint32_t par = (uint32_t)i & 1;
                const int64_t wn = next_w(w);
                const bool has_next = live(wn);
                const Item nx = make_item(p, has_next ? wn : w, has_next);
                uint64_t* nbar = &bars[slot ^ 1];
                if (i > 0) {  // the last item's accumulators and q, k tiles are read: this item's q, k
                    if (!pwait(&bars[7], par ^ 1, 52)) break;
                    issue_qk(make_item(p, w, true), &bars[slot]);
                }
                if (!pwait(&bars[slot], (uint32_t)(i >> 1) & 1, 51)) break;
                {  // phase A
                    tc_fence_after();
                    const uint32_t i128w = idesc_bf16(128, 128, false, false), i128 = idesc_bf16(128, 64, false, false),
                                   ixv = idesc_bf16(64, 128, true, true);
                    // [dQ~^T | S_in d_delta^T = -dw^T] = S_in [dO; d_delta]^T
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_bf16(tmem + 0, desc_kmajor(S(GS::SIN), D, ks), desc_kmajor(S(GS::DO), 2 * kC, ks),
                                 i128w, ks > 0);
                    // [V; delta] [dO; d_delta]^T: rows 0..63 give V d_delta^T (PR^T's first term) in columns
                    // 192..255; rows 64..127 give dAqk^T = delta dO^T in columns 128..191 and T^T = delta d_delta^T
                    // there after, where T = dINV INV^T = (d_delta V^T + dw K~^T) diag(beta) INV^T = d_delta u^T +
                    // dw w^T, which with dw = -d_delta S_in^T and delta = u - w S_in is d_delta delta^T
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_bf16(tmem + 128, desc_kmajor(S(GS::V), 2 * kC, ks), desc_kmajor(S(GS::DO), 2 * kC, ks),
                                 i128w, ks > 0);
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_bf16(tmem + 256, desc_kmajor(S(GS::DSO), D, ks), desc_kmajor(S(GS::DL), 2 * kC, ks),
                                 i128, ks > 0);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 320, desc_mnmajor(S(GS::INV), kC, ks), desc_mnmajor(S(GS::DDL), 2 * kC, ks),
                                 ixv, ks > 0);
                    mma_commit(&bars[2]);
                }
                if (!pwait(&bars[2], par, 53)) break;
                if (has_next) issue_a(nx, nbar);  // dO, delta, v and d_delta are consumed
                if (!pwait(&bars[8], par, 54)) break;  // dw, dN^T, T^T written
                {  // phase B, first part (operands from epilogue A): dAkk = -INV^T T (phase D), dXk^T = dw^T INV
                    tc_fence_after();
                    const uint32_t idd = idesc_neg_a(idesc_bf16(64, 64, true, false));
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 64, desc_mnmajor(S(GS::INV), kC, ks), desc_kmajor(S(GS::TT), kC, ks), idd,
                                 ks > 0);
                    const uint32_t ixk = idesc_bf16(128, 64, false, true);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 128, desc_kmajor(S(GS::DW), D, ks), desc_mnmajor(S(GS::INV), kC, ks), ixk,
                                 ks > 0);
                }
                if (!pwait(&bars[5], par, 58)) break;  // factor tiles written
                {  // phase B, second part (factor tiles): PR^T += K~ dw^T, Mkk = Kr Kc^T, dQr^T = Kc^T dN^T
                    tc_fence_after();
                    // PR^T's rows are lanes 0..63 of an M = 128 accumulator: K~ dw^T accumulates as an M = 128
                    // product whose rows 64..127 (from the 16 KB after the K~ tile) land on T^T, already read
                    const uint32_t ipr = idesc_bf16(128, 64, true, true), i64tt = idesc_bf16(64, 64, true, true);
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_bf16(tmem + 192, desc_mnmajor(S(GS::KT), D, ks), desc_mnmajor(S(GS::DW), D, ks), ipr, 1);
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_bf16(tmem + 320, desc_mnmajor(S(GS::KR), D, ks), desc_mnmajor(S(GS::KC), D, ks), i64tt,
                                 ks > 0);
                    const uint32_t imk = idesc_bf16(128, 64, false, true);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 384, desc_kmajor(S(GS::KC), D, ks), desc_mnmajor(S(GS::DN), kC, ks), imk,
                                 ks > 0);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 384, desc_kmajor(S(GS::KC), D, ks), desc_mnmajor(S(GS::DNL), kC, ks), imk, 1);
                    mma_commit(&bars[3]);
                }
                if (!pwait(&bars[3], par, 55)) break;
                if (!pwait(&bars[6], par, 56)) break;  // dM written, INV read
                {  // phase E
                    tc_fence_after();
                    if (has_next) issue_d(nx, nbar);  // INV is consumed
                    const uint32_t ik = idesc_bf16(128, 64, false, false), im = idesc_bf16(128, 64, false, true);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 64, desc_kmajor(S(GS::KC), D, ks), desc_kmajor(S(GS::DM), kC, ks), ik, ks > 0);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 320, desc_kmajor(S(GS::QR), D, ks), desc_kmajor(S(GS::DN), kC, ks), ik,
                                 ks > 0);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 320, desc_kmajor(S(GS::QR), D, ks), desc_kmajor(S(GS::DNL), kC, ks), ik, 1);
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_bf16(tmem + 320, desc_kmajor(S(GS::KR), D, ks), desc_mnmajor(S(GS::DM), kC, ks), im, 1);
                    mma_commit(&bars[4]);
                }
                if (!pwait(&bars[4], par, 57)) break;
                if (has_next) issue_e(nx, nbar, slot ^ 1);  // factor tiles, dN, dM, T are consumed
                // (fused) the next item's dS_out and d_delta may land: their bytes are expected by now
                if (FUSED && has_next) mbar_arrive_peer(rev_free);
            }
            if (live(w)) {  // a wait gave up: let copies already issued land before the block exits
                const long long t0 = clock64();
                while (clock64() - t0 < 2000000) {
                }
            }
        }
        __syncwarp();
    } else {
        float* xtot = reinterpret_cast<float*>(sm + GS::XTOT);
        float* xrg = reinterpret_cast<float*>(sm + GS::XRG);
        float* xrd = reinterpret_cast<float*>(sm + GS::XRD);
        float* xgc = reinterpret_cast<float*>(sm + GS::XGC);
        float* xt1 = reinterpret_cast<float*>(sm + GS::XT1);
        float* xdb = reinterpret_cast<float*>(sm + GS::XDB);
        const float* gt = reinterpret_cast<const float*>(sm + GS::GT);
        // the wait for phase E: per warp (a time-out is noticed at the next group barrier), or for the grouped
        // instantiation as a group, whose barrier orders the dbeta partials before their sum (per-warp waits
        // there spill that instantiation)
        auto phase_wait = [&](uint64_t* b, uint32_t parity, int code) {
            if constexpr (GROUPED) return wait_group<kSimt>(b, parity, ws.status, code, fail);
            warp_wait(b, parity, ws.status, code, fail);
            return true;
        };
        const int d = tid & 127, qtr = tid >> 7, q4 = warp & 3, cq = warp >> 2;
        const uint32_t lb = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
        const int rrow = 16 * q4 + lane;                // row of an M = 64 accumulator (lane < 16)
        const bool rv = lane < 16;
        int64_t w = w0;
        if (tid < kC && (!FUSED || live(w))) {
            const Item first = make_item(p, w, true);
            float* sb = reinterpret_cast<float*>(sm + GS::BETA);
            sb[tid] = tid < first.c ? __bfloat162float(beta[(first.r0 + tid) * HV + first.hv]) : 0.f;
        }
        // the next item's first row and row count, left by thread 0 while the current item runs (with packed
        // sequences a chunk-table look-up, two dependent global loads, that would otherwise stall the item start)
        int64_t* xrows = reinterpret_cast<int64_t*>(sm + GS::BARS + 96);
        for (int i = 0; live(w); ++i, w = next_w(w)) {
            const int slot = i & 1;
            const uint32_t par = (uint32_t)i & 1;
            // (the grouped instantiation looks up its own rows: the hand-off costs it registers)
            const Item cur = (GROUPED || i == 0) ? make_item(p, w, true) : handed_item(p, w, xrows);
            const int64_t wn = next_w(w);
            const float* sbeta = reinterpret_cast<const float*>(sm + GS::BETA + 256 * slot);
            const float* segc = reinterpret_cast<const float*>(sm + GS::EGC + 512 * slot);
            const int64_t r0 = cur.r0;
            const int c = cur.c, hv = cur.hv, h = cur.h;
            // dbeta of the item's rows: the eight partial sums of epilogue B/D in a fixed order
            auto store_dbeta = [&]() {
                if (tid < kC && tid < c)
                    db_out[(r0 + tid) * HV + hv] =
                        __float2bfloat16_rn(((xdb[tid] + xdb[64 + tid]) + (xdb[128 + tid] + xdb[192 + tid])) +
                                            ((xdb[256 + tid] + xdb[320 + tid]) + (xdb[384 + tid] + xdb[448 + tid])));
            };
            // the item's inputs: each warp waits on its own (the cumsum's barrier below absorbs the warps' skew)
            warp_wait(&bars[slot], (uint32_t)(i >> 1) & 1, ws.status, 41, fail);
            // Gamma2 of channel d for this thread's 16 rows (the canonical order of tc_intra)
            float G2[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int r = 16 * qtr + x;
                G2[x] = r < c ? gt[r * D + d] : 0.f;
            }
            quarter_cumsum_log2<1, kSimt>(G2, d, qtr, xtot, G2);
            const int rmid = (c - 1) >> 1;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                if (16 * qtr + x == rmid) xrg[d] = G2[x];
                if (16 * qtr + x == c - 1) xrg[128 + d] = G2[x];
            }
            float2 rd2 = bc2(0.f);  // even and odd columns accumulate separately, then add
#pragma unroll
            for (int c8 = 32 * qtr; c8 < 32 * qtr + 32; c8 += 8) {  // <S_in[d, v], dS_out[d, v]> over 32 columns v
                const uint4 a = *reinterpret_cast<const uint4*>(sm + GS::SIN + tile_off(d, c8, D));
                const uint4 b = *reinterpret_cast<const uint4*>(sm + GS::DSO + tile_off(d, c8, D));
                rd2 = fma2(f2(bf_lo(a.x), bf_hi(a.x)), f2(bf_lo(b.x), bf_hi(b.x)), rd2);
                rd2 = fma2(f2(bf_lo(a.y), bf_hi(a.y)), f2(bf_lo(b.y), bf_hi(b.y)), rd2);
                rd2 = fma2(f2(bf_lo(a.z), bf_hi(a.z)), f2(bf_lo(b.z), bf_hi(b.z)), rd2);
                rd2 = fma2(f2(bf_lo(a.w), bf_hi(a.w)), f2(bf_lo(b.w), bf_hi(b.w)), rd2);
            }
            xrd[qtr * 128 + d] = rd2.x + rd2.y;
            // phase A complete, the reference rows written and every warp past its reads of S_in and dS_out
            // (which the factor pass overwrites)
            if (!wait_group<kSimt>(&bars[2], par, ws.status, 42, fail)) break;
            const float ref = xrg[d], gC = xrg[128 + d];
            // per element only ep = 2^(G-ref) and em = 2^(ref-G) are evaluated; E = 2^G and
            // K^'s factor 2^(G_C-G) follow from them (the same formulas in both passes below)
            const float e_ref = exp2f(ref), e_cr = exp2f(gC - ref);
            tc_fence_after();
            {  // epilogue A: dw^T, dN^T and T^T row segments (16 columns), dv row segments (32 columns)
                const float br = rv ? sbeta[rrow] : 0.f;
                float x[16];
                // dw^T for key channel d (this thread's TMEM lane), chunk rows 16 * cq .. +15: the negated
                // S_in d_delta^T columns, to the transposed dw tile (row = key channel)
                tmem_ld16(tmem + lb + 64 + 16 * cq, x);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) x[u] = -x[u];
                for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::DW, d, 16 * cq + 8 * u, D, x + 8 * u);
                if (q4 >= 2) {  // lanes 64..127 of [V; delta] [dO; d_delta]^T: row i of dAqk^T and of T^T
                    const int ii = 32 * (q4 - 2) + lane;
                    tmem_ld16(tmem + lb + 128 + 16 * cq, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) {  // dN^T[i][r] = scale dAqk[r][i] for i <= r < c
                        const int r = 16 * cq + u;
                        x[u] = (ii <= r && r < c) ? p.scale * x[u] : 0.f;
                    }
                    for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::DN, ii, 16 * cq + 8 * u, kC, x + 8 * u);
#pragma unroll
                    for (int u = 0; u < 16; ++u) x[u] -= __bfloat162float(__float2bfloat16_rn(x[u]));
                    for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::DNL, ii, 16 * cq + 8 * u, kC, x + 8 * u);
                    tmem_ld16(tmem + lb + 192 + 16 * cq, x);  // T^T (bf16 operand of phase D)
                    tmem_ld_wait();
                    for (int u = 0; u < 2; ++u) st_tile_row8(sm + GS::TT, ii, 16 * cq + 8 * u, kC, x + 8 * u);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    tmem_ld16(tmem + lb + 320 + 32 * cq + 16 * hh, x);
                    tmem_ld_wait();
                    if (rv && rrow < c) {
                        bf16* dvrow = dv_out + ((r0 + rrow) * HV + hv) * D + 32 * cq + 16 * hh;
#pragma unroll
                        for (int u = 0; u < 16; u += 8) {
                            uint4 vv;
                            vv.x = pack2(br * x[u], br * x[u + 1]);
                            vv.y = pack2(br * x[u + 2], br * x[u + 3]);
                            vv.z = pack2(br * x[u + 4], br * x[u + 5]);
                            vv.w = pack2(br * x[u + 6], br * x[u + 7]);
                            *reinterpret_cast<uint4*>(dvrow + u) = vv;
                        }
                    }
                }
            }
            tc_fence_before();
            fence_async_smem();
            __syncwarp();  // this warp's part of epilogue A's tiles is written and its accumulators read
            if (lane == 0) mbar_arrive(&bars[8]);  // (all warps: operands of phase B's first part in place)
            tc_fence_after();
            // decayed factor tiles, stored transposed (row = key channel, column = chunk row): channel d,
            // this thread's 16 rows as two 16-byte row segments per tile (rows >= c are zero). Gamma2 goes
            // to TMEM columns 448 + 16 quarter .. +15 for the final epilogue, which reads q and k again.
            const ColAddr ad(d, kC);  // this thread's column in the 64-row q / k tiles
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                float kr[8], kc[8], qr[8], kt[8];
                uint32_t g2b[8];
#pragma unroll
                for (int x = 0; x < 8; x += 2) {  // rows r and r + 1 as packed fp32 pairs
                    const int r = 16 * qtr + 8 * h8 + x;
                    const bool in0 = r < c, in1 = r + 1 < c;
                    const uint32_t kb0 = in0 ? *reinterpret_cast<const uint16_t*>(sm + GS::K + ad.at(r)) : 0u;
                    const uint32_t qb0 = in0 ? *reinterpret_cast<const uint16_t*>(sm + GS::Q + ad.at(r)) : 0u;
                    const uint32_t kb1 = in1 ? *reinterpret_cast<const uint16_t*>(sm + GS::K + ad.at(r + 1)) : 0u;
                    const uint32_t qb1 = in1 ? *reinterpret_cast<const uint16_t*>(sm + GS::Q + ad.at(r + 1)) : 0u;
                    const float2 kv = f2(bf_lo(kb0), bf_lo(kb1)), qv = f2(bf_lo(qb0), bf_lo(qb1));
                    const float2 gm = f2(G2[8 * h8 + x], G2[8 * h8 + x + 1]);
                    g2b[x] = __float_as_uint(gm.x);
                    g2b[x + 1] = __float_as_uint(gm.y);
                    const float2 gd = add2(gm, bc2(-ref));
                    const float2 ep = f2(fast_exp2(gd.x), fast_exp2(gd.y)), em = f2(fast_exp2(-gd.x), fast_exp2(-gd.y));
                    const float2 E = mul2(ep, bc2(e_ref));
                    const float2 a = mul2(kv, ep), b = mul2(kv, em), cq2 = mul2(qv, ep), t = mul2(kv, E);
                    kr[x] = a.x, kr[x + 1] = a.y;
                    kc[x] = b.x, kc[x + 1] = b.y;
                    qr[x] = cq2.x, qr[x + 1] = cq2.y;
                    kt[x] = t.x, kt[x + 1] = t.y;
                }
                const int c0 = 16 * qtr + 8 * h8;
                st_tile_row8(sm + GS::KR, d, c0, D, kr);
                st_tile_row8(sm + GS::KC, d, c0, D, kc);
                st_tile_row8(sm + GS::QR, d, c0, D, qr);
                st_tile_row8(sm + GS::KT, d, c0, D, kt);
                tmem_st8(tmem + lb + 448 + (uint32_t)c0, g2b);
            }
            tmem_st_wait();
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[5]);  // (all warps: operands of phase B are in place)
            if (tid < kC) {  // beta of the next item to its shared slot, while phase B runs
                float nb = 0.f;
                if (live(wn)) {
                    const Item nx = make_item(p, wn, true);
                    if (tid < nx.c) nb = __bfloat162float(beta[(nx.r0 + tid) * HV + nx.hv]);
                    if (!GROUPED && tid == 0) {  // (read after this item's last group barrier)
                        xrows[0] = nx.r0;
                        xrows[1] = nx.c;
                    }
                }
                reinterpret_cast<float*>(sm + GS::BETA + 256 * (slot ^ 1))[tid] = nb;
            }
            warp_wait(&bars[3], par, ws.status, 43, fail);  // phase B complete
            tc_fence_after();
            {  // epilogue B/D: dbeta (INV and Akk parts), dM row segments
                if (q4 < 2) {  // INV part from PR^T row j (lanes 0..63 of an M = 128 accumulator), 16 columns
                    const int j = 32 * q4 + lane;
                    float x[16];
                    tmem_ld16(tmem + lb + 192 + 16 * cq, x);
                    tmem_ld_wait();
                    // INV[r][j], r = 16 cq + u: byte offset 128 r + (2 j ^ 16 (r % 8)) in the 64-row INV tile
                    const uint8_t* invc = sm + GS::INV + 16 * cq * 128;
                    const uint32_t j2 = (uint32_t)(2 * j);
                    float db = 0.f;
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const uint32_t o = (uint32_t)(u * 128) + (j2 ^ (uint32_t)((u & 7) << 4));
                        const float iv = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(invc + o) << 16);
                        db = fmaf(iv, x[u], db);
                    }
                    xdb[cq * 64 + j] = db;
                }
                const float br = rv ? sbeta[rrow] : 0.f;
                float db2 = 0.f;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {  // eight columns at a time (register budget)
                    const int j0 = 16 * cq + 8 * hh;
                    float a[8], m[8];
                    tmem_ld8(tmem + lb + 64 + j0, a);
                    tmem_ld8(tmem + lb + 320 + j0, m);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const bool in = j0 + u < rrow && rrow < c;
                        db2 = in ? fmaf(a[u], m[u], db2) : db2;
                        a[u] = in ? br * a[u] : 0.f;
                    }
                    if (rv) st_tile_row8(sm + GS::DM, rrow, j0, kC, a);
                }
                if (rv) xdb[256 + cq * 64 + rrow] = db2;
            }
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[6]);  // (all warps: dM is in place and INV has been read)
            if (!phase_wait(&bars[4], par, 46)) break;  // phase E complete
            if (GROUPED) store_dbeta();  // (after the group's barrier: every warp's dbeta partials are written)
            tc_fence_after();
            {  // final epilogue, channel d, rows 16 * quarter .. +15: dq, dk, dGamma -> dg
                // dGamma of each row replaces its Gamma2 in TMEM (columns 448 + row, read just before; the next
                // item's MMAs leave those columns alone) until the reverse cumsum below
                float dGC = 0.f;
                const float sc = p.scale, sce = p.scale * e_ref;
                // this thread's first output row and the row stride of dq / dk
                const int64_t o0 = ((r0 + 16 * qtr) * H + h) * D + d, rs = (int64_t)H * D;
                // grouped value heads: value head j of a group adds its dq, dk to the running fp32 sum of the
                // ones before it (kept per CTA in thread order, four rows per 16-byte slot, so that it stays
                // in L2), and the last one writes the bf16 result
                const int jg = GROUPED ? hv - h * G : 0;
                // this thread's column in the 64-row q / k tiles: byte offset of (r, d) = qk0 + 128 r + (dd2 ^ 16 (r % 8))
                const uint32_t qk0 = (uint32_t)((d >> 6) * kC * 128), dd2 = (uint32_t)((d & 63) * 2);
#pragma unroll
                for (int rb = 0; rb < 4; ++rb) {  // four rows at a time (register budget)
                    const uint32_t cb = (uint32_t)(16 * qtr + 4 * rb);
                    float aQt[4], aKh[4], aKr[4], aKc[4], aQr[4], aXk[4];
                    uint32_t g2u[4], kb[4], qb[4], dgb[4];
                    tmem_ld4(tmem + lb + 0 + cb, aQt);
                    tmem_ld4(tmem + lb + 256 + cb, aKh);
                    tmem_ld4(tmem + lb + 64 + cb, aKr);
                    tmem_ld4(tmem + lb + 320 + cb, aKc);
                    tmem_ld4(tmem + lb + 384 + cb, aQr);
                    tmem_ld4(tmem + lb + 128 + cb, aXk);
                    tmem_ld4u(tmem + lb + 448 + cb, g2u);
                    float gq[4], gk[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {  // raw k, q of this thread's channel (rows >= c read as zero)
                        const int r = 16 * qtr + 4 * rb + x;
                        const uint32_t o = qk0 + (uint32_t)r * 128u + (dd2 ^ (uint32_t)((r & 7) << 4));
                        kb[x] = r < c ? *reinterpret_cast<const uint16_t*>(sm + GS::K + o) : 0u;
                        qb[x] = r < c ? *reinterpret_cast<const uint16_t*>(sm + GS::Q + o) : 0u;
                    }
                    tmem_ld_wait();
                    if (rb == 3) {  // the accumulators and the q, k tiles of this item have been read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[7]);
                    }
#pragma unroll
                    for (int x = 0; x < 4; x += 2) {  // rows r and r + 1 as packed fp32 pairs
                        const int ii = 4 * rb + x, r = 16 * qtr + ii;
                        const float2 kv = f2(bf_lo(kb[x]), bf_lo(kb[x + 1])), qv = f2(bf_lo(qb[x]), bf_lo(qb[x + 1]));
                        const float2 gd = add2(f2(__uint_as_float(g2u[x]), __uint_as_float(g2u[x + 1])), bc2(-ref));
                        const float2 ep = f2(fast_exp2(gd.x), fast_exp2(gd.y)), em = f2(fast_exp2(-gd.x), fast_exp2(-gd.y));
                        const float2 E = mul2(ep, bc2(e_ref)), eh = mul2(em, bc2(e_cr));
                        const float2 bX = mul2(*reinterpret_cast<const float2*>(sbeta + r), f2(aXk[x], aXk[x + 1]));
                        const float2 aQt2 = f2(aQt[x], aQt[x + 1]), aQr2 = f2(aQr[x], aQr[x + 1]);
                        const float2 aKr2 = f2(aKr[x], aKr[x + 1]), aKc2 = f2(aKc[x], aKc[x + 1]);
                        const float2 aKh2 = f2(aKh[x], aKh[x + 1]);
                        // dq = E scale dQ~ + ep dQr;  dk = eh dK^ + E beta dXk + ep dKr + em dKc
                        const float2 dqv = mul2(ep, fma2(bc2(sce), aQt2, aQr2));
                        const float2 dkv =
                            fma2(ep, fma2(bc2(e_ref), bX, aKr2), mul2(em, fma2(bc2(e_cr), aKh2, aKc2)));
                        const float2 khk = mul2(aKh2, mul2(kv, eh));
                        // The factor values of the dGamma pair terms are the bf16 values the MMAs used (rounded
                        // two at a time here as in the factor tiles), so that each in-chunk pair's contributions
                        // to its two rows cancel in the chunk sum as they do exactly.
                        const float2 kE = mul2(kv, E), qp = mul2(qv, ep), kp = mul2(kv, ep), km = mul2(kv, em);
                        const uint32_t p1a = pack2(kE.x, qp.x), p1b = pack2(kE.y, qp.y);
                        const uint32_t p2a = pack2(kp.x, km.x), p2b = pack2(kp.y, km.y);
                        float2 dgv = fma2(mul2(bc2(sc), aQt2), mul2(qv, E), neg2(khk));
                        dgv = fma2(bX, f2(bf_lo(p1a), bf_lo(p1b)), dgv);
                        dgv = fma2(aQr2, f2(bf_hi(p1a), bf_hi(p1b)), dgv);
                        dgv = fma2(aKr2, f2(bf_lo(p2a), bf_lo(p2b)), dgv);
                        dgv = fma2(neg2(aKc2), f2(bf_hi(p2a), bf_hi(p2b)), dgv);
                        const bool in0 = r < c, in1 = r + 1 < c;
                        dgb[x] = __float_as_uint(in0 ? dgv.x : 0.f);
                        dgb[x + 1] = __float_as_uint(in1 ? dgv.y : 0.f);
                        gq[x] = dqv.x, gq[x + 1] = dqv.y;
                        gk[x] = dkv.x, gk[x + 1] = dkv.y;
                        if (in0) {
                            dGC += khk.x;
                            if (!GROUPED)
                                st_bf16_pair(reinterpret_cast<uint8_t*>(dq_out + o0 + ii * rs),
                                             reinterpret_cast<uint8_t*>(dk_out + o0 + ii * rs), dqv.x, dkv.x);
                        }
                        if (in1) {
                            dGC += khk.y;
                            if (!GROUPED)
                                st_bf16_pair(reinterpret_cast<uint8_t*>(dq_out + o0 + (ii + 1) * rs),
                                             reinterpret_cast<uint8_t*>(dk_out + o0 + (ii + 1) * rs), dqv.y, dkv.y);
                        }
                    }
                    tmem_st4(tmem + lb + 448 + cb, dgb);
                    if (GROUPED) {
                        float4* sq = reinterpret_cast<float4*>(ws.dqp) + ((int64_t)blockIdx.x * 4 + rb) * kSimt + tid;
                        float4* sk = reinterpret_cast<float4*>(ws.dkp) + ((int64_t)blockIdx.x * 4 + rb) * kSimt + tid;
                        if (jg > 0) {
                            const float4 a = *sq, b = *sk;
                            gq[0] += a.x, gq[1] += a.y, gq[2] += a.z, gq[3] += a.w;  // running sum + this head
                            gk[0] += b.x, gk[1] += b.y, gk[2] += b.z, gk[3] += b.w;
                        }
                        if (jg < G - 1) {
                            *sq = make_float4(gq[0], gq[1], gq[2], gq[3]);
                            *sk = make_float4(gk[0], gk[1], gk[2], gk[3]);
                        } else {
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                if (16 * qtr + 4 * rb + x < c)
                                    st_bf16_pair(reinterpret_cast<uint8_t*>(dq_out + o0 + (4 * rb + x) * rs),
                                                 reinterpret_cast<uint8_t*>(dk_out + o0 + (4 * rb + x) * rs), gq[x],
                                                 gk[x]);
                        }
                    }
                }
                // dg = reverse in-chunk cumsum of dGamma, whose last valid row also takes the Gamma_C terms
                // dGCt: in-quarter suffix sums and quarter totals first (one exchange), then per row the later
                // quarters' totals (added in the order 3, 2, 1) and dGCt where row c - 1 lies at or after it.
                float dG[16];
                tmem_st_wait();
                tmem_ld16(tmem + lb + 448 + 16 * qtr, dG);
                tmem_ld_wait();
                float run = 0.f;
#pragma unroll
                for (int x = 15; x >= 0; --x) {
                    run += dG[x];
                    dG[x] = run;
                }
                xgc[qtr * 128 + d] = dGC;
                xt1[qtr * 128 + d] = run;
                group_sync<kSimt>();
                if (*(volatile int*)fail) break;  // a warp's wait above gave up
                if (!GROUPED) store_dbeta();  // every warp's dbeta partials (epilogue B/D) are written
                const float dGCt = segc[d] * ((xrd[d] + xrd[128 + d]) + (xrd[256 + d] + xrd[384 + d])) +
                                   ((xgc[d] + xgc[128 + d]) + (xgc[256 + d] + xgc[384 + d]));
                const int qc = (c - 1) >> 4, xc = (c - 1) & 15;
                float carry = 0.f;
                for (int qq = 3; qq > qtr; --qq) carry += xt1[qq * 128 + d];
                if (qc > qtr) carry += dGCt;
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int r = 16 * qtr + x;
                    const float t = (qc == qtr && x <= xc) ? dG[x] + dGCt : dG[x];
                    if (r < c) dg_out[((r0 + r) * HV + hv) * D + d] = t + carry;
                }
            }
            // (no barrier here: the next item's first write to shared scratch follows its input barrier, which
            // every warp reaches only after this item's reads)
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <bool GROUPED>
__global__ void __launch_bounds__(kGradsThreads, 1)
    k_tc_grads(Prob p, const bf16* __restrict__ beta, bf16* __restrict__ dq_out, bf16* __restrict__ dk_out,
               bf16* __restrict__ dv_out, float* __restrict__ dg_out, bf16* __restrict__ db_out, TcWs ws,
               const __grid_constant__ GradMaps maps) {
    extern __shared__ uint8_t smraw[];
    grads_body<GROUPED, false>(p, beta, dq_out, dk_out, dv_out, dg_out, db_out, ws, maps, align1024(smraw), 0, 0);
}

// The sweep CTA of a fused reverse cluster: the reverse state-gradient pass of one (sequence, value head),
// chunks last to first, on 512 threads: thread t owns dS row k = t % 128, columns 32 (t / 128) .. +31, in
// fp32 registers. Per chunk, with dS the gradient of the state leaving it (dS_out):
//   d_delta = Aqk^T dO + K^ dS,   dS <- e^Gamma_C dS + Q~s^T dO - w^T d_delta,
// the arithmetic of the split reverse pass (tc_ds_rev) on the same operands, so the tiles are the same
// bits. Instead of writing dS_out and d_delta to the workspace, it pushes their bf16 tiles into the input
// regions of gradient CTA g = i % NG (cluster rank 1 + g), whose j-th item item i = g + NG j is (the bytes
// count on that CTA's input barrier of the item). Item i's two tiles are formed first; their pushes then
// wait until CTA g has finished its item j - 1 (its arrival on barrier kFree + g), whose factor tiles fill
// the dS_out region until then. Item i's tiles sit in buffer i % (NG + 1): they are rewritten by item
// i + NG + 1, which is formed only after the push of item i + NG has waited for CTA g to finish item i, so
// the push of item i has landed by then.
template <int NG>
__device__ __forceinline__ void rev_role(const Prob& p, const float* __restrict__ dht, float* __restrict__ dh0,
                                         const TcWs& ws, const CUtensorMap* tm_do, int n, int hv, uint8_t* sm) {
    static_assert(NG + 1 <= RevF::kBufs && RevF::kFree + NG <= 5, "buffers and barriers of the sweep CTA");
    constexpr int NR = kSimt;  // threads of the sweep
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + RevF::BARS);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 5);
    int* fail = reinterpret_cast<int*>(tslot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = tid & 127, vq = tid >> 7;
    const int HV = p.HV;
    int64_t bos, eos, c0;
    seq_range(p, n, bos, eos, c0);
    const int nts = (int)((eos - bos + kC - 1) / kC);
    if (tid == 0) {
        for (int x = 0; x < 5; ++x) mbar_init(&bars[x], 1);
        fence_mbar_init();
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    float S[32];
    {
        const float* src = dht ? dht + (((int64_t)n * HV + hv) * D + k) * D + 32 * vq : nullptr;
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = src ? src[j] : 0.f;
    }
    auto chunk = [&](int it) { return (c0 + it) * HV + hv; };
    auto issue1 = [&](int it) {  // operands of the first MMA group: K^, Q~s, Aqk, dO
        const int64_t ch = chunk(it);
        mbar_expect_tx(&bars[0], 3 * TCD + TCC);
        bulk_load(sm + RevF::KH, ws.kh + ch * TCD, TCD, &bars[0]);
        bulk_load(sm + RevF::QS, ws.qs + ch * TCD, TCD, &bars[0]);
        bulk_load(sm + RevF::AQK, ws.aqk + ch * TCC, TCC, &bars[0]);
        const int row = (int)(bos + (int64_t)it * kC);
        tma_load_3d(sm + RevF::DO, tm_do, 0, hv, row, &bars[0]);
        tma_load_3d(sm + RevF::DO + TCD / 2, tm_do, 64, hv, row, &bars[0]);
    };
    auto issue2 = [&](int it) {  // w (second MMA group) and e^Gamma_C (state update)
        const int64_t ch = chunk(it);
        mbar_expect_tx(&bars[1], TCD + 512);
        bulk_load(sm + RevF::W, ws.w + ch * TCD, TCD, &bars[1]);
        bulk_load(sm + RevF::EGC, ws.egc + ch * D, 512, &bars[1]);
    };
    // (the gradient CTAs' dS_out and d_delta regions and input barriers: rank 1 + g's copies of these addresses)
    const uint32_t dso_at = smem_u32(sm + GS::DSO), ddl_at = smem_u32(sm + GS::DDL), bar_at = smem_u32(sm + GS::BARS);
    tc_fence_before();
    group_sync<NR>();
    tc_fence_after();
    cluster_sync();  // every CTA's barriers are initialised
    const uint32_t tmem = *tslot;
    const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
    if (tid == 0 && nts > 0) {
        issue1(nts - 1);
        issue2(nts - 1);
    }
    uint32_t mph = 0;
    int i = 0;
    for (int it = nts - 1; it >= 0; --it, ++i) {
        const uint32_t ph = (uint32_t)i & 1;
        const int buf = i % (NG + 1), g = i % NG, j = i / NG;  // tile buffer, gradient CTA, its item index
        uint8_t* tS = sm + RevF::S0 + buf * TDD;   // bf16 dS_out: MMA operand and the pushed tile
        uint8_t* tD = sm + RevF::DD0 + buf * TCD;  // bf16 d_delta
#pragma unroll
        for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(tS, k, 32 * vq + c8, D, S + c8);
        fence_async_smem();
        if (!wait_group<NR>(&bars[0], ph, ws.status, 61, fail)) break;
        if (tid == 0) {
            tc_fence_after();
            // d_delta = Aqk^T dO + K^ dS (chunk rows on TMEM lanes, M = 64, N = 128)
            const uint32_t ida = idesc_bf16(64, 128, true, true), idb = idesc_bf16(64, 128, false, true);
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem, desc_mnmajor(smem_u32(sm + RevF::AQK), kC, ks),
                         desc_mnmajor(smem_u32(sm + RevF::DO), kC, ks), ida, ks > 0);
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem, desc_kmajor(smem_u32(sm + RevF::KH), kC, ks), desc_mnmajor(smem_u32(tS), D, ks), idb,
                         1);
            // dS accumulator = Q~s^T dO (M = 128, N = 128)
            const uint32_t idc = idesc_bf16(128, 128, true, true);
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem + 128, desc_mnmajor(smem_u32(sm + RevF::QS), kC, ks),
                         desc_mnmajor(smem_u32(sm + RevF::DO), kC, ks), idc, ks > 0);
            mma_commit(&bars[2]);
        }
        if (!wait_group<NR>(&bars[2], mph, ws.status, 63, fail)) break;
        mph ^= 1;
        if (tid == 0 && it > 0) issue1(it - 1);  // the first group's operands are consumed
        tc_fence_after();
        {  // d_delta rows into tD: row r = 16 (warp % 4) + lane (lane < 16), columns 32 (warp / 4) .. +31
            const int r = 16 * (warp & 3) + lane, cb = 32 * (warp >> 2);
            float acc[32];
            tmem_ld32(tmem + lq + cb, acc);
            tmem_ld_wait();
            if (lane < 16) {
#pragma unroll
                for (int c8 = 0; c8 < 32; c8 += 8) st_tile_row8(tD, r, cb + c8, kC, acc + c8);
            }
        }
        tc_fence_before();
        fence_async_smem();
        if (!wait_group<NR>(&bars[1], ph, ws.status, 64, fail)) break;
        if (tid == 0) {  // dS accumulator -= w^T d_delta
            tc_fence_after();
            const uint32_t id = idesc_neg_a(idesc_bf16(128, 128, true, true));
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tmem + 128, desc_mnmajor(smem_u32(sm + RevF::W), kC, ks), desc_mnmajor(smem_u32(tD), kC, ks),
                         id, 1);
            mma_commit(&bars[2]);
            // both tiles of item i, as soon as the gradient CTA has finished item i - 1; the gradient CTA
            // keeps d_delta's two 64-column halves TCD bytes apart
            if (j > 0 && !mbar_wait_cluster(&bars[RevF::kFree + g], (uint32_t)(j - 1) & 1, ws.status, 62)) {
                *(volatile int*)fail = 1;  // (read after the next group barrier)
            } else {
                const uint32_t r = 1 + (uint32_t)g;
                const uint32_t ibar = peer_addr(bar_at, r) + 8u * (uint32_t)(j & 1);  // CTA g's input barrier
                const uint32_t pddl = peer_addr(ddl_at, r);
                bulk_push(peer_addr(dso_at, r), tS, TDD, ibar);
                bulk_push(pddl, tD, TCD / 2, ibar);
                bulk_push(pddl + TCD, tD + TCD / 2, TCD / 2, ibar);
            }
        }
        const float e = reinterpret_cast<const float*>(sm + RevF::EGC)[k];
        if (!wait_group<NR>(&bars[2], mph, ws.status, 65, fail)) break;
        mph ^= 1;
        if (tid == 0 && it > 0) issue2(it - 1);  // w and e^Gamma_C are consumed
        tc_fence_after();
        {
            float acc[32];
            tmem_ld32(tmem + lq + 128 + 32 * vq, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 v = fma2(bc2(e), f2(S[j], S[j + 1]), f2(acc[j], acc[j + 1]));
                S[j] = v.x, S[j + 1] = v.y;
            }
        }
        tc_fence_before();
    }
    if (*(volatile int*)fail == 0) {
        if (dh0) {
            float* dst = dh0 + (((int64_t)n * HV + hv) * D + k) * D + 32 * vq;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[j] = S[j];
        }
    } else if (tid == 0) {  // a wait gave up: let copies already issued land before the cluster exits
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
    }
    tc_fence_before();
    group_sync<NR>();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// Fused reverse (state-gradient sweep and per-chunk gradients in one launch, dS_out and d_delta kept on
// chip): one cluster of 1 + NG CTAs per (sequence, value head), on 1 + NG SMs. CTA 0 runs the sweep
// (rev_role, warps 0..15; warp 16 only meets the cluster barriers); CTA 1 + g runs the gradient work of the
// sweep's chunks i with i % NG == g, in the sweep's order (grads_body), its dS_out and d_delta inputs pushed
// by CTA 0 into its shared memory. Equal key and value heads only (the grouped sum of dq, dk runs across
// sweeps).
template <int NG>
__global__ void __cluster_dims__(NG + 1, 1, 1) __launch_bounds__(kGradsThreads, 1)
    k_tc_rev_fused(Prob p, const float* __restrict__ dht, float* __restrict__ dh0, const bf16* __restrict__ beta,
                   bf16* __restrict__ dq_out, bf16* __restrict__ dk_out, bf16* __restrict__ dv_out,
                   float* __restrict__ dg_out, bf16* __restrict__ db_out, TcWs ws, const __grid_constant__ GradMaps maps) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = align1024(smraw);
    const int sweep = (int)cluster_index();
    const int hv = sweep % p.HV, n = sweep_seq(ws, sweep / p.HV);
    const int rank = (int)cluster_rank();
    if (rank == 0) {
        if (threadIdx.x < kSimt)
            rev_role<NG>(p, dht, dh0, ws, &maps.d_o, n, hv, sm);
        else
            cluster_sync();  // (the cluster's start barrier)
    } else {
        int64_t bos, eos, c0;
        seq_range(p, n, bos, eos, c0);
        const int64_t nts = (eos - bos + kC - 1) / kC;
        // this CTA's chunks of the sweep: it = nts - rank, nts - rank - NG, ... (none when nts < rank)
        grads_body<false, true>(p, beta, dq_out, dk_out, dv_out, dg_out, db_out, ws, maps, sm,
                                (c0 + nts - rank) * p.HV + hv, c0 * p.HV + hv, (int64_t)NG * p.HV, rank);
    }
    cluster_sync();  // no CTA leaves while another may still reach its shared memory
}

bool make_grad_maps(const Prob& p, const IO& io, GradMaps* m) {
    memset(m, 0, sizeof(*m));
    const int64_t rows = (int64_t)p.B * p.T;
    if (rows == 0) return true;
    const uint64_t rq = (uint64_t)p.H * D * 2, rv = (uint64_t)p.HV * D * 2;
    return make_tmap_bf16_3d(&m->q, io.q, D, p.H, rows, D * 2, rq, 64, 1, kC) &&
           make_tmap_bf16_3d(&m->k, io.k, D, p.H, rows, D * 2, rq, 64, 1, kC) &&
           make_tmap_bf16_3d(&m->v, io.v, D, p.HV, rows, D * 2, rv, 64, 1, kC) &&
           make_tmap_bf16_3d(&m->d_o, io.d_o, D, p.HV, rows, D * 2, rv, 64, 1, kC) &&
           make_tmap_f32_3d(&m->g, io.g, D, p.HV, rows, D * 4, (uint64_t)p.HV * D * 4, D, 1, kC);
}

}  // namespace

cudaError_t tc_grads(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st) {
    auto kern = p.HV != p.H ? k_tc_grads<true> : k_tc_grads<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGradsSmem);
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.B * p.T;
    if (p.NT == 0 || rows == 0) return cudaSuccess;
    GradMaps m;
    if (!make_grad_maps(p, io, &m)) return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // persistent: one CTA per SM, at most one per (chunk, key head) group and at most kGradsMaxCtas (the
    // CTAs the group-sum scratch is sized for)
    const bool grouped = p.HV != p.H;
    const int64_t groups = p.NT * p.H;
    int64_t grid = groups < nsm ? groups : nsm;
    if (grid > kGradsMaxCtas) grid = kGradsMaxCtas;
    if (grouped && (!ws.dqp || !ws.dkp)) return cudaErrorInvalidValue;
    kern<<<(unsigned)grid, kGradsThreads, kGradsSmem, st>>>(p, (const bf16*)io.beta, (bf16*)io.dq, (bf16*)io.dk,
                                                            (bf16*)io.dv, io.dg, (bf16*)io.dbeta, ws, m);
    note_launch("tc_grads", st);
    return cudaGetLastError();
}

cudaError_t tc_rev_fused(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st) {
    constexpr int NG = kFusedGradCtas;
    cudaError_t e = cudaFuncSetAttribute(k_tc_rev_fused<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGradsSmem);
    if (e != cudaSuccess) return e;
    if (p.HV != p.H) return cudaErrorInvalidValue;
    const int64_t sweeps = (int64_t)p.N * p.HV;
    if (sweeps == 0) return cudaSuccess;
    GradMaps m;
    if (!make_grad_maps(p, io, &m)) return cudaErrorInvalidValue;
    k_tc_rev_fused<NG><<<(unsigned)((NG + 1) * sweeps), kGradsThreads, kGradsSmem, st>>>(
        p, io.dht, io.dh0, (const bf16*)io.beta, (bf16*)io.dq, (bf16*)io.dk, (bf16*)io.dv, io.dg, (bf16*)io.dbeta,
        ws, m);
    note_launch("tc_rev_fused", st);
    return cudaGetLastError();
}

}  // namespace kda
