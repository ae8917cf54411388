// C-ABI layer of the KDA library: argument validation, workspace carving and
// launch sequencing. Declared in include/kda.h. Nothing here allocates device
// memory or synchronises (except kda_device_status, which is documented to).
#include <string.h>

#include "../../include/kda.h"
#include "../../include/kda_selftest.h"
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Validate dims; fills the device-side problem description (pointers unset).
kda_status check_dims(const kda_dims* d, Prob* p) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->B < 1 || d->T < 0 || d->H < 1 || d->HV < 1 || d->HV % d->H != 0) return KDA_ERR_INVALID_ARG;
    if (d->chunk != kC) return KDA_ERR_UNSUPPORTED;
    if (!((d->K == 64 || d->K == 128) && (d->V == 64 || d->V == 128))) return KDA_ERR_UNSUPPORTED;
    if (d->dtype != KDA_DTYPE_BF16 && d->dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (d->num_seqs < 1 || d->num_chunks < 0) return KDA_ERR_INVALID_ARG;
    if (d->HV > 65535 || d->num_seqs > 2147483647 || d->num_chunks > 2147483647) return KDA_ERR_UNSUPPORTED;
    memset(p, 0, sizeof(*p));
    p->B = d->B;
    p->T = d->T;
    p->H = d->H;
    p->HV = d->HV;
    p->K = d->K;
    p->V = d->V;
    p->N = d->num_seqs;
    p->NT = d->num_chunks;
    p->NTs = (d->T + kC - 1) / kC;
    p->scale = d->scale;
    return KDA_OK;
}

struct Layout {
    size_t status, gam, w, u, vn, inv, aqk, sin, dso, dvn, dqt, dkh, dw, dgc, dqp, dkp, total;
    // tensor-core path regions
    bool tc;
    size_t t_w, t_invb, t_kh, t_qs, t_vn, t_dvn, t_aqk, t_inv, t_sin, t_dso, t_egc, t_seg_e, t_seg_p, t_seg_s0, t_order;
};

// bf16 inputs with K = V = 128 run on the tensor-core path (forward and backward).
bool use_tc(const kda_dims* d, int pass) {
    // (the state passes put sequences on grid y, which holds at most 65535)
    return (pass == KDA_PASS_BWD || pass == KDA_PASS_FWD) && d->dtype == KDA_DTYPE_BF16 && d->K == 128 &&
           d->V == 128 && d->num_seqs <= 65535;
}

Layout layout(const Prob& p, int pass, bool tc) {
    Layout L;
    memset(&L, 0, sizeof(L));
    const size_t R = (size_t)p.B * p.T, HV = p.HV, K = p.K, V = p.V, NT = (size_t)p.NT, f = sizeof(float);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    L.status = take(kAlign);
    L.tc = tc;
    if (tc) {
        const size_t CH = NT * HV, TCD = (size_t)kC * 128 * 2, TCC = (size_t)kC * kC * 2, TDD = 128 * 128 * 2;
        L.t_w = take(CH * TCD);
        L.t_kh = take(CH * TCD);
        L.t_qs = take(CH * TCD);
        L.t_aqk = take(CH * TCC);
        L.t_inv = take(CH * TCC);
        L.t_invb = take(CH * TCC);
        L.t_egc = take(CH * 128 * f);
        L.t_order = take((size_t)p.N * sizeof(int));  // the sweep order of packed sequences
        const SegPlan sp = seg_plan(p);
        if (sp.len) {  // segmented state passes: three fp32 K x V matrices per (sequence, head, segment)
            const size_t segs = (size_t)p.N * HV * sp.M * 128 * 128 * f;
            L.t_seg_e = take(segs);
            L.t_seg_p = take(segs);
            L.t_seg_s0 = take(segs);
        }
        if (pass == KDA_PASS_FWD) {  // the forward keeps the state and delta on chip
            L.total = off;
            return L;
        }
        L.t_vn = take(CH * TCD);
        L.t_sin = take(CH * TDD);
        L.t_dvn = take(CH * TCD);
        L.t_dso = take(CH * TDD);
        if (p.HV != p.H) {  // the gradient kernel's running dq / dk group sums, 64 x 128 fp32 per CTA
            const size_t groups = NT * p.H, ctas = groups < (size_t)kGradsMaxCtas ? groups : kGradsMaxCtas;
            L.dqp = take(ctas * kC * 128 * f);
            L.dkp = take(ctas * kC * 128 * f);
        }
        L.total = off;
        return L;
    }
    L.gam = take(R * HV * K * f);
    L.w = take(R * HV * K * f);
    L.u = take(R * HV * V * f);
    L.vn = take(R * HV * V * f);
    L.inv = take(NT * HV * kC * kC * f);
    L.aqk = take(NT * HV * kC * kC * f);
    if (pass == KDA_PASS_BWD) {
        L.sin = take(NT * HV * K * V * f);
        L.dso = take(NT * HV * K * V * f);
        L.dvn = take(R * HV * V * f);
        L.dqt = take(R * HV * K * f);
        L.dkh = take(R * HV * K * f);
        L.dw = take(R * HV * K * f);
        L.dgc = take(NT * HV * K * f);
        if (p.HV != p.H) {
            L.dqp = take(R * HV * K * f);
            L.dkp = take(R * HV * K * f);
        }
    }
    L.total = off;
    return L;
}

Ws carve(void* base, const Layout& L) {
    char* b = (char*)base;
    Ws w;
    memset(&w, 0, sizeof(w));
    auto at = [&](size_t off) { return (float*)(b + off); };
    w.status = (int*)(b + L.status);
    w.gam = at(L.gam);
    w.w = at(L.w);
    w.u = at(L.u);
    w.vn = at(L.vn);
    w.inv = at(L.inv);
    w.aqk = at(L.aqk);
    if (L.sin) {
        w.sin = at(L.sin);
        w.dso = at(L.dso);
        w.dvn = at(L.dvn);
        w.dqt = at(L.dqt);
        w.dkh = at(L.dkh);
        w.dw = at(L.dw);
        w.dgc = at(L.dgc);
        if (L.dqp) {
            w.dqp = at(L.dqp);
            w.dkp = at(L.dkp);
        }
    }
    return w;
}

TcWs carve_tc(void* base, const Layout& L) {
    char* b = (char*)base;
    TcWs w;
    memset(&w, 0, sizeof(w));
    auto at = [&](size_t off) { return off ? (uint8_t*)(b + off) : nullptr; };  // 0: region absent
    w.status = (int*)(b + L.status);
    w.w = at(L.t_w);
    w.invb = at(L.t_invb);
    w.kh = at(L.t_kh);
    w.qs = at(L.t_qs);
    w.vn = at(L.t_vn);
    w.dvn = at(L.t_dvn);
    w.aqk = at(L.t_aqk);
    w.inv = at(L.t_inv);
    w.sin = at(L.t_sin);
    w.dso = at(L.t_dso);
    w.egc = (float*)at(L.t_egc);
    w.seg_e = (float*)at(L.t_seg_e);
    w.seg_p = (float*)at(L.t_seg_p);
    w.seg_s0 = (float*)at(L.t_seg_s0);
    w.seq_order = (int*)at(L.t_order);
    if (L.dqp) {
        w.dqp = (float*)at(L.dqp);
        w.dkp = (float*)at(L.dkp);
    }
    return w;
}

// Shared checks of the forward and backward inputs.
kda_status check_common(const kda_dims* dims, Prob* p, const void* q, const void* k, const void* v, const float* g,
                        const void* beta, const float* h0, const int64_t* cu, const int32_t* cidx,
                        const int64_t* coff, void* ws, size_t ws_bytes, int pass) {
    kda_status s = check_dims(dims, p);
    if (s != KDA_OK) return s;
    const bool packed = cu != nullptr;
    // (a packed batch of empty sequences has no chunk table to pass: chunk_idx may then be NULL)
    if (packed != (coff != nullptr) || (!packed && cidx) || (packed && !cidx && dims->num_chunks > 0))
        return KDA_ERR_INVALID_ARG;
    if (packed) {
        if (dims->B != 1) return KDA_ERR_INVALID_ARG;
    } else {
        if (dims->num_seqs != dims->B || dims->num_chunks != (int64_t)dims->B * p->NTs) return KDA_ERR_INVALID_ARG;
    }
    const size_t rows = (size_t)dims->B * dims->T;
    if (rows > 0 && (!q || !k || !v || !g || !beta)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, h0, cu, cidx, coff};
    for (const void* x : ptrs)
        if (x && !aligned16(x)) return KDA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws) || ws_bytes < layout(*p, pass, use_tc(dims, pass)).total) return KDA_ERR_WORKSPACE;
    p->cu = cu;
    p->cidx = cidx;
    p->coff = coff;
    return KDA_OK;
}

constexpr int kMaxLaunches = 64;
void* const* g_prof_events = nullptr;
int g_prof_n = 0;
thread_local const char* t_names[kMaxLaunches];
thread_local int t_count = 0;
thread_local const char* t_cuda_err = "no error";

kda_status cuda_fail(cudaError_t e) {
    t_cuda_err = cudaGetErrorString(e);
    return KDA_ERR_CUDA;
}

}  // namespace

void begin_launches(cudaStream_t st) {
    t_count = 0;
    if (g_prof_n > 0) cudaEventRecord((cudaEvent_t)g_prof_events[0], st);
}

void note_launch(const char* name, cudaStream_t st) {
    if (t_count < kMaxLaunches) t_names[t_count] = name;
    ++t_count;
    if (t_count < g_prof_n) cudaEventRecord((cudaEvent_t)g_prof_events[t_count], st);
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_set_profile_events(void* const* events, int32_t n_events) {
    if (n_events < 0 || (n_events > 0 && !events)) return KDA_ERR_INVALID_ARG;
    g_prof_events = n_events > 0 ? events : nullptr;
    g_prof_n = n_events;
    return KDA_OK;
}

extern "C" int32_t kda_last_launch_count(void) { return t_count; }

extern "C" const char* kda_last_cuda_error(void) { return t_cuda_err; }

extern "C" const char* kda_launch_name(int32_t i) {
    return (i >= 0 && i < t_count && i < kMaxLaunches) ? t_names[i] : nullptr;
}

extern "C" const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid size, pointer, alignment or cu_seqlens";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: valid but unsupported configuration";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call or kernel launch failed";
        case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown kda_status";
}

extern "C" kda_status kda_prepare_chunks(const int64_t* cu, int32_t num_seqs, int32_t chunk, int32_t* chunk_idx,
                                         int64_t* chunk_off, int64_t* num_chunks) {
    if (!cu || !num_chunks || num_seqs < 1 || chunk != kC || cu[0] != 0) return KDA_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int32_t n = 0; n < num_seqs; ++n) {
        if (cu[n + 1] < cu[n]) return KDA_ERR_INVALID_ARG;
        const int64_t nt = (cu[n + 1] - cu[n] + kC - 1) / kC;
        if (chunk_off) chunk_off[n] = total;
        if (chunk_idx)
            for (int64_t i = 0; i < nt; ++i) {
                chunk_idx[2 * (total + i)] = n;
                chunk_idx[2 * (total + i) + 1] = (int32_t)i;
            }
        total += nt;
    }
    if (chunk_off) chunk_off[num_seqs] = total;
    *num_chunks = total;
    return KDA_OK;
}

extern "C" size_t kda_workspace_bytes(const kda_dims* dims, int32_t pass) {
    Prob p;
    if (check_dims(dims, &p) != KDA_OK || (pass != KDA_PASS_FWD && pass != KDA_PASS_BWD)) return 0;
    return layout(p, pass, use_tc(dims, pass)).total;
}

extern "C" kda_status kda_chunk_fwd(const kda_dims* dims, const void* q, const void* k, const void* v,
                                    const float* g, const void* beta, const float* h0, const int64_t* cu_seqlens,
                                    const int32_t* chunk_idx, const int64_t* chunk_off, void* o, float* ht,
                                    float* states, void* ws, size_t ws_bytes, kda_stream_t stream) {
    Prob p;
    kda_status s = check_common(dims, &p, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, ws, ws_bytes,
                                KDA_PASS_FWD);
    if (s != KDA_OK) return s;
    if ((size_t)dims->B * dims->T > 0 && !o) return KDA_ERR_INVALID_ARG;
    for (const void* x : {(const void*)o, (const void*)ht, (const void*)states})
        if (x && !aligned16(x)) return KDA_ERR_INVALID_ARG;
    const Layout L = layout(p, KDA_PASS_FWD, use_tc(dims, KDA_PASS_FWD));
    cudaStream_t st = (cudaStream_t)stream;
    IO io;
    memset(&io, 0, sizeof(io));
    io.q = q; io.k = k; io.v = v; io.beta = beta; io.g = g; io.h0 = h0;
    io.o = o; io.ht = ht; io.states_out = states;
    cudaError_t e = cudaMemsetAsync((char*)ws + L.status, 0, kAlign, st);
    if (e != cudaSuccess) return cuda_fail(e);
    begin_launches(st);
    if (L.tc)
        e = tc_fwd(p, io, carve_tc(ws, L), st);
    else
        e = simt_fwd(p, dims->dtype == KDA_DTYPE_BF16, io, carve(ws, L), st);
    if (e != cudaSuccess) return cuda_fail(e);
    return KDA_OK;
}

namespace {
kda_status chunk_bwd(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                     const void* beta, const float* h0, const int64_t* cu_seqlens, const int32_t* chunk_idx,
                     const int64_t* chunk_off, const void* d_o, const float* dht, const float* states, void* dq,
                     void* dk, void* dv, float* dg, void* dbeta, float* dh0, void* ws, size_t ws_bytes,
                     kda_stream_t stream, bool fused) {
    Prob p;
    kda_status s = check_common(dims, &p, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, ws, ws_bytes,
                                KDA_PASS_BWD);
    if (s != KDA_OK) return s;
    if (dh0 && !h0) return KDA_ERR_INVALID_ARG;
    if ((size_t)dims->B * dims->T > 0 && (!d_o || !dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_INVALID_ARG;
    for (const void* x : {(const void*)d_o, (const void*)dht, (const void*)states, (const void*)dq,
                          (const void*)dk, (const void*)dv, (const void*)dg, (const void*)dbeta, (const void*)dh0})
        if (x && !aligned16(x)) return KDA_ERR_INVALID_ARG;
    const Layout L = layout(p, KDA_PASS_BWD, use_tc(dims, KDA_PASS_BWD));
    if (states && !L.tc) return KDA_ERR_UNSUPPORTED;  // saved states are consumed on the tensor-core path
    if (fused && (!L.tc || p.HV != p.H)) return KDA_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    IO io;
    memset(&io, 0, sizeof(io));
    io.q = q; io.k = k; io.v = v; io.beta = beta; io.d_o = d_o; io.g = g; io.h0 = h0; io.dht = dht;
    io.dq = dq; io.dk = dk; io.dv = dv; io.dbeta = dbeta; io.dg = dg; io.dh0 = dh0; io.states_in = states;
    cudaError_t e = cudaMemsetAsync((char*)ws + L.status, 0, kAlign, st);
    if (e != cudaSuccess) return cuda_fail(e);
    begin_launches(st);
    if (L.tc)
        e = tc_bwd(p, io, carve_tc(ws, L), st, 4, false, fused);
    else
        e = simt_bwd(p, dims->dtype == KDA_DTYPE_BF16, io, carve(ws, L), st);
    if (e != cudaSuccess) return cuda_fail(e);
    return KDA_OK;
}
}  // namespace

extern "C" kda_status kda_chunk_bwd(const kda_dims* dims, const void* q, const void* k, const void* v,
                                    const float* g, const void* beta, const float* h0, const int64_t* cu_seqlens,
                                    const int32_t* chunk_idx, const int64_t* chunk_off, const void* d_o,
                                    const float* dht, const float* states, void* dq, void* dk, void* dv, float* dg,
                                    void* dbeta, float* dh0, void* ws, size_t ws_bytes, kda_stream_t stream) {
    return chunk_bwd(dims, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, d_o, dht, states, dq, dk, dv, dg,
                     dbeta, dh0, ws, ws_bytes, stream, false);
}

extern "C" kda_status kda_chunk_bwd_fused(const kda_dims* dims, const void* q, const void* k, const void* v,
                                          const float* g, const void* beta, const float* h0,
                                          const int64_t* cu_seqlens, const int32_t* chunk_idx,
                                          const int64_t* chunk_off, const void* d_o, const float* dht,
                                          const float* states, void* dq, void* dk, void* dv, float* dg, void* dbeta,
                                          float* dh0, void* ws, size_t ws_bytes, kda_stream_t stream) {
    return chunk_bwd(dims, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, d_o, dht, states, dq, dk, dv, dg,
                     dbeta, dh0, ws, ws_bytes, stream, true);
}

extern "C" size_t kda_saved_bytes(const kda_dims* dims) {
    Prob p;
    if (check_dims(dims, &p) != KDA_OK || !use_tc(dims, KDA_PASS_BWD)) return 0;
    return layout(p, KDA_PASS_BWD, true).total;
}

extern "C" kda_status kda_chunk_fwd_save(const kda_dims* dims, const void* q, const void* k, const void* v,
                                         const float* g, const void* beta, const float* h0,
                                         const int64_t* cu_seqlens, const int32_t* chunk_idx, const int64_t* chunk_off,
                                         void* o, float* ht, void* saved, size_t saved_bytes, kda_stream_t stream) {
    Prob p;
    kda_status s = check_common(dims, &p, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, saved, saved_bytes,
                                KDA_PASS_BWD);
    if (s != KDA_OK) return s;
    if (!use_tc(dims, KDA_PASS_BWD)) return KDA_ERR_UNSUPPORTED;
    if ((size_t)dims->B * dims->T > 0 && !o) return KDA_ERR_INVALID_ARG;
    for (const void* x : {(const void*)o, (const void*)ht})
        if (x && !aligned16(x)) return KDA_ERR_INVALID_ARG;
    const Layout L = layout(p, KDA_PASS_BWD, true);
    cudaStream_t st = (cudaStream_t)stream;
    IO io;
    memset(&io, 0, sizeof(io));
    io.q = q; io.k = k; io.v = v; io.beta = beta; io.g = g; io.h0 = h0;
    io.o = o; io.ht = ht;
    cudaError_t e = cudaMemsetAsync((char*)saved + L.status, 0, kAlign, st);
    if (e != cudaSuccess) return cuda_fail(e);
    begin_launches(st);
    e = tc_fwd(p, io, carve_tc(saved, L), st);  // the backward layout: the state pass also keeps S_in and delta
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

extern "C" kda_status kda_chunk_bwd_from_saved(const kda_dims* dims, const void* q, const void* k, const void* v,
                                               const float* g, const void* beta, const float* h0,
                                               const int64_t* cu_seqlens, const int32_t* chunk_idx,
                                               const int64_t* chunk_off, const void* d_o, const float* dht,
                                               void* saved, size_t saved_bytes, void* dq, void* dk, void* dv, float* dg,
                                               void* dbeta, float* dh0, kda_stream_t stream) {
    Prob p;
    kda_status s = check_common(dims, &p, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, saved, saved_bytes,
                                KDA_PASS_BWD);
    if (s != KDA_OK) return s;
    if (!use_tc(dims, KDA_PASS_BWD)) return KDA_ERR_UNSUPPORTED;
    if (dh0 && !h0) return KDA_ERR_INVALID_ARG;
    if ((size_t)dims->B * dims->T > 0 && (!d_o || !dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_INVALID_ARG;
    for (const void* x : {(const void*)d_o, (const void*)dht, (const void*)dq, (const void*)dk, (const void*)dv,
                          (const void*)dg, (const void*)dbeta, (const void*)dh0})
        if (x && !aligned16(x)) return KDA_ERR_INVALID_ARG;
    const Layout L = layout(p, KDA_PASS_BWD, true);
    cudaStream_t st = (cudaStream_t)stream;
    IO io;
    memset(&io, 0, sizeof(io));
    io.q = q; io.k = k; io.v = v; io.beta = beta; io.d_o = d_o; io.g = g; io.h0 = h0; io.dht = dht;
    io.dq = dq; io.dk = dk; io.dv = dv; io.dbeta = dbeta; io.dg = dg; io.dh0 = dh0;
    cudaError_t e = cudaMemsetAsync((char*)saved + L.status, 0, kAlign, st);
    if (e != cudaSuccess) return cuda_fail(e);
    begin_launches(st);
    e = tc_bwd(p, io, carve_tc(saved, L), st, 4, true);
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

extern "C" kda_status kda_debug_bwd_stages(const kda_dims* dims, const void* q, const void* k, const void* v,
                                           const float* g, const void* beta, const float* h0,
                                           const int64_t* cu_seqlens, const int32_t* chunk_idx,
                                           const int64_t* chunk_off, const void* d_o, const float* dht, float* dh0,
                                           int32_t stages, void* ws, size_t ws_bytes, kda_stream_t stream) {
    Prob p;
    kda_status s = check_common(dims, &p, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, ws, ws_bytes,
                                KDA_PASS_BWD);
    if (s != KDA_OK) return s;
    if (!use_tc(dims, KDA_PASS_BWD)) return KDA_ERR_UNSUPPORTED;
    if (stages < 1 || stages > 4 || !d_o || (dh0 && !h0)) return KDA_ERR_INVALID_ARG;
    const Layout L = layout(p, KDA_PASS_BWD, true);
    cudaStream_t st = (cudaStream_t)stream;
    IO io;
    memset(&io, 0, sizeof(io));
    io.q = q; io.k = k; io.v = v; io.beta = beta; io.d_o = d_o; io.g = g; io.h0 = h0; io.dht = dht; io.dh0 = dh0;
    cudaError_t e = cudaMemsetAsync((char*)ws + L.status, 0, kAlign, st);
    if (e != cudaSuccess) return cuda_fail(e);
    begin_launches(st);
    e = tc_bwd(p, io, carve_tc(ws, L), st, stages);
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

extern "C" kda_status kda_debug_ws_region(const kda_dims* dims, int32_t pass, const char* name, size_t* offset,
                                          size_t* bytes) {
    Prob p;
    if (!name || !offset || !bytes || check_dims(dims, &p) != KDA_OK) return KDA_ERR_INVALID_ARG;
    const Layout L = layout(p, pass, use_tc(dims, pass));
    const struct {
        const char* n;
        size_t off;
    } tab[] = {{"w", L.t_w}, {"invb", L.t_invb}, {"kh", L.t_kh}, {"qs", L.t_qs}, {"vn", L.t_vn}, {"dvn", L.t_dvn},
               {"aqk", L.t_aqk}, {"inv", L.t_inv}, {"sin", L.t_sin}, {"dso", L.t_dso}, {"egc", L.t_egc},
               {"order", L.t_order}};
    if (!L.tc) return KDA_ERR_UNSUPPORTED;
    for (size_t i = 0; i < sizeof(tab) / sizeof(tab[0]); ++i)
        if (strcmp(tab[i].n, name) == 0) {
            *offset = tab[i].off;
            size_t end = L.total;
            for (size_t j = 0; j < sizeof(tab) / sizeof(tab[0]); ++j)
                if (tab[j].off > tab[i].off && tab[j].off < end) end = tab[j].off;
            *bytes = end - tab[i].off;
            return KDA_OK;
        }
    return KDA_ERR_INVALID_ARG;
}

extern "C" kda_status kda_device_status(const void* ws, kda_stream_t stream) {
    if (!ws) return KDA_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    int word = 0;
    e = cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return word == 0 ? KDA_OK : KDA_ERR_DEVICE_TIMEOUT;
}
