/*
 * KDA reference oracle: plain fp64 CPU token-by-token recurrence with a
 * hand-derived reverse-mode backward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file; it exists so the tests, the smoke check and the CPU
 * baseline leg of the benchmark can check the CUDA library against an
 * independent, obviously-correct computation. It shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes (Kimi Delta Attention, a gated delta rule with a
 * per-key-channel gate; the recurrence is the one stated for the method,
 * S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T and
 * o_t = scale * S_t^T q_t), written without changing it as
 *
 *     S'_t = Diag(exp g_t) S_{t-1}
 *     u_t  = v_t - S'_t^T k_t
 *     S_t  = S'_t + beta_t k_t u_t^T
 *     o_t  = scale * S_t^T q_t,          ht = S_T,  S_0 = h0 (or 0).
 *
 * The backward is reverse mode of L = sum(o * do) + sum(ht * dht), derived by
 * hand, token by token from t = T down to 1, with dS = dht (or 0):
 *
 *     dq_t  = scale * S_t do_t;          dS += scale * q_t do_t^T
 *     du    = beta_t * dS^T k_t;         dbeta_t = k_t^T dS u_t
 *     dv_t  = du;                        dk_t = beta_t dS u_t - S'_t du
 *     dS'   = dS - k_t du^T;             dg_t = rowsum(dS' (.) S'_t)
 *     dS    = Diag(exp g_t) dS'          (and dh0 = dS after t = 1).
 *
 * Grouped value heads (HV = G * H): value head hv reads key head h = hv / G
 * (the head map of the Triton backward kernels, "FLA chunk_bwd.py",
 * chunk_kda_bwd_kernel_dAv); dq and dk of key head h are the sum of the
 * per-value-head gradients over hv = h*G .. h*G+G-1 in ascending order (the
 * GVA reduction at the end of chunk_kda_bwd).
 *
 * Sequences are given as token offsets cu[0..N] into the packed row space
 * (the cu_seqlens convention of the same page). The state is checkpointed
 * every C tokens on the way forward and recomputed within a segment on the
 * way back. Optionally the per-chunk state S_in (state before a chunk's first
 * token) and dS_out (gradient w.r.t. the state after a chunk's last token,
 * before that chunk's own output terms are added) are written out; these are
 * the quantities the chunked form passes between chunks.
 *
 * Build: gcc -O2 -fPIC -shared (no -ffast-math: every sum has a fixed order).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int N, H, HV, K, V, C;
    const int64_t* cu;
    int64_t* choff; /* first global chunk of each sequence, [N+1] */
    double scale;
    const double *q, *k, *v, *g, *beta, *h0, *dout, *dht;
    double *o, *ht, *dq, *dk, *dv, *dg, *dbeta, *dh0, *s_in, *ds_out;
    int n_units;
    int next_unit;
    int failed;
    pthread_mutex_t lock;
} job_t;

/* One token of the forward recurrence, in place on S ([K][V] row-major).
 * Writes S' (the decayed state) to Sp and u to u. */
static void token_step(int K, int V, double* S, double* Sp, double* u,
                       const double* kt, const double* vt, const double* gt,
                       double bt) {
    for (int a = 0; a < K; ++a) {
        double e = exp(gt[a]);
        for (int c = 0; c < V; ++c) Sp[a * V + c] = e * S[a * V + c];
    }
    for (int c = 0; c < V; ++c) u[c] = vt[c];
    for (int a = 0; a < K; ++a) {
        double ka = kt[a];
        for (int c = 0; c < V; ++c) u[c] -= Sp[a * V + c] * ka;
    }
    for (int a = 0; a < K; ++a) {
        double bk = bt * kt[a];
        for (int c = 0; c < V; ++c) S[a * V + c] = Sp[a * V + c] + bk * u[c];
    }
}

static int run_unit(job_t* J, int n, int h) {
    const int H = J->H, HV = J->HV, K = J->K, V = J->V, C = J->C;
    const int G = HV / H;
    const int64_t bos = J->cu[n];
    const int64_t T = J->cu[n + 1] - bos;
    const int64_t nck = (T + C - 1) / C;
    const size_t KV = (size_t)K * V;
    const int do_bwd = (J->dq != NULL);

    double* ck = (double*)malloc((size_t)(nck + 1) * KV * sizeof(double));
    double* St = (double*)malloc((size_t)(C + 1) * KV * sizeof(double));
    double* S = (double*)malloc(KV * sizeof(double));
    double* Sp = (double*)malloc(KV * sizeof(double));
    double* dS = (double*)malloc(KV * sizeof(double));
    double* u = (double*)malloc((size_t)V * sizeof(double));
    double* du = (double*)malloc((size_t)V * sizeof(double));
    double* dSu = (double*)malloc((size_t)K * sizeof(double));
    if (!ck || !St || !S || !Sp || !dS || !u || !du || !dSu) {
        free(ck); free(St); free(S); free(Sp); free(dS); free(u); free(du); free(dSu);
        return 1;
    }

    for (int hv = h * G; hv < h * G + G; ++hv) {
        /* ---------------- forward ---------------- */
        if (J->h0) memcpy(S, J->h0 + ((size_t)n * HV + hv) * KV, KV * sizeof(double));
        else memset(S, 0, KV * sizeof(double));
        for (int64_t t = 0; t < T; ++t) {
            if (t % C == 0) memcpy(ck + (size_t)(t / C) * KV, S, KV * sizeof(double));
            const int64_t row = bos + t;
            const double* qt = J->q + ((size_t)row * H + h) * K;
            const double* kt = J->k + ((size_t)row * H + h) * K;
            const double* vt = J->v + ((size_t)row * HV + hv) * V;
            const double* gt = J->g + ((size_t)row * HV + hv) * K;
            const double bt = J->beta[(size_t)row * HV + hv];
            token_step(K, V, S, Sp, u, kt, vt, gt, bt);
            if (J->o) {
                double* ot = J->o + ((size_t)row * HV + hv) * V;
                for (int c = 0; c < V; ++c) ot[c] = 0.0;
                for (int a = 0; a < K; ++a) {
                    double qa = qt[a];
                    for (int c = 0; c < V; ++c) ot[c] += S[a * V + c] * qa;
                }
                for (int c = 0; c < V; ++c) ot[c] *= J->scale;
            }
        }
        memcpy(ck + (size_t)nck * KV, S, KV * sizeof(double));
        if (J->ht) memcpy(J->ht + ((size_t)n * HV + hv) * KV, S, KV * sizeof(double));
        if (J->s_in)
            for (int64_t i = 0; i < nck; ++i)
                memcpy(J->s_in + ((size_t)(J->choff[n] + i) * HV + hv) * KV, ck + (size_t)i * KV,
                       KV * sizeof(double));
        if (!do_bwd) continue;

        /* ---------------- backward ---------------- */
        if (J->dht) memcpy(dS, J->dht + ((size_t)n * HV + hv) * KV, KV * sizeof(double));
        else memset(dS, 0, KV * sizeof(double));
        for (int64_t seg = nck - 1; seg >= 0; --seg) {
            const int64_t t0 = seg * C;
            const int64_t t1 = (t0 + C < T) ? t0 + C : T;
            const int L = (int)(t1 - t0);
            /* recompute the states of this segment from its checkpoint */
            memcpy(St, ck + (size_t)seg * KV, KV * sizeof(double));
            for (int i = 0; i < L; ++i) {
                const int64_t row = bos + t0 + i;
                memcpy(St + (size_t)(i + 1) * KV, St + (size_t)i * KV, KV * sizeof(double));
                token_step(K, V, St + (size_t)(i + 1) * KV, Sp, u,
                           J->k + ((size_t)row * H + h) * K, J->v + ((size_t)row * HV + hv) * V,
                           J->g + ((size_t)row * HV + hv) * K, J->beta[(size_t)row * HV + hv]);
            }
            for (int i = L - 1; i >= 0; --i) {
                const int64_t row = bos + t0 + i;
                if (i == L - 1 && J->ds_out)
                    memcpy(J->ds_out + ((size_t)(J->choff[n] + seg) * HV + hv) * KV, dS,
                           KV * sizeof(double));
                const double* qt = J->q + ((size_t)row * H + h) * K;
                const double* kt = J->k + ((size_t)row * H + h) * K;
                const double* vt = J->v + ((size_t)row * HV + hv) * V;
                const double* gt = J->g + ((size_t)row * HV + hv) * K;
                const double bt = J->beta[(size_t)row * HV + hv];
                const double* dot = J->dout ? J->dout + ((size_t)row * HV + hv) * V : NULL;
                const double* Snew = St + (size_t)(i + 1) * KV;
                const double* Sold = St + (size_t)i * KV;
                double* dqt = J->dq + ((size_t)row * H + h) * K;
                double* dkt = J->dk + ((size_t)row * H + h) * K;
                double* dvt = J->dv + ((size_t)row * HV + hv) * V;
                double* dgt = J->dg + ((size_t)row * HV + hv) * K;

                /* output term o_t = scale * S_t^T q_t */
                if (dot) {
                    for (int a = 0; a < K; ++a) {
                        double acc = 0.0;
                        for (int c = 0; c < V; ++c) acc += Snew[a * V + c] * dot[c];
                        dqt[a] += J->scale * acc;
                    }
                    for (int a = 0; a < K; ++a) {
                        double sq = J->scale * qt[a];
                        for (int c = 0; c < V; ++c) dS[a * V + c] += sq * dot[c];
                    }
                }
                /* S' and u of this token */
                for (int a = 0; a < K; ++a) {
                    double e = exp(gt[a]);
                    for (int c = 0; c < V; ++c) Sp[a * V + c] = e * Sold[a * V + c];
                }
                for (int c = 0; c < V; ++c) u[c] = vt[c];
                for (int a = 0; a < K; ++a)
                    for (int c = 0; c < V; ++c) u[c] -= Sp[a * V + c] * kt[a];
                /* write term S_t = S' + beta k u^T */
                for (int c = 0; c < V; ++c) du[c] = 0.0;
                for (int a = 0; a < K; ++a)
                    for (int c = 0; c < V; ++c) du[c] += dS[a * V + c] * kt[a];
                for (int c = 0; c < V; ++c) du[c] *= bt;
                for (int a = 0; a < K; ++a) {
                    double acc = 0.0;
                    for (int c = 0; c < V; ++c) acc += dS[a * V + c] * u[c];
                    dSu[a] = acc;
                }
                double db = 0.0;
                for (int a = 0; a < K; ++a) db += kt[a] * dSu[a];
                J->dbeta[(size_t)row * HV + hv] = db;
                for (int c = 0; c < V; ++c) dvt[c] = du[c];
                for (int a = 0; a < K; ++a) {
                    double acc = 0.0;
                    for (int c = 0; c < V; ++c) acc += Sp[a * V + c] * du[c];
                    dkt[a] += bt * dSu[a] - acc;
                }
                /* u = v - S'^T k and S_t = S' + ... : dS' = dS - k du^T */
                for (int a = 0; a < K; ++a)
                    for (int c = 0; c < V; ++c) dS[a * V + c] -= kt[a] * du[c];
                /* S' = Diag(exp g) S_{t-1} */
                for (int a = 0; a < K; ++a) {
                    double acc = 0.0;
                    for (int c = 0; c < V; ++c) acc += dS[a * V + c] * Sp[a * V + c];
                    dgt[a] = acc;
                    double e = exp(gt[a]);
                    for (int c = 0; c < V; ++c) dS[a * V + c] *= e;
                }
            }
        }
        if (J->dh0) memcpy(J->dh0 + ((size_t)n * HV + hv) * KV, dS, KV * sizeof(double));
    }
    free(ck); free(St); free(S); free(Sp); free(dS); free(u); free(du); free(dSu);
    return 0;
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int idx = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (idx >= J->n_units) break;
        int n = idx / J->H, h = idx % J->H;
        if (run_unit(J, n, h)) {
            pthread_mutex_lock(&J->lock);
            J->failed = 1;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

/* Number of chunks of size C over all sequences (ceil per sequence). */
int64_t kda_oracle_num_chunks(const int64_t* cu, int N, int C) {
    int64_t total = 0;
    for (int n = 0; n < N; ++n) total += (cu[n + 1] - cu[n] + C - 1) / C;
    return total;
}

/*
 * Forward (and, when dq != NULL, backward) over all sequences and heads.
 * Layouts (row = packed token index):
 *   q, k, dq, dk : [rows, H, K]      v, do, o, dv : [rows, HV, V]
 *   g, dg        : [rows, HV, K]     beta, dbeta  : [rows, HV]
 *   h0, ht, dht, dh0 : [N, HV, K, V] s_in, ds_out : [num_chunks, HV, K, V]
 * dq, dk must be zero on entry (they accumulate over the value heads of a
 * group). Nullable: h0, dht, do (= zero), o, ht, s_in, ds_out, and the whole
 * backward set (dq, dk, dv, dg, dbeta, dh0 together; dh0 alone may be NULL).
 * nthreads <= 0 uses every online core. Returns 0 on success.
 */
int kda_oracle_run(int N, const int64_t* cu, int H, int HV, int K, int V, int C, double scale,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, const double* h0, const double* dout, const double* dht,
                   double* o, double* ht, double* dq, double* dk, double* dv, double* dg,
                   double* dbeta, double* dh0, double* s_in, double* ds_out, int nthreads) {
    if (N <= 0 || H <= 0 || HV <= 0 || HV % H != 0 || K <= 0 || V <= 0 || C <= 0) return 2;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return 2;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.N = N; J.H = H; J.HV = HV; J.K = K; J.V = V; J.C = C; J.cu = cu; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0; J.dout = dout; J.dht = dht;
    J.o = o; J.ht = ht; J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dh0 = dh0;
    J.s_in = s_in; J.ds_out = ds_out;
    J.choff = (int64_t*)malloc((size_t)(N + 1) * sizeof(int64_t));
    if (!J.choff) return 1;
    J.choff[0] = 0;
    for (int n = 0; n < N; ++n) J.choff[n + 1] = J.choff[n] + (cu[n + 1] - cu[n] + C - 1) / C;
    J.n_units = N * H;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads > J.n_units) nthreads = J.n_units;
    if (nthreads < 1) nthreads = 1;
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started;
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    free(J.choff);
    return J.failed ? 1 : 0;
}
