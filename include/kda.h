/*
 * kda.h — C ABI of the GB300 (sm_103a) chunk-parallel Kimi Delta Attention
 * library: the forward with saved chunk states, and the backward that
 * recomputes the forward it needs (or consumes saved states) and returns every
 * input gradient.
 *
 * The operation (Kimi Delta Attention, a gated delta rule with one decay per
 * key channel), per sequence and value head, with state S in R^{K x V}:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t,      S_0 = h0 (or 0),   ht = S_T
 *
 * computed in chunks of 64 tokens: an in-chunk cumulative sum of the gates,
 * the decayed in-chunk triangles Akk / Aqk and the WY inverse
 * (I + Akk)^{-1} (the "recompute w, u" step and the fused w/y kernel of FLA's
 * chunk_bwd.py page; "Step 1: Recompute U" of the FlashKDA backward (K2)
 * page), a sequential state pass over chunks, a reverse sequential pass of the
 * state gradient seeded by dht (the "bwd_dhu" step of chunk_kda_bwd, the
 * reverse chunk loop of the K2 kernel), per-chunk gradients, the reverse
 * in-chunk cumsum of dg, and the reduction of dq/dk over grouped value heads.
 *
 * Conventions for every entry point below:
 *   - Tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *     16-byte aligned, in the layouts listed. Outputs are fully overwritten.
 *   - Nothing here allocates device memory: scratch comes from the caller's
 *     workspace (size from kda_workspace_bytes). Kernels are enqueued on
 *     `stream` (a cudaStream_t, or NULL for the legacy default stream) and the
 *     calls return without synchronising.
 *   - Errors are returned as kda_status codes; nothing aborts or throws
 *     across the ABI. Argument errors are detected before any launch.
 *   - Layouts (row = packed token index b*T + t, or the cu_seqlens offset):
 *       q, k, dq, dk       [B, T, H,  K]   dtype (bf16 or fp32)
 *       v, do, o, dv       [B, T, HV, V]   dtype
 *       g, dg              [B, T, HV, K]   fp32, natural-log per-token decay
 *                                          (NOT cumsummed; dg is w.r.t. it)
 *       beta, dbeta        [B, T, HV]      dtype (post-sigmoid gate)
 *       h0, ht, dht, dh0   [N, HV, K, V]   fp32
 *       states             [num_chunks, HV, K, V] fp32: S entering each chunk
 *       cu_seqlens         int64 [N + 1]   (packed sequences; then B == 1)
 *       chunk_idx          int32 [num_chunks][2] = (sequence, chunk in seq);
 *                          may be NULL when num_chunks == 0
 *       chunk_off          int64 [N + 1]   first global chunk of each sequence
 *   - Value head hv reads key head hv / (HV / H).
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* kda_stream_t; /* a cudaStream_t */

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,    /* bad size, null or misaligned pointer, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. K not in {64,128}) */
    KDA_ERR_WORKSPACE = 3,      /* workspace null or smaller than kda_workspace_bytes */
    KDA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    KDA_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait gave up (see kda_device_status) */
} kda_status;

typedef enum { KDA_DTYPE_BF16 = 0, KDA_DTYPE_F32 = 1 } kda_dtype;

typedef enum { KDA_PASS_FWD = 0, KDA_PASS_BWD = 1 } kda_pass;

/*
 * Problem description.
 *   B, T      batch and tokens per sequence; with packed sequences B == 1 and
 *             T is the total packed length.
 *   H, HV     key heads and value heads, HV % H == 0.
 *   K, V      key and value head dims; each must be 64 or 128.
 *   chunk     must be 64 (the chunk size of the pages' kernels).
 *   num_seqs  N: B without cu_seqlens, len(cu_seqlens) - 1 with.
 *   num_chunks total chunks over all sequences (kda_prepare_chunks computes
 *             it for packed sequences; B * ceil(T / 64) otherwise).
 *   dtype     kda_dtype of q, k, v, beta, do and of o, dq, dk, dv, dbeta.
 *   scale     output scale (commonly K^-0.5).
 */
typedef struct {
    int32_t B, T, H, HV, K, V;
    int32_t chunk;
    int32_t num_seqs;
    int64_t num_chunks;
    int32_t dtype;
    float scale;
} kda_dims;

/* Human-readable name of a status code (static string). */
const char* kda_status_string(kda_status s);

/*
 * Build the chunk table of packed sequences on the host (the chunk index path
 * of the pages' varlen kernels, "prepare_chunk_indices"). Call once with
 * chunk_idx_host == NULL and chunk_off_host == NULL to get *num_chunks, then
 * again with buffers of 2 * num_chunks int32 and num_seqs + 1 int64.
 * cu_seqlens_host: HOST int64 [num_seqs + 1], cu[0] == 0, non-decreasing.
 * Empty sequences are allowed (they own no chunk).
 * Errors: KDA_ERR_INVALID_ARG on a null cu_seqlens/num_chunks, num_seqs < 1,
 * chunk != 64, or a decreasing / nonzero-starting cu_seqlens.
 */
kda_status kda_prepare_chunks(const int64_t* cu_seqlens_host, int32_t num_seqs, int32_t chunk,
                              int32_t* chunk_idx_host, int64_t* chunk_off_host, int64_t* num_chunks);

/* Bytes of device workspace kda_chunk_fwd (pass = KDA_PASS_FWD) or
 * kda_chunk_bwd (KDA_PASS_BWD) needs for these dims; 0 if dims are invalid. */
size_t kda_workspace_bytes(const kda_dims* dims, int32_t pass);

/*
 * Chunked forward: o, the final state ht and the state entering every chunk.
 *   q, k, v, g, beta (and optional h0) as in the layouts above.
 *   cu_seqlens, chunk_idx, chunk_off: all NULL (B equal-length sequences) or
 *     all non-NULL device arrays (packed sequences, B == 1); chunk_idx may be
 *     NULL for a packed batch with no chunk (every sequence empty).
 *   o: required. ht, states: nullable (skipped when NULL).
 *   ws / ws_bytes: device workspace of at least kda_workspace_bytes(FWD).
 * Errors: KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE before
 * any launch; KDA_ERR_CUDA if a launch fails.
 */
kda_status kda_chunk_fwd(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                         const void* beta, const float* h0, const int64_t* cu_seqlens, const int32_t* chunk_idx,
                         const int64_t* chunk_off, void* o, float* ht, float* states, void* ws, size_t ws_bytes,
                         kda_stream_t stream);

/*
 * Chunked backward of L = sum(o * do) + sum(ht * dht): dq, dk (already summed
 * over each key head's value heads), dv, dg, dbeta and dh0.
 *   do: required; dht: nullable (zero).
 *   states: NULL to recompute the forward state pass inside the call (the
 *     default recompute path); or the states saved by kda_chunk_fwd for the
 *     same inputs, which replaces the sequential forward state pass by a
 *     chunk-parallel load (bf16 with K = V = 128 only; KDA_ERR_UNSUPPORTED
 *     otherwise). With the states of the same build's forward the results
 *     equal the recompute path's bit for bit.
 *   dh0: nullable; must be NULL when h0 is NULL.
 *   Other arguments as kda_chunk_fwd; ws of at least kda_workspace_bytes(BWD).
 * Errors: as kda_chunk_fwd.
 */
kda_status kda_chunk_bwd(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                         const void* beta, const float* h0, const int64_t* cu_seqlens, const int32_t* chunk_idx,
                         const int64_t* chunk_off, const void* d_o, const float* dht, const float* states,
                         void* dq, void* dk, void* dv, float* dg, void* dbeta, float* dh0, void* ws,
                         size_t ws_bytes, kda_stream_t stream);

/*
 * Backward with a fused reverse pass: the same results as kda_chunk_bwd, bit
 * for bit, with the reverse state-gradient sweep and the per-chunk gradients
 * run as one launch in which the state gradient never leaves the chip (the
 * structure of the FlashKDA backward (K2) page's kernel: one sweep per
 * (sequence, head) over the chunks from last to first with dS resident in
 * shared memory, the per-chunk gradient work inside the sweep).
 * Per (sequence, value head) a cluster of three CTAs on three SMs: one carries
 * dS in registers through the sweep, the other two compute the chunks' dq, dk,
 * dv, dbeta and dg (alternate chunks each); each chunk's dS_out and d_delta
 * tiles pass from the first to the one that takes the chunk through
 * distributed shared memory instead of the workspace.
 * Arguments, layouts, workspace and errors as kda_chunk_bwd, plus
 * KDA_ERR_UNSUPPORTED off the tensor-core path (bf16, K = V = 128) or when
 * HV != H. The split path (kda_chunk_bwd) is the faster one on the workloads
 * measured here; this entry point is the alternative structure.
 */
kda_status kda_chunk_bwd_fused(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                               const void* beta, const float* h0, const int64_t* cu_seqlens, const int32_t* chunk_idx,
                               const int64_t* chunk_off, const void* d_o, const float* dht, const float* states,
                               void* dq, void* dk, void* dv, float* dg, void* dbeta, float* dh0, void* ws,
                               size_t ws_bytes, kda_stream_t stream);

/*
 * Backward from a saved forward context (bf16 inputs with K = V = 128 only).
 *
 * The backward needs, per chunk, the WY factors (w, INV, INV diag(beta)), the
 * decayed key/query factors, the in-chunk triangle Aqk, e^Gamma_C, the state
 * entering the chunk and delta = u - w S_in: the quantities FLA's chunk_kda_bwd
 * takes from the forward instead of recomputing them when recomputation is
 * disabled (the "FLA chunk_bwd.py" page: w, u, qg, kg, v_new and h of its
 * disable_recompute branch). kda_chunk_fwd_save runs the forward and keeps all
 * of them, as bf16 tiles in the layout the backward's MMAs read, in `saved`;
 * kda_chunk_bwd_from_saved then runs only the reverse state-gradient pass and
 * the per-chunk gradients (no intra-chunk pass, no forward state pass). Its
 * results equal kda_chunk_bwd's bit for bit on the same inputs.
 *
 * kda_saved_bytes: bytes of the saved context for these dims (equal to
 *   kda_workspace_bytes(dims, KDA_PASS_BWD)); 0 if the dims are invalid or not
 *   on this path (not bf16 with K = V = 128).
 * kda_chunk_fwd_save: as kda_chunk_fwd (o, ht; no fp32 states) and writes the
 *   context into `saved` (device, 16-byte aligned, at least kda_saved_bytes).
 * kda_chunk_bwd_from_saved: as kda_chunk_bwd with `saved` (from
 *   kda_chunk_fwd_save on the same inputs and dims) as both the saved context
 *   and the workspace. It reads the context and overwrites only the backward's
 *   own scratch regions of the buffer, so it may be called again with the same
 *   buffer. Calls that overlap on the GPU with the same buffer race.
 * Errors: those of kda_chunk_fwd / kda_chunk_bwd; KDA_ERR_UNSUPPORTED off this
 * path; KDA_ERR_WORKSPACE when `saved` is null, misaligned or too small.
 * kda_device_status(saved, stream) reports bounded device waits of either call.
 */
size_t kda_saved_bytes(const kda_dims* dims);
kda_status kda_chunk_fwd_save(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                              const void* beta, const float* h0, const int64_t* cu_seqlens, const int32_t* chunk_idx,
                              const int64_t* chunk_off, void* o, float* ht, void* saved, size_t saved_bytes,
                              kda_stream_t stream);
kda_status kda_chunk_bwd_from_saved(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                                    const void* beta, const float* h0, const int64_t* cu_seqlens,
                                    const int32_t* chunk_idx, const int64_t* chunk_off, const void* d_o,
                                    const float* dht, void* saved, size_t saved_bytes, void* dq, void* dk, void* dv,
                                    float* dg, void* dbeta, float* dh0, kda_stream_t stream);

/*
 * Status word that device-side bounded waits write into the workspace of the
 * last call (KDA_OK when none gave up). Synchronises `stream`, then reads it.
 * ws: the workspace passed to that call.
 */
kda_status kda_device_status(const void* ws, kda_stream_t stream);

/*
 * Backward without a caller workspace, for callers that cannot allocate.
 *
 * Some callers cannot call cudaMalloc or any other allocating routine where
 * they run the backward (for example a plugin running inside another
 * engine's enqueue/execute phase, where allocation is forbidden or would
 * synchronise the device, or a process whose device memory is all reserved by
 * another allocator), so they cannot pass a workspace either. This variant of
 * kda_chunk_bwd (always the recompute path: no saved states) uses a fixed
 * scratch array of KDA_NOALLOC_SCRATCH_BYTES that the library keeps in device
 * memory on every GPU that loads it, until the process exits. It allocates
 * nothing; the caller still passes every input and output, as for
 * kda_chunk_bwd.
 *   - Set-up: the array's device address is looked up once per device, with
 *     that device current, by kda_noalloc_prepare (or by the first call on
 *     the device if prepare was not called). With CUDA's lazy module loading
 *     that first look-up also loads the module and commits the 64 MiB array,
 *     so it needs that much free device memory: call kda_noalloc_prepare in
 *     the caller's set-up phase, before any execute phase or stream capture.
 *   - The address stays valid for the life of the device's context; after a
 *     device reset (cudaDeviceReset), call kda_noalloc_prepare again.
 *   - Every call shares the one array and it keeps the last call's contents
 *     (each call clears the status word it needs at zero). Calls whose
 *     execution overlaps on the GPU (several streams or host threads) race
 *     on it: serialise them.
 *   - Errors: those of kda_chunk_bwd, returned before any launch, plus
 *     KDA_ERR_WORKSPACE when the problem needs more than
 *     KDA_NOALLOC_SCRATCH_BYTES (kda_workspace_bytes(dims, KDA_PASS_BWD) >
 *     KDA_NOALLOC_SCRATCH_BYTES). A bounded device wait that gives up is
 *     reported by kda_noalloc_device_status, not by the call itself.
 * This entry point has no counterpart in the paper; it is a deployment aid.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
kda_status kda_chunk_bwd_noalloc(const kda_dims* dims, const void* q, const void* k, const void* v, const float* g,
                                 const void* beta, const float* h0, const int64_t* cu_seqlens,
                                 const int32_t* chunk_idx, const int64_t* chunk_off, const void* d_o,
                                 const float* dht, void* dq, void* dk, void* dv, float* dg, void* dbeta, float* dh0,
                                 kda_stream_t stream);

/* Set-up of kda_chunk_bwd_noalloc on the current device: loads the module and
 * looks up (again) the scratch array's device address. Allocates nothing
 * beyond the module's own static array. KDA_ERR_CUDA if the look-up fails. */
kda_status kda_noalloc_prepare(void);

/* kda_device_status for kda_chunk_bwd_noalloc: synchronises `stream`, then
 * reads the status word the last call on the current device left in the
 * shared scratch (KDA_OK, or KDA_ERR_DEVICE_TIMEOUT if a bounded wait gave up). */
kda_status kda_noalloc_device_status(kda_stream_t stream);

/*
 * Per-kernel timing hook (for benchmarks and profiling; off by default).
 * After kda_set_profile_events(events, n) with n >= 1 caller-created
 * cudaEvent_t handles, every later kda_chunk_fwd / kda_chunk_bwd call records
 * events[0] on its stream before its first kernel and events[i + 1] right
 * after its i-th kernel launch (while i + 1 < n). The elapsed time between
 * consecutive events is then the device time of each launch in stream order.
 * kda_set_profile_events(NULL, 0) turns it off. Process-wide setting; not for
 * concurrent use from several host threads. Errors: KDA_ERR_INVALID_ARG if
 * events is NULL with n > 0, or n < 0.
 */
kda_status kda_set_profile_events(void* const* events, int32_t n_events);

/* Number of kernel launches the last kda_chunk_fwd / kda_chunk_bwd call made
 * on this host thread, and the name of the i-th (static string, NULL if out of range). */
int32_t kda_last_launch_count(void);

/* Text of the CUDA error behind the last KDA_ERR_CUDA returned on this host
 * thread (static string; "no error" if none). */
const char* kda_last_cuda_error(void);
const char* kda_launch_name(int32_t i);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
