// Internal interfaces between the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

struct Prob;

// Caller tensors of one call (device pointers; see include/kda.h for layouts).
struct IO {
    const void *q, *k, *v, *beta, *d_o;
    const float *g, *h0, *dht;
    void *o, *dq, *dk, *dv, *dbeta;
    float *ht, *states_out, *dg, *dh0;
    const float* states_in;  // the forward's saved chunk states (backward), or null
};

// Workspace carved from the caller's buffer (fp32 unless noted).
//   per token and value head:   gam [R,HV,K] (log2 cumsum), w [R,HV,K],
//     u [R,HV,V], vn (delta) [R,HV,V], dvn (d_delta) [R,HV,V], dqt, dkh, dw
//     [R,HV,K], dqp, dkp [R,HV,K] (per-value-head dq/dk before the group sum)
//   per chunk and value head:   inv, aqk [NT,HV,C,C], sin, dso [NT,HV,K,V],
//     dgc [NT,HV,K]
//   status: device status word(s) written by bounded waits.
struct Ws {
    float *gam, *w, *u, *vn, *dvn, *dqt, *dkh, *dw, *dqp, *dkp;
    float *inv, *aqk, *sin, *dso, *dgc;
    int* status;
};

// Launch bookkeeping of the current call: begin_launches() at the start of a
// call, note_launch() right after every kernel launch (records the caller's
// profiling events, if any, and the launch name).
void begin_launches(cudaStream_t st);
void note_launch(const char* name, cudaStream_t st);

cudaError_t simt_fwd(const Prob& p, bool bf16, const IO& io, const Ws& ws, cudaStream_t st);
cudaError_t simt_bwd(const Prob& p, bool bf16, const IO& io, const Ws& ws, cudaStream_t st);

// Workspace of the tensor-core path (bf16, K = V = 128). Per chunk-head
// ch = chunk * HV + hv, bf16 tiles in the operand layout of tc_util.cuh:
//   w, kh (K^), qs (scale Q~), vn (delta), dvn (d_delta): 64 x 128 (16 KB)
//   aqk, inv, invb (INV diag(beta)): 64 x 64 (8 KB);  sin, dso: 128 x 128 (32 KB)
//   egc: 128 fp32 (e^Gamma_C per key channel)
// dqp, dkp (grouped value heads only): per gradient-kernel CTA, the running fp32 dq / dk sum of a
// (chunk, key head) group over its value heads, 64 x 128 values in the CTA's thread order.
constexpr int kGradsMaxCtas = 256;
struct TcWs {
    uint8_t *w, *invb, *kh, *qs, *vn, *dvn, *aqk, *inv, *sin, *dso;
    float *egc, *dqp, *dkp;
    // segmented state passes (long sequences, few sweeps): per (sequence, value head, segment) fp32
    // K x V end states from a zero start, K x K transitions and start states
    float *seg_e, *seg_p, *seg_s0;
    // packed sequences: the sequence indices by decreasing chunk count (the order in which the sweeps of the
    // state passes are launched, longest first), or null for the natural order
    int* seq_order;
    int* status;
};

#ifdef __CUDACC__
// The sequence of the y-th sweep row of a state-pass launch (grid y = sequence).
__device__ __forceinline__ int sweep_seq(const TcWs& ws, int y) { return ws.seq_order ? ws.seq_order[y] : y; }
#endif

// Segmented sweeps of the state passes: segment m of a sequence covers chunks
// [m * len, min((m + 1) * len, chunks)); len = 0 means no segmentation.
// Chosen from the problem alone (dense batches with few sweeps and long sequences).
struct SegPlan {
    int len, M;
};
SegPlan seg_plan(const Prob& p);

// The tensor-core path handles bf16 inputs with K = V = 128.
bool tc_path_ok(const Prob& p, bool bf16);
// The tensor-core forward: intra, state pass (ht and the fp32 chunk states
// when requested), output.
cudaError_t tc_fwd(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st);
// Runs the first `stages` stages of the tensor-core backward (1: intra,
// 2: + state pass, or the load of io.states_in, 3: + reverse pass,
// 4: + gradients). With from_saved, the workspace holds a saved context (the
// forward's intra tiles, S_in and delta, written by tc_fwd into a backward-
// layout workspace) and stages 1 and 2 are skipped. With fused, stages 3 and 4 run as one launch
// (tc_rev_fused; equal key and value heads only).
cudaError_t tc_bwd(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st, int stages, bool from_saved = false,
                   bool fused = false);
// The per-chunk gradient stage (dq, dk summed over the value heads of a group in the same kernel).
cudaError_t tc_grads(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st);
// The fused reverse: per (sequence, value head) a cluster of three CTAs, one running the reverse
// state-gradient sweep and two the per-chunk gradients of its chunks (alternate chunks each), dS_out
// and d_delta passed to them in shared memory (H == HV).
cudaError_t tc_rev_fused(const Prob& p, const IO& io, const TcWs& ws, cudaStream_t st);

}  // namespace kda
