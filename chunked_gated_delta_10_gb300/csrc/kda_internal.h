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

}  // namespace kda
