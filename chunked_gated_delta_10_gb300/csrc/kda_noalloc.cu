// kda_chunk_bwd_noalloc: the backward for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the backward: a plugin executing inside another engine's
// enqueue/execute phase, where allocation is forbidden or would implicitly
// synchronise the device; or a process whose device memory is entirely
// reserved up front by another allocator. Such callers also cannot hand the
// library a workspace of their own. This entry point therefore takes its
// scratch from a fixed-size array in the library's own device memory (a
// file-scope __device__ array below), so the caller passes only its inputs and
// outputs.
//
// Properties of that scratch:
//   - Its size is fixed (KDA_NOALLOC_SCRATCH_BYTES). Every GPU that loads this
//     part of the library holds it until the process exits. With CUDA's lazy
//     module loading the array is committed when this file's module is first
//     loaded on a device, i.e. at the first kda_noalloc_prepare or
//     kda_chunk_bwd_noalloc call there: that first call needs 64 MiB of free
//     device memory and belongs in the caller's set-up phase.
//   - The cached address is valid for the life of the device's context; after
//     a device reset, call kda_noalloc_prepare again before the next call.
//   - All calls share it, and it keeps the last call's contents. The backward
//     fully writes every scratch region before reading it; the one word that
//     must start at zero (the device status word) is cleared by every call on
//     the call's stream. Calls whose execution overlaps on the GPU (several
//     streams, or several host threads) race on the scratch and give wrong
//     results: serialise them.
#include <mutex>

#include "../../include/kda.h"

namespace {

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is obtained with
// cudaGetSymbolAddress while that device is current: once per device, or again
// when `refresh` is set (kda_noalloc_prepare, e.g. after a device reset).
kda_status scratch_address(void** out, bool refresh) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_setup_lock);
    if (!g_scratch_ptr[dev] || refresh) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_noalloc_prepare(void) {
    void* scratch = nullptr;
    return scratch_address(&scratch, true);
}

extern "C" kda_status kda_chunk_bwd_noalloc(const kda_dims* dims, const void* q, const void* k, const void* v,
                                            const float* g, const void* beta, const float* h0,
                                            const int64_t* cu_seqlens, const int32_t* chunk_idx,
                                            const int64_t* chunk_off, const void* d_o, const float* dht, void* dq,
                                            void* dk, void* dv, float* dg, void* dbeta, float* dh0,
                                            kda_stream_t stream) {
    const size_t need = kda_workspace_bytes(dims, KDA_PASS_BWD);
    if (need == 0)  // invalid dims: let the regular validation name the error (nothing is launched)
        return kda_chunk_bwd(dims, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, d_o, dht, nullptr, dq, dk,
                             dv, dg, dbeta, dh0, nullptr, 0, stream);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const kda_status s = scratch_address(&scratch, false);
    if (s != KDA_OK) return s;
    return kda_chunk_bwd(dims, q, k, v, g, beta, h0, cu_seqlens, chunk_idx, chunk_off, d_o, dht, nullptr, dq, dk,
                         dv, dg, dbeta, dh0, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}

// The status word sits at the start of the scratch, where kda_chunk_bwd places it in any workspace.
extern "C" kda_status kda_noalloc_device_status(kda_stream_t stream) {
    void* scratch = nullptr;
    const kda_status s = scratch_address(&scratch, false);
    if (s != KDA_OK) return s;
    return kda_device_status(scratch, stream);
}
