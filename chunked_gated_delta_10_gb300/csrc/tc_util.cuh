// Blackwell (sm_100 family, built for sm_103a) tensor-core, TMEM, TMA and
// mbarrier primitives as inline PTX, used by the KDA tensor-core kernels.
//
// Shared-memory operand convention: every bf16 operand tile is a row-major
// matrix X[R][cols] stored as blocks of 64 columns (128 bytes per row), each
// block R x 128 B with the 128-byte swizzle (16-byte chunk c of row r stored at
// chunk c ^ (r % 8)); blocks follow each other every R * 128 bytes and the
// tile base is 1024-byte aligned. This is exactly what a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B and a {64, R} box writes. The same tile serves as
//   - a K-major operand (rows = M or N, reduction over the columns), or
//   - an MN-major operand (columns = M or N, reduction over the rows),
// selected by the shared-memory descriptor and the instruction descriptor.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {
namespace tc {

// A bounded wait gives up after this many SM clock cycles (about 1 s).
constexpr long long kWaitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait for phase `parity` of `bar` to complete, for at most `limit` SM cycles.
// On time-out, writes `code` to *status (if non-null) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, int code,
                                         long long limit = kWaitCycles) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (clock64() - t0 > limit) {
            if (status) *(volatile int*)status = code;
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------- fences
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// --------------------------------------------------------------------- TMEM
// Executed by one full warp. Writes the TMEM base address to *dst (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of warp w (w % 4 = q)
// receives lane 32q + t, columns col .. col+31 (taddr = base + (32q << 16) + col).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// As tmem_ld32 with 8 consecutive columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// As tmem_ld8, raw 32-bit values.
__device__ __forceinline__ void tmem_ld8u(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
// As tmem_ld32 with 4 consecutive columns.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float* v) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
// As tmem_ld4, raw 32-bit values.
__device__ __forceinline__ void tmem_ld4u(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
// Store 8 consecutive 32-bit columns of this thread's lane (same addressing as tmem_ld32);
// tmem_st_wait() completes the warp's outstanding stores.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
// As tmem_st8 with 4 consecutive columns.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// As tmem_ld32 with 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version
    d |= (uint64_t)2 << 61;  // SWIZZLE_128B
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Descriptor of the 16-deep reduction step `ks` of an operand tile (see the
// convention at the top). K-major: tile rows = M/N, reduction along columns.
// The start-address field holds (address >> 4) in 14 bits, and shared-memory
// addresses stay below 2^18 bytes, so the descriptor of (tile + off) is the
// tile's descriptor plus off >> 4: one add per K step once the tile's
// descriptor is formed (offsets are compile-time constants in unrolled loops).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int rows, int ks) {
    return sdesc(tile, 16, 1024) + (uint64_t)(((ks >> 2) * rows * 128 + (ks & 3) * 32) >> 4);
}
// MN-major: tile rows = reduction, columns = M/N (blocks of 64 columns).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int rows, int ks) {
    return sdesc(tile, (uint32_t)(rows * 128), 1024) + (uint64_t)((ks * 16 * 128) >> 4);
}

// D[tmem] (+)= A * B^T, one instruction of K = 16 (issued by one thread).
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Byte offset of element (r, c) of a bf16 operand tile with R rows (see top).
__device__ __forceinline__ uint32_t tile_off(int r, int c, int R) {
    const uint32_t off = (uint32_t)((c >> 6) * R * 128 + r * 128 + (c & 63) * 2);
    return off ^ (((off >> 7) & 7u) << 4);
}


// ------------------------------------------------- tiles, bulk copies, waits
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ void st_tile(uint8_t* tile, int r, int c, int R, float x) {
    *reinterpret_cast<__nv_bfloat16*>(tile + tile_off(r, c, R)) = __float2bfloat16_rn(x);
}
__device__ __forceinline__ float ld_tile(const uint8_t* tile, int r, int c, int R) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + tile_off(r, c, R)));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// Row r, columns c0 .. c0+7 of a tile with R rows, as one 16-byte store.
__device__ __forceinline__ void st_tile_row8(uint8_t* tile, int r, int c0, int R, const float* x) {
    uint4 v;
    v.x = pack2(x[0], x[1]);
    v.y = pack2(x[2], x[3]);
    v.z = pack2(x[4], x[5]);
    v.w = pack2(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + tile_off(r, c0, R)) = v;
}

// Row r, columns c0 .. c0+7 of a bf16 tile with R rows, as one 16-byte load.
__device__ __forceinline__ void ld_tile_row8(const uint8_t* tile, int r, int c0, int R, float* x) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + tile_off(r, c0, R));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// The same 16 bytes unconverted, and element i (0..7) of such a group as fp32.
__device__ __forceinline__ uint4 ld_raw16(const uint8_t* tile, int r, int c0, int R) {
    return *reinterpret_cast<const uint4*>(tile + tile_off(r, c0, R));
}
__device__ __forceinline__ float bf16_at(const uint4& v, int i) {
    const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
    return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
}

// Bulk copy shared -> global (16-byte aligned, size % 16 == 0) and its group ops.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster; orders each thread's earlier accesses (and mbarrier inits
// fenced by fence_mbar_init) before the other CTAs' later ones.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address in the shared memory of cluster CTA `rank` of the variable at this CTA's shared address `a`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Bulk copy from this CTA's shared memory into another cluster CTA's (dst and its mbarrier as
// peer_addr addresses; 16-byte aligned, size % 16 == 0). Completion is counted in bytes on that
// mbarrier; nothing here tells when the source has been read.
__device__ __forceinline__ void bulk_push(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "r"(smem_u32(src)), "r"(bytes), "r"(mbar)
                 : "memory");
}
// Arrive on another cluster CTA's mbarrier (a peer_addr address), releasing this thread's earlier
// accesses at cluster scope.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t mbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// Bounded wait on this CTA's mbarrier whose arrivals come from other CTAs of the cluster (acquire at
// cluster scope); on time-out writes `code` to *status and returns false.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status, int code) {
    auto poll = [&]() {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        return done != 0;
    };
    if (poll()) return true;
    const long long t0 = clock64();
    while (!poll()) {
        if (clock64() - t0 > kWaitCycles) {
            if (status) *(volatile int*)status = code;
            return false;
        }
    }
    return true;
}

// Negated-A variant of the __nv_bfloat16 instruction descriptor.
__host__ __device__ constexpr uint32_t idesc_neg_a(uint32_t id) { return id | (1u << 13); }

// Barrier 1 over threads 0 .. N-1 of the block (a multiple of 32): the group of
// warps that shares a phase while other warps of the block run on their own.
template <int N>
__device__ __forceinline__ void group_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Uniform bounded wait on (bar, parity): warp 0 polls the barrier while the other
// warps park in the CTA barrier (issuing nothing); the barrier then orders the
// observed completion before every thread's later accesses (callers that read
// TMEM next add tcgen05.fence::after_thread_sync). If the poll gives up, *fail
// becomes nonzero for all after the barrier.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int* status, int code, int* fail) {
    if (threadIdx.x < 32 && !mbar_wait(bar, parity, status, code)) *(volatile int*)fail = 1;
    __syncthreads();
    return *(volatile int*)fail == 0;
}
// wait_all on two barriers at once: one poll by warp 0 of each, then one CTA barrier.
__device__ __forceinline__ bool wait_all2(uint64_t* bar_a, uint32_t par_a, int code_a, uint64_t* bar_b, uint32_t par_b,
                                          int code_b, int* status, int* fail) {
    if (threadIdx.x < 32 && (!mbar_wait(bar_a, par_a, status, code_a) || !mbar_wait(bar_b, par_b, status, code_b)))
        *(volatile int*)fail = 1;
    __syncthreads();
    return *(volatile int*)fail == 0;
}
// Per-warp bounded wait (every lane polls, so every lane acquires the completed phase): no CTA barrier. On
// time-out *fail becomes nonzero and the warp goes on; the caller's next group barrier reads *fail and
// leaves the loop, so that no warp waits at a barrier another warp has left.
__device__ __forceinline__ void warp_wait(uint64_t* bar, uint32_t parity, int* status, int code, int* fail) {
    if (!mbar_wait(bar, parity, status, code)) *(volatile int*)fail = 1;
    __syncwarp();
}
// The same for the group of threads 0 .. N-1 (group_sync); *fail must be written
// by no thread outside the group, so that every thread of the group reads the
// same value after the barrier.
template <int N>
__device__ __forceinline__ bool wait_group(uint64_t* bar, uint32_t parity, int* status, int code, int* fail) {
    if (threadIdx.x < 32 && !mbar_wait(bar, parity, status, code)) *(volatile int*)fail = 1;
    group_sync<N>();
    return *(volatile int*)fail == 0;
}

// Column addressing of a bf16 operand tile: for a fixed column c, the byte offset
// of element (r, c) is o[r % 8] + 128 r (the swizzle only permutes the 16-byte
// chunks of a row, by r % 8). Inside fully unrolled row loops every access is
// then a single shared-memory load or store with an immediate offset.
struct ColAddr {
    uint32_t o[8];
    __device__ __forceinline__ ColAddr(int c, int R) {
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = (uint32_t)((c >> 6) * R * 128 + (((c & 63) * 2) ^ (k << 4)));
    }
    __device__ __forceinline__ uint32_t at(int r) const { return o[r & 7] + (uint32_t)(r * 128); }
};
__device__ __forceinline__ float ld_col(const uint8_t* tile, const ColAddr& a, int r) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + a.at(r)));
}
__device__ __forceinline__ void st_col(uint8_t* tile, const ColAddr& a, int r, float x) {
    *reinterpret_cast<__nv_bfloat16*>(tile + a.at(r)) = __float2bfloat16_rn(x);
}
// Two values rounded to bf16 by one packed conversion, stored as 16-bit halves at two addresses.
__device__ __forceinline__ void st_bf16_pair(uint8_t* pa, uint8_t* pb, float a, float b) {
    const uint32_t v = pack2(a, b);
    *reinterpret_cast<uint16_t*>(pa) = (uint16_t)(v & 0xffffu);
    *reinterpret_cast<uint16_t*>(pb) = (uint16_t)(v >> 16);
}
// Rows r and r + 1 of the column a of a tile, one packed conversion.
__device__ __forceinline__ void st_col_pair(uint8_t* tile, const ColAddr& a, int r, float x0, float x1) {
    st_bf16_pair(tile + a.at(r), tile + a.at(r + 1), x0, x1);
}
// Packed fp32 pairs: one instruction for two IEEE fp32 operations (each lane rounds as its scalar form).
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 bc2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }
// The two bf16 halves of a packed pair, widened: low (first) and high (second) element.
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// In-chunk cumulative sum of g for key channel d in log2 units, in one
// canonical order that every kernel reproduces exactly whatever its thread
// layout: rows are split in four quarters of 16; for row r of quarter q,
//   G2(r) = (off_q + run_q(r)) * log2(e),  run_q(r) = sum of g over rows 16q..r
// (in row order), off_0 = 0, off_q = off_{q-1} + T_{q-1}, T_q = run_q(15).
// Rows >= c add nothing. The calling thread owns quarters q0 .. q0+NQ-1:
// load_g_quarters fetches its g values (issued early, ahead of other
// copies, since the cumsum heads each kernel's critical path) and
// quarter_cumsum_log2 forms G2; `tot` is 4 x 128 floats of shared scratch.
// quarter_cumsum_log2 contains a barrier: __syncthreads(), or with kGroup > 0
// named barrier 1 over the first kGroup threads of the block (group_sync).
template <int NQ>
__device__ __forceinline__ void load_g_quarters(const float* __restrict__ g, int64_t r0, int c, int HV, int hv, int d,
                                                int q0, float (&gv)[16 * NQ]) {
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * (q0 + qi) + i;
            gv[16 * qi + i] = r < c ? g[((r0 + r) * HV + hv) * 128 + d] : 0.f;
        }
}
template <int NQ, int kGroup = 0>
__device__ __forceinline__ void quarter_cumsum_log2(const float (&gv)[16 * NQ], int d, int q0, float* tot,
                                                    float (&G2)[16 * NQ]) {
    float run[16 * NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            acc += gv[16 * qi + i];
            run[16 * qi + i] = acc;
        }
        tot[(q0 + qi) * 128 + d] = acc;
    }
    if constexpr (kGroup > 0)
        group_sync<kGroup>();
    else
        __syncthreads();
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        float off = 0.f;
        for (int qq = 0; qq < q0 + qi; ++qq) off += tot[qq * 128 + d];
#pragma unroll
        for (int i = 0; i < 16; ++i) G2[16 * qi + i] = (off + run[16 * qi + i]) * 1.4426950408889634f;
    }
}

// The same canonical order for a thread that owns the key-channel pair d0, d0 + 1
// (d0 even) over the 16 rows of quarter qt: load_g_pair fetches the gate values into
// gv[16 * ch + i] (channel d0 + ch, row 16 qt + i; issued early), pair_cumsum_log2
// turns them into Gamma2 in place. `tot` is 4 x 128 floats of shared scratch;
// pair_cumsum_log2 contains a __syncthreads().
__device__ __forceinline__ void load_g_pair(const float* __restrict__ g, int64_t r0, int c, int HV, int hv, int d0,
                                            int qt, float (&gv)[32]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 16 * qt + i;
        const float2 x = r < c ? *reinterpret_cast<const float2*>(g + ((r0 + r) * HV + hv) * 128 + d0)
                               : make_float2(0.f, 0.f);
        gv[i] = x.x;
        gv[16 + i] = x.y;
    }
}
__device__ __forceinline__ void pair_cumsum_log2(float (&G2)[32], int d0, int qt, float* tot) {
    float run[32];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            acc += G2[16 * ch + i];
            run[16 * ch + i] = acc;
        }
        tot[qt * 128 + d0 + ch] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        float off = 0.f;
        for (int qq = 0; qq < qt; ++qq) off += tot[qq * 128 + d0 + ch];
#pragma unroll
        for (int i = 0; i < 16; ++i) G2[16 * ch + i] = (off + run[16 * ch + i]) * 1.4426950408889634f;
    }
}

}  // namespace tc
}  // namespace kda
