// Host-side encoding of TMA tensor maps (driver entry point looked up at run
// time, so the library does not link libcuda).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace kda {

// 2-D bf16 tensor map over a row-major matrix of `outer` rows of `inner`
// elements with `row_bytes` between rows, box {box_inner, box_outer}, 128-byte
// swizzle. Returns false if encoding fails.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                       uint32_t box_inner, uint32_t box_outer);

// 3-D bf16 tensor map: dims {d0 (contiguous), d1, d2}, byte strides s1, s2,
// box {b0, b1, b2}, 128-byte swizzle.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                       uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);

// 3-D fp32 tensor map, same dims / strides / box convention, no swizzle
// (the box lands in shared memory as a dense row-major block).
bool make_tmap_f32_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                      uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);

}  // namespace kda
