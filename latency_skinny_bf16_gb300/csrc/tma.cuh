// tma.cuh -- tensor-map copies (the TMA engine's tiled mode), shared by the
// kernels that stream W through them (tcgen05 GEMM, cluster split-K).
//
// Every map here views bf16 data with 64-element (128-byte) inner boxes and
// the 128-byte swizzle: inside each 1024-byte block of eight 128-byte rows,
// the 16-byte piece c of row r lands at piece c ^ (r & 7).  Destinations are
// 1024-byte aligned, so that pattern holds from the start of every box.
// Elements outside the tensor arrive as zeros and count toward the
// mbarrier's transaction bytes like any other.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace skinny {

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Box at (c0 = K element, c1 = row) of a 2-D tensor map into shared memory,
// completing on `bar`.  c0 is a multiple of 64 (128 bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar) : "memory");
}
// Box at (0, c1 = row, c2 = 64-element K box) of a 3-D view [K/64][rows][64].
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}
// Byte offset of the 16-byte piece `c` (8 elements; c / 8 selects the 64-element
// box) of row `r` in a run of boxes of `rows` rows each (rows a multiple of 8).
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Host side (tmem_gemm.cu).  bf16 [rows, cols] with row stride ld (elements),
// boxes of 64 columns x box_rows rows; false when the driver refuses the map.
bool encode_bf16_2d(CUtensorMap *map, const void *ptr, int cols, int rows, int64_t ld, int box_rows);
// A 3-D view [cols / 64][rows][64] (cols a multiple of 64), boxes of
// kb x box_rows x 64: one copy moves kb consecutive 64-column boxes.
bool encode_bf16_3d(CUtensorMap *map, const void *ptr, int cols, int rows, int64_t ld, int box_rows, int kb);

}  // namespace skinny
