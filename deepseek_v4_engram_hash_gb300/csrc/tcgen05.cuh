// tcgen05.cuh -- pieces the two tensor-core GEMMs share (gemm_tc.cu: one CTA
// a 128 x 256 tile; gemm_tc2.cu: a CTA pair a 256 x 256 tile): the shared-
// memory and instruction descriptors, the tcgen05 fences, the 32-column
// tensor-memory load, the grouped tile order and the TMA tensor maps.
#pragma once

#include "common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace engram {
namespace tcg {

constexpr int BK = 64;          // k step: one 128-byte swizzle row of bf16

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle:
// rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), the
// leading byte offset unused for this layout (encoded 1), version 1 in bits
// 46..47, layout type 2 (SWIZZLE_128B) in bits 61..63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor, kind::f16: f32 accumulator (bits 4..5 = 1), bf16 A
// and B (bits 7..9 = 1, 10..12 = 1), both K-major, N >> 3 in bits 17..22,
// M >> 4 in bits 24..28 (M of the whole CTA group).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive f32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Tile order within a layer: groups of group_m row tiles; inside a group,
// row tiles fastest, then column tiles.  The CTAs running at one time then
// share a few x row blocks and a few wkv column blocks, both L2-resident, even
// when x itself is larger than L2.
__device__ __forceinline__ void tile_coords(int r, int m_tiles, int n_tiles, int group_m, int &mt, int &nt) {
    const int per_group = group_m * n_tiles;
    const int g = r / per_group, idx = r % per_group;
    const int gsz = min(group_m, m_tiles - g * group_m);
    mt = g * group_m + idx % gsz;
    nt = idx / gsz;
}

// Group size in 128-row tiles: all row tiles in one group up to 32 (x of one
// group <= 50 MB at K = 6144, so wkv streams from DRAM once); beyond, equal
// groups of about 24.  Measured on one V4.1 layer with the one-CTA kernel:
// 4096 tokens 1.73 PF/s with one group of 32 against 1.69 with 16; 12 288
// tokens 1.83 PF/s with four groups of 24 against 1.78 with three of 32 and
// 1.73 with six of 16; the pair kernel's sweep agreed within 0.5 %.
inline int group_rows128(int m_tiles128) {
    if (m_tiles128 <= 32) return m_tiles128 < 1 ? 1 : m_tiles128;
    const int groups = (m_tiles128 + 23) / 24;
    return (m_tiles128 + groups - 1) / groups;
}

// 2D bf16 tensor map over [outer, inner] (inner contiguous), box {BK, box_outer},
// 128-byte swizzle; false if the driver entry point is missing or refuses.
bool make_map(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_outer);
bool have_tensor_maps();

}  // namespace tcg
}  // namespace engram
