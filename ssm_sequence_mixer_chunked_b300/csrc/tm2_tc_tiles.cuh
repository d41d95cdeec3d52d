// tm2_tc_tiles.cuh -- small shared-memory tile helpers of the tensor-core kernels (16-bit
// [rows][64] tiles in the 128-byte swizzled layout that TMA and the MMA descriptors use).
#pragma once
#include "tm2_sm100.cuh"

namespace tm2 {
namespace tctile {

// 16-byte piece `piece` of a [rows][64] 16-bit swizzled tile: bf16 -> fp16 into another tile
TM2_DEV void tile_bf16_to_f16(uint32_t src, uint32_t dst, int piece) {
    uint32_t x[4];
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]) : "r"(src + piece * 16));
    st_shared_v4(dst + piece * 16, bf16x2_to_f16x2(x[0]), bf16x2_to_f16x2(x[1]), bf16x2_to_f16x2(x[2]),
                 bf16x2_to_f16x2(x[3]));
}
// element (row, col) of a [rows][64] 16-bit swizzled tile
TM2_DEV uint32_t swz_elem(int row, int col) { return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2; }
// the normaliser matrix in two steps, so that its global loads can be issued before a wait:
// z_tiles_load reads this thread's 16 values of z[4096] (256 threads), z_tiles_store writes
// zm[m][n] = scale * z[m*64 + n] as hi + lo fp16 K-major tiles
TM2_DEV void z_tiles_load(const float* __restrict__ z, int t256, float4 (&r)[4]) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int pc = t256 + 256 * it, m = pc >> 3, k8 = pc & 7;
        r[2 * it] = *reinterpret_cast<const float4*>(z + m * 64 + k8 * 8);
        r[2 * it + 1] = *reinterpret_cast<const float4*>(z + m * 64 + k8 * 8 + 4);
    }
}
TM2_DEV void z_tiles_store(uint8_t* hi, uint8_t* lo, const float4 (&r)[4], float scale, int t256) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int pc = t256 + 256 * it, m = pc >> 3, k8 = pc & 7;
        const float4 a0 = r[2 * it], a1 = r[2 * it + 1];
        const float v[8] = {a0.x * scale, a0.y * scale, a0.z * scale, a0.w * scale,
                            a1.x * scale, a1.y * scale, a1.z * scale, a1.w * scale};
        uint32_t h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            h[u] = pack_f16x2(v[2 * u], v[2 * u + 1]);
            const __half2 h2 = *reinterpret_cast<const __half2*>(&h[u]);
            l[u] = pack_f16x2(v[2 * u] - __low2float(h2), v[2 * u + 1] - __high2float(h2));
        }
        const uint32_t off = m * 128 + ((k8 ^ (m & 7)) << 4);
        st_shared_v4(smem_u32(hi) + off, h[0], h[1], h[2], h[3]);
        st_shared_v4(smem_u32(lo) + off, l[0], l[1], l[2], l[3]);
    }
}

}  // namespace tctile
}  // namespace tm2
