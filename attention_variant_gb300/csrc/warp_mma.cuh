// warp_mma.cuh -- warp-level bf16 tensor-core helpers for kernels whose
// contractions are a few rows per warp (the decode kernel): ldmatrix fragment
// loads from 128-byte-swizzled shared-memory tiles and the m16n8k16 MMA with
// fp32 accumulation.
//
// Fragment layout of mma.m16n8k16 (g = lane / 4, t = lane % 4):
//   A (16 x 16): a0 (row g, cols 2t, 2t+1), a1 (row g+8, same cols),
//                a2 (row g, cols 2t+8, 2t+9), a3 (row g+8, cols 2t+8, 2t+9)
//   B (16 x 8):  b0 (rows 2t, 2t+1, col g), b1 (rows 2t+8, 2t+9, col g)
//   C (16 x 8):  c0, c1 (row g, cols 2t, 2t+1), c2, c3 (row g+8, same cols)
// A tile of 64 bf16 per row is 128 bytes; the TMA's 128-byte swizzle puts the
// 16-byte unit u of row r at position u ^ (r mod 8).
#pragma once

#include "ptx.cuh"

namespace fl {
namespace wm {

// Byte offset of 16-byte unit u of row r inside a swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int u)
{
    return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// d += a b for one 16 x 8 tile, K = 16 (bf16 in, fp32 accumulate)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// B fragments of an operand whose n index runs along the tile's rows (the
// tile row holds the k values contiguously, as K[key][dim] for S = Q K^T):
// rows n0 .. n0+15, k-step kk (dims 16 kk .. 16 kk + 15).  b[0], b[1] for
// n-tile n0 .. n0+7 and b[2], b[3] for n0+8 .. n0+15.
__device__ __forceinline__ void ldsm_b_rows(uint32_t tile, int n0, int kk, uint32_t (&b)[4])
{
    const int lane = threadIdx.x & 31, mi = lane >> 3, ri = lane & 7;
    ldsm_x4(tile + swz(n0 + ri + ((mi >> 1) << 3), 2 * kk + (mi & 1)), b[0], b[1], b[2], b[3]);
}

// B fragments of an operand whose k index runs along the tile's rows (as
// V[key][dim] for O = P V): rows (k) k0 .. k0+15, columns (n) 16 u2 ..
// 16 u2 + 15 as two n-tiles: b[0], b[1] for columns 16 u2 .. +7, b[2], b[3]
// for 16 u2 + 8 .. +15.
__device__ __forceinline__ void ldsm_b_cols(uint32_t tile, int k0, int u2, uint32_t (&b)[4])
{
    const int lane = threadIdx.x & 31, mi = lane >> 3, ri = lane & 7;
    ldsm_x4_t(tile + swz(k0 + ri + ((mi & 1) << 3), 2 * u2 + (mi >> 1)), b[0], b[1], b[2], b[3]);
}

} // namespace wm
} // namespace fl
