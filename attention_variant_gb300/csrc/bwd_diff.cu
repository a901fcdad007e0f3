// bwd_diff.cu -- the combining step of the differential-attention backward.
//
// The backward of O = softmax(s Q1 K1^T) V - lambda softmax(s Q2 K2^T) V is
// assembled on the host from the standard kind's kernels: stream t's
// gradients are those of one softmax attention with output gradient
// c_t dO (c = 1, -lambda), and every gradient of softmax(Q K^T) V is linear in
// the output gradient, so the standard backward runs with dO itself and the
// coefficient is applied here.  A value head dimension of 128 runs as two
// 64-column halves of V, O and dO: dS = P (dP - D) is a sum over the halves
// (dP and D are sums over value columns), so dQ and dK of the whole are the
// halves' sums, and each half of dV is its own.  This kernel forms
//     out[row, 0:64] = sum_p coef[p] in_p[row, 0:64]
// in fp32 from up to two bf16 partials and rounds once to bf16.
#include <cuda_bf16.h>
#include <cstdint>

#include "launch.h"

namespace fl {
namespace {

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b); // .x = a (low half)
    return *reinterpret_cast<const uint32_t *>(&h);
}

// One thread per 8 columns (16 bytes) of one row; rows are (b, position, head)
// of the output view.
__global__ void __launch_bounds__(256) diff_bwd_combine_kernel(const DiffCombine c)
{
    const int64_t n = c.rows * 8;
    for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < n;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = idx >> 3;
        const int part = static_cast<int>(idx & 7);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            if (!c.in[p])
                continue;
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(c.in[p] + row * 64) + part);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] = fmaf(c.coef[p], lo_bf16(ws[e]), acc[2 * e]);
                acc[2 * e + 1] = fmaf(c.coef[p], hi_bf16(ws[e]), acc[2 * e + 1]);
            }
        }
        const int64_t h = row % c.heads, bs = row / c.heads;
        const int64_t s = bs % c.S, b = bs / c.S;
        uint4 *dst = reinterpret_cast<uint4 *>(c.out + b * c.o_sb + s * c.o_ss + h * c.o_sh) + part;
        *dst = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]), pack2(acc[4], acc[5]),
                          pack2(acc[6], acc[7]));
    }
}

} // namespace

cudaError_t launch_diff_bwd_combine(const DiffCombine &c, int sm_count, cudaStream_t stream)
{
    if (c.rows <= 0)
        return cudaSuccess;
    const int64_t threads = c.rows * 8;
    const int64_t want = (threads + 255) / 256;
    const int64_t cap = int64_t(sm_count) * 16; // grid-stride beyond that
    const int grid = static_cast<int>(want < cap ? want : cap);
    diff_bwd_combine_kernel<<<grid, 256, 0, stream>>>(c);
    return cudaGetLastError();
}

} // namespace fl
