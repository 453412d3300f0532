// One lane's share of an OFT block rotation (bf16), shared by the rotation
// kernels of libscute.so.
//
// OFT multiplies the layer input by a block-diagonal rotation (article "Scute:
// Exact Batched Serving for PEFT Adapters Beyond LoRA", paper-daily.com,
// sections "What problem is it solving?" and "Where is the cheapest place to
// compute the remaining slots?").  A warp moves one row of 256 columns, lane l
// holding columns [8l, 8l + 8) as one 16-byte word; the four lanes 4b..4b+3
// hold one 32-column block.  rotate_lane returns lane l's 8 outputs of
// x'[j] = sum_i x[i] R[i][j] over its block, reading row j of the
// block-transposed copy Rt (Rt[b][j][i] = R[b][i][j], 32 contiguous bf16 per
// j) through L1.  Every lane of the warp must call it (the block's inputs
// arrive by shuffle); `compute` is false for lanes past the row's end, whose
// result is not used.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace scute {

__device__ __forceinline__ uint4 rotate_lane(uint4 xv, const __nv_bfloat16 *Rt, int col, bool compute) {
    const int lane = threadIdx.x & 31;
    uint32_t xin[16];
    const uint32_t *mine = reinterpret_cast<const uint32_t *>(&xv);
    const int base = lane & ~3;
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
        for (int w = 0; w < 4; ++w) xin[s4 * 4 + w] = __shfl_sync(0xffffffffu, mine[w], base + s4);
    uint4 o = xv;
    if (!compute) return o;
    float xf[32];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xin[p]));
        xf[2 * p] = f.x;
        xf[2 * p + 1] = f.y;
    }
    const int b = col / 32, j0 = col % 32;
    const uint4 *Rrow = reinterpret_cast<const uint4 *>(Rt + ((size_t)b * 32 + j0) * 32);
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = __ldg(Rrow + e * 4 + q);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 f = __bfloat1622float2(h[t]);
                acc = fmaf(xf[q * 8 + 2 * t], f.x, acc);
                acc = fmaf(xf[q * 8 + 2 * t + 1], f.y, acc);
            }
        }
        y[e] = acc;
    }
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
    for (int t = 0; t < 4; ++t) h[t] = __floats2bfloat162_rn(y[2 * t], y[2 * t + 1]);
    return o;
}

}  // namespace scute
