// Separate-pass placements of two live slots, for validating the byte model.
//
// The article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA"
// (paper-daily.com, section "Where is the cheapest place to compute the
// remaining slots?") checks its zero-parameter time model on OFT's input
// rotation run as its own pass before the shared GEMM and on ways of applying
// DoRA's s outside the expand.  The decode step normally does both inside its
// one launch; these kernels move them out again, so that the model's
// prediction for the extra launch (its bytes over the bandwidth plus one
// launch cost) can be set against a measurement.  Both placements keep the
// layer's result exact:
//   * oft_pass: x_rot[t] = x[t] R_a(t) for rotated tokens, x[t] otherwise, in
//     token order, for every call of a batch in one launch; the step then
//     reads x_rot and rotates nothing;
//   * s_pass: out[t] *= s_a(t) for the tokens whose adapter is a DoRA or
//     (IA)^3 one with a live s, for every call in one launch; the step then
//     leaves s out for those tokens and, for DoRA, expands with B' whose s is
//     not folded in (y = s * (x W + v B)).
#include "internal.h"
#include "oft_lane.cuh"
#include "ptx.cuh"

namespace scute {

namespace {

__device__ __forceinline__ int token_adapter(const PassArgs &p, int t) {
    const int id = p.ids[t];
    return (id >= 0 && id < p.A && p.method_tab[id] >= 0) ? id : -1;
}

// grid (256-column chunks, 32-token groups, calls); one warp per token row.
__global__ void __launch_bounds__(256) oft_pass_kernel(const __grid_constant__ PassArgs p) {
    const PassCall &k = p.call[blockIdx.z];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = blockIdx.x * 256 + lane * 8;
    if (blockIdx.x * 256 >= k.d_in) return;   // uniform: this call is narrower
    const bool colok = col < k.d_in;
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(k.x);
    __nv_bfloat16 *xo = reinterpret_cast<__nv_bfloat16 *>(k.xo);
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        const int t = blockIdx.y * 32 + warp * 4 + r;
        if (t >= p.n) break;   // uniform across the warp
        const int a = token_adapter(p, t);
        const __nv_bfloat16 *Rt = a >= 0 ? reinterpret_cast<const __nv_bfloat16 *>(k.slots[a].Rt) : nullptr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (colok) v = *reinterpret_cast<const uint4 *>(x + (size_t)t * k.d_in + col);
        if (Rt != nullptr) v = rotate_lane(v, Rt, col, colok);
        if (colok) *reinterpret_cast<uint4 *>(xo + (size_t)t * k.d_in + col) = v;
    }
}

// grid (2048-column chunks, tokens, calls); 8 columns per thread.
__global__ void __launch_bounds__(256) s_pass_kernel(const __grid_constant__ PassArgs p) {
    const PassCall &k = p.call[blockIdx.z];
    const int t = blockIdx.y;
    const int j0 = (blockIdx.x * 256 + threadIdx.x) * 8;
    if (j0 >= k.d_out) return;
    const int a = token_adapter(p, t);
    if (a < 0) return;
    const int m = p.method_tab[a];
    const float *s = k.slots[a].s;
    if ((m != RANK_DORA && m != RANK_IA3) || s == nullptr) return;
    const float4 s0 = __ldg(reinterpret_cast<const float4 *>(s + j0));
    const float4 s1 = __ldg(reinterpret_cast<const float4 *>(s + j0 + 4));
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    if (p.out_f32) {
        float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(k.out) + (size_t)t * k.d_out + j0);
        float4 u = o[0], w = o[1];
        u.x *= sv[0]; u.y *= sv[1]; u.z *= sv[2]; u.w *= sv[3];
        w.x *= sv[4]; w.y *= sv[5]; w.z *= sv[6]; w.w *= sv[7];
        o[0] = u;
        o[1] = w;
    } else {
        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(k.out) + (size_t)t * k.d_out + j0);
        uint4 u = *o;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            h[e] = __floats2bfloat162_rn(f.x * sv[2 * e], f.y * sv[2 * e + 1]);
        }
        *o = u;
    }
}

}  // namespace

cudaError_t launch_oft_pass(const PassArgs &p, int max_d_in, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((max_d_in + 255) / 256), (unsigned)((p.n + 31) / 32), (unsigned)p.n_calls);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, oft_pass_kernel, p);
}

cudaError_t launch_s_pass(const PassArgs &p, int max_d_out, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((max_d_out + 2047) / 2048), (unsigned)p.n, (unsigned)p.n_calls);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, s_pass_kernel, p);
}

}  // namespace scute
