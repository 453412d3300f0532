// Segmented shrink / expand of the owned low-rank term (LoRA, DoRA, raw
// normal form), after the fold rule has put c and d into A and e into B:
//     v_t   = x_t A'_a                      (shrink, fp32, K split in KS parts)
//     out_t += v_t B'_a                     (expand, read-modify-write)
// (article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA",
// paper-daily.com, section "The big picture": the shrink multiplies the input
// by A down to rank dimensions, the expand multiplies by B and adds the result
// to h; section "Which slots can be merged at load?" for the folds).
//
// Both kernels take one CTA per (segment, chunk).  Segments come from the
// indexing kernel, so every CTA serves exactly one adapter and streams that
// adapter's A' (stored [rank][d_in]) or B' ([rank][d_out]) with 16-byte loads,
// while the segment's rows reuse it from L1.  The shrink reads the original x
// through the sort permutation (the low-rank term acts on x, not on x R).
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&v)[8]) {
    if constexpr (sizeof(T) == 2) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            v[2 * e] = f.x;
            v[2 * e + 1] = f.y;
        }
    } else {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        const float4 b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T, int RM>
__global__ void __launch_bounds__(256) lr_shrink_kernel(const T *__restrict__ x, int d_in,
                                                        const int *__restrict__ perm,
                                                        const int *__restrict__ seg_start,
                                                        const int *__restrict__ seg_aid,
                                                        const IndexMeta *__restrict__ meta,
                                                        const Slot *__restrict__ slots, float *v_part,
                                                        int max_tokens, int kchunk) {
    ptx::grid_dep_wait();
    const int seg = blockIdx.x;
    if (seg >= meta->n_seg) return;
    const int a = seg_aid[seg];
    if (a < 0) return;
    const T *A = reinterpret_cast<const T *>(slots[a].A);
    const int r = slots[a].rank;
    if (A == nullptr || r <= 0) return;
    const int k0 = blockIdx.y * kchunk;
    if (k0 >= d_in) return;
    const int k1 = min(d_in, k0 + kchunk);
    const int rs = seg_start[seg], re = seg_start[seg + 1];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *vp = v_part + (size_t)blockIdx.y * max_tokens * MAX_RANK;
    for (int i = rs + w; i < re; i += 8) {
        float acc[RM];
#pragma unroll
        for (int q = 0; q < RM; ++q) acc[q] = 0.f;
        const T *src = x + (size_t)perm[i] * d_in;
        for (int k = k0 + lane * 8; k < k1; k += 256) {
            float xv[8];
            load8(src + k, xv);
#pragma unroll
            for (int q = 0; q < RM; ++q) {
                if (q < r) {
                    float av[8];
                    load8(A + (size_t)q * d_in + k, av);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[q] = fmaf(xv[e], av[e], acc[q]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < RM; ++q) {
            if (q < r) {
                const float s = warp_sum(acc[q]);
                if (lane == 0) vp[(size_t)i * MAX_RANK + q] = s;
            }
        }
    }
}

template <typename T, int RM>
__global__ void __launch_bounds__(256) lr_expand_kernel(const float *__restrict__ v_part, int ks,
                                                        int max_tokens, int d_out,
                                                        const int *__restrict__ perm,
                                                        const int *__restrict__ seg_start,
                                                        const int *__restrict__ seg_aid,
                                                        const IndexMeta *__restrict__ meta,
                                                        const Slot *__restrict__ slots, void *out,
                                                        int out_f32) {
    __shared__ float vs[8][RM];
    ptx::grid_dep_wait();
    const int seg = blockIdx.x;
    if (seg >= meta->n_seg) return;
    const int a = seg_aid[seg];
    if (a < 0) return;
    const T *B = reinterpret_cast<const T *>(slots[a].B);
    const int r = slots[a].rank;
    if (B == nullptr || r <= 0) return;
    const int rs = seg_start[seg], re = seg_start[seg + 1];
    const int j0 = (blockIdx.y * 256 + threadIdx.x) * 8;
    for (int rb = rs; rb < re; rb += 8) {
        const int nr = min(8, re - rb);
        for (int e = threadIdx.x; e < 8 * RM; e += 256) {
            const int rr = e / RM, q = e % RM;
            float v = 0.f;
            if (rr < nr && q < r)
                for (int s = 0; s < ks; ++s) v += v_part[((size_t)s * max_tokens + rb + rr) * MAX_RANK + q];
            vs[rr][q] = v;
        }
        __syncthreads();
        if (j0 < d_out) {
            float acc[8][8];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[rr][e] = 0.f;
#pragma unroll 4
            for (int q = 0; q < r; ++q) {
                float bv[8];
                load8(B + (size_t)q * d_out + j0, bv);
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const float vq = vs[rr][q];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[rr][e] = fmaf(vq, bv[e], acc[rr][e]);
                }
            }
            for (int rr = 0; rr < nr; ++rr) {
                const size_t o = (size_t)perm[rb + rr] * d_out + j0;
                if (out_f32) {
                    float4 *p = reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + o);
                    float4 u = p[0], w = p[1];
                    u.x += acc[rr][0]; u.y += acc[rr][1]; u.z += acc[rr][2]; u.w += acc[rr][3];
                    w.x += acc[rr][4]; w.y += acc[rr][5]; w.z += acc[rr][6]; w.w += acc[rr][7];
                    p[0] = u;
                    p[1] = w;
                } else {
                    uint4 *p = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out) + o);
                    uint4 u = *p;
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h[e]);
                        h[e] = __floats2bfloat162_rn(f.x + acc[rr][2 * e], f.y + acc[rr][2 * e + 1]);
                    }
                    *p = u;
                }
            }
        }
        __syncthreads();
    }
}

template <typename T, int RM>
cudaError_t launch_lr(const T *x, int d_in, int d_out, int seg_bound, const int *perm,
                      const int *seg_start, const int *seg_aid, const IndexMeta *meta,
                      const Slot *slots, float *v_part, int max_tokens, void *out, int out_f32,
                      cudaStream_t st, bool pdl) {
    int kchunk = 0;
    const int ks = lowrank_ks(d_in, &kchunk);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)seg_bound, (unsigned)ks, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lr_shrink_kernel<T, RM>, x, d_in, perm, seg_start, seg_aid,
                                       meta, slots, v_part, max_tokens, kchunk);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)seg_bound, (unsigned)((d_out + 2047) / 2048), 1);
    return cudaLaunchKernelEx(&cfg, lr_expand_kernel<T, RM>, (const float *)v_part, ks, max_tokens, d_out,
                              perm, seg_start, seg_aid, meta, slots, out, out_f32);
}

}  // namespace

cudaError_t launch_lowrank(bool f32, const void *x, int d_in, int d_out, int n, int seg_bound,
                           const int *perm, const int *seg_start, const int *seg_aid,
                           const IndexMeta *meta, const Slot *slots, float *v_part, int max_tokens,
                           void *out, int out_f32, cudaStream_t st, bool pdl, int max_rank) {
    (void)n;
    if (f32) {
        if (max_rank <= 16)
            return launch_lr<float, 16>((const float *)x, d_in, d_out, seg_bound, perm, seg_start, seg_aid,
                                        meta, slots, v_part, max_tokens, out, out_f32, st, pdl);
        return launch_lr<float, 64>((const float *)x, d_in, d_out, seg_bound, perm, seg_start, seg_aid,
                                    meta, slots, v_part, max_tokens, out, out_f32, st, pdl);
    }
    if (max_rank <= 16)
        return launch_lr<__nv_bfloat16, 16>((const __nv_bfloat16 *)x, d_in, d_out, seg_bound, perm,
                                            seg_start, seg_aid, meta, slots, v_part, max_tokens, out,
                                            out_f32, st, pdl);
    return launch_lr<__nv_bfloat16, 64>((const __nv_bfloat16 *)x, d_in, d_out, seg_bound, perm, seg_start,
                                        seg_aid, meta, slots, v_part, max_tokens, out, out_f32, st, pdl);
}

}  // namespace scute
