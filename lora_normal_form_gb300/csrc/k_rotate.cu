// OFT input rotation prologue: x'[i] = x[perm[i]] R_a, written in sorted row
// order into the GEMM's token operand.
//
// OFT multiplies each layer input by its tenant's block-diagonal rotation
// before the shared GEMM, in its own pass, so that the rotated rows still share
// the base weight (article "Scute: Exact Batched Serving for PEFT Adapters
// Beyond LoRA", paper-daily.com, section "Where is the cheapest place to
// compute the remaining slots?").  Rows of every other adapter are copied
// unchanged, so the GEMM reads one contiguous token operand in sorted order.
//
// fp32 contexts (gather_rotate_kernel): x = 256-column chunk (8 blocks of 32),
// y = run of sorted rows; a CTA stages its adapter's 8 blocks of R in shared
// memory once per run of one adapter, and writes each value as three tf32
// parts [hi | hi | lo] for the split-precision GEMM (hi = tf32(v), lo = v - hi).
// bf16 contexts: gather_rotate_bf16_kernel below.
#include "internal.h"
#include "oft_lane.cuh"
#include "ptx.cuh"

namespace scute {

namespace {

template <typename T>
__device__ __forceinline__ float ldf(const T *p) {
    if constexpr (sizeof(T) == 2) return __bfloat162float(*p);
    else return *p;
}

template <typename T>
__global__ void __launch_bounds__(256) gather_rotate_kernel(const T *__restrict__ x, int d_in, int n,
                                                            const int *__restrict__ perm,
                                                            const int *__restrict__ aid_s,
                                                            const Slot *__restrict__ slots, T *xs,
                                                            int kdim, int rows_per_cta) {
    __shared__ float Rs[8][OFT_BLK][OFT_BLK];
    __shared__ float xrow[256];
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int tid = threadIdx.x;
    const int col0 = blockIdx.x * 256;
    const int ncols = min(256, d_in - col0);
    const int blk = tid >> 5, cc = tid & 31;
    const int r0 = blockIdx.y * rows_per_cta;
    const int r1 = min(n, r0 + rows_per_cta);
    int cur = -2;
    for (int i = r0; i < r1; ++i) {
        const int a = aid_s[i];
        const T *R = a >= 0 ? reinterpret_cast<const T *>(slots[a].R) : nullptr;
        const T *src = x + (size_t)perm[i] * d_in + col0;
        float val = 0.f;
        if (R == nullptr) {
            if (tid < ncols) val = ldf(src + tid);
        } else {
            if (a != cur) {
                __syncthreads();
                const T *Rb = R + (size_t)(col0 / OFT_BLK) * OFT_BLK * OFT_BLK;
                const int nel = (ncols / OFT_BLK) * OFT_BLK * OFT_BLK;
                for (int e = tid; e < nel; e += 256) (&Rs[0][0][0])[e] = ldf(Rb + e);
                cur = a;
            }
            xrow[tid] = tid < ncols ? ldf(src + tid) : 0.f;
            __syncthreads();
            if (tid < ncols) {
                float acc = 0.f;
#pragma unroll 8
                for (int m = 0; m < OFT_BLK; ++m) acc = fmaf(xrow[blk * OFT_BLK + m], Rs[blk][m][cc], acc);
                val = acc;
            }
            __syncthreads();
        }
        if (tid < ncols) {
            T *dst = xs + (size_t)i * kdim + col0 + tid;
            if constexpr (sizeof(T) == 2) {
                *dst = __float2bfloat16_rn(val);
            } else {
                const float hi = ptx::to_tf32(val);
                dst[0] = hi;
                dst[d_in] = hi;
                dst[2 * d_in] = val - hi;
            }
        }
    }
}

// bf16 contexts: one warp per sorted row, which it moves whole, eight 256-column
// chunks at a time (lane l holds columns [8l, 8l + 8) of each chunk as one
// 16-byte word, so every load of the eight is in flight before the first
// store, and a row's bytes are read and written in one pass); a rotated row's
// lanes compute their block outputs with rotate_lane (oft_lane.cuh), reading
// R through L1.  No shared memory and no barrier: every row is independent.
// x is read once (cache-streaming), so that x', which the shrinks and the GEMM
// read next, keeps its place in L2.
__global__ void __launch_bounds__(256) gather_rotate_bf16_kernel(const __nv_bfloat16 *__restrict__ x, int d_in,
                                                                 int n, const int *__restrict__ perm,
                                                                 const int *__restrict__ aid_s,
                                                                 const Slot *__restrict__ slots,
                                                                 __nv_bfloat16 *xs, int kdim) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + warp;
    if (i >= n) return;   // whole warps; no barrier below
    const int a = aid_s[i];
    const __nv_bfloat16 *Rt = a >= 0 ? reinterpret_cast<const __nv_bfloat16 *>(slots[a].Rt) : nullptr;
    const __nv_bfloat16 *src = x + (size_t)perm[i] * d_in;
    __nv_bfloat16 *dst = xs + (size_t)i * kdim;
    const int nch = (d_in + 255) / 256;
    for (int c0 = 0; c0 < nch; c0 += 8) {
        uint4 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int col = (c0 + u) * 256 + lane * 8;
            xv[u] = make_uint4(0u, 0u, 0u, 0u);
            if (c0 + u < nch && col < d_in) xv[u] = __ldcs(reinterpret_cast<const uint4 *>(src + col));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (c0 + u >= nch) break;   // uniform across the warp
            const int col = (c0 + u) * 256 + lane * 8;
            const bool colok = col < d_in;
            uint4 o = xv[u];
            if (Rt != nullptr) o = rotate_lane(xv[u], Rt, col, colok);
            if (colok) *reinterpret_cast<uint4 *>(dst + col) = o;
        }
    }
}

}  // namespace

cudaError_t launch_gather_rotate(bool f32, const void *x, int d_in, int n, const int *perm,
                                 const int *aid_s, const Slot *slots, void *xs, int kdim,
                                 cudaStream_t st, bool pdl) {
    const int rows = n <= 256 ? 4 : 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((d_in + 255) / 256), (unsigned)((n + rows - 1) / rows), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (f32)
        return cudaLaunchKernelEx(&cfg, gather_rotate_kernel<float>, (const float *)x, d_in, n, perm,
                                  aid_s, slots, (float *)xs, kdim, rows);
    cfg.gridDim = dim3((unsigned)((n + 7) / 8), 1, 1);
    return cudaLaunchKernelEx(&cfg, gather_rotate_bf16_kernel, (const __nv_bfloat16 *)x, d_in, n, perm, aid_s,
                              slots, (__nv_bfloat16 *)xs, kdim);
}

}  // namespace scute
