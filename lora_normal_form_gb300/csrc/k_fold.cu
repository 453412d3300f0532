// Registration-time kernels: K-major copies of the shared weights and the fold
// rule applied to an adapter's own tensors (article "Scute: Exact Batched
// Serving for PEFT Adapters Beyond LoRA", paper-daily.com, section "Which slots
// can be merged at load?": (xA) * d = x (A diag(d)); DoRA's e folds into its B
// and c into its A; section "How does Scute plug into vLLM?": DoRA's s is the
// learned length over the norm of each column of W + cAB, computed at load).
// None of these runs inside scute_linear.
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

template <typename T>
__device__ __forceinline__ float ldf(const T *p) {
    if constexpr (sizeof(T) == 2) return __bfloat162float(*p);
    else return *p;
}
template <typename T>
__device__ __forceinline__ void stf(T *p, float v) {
    if constexpr (sizeof(T) == 2) *p = __float2bfloat16_rn(v);
    else *p = v;
}

// src [rows][cols] -> dst [cols][kdim].  pattern 0: dst[c][r] = src[r][c].
// pattern 1 (fp32 weight side of the split-precision GEMM): the row holds
// [hi | lo | hi] of src[:, c], hi = tf32(v), lo = v - hi, so that against
// activations stored [hi | hi | lo] one K-long dot product sums
// hi*hi + lo*hi + hi*lo.
template <typename T>
__global__ void transpose_kernel(const T *__restrict__ src, int rows, int cols, T *dst, int kdim,
                                 int pattern) {
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
        const int r = r0 + k, c = c0 + threadIdx.x;
        tile[k][threadIdx.x] = (r < rows && c < cols) ? ldf(src + (size_t)r * cols + c) : 0.f;
    }
    __syncthreads();
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
        const int c = c0 + k, r = r0 + threadIdx.x;
        if (c < cols && r < rows) {
            const float v = tile[threadIdx.x][k];
            T *d = dst + (size_t)c * kdim;
            if (pattern == 0) {
                stf(d + r, v);
            } else {
                const float hi = ptx::to_tf32(v);
                stf(d + r, hi);
                stf(d + rows + r, v - hi);
                stf(d + 2 * rows + r, hi);
            }
        }
    }
}

// A [d_in][rank] -> A' [rank][d_in] = c * A[k][q] * d[q]
template <typename T>
__global__ void fold_A_kernel(const T *__restrict__ A, int d_in, int rank, float c,
                              const float *__restrict__ d, T *Aout) {
    const size_t total = (size_t)d_in * rank;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x) {
        const int q = (int)(e / d_in), k = (int)(e % d_in);
        float v = ldf(A + (size_t)k * rank + q) * c;
        if (d) v *= d[q];
        stf(Aout + e, v);
    }
}

// B [rank][d_out] -> B' = B diag(e) diag(s)
template <typename T>
__global__ void fold_B_kernel(const T *__restrict__ B, int rank, int d_out, const float *__restrict__ e,
                              const float *__restrict__ s, T *Bout) {
    const size_t total = (size_t)d_out * rank;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int j = (int)(i % d_out);
        float v = ldf(B + i);
        if (e) v *= e[j];
        if (s) v *= s[j];
        stf(Bout + i, v);
    }
}

// DoRA: s[j] = m[j] / || W[:, j] + c sum_q A[:, q] B[q, j] ||_2, one warp per
// column, squares accumulated in float64.  W is read from the K-major copy
// (W[k][j] = Wt[j][k]; an fp32 context stores [hi | lo | hi] and hi + lo is
// the original value exactly).
template <typename T>
__global__ void dora_scale_kernel(const T *__restrict__ Wt, int kdim, int d_in, int d_out,
                                  const T *__restrict__ A, const T *__restrict__ B, int rank, float c,
                                  const float *__restrict__ m, float *s_out, int *err) {
    const int warps = blockDim.x >> 5;
    const int j = blockIdx.x * warps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (j >= d_out) return;
    double bcol[MAX_RANK];
    for (int q = 0; q < rank; ++q) bcol[q] = (double)ldf(B + (size_t)q * d_out + j);
    double acc = 0.0;
    const T *w = Wt + (size_t)j * kdim;
    for (int k = lane; k < d_in; k += 32) {
        double v = (double)ldf(w + k);
        if (sizeof(T) == 4) v += (double)ldf(w + d_in + k);
        double ab = 0.0;
        for (int q = 0; q < rank; ++q) ab += (double)ldf(A + (size_t)k * rank + q) * bcol[q];
        v += (double)c * ab;
        acc += v * v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        if (!(acc > 0.0)) {
            atomicOr(err, 1);
            s_out[j] = 0.f;
        } else {
            s_out[j] = (float)((double)m[j] / sqrt(acc));
        }
    }
}

__global__ void scale_vec_kernel(const float *v, float c, float *out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = v[i] * c;
}

__global__ void transpose_blocks_kernel(const __nv_bfloat16 *src, __nv_bfloat16 *dst) {
    __shared__ __nv_bfloat16 t[32][33];
    const size_t b = blockIdx.x;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) t[i][threadIdx.x] = src[b * 1024 + i * 32 + threadIdx.x];
    __syncthreads();
    for (int j = threadIdx.y; j < 32; j += blockDim.y) dst[b * 1024 + j * 32 + threadIdx.x] = t[threadIdx.x][j];
}

int blocks_for(size_t total, int threads) {
    size_t b = (total + threads - 1) / threads;
    return (int)(b > 4096 ? 4096 : (b < 1 ? 1 : b));
}

}  // namespace

cudaError_t launch_transpose_w(bool f32, const void *W, int rows, int cols, void *Wt, int kdim,
                               int pattern, cudaStream_t st) {
    (void)cudaGetLastError();
    dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
    if (f32)
        transpose_kernel<float><<<grid, block, 0, st>>>((const float *)W, rows, cols, (float *)Wt, kdim,
                                                        pattern);
    else
        transpose_kernel<__nv_bfloat16><<<grid, block, 0, st>>>((const __nv_bfloat16 *)W, rows, cols,
                                                                (__nv_bfloat16 *)Wt, kdim, 0);
    return cudaGetLastError();
}

cudaError_t launch_fold_A(bool f32, const void *A, int d_in, int rank, float c, const float *d,
                          void *Aout, cudaStream_t st) {
    (void)cudaGetLastError();
    const int b = blocks_for((size_t)d_in * rank, 256);
    if (f32)
        fold_A_kernel<float><<<b, 256, 0, st>>>((const float *)A, d_in, rank, c, d, (float *)Aout);
    else
        fold_A_kernel<__nv_bfloat16><<<b, 256, 0, st>>>((const __nv_bfloat16 *)A, d_in, rank, c, d,
                                                        (__nv_bfloat16 *)Aout);
    return cudaGetLastError();
}

cudaError_t launch_fold_B(bool f32, const void *B, int rank, int d_out, const float *e,
                          const float *s, void *Bout, cudaStream_t st) {
    (void)cudaGetLastError();
    const int b = blocks_for((size_t)d_out * rank, 256);
    if (f32)
        fold_B_kernel<float><<<b, 256, 0, st>>>((const float *)B, rank, d_out, e, s, (float *)Bout);
    else
        fold_B_kernel<__nv_bfloat16><<<b, 256, 0, st>>>((const __nv_bfloat16 *)B, rank, d_out, e, s,
                                                        (__nv_bfloat16 *)Bout);
    return cudaGetLastError();
}

cudaError_t launch_dora_scale(bool f32, const void *Wt, int kdim, int d_in, int d_out,
                              const void *A, const void *B, int rank, float c,
                              const float *m, float *s_out, int *err, cudaStream_t st) {
    (void)cudaGetLastError();
    const int warps = 8;
    dim3 grid((d_out + warps - 1) / warps), block(32 * warps);
    if (f32)
        dora_scale_kernel<float><<<grid, block, 0, st>>>((const float *)Wt, kdim, d_in, d_out,
                                                         (const float *)A, (const float *)B, rank, c, m,
                                                         s_out, err);
    else
        dora_scale_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(
            (const __nv_bfloat16 *)Wt, kdim, d_in, d_out, (const __nv_bfloat16 *)A,
            (const __nv_bfloat16 *)B, rank, c, m, s_out, err);
    return cudaGetLastError();
}

cudaError_t launch_scale_vec(const float *v, float c, float *out, int n, cudaStream_t st) {
    (void)cudaGetLastError();
    scale_vec_kernel<<<(n + 255) / 256, 256, 0, st>>>(v, c, out, n);
    return cudaGetLastError();
}

cudaError_t launch_transpose_blocks(const void *src, void *dst, int n_blk, cudaStream_t st) {
    (void)cudaGetLastError();
    if (n_blk <= 0) return cudaSuccess;
    transpose_blocks_kernel<<<n_blk, dim3(32, 8), 0, st>>>(reinterpret_cast<const __nv_bfloat16 *>(src),
                                                         reinterpret_cast<__nv_bfloat16 *>(dst));
    return cudaGetLastError();
}

}  // namespace scute
