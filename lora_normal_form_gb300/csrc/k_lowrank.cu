// Segmented shrink / expand of the owned low-rank term (LoRA, DoRA, raw
// normal form), after the fold rule has put c and d into A and e into B:
//     v_t   = x_t A'_a                      (shrink, fp32, K split in KS parts)
//     out_t += v_t B'_a                     (expand, read-modify-write)
// (article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA",
// paper-daily.com, section "The big picture": the shrink multiplies the input
// by A down to rank dimensions, the expand multiplies by B and adds the result
// to h; section "Which slots can be merged at load?" for the folds).
//
// Work is cut into units of at most 32 sorted rows of one segment (the
// indexing kernel lists them: seg_unit[s] counts the units before segment s),
// so that every CTA serves one adapter, long prefill segments are spread over
// many CTAs, and the many short segments of a decode-like batch each get
// their own:
//   * shrink: grid (units, K chunks); the unit's (row, 16-rank group) items
//     are spread over the 8 warps; lane l covers 8 consecutive k per
//     256-wide step with 16-byte loads of x and of 16 rows of A', and a
//     transposing butterfly of 16 shuffles sums the 16 ranks over the warp;
//     partial sums per K chunk go to v_part[chunk][row][rank];
//   * expand: grid (units, 2048-column chunks); the CTA first sums the K
//     chunks of its rows' v into shared memory, then each thread owns 8
//     output columns, loads 16-byte slices of B' eight ranks at a time (shared
//     by 4 rows per pass) and adds into out in place.
// The shrink reads the original x through the sort permutation (the low-rank
// term acts on x, not on x R).
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

constexpr int LR_GROUP = 16;  // ranks reduced per butterfly

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

// The rows [r0, r1) and adapter of work unit u, or false when u is past the
// last unit or its segment has no adapter.
__device__ __forceinline__ bool unit_rows(int u, const int *__restrict__ seg_start, const int *__restrict__ seg_aid,
                                          const int *__restrict__ seg_unit, const IndexMeta *__restrict__ meta,
                                          int &r0, int &r1, int &a) {
    const int n_seg = meta->n_seg;
    if (u >= seg_unit[n_seg]) return false;
    int lo = 0, hi = n_seg - 1;   // the last segment whose first unit is <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_unit[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    a = seg_aid[lo];
    r0 = seg_start[lo] + (u - seg_unit[lo]) * SEG_UNIT_ROWS;
    r1 = min(seg_start[lo + 1], r0 + SEG_UNIT_ROWS);
    return a >= 0;
}

template <typename T>
__global__ void __launch_bounds__(256, 3) lr_shrink_kernel(const T *__restrict__ x, int d_in,
                                                           const int *__restrict__ perm,
                                                           const int *__restrict__ seg_start,
                                                           const int *__restrict__ seg_aid,
                                                           const int *__restrict__ seg_unit,
                                                           const IndexMeta *__restrict__ meta,
                                                           const Slot *__restrict__ slots, float *v_part,
                                                           int max_tokens, int kchunk) {
    ptx::grid_dep_wait();
    int r0, r1, a;
    if (!unit_rows(blockIdx.x, seg_start, seg_aid, seg_unit, meta, r0, r1, a)) return;
    const T *A = reinterpret_cast<const T *>(slots[a].A);
    const int r = slots[a].rank;
    if (A == nullptr || r <= 0) return;
    extern __shared__ uint4 lr_smem[];
    T *As = reinterpret_cast<T *>(lr_smem);   // [LR_GROUP][kchunk]: one rank group of A' over the K chunk
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = blockIdx.y * kchunk;
    const int k1 = min(d_in, k0 + kchunk);
    constexpr int V = 16 / sizeof(T);         // elements per 16-byte word
    float *vp = v_part + (size_t)blockIdx.y * max_tokens * MAX_RANK;
#pragma unroll 1
    for (int g0 = 0; g0 < r; g0 += LR_GROUP) {
        const int nq = min(LR_GROUP, r - g0);
        // the rank group of A' over this K chunk, staged once for every row
        __syncthreads();
        const int wpr = kchunk / V;   // 16-byte words per staged row
        // eight words per thread per round, all loads of a round issued first
#pragma unroll 1
        for (int e0 = 0; e0 < LR_GROUP * wpr; e0 += 8 * 256) {
            uint4 val[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i * 256 + threadIdx.x;
                const int q = e / wpr, k = k0 + (e - q * wpr) * V;
                val[i] = make_uint4(0u, 0u, 0u, 0u);
                if (e < LR_GROUP * wpr && q < nq && k < k1)
                    val[i] = *reinterpret_cast<const uint4 *>(A + (size_t)(g0 + q) * d_in + k);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i * 256 + threadIdx.x;
                if (e < LR_GROUP * wpr) lr_smem[e] = val[i];
            }
        }
        __syncthreads();
        // warp w takes rows w, w + 8, ... of the unit; a row's K chunk is read
        // in steps of 256 (8 per lane), eight steps' x loads issued together
#pragma unroll 1
        for (int row = r0 + w; row < r1; row += 8) {
            const T *src = x + (size_t)perm[row] * d_in;
            float v[LR_GROUP];
#pragma unroll
            for (int q = 0; q < LR_GROUP; ++q) v[q] = 0.f;
#pragma unroll 1
            for (int kb = k0 + lane * 8; kb < k1; kb += 2048) {
                uint4 xu[8][16 / V == 1 ? 1 : 2];
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int h = 0; h < (16 / V == 1 ? 1 : 2); ++h)
                        xu[u][h] = kb + u * 256 < k1 ? *reinterpret_cast<const uint4 *>(src + kb + u * 256 + h * V)
                                                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = kb + u * 256;
                    if (k >= k1) break;
                    float xv[8];
                    load8(reinterpret_cast<const T *>(&xu[u][0]), xv);
#pragma unroll
                    for (int q = 0; q < LR_GROUP; ++q) {
                        if (q < nq) {
                            float av[8];
                            load8(As + (size_t)q * kchunk + (k - k0), av);
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[q] = fmaf(xv[e], av[e], v[q]);
                        }
                    }
                }
            }
            // transposing butterfly: after it, lanes 2i and 2i + 1 hold the
            // warp's sum for rank g0 + i
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                const int o = 16 >> st, half = 8 >> st;
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
            const int q = lane >> 1;
            if ((lane & 1) == 0 && q < nq) vp[(size_t)row * MAX_RANK + g0 + q] = v[0];
        }
    }
}

template <typename T, int RM>
__global__ void __launch_bounds__(256, 2) lr_expand_kernel(const float *__restrict__ v_part, int ks,
                                                           int max_tokens, int d_out,
                                                           const int *__restrict__ perm,
                                                           const int *__restrict__ seg_start,
                                                           const int *__restrict__ seg_aid,
                                                           const int *__restrict__ seg_unit,
                                                           const IndexMeta *__restrict__ meta,
                                                           const Slot *__restrict__ slots, void *out,
                                                           int out_f32) {
    __shared__ float vs[SEG_UNIT_ROWS][RM];
    ptx::grid_dep_wait();
    int r0, r1, a;
    if (!unit_rows(blockIdx.x, seg_start, seg_aid, seg_unit, meta, r0, r1, a)) return;
    const T *B = reinterpret_cast<const T *>(slots[a].B);
    const int r = slots[a].rank;
    if (B == nullptr || r <= 0) return;
    const int tid = threadIdx.x;
    const int nr = r1 - r0;
    for (int e = tid; e < SEG_UNIT_ROWS * RM; e += 256) {
        const int rr = e / RM, q = e - rr * RM;
        float v = 0.f;
        if (rr < nr && q < r) {
            // the K-chunk partials are loaded together, then added in order
            float pv[KS_MAX];
#pragma unroll
            for (int s = 0; s < KS_MAX; ++s)
                pv[s] = s < ks ? v_part[((size_t)s * max_tokens + r0 + rr) * MAX_RANK + q] : 0.f;
#pragma unroll
            for (int s = 0; s < KS_MAX; ++s) v += pv[s];
        }
        vs[rr][q] = v;
    }
    __syncthreads();
    const int j0 = (blockIdx.y * 256 + tid) * 8;
    if (j0 >= d_out) return;
constexpr int RG = 4;   // rows per pass (one slice of B' serves all of them)
#pragma unroll 1
    for (int g = 0; g < nr; g += RG) {
        const int ng = min(RG, nr - g);
        // the rows' old outputs are requested first, so that their latency
        // overlaps the loads of B' and the products below
        uint4 oldb[RG];
        float4 oldf[RG][2];
        if (!out_f32) {
            const __nv_bfloat16 *ob = reinterpret_cast<const __nv_bfloat16 *>(out);
#pragma unroll
            for (int rr = 0; rr < RG; ++rr)
                if (rr < ng) oldb[rr] = *reinterpret_cast<const uint4 *>(ob + (size_t)perm[r0 + g + rr] * d_out + j0);
        } else {
            const float *of = reinterpret_cast<const float *>(out);
#pragma unroll
            for (int rr = 0; rr < RG; ++rr)
                if (rr < ng) {
                    const float4 *p = reinterpret_cast<const float4 *>(of + (size_t)perm[r0 + g + rr] * d_out + j0);
                    oldf[rr][0] = p[0];
                    oldf[rr][1] = p[1];
                }
        }
        float acc[RG][8];
#pragma unroll
        for (int rr = 0; rr < RG; ++rr)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[rr][e] = 0.f;
#pragma unroll 1
        for (int q0 = 0; q0 < r; q0 += 8) {
            // eight ranks' slices of B' loaded (as stored) before any is used
            constexpr int W = sizeof(T) == 2 ? 1 : 2;   // 16-byte words per 8 values
            uint4 bq[8][W];
#pragma unroll
            for (int q = 0; q < 8; ++q)
#pragma unroll
                for (int h = 0; h < W; ++h)
                    bq[q][h] = q0 + q < r ? *reinterpret_cast<const uint4 *>(B + (size_t)(q0 + q) * d_out + j0 + h * 4)
                                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float bv[8];
                load8(reinterpret_cast<const T *>(&bq[q][0]), bv);
#pragma unroll
                for (int rr = 0; rr < RG; ++rr) {
                    if (rr < ng) {
                        const float vq = vs[g + rr][(q0 + q) & (RM - 1)];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[rr][e] = fmaf(vq, bv[e], acc[rr][e]);
                    }
                }
            }
        }
        if (!out_f32) {
            __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(out);
#pragma unroll
            for (int rr = 0; rr < RG; ++rr) {
                if (rr >= ng) continue;
                __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&oldb[rr]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h[e]);
                    h[e] = __floats2bfloat162_rn(f.x + acc[rr][2 * e], f.y + acc[rr][2 * e + 1]);
                }
                *reinterpret_cast<uint4 *>(ob + (size_t)perm[r0 + g + rr] * d_out + j0) = oldb[rr];
            }
        } else {
            float *of = reinterpret_cast<float *>(out);
#pragma unroll
            for (int rr = 0; rr < RG; ++rr) {
                if (rr >= ng) continue;
                float4 *p = reinterpret_cast<float4 *>(of + (size_t)perm[r0 + g + rr] * d_out + j0);
                float4 u = oldf[rr][0], w = oldf[rr][1];
                u.x += acc[rr][0]; u.y += acc[rr][1]; u.z += acc[rr][2]; u.w += acc[rr][3];
                w.x += acc[rr][4]; w.y += acc[rr][5]; w.z += acc[rr][6]; w.w += acc[rr][7];
                p[0] = u;
                p[1] = w;
            }
        }
    }
}

// The expand for bf16 outputs and ranks <= 16: the thread's 16 slices of B'
// stay in registers for every row of the unit, and the next row pair's old
// outputs are in flight while the current pair is formed.
__global__ void __launch_bounds__(256, 2) lr_expand16_kernel(const float *__restrict__ v_part, int ks,
                                                            int max_tokens, int d_out,
                                                            const int *__restrict__ perm,
                                                            const int *__restrict__ seg_start,
                                                            const int *__restrict__ seg_aid,
                                                            const int *__restrict__ seg_unit,
                                                            const IndexMeta *__restrict__ meta,
                                                            const Slot *__restrict__ slots, void *out) {
    using T = __nv_bfloat16;
    __shared__ float vs[SEG_UNIT_ROWS][16];
    ptx::grid_dep_wait();
    int r0, r1, a;
    if (!unit_rows(blockIdx.x, seg_start, seg_aid, seg_unit, meta, r0, r1, a)) return;
    const T *B = reinterpret_cast<const T *>(slots[a].B);
    const int r = slots[a].rank;
    if (B == nullptr || r <= 0) return;
    const int tid = threadIdx.x;
    const int nr = r1 - r0;
    for (int e = tid; e < SEG_UNIT_ROWS * 16; e += 256) {
        const int rr = e / 16, q = e - rr * 16;
        float v = 0.f;
        if (rr < nr && q < r) {
            float pv[KS_MAX];
#pragma unroll
            for (int s = 0; s < KS_MAX; ++s)
                pv[s] = s < ks ? v_part[((size_t)s * max_tokens + r0 + rr) * MAX_RANK + q] : 0.f;
#pragma unroll
            for (int s = 0; s < KS_MAX; ++s) v += pv[s];
        }
        vs[rr][q] = v;
    }
    __syncthreads();
    const int j0 = (blockIdx.y * 256 + tid) * 8;
    if (j0 >= d_out) return;
    // rank <= 16, bf16: the thread's 16 slices of B' stay in registers
    // for every row of the unit, and the next row pair's old outputs
    // are in flight while the current pair is formed
    const __nv_bfloat16 *Bb = reinterpret_cast<const __nv_bfloat16 *>(B) + j0;
    __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(out);
    uint4 bq[16];
#pragma unroll
    for (int q = 0; q < 16; ++q)
        bq[q] = q < r ? *reinterpret_cast<const uint4 *>(Bb + (size_t)q * d_out) : make_uint4(0u, 0u, 0u, 0u);
    constexpr int RP = 2;   // rows per step
    uint4 cur[RP], nxt[RP];
#pragma unroll
    for (int rr = 0; rr < RP; ++rr)
        if (rr < nr) cur[rr] = *reinterpret_cast<const uint4 *>(ob + (size_t)perm[r0 + rr] * d_out + j0);
#pragma unroll 1
    for (int g = 0; g < nr; g += RP) {
#pragma unroll
        for (int rr = 0; rr < RP; ++rr)
            if (g + RP + rr < nr)
                nxt[rr] = *reinterpret_cast<const uint4 *>(ob + (size_t)perm[r0 + g + RP + rr] * d_out + j0);
        // the slices are converted afresh for every row pair: held converted
        // across the loop they would need 128 registers
#pragma unroll
        for (int q = 0; q < 16; ++q) asm volatile("" : "+r"(bq[q].x), "+r"(bq[q].y), "+r"(bq[q].z), "+r"(bq[q].w));
        float acc[RP][8];
#pragma unroll
        for (int rr = 0; rr < RP; ++rr)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[rr][e] = 0.f;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            float bv[8];
            load8(reinterpret_cast<const T *>(&bq[q]), bv);
#pragma unroll
            for (int rr = 0; rr < RP; ++rr) {
                const float vq = vs[(g + rr) & (SEG_UNIT_ROWS - 1)][q];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[rr][e] = fmaf(vq, bv[e], acc[rr][e]);
            }
        }
#pragma unroll
        for (int rr = 0; rr < RP; ++rr) {
            if (g + rr >= nr) continue;
            __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&cur[rr]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h[e]);
                h[e] = __floats2bfloat162_rn(f.x + acc[rr][2 * e], f.y + acc[rr][2 * e + 1]);
            }
            *reinterpret_cast<uint4 *>(ob + (size_t)perm[r0 + g + rr] * d_out + j0) = cur[rr];
        }
#pragma unroll
        for (int rr = 0; rr < RP; ++rr) cur[rr] = nxt[rr];
    }
}

template <typename T, int RM>
cudaError_t launch_lr(const T *x, int d_in, int d_out, int unit_bound, const int *perm, const int *seg_start,
                      const int *seg_aid, const int *seg_unit, const IndexMeta *meta, const Slot *slots,
                      float *v_part, int max_tokens, void *out, int out_f32, cudaStream_t st, bool pdl,
                      bool shrink, bool expand) {
    int kchunk = 0;
    const int ks = lowrank_ks(d_in, &kchunk);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)unit_bound, (unsigned)ks, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    static std::atomic<unsigned long long> attr_done{0};
    cudaError_t e = cudaSuccess;
    if (shrink) {
        e = allow_max_dynamic_smem(lr_shrink_kernel<T>, attr_done);
        if (e != cudaSuccess) return e;
        cfg.dynamicSmemBytes = (size_t)LR_GROUP * kchunk * sizeof(T);
        e = cudaLaunchKernelEx(&cfg, lr_shrink_kernel<T>, x, d_in, perm, seg_start, seg_aid, seg_unit, meta, slots,
                               v_part, max_tokens, kchunk);
        if (e != cudaSuccess) return e;
    }
    if (!expand) return cudaSuccess;
    cfg.dynamicSmemBytes = 0;
    cfg.gridDim = dim3((unsigned)unit_bound, (unsigned)((d_out + 2047) / 2048), 1);
    if (sizeof(T) == 2 && RM == 16 && !out_f32)
        return cudaLaunchKernelEx(&cfg, lr_expand16_kernel, (const float *)v_part, ks, max_tokens, d_out, perm,
                                  seg_start, seg_aid, seg_unit, meta, slots, out);
    return cudaLaunchKernelEx(&cfg, lr_expand_kernel<T, RM>, (const float *)v_part, ks, max_tokens, d_out, perm,
                              seg_start, seg_aid, seg_unit, meta, slots, out, out_f32);
}

}  // namespace

cudaError_t launch_lowrank(bool f32, const void *x, int d_in, int d_out, int unit_bound, const int *perm,
                           const int *seg_start, const int *seg_aid, const int *seg_unit,
                           const IndexMeta *meta, const Slot *slots, float *v_part, int max_tokens, void *out,
                           int out_f32, cudaStream_t st, bool pdl, int max_rank, bool shrink, bool expand) {
    if (f32) {
        if (max_rank <= 16)
            return launch_lr<float, 16>((const float *)x, d_in, d_out, unit_bound, perm, seg_start, seg_aid, seg_unit,
                                        meta, slots, v_part, max_tokens, out, out_f32, st, pdl, shrink, expand);
        return launch_lr<float, 64>((const float *)x, d_in, d_out, unit_bound, perm, seg_start, seg_aid, seg_unit,
                                    meta, slots, v_part, max_tokens, out, out_f32, st, pdl, shrink, expand);
    }
    if (max_rank <= 16)
        return launch_lr<__nv_bfloat16, 16>((const __nv_bfloat16 *)x, d_in, d_out, unit_bound, perm, seg_start,
                                            seg_aid, seg_unit, meta, slots, v_part, max_tokens, out, out_f32, st, pdl,
                                            shrink, expand);
    return launch_lr<__nv_bfloat16, 64>((const __nv_bfloat16 *)x, d_in, d_out, unit_bound, perm, seg_start, seg_aid,
                                        seg_unit, meta, slots, v_part, max_tokens, out, out_f32, st, pdl, shrink, expand);
}

}  // namespace scute
