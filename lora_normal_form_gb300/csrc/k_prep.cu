// Decode-batch prologue: everything of one adapted-layer call that depends only
// on x and the ids, in one launch.
//
// For a small batch (n <= 128 tokens) every CTA orders the ids itself in
// shared memory (key = (method, adapter id), ties in token order: the same
// stable grouping the stand-alone indexing kernel produces), then serves one
// work item:
//   * gather / rotate   x'[i] = x[perm[i]] R_a for OFT rows, a copy otherwise;
//                       per 256-column chunk one CTA copies the unrotated rows
//                       and one CTA per rotated segment rotates its rows (article "Scute: Exact
//                       Batched Serving for PEFT Adapters Beyond LoRA",
//                       paper-daily.com, section "Where is the cheapest place
//                       to compute the remaining slots?": OFT's rotation runs
//                       in its own pass before the shared GEMM);
//   * low-rank shrink   v[i][q] = x_i A'_a[q] for 4 ranks of one segment
//                       (section "The big picture": the shrink multiplies the
//                       input by A down to rank dimensions; c and d already
//                       folded into A');
//   * VeRA shrink       U[i][q] = d_a[q] (x_i A_sh)[q] for 4 of the shared
//                       ranks over all VeRA rows (section "Where is the cheapest
//                       place...": x A for the batch's VeRA rows, scaled by the
//                       row's tenant's d).
// CTA 0 also writes the index (perm, per-row adapter, segments, per-method
// counts) that the fused GEMM's epilogue reads.  The low-rank and VeRA
// intermediates stay in fp32 / bf16 and are consumed by the fused GEMM.
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

constexpr int PREP_THREADS = 256;
constexpr int SHRINK_ROWS = 4;    // rows per pass of the shrink
constexpr int SHRINK_Q = 4;       // ranks per shrink work item
constexpr int ROT_ROWS = 16;      // rows rotated per batch

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

struct PrepSmem {
    uint32_t key[PREP_MAX_TOKENS];      // key of token t
    int perm[PREP_MAX_TOKENS];          // sorted row -> token
    uint32_t skey[PREP_MAX_TOKENS];     // key of sorted row
    int seg_start[PREP_MAX_TOKENS + 1];
    int seg_aid[PREP_MAX_TOKENS];
    int seg_rank[PREP_MAX_TOKENS];
    const void *row_R[PREP_MAX_TOKENS]; // rotation of each sorted row (null = copy)
    int seg_lr[PREP_MAX_TOKENS];        // segment has an owned low-rank term
    int row_lr[PREP_MAX_TOKENS];        // sorted row's adapter has an owned term
    int warp_tot[33];
    int count[N_RANKS], offset[N_RANKS], segc[N_RANKS];
    int n_seg, bad;
    float red[PREP_THREADS / 32][32];
    const float *row_vd[PREP_MAX_TOKENS]; // VeRA d of each sorted row
    float R[8][OFT_BLK][OFT_BLK];
    float xrows[ROT_ROWS][256];
};

// x_i A_rows^T for up to 4 rows of A (each [d_in], bf16) and the sorted rows
// [r0, r1); emit(i, q, value) is called by one thread per (row, q).  Each
// thread covers 8 consecutive k per pass, loading its A and x vectors before
// any multiply; a warp then reduces its 16 partial sums (4 rows x 4 ranks)
// with a transposing butterfly (16 shuffles) so that lanes 2s and 2s+1 hold
// sum s, and the 8 warps' sums are added in a fixed order.
template <typename Emit>
__device__ void shrink(const __nv_bfloat16 *x, int d_in, const int *perm, int r0, int r1,
                       const __nv_bfloat16 *Arows, int nq, PrepSmem &sm, Emit emit) {
    constexpr int NV = SHRINK_ROWS * SHRINK_Q;   // 16
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int rc = r0; rc < r1; rc += SHRINK_ROWS) {
        const int nr = min(SHRINK_ROWS, r1 - rc);
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = 0.f;
#pragma unroll 2
        for (int k = tid * 8; k < d_in; k += PREP_THREADS * 8) {
            float a[SHRINK_Q][8], xv[SHRINK_ROWS][8];
#pragma unroll
            for (int q = 0; q < SHRINK_Q; ++q) {
                if (q < nq) load8(Arows + (size_t)q * d_in + k, a[q]);
                else
#pragma unroll
                    for (int e = 0; e < 8; ++e) a[q][e] = 0.f;
            }
#pragma unroll
            for (int r = 0; r < SHRINK_ROWS; ++r) {
                if (r < nr) load8(x + (size_t)perm[rc + r] * d_in + k, xv[r]);
                else
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[r][e] = 0.f;
            }
#pragma unroll
            for (int r = 0; r < SHRINK_ROWS; ++r)
#pragma unroll
                for (int q = 0; q < SHRINK_Q; ++q)
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[r * SHRINK_Q + q] = fmaf(xv[r][e], a[q][e], v[r * SHRINK_Q + q]);
        }
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
        if ((lane & 1) == 0) sm.red[w][lane >> 1] = v[0];
        __syncthreads();
        if (tid < NV) {
            const int r = tid / SHRINK_Q, q = tid % SHRINK_Q;
            float s = 0.f;
#pragma unroll
            for (int ww = 0; ww < PREP_THREADS / 32; ++ww) s += sm.red[ww][tid];
            if (r < nr && q < nq) emit(rc + r, q, s);
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(PREP_THREADS, 2) prep_kernel(const __grid_constant__ PrepArgs p) {
    extern __shared__ uint8_t smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int n = p.n;
    const uint32_t A = (uint32_t)p.A;
    const uint32_t base_key = (uint32_t)RANK_BASE * A;

    ptx::grid_dep_wait();
    ptx::grid_dep_launch();

    // ---- order the ids (every CTA): rank of each token among (key, token)
    if (tid == 0) sm.bad = 0;
    if (tid < N_RANKS) { sm.count[tid] = 0; sm.segc[tid] = 0; }
    // the id's method and its slot pointers are fetched together (one round
    // of dependent loads), then carried to the token's sorted row
    const void *tR = nullptr;
    const float *tvd = nullptr;
    int t_lr = 0;
    if (tid < n) {
        const int id = p.ids[tid];
        int m = -1;
        if (id >= 0 && id < p.A) {
            m = p.method_tab[id];
            const Slot &sl = p.slots[id];
            tR = sl.R;
            tvd = sl.vd;
            t_lr = sl.A != nullptr && sl.rank > 0;
        }
        if (m < 0 && id != -1) sm.bad = 1;
        if (m < 0) { tR = nullptr; tvd = nullptr; t_lr = 0; }
        sm.key[tid] = m >= 0 ? (uint32_t)m * A + (uint32_t)id : base_key;
    }
    __syncthreads();
    if (tid < n) {
        const uint32_t kt = sm.key[tid];
        int r = 0;
        for (int u = 0; u < n; ++u) {
            const uint32_t ku = sm.key[u];
            r += (ku < kt) || (ku == kt && u < tid);
        }
        sm.perm[r] = tid;
        sm.skey[r] = kt;
        sm.row_R[r] = tR;
        sm.row_vd[r] = tvd;
        sm.row_lr[r] = t_lr;
    }
    __syncthreads();
    // segments: runs of one key in sorted order
    const bool head = tid < n && (tid == 0 || sm.skey[tid] != sm.skey[tid - 1]);
    const int incl = warp_incl_scan(head ? 1 : 0);
    if (lane == 31) sm.warp_tot[w] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int k = 0; k < PREP_THREADS / 32; ++k) {
            const int c = sm.warp_tot[k];
            sm.warp_tot[k] = run;
            run += c;
        }
        sm.n_seg = run;
    }
    __syncthreads();
    int aid = -1, rank = RANK_BASE;
    if (tid < n) {
        const uint32_t k = sm.skey[tid];
        rank = (int)(k / A);
        aid = rank >= RANK_BASE ? -1 : (int)(k - (uint32_t)rank * A);
        atomicAdd(&sm.count[rank], 1);
        if (head) {
            const int s = sm.warp_tot[w] + incl - 1;
            sm.seg_start[s] = tid;
            sm.seg_aid[s] = aid;
            sm.seg_rank[s] = rank;
            sm.seg_lr[s] = sm.row_lr[tid];
            atomicAdd(&sm.segc[rank], 1);
        }
    }
    if (tid == 0) sm.seg_start[sm.n_seg] = n;
    __syncthreads();
    if (tid == 0) {
        int off = 0;
        for (int r = 0; r < N_RANKS; ++r) {
            sm.offset[r] = off;
            off += sm.count[r];
        }
    }
    __syncthreads();

    const int b = blockIdx.x;
    if (b == 0) {
        // ---- the index, for the fused GEMM
        if (tid < n) {
            p.perm[tid] = sm.perm[tid];
            p.aid_s[tid] = aid;
        }
        if (tid < sm.n_seg) {
            p.seg_start[tid] = sm.seg_start[tid];
            p.seg_aid[tid] = sm.seg_aid[tid];
        }
        if (tid == 0) {
            p.seg_start[sm.n_seg] = n;
            p.meta->n_seg = sm.n_seg;
            for (int r = 0; r < N_RANKS; ++r) {
                p.meta->count[r] = sm.count[r];
                p.meta->offset[r] = sm.offset[r];
                p.meta->seg_count[r] = sm.segc[r];
            }
            if (sm.bad) atomicOr(p.status, STATUS_BAD_ADAPTER);
        }
    }

    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(p.x);
    if (b < p.n_rot) {
        // ================= gather / rotate: item = (256-column chunk, part);
        // part 0 copies every unrotated row of the chunk, part k >= 1 rotates
        // the k-th rotated segment (one adapter's rows) of the chunk
        const int chunks = (p.d_in + 255) / 256;
        const int chunk = b % chunks, part = b / chunks;
        const int col0 = chunk * 256;
        const int ncols = min(256, p.d_in - col0);
        __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(p.xs);
        if (part == 0) {
            // 32 threads x 8 columns per row; each warp handles rows w, w+8, ...
            // and issues up to 8 row loads before storing any
            const int c = lane * 8;
            for (int i0 = w; i0 < n; i0 += 8 * (PREP_THREADS / 32)) {
                uint4 buf[8];
                bool live[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * (PREP_THREADS / 32);
                    live[u] = i < n && c < ncols && sm.row_R[i] == nullptr;
                    if (live[u]) buf[u] = *reinterpret_cast<const uint4 *>(x + (size_t)sm.perm[i] * p.d_in + col0 + c);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * (PREP_THREADS / 32);
                    if (live[u]) *reinterpret_cast<uint4 *>(xs + (size_t)i * p.kdim + col0 + c) = buf[u];
                }
            }
            return;
        }
        int seg = -1, seen = 0;
        for (int sgi = 0; sgi < sm.n_seg; ++sgi) {
            if (sm.row_R[sm.seg_start[sgi]] == nullptr) continue;
            if (++seen == part) { seg = sgi; break; }
        }
        if (seg < 0) return;
        const int s0 = sm.seg_start[seg], s1 = sm.seg_start[seg + 1];
        const __nv_bfloat16 *Rb = reinterpret_cast<const __nv_bfloat16 *>(sm.row_R[s0]) +
                                  (size_t)(col0 / OFT_BLK) * OFT_BLK * OFT_BLK;
        const int nvec = (ncols / OFT_BLK) * OFT_BLK * OFT_BLK / 8;   // <= 4 per thread
        {
            uint4 rbuf[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = tid + u * PREP_THREADS;
                if (e < nvec) rbuf[u] = *reinterpret_cast<const uint4 *>(Rb + (size_t)e * 8);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = tid + u * PREP_THREADS;
                if (e < nvec) {
                    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&rbuf[u]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 f = __bfloat1622float2(h[q]);
                        (&sm.R[0][0][0])[e * 8 + 2 * q] = f.x;
                        (&sm.R[0][0][0])[e * 8 + 2 * q + 1] = f.y;
                    }
                }
            }
        }
        // R's 8 blocks of this chunk and up to ROT_ROWS rows of x are staged
        // with 16-byte loads; every thread then produces one column per row
        for (int r0 = s0; r0 < s1; r0 += ROT_ROWS) {
            const int nr = min(ROT_ROWS, s1 - r0);
            {
                uint4 xbuf[2];   // ROT_ROWS * 32 vectors over 256 threads
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = tid + u * PREP_THREADS, rr = e >> 5, c = (e & 31) * 8;
                    if (rr < nr && c < ncols)
                        xbuf[u] = *reinterpret_cast<const uint4 *>(x + (size_t)sm.perm[r0 + rr] * p.d_in + col0 + c);
                    else
                        xbuf[u] = make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = tid + u * PREP_THREADS, rr = e >> 5, c = (e & 31) * 8;
                    if (rr < nr) {
                        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&xbuf[u]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __bfloat1622float2(h[q]);
                            sm.xrows[rr][c + 2 * q] = f.x;
                            sm.xrows[rr][c + 2 * q + 1] = f.y;
                        }
                    }
                }
            }
            __syncthreads();
            if (tid < ncols) {
                const int blk = tid >> 5, cc = tid & 31;
                for (int rr = 0; rr < nr; ++rr) {
                    float acc = 0.f;
#pragma unroll 8
                    for (int m = 0; m < OFT_BLK; ++m)
                        acc = fmaf(sm.xrows[rr][blk * OFT_BLK + m], sm.R[blk][m][cc], acc);
                    xs[(size_t)(r0 + rr) * p.kdim + col0 + tid] = __float2bfloat16_rn(acc);
                }
            }
            __syncthreads();
        }
        return;
    }
    if (b < p.n_rot + p.n_lr) {
        // ================= low-rank shrink: 4 ranks of one owned-term segment
        const int item = b - p.n_rot;
        const int ordinal = item / p.lr_groups, g = item % p.lr_groups;
        int seg = -1, seen = 0;
        for (int s = 0; s < sm.n_seg; ++s) {
            if (!sm.seg_lr[s]) continue;
            if (seen == ordinal) { seg = s; break; }
            ++seen;
        }
        if (seg < 0) return;
        const int a = sm.seg_aid[seg];
        const int r = p.slots[a].rank;
        const int q0 = g * SHRINK_Q;
        if (q0 >= r) return;
        const int nq = min(SHRINK_Q, r - q0);
        const __nv_bfloat16 *Arows = reinterpret_cast<const __nv_bfloat16 *>(p.slots[a].A) + (size_t)q0 * p.d_in;
        float *v = p.v;
        const int ldv = p.v_ld;
        shrink(x, p.d_in, sm.perm, sm.seg_start[seg], sm.seg_start[seg + 1], Arows, nq, sm,
               [&](int i, int q, float s) { v[(size_t)i * ldv + q0 + q] = s; });
        return;
    }
    {
        // ================= VeRA shrink: 4 shared ranks over all VeRA rows
        const int g = b - p.n_rot - p.n_lr;
        const int q0 = g * SHRINK_Q;
        if (q0 >= p.rv) return;
        const int nq = min(SHRINK_Q, p.rv - q0);
        const int r0 = sm.offset[RANK_VERA], r1 = r0 + sm.count[RANK_VERA];
        if (r1 <= r0) return;
        const __nv_bfloat16 *Arows = reinterpret_cast<const __nv_bfloat16 *>(p.Ash) + (size_t)q0 * p.d_in;
        __nv_bfloat16 *U = reinterpret_cast<__nv_bfloat16 *>(p.U);
        const int ldu = p.u_ld;
        const Slot *slots = p.slots;
        (void)slots;
        shrink(x, p.d_in, sm.perm, r0, r1, Arows, nq, sm, [&](int i, int q, float s) {
            const float *d = sm.row_vd[i];
            U[(size_t)i * ldu + q0 + q] = __float2bfloat16_rn(d ? s * d[q0 + q] : 0.f);
        });
    }
}

}  // namespace

size_t prep_smem_bytes() { return sizeof(PrepSmem); }

cudaError_t launch_prep(const PrepArgs &p, int grid, cudaStream_t st, bool pdl) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = allow_max_dynamic_smem(prep_kernel);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(PREP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = sizeof(PrepSmem);
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prep_kernel, p);
}

}  // namespace scute
