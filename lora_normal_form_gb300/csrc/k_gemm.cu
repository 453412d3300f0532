// tcgen05 / TMEM / TMA GEMM with the normal-form epilogues.
//
// One kernel serves the three dense contractions of the adapted layer:
//   EPI_BASE    out[token] = (x' W) * s[a] + b[a]        the shared base GEMM
//               (article "Scute: Exact Batched Serving for PEFT Adapters
//               Beyond LoRA", paper-daily.com, section "The big picture": h = xW
//               once for the whole batch; s is applied "where the output tile
//               already is", section "Where is the cheapest place to compute the
//               remaining slots?")
//   EPI_VERA_D  U = (X_v A_sh) * d[a]                     VeRA shared shrink
//   EPI_VERA_E  out[token] += (U B_sh) * e[a]             VeRA shared expand
//               (same section: VeRA's shared matrices multiplied for the whole
//               batch at once, rows scaled by their tenant's d and e, rows that
//               do not belong to a VeRA tenant skipped)
//
// Shape of one work tile: D[128 x BN] = P[128 rows, K] * Q[BN rows, K]^T with
// both operands K-major.  For small token counts (decode) the features sit on
// the 128-row P side and the tokens on the BN side (P = W^T, Q = x'), and the
// K dimension is split over a thread-block cluster whose partial tiles are
// reduced through distributed shared memory.  For large token counts
// (prefill) tokens sit on P and features on Q, and a persistent grid walks the
// tiles with a double-buffered TMEM accumulator.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs from one thread, warps 2..5 drain TMEM (tcgen05.ld) and run
// the epilogue.  Every mbarrier wait is bounded (a time limit on %globaltimer);
// on expiry the CTA records STATUS_TIMEOUT, drains what it issued, frees TMEM
// and returns.
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

constexpr int GEMM_THREADS = 192;
constexpr int MAX_STAGES = 8;
constexpr int TILE_M = 128;
constexpr int BOX_ROWS = 64;
constexpr int BOX_BYTES = BOX_ROWS * 128;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s per wait
constexpr int CTRL_BYTES = 256;

// Shared-memory matrix descriptor for a K-major tile in the canonical
// 128-byte-swizzle layout that TMA writes: rows of 128 bytes, 8-row atoms of
// 1024 bytes stacked along M/N (stride byte offset 1024).  The tile base is
// 1024-byte aligned, so the base-offset field is 0; advancing K by 32 bytes
// inside the atom adds 2 to the 16-byte-unit start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset
    d |= (uint64_t)1 << 46;                     // descriptor version
    d |= (uint64_t)2 << 61;                     // 128-byte swizzle
    return d;
}

// Instruction descriptor: f32 accumulator, A/B bf16 (1) or tf32 (2), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc(bool tf32, int M, int N) {
    return (1u << 4) | ((tf32 ? 2u : 1u) << 7) | ((tf32 ? 2u : 1u) << 10) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Ctrl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Ctrl) <= CTRL_BYTES, "control block");

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's
// abort flag) when the time limit passes, or when another role aborted.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      bool honour_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (honour_abort && *abort_flag) return false;
        if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void store_elem(void *out, int f32, size_t idx, float v, bool add) {
    if (f32) {
        float *o = reinterpret_cast<float *>(out) + idx;
        *o = add ? (*o + v) : v;
    } else {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(out) + idx;
        const float prev = add ? __bfloat162float(*o) : 0.f;
        *o = __float2bfloat16_rn(prev + v);
    }
}

// Per-row context of the epilogue: which output row and which live vectors.
struct RowCtx {
    long long out_row;     // token index (output row) or U row
    const float *v1;       // s (BASE), d (VERA_D), e (VERA_E)
    const float *v2;       // b (BASE)
};

__device__ __forceinline__ RowCtx row_ctx(const GemmArgs &g, int i, int sorted_base) {
    RowCtx r;
    const int srow = sorted_base + i;
    const int a = g.aid_s[srow];
    r.v1 = nullptr;
    r.v2 = nullptr;
    if (g.epi == EPI_VERA_D) {
        r.out_row = i;
        if (a >= 0) r.v1 = g.slots[a].vd;
    } else {
        r.out_row = g.perm[srow];
        if (a >= 0) {
            if (g.epi == EPI_BASE) {
                r.v1 = g.slots[a].s;
                r.v2 = g.slots[a].b;
            } else {
                r.v1 = g.slots[a].ve;
            }
        }
    }
    return r;
}

// One output element.
__device__ __forceinline__ void emit1(const GemmArgs &g, const RowCtx &r, int j, float acc) {
    if (g.epi == EPI_BASE) {
        float v = acc;
        if (r.v1) v *= __ldg(r.v1 + j);
        if (r.v2) v += __ldg(r.v2 + j);
        store_elem(g.out, g.out_f32, (size_t)r.out_row * g.ld_out + j, v, false);
    } else if (g.epi == EPI_VERA_E) {
        float v = acc;
        if (r.v1) v *= __ldg(r.v1 + j);
        store_elem(g.out, g.out_f32, (size_t)r.out_row * g.ld_out + j, v, true);
    } else {
        float v = r.v1 ? acc * __ldg(r.v1 + j) : 0.f;
        if (g.u_split3) {
            float *U = reinterpret_cast<float *>(g.U) + (size_t)r.out_row * g.ldu;
            const float hi = ptx::to_tf32(v);
            U[j] = hi;
            U[g.u_rank + j] = hi;
            U[2 * g.u_rank + j] = v - hi;
        } else {
            reinterpret_cast<__nv_bfloat16 *>(g.U)[(size_t)r.out_row * g.ldu + j] =
                __float2bfloat16_rn(v);
        }
    }
}

// 32 consecutive features [j0, j0+32) of one row (normal orientation).
__device__ __forceinline__ void emit32(const GemmArgs &g, const RowCtx &r, int j0,
                                       const float (&acc)[32]) {
    float v[32];
    if (g.epi == EPI_VERA_D) {
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
            float4 d4 = r.v1 ? __ldg(reinterpret_cast<const float4 *>(r.v1 + j0 + k))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            v[k] = acc[k] * d4.x; v[k + 1] = acc[k + 1] * d4.y;
            v[k + 2] = acc[k + 2] * d4.z; v[k + 3] = acc[k + 3] * d4.w;
        }
        if (g.u_split3) {
            float *U = reinterpret_cast<float *>(g.U) + (size_t)r.out_row * g.ldu;
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                float4 hi, lo;
                hi.x = ptx::to_tf32(v[k]); hi.y = ptx::to_tf32(v[k + 1]);
                hi.z = ptx::to_tf32(v[k + 2]); hi.w = ptx::to_tf32(v[k + 3]);
                lo.x = v[k] - hi.x; lo.y = v[k + 1] - hi.y; lo.z = v[k + 2] - hi.z; lo.w = v[k + 3] - hi.w;
                *reinterpret_cast<float4 *>(U + j0 + k) = hi;
                *reinterpret_cast<float4 *>(U + g.u_rank + j0 + k) = hi;
                *reinterpret_cast<float4 *>(U + 2 * g.u_rank + j0 + k) = lo;
            }
        } else {
            __nv_bfloat16 *U = reinterpret_cast<__nv_bfloat16 *>(g.U) + (size_t)r.out_row * g.ldu + j0;
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
                uint4 pk;
                __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(v[k + 2 * e], v[k + 2 * e + 1]);
                *reinterpret_cast<uint4 *>(U + k) = pk;
            }
        }
        return;
    }
    const bool add = (g.epi == EPI_VERA_E);
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
        float4 s4 = r.v1 ? __ldg(reinterpret_cast<const float4 *>(r.v1 + j0 + k))
                         : make_float4(1.f, 1.f, 1.f, 1.f);
        float4 b4 = r.v2 ? __ldg(reinterpret_cast<const float4 *>(r.v2 + j0 + k))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        v[k] = acc[k] * s4.x + b4.x; v[k + 1] = acc[k + 1] * s4.y + b4.y;
        v[k + 2] = acc[k + 2] * s4.z + b4.z; v[k + 3] = acc[k + 3] * s4.w + b4.w;
    }
    if (g.out_f32) {
        float *o = reinterpret_cast<float *>(g.out) + (size_t)r.out_row * g.ld_out + j0;
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
            float4 w = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
            if (add) {
                float4 p = *reinterpret_cast<float4 *>(o + k);
                w.x += p.x; w.y += p.y; w.z += p.z; w.w += p.w;
            }
            *reinterpret_cast<float4 *>(o + k) = w;
        }
    } else {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(g.out) + (size_t)r.out_row * g.ld_out + j0;
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
            uint4 pk;
            if (add) {
                uint4 prev = *reinterpret_cast<uint4 *>(o + k);
                const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&prev);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = __bfloat1622float2(q2[e]);
                    v[k + 2 * e] += f.x;
                    v[k + 2 * e + 1] += f.y;
                }
            }
            __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
            for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(v[k + 2 * e], v[k + 2 * e + 1]);
            *reinterpret_cast<uint4 *>(o + k) = pk;
        }
    }
}

template <int BN, bool TF32>
__global__ void __launch_bounds__(GEMM_THREADS, BN == 64 ? 2 : 1)
    gemm_tc_kernel(const __grid_constant__ GemmArgs g) {
    constexpr int STAGE_BYTES = TILE_M * 128 + BN * 128;
    constexpr uint32_t NCOLS = 2 * BN;
    constexpr int KE = TF32 ? 32 : 64;  // elements per 128-byte K block
    constexpr uint32_t IDESC = instr_desc(TF32, TILE_M, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int stages = g.stages;
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + stages * STAGE_BYTES);
    volatile int *abort_flag = &ctrl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool sched_dep = (g.tok_cnt != nullptr) || (g.tok_base != nullptr);
    if (sched_dep) ptx::grid_dep_wait();

    // ---- tile schedule
    const int n_tok = g.tok_cnt ? *g.tok_cnt : g.n_tok_host;
    const int tok_base = g.tok_base ? *g.tok_base : 0;
    const int sorted_base = g.sorted_base ? *g.sorted_base : 0;
    const int TOKT = g.tok_on_p ? TILE_M : BN;
    const int n_tt = (n_tok + TOKT - 1) / TOKT;
    const int n_tiles = g.n_ft * n_tt;
    const int splits = g.splits;
    const int crank = splits > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int tile0 = splits > 1 ? (int)(blockIdx.x / splits) : (int)blockIdx.x;
    const int tstep = splits > 1 ? n_tiles : (int)gridDim.x;  // one tile per cluster when split
    if (tile0 >= n_tiles) return;  // uniform across a cluster
    const int kb0 = (int)((long long)crank * g.kblocks / splits);
    const int kb1 = (int)((long long)(crank + 1) * g.kblocks / splits);

    // ---- set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->tfull[a]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->tempty[a]), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&ctrl->drain), 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&g.mapP);
        ptx::prefetch_tmap(&g.mapQ);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctrl->tmem_base), NCOLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl->tmem_base;

    if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool dep_done = sched_dep;
            for (int tile = tile0; tile < n_tiles; tile += tstep) {
                const int ft = tile % g.n_ft, tt = tile / g.n_ft;
                const int prow = g.tok_on_p ? tok_base + tt * TILE_M : ft * TILE_M;
                const int qrow = g.tok_on_p ? ft * BN : tok_base + tt * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar(ptx::smem_u32(&ctrl->empty[stage]), phase ^ 1, abort_flag)) goto prod_done;
                    const uint32_t fb = ptx::smem_u32(&ctrl->full[stage]);
                    const uint32_t sP = ptx::smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sQ = sP + TILE_M * 128;
                    const int kc = kb * KE;
                    ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    if (!g.tok_on_p) {
                        // P (weights) does not depend on earlier kernels: it is
                        // fetched before the grid dependency resolves.
                        ptx::tma_load_2d(sP, &g.mapP, kc, prow, fb);
                        ptx::tma_load_2d(sP + BOX_BYTES, &g.mapP, kc, prow + BOX_ROWS, fb);
                        if (!dep_done) { ptx::grid_dep_wait(); dep_done = true; }
#pragma unroll
                        for (int j = 0; j < BN / BOX_ROWS; ++j)
                            ptx::tma_load_2d(sQ + j * BOX_BYTES, &g.mapQ, kc, qrow + j * BOX_ROWS, fb);
                    } else {
                        if (!dep_done) { ptx::grid_dep_wait(); dep_done = true; }
                        ptx::tma_load_2d(sP, &g.mapP, kc, prow, fb);
                        ptx::tma_load_2d(sP + BOX_BYTES, &g.mapP, kc, prow + BOX_ROWS, fb);
#pragma unroll
                        for (int j = 0; j < BN / BOX_ROWS; ++j)
                            ptx::tma_load_2d(sQ + j * BOX_BYTES, &g.mapQ, kc, qrow + j * BOX_ROWS, fb);
                    }
                    ++issued;
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
            }
        prod_done:
            // every issued copy must have landed before the CTA may exit
            {
                const int m_max = issued < stages ? (int)issued : stages;
                for (int m = 1; m <= m_max; ++m) {
                    const int s = (stage - m + stages) % stages;
                    const uint32_t ph = (s < stage) ? phase : (phase ^ 1);
                    wait_bar(ptx::smem_u32(&ctrl->full[s]), ph, abort_flag, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = tile0; tile < n_tiles; tile += tstep) {
                if (!wait_bar(ptx::smem_u32(&ctrl->tempty[acc]), acc_phase ^ 1, abort_flag)) goto mma_done;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar(ptx::smem_u32(&ctrl->full[stage]), phase, abort_flag)) goto mma_done;
                    ptx::tc_fence_after();
                    const uint32_t sP = ptx::smem_u32(smem + stage * STAGE_BYTES);
                    const uint64_t da = sw128_desc(sP);
                    const uint64_t db = sw128_desc(sP + TILE_M * 128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (kb > kb0 || kk > 0) ? 1u : 0u;
                        if (TF32)
                            ptx::mma_tf32(d_tmem, da + 2 * kk, db + 2 * kk, IDESC, accum);
                        else
                            ptx::mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, IDESC, accum);
                    }
                    ptx::mma_commit(ptx::smem_u32(&ctrl->empty[stage]));
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
                ptx::mma_commit(ptx::smem_u32(&ctrl->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
        mma_done:
            // all MMAs this thread issued must finish before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&ctrl->drain));
            wait_bar(ptx::smem_u32(&ctrl->drain), 0, abort_flag, false);
        }
        __syncwarp();
    } else {
        // ================================================= epilogue warps
        ptx::grid_dep_wait();
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = tile0; tile < n_tiles; tile += tstep) {
            if (!wait_bar(ptx::smem_u32(&ctrl->tfull[acc]), acc_phase, abort_flag)) break;
            ptx::tc_fence_after();
            const int ft = tile % g.n_ft, tt = tile / g.n_ft;
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (splits > 1) {
                // partial tile -> own shared memory, [token][128 features]
                float *red = reinterpret_cast<float *>(smem);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    ptx::tmem_ld32(tb + c * 32, v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) red[(c * 32 + k) * TILE_M + row] = v[k];
                }
            } else if (!g.tok_on_p) {
                // features on rows, tokens on columns
                const int j = ft * TILE_M + row;
                int last_i = -1;
                RowCtx rc;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    ptx::tmem_ld32(tb + c * 32, v);
                    if (c == BN / 32 - 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[acc]));
                    }
                    if (j < g.n_feat) {
#pragma unroll 1
                        for (int k = 0; k < 32; ++k) {
                            const int i = tt * BN + c * 32 + k;
                            if (i >= n_tok) break;
                            if (i != last_i) { rc = row_ctx(g, i, sorted_base); last_i = i; }
                            emit1(g, rc, j, v[k]);
                        }
                    }
                }
            } else {
                // tokens on rows, features on columns
                const int i = tt * TILE_M + row;
                const bool live = i < n_tok;
                RowCtx rc;
                if (live) rc = row_ctx(g, i, sorted_base);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    ptx::tmem_ld32(tb + c * 32, v);
                    if (c == BN / 32 - 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[acc]));
                    }
                    const int j0 = ft * BN + c * 32;
                    if (live && j0 < g.n_feat) emit32(g, rc, j0, v);
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();

    if (splits > 1) {
        // ---- cluster split-K: reduce the partial tiles through DSMEM
        ptx::cluster_sync();
        int any_abort = 0;
        const uint32_t red_base = ptx::smem_u32(smem);
        for (int r = 0; r < splits; ++r)
            any_abort |= ptx::ld_dsmem_s32(ptx::mapa(ptx::smem_u32(&ctrl->abort), (uint32_t)r));
        if (!any_abort && warp >= 2) {
            const int et = threadIdx.x - 64;
            const int FR = TILE_M / splits;   // feature rows finalised by this CTA
            const int fl = et % FR, tg = et / FR, TG = 128 / FR;
            const int f = crank * FR + fl;
            const int ft = tile0 % g.n_ft, tt = tile0 / g.n_ft;
            const int j = ft * TILE_M + f;
            uint32_t rb[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) rb[r] = r < splits ? ptx::mapa(red_base, (uint32_t)r) : 0u;
            if (j < g.n_feat) {
                int last_i = -1;
                RowCtx rc;
#pragma unroll 1
                for (int t = tg; t < BN; t += TG) {
                    const int i = tt * BN + t;
                    if (i >= n_tok) break;
                    float sum = 0.f;
                    const uint32_t off = (uint32_t)(t * TILE_M + f) * 4u;
#pragma unroll
                    for (int r = 0; r < 8; ++r)
                        if (r < splits) sum += ptx::ld_dsmem_f32(rb[r] + off);
                    if (i != last_i) { rc = row_ctx(g, i, sorted_base); last_i = i; }
                    emit1(g, rc, j, sum);
                }
            }
        }
        ptx::cluster_sync();
    }

    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, NCOLS);
    }
    if (threadIdx.x == 0 && ctrl->abort) atomicOr(g.status, STATUS_TIMEOUT);
}

template <int BN, bool TF32>
cudaError_t launch_one(const GemmArgs &g, const GemmPlan &p, cudaStream_t st, bool pdl) {
    static bool attr_set = false;
    auto kern = gemm_tc_kernel<BN, TF32>;
    if (!attr_set) {
        cudaError_t e = allow_max_dynamic_smem(kern);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (p.splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)p.splits;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, g);
}

}  // namespace

GemmPlan plan_gemm(int n_tok, int n_feat, int kblocks, bool tok_on_p, bool tf32, int num_sms) {
    GemmPlan p{};
    p.tf32 = tf32 ? 1 : 0;
    if (tok_on_p) {
        // prefill orientation: 128 tokens x 256 features, persistent tiles
        p.bn = 256;
        p.splits = 1;
        p.stages = 4;
        const int tiles = ((n_tok + TILE_M - 1) / TILE_M) * ((n_feat + p.bn - 1) / p.bn);
        p.grid = tiles < num_sms ? tiles : num_sms;
    } else {
        // decode orientation: 128 features x BN tokens, K split over a cluster
        p.bn = n_tok <= 64 ? 64 : (n_tok <= 128 ? 128 : 256);
        const int n_ft = (n_feat + TILE_M - 1) / TILE_M;
        const int n_tt = (n_tok + p.bn - 1) / p.bn;
        const int tiles = n_ft * n_tt;
        const int per_sm = p.bn == 64 ? 2 : 1;
        const int target = per_sm * num_sms;
        p.stages = p.bn == 64 ? 4 : (p.bn == 128 ? 5 : 4);
        int s = 1;
        while (s < 8 && tiles * (s * 2) <= target && kblocks / (s * 2) >= 4) s *= 2;
        p.splits = s;
        p.grid = tiles * s;
    }
    if (p.grid < 1) p.grid = 1;
    const int stage_bytes = TILE_M * 128 + p.bn * 128;
    p.smem = 1024 + (size_t)p.stages * stage_bytes + CTRL_BYTES;
    return p;
}

cudaError_t launch_gemm(const GemmArgs &g, const GemmPlan &p, cudaStream_t st, bool pdl) {
    if (p.tf32) {
        switch (p.bn) {
            case 64: return launch_one<64, true>(g, p, st, pdl);
            case 128: return launch_one<128, true>(g, p, st, pdl);
            default: return launch_one<256, true>(g, p, st, pdl);
        }
    }
    switch (p.bn) {
        case 64: return launch_one<64, false>(g, p, st, pdl);
        case 128: return launch_one<128, false>(g, p, st, pdl);
        default: return launch_one<256, false>(g, p, st, pdl);
    }
}

}  // namespace scute
