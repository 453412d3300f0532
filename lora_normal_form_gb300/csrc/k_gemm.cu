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
// K dimension is split over a thread-block cluster: each CTA of the cluster
// writes its partial tile to an L2-resident workspace in global memory, and
// after a cluster barrier the CTAs read back each other's slices and sum
// them.  For large token counts
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
constexpr int CTRL_BYTES = 512;
constexpr size_t GEMM_SMEM_MAX = 227 * 1024;   // dynamic shared memory of one CTA
// token stride of the partial tiles in shared memory: 128 features plus 4
// floats of padding, so the tokens a warp reads start on different banks
constexpr int RED_LD = TILE_M + 4;

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

// The same for the 64-byte-swizzle layout: rows of 64 bytes, 8-row atoms of
// 512 bytes (stride byte offset 512); 16-byte unit u of row r sits at unit
// u ^ ((r >> 1) & 3).  Base 1024-byte aligned; K advances 32 bytes (+2) per
// 16 bf16 elements.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused here)
    d |= (uint64_t)(512 >> 4) << 32;            // stride byte offset
    d |= (uint64_t)1 << 46;                     // descriptor version
    d |= (uint64_t)4 << 61;                     // 64-byte swizzle
    return d;
}
__device__ __forceinline__ uint32_t sw64_offset(int r, int unit) {
    return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + ((unit ^ ((r >> 1) & 3)) << 4));
}

// Instruction descriptor: f32 accumulator, A/B bf16 (1) or tf32 (2), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc(bool tf32, int M, int N) {
    return (1u << 4) | ((tf32 ? 2u : 1u) << 7) | ((tf32 ? 2u : 1u) << 10) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Owned low-rank expand on the tensor cores (tokens on P, bf16): per tile one
// extra K block of LR_KSTEPS x 16 columns, A = the rows' v (each row in the
// columns of its adapter's k-steps, zeros elsewhere), B = the tile's features
// of each adapter's B, both K-major in the 64-byte-swizzle layout.
// bytes between rows of a tile's staged bf16 output (the 16 extra bytes put
// the rows read by one quarter-warp in different banks)
__host__ __device__ constexpr int out_pitch(int bn) { return bn * 2 + 16; }

constexpr int LR_KSTEPS = 2;
constexpr int LR_A_BYTES = TILE_M * 64;

struct Ctrl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t lrfull;                // the tile's low-rank operands are in shared memory (128 arrivals)
    uint32_t tmem_base;
    int abort;
    // per tile parity: k-steps the MMA issues, each k-step's adapter (-2 none),
    // its first k-step, rank and B, and the epilogue warps' counts of k-steps
    int lr_steps[2];
    int lr_aid[2][LR_KSTEPS], lr_k0[2][LR_KSTEPS], lr_rank[2][LR_KSTEPS];
    int lr_wsum[2][4];
    const void *lr_B[2][LR_KSTEPS];
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

// Per-token context of the epilogue: which output row and which live slots.
struct TokMeta {
    long long out_row;     // token index (output row) or U row
    const float *v1;       // s (BASE), d (VERA_D), e (VERA_E)
    const float *v2;       // b (BASE)
    const void *B;         // fused owned B' [rank][n_feat] (BASE)
    const void *Bm;        // tokens on P: B for the tensor-core expand, added before s
                           // (B' when the adapter has no s, DoRA's B without s; null = none)
    const float *ve;       // fused VeRA e (BASE)
    int rank;              // fused owned rank
    int vera;              // fused: the row is a VeRA row
};

__device__ __forceinline__ TokMeta tok_meta(const GemmArgs &g, int i, int sorted_base) {
    TokMeta m;
    const int srow = sorted_base + i;
    const int a = g.aid_s[srow];
    m.v1 = nullptr;
    m.v2 = nullptr;
    m.B = nullptr;
    m.Bm = nullptr;
    m.ve = nullptr;
    m.rank = 0;
    m.vera = 0;
    if (g.epi == EPI_VERA_D) {
        m.out_row = i;
        if (a >= 0) m.v1 = g.slots[a].vd;
        return m;
    }
    m.out_row = g.perm[srow];
    if (a < 0) return m;
    const Slot &sl = g.slots[a];
    if (g.epi == EPI_VERA_E) {
        m.v1 = sl.ve;
        return m;
    }
    m.v1 = sl.s;
    m.v2 = sl.b;
    if (g.v && sl.B && sl.rank > 0) {
        m.B = sl.B;
        m.Bm = sl.s ? sl.Bu : sl.B;
        m.rank = sl.rank;
    }
    if (g.vera_kb && sl.vd) {
        m.vera = 1;
        m.ve = sl.ve;
    }
    return m;
}

// 32 consecutive features [j0, j0+32) of one row (tokens-on-P orientation).
// vsrc: the row's K-chunk partials of the owned low-rank intermediate when its
// expand is added here on the CUDA cores (bf16 contexts; the tensor-core expand
// did not take the row), else null.
__device__ __forceinline__ void emit32(const GemmArgs &g, const TokMeta &r, int j0, const float (&acc)[32],
                                       const float *vsrc) {
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
    if (vsrc) {
        // owned low-rank expand: y += v_t B'[:, j0:j0+32], four ranks per
        // batch (v summed over the K chunks in chunk order)
        const __nv_bfloat16 *B = reinterpret_cast<const __nv_bfloat16 *>(r.B) + j0;
#pragma unroll 1
        for (int q0 = 0; q0 < r.rank; q0 += 4) {
            float4 vs = __ldg(reinterpret_cast<const float4 *>(vsrc + q0));
            for (int s = 1; s < g.v_ks; ++s) {
                const float4 t = __ldg(reinterpret_cast<const float4 *>(vsrc + s * g.v_kstride + q0));
                vs.x += t.x; vs.y += t.y; vs.z += t.z; vs.w += t.w;
            }
            const float vv[4] = {vs.x, vs.y, vs.z, vs.w};
            uint4 bq[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    bq[u][h] = q0 + u < r.rank ? __ldg(reinterpret_cast<const uint4 *>(B + (size_t)(q0 + u) * g.n_feat) + h)
                                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float vq = q0 + u < r.rank ? vv[u] : 0.f;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&bq[u][h]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(b2[e]);
                        v[h * 8 + 2 * e] = fmaf(vq, f.x, v[h * 8 + 2 * e]);
                        v[h * 8 + 2 * e + 1] = fmaf(vq, f.y, v[h * 8 + 2 * e + 1]);
                    }
                }
            }
        }
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

// Eight consecutive features [j0, j0+8) of token m (features-on-P orientation):
// base / VeRA accumulators in, slots applied, eight outputs stored with one
// vector store.  All loads of one item are independent 16-byte loads.
__device__ __forceinline__ void emit8(const GemmArgs &g, const TokMeta &m, const float *vrow, int j0,
                                      const float (&acc)[8], const float (&vacc)[8]) {
    float y[8];
    if (g.epi == EPI_VERA_D) {
        if (m.v1) {
            const float4 d0 = __ldg(reinterpret_cast<const float4 *>(m.v1 + j0));
            const float4 d1 = __ldg(reinterpret_cast<const float4 *>(m.v1 + j0 + 4));
            y[0] = acc[0] * d0.x; y[1] = acc[1] * d0.y; y[2] = acc[2] * d0.z; y[3] = acc[3] * d0.w;
            y[4] = acc[4] * d1.x; y[5] = acc[5] * d1.y; y[6] = acc[6] * d1.z; y[7] = acc[7] * d1.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = 0.f;
        }
        if (g.u_split3) {
            float *U = reinterpret_cast<float *>(g.U) + (size_t)m.out_row * g.ldu + j0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float hi = ptx::to_tf32(y[k]);
                U[k] = hi;
                U[g.u_rank + k] = hi;
                U[2 * g.u_rank + k] = y[k] - hi;
            }
        } else {
            uint4 pk;
            __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
            for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
            *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(g.U) + (size_t)m.out_row * g.ldu + j0) = pk;
        }
        return;
    }
    if (g.epi == EPI_BASE) {
        float s8[8], b8[8];
        if (m.v1) {
            const float4 a0 = __ldg(reinterpret_cast<const float4 *>(m.v1 + j0));
            const float4 a1 = __ldg(reinterpret_cast<const float4 *>(m.v1 + j0 + 4));
            s8[0] = a0.x; s8[1] = a0.y; s8[2] = a0.z; s8[3] = a0.w; s8[4] = a1.x; s8[5] = a1.y; s8[6] = a1.z; s8[7] = a1.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) s8[k] = 1.f;
        }
        if (m.v2) {
            const float4 a0 = __ldg(reinterpret_cast<const float4 *>(m.v2 + j0));
            const float4 a1 = __ldg(reinterpret_cast<const float4 *>(m.v2 + j0 + 4));
            b8[0] = a0.x; b8[1] = a0.y; b8[2] = a0.z; b8[3] = a0.w; b8[4] = a1.x; b8[5] = a1.y; b8[6] = a1.z; b8[7] = a1.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) b8[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = acc[k] * s8[k] + b8[k];
        if (m.B) {
            // owned low-rank expand: y += v_t B'[:, j0:j0+8], 8 ranks per batch of loads
            const __nv_bfloat16 *B = reinterpret_cast<const __nv_bfloat16 *>(m.B) + j0;
            for (int q0 = 0; q0 < m.rank; q0 += 8) {
                uint4 bq[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q0 + q < m.rank) bq[q] = __ldg(reinterpret_cast<const uint4 *>(B + (size_t)(q0 + q) * g.n_feat));
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (q0 + q < m.rank) {
                        const float vq = vrow[q0 + q];
                        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&bq[q]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(h[e]);
                            y[2 * e] = fmaf(vq, f.x, y[2 * e]);
                            y[2 * e + 1] = fmaf(vq, f.y, y[2 * e + 1]);
                        }
                    }
                }
            }
        }
        if (m.vera) {
            if (m.ve) {
                const float4 a0 = __ldg(reinterpret_cast<const float4 *>(m.ve + j0));
                const float4 a1 = __ldg(reinterpret_cast<const float4 *>(m.ve + j0 + 4));
                y[0] += vacc[0] * a0.x; y[1] += vacc[1] * a0.y; y[2] += vacc[2] * a0.z; y[3] += vacc[3] * a0.w;
                y[4] += vacc[4] * a1.x; y[5] += vacc[5] * a1.y; y[6] += vacc[6] * a1.z; y[7] += vacc[7] * a1.w;
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) y[k] += vacc[k];
            }
        }
    } else {  // EPI_VERA_E: out += acc * e
        if (m.v1) {
            const float4 a0 = __ldg(reinterpret_cast<const float4 *>(m.v1 + j0));
            const float4 a1 = __ldg(reinterpret_cast<const float4 *>(m.v1 + j0 + 4));
            y[0] = acc[0] * a0.x; y[1] = acc[1] * a0.y; y[2] = acc[2] * a0.z; y[3] = acc[3] * a0.w;
            y[4] = acc[4] * a1.x; y[5] = acc[5] * a1.y; y[6] = acc[6] * a1.z; y[7] = acc[7] * a1.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = acc[k];
        }
    }
    const bool add = g.epi == EPI_VERA_E;
    if (g.out_f32) {
        float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(g.out) + (size_t)m.out_row * g.ld_out + j0);
        float4 w0 = make_float4(y[0], y[1], y[2], y[3]), w1 = make_float4(y[4], y[5], y[6], y[7]);
        if (add) {
            const float4 p0 = o[0], p1 = o[1];
            w0.x += p0.x; w0.y += p0.y; w0.z += p0.z; w0.w += p0.w;
            w1.x += p1.x; w1.y += p1.y; w1.z += p1.z; w1.w += p1.w;
        }
        o[0] = w0;
        o[1] = w1;
    } else {
        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(g.out) + (size_t)m.out_row * g.ld_out + j0);
        if (add) {
            const uint4 prev = *o;
            const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&prev);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(q2[e]);
                y[2 * e] += f.x;
                y[2 * e + 1] += f.y;
            }
        }
        uint4 pk;
        __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
        for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
        *o = pk;
    }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// barrier of the 128 epilogue threads that also returns whether v held on all of them
__device__ __forceinline__ bool vs_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

// SO: the VeRA expand with its rows of out staged in shared memory (tokens on
// P, bf16; a separate instance, so that the other launches' code is unchanged)
template <int BN, bool TF32, bool SO>
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
    // tokens on P with an owned low-rank term (bf16): its expand runs on the
    // tensor cores as one extra K block per tile, from operands the epilogue
    // warps write after the ring: A (128 rows x 64 bytes), then B (BN rows)
    const bool lr_fused = g.tok_on_p && g.v != nullptr;
    uint8_t *lr_buf = smem + stages * STAGE_BYTES;
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(lr_buf + (lr_fused ? LR_A_BYTES + BN * 64 : 0));
    TokMeta *tmeta = reinterpret_cast<TokMeta *>(reinterpret_cast<uint8_t *>(ctrl) + CTRL_BYTES);
    // features on P: per-token metadata, then the tokens' v
    float *vtile = reinterpret_cast<float *>(tmeta + BN);
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
    // fused VeRA expand K blocks of this CTA: j = crank, crank + splits, ...
    const bool my_vera = g.vera_kb > crank;
    const int n_vera_ranks = g.vera_kb < splits ? g.vera_kb : splits;

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
        ptx::mbar_init(ptx::smem_u32(&ctrl->lrfull), 128);
        ctrl->abort = 0;
        for (int p = 0; p < 2; ++p) {
            ctrl->lr_steps[p] = 0;
            for (int j = 0; j < LR_KSTEPS; ++j) ctrl->lr_aid[p][j] = -2;
        }
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&g.mapP);
        ptx::prefetch_tmap(&g.mapQ);
        if (g.vera_kb) {
            ptx::prefetch_tmap(&g.mapVP);
            ptx::prefetch_tmap(&g.mapVQ);
        }
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
            if (g.p_base && !g.tok_on_p && splits > 0) {
                // the weights do not depend on earlier kernels: ask L2 for this
                // CTA's whole K range of its 128 rows now, so the ring below
                // finds them there instead of waiting on DRAM stage by stage
                const int prow0 = (tile0 % g.n_ft) * TILE_M;
                const long long off = (long long)kb0 * 128;
                long long want = (long long)(kb1 - kb0) * 128;
                if (off + want > g.p_pitch) want = g.p_pitch - off;   // ragged K tail stays inside the row
                const uint32_t bytes = want > 0 ? (uint32_t)(want & ~15ll) : 0u;
                const uint8_t *base = reinterpret_cast<const uint8_t *>(g.p_base) + off;
                for (int r = 0; bytes && r < TILE_M && prow0 + r < g.p_rows; ++r)
                    ptx::bulk_prefetch_l2(base + (size_t)(prow0 + r) * g.p_pitch, bytes);
            }
            for (int tile = tile0; tile < n_tiles; tile += tstep) {
                const int ft = tile % g.n_ft, tt = tile / g.n_ft;
                const int prow = g.tok_on_p ? tok_base + tt * TILE_M : ft * TILE_M;
                const int qrow = g.tok_on_p ? ft * BN : tok_base + tt * BN;
                const int nkb = (kb1 - kb0) + (my_vera ? (g.vera_kb - crank + splits - 1) / splits : 0);
                for (int it = 0; it < nkb; ++it) {
                    const bool vblk = it >= kb1 - kb0;
                    const int kc = vblk ? (crank + (it - (kb1 - kb0)) * splits) * KE : (kb0 + it) * KE;
                    const CUtensorMap *mP = vblk ? &g.mapVP : &g.mapP;
                    const CUtensorMap *mQ = vblk ? &g.mapVQ : &g.mapQ;
                    if (!wait_bar(ptx::smem_u32(&ctrl->empty[stage]), phase ^ 1, abort_flag)) goto prod_done;
                    const uint32_t fb = ptx::smem_u32(&ctrl->full[stage]);
                    const uint32_t sP = ptx::smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sQ = sP + TILE_M * 128;
                    ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    if (!g.tok_on_p) {
                        // P (weights) does not depend on earlier kernels: it is
                        // fetched before the grid dependency resolves.
                        ptx::tma_load_2d(sP, mP, kc, prow, fb);
                        ptx::tma_load_2d(sP + BOX_BYTES, mP, kc, prow + BOX_ROWS, fb);
                        if (!dep_done) { ptx::grid_dep_wait(); dep_done = true; }
#pragma unroll
                        for (int j = 0; j < BN / BOX_ROWS; ++j)
                            ptx::tma_load_2d(sQ + j * BOX_BYTES, mQ, kc, qrow + j * BOX_ROWS, fb);
                    } else {
                        if (!dep_done) { ptx::grid_dep_wait(); dep_done = true; }
                        ptx::tma_load_2d(sP, mP, kc, prow, fb);
                        ptx::tma_load_2d(sP + BOX_BYTES, mP, kc, prow + BOX_ROWS, fb);
#pragma unroll
                        for (int j = 0; j < BN / BOX_ROWS; ++j)
                            ptx::tma_load_2d(sQ + j * BOX_BYTES, mQ, kc, qrow + j * BOX_ROWS, fb);
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
            uint32_t lr_par = 0;
            for (int tile = tile0; tile < n_tiles; tile += tstep) {
                if (!wait_bar(ptx::smem_u32(&ctrl->tempty[acc]), acc_phase ^ 1, abort_flag)) goto mma_done;
                ptx::tc_fence_after();
                const int nb = kb1 - kb0;
                const int nkb = nb + (my_vera ? (g.vera_kb - crank + splits - 1) / splits : 0);
                for (int it = 0; it < nkb; ++it) {
                    const bool vblk = it >= nb;
                    // the fused VeRA product accumulates into the second buffer
                    const uint32_t d_tmem = tmem_base + (uint32_t)((vblk ? 1 : acc) * BN);
                    const bool first = vblk ? (it == nb) : (it == 0);
                    if (!wait_bar(ptx::smem_u32(&ctrl->full[stage]), phase, abort_flag)) goto mma_done;
                    ptx::tc_fence_after();
                    const uint32_t sP = ptx::smem_u32(smem + stage * STAGE_BYTES);
                    const uint64_t da = sw128_desc(sP);
                    const uint64_t db = sw128_desc(sP + TILE_M * 128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (!first || kk > 0) ? 1u : 0u;
                        if (TF32)
                            ptx::mma_tf32(d_tmem, da + 2 * kk, db + 2 * kk, IDESC, accum);
                        else
                            ptx::mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, IDESC, accum);
                    }
                    ptx::mma_commit(ptx::smem_u32(&ctrl->empty[stage]));
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
                if (lr_fused) {
                    // the owned low-rank expand of this tile, into the same
                    // accumulator (its rows are added before s is applied)
                    if (!wait_bar(ptx::smem_u32(&ctrl->lrfull), lr_par, abort_flag)) goto mma_done;
                    ptx::tc_fence_after();
                    const int steps = ctrl->lr_steps[lr_par];
                    const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                    const uint64_t da = sw64_desc(ptx::smem_u32(lr_buf));
                    const uint64_t db = sw64_desc(ptx::smem_u32(lr_buf + LR_A_BYTES));
                    for (int j = 0; j < steps && j < LR_KSTEPS; ++j)
                        ptx::mma_bf16(d_tmem, da + 2 * j, db + 2 * j, IDESC, 1u);
                    lr_par ^= 1u;
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
        const int et = threadIdx.x - 64;   // 0..127
        const int q = warp & 3;            // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;
        if (!g.tok_on_p) {
            // one token tile (n_tok <= BN): per-token metadata and the owned
            // low-rank intermediate go to shared memory while the K loop runs
            for (int t = et; t < BN; t += 128)
                if (t < n_tok) tmeta[t] = tok_meta(g, t, sorted_base);
            if (g.v) {
                const int R = g.lr_rmax;
                for (int e = et; e < BN * R; e += 128) {
                    const int t = e / R, c = e - t * R;
                    vtile[e] = t < n_tok ? g.v[(size_t)(sorted_base + t) * g.v_ld + c] : 0.f;
                }
            }
            epi_bar();
            // warm L2 with the epilogue's per-token operands of this CTA's items
            // while the K loop streams the weights
            {
                const int FR = TILE_M / splits, G8 = FR / 8;
                const int ft = tile0 % g.n_ft;
                const int nt = min(BN, n_tok);
                for (int item = et; item < nt * G8; item += 128) {
                    const int t = item / G8, fg = item - t * G8;
                    const int j0 = ft * TILE_M + crank * FR + fg * 8;
                    if (j0 >= g.n_feat) continue;
                    const TokMeta &m = tmeta[t];
                    if (m.v1) ptx::prefetch_l2(m.v1 + j0);
                    if (m.v2) ptx::prefetch_l2(m.v2 + j0);
                    if (m.ve) ptx::prefetch_l2(m.ve + j0);
                    if (m.B) {
                        const __nv_bfloat16 *B = reinterpret_cast<const __nv_bfloat16 *>(m.B) + j0;
                        for (int q = 0; q < m.rank; ++q) ptx::prefetch_l2(B + (size_t)q * g.n_feat);
                    }
                }
            }
        }
        int acc = 0;
        uint32_t acc_phase = 0;
        // tokens on P with an owned low-rank term: before each tile's
        // accumulator wait, the epilogue warps write that tile's low-rank
        // operands (the buffer is free: the previous tile's accumulator, which
        // includes its low-rank MMAs, is complete)
        const uint32_t lrfull = ptx::smem_u32(&ctrl->lrfull);
        uint32_t lr_par = 0;
        // VeRA expand, tokens on P, bf16 out: staged rows of out and e slices
        constexpr bool stage_out = SO && !TF32;
        uint8_t *obuf = reinterpret_cast<uint8_t *>(ctrl) + CTRL_BYTES;
        float *ebuf = reinterpret_cast<float *>(obuf + TILE_M * out_pitch(BN));
        const float *ew = nullptr;
        bool ok = true;            // this thread's wait of the previous tile succeeded
        for (int tile = tile0; tile < n_tiles; tile += tstep) {
            const int ft = tile % g.n_ft, tt = tile / g.n_ft;
            int i = 0;
            bool live = false;
            TokMeta rc;
            const float *vsrc = nullptr;
            if (lr_fused) {
                const int par = (int)lr_par;
                i = tt * TILE_M + row;
                live = i < n_tok;
                int a = -1, prev = -2;
                if (live) {
                    rc = tok_meta(g, i, sorted_base);
                    a = g.aid_s[sorted_base + i];
                    if (row > 0) prev = g.aid_s[sorted_base + i - 1];
                }
                const bool own = live && rc.B != nullptr;
                const bool mma_ok = own && rc.Bm != nullptr && rc.rank <= 16 * LR_KSTEPS;
                // k-steps in row order: the first row of each adapter in the
                // tile asks for ceil(rank / 16) of them
                const int need = (mma_ok && prev != a) ? (rc.rank + 15) / 16 : 0;
                int incl = need;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                if (lane == 31) ctrl->lr_wsum[par][q] = incl;
                // every thread is done with the previous tile, and every wait
                // of it succeeded
                if (!vs_all(ok)) break;
                if (et == 0) {
                    ctrl->lr_steps[par ^ 1] = 0;
                    for (int j = 0; j < LR_KSTEPS; ++j) ctrl->lr_aid[par ^ 1][j] = -2;
                }
                if (need > 0) {
                    int k0 = incl - need;
                    for (int w = 0; w < q; ++w) k0 += ctrl->lr_wsum[par][w];
                    if (k0 + need <= LR_KSTEPS) {
                        for (int j = k0; j < k0 + need; ++j) {
                            ctrl->lr_aid[par][j] = a;
                            ctrl->lr_k0[par][j] = k0;
                            ctrl->lr_rank[par][j] = rc.rank;
                            ctrl->lr_B[par][j] = rc.Bm;
                        }
                        atomicMax(&ctrl->lr_steps[par], k0 + need);
                    }
                }
                epi_bar();   // the tile's k-steps are assigned
                int k0 = -1;
                if (mma_ok)
                    for (int j = 0; j < LR_KSTEPS; ++j)
                        if (ctrl->lr_aid[par][j] == a) { k0 = j; break; }
                if (own && k0 < 0) vsrc = g.v + (size_t)(sorted_base + i) * g.v_ld;
                // A: this row's v (summed over the K chunks in chunk order,
                // rounded to bf16) in its adapter's k-steps, zeros elsewhere
                {
                    float vv[16 * LR_KSTEPS];
#pragma unroll
                    for (int c = 0; c < 16 * LR_KSTEPS; ++c) vv[c] = 0.f;
                    if (k0 >= 0) {
                        const float *src = g.v + (size_t)(sorted_base + i) * g.v_ld;
#pragma unroll
                        for (int c4 = 0; c4 < 4 * LR_KSTEPS; ++c4) {
                            const int qq = 4 * c4 - 16 * k0;
                            if (qq >= 0 && qq < rc.rank) {
                                float4 sum = __ldg(reinterpret_cast<const float4 *>(src + qq));
                                for (int s = 1; s < g.v_ks; ++s) {
                                    const float4 t = __ldg(reinterpret_cast<const float4 *>(src + s * g.v_kstride + qq));
                                    sum.x += t.x; sum.y += t.y; sum.z += t.z; sum.w += t.w;
                                }
                                vv[4 * c4] = sum.x;
                                vv[4 * c4 + 1] = qq + 1 < rc.rank ? sum.y : 0.f;
                                vv[4 * c4 + 2] = qq + 2 < rc.rank ? sum.z : 0.f;
                                vv[4 * c4 + 3] = qq + 3 < rc.rank ? sum.w : 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2 * LR_KSTEPS; ++u) {
                        uint4 pk;
                        __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                        for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(vv[8 * u + 2 * e], vv[8 * u + 2 * e + 1]);
                        *reinterpret_cast<uint4 *>(lr_buf + sw64_offset(row, u)) = pk;
                    }
                }
                // B: for features n of this tile, each k-step's 16 rank rows of
                // its adapter's B at column n (zeros past the rank, past the
                // features, and in k-steps no adapter took)
                for (int n = et; n < BN; n += 128) {
                    const int col = ft * BN + n;
#pragma unroll
                    for (int j = 0; j < LR_KSTEPS; ++j) {
                        const int aj = ctrl->lr_aid[par][j];
                        float bv[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) bv[e] = 0.f;
                        if (aj != -2 && col < g.n_feat) {
                            const __nv_bfloat16 *Bj = reinterpret_cast<const __nv_bfloat16 *>(ctrl->lr_B[par][j]);
                            const int q0 = 16 * (j - ctrl->lr_k0[par][j]);
                            const int rk = ctrl->lr_rank[par][j];
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                if (q0 + e < rk) bv[e] = __bfloat162float(Bj[(size_t)(q0 + e) * g.n_feat + col]);
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint4 pk;
                            __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                            for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(bv[8 * h + 2 * e], bv[8 * h + 2 * e + 1]);
                            *reinterpret_cast<uint4 *>(lr_buf + LR_A_BYTES + sw64_offset(n, 2 * j + h)) = pk;
                        }
                    }
                }
                // generic-proxy writes made visible to the tensor cores, then
                // the MMA issuer may read them
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                ptx::mbar_arrive(lrfull);
                lr_par ^= 1u;
                ok = wait_bar(ptx::smem_u32(&ctrl->tfull[acc]), acc_phase, abort_flag);
                if (!ok) continue;   // every thread learns of it at the next tile's vote
            } else if (stage_out) {
                // this warp's 32 rows of out at the tile's features, and the
                // e slice of its first row's adapter, copied to shared memory
                // while the accumulator forms (one row per warp instruction)
                i = tt * TILE_M + row;
                live = i < n_tok;
                if (live) rc = tok_meta(g, i, sorted_base);
                const int cols = min(BN, g.n_feat - ft * BN);
                const long long my_orow = live ? rc.out_row : 0;
                for (int r = 0; r < 32; ++r) {
                    const long long orow_r = __shfl_sync(0xffffffffu, my_orow, r);
                    const int live_r = __shfl_sync(0xffffffffu, live ? 1 : 0, r);
                    if (live_r && lane * 16 < cols * 2)
                        ptx::cp_async16(ptx::smem_u32(obuf + (q * 32 + r) * out_pitch(BN) + lane * 16),
                                        reinterpret_cast<const __nv_bfloat16 *>(g.out) + orow_r * g.ld_out +
                                            (size_t)ft * BN + lane * 8);
                }
                ew = reinterpret_cast<const float *>(__shfl_sync(
                    0xffffffffu, (unsigned long long)(live ? rc.v1 : nullptr), 0));
                if (ew)
                    for (int k = lane; k * 4 < cols; k += 32)
                        ptx::cp_async16(ptx::smem_u32(ebuf + q * BN + 4 * k), ew + (size_t)ft * BN + 4 * k);
                ptx::cp_async_commit();
                if (!wait_bar(ptx::smem_u32(&ctrl->tfull[acc]), acc_phase, abort_flag)) break;
                ptx::cp_async_wait_all();
                __syncwarp();
            } else {
                if (!wait_bar(ptx::smem_u32(&ctrl->tfull[acc]), acc_phase, abort_flag)) break;
            }
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const uint32_t tbv = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)BN;
            if (!g.tok_on_p) {
                // features on rows, tokens on columns.  The (partial) tile is
                // written as [token][128 features]: to shared memory when the
                // CTA owns all of K, else to this CTA's slot of the workspace
                // for the cluster's reduction through L2
                float *red = splits > 1 ? g.part + (size_t)blockIdx.x * g.part_stride
                                        : reinterpret_cast<float *>(smem);
                const int ld = splits > 1 ? TILE_M : RED_LD;
                float *redv = red + BN * ld;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    ptx::tmem_ld32(tb + c * 32, v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) red[(c * 32 + k) * ld + row] = v[k];
                    if (my_vera) {
                        ptx::tmem_ld32(tbv + c * 32, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) redv[(c * 32 + k) * ld + row] = v[k];
                    }
                }
            } else if (stage_out) {
                // out += acc * e on the staged rows, then the warp writes its
                // 32 rows back, one row per instruction
                const int cols = min(BN, g.n_feat - ft * BN);
                uint8_t *orow = obuf + row * out_pitch(BN);
                const bool e_sh = live && rc.v1 != nullptr && rc.v1 == ew;
                // y = acc * e + old for 32 features [32c, 32c + 32) of this row
                auto add_chunk = [&](int c, const float (&v)[32]) {
                    if (!live || c * 32 >= cols) return;
                    const float *ep = e_sh ? ebuf + q * BN + c * 32
                                           : (rc.v1 ? rc.v1 + (size_t)ft * BN + c * 32 : nullptr);
                    uint4 *op = reinterpret_cast<uint4 *>(orow + c * 64);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        float e8[8];
                        if (ep) {
                            const float4 a0 = e_sh ? reinterpret_cast<const float4 *>(ep)[2 * h]
                                                   : __ldg(reinterpret_cast<const float4 *>(ep) + 2 * h);
                            const float4 a1 = e_sh ? reinterpret_cast<const float4 *>(ep)[2 * h + 1]
                                                   : __ldg(reinterpret_cast<const float4 *>(ep) + 2 * h + 1);
                            e8[0] = a0.x; e8[1] = a0.y; e8[2] = a0.z; e8[3] = a0.w;
                            e8[4] = a1.x; e8[5] = a1.y; e8[6] = a1.z; e8[7] = a1.w;
                        } else {
#pragma unroll
                            for (int k = 0; k < 8; ++k) e8[k] = 1.f;
                        }
                        const uint4 prev = op[h];
                        const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&prev);
                        uint4 pk;
                        __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(q2[e]);
                            p2[e] = __floats2bfloat162_rn(v[8 * h + 2 * e] * e8[2 * e] + f.x,
                                                          v[8 * h + 2 * e + 1] * e8[2 * e + 1] + f.y);
                        }
                        op[h] = pk;
                    }
                };
                // two accumulator chunks in flight per wait
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 2) {
                    float v0[32], v1[32];
                    ptx::tmem_ld32x2(tb + c * 32, tb + (c + 1) * 32, v0, v1);
                    if (c + 2 == BN / 32) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[acc]));
                    }
                    add_chunk(c, v0);
                    add_chunk(c + 1, v1);
                }
                __syncwarp();
                const long long my_orow = live ? rc.out_row : 0;
                for (int r = 0; r < 32; ++r) {
                    const long long orow_r = __shfl_sync(0xffffffffu, my_orow, r);
                    const int live_r = __shfl_sync(0xffffffffu, live ? 1 : 0, r);
                    if (live_r && lane * 16 < cols * 2)
                        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(g.out) + orow_r * g.ld_out +
                                                   (size_t)ft * BN + lane * 8) =
                            *reinterpret_cast<const uint4 *>(obuf + (q * 32 + r) * out_pitch(BN) + lane * 16);
                }
                __syncwarp();   // the rows are read before the next tile's copies land
            } else {
                // tokens on rows, features on columns
                if (!lr_fused) {
                    i = tt * TILE_M + row;
                    live = i < n_tok;
                    if (live) rc = tok_meta(g, i, sorted_base);
                }
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
                    if (live && j0 < g.n_feat) emit32(g, rc, j0, v, vsrc);
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (stage_out) ptx::cp_async_wait_all();   // no copy in flight at exit
    }

    ptx::tc_fence_before();
    __syncthreads();

    if (!g.tok_on_p) {
        // ---- features-on-P epilogue: sum the cluster's K-split partial tiles
        // (written to the workspace before the cluster barrier, which orders
        // them at cluster scope), then apply the slots to items of (token,
        // 8 consecutive features)
        if (splits > 1) ptx::cluster_sync();
        int any_abort = 0;
        {
            int ab[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                ab[r] = r < splits ? (splits > 1 ? ptx::ld_dsmem_s32(ptx::mapa(ptx::smem_u32(&ctrl->abort), (uint32_t)r))
                                                 : ctrl->abort)
                                   : 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) any_abort |= ab[r];
        }
        // the peers' abort flags were the last reads of their shared memory
        if (splits > 1) ptx::cluster_arrive_relaxed();
        if (!any_abort && warp >= 2) {
            const int et = threadIdx.x - 64;
            const int FR = TILE_M / splits;   // feature rows finalised by this CTA
            const int G8 = FR / 8;            // 8-feature groups per token
            const int ft = tile0 % g.n_ft;
            const int R = g.lr_rmax;
            const int nt = min(BN, n_tok);
            const int ld = splits > 1 ? TILE_M : RED_LD;
            const float *base0 = splits > 1 ? g.part + (size_t)(blockIdx.x - crank) * g.part_stride
                                            : reinterpret_cast<const float *>(smem);
            const size_t vstride = (size_t)BN * ld;
#pragma unroll 1
            for (int item = et; item < nt * G8; item += 128) {
                const int t = item / G8, fg = item - t * G8;
                const int f0 = crank * FR + fg * 8;
                const int j0 = ft * TILE_M + f0;
                if (j0 >= g.n_feat) continue;
                const size_t off = (size_t)t * ld + f0;
                // partial tiles of the cluster are loaded four ranks at a time,
                // all loads of a batch before any add, so their latencies overlap
                float acc[8], vacc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) { acc[k] = 0.f; vacc[k] = 0.f; }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float4 pb[8], pv[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int r = h * 4 + u;
                        const float4 *src = reinterpret_cast<const float4 *>(base0 + (size_t)r * g.part_stride + off);
                        const float4 *srcv = reinterpret_cast<const float4 *>(base0 + (size_t)r * g.part_stride + off + vstride);
                        if (splits == 1) {
                            // the tile is in this CTA's shared memory
                            if (r == 0) { pb[0] = src[0]; pb[1] = src[1]; }
                            if (r < n_vera_ranks) { pv[2 * u] = srcv[0]; pv[2 * u + 1] = srcv[1]; }
                        } else {
                            // peers' slices in L2 (never cached in this SM's L1)
                            if (r < splits) { pb[2 * u] = __ldcg(src); pb[2 * u + 1] = __ldcg(src + 1); }
                            if (r < n_vera_ranks) { pv[2 * u] = __ldcg(srcv); pv[2 * u + 1] = __ldcg(srcv + 1); }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int r = h * 4 + u;
                        if (r < splits) {
                            acc[0] += pb[2 * u].x; acc[1] += pb[2 * u].y; acc[2] += pb[2 * u].z; acc[3] += pb[2 * u].w;
                            acc[4] += pb[2 * u + 1].x; acc[5] += pb[2 * u + 1].y; acc[6] += pb[2 * u + 1].z; acc[7] += pb[2 * u + 1].w;
                        }
                        if (r < n_vera_ranks) {
                            vacc[0] += pv[2 * u].x; vacc[1] += pv[2 * u].y; vacc[2] += pv[2 * u].z; vacc[3] += pv[2 * u].w;
                            vacc[4] += pv[2 * u + 1].x; vacc[5] += pv[2 * u + 1].y; vacc[6] += pv[2 * u + 1].z; vacc[7] += pv[2 * u + 1].w;
                        }
                    }
                }
                emit8(g, tmeta[t], vtile + t * R, j0, acc, vacc);
            }
        }
    }

    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, NCOLS);
    }
    if (threadIdx.x == 0 && ctrl->abort) atomicOr(g.status, STATUS_TIMEOUT);
    if (!g.tok_on_p && splits > 1) ptx::cluster_wait();
}

template <int BN, bool TF32, bool SO = false>
cudaError_t launch_one(const GemmArgs &g, const GemmPlan &p, cudaStream_t st, bool pdl) {
    static std::atomic<unsigned long long> attr_done{0};
    auto kern = gemm_tc_kernel<BN, TF32, SO>;
    {
        const cudaError_t e = allow_max_dynamic_smem(kern, attr_done);
        if (e != cudaSuccess) return e;
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

// Dynamic shared memory of one launch.  Tokens on P with an owned low-rank
// term (lr_rmax > 0): the tensor-core expand's operands follow the ring.
size_t gemm_smem_bytes(int bn, int stages, int lr_rmax, bool tok_on_p, bool stage_out = false) {
    const size_t stage_bytes = (size_t)TILE_M * 128 + (size_t)bn * 128;
    const size_t epi = tok_on_p ? (lr_rmax > 0 ? (size_t)LR_A_BYTES + (size_t)bn * 64 : 0)
                                : (size_t)bn * sizeof(TokMeta) + (size_t)bn * lr_rmax * sizeof(float);
    const size_t so = stage_out ? (size_t)TILE_M * out_pitch(bn) + (size_t)4 * bn * sizeof(float) : 0;
    return 1024 + (size_t)stages * stage_bytes + CTRL_BYTES + epi + so;
}

GemmPlan plan_gemm(int n_tok, int n_feat, int kblocks, bool tok_on_p, bool tf32, int num_sms, int lr_rmax,
                   bool stage_out) {
    GemmPlan p{};
    p.tf32 = tf32 ? 1 : 0;
    if (tok_on_p) {
        // prefill orientation: 128 tokens x 256 features, persistent tiles; a
        // narrow product (the VeRA shrink to the shared rank) takes 64-feature
        // tiles, so that more CTAs share its K loop
        p.bn = n_feat <= 256 ? 64 : 256;
        p.splits = 1;
        p.stages = 4;
        while (p.stages > 2 && gemm_smem_bytes(p.bn, p.stages, lr_rmax, true, stage_out) > GEMM_SMEM_MAX) --p.stages;
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
        // two CTAs of the 64-token tile share an SM: keep both within its shared memory
        while (p.bn == 64 && p.stages > 2 && 2 * (gemm_smem_bytes(p.bn, p.stages, lr_rmax, false) + 1024) > 228 * 1024)
            --p.stages;
        int s = 1;
        while (s < 8 && tiles * (s * 2) <= target && kblocks / (s * 2) >= 4) s *= 2;
        p.splits = s;
        p.grid = tiles * s;
    }
    if (p.grid < 1) p.grid = 1;
    p.smem = gemm_smem_bytes(p.bn, p.stages, lr_rmax, tok_on_p, tok_on_p && stage_out);
    return p;
}

cudaError_t launch_gemm(const GemmArgs &g, const GemmPlan &p, cudaStream_t st, bool pdl) {
    // the staged-output instance (its shared memory is in the plan) for the
    // VeRA expand of bf16 outputs with tokens on P
    const bool so = g.stage_out && g.tok_on_p && g.epi == EPI_VERA_E && !g.out_f32;
    if (p.tf32) {
        switch (p.bn) {
            case 64: return launch_one<64, true>(g, p, st, pdl);
            case 128: return launch_one<128, true>(g, p, st, pdl);
            default: return launch_one<256, true>(g, p, st, pdl);
        }
    }
    switch (p.bn) {
        case 64: return so ? launch_one<64, false, true>(g, p, st, pdl) : launch_one<64, false>(g, p, st, pdl);
        case 128: return launch_one<128, false>(g, p, st, pdl);
        default: return so ? launch_one<256, false, true>(g, p, st, pdl) : launch_one<256, false>(g, p, st, pdl);
    }
}

}  // namespace scute
