// Decode step: every projection of one batched call in one persistent launch.
//
// The adapted layer of the article "Scute: Exact Batched Serving for PEFT
// Adapters Beyond LoRA" (paper-daily.com), section "The big picture: six extra
// slots in the LoRA computation":
//     F_a(x) = ((x R_a) W) * s_a + b_a + (x A'_a) B'_a + (((x A_sh) * d_a) B_sh) * e_a
// with the slots already folded at load (section "Which slots can be merged at
// load?").  For a decode batch (n <= 128 tokens) the work of every layer of
// the call is one HBM stream of the base weights, so the launch is organised
// around that stream (section "Where is the cheapest place to compute the
// remaining slots?": the extra work is priced in bytes moved):
//
//   * prologue, on the epilogue warps of every CTA while the weights start to
//     stream: the ids are ordered by (method, adapter) in shared memory; the
//     token operand x' (x R_a for rotated rows, x otherwise, kept in token
//     order) is written per layer (a layer with no rotation adapter needs
//     none: its base tiles read x itself); the owned low-rank term runs per
//     adapter segment and group of 8 ranks: the shrink v = x A'_a, then at
//     once, by the same CTA, the expand b + v B'_a over every output feature
//     of the layer, into fp32 rows that the tiles' finishers read;
//   * VeRA shared shrink U = (x' A_sh) * d_a on tcgen05, cut into short
//     K-chunks that are the first work of many CTAs; a VeRA token is never
//     rotated, so the chunks read x itself and start at once, and U is written
//     right after the token operands, long before the base tiles reach their
//     VeRA blocks;
//   * base tiles D[128 features x BN tokens] = W^T x'^T on tcgen05 (TMA-fed,
//     TMEM accumulators), each tile's K loop followed by the VeRA expand
//     U B_sh as extra K blocks into a second accumulator; the 64-wide K blocks
//     of all tiles of all layers are split over the CTAs in contiguous ranges
//     (stream-K).  The CTA holding a tile's first block finishes it: the CTAs
//     sharing the tile publish their partial tiles, and the finisher adds them
//     in CTA order to its own accumulator and applies s, b + v B' and the VeRA
//     e in its epilogue.
//
// Waits between CTAs (token operand written, U written, v written) are
// counters in global memory, read with acquire loads and bounded in time; the
// launch is cooperative, so every CTA is resident.  Every mbarrier wait is
// bounded too; on expiry a CTA records STATUS_TIMEOUT, raises the launch-wide
// abort flag, drains what it issued, frees TMEM and returns.
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs, warps 2..9 run the prologue and then the epilogues.
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

constexpr int THREADS = 320;
constexpr int EPI_THREADS = 256;              // warps 2..9
constexpr int EPI_WARPS = EPI_THREADS / 32;
constexpr int TILE_M = 128;
constexpr int BOX_ROWS = 64;
constexpr int BOX_BYTES = BOX_ROWS * 128;
constexpr int P_BYTES = TILE_M * 128;
constexpr int MAX_STAGES = 8;
constexpr uint64_t WAIT_NS = 2000000000ull;   // 2 s per wait
constexpr int RED = TILE_M + 4;               // token-row stride of a transposed chunk (floats)
constexpr int XB_FLOATS = 2 * 32 * RED;       // main + VeRA chunk of 32 tokens
constexpr int NTOK = STEP_MAX_TOKENS;
constexpr int NCALL = STEP_MAX_CALLS;
constexpr int LR_Q = 8;                       // ranks per low-rank shrink item
constexpr int LR_ROWS = 2;                    // rows per pass of the shrink

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// f32 accumulator, bf16 A and B, both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Ctrl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t tfull[4];
    uint64_t tempty[4];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;          // this CTA gave up a wait
    int flag;           // broadcast among the epilogue warps
    int meta_call;      // call whose token metadata is staged (-1: none)
    int n_seg;
    int bad;
    int warp_tot[EPI_WARPS];
    int n_oft[NCALL], n_lrs[NCALL];
    int it0[NCALL + 1];   // first low-rank item of each call, in the order a.it_call
    int done[NCALL];      // low-rank items this CTA finished per call
};
constexpr int CTRL_BYTES = 512;
static_assert(sizeof(Ctrl) <= CTRL_BYTES, "control block");

// Per-token slots of one layer, as the epilogue uses them.
struct TokMeta {
    const float *s, *b, *ve, *vd;
    const __nv_bfloat16 *B;
    int rank;    // owned rank applied in the epilogue (0: none)
    int vera;    // the token takes the VeRA expand
};

struct Fixed {
    long long start[STEP_MAX_GRID + 1];   // stream-K range of each CTA
    uint32_t key[NTOK], skey[NTOK];
    int perm[NTOK];                       // sorted row -> token
    int tok_aid[NTOK];                    // token -> adapter (-1: base only)
    int tok_seg[NTOK];                    // token -> segment
    int seg_start[NTOK + 1], seg_aid[NTOK];
    const __nv_bfloat16 *segR[NCALL][NTOK];   // per call: transposed rotation of each segment (null: none)
    const __nv_bfloat16 *segA[NCALL][NTOK];   // per call: owned A' of each segment (null: none)
    uint8_t segRank[NCALL][NTOK];
    uint8_t oft_list[NCALL][NTOK];            // per call: segments with a rotation
    uint8_t lr_list[NCALL][NTOK];             // per call: segments with an owned term
    uint32_t oft_mask[NCALL][NTOK / 32];      // per call: tokens whose row is rotated
    TokMeta tmeta[NTOK];
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The same barrier as a vote: true when v holds in all 256 epilogue threads.
// A wait that some warps see end and others see give up must not split them
// (the split would leave both halves at different barriers for good), so the
// epilogue acts on the vote of every such wait.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&v)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

// Bounded wait on an mbarrier phase; gives up when the time limit passes or
// when this CTA or another one has given up.  The launch-wide abort flag lives
// in global memory and is read only every few microseconds, so that waiting
// warps do not keep one L2 line busy; with nap set the warp sleeps between
// polls (for waits that are not on the streaming path).
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      const int *gabort, bool honour_abort = true, bool nap = false) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint64_t next_global = t0 + 4000;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (nap) __nanosleep(128);
        if (honour_abort && *abort_flag) return false;
        const uint64_t now = ptx::globaltimer();
        if (honour_abort && now > next_global) {
            if (*reinterpret_cast<const volatile int *>(gabort)) {
                *abort_flag = 1;
                return false;
            }
            next_global = now + 4000;
        }
        if (now - t0 > WAIT_NS) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait until the counter at p reaches target (acquire).
__device__ __noinline__ bool wait_count(const int *p, int target, volatile int *abort_flag, const int *gabort) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if (*abort_flag || *reinterpret_cast<const volatile int *>(gabort)) {
            *abort_flag = 1;
            return false;
        }
        if (ptx::globaltimer() - t0 > WAIT_NS) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Non-blocking look at a counter (acquire).
__device__ __forceinline__ bool count_reached(const int *p, int target) { return ld_acquire(p) >= target; }

// ---------------------------------------------------------------- schedule
struct ULoc {      // one VeRA shrink unit: K blocks [kb0, kb1) of VeRA tile vt of call c
    int c, vt, kb0, kb1;
};
__device__ __forceinline__ ULoc ulocate(const StepArgs &a, int u) {
    int c = 0;
    while (c + 1 < a.n_calls && a.call[c + 1].vs_unit0 <= u) ++c;
    const StepCall &k = a.call[c];
    const int l = u - k.vs_unit0;
    ULoc r;
    r.c = c;
    r.vt = l / k.vs_chunks;
    const int ch = l - r.vt * k.vs_chunks;
    r.kb0 = ch * a.vs_ch;
    r.kb1 = min(k.kblocks, r.kb0 + a.vs_ch);
    return r;
}

struct MLoc {      // the main tile that holds stream-K block b
    int c, tile, kb, nkb;
    long long tb0;
};
__device__ __forceinline__ MLoc mlocate(const StepArgs &a, long long b) {
    int c = 0;
    while (c + 1 < a.n_calls && a.call[c + 1].blk0 <= b) ++c;
    const StepCall &k = a.call[c];
    const int mpt = k.kblocks + k.vkb;
    const long long l = b - k.blk0;
    MLoc r;
    r.c = c;
    r.tile = (int)(l / mpt);
    r.kb = (int)(l - (long long)r.tile * mpt);
    r.nkb = mpt;
    r.tb0 = k.blk0 + (long long)r.tile * mpt;
    return r;
}

// The CTA whose range holds main block b.
__device__ __forceinline__ int owner(const Fixed &fx, int G, long long b) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (fx.start[mid] <= b) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------- epilogue pieces
// Write this warp's half of a 128-row accumulator plane (TMEM columns
// [tcol, tcol + BN)) as rows of the partial tile [token][128] fp32 (tokens < n).
__device__ __forceinline__ void publish(uint32_t tcol, float *dst, int n, int BN, int row, int half) {
    const int per = BN / 64;   // 32-column chunks per warp
    for (int c = half * per; c < (half + 1) * per; ++c) {
        if (c * 32 >= n) break;   // uniform across the warp
        float v[32];
        ptx::tmem_ld32(tcol + c * 32, v);
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (c * 32 + k < n) dst[(size_t)(c * 32 + k) * TILE_M + row] = v[k];
    }
}

// Count this CTA's arrival at a shared tile; true for the last of n_ctr.
__device__ __forceinline__ bool arrive(int *cnt, int n_ctr, Ctrl *ctrl, int et) {
    __threadfence();
    epi_bar();
    if (et == 0) {
        const int old = atomicAdd(cnt, 1);
        const int last = old == n_ctr - 1;
        if (last) atomicExch(cnt, 0);
        ctrl->flag = last;
    }
    epi_bar();
    const bool last = ctrl->flag != 0;
    if (last) __threadfence();
    return last;
}

// Stage the per-token slots of call c (all epilogue threads).
__device__ void stage_meta(const StepArgs &a, int c, Fixed &fx, Ctrl *ctrl, int et) {
    if (ctrl->meta_call == c) return;
    epi_bar();
    const StepCall &k = a.call[c];
    for (int t = et; t < a.n; t += EPI_THREADS) {
        TokMeta m;
        m.s = m.b = m.ve = m.vd = nullptr;
        m.B = nullptr;
        m.rank = 0;
        m.vera = 0;
        const int aid = fx.tok_aid[t];
        if (aid >= 0) {
            const Slot &sl = k.slots[aid];
            // s placed in a separate pass: DoRA and (IA)^3 tokens leave it out
            // here, and DoRA expands with B' whose s is not folded in
            const int meth = a.method_tab[aid];
            const bool spass = (a.variant & VARIANT_S_PASS) && (meth == RANK_DORA || meth == RANK_IA3);
            m.s = spass ? nullptr : sl.s;
            m.b = sl.b;
            if (k.lr_rmax > 0 && sl.B && sl.rank > 0) {
                m.B = reinterpret_cast<const __nv_bfloat16 *>(spass && sl.Bu ? sl.Bu : sl.B);
                m.rank = sl.rank;
            }
            m.vd = sl.vd;
            if (k.vkb > 0 && sl.vd) {
                m.vera = 1;
                m.ve = sl.ve;
            }
        }
        fx.tmeta[t] = m;
    }
    if (et == 0) ctrl->meta_call = c;
    epi_bar();
}

__device__ __forceinline__ void ld_vec8(const float *p, bool ok, float fill, float (&v)[8]) {
    if (ok) {
        const float4 a0 = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 a1 = __ldg(reinterpret_cast<const float4 *>(p + 4));
        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w; v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = fill;
    }
}

// Add the partial rows [t][f0, f0+8) of one plane of a partial slot.
__device__ __forceinline__ void add_part(const float *src, float (&acc)[8]) {
    const float4 p0 = __ldcg(reinterpret_cast<const float4 *>(src));
    const float4 p1 = __ldcg(reinterpret_cast<const float4 *>(src + 4));
    acc[0] += p0.x; acc[1] += p0.y; acc[2] += p0.z; acc[3] += p0.w;
    acc[4] += p1.x; acc[5] += p1.y; acc[6] += p1.z; acc[7] += p1.w;
}

// x_i A_rows^T for up to LR_Q rows of A (each [d_in], bf16) and the sorted
// rows [r0, r1) (tokens perm[r]); emit(token, q, value) once per (row, q).
// Each of the 256 threads covers 8 consecutive k per pass; a warp reduces its
// 16 partial sums (2 rows x 8 ranks) with a transposing butterfly, and the 8
// warps' sums are added in a fixed order.
template <typename Emit>
__device__ void shrink256(const __nv_bfloat16 *x, int d_in, const int *perm, int r0, int r1,
                          const __nv_bfloat16 *Arows, int nq, float *red, int et, Emit emit) {
    const int lane = et & 31, w = et >> 5;
    for (int rc = r0; rc < r1; rc += LR_ROWS) {
        const int nr = min(LR_ROWS, r1 - rc);
        float v[LR_ROWS * LR_Q];
#pragma unroll
        for (int i = 0; i < LR_ROWS * LR_Q; ++i) v[i] = 0.f;
        const __nv_bfloat16 *xr[LR_ROWS];
#pragma unroll
        for (int r = 0; r < LR_ROWS; ++r) xr[r] = x + (size_t)perm[rc + (r < nr ? r : 0)] * d_in;
        // one pass of 8 k per thread per iteration; the next iteration's
        // operands are loaded while the current ones are multiplied, and the
        // loop stays rolled so that its code is short
        uint4 au[LR_Q], xu[LR_ROWS];
        auto load = [&](int k0) {
            const bool in = k0 < d_in;
#pragma unroll
            for (int q = 0; q < LR_Q; ++q)
                au[q] = (in && q < nq) ? *reinterpret_cast<const uint4 *>(Arows + (size_t)q * d_in + k0) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int r = 0; r < LR_ROWS; ++r)
                xu[r] = (in && r < nr) ? *reinterpret_cast<const uint4 *>(xr[r] + k0) : make_uint4(0u, 0u, 0u, 0u);
        };
        load(et * 8);
#pragma unroll 1
        for (int kk = et * 8; kk < d_in; kk += EPI_THREADS * 8) {
            uint4 ca[LR_Q], cx[LR_ROWS];
#pragma unroll
            for (int q = 0; q < LR_Q; ++q) ca[q] = au[q];
#pragma unroll
            for (int r = 0; r < LR_ROWS; ++r) cx[r] = xu[r];
            load(kk + EPI_THREADS * 8);
            float xv[LR_ROWS][8];
#pragma unroll
            for (int r = 0; r < LR_ROWS; ++r) unpack8(cx[r], xv[r]);
#pragma unroll
            for (int q = 0; q < LR_Q; ++q) {
                float av[8];
                unpack8(ca[q], av);
#pragma unroll
                for (int r = 0; r < LR_ROWS; ++r)
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[r * LR_Q + q] = fmaf(xv[r][e], av[e], v[r * LR_Q + q]);
            }
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
        if ((lane & 1) == 0) red[w * 16 + (lane >> 1)] = v[0];
        epi_bar();
        if (et < 16) {
            const int r = et / LR_Q, q = et % LR_Q;
            float s = 0.f;
#pragma unroll
            for (int ww = 0; ww < EPI_WARPS; ++ww) s += red[ww * 16 + et];
            if (r < nr && q < nq) emit(perm[rc + r], q, s);
        }
        epi_bar();
    }
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(THREADS, 1) step_kernel(const __grid_constant__ StepArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t *sbase = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int BN = a.bn, S = a.stages, G = a.grid, me = (int)blockIdx.x;
    const int STAGE = P_BYTES + BN * 128;
    // accumulator buffers (a base and a VeRA accumulator each): four when
    // they fit TMEM's 512 columns, so that the MMA can run up to four
    // segments ahead of the epilogue warps
    const int NB = BN <= 64 ? 4 : 2;
    const uint32_t NCOLS = (uint32_t)(2 * NB * BN);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(sbase + S * STAGE);
    Fixed &fx = *reinterpret_cast<Fixed *>(sbase + S * STAGE + CTRL_BYTES);
    float *xb = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(&fx) + sizeof(Fixed));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &ctrl->abort;
    int *sync = a.sync;
    const int *gabort = sync + SY_ABORT;
    const size_t SLOT = (size_t)2 * TILE_M * BN;   // floats per partial slot

    // ---- set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < NB; ++b) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->tfull[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->tempty[b]), EPI_WARPS);
        }
        ptx::mbar_init(ptx::smem_u32(&ctrl->drain), 1);
        ctrl->abort = 0;
        ctrl->meta_call = -1;
        ctrl->bad = 0;
        for (int c = 0; c < NCALL; ++c) ctrl->done[c] = 0;
        ptx::fence_mbar_init();
    }
    for (int i = threadIdx.x; i <= G; i += THREADS) fx.start[i] = a.start[i];
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctrl->tmem_base), NCOLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const long long ms = fx.start[me], mend = fx.start[me + 1];

    if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            for (int c = 0; c < a.n_calls; ++c) {
                ptx::prefetch_tmap(&a.call[c].mapW);
                ptx::prefetch_tmap(&a.call[c].mapXs);
                if (a.call[c].vs_x || a.call[c].xs_direct) ptx::prefetch_tmap(&a.call[c].mapX);
            }
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            // every weight box is read by exactly one CTA once: let it leave L2
            // first, ahead of the token operands, slots and partial tiles
            const uint64_t once = ptx::make_policy_evict_first();
            unsigned xs_ok = 0, u_ok = 0;
            for (int c = 0; c < a.n_calls; ++c)
                if (a.call[c].xs_direct) xs_ok |= 1u << c;   // read from x: nothing to wait for
            bool ok = true;
            // stages whose weight boxes are issued but whose token-operand
            // boxes wait until the prologue has written that call's x'
            int pend_n = 0, pend_head = 0;
            uint32_t pend_sQ[MAX_STAGES], pend_fb[MAX_STAGES];
            int pend_kc[MAX_STAGES], pend_c[MAX_STAGES];
            auto issue_q = [&](uint32_t sQ, uint32_t fb, const CUtensorMap *mq, int kc) {
                for (int j = 0; j < BN / BOX_ROWS; ++j) ptx::tma_load_2d(sQ + j * BOX_BYTES, mq, kc, j * BOX_ROWS, fb);
            };
            auto xs_ready = [&](int c, bool block) -> bool {
                if ((xs_ok >> c) & 1u) return true;
                const int target = a.grid + a.hold;   // every CTA adds one per call
                if (block) {
                    if (!wait_count(sync + SY_XS + c, target, abort_flag, gabort)) return false;
                } else if (!count_reached(sync + SY_XS + c, target)) {
                    return false;
                }
                fence_proxy_async_global();
                xs_ok |= 1u << c;
                return true;
            };
            // issue pending token boxes in order; with block, wait for them
            auto flush = [&](bool block) -> bool {
                while (pend_n > 0) {
                    const int i = pend_head;
                    if (!xs_ready(pend_c[i], block)) {
                        if (!block) return true;
                        // gave up: issue them anyway (in bounds) so that every
                        // barrier completes and the copies can be drained
                        while (pend_n > 0) {
                            const int j = pend_head;
                            issue_q(pend_sQ[j], pend_fb[j], &a.call[pend_c[j]].mapXs, pend_kc[j]);
                            pend_head = (pend_head + 1) % MAX_STAGES;
                            --pend_n;
                        }
                        return false;
                    }
                    issue_q(pend_sQ[i], pend_fb[i], &a.call[pend_c[i]].mapXs, pend_kc[i]);
                    pend_head = (pend_head + 1) % MAX_STAGES;
                    --pend_n;
                }
                return true;
            };
            // one stage: P rows [prow, prow + 128) and the token operand, both at K offset kc
            auto issue = [&](const CUtensorMap *mp, int prow, const CUtensorMap *mq, int kc, int c, bool xs_dep) -> bool {
                if (pend_n == S && !flush(true)) return false;
                if (!wait_bar(ptx::smem_u32(&ctrl->empty[stage]), phase ^ 1, abort_flag, gabort)) return false;
                const uint32_t fb = ptx::smem_u32(&ctrl->full[stage]);
                const uint32_t sP = ptx::smem_u32(sbase + stage * STAGE);
                const uint32_t sQ = sP + P_BYTES;
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)STAGE);
                ptx::tma_load_2d_hint(sP, mp, kc, prow, fb, once);
                ptx::tma_load_2d_hint(sP + BOX_BYTES, mp, kc, prow + BOX_ROWS, fb, once);
                if (!xs_dep) {
                    issue_q(sQ, fb, mq, kc);
                } else {
                    flush(false);
                    if (pend_n == 0 && xs_ready(c, false)) {
                        issue_q(sQ, fb, mq, kc);
                    } else {
                        const int i = (pend_head + pend_n) % MAX_STAGES;
                        pend_sQ[i] = sQ;
                        pend_fb[i] = fb;
                        pend_kc[i] = kc;
                        pend_c[i] = c;
                        ++pend_n;
                    }
                }
                ++issued;
                if (++stage == S) { stage = 0; phase ^= 1; }
                return true;
            };
            for (int u = me; ok && u < a.n_units; u += G) {
                const ULoc U = ulocate(a, u);
                const StepCall &k = a.call[U.c];
                for (int kb = U.kb0; ok && kb < U.kb1; ++kb)
                    ok = k.vs_x ? issue(&k.mapAsh, U.vt * TILE_M, &k.mapX, kb * 64, U.c, false)
                                : issue(&k.mapAsh, U.vt * TILE_M, &k.mapXs, kb * 64, U.c, true);
            }
            const uint32_t s0 = ptx::smem_u32(sbase);
            for (long long b = ms; ok && b < mend;) {
                const MLoc L = mlocate(a, b);
                const StepCall &k = a.call[L.c];
                const long long se = min(mend, L.tb0 + L.nkb);
                int kb = L.kb;
                const long long bm = min(se, L.tb0 + (long long)k.kblocks);   // end of the main blocks
                while (ok && b < se) {
                    if (b < bm && pend_n == 0 && xs_ready(L.c, false)) {
                        // steady state: the call's x' is written and nothing
                        // waits, so the segment's main blocks take a short path
                        const CUtensorMap *mW = &k.mapW, *mQ = k.xs_direct ? &k.mapX : &k.mapXs;
                        const int prow = L.tile * TILE_M;
                        for (; b < bm; ++b, ++kb) {
                            const uint32_t eb = ptx::smem_u32(&ctrl->empty[stage]);
                            if (!ptx::mbar_try_wait(eb, phase ^ 1) && !wait_bar(eb, phase ^ 1, abort_flag, gabort)) {
                                ok = false;
                                break;
                            }
                            const uint32_t fb = ptx::smem_u32(&ctrl->full[stage]);
                            const uint32_t sP = s0 + (uint32_t)(stage * STAGE);
                            ptx::mbar_arrive_expect_tx(fb, (uint32_t)STAGE);
                            ptx::tma_load_2d_hint(sP, mW, kb * 64, prow, fb, once);
                            ptx::tma_load_2d_hint(sP + BOX_BYTES, mW, kb * 64, prow + BOX_ROWS, fb, once);
                            for (int j = 0; j < BN / BOX_ROWS; ++j)
                                ptx::tma_load_2d(sP + P_BYTES + j * BOX_BYTES, mQ, kb * 64, j * BOX_ROWS, fb);
                            ++issued;
                            if (++stage == S) { stage = 0; phase ^= 1; }
                        }
                        continue;
                    }
                    // one block the general way (token operand not yet written,
                    // stages pending, or a VeRA block); the short path is tried
                    // again before the next one
                    const bool vb = kb >= k.kblocks;
                    if (vb && !((u_ok >> L.c) & 1u)) {
                        // this CTA's own pending stages may be what U waits for
                        ok = flush(true) && wait_count(sync + SY_U + L.c, k.n_vt, abort_flag, gabort);
                        if (!ok) break;
                        fence_proxy_async_global();
                        u_ok |= 1u << L.c;
                    }
                    ok = vb ? issue(&k.mapBsh, L.tile * TILE_M, &k.mapU, (kb - k.kblocks) * 64, L.c, false)
                            : issue(&k.mapW, L.tile * TILE_M, k.xs_direct ? &k.mapX : &k.mapXs, kb * 64, L.c,
                                    !k.xs_direct);
                    ++b;
                    ++kb;
                }
            }
            flush(true);
            // every issued copy must have landed before the CTA may exit
            const int m_max = issued < S ? (int)issued : S;
            for (int m = 1; m <= m_max; ++m) {
                const int s = (stage - m + S) % S;
                const uint32_t ph = (s < stage) ? phase : (phase ^ 1);
                wait_bar(ptx::smem_u32(&ctrl->full[s]), ph, abort_flag, gabort, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0) {
            const uint32_t IDESC = idesc_bf16(TILE_M, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, bph = 0;
            bool ok = true;
            // one segment: nblk K blocks starting at kb_first; blocks at or
            // beyond kmain go to the second (VeRA) accumulator of the buffer
            auto segment = [&](int nblk, int kb_first, int kmain) -> bool {
                if (!wait_bar(ptx::smem_u32(&ctrl->tempty[buf]), bph ^ 1, abort_flag, gabort)) return false;
                ptx::tc_fence_after();
                bool fm = true, fv = true;
                for (int i = 0; i < nblk; ++i) {
                    const bool vb = kb_first + i >= kmain;
                    if (!wait_bar(ptx::smem_u32(&ctrl->full[stage]), phase, abort_flag, gabort)) return false;
                    ptx::tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(buf * 2 * BN + (vb ? BN : 0));
                    const uint32_t sP = ptx::smem_u32(sbase + stage * STAGE);
                    const uint64_t da = sw128_desc(sP), db = sw128_desc(sP + P_BYTES);
                    const bool first = vb ? fv : fm;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(d, da + 2 * kk, db + 2 * kk, IDESC, (kk > 0 || !first) ? 1u : 0u);
                    if (vb) fv = false;
                    else fm = false;
                    ptx::mma_commit(ptx::smem_u32(&ctrl->empty[stage]));
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                ptx::mma_commit(ptx::smem_u32(&ctrl->tfull[buf]));
                if (++buf == NB) { buf = 0; bph ^= 1; }
                return true;
            };
            for (int u = me; ok && u < a.n_units; u += G) {
                const ULoc U = ulocate(a, u);
                ok = segment(U.kb1 - U.kb0, U.kb0, 1 << 30);
            }
            for (long long b = ms; ok && b < mend;) {
                const MLoc L = mlocate(a, b);
                const long long se = min(mend, L.tb0 + L.nkb);
                ok = segment((int)(se - b), L.kb, a.call[L.c].kblocks);
                b = se;
            }
            // all MMAs issued here must finish before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&ctrl->drain));
            wait_bar(ptx::smem_u32(&ctrl->drain), 0, abort_flag, gabort, false);
        }
        __syncwarp();
    } else {
        // ================================================= prologue, then epilogues
        const int et = threadIdx.x - 64;   // 0..255
        const int ew = et >> 5;            // epilogue warp 0..7
        const int q4 = warp & 3;           // TMEM lane quadrant this warp may read
        const int half = ew >> 2;          // which half of the columns (or planes) it drains
        const int row = q4 * 32 + lane;
        const int n = a.n;
        const uint32_t A = (uint32_t)a.A;

        // ---- order the ids: key = (method, adapter), ties in token order
        {
            const uint32_t base_key = (uint32_t)RANK_BASE * A;
            if (et < n) {
                const int id = a.ids[et];
                int m = -1;
                if (id >= 0 && id < a.A) m = a.method_tab[id];
                if (m < 0 && id != -1) ctrl->bad = 1;
                fx.tok_aid[et] = m >= 0 ? id : -1;
                fx.key[et] = m >= 0 ? (uint32_t)m * A + (uint32_t)id : base_key;
            }
            epi_bar();
            if (et < n) {
                const uint32_t kt = fx.key[et];
                int r = 0;
                for (int u = 0; u < n; ++u) {
                    const uint32_t ku = fx.key[u];
                    r += (ku < kt) || (ku == kt && u < et);
                }
                fx.perm[r] = et;
                fx.skey[r] = kt;
            }
            epi_bar();
            const bool head = et < n && (et == 0 || fx.skey[et] != fx.skey[et - 1]);
            const int incl = warp_incl_scan(head ? 1 : 0);
            if (lane == 31) ctrl->warp_tot[ew] = incl;
            epi_bar();
            int off = 0, tot = 0;
            for (int w = 0; w < EPI_WARPS; ++w) {
                if (w < ew) off += ctrl->warp_tot[w];
                tot += ctrl->warp_tot[w];
            }
            if (et < n) {
                const int s = off + incl - 1;   // segment of sorted row et
                fx.tok_seg[fx.perm[et]] = s;
                if (head) {
                    const uint32_t k = fx.skey[et];
                    const int rank = (int)(k / A);
                    fx.seg_start[s] = et;
                    fx.seg_aid[s] = rank >= RANK_BASE ? -1 : (int)(k - (uint32_t)rank * A);
                }
            }
            if (et == 0) {
                fx.seg_start[tot] = n;
                ctrl->n_seg = tot;
                if (me == 0 && ctrl->bad) atomicOr(a.status, STATUS_BAD_ADAPTER);
            }
            epi_bar();
        }
        // ---- every call's slots per segment, fetched in one round
        {
            const int n_seg = ctrl->n_seg;
            constexpr int PER = NCALL * NTOK / EPI_THREADS;
            const __nv_bfloat16 *R[PER], *Ao[PER];
            int rk[PER];
            // every slot load of this thread is issued before any is used
#pragma unroll
            for (int r = 0; r < PER; ++r) {
                const int e = et + r * EPI_THREADS, c = e / NTOK, s = e - c * NTOK;
                const int aid = (c < a.n_calls && s < n_seg) ? fx.seg_aid[s] : -1;
                R[r] = Ao[r] = nullptr;
                rk[r] = 0;
                if (aid >= 0) {
                    const StepCall &k = a.call[c];
                    const Slot &sl = k.slots[aid];
                    // rotation placed in a separate pass: x is already rotated
                    R[r] = (a.variant & VARIANT_OFT_PASS) ? nullptr : reinterpret_cast<const __nv_bfloat16 *>(sl.Rt);
                    if (sl.A && sl.rank > 0 && k.lr_rmax > 0) {
                        Ao[r] = reinterpret_cast<const __nv_bfloat16 *>(sl.A);
                        rk[r] = sl.rank;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < PER; ++r) {
                const int e = et + r * EPI_THREADS, c = e / NTOK, s = e - c * NTOK;
                if (c >= a.n_calls || s >= n_seg) continue;
                fx.segR[c][s] = R[r];
                fx.segA[c][s] = Ao[r];
                fx.segRank[c][s] = (uint8_t)rk[r];
            }
            epi_bar();
            if (ew < a.n_calls) {
                // warp ew lists call ew's rotated and owned-term segments and
                // marks its rotated tokens
                const int c = ew;
                const uint32_t lt = (1u << lane) - 1u;
                int no = 0, nl = 0;
                for (int s0 = 0; s0 < n_seg; s0 += 32) {
                    const int s = s0 + lane;
                    const bool o = s < n_seg && fx.segR[c][s] != nullptr;
                    const bool l = s < n_seg && fx.segA[c][s] != nullptr;
                    const uint32_t mo = __ballot_sync(0xffffffffu, o), ml = __ballot_sync(0xffffffffu, l);
                    if (o) fx.oft_list[c][no + __popc(mo & lt)] = (uint8_t)s;
                    if (l) fx.lr_list[c][nl + __popc(ml & lt)] = (uint8_t)s;
                    no += __popc(mo);
                    nl += __popc(ml);
                }
                for (int t0 = 0; t0 < NTOK; t0 += 32) {
                    const int t = t0 + lane;
                    const bool rot = t < n && fx.segR[c][fx.tok_seg[t]] != nullptr;
                    const uint32_t m = __ballot_sync(0xffffffffu, rot);
                    if (lane == 0) fx.oft_mask[c][t0 / 32] = m;
                }
                if (lane == 0) {
                    ctrl->n_oft[c] = no;
                    ctrl->n_lrs[c] = nl;
                }
            }
            epi_bar();
            if (et == 0) {
                // the batch's low-rank items: (segment, group of 8 ranks) of
                // every call with owned terms, in the host's order of the calls
                // (most work per item first); a.it_ng: rank groups per segment
                int acc = 0;
                ctrl->it0[0] = 0;
#pragma unroll
                for (int o = 0; o < NCALL; ++o) {
                    if (o < a.n_calls) acc += ctrl->n_lrs[a.it_call[o]] * a.it_ng[o];
                    ctrl->it0[o + 1] = acc;
                }
            }
            epi_bar();
        }

        int buf = 0;
        uint32_t bph = 0;
        bool ok = true;
        const uint32_t tq = tmem + ((uint32_t)(q4 * 32) << 16);
        float *xbm = xb, *xbv = xb + 32 * RED;
        // VeRA shrink unit u (a CTA has at most one; it is the first use of the
        // TMEM buffers): publish the partial sums, or, arriving last, write U
        auto unit_epi = [&](int u) -> bool {
            const ULoc U = ulocate(a, u);
            const StepCall &k = a.call[U.c];
            if (!epi_all(wait_bar(ptx::smem_u32(&ctrl->tfull[buf]), bph, abort_flag, gabort, true, true))) return false;
            ptx::tc_fence_after();
            const uint32_t tcol = tq + (uint32_t)(buf * 2 * BN);
            const int nctr = k.vs_chunks;
            const int u0 = k.vs_unit0 + U.vt * nctr;
            bool last = true;
            if (nctr > 1) {
                publish(tcol, a.part + (size_t)u * SLOT, n, BN, row, half);
                last = arrive(sync + SY_VTILE + U.c * STEP_MAX_VTILES + U.vt, nctr, ctrl, et);
            }
            if (last) {
                // U[t][q] = (x' A_sh)[t][q] * d_a(t)[q] for VeRA tokens, 0 otherwise
                stage_meta(a, U.c, fx, ctrl, et);
                const int r0 = U.vt * TILE_M;
                __nv_bfloat16 *Ub = reinterpret_cast<__nv_bfloat16 *>(k.U);
                for (int c32 = 0; c32 * 32 < n; ++c32) {
                    // a lone contributor's tile comes from TMEM; otherwise every
                    // published partial is summed in unit order, this CTA's too,
                    // so the result does not depend on which CTA finished last
                    if (half == 0 && nctr == 1) {
                        float v[32];
                        ptx::tmem_ld32(tcol + c32 * 32, v);
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) xbm[kk * RED + row] = v[kk];
                    }
                    epi_bar();
                    int t[2], q0[2], g[2], kk[2];
                    bool live[2];
                    float acc[2][8];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const int it = et + p * EPI_THREADS;
                        kk[p] = it >> 4;
                        g[p] = it & 15;
                        t[p] = c32 * 32 + kk[p];
                        q0[p] = r0 + g[p] * 8;
                        live[p] = t[p] < n && q0[p] < k.krv;
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[p][e] = nctr == 1 ? xbm[kk[p] * RED + g[p] * 8 + e] : 0.f;
                    }
#pragma unroll 4
                    for (int j = 0; j < (nctr > 1 ? nctr : 0); ++j) {
                        const float *src = a.part + (size_t)(u0 + j) * SLOT;
#pragma unroll
                        for (int p = 0; p < 2; ++p)
                            if (live[p]) add_part(src + (size_t)t[p] * TILE_M + g[p] * 8, acc[p]);
                    }
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        if (!live[p]) continue;
                        const float *vd = fx.tmeta[t[p]].vd;
                        uint4 pk;
                        __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
                        if (vd && q0[p] < k.rv) {
                            float d8[8];
                            ld_vec8(vd + q0[p], true, 0.f, d8);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                p2[e] = __floats2bfloat162_rn(acc[p][2 * e] * d8[2 * e], acc[p][2 * e + 1] * d8[2 * e + 1]);
                        } else {
                            pk = make_uint4(0u, 0u, 0u, 0u);
                        }
                        *reinterpret_cast<uint4 *>(Ub + (size_t)t[p] * k.krv + q0[p]) = pk;
                    }
                    epi_bar();
                }
                fence_proxy_async_global();
                __threadfence();
                epi_bar();
                if (et == 0) atomicAdd(sync + SY_U + U.c, 1);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[buf]));
            if (++buf == NB) { buf = 0; bph ^= 1; }
            return true;
        };

        // ---- token operands x' of every call, in warp-sized units spread
        // over all epilogue warps of the launch: copies of 8 unrotated rows x
        // 256 columns, then rotations of one 32x32 block of one rotated
        // segment (lane l reads row l of the transposed block; the rows'
        // inputs arrive by shuffle; the next unit's operands are loaded while
        // the current one is computed).  Each CTA then adds one per call.
        {
            const int W = G * EPI_WARPS, gw = me * EPI_WARPS + ew;
            int ubase = 0;
            for (int c = 0; c < a.n_calls; ++c) {
                const StepCall &k = a.call[c];
                if (k.xs_direct) continue;   // its base tiles read x itself
                const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(k.x);
                __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(k.xs);
                const int ccols = (k.d_in + 255) / 256, units = ccols * ((n + 7) / 8);
#pragma unroll 1
                for (int u = ((gw - ubase) % W + W) % W; u < units; u += W) {
                    const int rg = u / ccols, cc = u - rg * ccols;
                    const int col = cc * 256 + lane * 8;
                    if (col >= k.d_in) continue;
                    uint4 buf[8];
                    bool live[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int t = rg * 8 + r;
                        live[r] = t < n && !((fx.oft_mask[c][t >> 5] >> (t & 31)) & 1u);
                        if (live[r]) buf[r] = *reinterpret_cast<const uint4 *>(x + (size_t)t * k.d_in + col);
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int t = rg * 8 + r;
                        if (live[r]) *reinterpret_cast<uint4 *>(xs + (size_t)t * k.kdim + col) = buf[r];
                    }
                }
                ubase += units;
            }
            // rotation units of every call, one sequence in call order; a warp
            // takes four of its units at a time (whichever calls they belong
            // to) and issues every load of the four before computing any
            int rbase[NCALL + 1];
            rbase[0] = 0;
            for (int c = 0; c < NCALL; ++c)
                rbase[c + 1] = rbase[c] + (c < a.n_calls ? ctrl->n_oft[c] * (a.call[c].d_in / OFT_BLK) : 0);
            const int rtot = rbase[NCALL];
#pragma unroll 1
            for (int g0 = gw; g0 < rtot; g0 += 4 * W) {
                uint4 rq[4][4];
                float xv[4][4];
                int blk[4], r0[4], r1[4], ci[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int g = g0 + i * W;
                    r0[i] = r1[i] = blk[i] = ci[i] = 0;
                    if (g < rtot) {
                        int c = 0;
                        while (g >= rbase[c + 1]) ++c;
                        ci[i] = c;
                        const int nblk = a.call[c].d_in / OFT_BLK;
                        const int uu = g - rbase[c], s_ord = uu / nblk;
                        blk[i] = uu - s_ord * nblk;
                        const int seg = fx.oft_list[c][s_ord];
                        r0[i] = fx.seg_start[seg];
                        r1[i] = fx.seg_start[seg + 1];
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            fx.segR[c][seg] + (size_t)blk[i] * OFT_BLK * OFT_BLK + lane * OFT_BLK);
#pragma unroll
                        for (int q = 0; q < 4; ++q) rq[i][q] = src[q];
                    }
                    const StepCall &k = a.call[ci[i]];
                    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(k.x);
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
                        xv[i][rr] = r0[i] + rr < r1[i]
                                        ? __bfloat162float(x[(size_t)fx.perm[r0[i] + rr] * k.d_in + blk[i] * OFT_BLK + lane])
                                        : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (r0[i] >= r1[i]) continue;   // uniform across the warp
                    const StepCall &k = a.call[ci[i]];
                    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(k.x);
                    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(k.xs);
                    float rc[OFT_BLK];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float f8[8];
                        unpack8(rq[i][q], f8);
#pragma unroll
                        for (int e = 0; e < 8; ++e) rc[q * 8 + e] = f8[e];
                    }
#pragma unroll 1
                    for (int r = r0[i]; r < r1[i]; ++r) {
                        const int rr = r - r0[i];
                        const float xr = rr == 0 ? xv[i][0] : rr == 1 ? xv[i][1] : rr == 2 ? xv[i][2] : rr == 3 ? xv[i][3]
                                       : __bfloat162float(x[(size_t)fx.perm[r] * k.d_in + blk[i] * OFT_BLK + lane]);
                        float acc = 0.f;
#pragma unroll
                        for (int m = 0; m < OFT_BLK; ++m) acc = fmaf(__shfl_sync(0xffffffffu, xr, m), rc[m], acc);
                        xs[(size_t)fx.perm[r] * k.kdim + blk[i] * OFT_BLK + lane] = __float2bfloat16_rn(acc);
                    }
                }
            }
            fence_proxy_async_global();
            __threadfence();
            epi_bar();
            if (et == 0)
                for (int c = 0; c < a.n_calls; ++c) atomicAdd(sync + SY_XS + c, 1);
        }

        // ---- the VeRA shrink unit of this CTA, if any: U is written before
        // the low-rank items, so that the tiles' VeRA blocks wait little
        for (int u = me; ok && u < a.n_units; u += G) ok = unit_epi(u);

        // ---- owned low-rank items (CTA-sized): ranks [q0, q0 + 8) of one
        // adapter segment.  The shrink v = x A' of the segment's rows goes to
        // shared memory; the expand then runs at once over every output
        // feature of the layer: plane g = q0 / 8 of the call's rows gets
        // (b, for g = 0) + sum over those ranks of v_q B'_q, so that the
        // finishers read b + v B' as the sum of the token's planes, in order.
        float *red = xb;                        // shrink reduction scratch
        float *vloc = xb + EPI_WARPS * 32;      // [token][8] v of the current item
        // Items are dealt round-robin from the last CTA down: the first CTAs
        // hold the VeRA shrink units, whose epilogues come first.
        const int n_it = ctrl->it0[a.n_calls];
        for (int it = G - 1 - me; it < n_it; it += G) {
            int o = 0;
            while (it >= ctrl->it0[o + 1]) ++o;
            const int c = a.it_call[o];
            const int kk = it - ctrl->it0[o];
            const StepCall &k = a.call[c];
            // the low-rank term acts on x, not on x R (x0: the caller's x even
            // when the token operand comes from a separately rotated copy)
            const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(k.x0);
            const int ng = (k.lr_rmax + LR_Q - 1) / LR_Q;
            const int s_ord = kk / ng, qg = kk - s_ord * ng;   // s_ord < n_lrs[c] by construction
            {
                const int seg = fx.lr_list[c][s_ord];
                const int r0 = fx.seg_start[seg], r1 = fx.seg_start[seg + 1];
                const int rk = fx.segRank[c][seg];
                const int q0 = qg * LR_Q;
                if (q0 < rk) {
                    const int nq = min(LR_Q, rk - q0);
                    shrink256(x, k.d_in, fx.perm, r0, r1, fx.segA[c][seg] + (size_t)q0 * k.d_in, nq, red, et,
                              [&](int t, int q, float v) { vloc[t * LR_Q + q] = v; });
                    // (shrink256 ends at a barrier: every v of the item is in vloc)
                    stage_meta(a, c, fx, ctrl, et);
                    const TokMeta &m = fx.tmeta[fx.perm[r0]];   // the segment's adapter
                    float *plane = k.pre + (size_t)qg * NTOK * k.d_out;
#pragma unroll 1
                    for (int f = et * 8; f < k.d_out; f += EPI_THREADS * 8) {
                        uint4 bq[LR_Q];
#pragma unroll
                        for (int q = 0; q < LR_Q; ++q)
                            if (q < nq) bq[q] = __ldg(reinterpret_cast<const uint4 *>(m.B + f + (size_t)(q0 + q) * k.d_out));
                        float bb[8];
                        ld_vec8(m.b + f, qg == 0 && m.b != nullptr, 0.f, bb);
#pragma unroll 1
                        for (int r = r0; r < r1; ++r) {
                            const int t = fx.perm[r];
                            float y[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) y[e] = bb[e];
#pragma unroll
                            for (int q = 0; q < LR_Q; ++q) {
                                if (q < nq) {
                                    float bf[8];
                                    unpack8(bq[q], bf);
                                    const float vq = vloc[t * LR_Q + q];
#pragma unroll
                                    for (int e = 0; e < 8; ++e) y[e] = fmaf(vq, bf[e], y[e]);
                                }
                            }
                            float4 *dp = reinterpret_cast<float4 *>(plane + (size_t)t * k.d_out + f);
                            dp[0] = make_float4(y[0], y[1], y[2], y[3]);
                            dp[1] = make_float4(y[4], y[5], y[6], y[7]);
                        }
                    }
                    epi_bar();   // vloc is rewritten by the next item
                }
            }
            if (et == 0) ++ctrl->done[c];
        }
        // completed low-rank items are published once per CTA: every thread's
        // writes made visible, then one counter add per call
        __threadfence();
        epi_bar();
        if (et == 0)
            for (int c = 0; c < a.n_calls; ++c)
                if (ctrl->done[c]) atomicAdd(sync + SY_LR + c, ctrl->done[c]);
        epi_bar();

        // ---- epilogues, one per segment of this CTA's work, in issue order
        unsigned lr_ok = 0;      // calls whose b + v B' rows this CTA has waited for
        for (long long b = ms; ok && b < mend;) {
            const MLoc L = mlocate(a, b);
            const StepCall &k = a.call[L.c];
            const long long se = min(mend, L.tb0 + L.nkb);
            const int gtile = k.tile0 + L.tile;
            const int f0 = L.tile * TILE_M;
            // The CTA that holds a tile's first block finishes the tile.  It
            // reaches that tile at the end of its range, while the CTAs that
            // share the tile hold it at the start of theirs and publish their
            // partial sums early; waits therefore only run from a CTA to
            // higher-numbered ones, and nothing waits in a cycle.
            const bool fin = b == L.tb0;
            float *own = a.part + (size_t)(a.n_units + gtile + me) * SLOT;
            if (fin && k.lr_rmax > 0 && !((lr_ok >> L.c) & 1u)) {
                // b + v B' rows of the call: every low-rank item done
                epi_bar();
                const int n_lr_items = ctrl->n_lrs[L.c] * ((k.lr_rmax + LR_Q - 1) / LR_Q);
                if (et == 0) ctrl->flag = wait_count(sync + SY_LR + L.c, n_lr_items, abort_flag, gabort) ? 1 : 0;
                epi_bar();
                if (!ctrl->flag) { ok = false; break; }
                lr_ok |= 1u << L.c;
            }
            const int lastc = fin ? owner(fx, G, L.tb0 + L.nkb - 1) : me;
            if (!epi_all(wait_bar(ptx::smem_u32(&ctrl->tfull[buf]), bph, abort_flag, gabort, true, true))) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t tcol = tq + (uint32_t)(buf * 2 * BN);
            const bool my_v = k.vkb > 0 && se - L.tb0 > k.kblocks;
            if (!fin) {
                // hand this CTA's part of the tile to the tile's finisher
                if (b - L.tb0 < k.kblocks) publish(tcol, own, n, BN, row, half);
                if (my_v) publish(tcol + BN, own + (size_t)TILE_M * BN, n, BN, row, half);
                __threadfence();
                epi_bar();
                if (et == 0) atomicAdd(sync + SY_TILE + gtile, 1);
            } else {
                int others = 0;
                for (int j = me + 1; j <= lastc; ++j) others += fx.start[j + 1] > fx.start[j] ? 1 : 0;
                if (others > 0) {
                    epi_bar();
                    if (et == 0) {
                        ctrl->flag = wait_count(sync + SY_TILE + gtile, others, abort_flag, gabort) ? 1 : 0;
                    }
                    epi_bar();
                    if (!ctrl->flag) ok = false;
                    __threadfence();
                }
                if (ok) {
                    stage_meta(a, L.c, fx, ctrl, et);
                    for (int c32 = 0; c32 * 32 < n; ++c32) {
                        // operands first: none of them depends on the accumulator
                        float s8[2][8], e8[2][8], p8[2][8], oth[2][8], voth[2][8];
                        int t[2], g[2];
                        bool live[2];
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
                            const int it = c32 * 2 * EPI_THREADS + p * EPI_THREADS + et;
                            t[p] = it >> 4;
                            g[p] = it & 15;
                            const int j0 = f0 + g[p] * 8;
                            live[p] = t[p] < n && j0 < k.d_out;
                            const TokMeta &m = fx.tmeta[live[p] ? t[p] : 0];
                            ld_vec8(m.s + j0, live[p] && m.s != nullptr, 1.f, s8[p]);
                            ld_vec8(m.ve + j0, live[p] && m.vera && m.ve != nullptr, 0.f, e8[p]);
#pragma unroll
                            for (int e = 0; e < 8; ++e) { oth[p][e] = 0.f; voth[p][e] = 0.f; }
                            if (live[p] && m.rank > 0) {
                                // b + v B': the token's rank-group planes, in order
#pragma unroll
                                for (int e = 0; e < 8; ++e) p8[p][e] = 0.f;
#pragma unroll 1
                                for (int pg = 0; pg * LR_Q < m.rank; ++pg)
                                    add_part(k.pre + ((size_t)pg * NTOK + t[p]) * k.d_out + j0, p8[p]);
                            } else {
                                ld_vec8(m.b + j0, live[p] && m.b != nullptr, 0.f, p8[p]);
                            }
                        }
                        // the sharers' partial tiles, in CTA order
#pragma unroll 1
                        for (int j = me + 1; j <= lastc; ++j) {
                            if (fx.start[j + 1] <= fx.start[j]) continue;
                            const long long lo = max(L.tb0, fx.start[j]), hi = min(L.tb0 + L.nkb, fx.start[j + 1]);
                            const bool om = lo - L.tb0 < k.kblocks, ov = k.vkb > 0 && hi - L.tb0 > k.kblocks;
                            const float *sp = a.part + (size_t)(a.n_units + gtile + j) * SLOT;
#pragma unroll
                            for (int p = 0; p < 2; ++p) {
                                if (!live[p]) continue;
                                const float *q = sp + (size_t)t[p] * TILE_M + g[p] * 8;
                                if (om) add_part(q, oth[p]);
                                if (ov) add_part(q + (size_t)TILE_M * BN, voth[p]);
                            }
                        }
                        // this CTA's own sums come from TMEM: half 0 drains the
                        // base accumulator, half 1 the VeRA one
                        if (half == 0 || my_v) {
                            float *dstp = half == 0 ? xbm : xbv;
                            float v[32];
                            ptx::tmem_ld32(tcol + (half ? BN : 0) + c32 * 32, v);
#pragma unroll
                            for (int kk = 0; kk < 32; ++kk) dstp[kk * RED + row] = v[kk];
                        }
                        epi_bar();
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
                            if (!live[p]) continue;
                            const int kk = t[p] - c32 * 32, j0 = f0 + g[p] * 8;
                            // y = acc s + (b + v B') + vacc e
                            float y[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float acc = xbm[kk * RED + g[p] * 8 + e] + oth[p][e];
                                const float vacc = (my_v ? xbv[kk * RED + g[p] * 8 + e] : 0.f) + voth[p][e];
                                y[e] = fmaf(vacc, e8[p][e], fmaf(acc, s8[p][e], p8[p][e]));
                            }
                            if (k.out_f32) {
                                float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(k.out) + (size_t)t[p] * k.d_out + j0);
                                o[0] = make_float4(y[0], y[1], y[2], y[3]);
                                o[1] = make_float4(y[4], y[5], y[6], y[7]);
                            } else {
                                uint4 pk;
                                __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                                for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
                                *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(k.out) + (size_t)t[p] * k.d_out + j0) = pk;
                            }
                        }
                        epi_bar();
                        // the slot rows of this chunk are not read again: drop
                        // them from L2 without writing them back (threads below
                        // 128 take the base planes, the others the VeRA planes)
                        const int tl = c32 * 32 + ((et & 127) >> 2);
                        if (tl < n) {
                            const size_t off = (size_t)tl * TILE_M + (et & 3) * 32 + (et < 128 ? 0 : (size_t)TILE_M * BN);
#pragma unroll 1
                            for (int j = me + 1; j <= lastc; ++j) {
                                if (fx.start[j + 1] <= fx.start[j]) continue;
                                const long long lo = max(L.tb0, fx.start[j]), hi = min(L.tb0 + L.nkb, fx.start[j + 1]);
                                const bool om = lo - L.tb0 < k.kblocks, ov = k.vkb > 0 && hi - L.tb0 > k.kblocks;
                                if (et < 128 ? om : ov) ptx::discard_l2(a.part + (size_t)(a.n_units + gtile + j) * SLOT + off);
                            }
                        }
                    }
                }
                // every sharer has counted: clear the tile's counter for the next launch
                if (others > 0 && ok && et == 0) sync[SY_TILE + gtile] = 0;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[buf]));
            if (++buf == NB) { buf = 0; bph ^= 1; }
            b = se;
        }
    }

    // ---- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, NCOLS);
    }
    if (threadIdx.x == 0) {
        if (ctrl->abort) {
            atomicOr(a.status, STATUS_TIMEOUT);
            atomicExch(sync + SY_ABORT, 1);
        }
        __threadfence();
        const int old = atomicAdd(sync + SY_EXIT, 1);
        if (old == G - 1) {
            // every CTA has left: clear the counters for the next launch
            __threadfence();
            const bool aborted = atomicAdd(sync + SY_ABORT, 0) != 0;
            for (int c = 0; c < a.n_calls; ++c) {
                sync[SY_XS + c] = 0;
                sync[SY_LR + c] = 0;
                sync[SY_U + c] = 0;
            }
            if (aborted) {
                for (int i = 0; i < STEP_MAX_CALLS * STEP_MAX_VTILES; ++i) sync[SY_VTILE + i] = 0;
                for (int i = 0; i < a.n_tiles; ++i) sync[SY_TILE + i] = 0;
            }
            sync[SY_ABORT] = 0;
            sync[SY_EXIT] = 0;
            __threadfence();
        }
    }
}

}  // namespace

size_t step_smem_bytes(int bn, int stages, int rmax) {
    (void)rmax;   // the low-rank intermediates live in the transposition scratch
    return 1024 + (size_t)stages * (P_BYTES + bn * 128) + CTRL_BYTES + sizeof(Fixed) + XB_FLOATS * sizeof(float);
}

cudaError_t launch_step(const StepArgs &a, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_done{0};
    {
        const cudaError_t e = allow_max_dynamic_smem(step_kernel, attr_done);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    // one CTA per SM: a CTA holds up to all 512 TMEM columns and waits on the
    // others, so two on one SM must never be possible; more than half of the
    // SM's shared memory guarantees it whatever the register count
    size_t smem = step_smem_bytes(a.bn, a.stages, a.rmax);
    if (smem < (size_t)120 * 1024) smem = (size_t)120 * 1024;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, step_kernel, a);
}

}  // namespace scute
