// Segmented owned low-rank shrink on the tensor cores (bf16, the per-kernel
// path of prefill-sized batches):
//     v_t = x_t A'_a        for the sorted rows t of every owned-term segment
// (article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA",
// paper-daily.com, section "The big picture": the shrink multiplies the input
// down to rank dimensions; section "Which slots can be merged at load?": c and
// d are already folded into A').
//
// Work unit: up to 128 consecutive sorted rows of ONE segment (the indexing
// kernel lists them: seg_tile[s] counts the tiles before segment s) and one K
// chunk of the input (the chunks of the CUDA-core shrink, so that the same
// expand kernel sums them).  Per 64-wide K block, TMA brings the 128 token
// rows from the sorted token operand (x' = x wherever no owned-term row is
// rotated, which the host checks before choosing this kernel) and the
// segment's rows of A' through a tensor map of the adapter's own (made at
// registration, box = the rank rounded up to 16 rows, rows past the rank read
// as zero); one thread issues tcgen05.mma (M = 128 rows, N = that box, K = 16
// four times) into a TMEM accumulator.  The epilogue warps read the
// accumulator back (lane = row) and write v_part[chunk][row][q] for the rows
// of the segment and q < rank; rows of other segments in the tile are
// discarded.  The tensor cores leave the shrink bound by the bytes of x it
// reads, where the CUDA-core kernel is bound by its dependent loads.
//
// Warp roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues the
// MMAs, warps 2..5 drain TMEM.  Every wait is bounded (2 s); on expiry the CTA
// records STATUS_TIMEOUT, drains what it issued, frees TMEM and returns.
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

constexpr int THREADS = 192;
// Pipeline stages: 6 for a shrink that has the SMs to itself; fewer when the
// low-rank and the VeRA shrink run side by side, so that a CTA of each fits in
// one SM's shared memory (BESIDE_LR + BESIDE_VS stages of 24 KB, plus two
// control blocks and alignment pads, within 227 KB)
constexpr int STAGES_ALONE = 6;
constexpr int BESIDE_LR = 4;
constexpr int BESIDE_VS = 5;
constexpr int MAX_STAGES = 6;
constexpr int TILE_ROWS = 128;
constexpr int BOX_ROWS = 64;
constexpr int BOX_BYTES = BOX_ROWS * 128;
constexpr int XB = TILE_ROWS * 128;   // token rows of one K block
constexpr int AB = 64 * 128;          // at most 64 rank rows of A' of one K block
constexpr int STAGE = XB + AB;
constexpr int ACC_COLS = 64;          // one accumulator: up to 64 ranks
constexpr uint64_t WAIT_NS = 2000000000ull;

struct Ctrl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
constexpr int CTRL_BYTES = 256;
static_assert(sizeof(Ctrl) <= CTRL_BYTES, "control block");
static_assert(BESIDE_LR <= MAX_STAGES && BESIDE_VS <= MAX_STAGES && STAGES_ALONE <= MAX_STAGES, "stages");
static_assert(2 * (1024 + CTRL_BYTES) + (BESIDE_LR + BESIDE_VS) * (XB + AB) + 2 * 1024 <= 228 * 1024,
              "a low-rank and a VeRA shrink CTA side by side in one SM");

// K-major tile in the 128-byte-swizzle layout TMA writes (8-row atoms of
// 1024 bytes stacked along M / N).
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
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      bool honour_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (honour_abort && *abort_flag) return false;
        if (ptx::globaltimer() - t0 > WAIT_NS) {
            *abort_flag = 1;
            return false;
        }
    }
}

// One work unit: rows [r0, r1) of a segment with an owned term, K chunk ch,
// the adapter's rank, its box rows (rank rounded up to 16) and A' map.  Every
// role walks the same units and skips the same ones (segments without an
// owned term), reading the same read-only data.
struct Unit {
    int r0, r1, ch, rank, nb;
    const void *mapA;
};

__device__ __forceinline__ bool unit_at(const LrTcArgs &p, int u, Unit &U) {
    const int n_seg = p.meta->n_seg;
    const int n_tiles = p.seg_tile[n_seg];
    if (u >= n_tiles * p.ks) return false;
    const int tile = u / p.ks;
    U.ch = u - tile * p.ks;
    int lo = 0, hi = n_seg - 1;   // the last segment whose first tile is <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg_tile[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    U.r0 = p.seg_start[lo] + (tile - p.seg_tile[lo]) * TILE_ROWS;
    U.r1 = min(p.seg_start[lo + 1], U.r0 + TILE_ROWS);
    U.rank = 0;
    U.nb = 0;
    U.mapA = nullptr;
    const int a = p.seg_aid[lo];
    if (a >= 0) {
        const Slot &sl = p.slots[a];
        if (sl.A && sl.rank > 0 && sl.mapA) {
            U.rank = sl.rank;
            U.nb = (sl.rank + 15) & ~15;
            U.mapA = sl.mapA;
        }
    }
    return true;
}

template <int NST>
__global__ void __launch_bounds__(THREADS, 1) lr_shrink_tc_kernel(const __grid_constant__ LrTcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + NST * STAGE);
    volatile int *abort_flag = &ctrl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the segments come from the indexing kernel, the token rows from the
    // rotation kernel: wait for the previous launches before reading either.
    // The next launch may start at once: a VeRA shrink reads nothing written
    // here and waits for this grid only before it exits; the base GEMM waits
    // for it before it reads v
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->tfull[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->tempty[b]), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&ctrl->drain), 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.mapX);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctrl->tmem_base), 2 * ACC_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;

    if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            Unit U;
            for (int u = blockIdx.x; unit_at(p, u, U); u += gridDim.x) {
                if (U.rank == 0) continue;
                ptx::prefetch_tmap(U.mapA);
                const int kb0 = U.ch * p.chunk_blocks, kb1 = min(p.kblocks, kb0 + p.chunk_blocks);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar(ptx::smem_u32(&ctrl->empty[stage]), phase ^ 1, abort_flag)) goto prod_done;
                    const uint32_t fb = ptx::smem_u32(&ctrl->full[stage]);
                    const uint32_t sX = ptx::smem_u32(smem + stage * STAGE);
                    ptx::mbar_arrive_expect_tx(fb, (uint32_t)(XB + U.nb * 128));
                    ptx::tma_load_2d(sX, &p.mapX, kb * 64, U.r0, fb);
                    ptx::tma_load_2d(sX + BOX_BYTES, &p.mapX, kb * 64, U.r0 + BOX_ROWS, fb);
                    ptx::tma_load_2d(sX + XB, U.mapA, kb * 64, 0, fb);
                    ++issued;
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
        prod_done:
            // every issued copy must have landed before the CTA may exit
            {
                const int m_max = issued < NST ? (int)issued : NST;
                for (int m = 1; m <= m_max; ++m) {
                    const int s = (stage - m + NST) % NST;
                    const uint32_t ph = (s < stage) ? phase : (phase ^ 1);
                    wait_bar(ptx::smem_u32(&ctrl->full[s]), ph, abort_flag, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            Unit U;
            for (int u = blockIdx.x; unit_at(p, u, U); u += gridDim.x) {
                if (U.rank == 0) continue;
                if (!wait_bar(ptx::smem_u32(&ctrl->tempty[acc]), acc_phase ^ 1, abort_flag)) goto mma_done;
                ptx::tc_fence_after();
                const uint32_t idesc = idesc_bf16(TILE_ROWS, U.nb);
                const uint32_t d_tmem = tmem + (uint32_t)(acc * ACC_COLS);
                const int kb0 = U.ch * p.chunk_blocks, kb1 = min(p.kblocks, kb0 + p.chunk_blocks);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar(ptx::smem_u32(&ctrl->full[stage]), phase, abort_flag)) goto mma_done;
                    ptx::tc_fence_after();
                    const uint32_t sX = ptx::smem_u32(smem + stage * STAGE);
                    const uint64_t da = sw128_desc(sX), db = sw128_desc(sX + XB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(ptx::smem_u32(&ctrl->empty[stage]));
                    if (++stage == NST) { stage = 0; phase ^= 1; }
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
        const int q = warp & 3;   // TMEM lane quadrant this warp may read
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        Unit U;
        for (int u = blockIdx.x; unit_at(p, u, U); u += gridDim.x) {
            if (U.rank == 0) continue;
            if (!wait_bar(ptx::smem_u32(&ctrl->tfull[acc]), acc_phase, abort_flag)) break;
            ptx::tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            float v0[32], v1[32];
            ptx::tmem_ld32(tb, v0);
            if (U.nb > 32) ptx::tmem_ld32(tb + 32, v1);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[acc]));
            const int r = U.r0 + row;
            if (r < U.r1) {
                float *vp = p.v_part + ((size_t)U.ch * p.max_tokens + r) * MAX_RANK;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c < U.rank) vp[c] = v0[c];
                if (U.nb > 32) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (32 + c < U.rank) vp[32 + c] = v1[c];
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    // ---- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 2 * ACC_COLS);
    }
    if (threadIdx.x == 0 && ctrl->abort) atomicOr(p.status, STATUS_TIMEOUT);
}

// ---------------------------------------------------------------- VeRA shared shrink
// U_t = (x_t A_sh) * d_a(t) over the batch's VeRA rows (a contiguous range of
// the sorted rows), for prefill-sized batches: units of 128 rows x 64 shared
// ranks x one of ks K chunks, so that even a few hundred VeRA rows keep every
// SM streaming (one CTA per 128 x rank tile over the whole of K would leave
// most idle).  Each unit writes its partial tile (fp32) to a workspace and
// counts itself; the last unit of a tile adds the ks partials in chunk order,
// applies d and writes U (bf16): the result does not depend on which CTA
// finishes last.
__device__ __forceinline__ void vs_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// The same barrier as a vote: true when v holds in all 128 epilogue threads
// (a wait that some warps see end and others see give up must not split them).
__device__ __forceinline__ bool vs_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

template <int NST>
__global__ void __launch_bounds__(THREADS, 1) vera_shrink_tc_kernel(const __grid_constant__ VsTcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + NST * STAGE);
    __shared__ int s_last;
    volatile int *abort_flag = &ctrl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // segments and token rows come from earlier launches.  Launched right
    // after the low-rank shrink (which starts its dependents once its own wait
    // is over, so both are complete here), it runs beside that grid and waits
    // for it only before it exits, so that the launch after this one sees v
    if (!p.after_lr) ptx::grid_dep_wait();
    const int base = p.meta->offset[RANK_VERA], count = p.meta->count[RANK_VERA];
    const int n_rt = (count + TILE_ROWS - 1) / TILE_ROWS;
    const int per_rt = p.n_nt * p.ks;
    const int n_units = n_rt * per_rt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&ctrl->tfull[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&ctrl->tempty[b]), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&ctrl->drain), 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.mapX);
        ptx::prefetch_tmap(&p.mapA);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctrl->tmem_base), 2 * ACC_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;

    if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
                const int rt = u / per_rt, rem = u - rt * per_rt, nt = rem / p.ks, ch = rem - nt * p.ks;
                const int kb0 = ch * p.chunk_blocks, kb1 = min(p.kblocks, kb0 + p.chunk_blocks);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar(ptx::smem_u32(&ctrl->empty[stage]), phase ^ 1, abort_flag)) goto prod_done;
                    const uint32_t fb = ptx::smem_u32(&ctrl->full[stage]);
                    const uint32_t sX = ptx::smem_u32(smem + stage * STAGE);
                    ptx::mbar_arrive_expect_tx(fb, (uint32_t)(XB + BOX_BYTES));
                    ptx::tma_load_2d(sX, &p.mapX, kb * 64, base + rt * TILE_ROWS, fb);
                    ptx::tma_load_2d(sX + BOX_BYTES, &p.mapX, kb * 64, base + rt * TILE_ROWS + BOX_ROWS, fb);
                    ptx::tma_load_2d(sX + XB, &p.mapA, kb * 64, nt * 64, fb);
                    ++issued;
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
        prod_done:
            {
                const int m_max = issued < NST ? (int)issued : NST;
                for (int m = 1; m <= m_max; ++m) {
                    const int s = (stage - m + NST) % NST;
                    const uint32_t ph = (s < stage) ? phase : (phase ^ 1);
                    wait_bar(ptx::smem_u32(&ctrl->full[s]), ph, abort_flag, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t idesc = idesc_bf16(TILE_ROWS, 64);
            for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
                const int rt = u / per_rt, rem = u - rt * per_rt, nt = rem / p.ks, ch = rem - nt * p.ks;
                (void)rt;
                (void)nt;
                const int kb0 = ch * p.chunk_blocks, kb1 = min(p.kblocks, kb0 + p.chunk_blocks);
                if (!wait_bar(ptx::smem_u32(&ctrl->tempty[acc]), acc_phase ^ 1, abort_flag)) goto mma_done;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * ACC_COLS);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bar(ptx::smem_u32(&ctrl->full[stage]), phase, abort_flag)) goto mma_done;
                    ptx::tc_fence_after();
                    const uint32_t sX = ptx::smem_u32(smem + stage * STAGE);
                    const uint64_t da = sw128_desc(sX), db = sw128_desc(sX + XB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(ptx::smem_u32(&ctrl->empty[stage]));
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
                ptx::mma_commit(ptx::smem_u32(&ctrl->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
        mma_done:
            ptx::mma_commit(ptx::smem_u32(&ctrl->drain));
            wait_bar(ptx::smem_u32(&ctrl->drain), 0, abort_flag, false);
        }
        __syncwarp();
    } else {
        // ================================================= epilogue warps
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            const int rt = u / per_rt, rem = u - rt * per_rt, nt = rem / p.ks, ch = rem - nt * p.ks;
            if (!vs_all(wait_bar(ptx::smem_u32(&ctrl->tfull[acc]), acc_phase, abort_flag))) break;
            ptx::tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            float v0[32], v1[32];
            ptx::tmem_ld32(tb, v0);
            ptx::tmem_ld32(tb + 32, v1);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ctrl->tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            const int i = rt * TILE_ROWS + row;   // VeRA row
            if (i < count) {
                float4 *dst = reinterpret_cast<float4 *>(p.part + ((size_t)ch * p.max_tokens + i) * p.rv + nt * 64);
#pragma unroll
                for (int c = 0; c < 8; ++c) dst[c] = make_float4(v0[4 * c], v0[4 * c + 1], v0[4 * c + 2], v0[4 * c + 3]);
#pragma unroll
                for (int c = 0; c < 8; ++c) dst[8 + c] = make_float4(v1[4 * c], v1[4 * c + 1], v1[4 * c + 2], v1[4 * c + 3]);
            }
            // count this unit; the last of the tile's ks units finishes it
            __threadfence();
            vs_bar();
            if (et == 0) {
                int *ctr = p.ctr + VS_CTR_TILES + rt * p.n_nt + nt;
                const int old = atomicAdd(ctr, 1);
                s_last = old == p.ks - 1;
                if (s_last) atomicExch(ctr, 0);   // every unit of the tile has counted
            }
            vs_bar();
            if (s_last && i < count) {
                __threadfence();
                float sum[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) sum[c] = 0.f;
                for (int k = 0; k < p.ks; ++k) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(p.part + ((size_t)k * p.max_tokens + i) * p.rv + nt * 64);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float4 f = __ldcg(src + c);
                        sum[4 * c] += f.x;
                        sum[4 * c + 1] += f.y;
                        sum[4 * c + 2] += f.z;
                        sum[4 * c + 3] += f.w;
                    }
                }
                const int a = p.aid_s[base + i];
                const float *vd = a >= 0 ? p.slots[a].vd : nullptr;
                __nv_bfloat16 *U = reinterpret_cast<__nv_bfloat16 *>(p.U) + (size_t)i * p.ldu + nt * 64;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 pk;
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 8 * c + 2 * e;
                        const float d0 = vd ? vd[nt * 64 + j] : 0.f, d1 = vd ? vd[nt * 64 + j + 1] : 0.f;
                        h[e] = __floats2bfloat162_rn(sum[j] * d0, sum[j + 1] * d1);
                    }
                    reinterpret_cast<uint4 *>(U)[c] = pk;
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 2 * ACC_COLS);
    }
    if (threadIdx.x == 0) {
        if (ctrl->abort) {
            atomicOr(p.status, STATUS_TIMEOUT);
            atomicExch(p.ctr + VS_CTR_ABORT, 1);
        }
        // the last CTA out clears the tile counters a launch that gave up left
        __threadfence();
        if (atomicAdd(p.ctr + VS_CTR_EXIT, 1) == (int)gridDim.x - 1) {
            __threadfence();
            if (atomicAdd(p.ctr + VS_CTR_ABORT, 0) != 0)
                for (int t = 0; t < n_rt * p.n_nt; ++t) p.ctr[VS_CTR_TILES + t] = 0;
            p.ctr[VS_CTR_ABORT] = 0;
            p.ctr[VS_CTR_EXIT] = 0;
            __threadfence();
        }
    }
    if (p.after_lr) ptx::grid_dep_wait();
    ptx::grid_dep_launch();
}

}  // namespace

size_t shrink_tc_smem_bytes(int stages) { return 1024 + (size_t)stages * STAGE + CTRL_BYTES; }

namespace {

template <typename Args>
cudaError_t launch_shrink(void (*kernel)(Args), std::atomic<unsigned long long> &done, const Args &p, int grid,
                          int stages, cudaStream_t st, bool pdl) {
    {
        const cudaError_t e = allow_max_dynamic_smem(kernel, done);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = shrink_tc_smem_bytes(stages);
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

cudaError_t launch_lr_shrink_tc(const LrTcArgs &p, int grid, cudaStream_t st, bool pdl, bool beside) {
    static std::atomic<unsigned long long> done_alone{0}, done_beside{0};
    if (beside) return launch_shrink(lr_shrink_tc_kernel<BESIDE_LR>, done_beside, p, grid, BESIDE_LR, st, pdl);
    return launch_shrink(lr_shrink_tc_kernel<STAGES_ALONE>, done_alone, p, grid, STAGES_ALONE, st, pdl);
}

cudaError_t launch_vera_shrink_tc(const VsTcArgs &p, int grid, cudaStream_t st, bool pdl) {
    static std::atomic<unsigned long long> done_alone{0}, done_beside{0};
    if (p.after_lr) return launch_shrink(vera_shrink_tc_kernel<BESIDE_VS>, done_beside, p, grid, BESIDE_VS, st, pdl);
    return launch_shrink(vera_shrink_tc_kernel<STAGES_ALONE>, done_alone, p, grid, STAGES_ALONE, st, pdl);
}

}  // namespace scute
