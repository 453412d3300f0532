// Token -> segment indexing (one CTA).
//
// The batched layer works per adapter segment (article "Scute: Exact Batched
// Serving for PEFT Adapters Beyond LoRA", paper-daily.com, section "The big
// picture": shrink and expand per adapter segment; section "Where is the
// cheapest place to compute the remaining slots?": each tile belongs to one
// adapter).  This kernel orders the tokens by the key (method, adapter id) with
// ties kept in token order, so that every method's rows and every adapter's
// rows are contiguous, and emits:
//   perm[i]        token of sorted row i
//   aid_s[i]       adapter of sorted row i (-1 = base only)
//   seg_start/aid  maximal runs of one key
//   meta           rows, first row and segments per method
//   seg_unit       (optional) chunks of SEG_UNIT_ROWS rows before each segment
// Ids that name no registered adapter become base-only rows and set
// STATUS_BAD_ADAPTER.
//
// Sort: each token becomes the 32-bit word (key << 16) | token, sorted by a
// least-significant-digit counting sort on the key.  The keys are below
// 6 A + 1 (A = the adapter ids' bound), so for A <= 85 one pass on a digit of
// 8 or 9 bits orders them completely; otherwise two passes take the key's two
// bytes.  A pass is stable: warp w owns a contiguous run of the input, counts
// digits with __match_any_sync, and scatters in order through per-(warp,
// digit) offsets laid out digit-major, warp-minor.
#include "internal.h"
#include "ptx.cuh"

namespace scute {

namespace {

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Exclusive scan of one value per thread over the whole block (<= 1024
// threads).  Returns the exclusive prefix; *total receives the block sum.
__device__ int block_excl_scan(int v, int *s_warp, int *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int incl = warp_incl_scan(v);
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int x = lane < nw ? s_warp[lane] : 0;
        const int xi = warp_incl_scan(x);
        if (lane < nw) s_warp[lane] = xi - x;  // exclusive prefix of warp totals
        if (lane == nw - 1) s_warp[32] = xi;
    }
    __syncthreads();
    const int r = s_warp[w] + incl - v;
    if (total) *total = s_warp[32];
    __syncthreads();
    return r;
}

// One stable pass on the digit (v >> shift) & (DIG - 1); DIG <= blockDim.x
// (256 or 512 digits; hist holds nw x DIG counters).
template <int DIG>
__device__ void radix_pass(const uint32_t *src, uint32_t *dst, int n, int shift, int *hist,
                           int *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
    int chunk = (n + nw - 1) / nw;
    chunk = (chunk + 31) & ~31;
    const int beg = w * chunk;
    const int end = min(n, beg + chunk);
    for (int i = tid; i < nw * DIG; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int base = beg; base < end; base += 32) {
        const int i = base + lane;
        const bool valid = i < end;
        // lanes past the end get distinct digits no valid lane has
        const uint32_t d = valid ? ((src[i] >> shift) & (uint32_t)(DIG - 1)) : ((uint32_t)DIG + lane);
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (valid && lane == __ffs(peers) - 1) hist[w * DIG + d] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    int tot = 0;
    if (tid < DIG) {
#pragma unroll 8
        for (int k = 0; k < nw; ++k) tot += hist[k * DIG + tid];
    }
    const int excl = block_excl_scan(tid < DIG ? tot : 0, s_warp, nullptr);
    if (tid < DIG) {
        int run = excl;
#pragma unroll 8
        for (int k = 0; k < nw; ++k) {
            const int c = hist[k * DIG + tid];
            hist[k * DIG + tid] = run;
            run += c;
        }
    }
    __syncthreads();
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = beg; base < end; base += 32) {
        const int i = base + lane;
        const bool valid = i < end;
        const uint32_t v = valid ? src[i] : 0u;
        const uint32_t d = valid ? ((v >> shift) & (uint32_t)(DIG - 1)) : ((uint32_t)DIG + lane);
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        int pos = 0;
        if (valid) pos = hist[w * DIG + d] + __popc(peers & lt);
        __syncwarp();
        if (valid) {
            dst[pos] = v;
            if (lane == __ffs(peers) - 1) hist[w * DIG + d] += __popc(peers);
        }
        __syncwarp();
    }
    __syncthreads();
}

__global__ void __launch_bounds__(1024) index_kernel(const int32_t *ids, int n, const int8_t *method_tab,
                                                     int A, int *perm, int *aid_s, int *seg_start,
                                                     int *seg_aid, IndexMeta *meta, int *status,
                                                     int *seg_unit, int *seg_tile, int key_bits) {
    extern __shared__ uint32_t sm[];
    uint32_t *bufA = sm;
    uint32_t *bufB = sm + n;
    int *hist = reinterpret_cast<int *>(bufB + n);
    // the method table follows the counters of the widest pass this launch runs
    int8_t *s_tab = reinterpret_cast<int8_t *>(hist + (blockDim.x >> 5) * (key_bits == 9 ? 512 : 256));
    __shared__ int s_warp[33];
    __shared__ int s_count[N_RANKS], s_segc[N_RANKS];
    __shared__ int s_bad;

    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    if (tid < N_RANKS) { s_count[tid] = 0; s_segc[tid] = 0; }
    const uint32_t base_key = (uint32_t)RANK_BASE * (uint32_t)A;
    // the method table and every id of this thread are requested together
    // (one round of global loads), the ids' methods then read from shared
    // memory.  ids per thread, at most: n <= 2048 runs 256 or 512 threads,
    // larger n 1024
    constexpr int PER_T = INDEX_MAX_TOKENS / 1024;
    static_assert(PER_T * 256 >= 2048, "ids per thread for the 256-thread launch");
    int idv[PER_T], mv[PER_T];
    for (int e = tid; e < A; e += blockDim.x) s_tab[e] = method_tab[e];
#pragma unroll
    for (int j = 0; j < PER_T; ++j) {
        const int t = tid + j * (int)blockDim.x;
        idv[j] = t < n ? ids[t] : -1;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < PER_T; ++j) {
        mv[j] = -1;
        if (idv[j] >= 0 && idv[j] < A) mv[j] = s_tab[idv[j]];
    }
#pragma unroll
    for (int j = 0; j < PER_T; ++j) {
        const int t = tid + j * (int)blockDim.x;
        if (t >= n) break;
        const int id = idv[j], m = mv[j];
        if (m < 0 && id != -1) s_bad = 1;
        const uint32_t key = m >= 0 ? (uint32_t)m * (uint32_t)A + (uint32_t)id : base_key;
        bufA[t] = (key << 16) | (uint32_t)t;
    }
    __syncthreads();
    // keys of at most key_bits bits: one pass (the sorted words land in bufB)
    // or two (back in bufA); `spare` is the other buffer
    uint32_t *sorted = bufA, *spare = bufB;
    if (key_bits <= 8) {
        radix_pass<256>(bufA, bufB, n, 16, hist, s_warp);
        sorted = bufB;
        spare = bufA;
    } else if (key_bits == 9) {
        radix_pass<512>(bufA, bufB, n, 16, hist, s_warp);
        sorted = bufB;
        spare = bufA;
    } else {
        radix_pass<256>(bufA, bufB, n, 16, hist, s_warp);
        radix_pass<256>(bufB, bufA, n, 24, hist, s_warp);
    }

    // the per-row outputs, with consecutive threads on consecutive rows (one
    // SM writes them all: a strided pattern would cost a store sector per row)
    for (int i = tid; i < n; i += blockDim.x) {
        const uint32_t v = sorted[i];
        const uint32_t key = v >> 16;
        const int rank = (int)(key / (uint32_t)A);
        perm[i] = (int)(v & 0xFFFFu);
        aid_s[i] = rank >= RANK_BASE ? -1 : (int)(key - (uint32_t)rank * (uint32_t)A);
    }
    // segments: runs of one key; each thread owns a contiguous run of rows
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int r0 = min(n, tid * per), r1 = min(n, r0 + per);
    int nflag = 0;
    for (int i = r0; i < r1; ++i)
        if (i == 0 || (sorted[i - 1] >> 16) != (sorted[i] >> 16)) ++nflag;
    int total = 0;
    int s = block_excl_scan(nflag, s_warp, &total);
    for (int i = r0; i < r1; ++i) {
        const uint32_t key = sorted[i] >> 16;
        if (i == 0 || (sorted[i - 1] >> 16) != key) {
            const int rank = (int)(key / (uint32_t)A);
            seg_start[s] = i;
            seg_aid[s] = rank >= RANK_BASE ? -1 : (int)(key - (uint32_t)rank * (uint32_t)A);
            spare[s] = (uint32_t)rank;   // (free once the sort is done)
            ++s;
        }
    }
    if (tid == 0) seg_start[total] = n;
    __syncthreads();
    // rows and segments per method, one shared atomic per segment (one per
    // row would serialise on the few method counters)
    for (int q = tid; q < total; q += blockDim.x) {
        const int rank = (int)spare[q];
        atomicAdd(&s_count[rank], seg_start[q + 1] - seg_start[q]);
        atomicAdd(&s_segc[rank], 1);
    }
    __syncthreads();
    // work units of the segmented kernels: each segment cut into chunks of
    // SEG_UNIT_ROWS and of SEG_TILE_ROWS rows; seg_unit[s] / seg_tile[s] =
    // chunks of the segments before s.  Both counts share one scan, packed
    // in 16-bit halves (each total is below n / 32 + n <= 16896)
    if (seg_unit || seg_tile) {
        static_assert(INDEX_MAX_TOKENS / SEG_UNIT_ROWS + INDEX_MAX_TOKENS < (1 << 15), "packed unit counts");
        auto chunks = [&](int q) {
            const int rows = seg_start[q + 1] - seg_start[q];
            return (rows + SEG_UNIT_ROWS - 1) / SEG_UNIT_ROWS + (((rows + SEG_TILE_ROWS - 1) / SEG_TILE_ROWS) << 16);
        };
        const int per_s = (total + blockDim.x - 1) / blockDim.x;
        const int s0 = min(total, tid * per_s), s1 = min(total, s0 + per_s);
        int u = 0;
        for (int q = s0; q < s1; ++q) u += chunks(q);
        int tot_u = 0;
        int ex = block_excl_scan(u, s_warp, &tot_u);
        for (int q = s0; q < s1; ++q) {
            if (seg_unit) seg_unit[q] = ex & 0xFFFF;
            if (seg_tile) seg_tile[q] = ex >> 16;
            ex += chunks(q);
        }
        if (tid == 0) {
            if (seg_unit) seg_unit[total] = tot_u & 0xFFFF;
            if (seg_tile) seg_tile[total] = tot_u >> 16;
        }
    }
    if (tid == 0) {
        meta->n_seg = total;
        int off = 0;
        for (int r = 0; r < N_RANKS; ++r) {
            meta->count[r] = s_count[r];
            meta->offset[r] = off;
            meta->seg_count[r] = s_segc[r];
            off += s_count[r];
        }
        if (s_bad) atomicOr(status, STATUS_BAD_ADAPTER);
    }
}

}  // namespace

cudaError_t launch_index(const int32_t *ids, int n, const int8_t *method_tab, int max_adapters,
                         int *perm, int *aid_s, int *seg_start, int *seg_aid, IndexMeta *meta,
                         int *status, cudaStream_t st, int *seg_unit, int *seg_tile) {
    static std::atomic<unsigned long long> attr_done{0};
    {
        const cudaError_t e = allow_max_dynamic_smem(index_kernel, attr_done);
        if (e != cudaSuccess) return e;
    }
    // the largest key is the base rows' 6 A: its bit count picks the passes;
    // a 512-digit pass needs a thread per digit
    int key_bits = 1;
    while (key_bits < 16 && ((uint32_t)RANK_BASE * (uint32_t)max_adapters >> key_bits) != 0u) ++key_bits;
    const int threads = n <= 2048 ? (key_bits == 9 ? 512 : 256) : 1024;
    const int digits = key_bits == 9 ? 512 : 256;
    const size_t smem = (size_t)2 * n * sizeof(uint32_t) + (size_t)(threads / 32) * digits * sizeof(int) +
                        (((size_t)max_adapters + 15) & ~(size_t)15);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, index_kernel, ids, n, method_tab, max_adapters, perm, aid_s,
                              seg_start, seg_aid, meta, status, seg_unit, seg_tile, key_bits);
}

}  // namespace scute
