// Internal declarations shared by the kernels and the host runtime of
// libscute.so.  Nothing here is part of the C ABI (include/scute.h is).
#pragma once

#include <cuda.h>  // CUtensorMap type only; the driver entry point is fetched at run time
#include <cuda_bf16.h>
#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>

namespace scute {

// Method ranks: the order tokens are grouped in (base-only tokens last).
enum : int {
    RANK_LORA = 0, RANK_DORA = 1, RANK_IA3 = 2, RANK_VERA = 3, RANK_OFT = 4, RANK_NF = 5,
    RANK_BASE = 6, N_RANKS = 7
};

// Device status word bits (read back by scute_sync_status).
enum : int { STATUS_BAD_ADAPTER = 1, STATUS_TIMEOUT = 2 };

constexpr int OFT_BLK = 32;
constexpr int MAX_RANK = 64;          // owned low-rank term
constexpr int KS_MAX = 8;             // K splits of the low-rank shrink
constexpr int INDEX_MAX_TOKENS = 16384;

// One (layer, adapter) entry of the device slot table: the folded normal form
// of that adapter on that layer.  A null pointer is the identity value.
struct Slot {
    const float *s;    // [d_out] live column factor (DoRA, (IA)^3, NF)
    const float *b;    // [d_out] live shift (NF)
    const void *R;     // [d_in/32][32][32] live input rotation (OFT, NF)
    const void *A;     // owned A' = c A diag(d), stored [rank][d_in]
    const void *B;     // owned B' = B diag(e), stored [rank][d_out]
    const float *vd;   // VeRA d [shared rank] (c folded in); null = no shared term
    const float *ve;   // VeRA e [d_out]; null = ones
    const void *Rt;    // R with every 32x32 block transposed (bf16 contexts; null = no R)
    const void *Bu;    // DoRA: B' without its s folded in (the separate-s-pass placement,
                       // and the prefill expand that runs before s is applied)
    const void *mapA;  // bf16: CUtensorMap of A' (box 64 columns x rank rounded up to 16 rows)
    int rank;          // rank of the owned term (0 = none)
    int pad;
};

// Separate-pass placements of live slots (scute_set_variant; the same codes as
// SCUTE_VARIANT_OFT_PASS and SCUTE_VARIANT_S_PASS).
enum : int { VARIANT_OFT_PASS = 1, VARIANT_S_PASS = 2 };

// Results of the token indexing kernel beyond the per-row arrays.
struct IndexMeta {
    int n_seg;
    int count[N_RANKS];       // sorted rows per method rank
    int offset[N_RANKS];      // first sorted row per method rank
    int seg_count[N_RANKS];   // segments per method rank
};
static_assert(sizeof(IndexMeta) == 22 * sizeof(int), "IndexMeta layout");

// ---------------------------------------------------------------- GEMM
// D[128 x BN] += P[128 rows, K] * Q[BN rows, K]^T on tcgen05, both operands
// K-major in 128-byte swizzled shared-memory tiles loaded by TMA.
enum : int { EPI_BASE = 0, EPI_VERA_D = 1, EPI_VERA_E = 2 };

struct GemmArgs {
    CUtensorMap mapP;          // P operand: 128-row tiles
    CUtensorMap mapQ;          // Q operand: BN-row tiles
    CUtensorMap mapVP;         // fused VeRA expand: P = B_sh^T [d_out][rv]
    CUtensorMap mapVQ;         // fused VeRA expand: Q = U [tokens][rv] (sorted rows)
    int kblocks;               // K extent in 128-byte blocks
    int n_ft;                  // tiles along the feature dimension
    int n_feat;                // features (d_out, or the shared rank)
    int tok_on_p;              // 1: P rows are tokens; 0: Q rows are tokens
    int n_tok_host;            // token rows when tok_cnt is null (and the grid bound)
    const int *tok_cnt;        // device token-row count (VeRA rows) or null
    const int *tok_base;       // device row offset of the token operand's TMA coordinates
    const int *sorted_base;    // device offset from token row to sorted row
    int splits;                // K splits = cluster size (1 = persistent tile loop)
    int stages;                // shared-memory pipeline depth
    int epi;                   // EPI_*
    int out_f32;               // output element type (1 float, 0 bf16)
    int ld_out;                // output row pitch in elements
    int ldu;                   // U row pitch in elements
    int u_split3;              // U holds [hi | hi | lo] tf32 parts (fp32 context)
    int u_rank;                // shared rank (for the split layout)
    const Slot *slots;         // slot table row of this layer: slots[adapter]
    const int *perm;           // sorted row -> token
    const int *aid_s;          // sorted row -> adapter (-1 base)
    void *out;                 // [n, ld_out]
    void *U;                   // VeRA intermediate
    int *status;
    // fused epilogue
    int vera_kb;               // VeRA expand K blocks folded into this GEMM (0 = none; features on P)
    int stage_out;             // EPI_VERA_E, tokens on P, bf16 out: each tile's rows of out are
                               // read into shared memory before its accumulator is complete
                               // and written back with coalesced stores
    // owned low-rank intermediate (null = none).  Features on P: v[row * v_ld + q].
    // Tokens on P (bf16): the K-chunk partials of the shrink, summed in chunk
    // order, v[s * v_kstride + row * v_ld + q] for s < v_ks; the expand runs as
    // an extra tensor-core K block of each tile (rows of adapters with an s
    // other than DoRA's, or beyond the block's k-steps, on the CUDA cores in
    // the epilogue), so out is written once
    const float *v;
    int v_ld;
    int v_ks;
    long long v_kstride;
    int lr_rmax;               // largest owned rank on the layer (features on P: v columns per token)
    // the P operand's rows in global memory (features-on-P orientation): each
    // CTA asks L2 for its whole K range of them at start
    const void *p_base;
    long long p_pitch;         // bytes between rows
    int p_rows;
    // K-split partial tiles: CTA b of a cluster writes [token][128] fp32 (and
    // the VeRA plane after it) at part + b * part_stride; the cluster's CTAs
    // then read each other's slices from L2
    float *part;
    long long part_stride;     // floats per CTA
};
// floats of K-split workspace one GEMM launch needs
inline size_t gemm_part_floats(int grid, int bn, bool vera) {
    return (size_t)grid * (size_t)bn * 128 * (vera ? 2 : 1);
}
constexpr size_t PART_WORKSPACE_FLOATS = (size_t)8 << 20;   // 32 MiB

struct GemmPlan {
    int bn;        // 64, 128 or 256
    int splits;    // 1, 2, 4, 8
    int stages;
    int grid;
    int tf32;
    size_t smem;
};

GemmPlan plan_gemm(int n_tok, int n_feat, int kblocks, bool tok_on_p, bool tf32, int num_sms,
                   int lr_rmax = 0, bool stage_out = false);
cudaError_t launch_gemm(const GemmArgs &g, const GemmPlan &p, cudaStream_t st, bool pdl);

// K splits of the owned low-rank shrink: chunks of about 2048 elements, at
// most KS_MAX of them, each a multiple of 256 elements.
inline int lowrank_ks(int d_in, int *kchunk_out) {
    int ks = (d_in + 2047) / 2048;
    if (ks > KS_MAX) ks = KS_MAX;
    int kchunk = (d_in + ks - 1) / ks;
    kchunk = (kchunk + 255) / 256 * 256;
    ks = (d_in + kchunk - 1) / kchunk;
    if (kchunk_out) *kchunk_out = kchunk;
    return ks;
}

// Raise a kernel's dynamic shared-memory limit to the device's opt-in maximum
// less its static shared memory.  A function attribute belongs to one device
// context, so the raise is made once per (kernel, device): `done` holds one bit
// per device id below 64 (devices beyond that ask on every launch).  Two host
// threads racing on the first launch both set the same value, which is
// harmless.
template <typename K>
cudaError_t allow_max_dynamic_smem(K kernel, std::atomic<unsigned long long> &done) {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}


// ---------------------------------------------------------------- decode step
// Every projection of one batched call (up to STEP_MAX_CALLS layers over the
// same n <= 128 tokens) in one persistent cooperative launch: the prologue
// work (gather / OFT rotation of the token operand, owned low-rank shrink) on
// the epilogue warps, the VeRA shared shrink as tcgen05 K-chunks, and every
// layer's base GEMM tiles with the VeRA expand K blocks, split over the CTAs
// by contiguous ranges of 64-wide K blocks (stream-K), partial tiles summed
// by the CTA holding each tile's first block.
constexpr int STEP_MAX_CALLS = 8;
constexpr int STEP_MAX_TOKENS = 128;
// stream-block charge of one decode low-rank item: (d_in + d_out) / this
constexpr int ITEM_FEATURES_PER_BLOCK = 1152;
constexpr int STEP_MAX_GRID = 190;
constexpr int STEP_MAX_VTILES = 8;     // VeRA shrink tiles per call (shared rank <= 1024)

// Layout of the step's int counter array (device, zero between launches).
enum : int {
    SY_XS = 0,           // [call] prologue items that wrote the call's token operand
    SY_LR = 8,           // [call] low-rank shrink items done
    SY_U = 16,           // [call] VeRA shrink tiles finished
    SY_EXIT = 24,        // CTAs that left
    SY_ABORT = 25,       // a CTA gave up a wait
    SY_VTILE = 32,       // [call * 8 + tile] arrivals at a VeRA shrink tile
    SY_TILE = 96         // [main tile] arrivals
};
constexpr int STEP_SYNC_INTS = 1 << 16;

struct StepCall {
    CUtensorMap mapW;          // W^T [d_out][kdim]
    CUtensorMap mapXs;         // token operand [128][kdim]
    CUtensorMap mapAsh;        // A_sh^T [rv][kdim]
    CUtensorMap mapBsh;        // B_sh^T [d_out][krv]
    CUtensorMap mapU;          // VeRA intermediate [128][krv]
    CUtensorMap mapX;          // token-operand source [n][d_in] (read directly when vs_x / xs_direct)
    const void *x;             // [n][d_in] token-operand source (the caller's x, or its rotated copy)
    const void *x0;            // [n][d_in] the caller's x (low-rank shrink input)
    void *xs;                  // [128][kdim]
    void *U;                   // [128][krv]
    float *pre;                // [ceil(lr_rmax / 8)][128][d_out] fp32: b + v B' per group of 8 ranks
    void *out;                 // [n][d_out]
    const Slot *slots;         // the layer's slot row
    const void *Wt;            // W^T base (L2 prefetch)
    long long blk0;            // first main block (stream-K order)
    int d_in, kdim, d_out, krv, rv;
    int kblocks;               // 64-wide K blocks of the base GEMM
    int vkb;                   // VeRA expand K blocks per main tile (0: none)
    int n_ft;                  // main tiles (128 features each)
    int n_vt;                  // VeRA shrink tiles (128 shared ranks each; 0: none)
    int vs_chunks;             // VeRA shrink units per VeRA tile
    int vs_unit0;              // first VeRA shrink unit
    int tile0;                 // first main tile id
    int lr_rmax;               // largest owned rank (0: no low-rank shrink)
    int out_f32;
    int lr_items;              // owned low-rank shrink items
    int lr_item0;              // first low-rank item
    int vs_x;                  // VeRA shrink reads x itself (no wait for x')
    int xs_direct;             // no row of this call is rotated: the base tiles read x itself
};

struct StepArgs {
    StepCall call[STEP_MAX_CALLS];
    int n_calls, n, A, bn, stages, grid;
    const int32_t *ids;
    const int8_t *method_tab;
    int *status;
    float *part;               // partial tiles: slot * 2 planes * 128 * bn floats
    int *sync;
    long long t_main;          // main K blocks over all calls
    long long w_total;         // main + VeRA shrink K blocks + low-rank item charges
    int n_units;               // VeRA shrink units (<= grid)
    int vs_ch;                 // K blocks per VeRA shrink unit
    int n_tiles;               // main tiles over all calls
    int n_items;               // prologue items over all calls
    int rmax;                  // largest lr_rmax
    int hold;                  // extra count the token-operand wait needs (failure-path test)
    int variant;               // VARIANT_*: slots applied by separate passes instead
    int it_call[STEP_MAX_CALLS];   // calls in the order their low-rank items are dealt
    int it_ng[STEP_MAX_CALLS];     // rank groups of 8 per owned-term segment, in that order
    long long start[STEP_MAX_GRID + 1];   // main-block range of each CTA: [start[i], start[i+1])
};

size_t step_smem_bytes(int bn, int stages, int rmax);
cudaError_t launch_step(const StepArgs &a, cudaStream_t st);

// ---------------------------------------------------------------- separate passes
struct PassCall {
    const void *x;     // oft_pass: input [n][d_in]
    void *xo;          // oft_pass: rotated copy [n][d_in]
    void *out;         // s_pass: output [n][d_out], scaled in place
    const Slot *slots;
    int d_in, d_out;
};
struct PassArgs {
    PassCall call[STEP_MAX_CALLS];
    int n_calls, n, A, out_f32;
    const int32_t *ids;
    const int8_t *method_tab;
};
cudaError_t launch_oft_pass(const PassArgs &p, int max_d_in, cudaStream_t st);
cudaError_t launch_s_pass(const PassArgs &p, int max_d_out, cudaStream_t st);

// ---------------------------------------------------------------- other kernels
// Token indexing (one CTA).  seg_unit (optional, n_seg + 1 ints): the
// segmented low-rank kernels' work units, every segment cut into chunks of
// SEG_UNIT_ROWS sorted rows; seg_unit[s] counts the chunks before segment s.
// seg_tile (optional, n_seg + 1 ints): the same with SEG_TILE_ROWS rows, the
// tiles of the tensor-core shrink.
constexpr int SEG_UNIT_ROWS = 32;
constexpr int SEG_TILE_ROWS = 128;
cudaError_t launch_index(const int32_t *ids, int n, const int8_t *method_tab, int max_adapters,
                         int *perm, int *aid_s, int *seg_start, int *seg_aid, IndexMeta *meta,
                         int *status, cudaStream_t st, int *seg_unit = nullptr, int *seg_tile = nullptr);

// Copies of up to COPY_MAX_SEGS buffers in one launch (k_copy.cu): each
// source and destination a device-visible address (device memory, or the
// device address of pinned, mapped host memory).
constexpr int COPY_MAX_SEGS = 2 * 8 + 1;
struct CopySegs {
    const void *src[COPY_MAX_SEGS];
    void *dst[COPY_MAX_SEGS];
    size_t bytes[COPY_MAX_SEGS];
    int n;
};
cudaError_t launch_copy_segments(const CopySegs &s, cudaStream_t st);

cudaError_t launch_gather_rotate(bool f32, const void *x, int d_in, int n, const int *perm,
                                 const int *aid_s, const Slot *slots, void *xs, int kdim,
                                 cudaStream_t st, bool pdl);

// Segmented owned low-rank shrink and expand over the units of launch_index
// (unit_bound: a host-side bound on their number); with shrink false only the
// expand runs (its v_part written by the tensor-core shrink below), with
// expand false only the shrink (the expand then runs in the base GEMM's
// epilogue).
cudaError_t launch_lowrank(bool f32, const void *x, int d_in, int d_out, int unit_bound, const int *perm,
                           const int *seg_start, const int *seg_aid, const int *seg_unit,
                           const IndexMeta *meta, const Slot *slots, float *v_part, int max_tokens, void *out,
                           int out_f32, cudaStream_t st, bool pdl, int max_rank, bool shrink = true,
                           bool expand = true);

// Segmented owned low-rank shrink on the tensor cores (bf16): units = the
// SEG_TILE_ROWS-row tiles of launch_index x the K chunks of lowrank_ks, each
// writing v_part[chunk][sorted row][rank] like the CUDA-core shrink.  Reads the
// sorted token operand, so it serves layers where no owned-term row is rotated.
struct LrTcArgs {
    CUtensorMap mapX;          // sorted token operand [max_tokens][d_in] (box 64 rows x 128 B)
    int kblocks;               // 64-wide K blocks of d_in
    int ks;                    // K chunks (lowrank_ks)
    int chunk_blocks;          // K blocks per chunk
    int max_tokens;            // row pitch of a v_part chunk
    const int *seg_start, *seg_aid, *seg_tile;
    const IndexMeta *meta;
    const Slot *slots;
    float *v_part;             // [ks][max_tokens][MAX_RANK]
    int *status;
};
size_t shrink_tc_smem_bytes(int stages);
// VeRA shared shrink on the tensor cores for prefill-sized batches (bf16,
// shared rank a multiple of 64): units of 128 VeRA rows x 64 shared ranks x
// one of ks K chunks; partial tiles in `part`, the last unit of a tile sums
// them in chunk order, applies d and writes U (bf16, row = VeRA row).
// ctr: [VS_CTR_TILES + tiles] ints, zero between launches.
enum : int { VS_CTR_EXIT = 0, VS_CTR_ABORT = 1, VS_CTR_TILES = 2 };
constexpr int VS_CTR_INTS = 4096;
constexpr int VS_KS = 4;               // K chunks
struct VsTcArgs {
    CUtensorMap mapX;          // sorted token operand [max_tokens][d_in]
    CUtensorMap mapA;          // A_sh^T [rv][d_in] (box 64 rows x 128 B)
    int kblocks, ks, chunk_blocks;
    int n_nt;                  // rv / 64
    int rv, ldu, max_tokens;
    const IndexMeta *meta;     // offset / count of the VeRA rows
    const int *aid_s;
    const Slot *slots;
    float *part;               // [ks][max_tokens][rv]
    int *ctr;
    void *U;                   // bf16 [VeRA rows][ldu]
    int *status;
    int after_lr;              // launched right after the tensor-core low-rank shrink
};
cudaError_t launch_vera_shrink_tc(const VsTcArgs &p, int grid, cudaStream_t st, bool pdl);
// beside: a VeRA shrink is launched right after it, to run beside it
cudaError_t launch_lr_shrink_tc(const LrTcArgs &p, int grid, cudaStream_t st, bool pdl, bool beside);

// registration-time kernels
cudaError_t launch_transpose_w(bool f32, const void *W, int rows, int cols, void *Wt, int kdim,
                               int pattern, cudaStream_t st);
cudaError_t launch_fold_A(bool f32, const void *A, int d_in, int rank, float c, const float *d,
                          void *Aout, cudaStream_t st);
cudaError_t launch_fold_B(bool f32, const void *B, int rank, int d_out, const float *e,
                          const float *s, void *Bout, cudaStream_t st);
cudaError_t launch_dora_scale(bool f32, const void *Wt, int kdim, int d_in, int d_out,
                              const void *A, const void *B, int rank, float c,
                              const float *m, float *s_out, int *err, cudaStream_t st);
cudaError_t launch_scale_vec(const float *v, float c, float *out, int n, cudaStream_t st);
// dst[b][j][i] = src[b][i][j] for n_blk 32x32 bf16 blocks
cudaError_t launch_transpose_blocks(const void *src, void *dst, int n_blk, cudaStream_t st);

}  // namespace scute
