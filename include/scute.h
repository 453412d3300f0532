/*
 * scute.h -- C ABI of libscute.so: the adapted linear layer in normal form,
 * evaluated for a heterogeneous batch in which every token carries its own
 * adapter id, on one NVIDIA GB300 (sm_103a).
 *
 * What is computed.  For a token x (row vector, [d_in]) routed to adapter a,
 *
 *     F_a(x) = ((x R) W) * s + b + sum_k c_k (((x A_k) * d_k) B_k * e_k)
 *
 * the "normal form" of the article "Scute: Exact Batched Serving for PEFT
 * Adapters Beyond LoRA" (paper-daily.com), section "The big picture: six extra
 * slots in the LoRA computation".  W is the layer's shared base weight.  LoRA,
 * DoRA, (IA)^3, VeRA and OFT adapters are written into the slots at
 * registration; the fold rule of section "Which slots can be merged at load?"
 * multiplies every slot next to a tensor the adapter owns into that tensor, and
 * keeps live the slots next to shared tensors (s, b, R next to W; VeRA's d and
 * e next to the shared VeRA pair).  Tokens with id -1 get x W.
 *
 * Conventions used by every call below.
 *   - Row-major, row-vector orientation: x [n, d_in], W [d_in, d_out],
 *     A [d_in, rank], B [rank, d_out], out [n, d_out].
 *   - Matrices (W, A, B, R, shared VeRA A/B, x, out) are in the context dtype
 *     (bf16 or fp32).  A bf16 context may also write an fp32 `out`.
 *     Vectors (s, b, d, e, DoRA magnitude, (IA)^3 l) are always float32.
 *   - OFT rotations are explicit 32x32 blocks: R [d_in/32, 32, 32]; block k
 *     acts on input features [32k, 32k+32).
 *   - Setup calls (create, add_layer, set_shared, register, unregister) accept
 *     host or device pointers (the library copies through unified addressing)
 *     and may synchronise the device.  The library owns every tensor it keeps:
 *     caller buffers may be freed as soon as a setup call returns.
 *   - scute_linear is asynchronous on the caller's stream, allocates nothing,
 *     never synchronises and can be captured in a CUDA graph.  Errors the device
 *     detects (an id that names no adapter, a wait that timed out) are recorded
 *     in a status word read by scute_sync_status.  No call traps or hangs.
 *   - A context is thread-compatible, not thread-safe: calls on one context
 *     must be serialised by the caller, and its scute_linear calls must be
 *     ordered on the device (one stream, or streams joined by events), because
 *     they share the context's workspace.
 */
#ifndef SCUTE_H
#define SCUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct scute_ctx scute_ctx;

/* Adapter methods.  The order is also the order tokens are grouped in. */
typedef enum {
    SCUTE_LORA = 0, /* owned A, B and scalar c                                   */
    SCUTE_DORA = 1, /* owned A, B, c and learned column lengths (magnitude)      */
    SCUTE_IA3  = 2, /* l on key / value / up projections (the s slot)           */
    SCUTE_VERA = 3, /* per-adapter d, e around the layer's shared VeRA pair     */
    SCUTE_OFT  = 4, /* block-diagonal input rotation R (32x32 blocks)           */
    SCUTE_NF   = 5  /* raw normal-form slots: s, b, R and one owned term        */
} scute_method;

typedef enum { SCUTE_BF16 = 0, SCUTE_FP32 = 1 } scute_dtype;

typedef enum {
    SCUTE_OK = 0,
    SCUTE_ERR_ARG = 1,          /* null pointer, bad enum, out-of-range id/layer   */
    SCUTE_ERR_SHAPE = 2,        /* dimension not allowed (see each call)          */
    SCUTE_ERR_DTYPE = 3,        /* dtype combination not allowed                   */
    SCUTE_ERR_OOM = 4,          /* device allocation failed                        */
    SCUTE_ERR_BAD_ADAPTER = 5,  /* a token id named no registered adapter          */
    SCUTE_ERR_CUDA = 6,         /* a CUDA runtime call failed (see last_error)     */
    SCUTE_ERR_TIMEOUT = 7,      /* a bounded device-side wait gave up              */
    SCUTE_ERR_UNSUPPORTED = 8,  /* valid but outside what this build supports      */
    SCUTE_ERR_NO_DEVICE = 9     /* no usable sm_103 device                        */
} scute_status;

/* Limits of this build. */
#define SCUTE_MAX_TOKENS    16384  /* tokens per scute_linear call                 */
#define SCUTE_MAX_ADAPTERS  8192   /* registered adapters per context              */
#define SCUTE_MAX_RANK      64     /* rank of an owned low-rank term               */
#define SCUTE_MAX_SHARED_RANK 1024 /* rank of a layer's shared VeRA pair           */
#define SCUTE_OFT_BLOCK     32

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int scute_version(void);

/* Create a context on CUDA device `device`.
 *   dtype          storage/compute dtype of matrices and activations;
 *   max_tokens     largest n of a scute_linear call (1..SCUTE_MAX_TOKENS);
 *   max_adapters   adapter ids are 0..max_adapters-1 (1..SCUTE_MAX_ADAPTERS);
 *   max_layers     layer ids are 0..max_layers-1.
 * The context allocates its workspace here and grows it in scute_add_layer and
 * scute_set_shared.  Returns SCUTE_ERR_NO_DEVICE when the device is not sm_103. */
scute_status scute_create(scute_ctx **ctx, int device, scute_dtype dtype, int max_tokens,
                          int max_adapters, int max_layers);

/* Free every device allocation of the context (synchronises the device). */
void scute_destroy(scute_ctx *ctx);

/* Last error message of this context (static storage owned by the context). */
const char *scute_last_error(const scute_ctx *ctx);

/* Add base layer `layer` with shared weight W [d_in, d_out] (row-major, context
 * dtype).  The base GEMM h = xW is computed once for the whole batch (article,
 * "The big picture").  d_in and d_out must be positive multiples of 32
 * (SCUTE_ERR_SHAPE otherwise).  The library keeps a K-major copy of W. */
scute_status scute_add_layer(scute_ctx *ctx, int layer, int d_in, int d_out, const void *W);

/* Set the shared VeRA pair of `layer`: A_sh [d_in, rank], B_sh [rank, d_out]
 * (context dtype), shared by every VeRA adapter on that layer (article, "Which
 * slots can be merged at load?": VeRA's A and B are shared, rank 256 there).
 * rank must be a positive multiple of 32 and at most SCUTE_MAX_SHARED_RANK. */
scute_status scute_set_shared(scute_ctx *ctx, int layer, int rank, const void *A_sh,
                              const void *B_sh);

/* One layer's raw (unfolded) tensors of an adapter.  NULL = slot absent
 * (identity).  Which fields a method reads:
 *   LORA  A [d_in, rank], B [rank, d_out], c (= alpha / rank), rank
 *   DORA  A, B, c, rank, magnitude [d_out] (learned column length m)
 *   IA3   l [d_out]
 *   VERA  d [shared rank], e [d_out], c  (the layer must have a shared pair;
 *         c scales the shared term and is applied as given, like every other
 *         term's c: 1 for plain VeRA, 0 switches the term off)
 *   OFT   R [d_in/32, 32, 32]
 *   NF    any of s [d_out], b [d_out], R, and one owned term A, B, rank, c with
 *         optional d [rank] and e [d_out]
 * Layers of an adapter that are not listed get identity slots (n_layers may
 * be 0: the adapter then leaves every layer unchanged). */
typedef struct {
    int layer;
    int rank;
    float c;
    const void *A;
    const void *B;
    const float *d;
    const float *e;
    const float *s;
    const float *b;
    const void *R;
    const float *magnitude;
    const float *l;
} scute_layer_tensors;

/* Register an adapter: validate, copy to the device and apply the fold rule
 * (article, "Which slots can be merged at load?" and "How does Scute plug
 * into vLLM?"):
 *   - c and d of an owned term go into A:  A' = c A diag(d);
 *   - e of an owned term goes into B:      B' = B diag(e);
 *   - DoRA: s = m / ||column of (W + cAB)|| (L2 over d_in, accumulated in
 *     float64) stays live on the base path, and the same factor is folded into
 *     B as its e;  a zero column norm returns SCUTE_ERR_ARG;
 *   - (IA)^3: l becomes the live s slot;
 *   - VeRA: d and e stay live next to the shared pair;
 *   - OFT: the blocks of R stay live (they sit next to W).
 * Writes the new adapter id (lowest free id) to *adapter_id_out.
 * Errors: SCUTE_ERR_ARG (bad method / missing tensor / unknown layer / no free
 * id), SCUTE_ERR_SHAPE, SCUTE_ERR_UNSUPPORTED (rank > SCUTE_MAX_RANK, or R
 * combined with a VeRA term), SCUTE_ERR_OOM.  On error nothing is registered. */
scute_status scute_register_adapter(scute_ctx *ctx, scute_method method,
                                    const scute_layer_tensors *t, int n_layers,
                                    int32_t *adapter_id_out);

/* Remove an adapter and free its tensors.  Synchronises the device first, so
 * no in-flight call can still read them.  Its id becomes free. */
scute_status scute_unregister_adapter(scute_ctx *ctx, int32_t adapter_id);

/* The adapted linear layer for a heterogeneous batch (the hot path).
 *   x            device [n, d_in], context dtype;
 *   adapter_ids  device int32 [n]; -1 = base only.  An id that names no
 *                registered adapter is treated as -1 and recorded as
 *                SCUTE_ERR_BAD_ADAPTER in the status word;
 *   n            0..max_tokens (n = 0 returns SCUTE_OK without launching);
 *   out          device [n, d_out] in out_dtype (FP32 or, for a bf16 context,
 *                BF16); overwritten.
 *   stream       a cudaStream_t (NULL = legacy default stream).
 * Steps, all on the device: token indexing (stable grouping by method and
 * adapter id), the OFT input rotation into a workspace copy of x, the base
 * GEMM on tcgen05 tensor cores with the s / b epilogue gathered by adapter,
 * the owned low-rank shrink and expand, and the VeRA shared-pair GEMMs.  A
 * decode batch (bf16 context, n <= 128) runs all of them in one persistent
 * launch (scute_linear_batch with one call).
 * Returns after enqueueing; x, adapter_ids and out must stay valid until the
 * stream reaches the call. */
scute_status scute_linear(scute_ctx *ctx, const void *x, const int32_t *adapter_ids, int64_t n,
                          int layer, void *out, scute_dtype out_dtype, void *stream);

/* scute_linear with HOST buffers: copies x and adapter_ids from host memory
 * into context-owned device staging, runs scute_linear and copies `out` back,
 * all enqueued on `stream`; a bf16-context batch of at most 128 tokens stores
 * into a pinned, mapped, 16-byte-aligned `out_host` directly (unless the
 * separate s pass of scute_set_variant is on).  Pinned host memory keeps it
 * asynchronous; the caller synchronises the stream before reading
 * `out_host`. */
scute_status scute_linear_host(scute_ctx *ctx, const void *x_host, const int32_t *ids_host,
                               int64_t n, int layer, void *out_host, scute_dtype out_dtype,
                               void *stream);

/* Several layers over the same tokens in one call: for each i < n_calls,
 * calls[i].out receives the adapted layer calls[i].layer applied to
 * calls[i].x, all with the one adapter_ids vector (the projections of a
 * transformer block that read the same batch, such as q, k and v, or gate and
 * up).  The results are those of n_calls scute_linear calls up to the order of
 * floating-point sums.
 *   calls    HOST array of n_calls entries (0..SCUTE_MAX_CALLS); each x and out
 *            as for scute_linear (device, 16-byte aligned); an out may not
 *            overlap any call's x or out.  A layer may appear more than once.
 * A decode batch (bf16 context, n <= 128) runs as ONE persistent cooperative
 * launch that streams every listed layer's weights once, split over all SMs
 * in contiguous runs of 64-wide K blocks (section "Where is the cheapest place
 * to compute the remaining slots?" of the article prices the extra slots in
 * bytes moved; this launch keeps the one large byte stream, the base weights,
 * continuous).  Other batches run the calls one after another.  Errors as for
 * scute_linear; nothing is enqueued when an argument is rejected.  Calls on one
 * context must be ordered on the device (they share its workspace). */
#define SCUTE_MAX_CALLS 8
typedef struct scute_call {
    const void *x;   /* [n, d_in of layer] */
    int layer;
    void *out;       /* [n, d_out of layer] */
} scute_call;
scute_status scute_linear_batch(scute_ctx *ctx, const scute_call *calls, int n_calls,
                                const int32_t *adapter_ids, int64_t n, scute_dtype out_dtype,
                                void *stream);

/* scute_linear_batch with HOST buffers (every x and out, and adapter_ids, in
 * host memory): the inputs are copied into context-owned device staging, the
 * batch runs, the outputs are copied back, all enqueued on `stream`.  When
 * every input buffer is pinned and mapped, one kernel launch moves all of
 * them through their device addresses; otherwise each is one asynchronous
 * copy.  A bf16-context batch of at most 128 tokens whose output buffers are
 * all pinned, mapped and 16-byte aligned has its outputs stored straight
 * into them by the step (unless the separate s pass of scute_set_variant is
 * on); other pinned, mapped outputs take one scatter launch after the batch,
 * and any other output one copy each.  The caller synchronises the stream
 * before reading the outputs. */
scute_status scute_linear_batch_host(scute_ctx *ctx, const scute_call *calls, int n_calls,
                                     const int32_t *ids_host, int64_t n, scute_dtype out_dtype,
                                     void *stream);

/* Synchronise the device and return (then clear) the device status word:
 * SCUTE_OK, SCUTE_ERR_BAD_ADAPTER or SCUTE_ERR_TIMEOUT (timeout wins). */
scute_status scute_sync_status(scute_ctx *ctx);

/* Token indexing alone, for inspection.  Runs the same kernel scute_linear
 * runs and copies its results into caller device buffers on `stream`:
 *   perm       int32 [n]     sorted position -> token index;
 *   aid_sorted int32 [n]     adapter of each sorted row (-1 = base);
 *   seg_start  int32 [n + 1] first sorted row of each segment, then n;
 *   seg_aid    int32 [n]     adapter of each segment;
 *   counts     int32 [22]    n_seg, rows per method (7: LoRA, DoRA, (IA)^3,
 *                            VeRA, OFT, NF, base), first row per method (7),
 *                            segments per method (7).
 * Only the first n_seg entries of seg_aid and n_seg + 1 of seg_start are set. */
scute_status scute_debug_index(scute_ctx *ctx, const int32_t *adapter_ids, int64_t n,
                               int32_t *perm, int32_t *aid_sorted, int32_t *seg_start,
                               int32_t *seg_aid, int32_t *counts, void *stream);

/* ---------------------------------------------------------------- token indexing without a context
 * The article has no counterpart of this call: it is a service of this
 * library for callers that cannot allocate device memory.  Typical ones: a
 * batch scheduler or router in a process whose serving engine has already
 * reserved its device memory pool (most of HBM goes to the KV cache), where a
 * new allocation fails or takes memory the pool counts on; and code on a
 * latency-critical path, where cudaMalloc and cudaFree may synchronise the
 * device.  Such callers still want the adapter segments a batch forms, but
 * cannot create a context (scute_create allocates its workspaces).
 *
 * Runs the kernel scute_debug_index runs, on the CURRENT device and `stream`,
 * with the same outputs (perm, aid_sorted, seg_start, seg_aid, counts: layout
 * as for scute_debug_index; all device buffers of the caller), and
 *   method_of_adapter  HOST int8 [n_adapters]: the scute_method of each
 *                      adapter id, or -1 where the id names no adapter;
 *                      copied with cudaMemcpyAsync (pageable memory may be
 *                      reused when the call returns; pinned memory must stay
 *                      unchanged until the stream has passed the call);
 *   flags              device int32 [1] or NULL: nonzero when an id in
 *                      adapter_ids named no adapter (those tokens become
 *                      base-only rows, as in scute_linear).
 * Scratch: a file-scope device array of SCUTE_NOALLOC_SCRATCH_BYTES (the method
 * table and a status word), located once per device with cudaGetSymbolAddress
 * on the first call made while that device is current.  That first call may
 * load the library's module, so make it before any stream capture.  The
 * address is kept for the life of the process: do not use this call on a
 * device after cudaDeviceReset (or any teardown of its primary context) in
 * the same process.  Nothing
 * is allocated: no cudaMalloc, cudaFree or allocating library routine.
 * Overlapping calls on one device (other streams, other host threads) share
 * the array and race; order them on the device.
 * Errors (nothing is launched): SCUTE_ERR_ARG for a null output, n < 0,
 * n_adapters < 1 or a method code outside -1..5; SCUTE_ERR_UNSUPPORTED for
 * n > SCUTE_MAX_TOKENS or n_adapters > SCUTE_NOALLOC_MAX_ADAPTERS (the static
 * table's size); SCUTE_ERR_NO_DEVICE when the current device is not sm_103;
 * SCUTE_ERR_CUDA when a CUDA call fails. */
#define SCUTE_NOALLOC_MAX_ADAPTERS 8192
#define SCUTE_NOALLOC_SCRATCH_BYTES (256 + SCUTE_NOALLOC_MAX_ADAPTERS)
scute_status scute_index_tokens_noalloc(const int8_t *method_of_adapter, int32_t n_adapters,
                                        const int32_t *adapter_ids, int64_t n, int32_t *perm,
                                        int32_t *aid_sorted, int32_t *seg_start, int32_t *seg_aid,
                                        int32_t *counts, int32_t *flags, void *stream);

/* ---------------------------------------------------------------- byte model
 * Zero-parameter byte and time model (article, section "Where is the cheapest
 * place to compute the remaining slots?": added time = extra bytes / memory
 * bandwidth + extra launches x launch cost; bytes are what adapter work is
 * measured in).
 *
 * For one call it lists every kernel launch the library makes for it, with the
 * bytes that launch must move to and from device memory (each operand read
 * once, each result written once; intermediates a launch keeps to itself are
 * not counted: a lower bound that measured DRAM bytes are compared against)
 * and its floating-point operations, plus the call's algorithmic bytes: W once,
 * each distinct adapter's live (post-fold) tensors once, the shared VeRA pair
 * once when a VeRA token is present, x read, out written and the ids read.
 * Launch plans: a bf16 batch of at most 128 tokens is ONE launch ("step") over
 * every layer of the call, with "oft_pass" before it and "s_pass" after it
 * when the variant flags place those slots in passes of their own
 * (scute_set_variant; the step's own bytes then lose R, or the DoRA and
 * (IA)^3 s vectors); otherwise each layer takes the per-kernel plan
 * ("index", "rotate", "base_gemm", "lr_shrink", "lr_expand", "vera_shrink",
 * "vera_expand"; in a bf16 context above 256 tokens "lr_shrink" and, for a
 * shared rank that is a multiple of 64, "vera_shrink" come before
 * "base_gemm", which takes in the owned expand).  Pure host arithmetic: no device work, no context needed for
 * scute_byte_model and scute_byte_model_batch. */
#define SCUTE_BM_MAX_KERNELS 64
typedef struct {
    int n_kernels;                          /* launches of the call            */
    char name[SCUTE_BM_MAX_KERNELS][24];    /* kernel names                    */
    int64_t bytes[SCUTE_BM_MAX_KERNELS];    /* bytes read + written per launch */
    int64_t flops[SCUTE_BM_MAX_KERNELS];    /* 2 x multiply-adds per launch    */
    int64_t algorithmic_bytes;              /* minimal bytes of the call       */
    int64_t adapter_bytes;                  /* live adapter tensors + shared pair */
    int64_t base_weight_bytes;              /* W                               */
    int32_t distinct_adapters;              /* distinct valid ids in the batch */
} scute_byte_report;

/* One registered adapter as the byte model sees one layer of it.
 * method = -1 marks an unregistered id. */
typedef struct {
    int method;
    int rank;          /* owned low-rank rank on this layer (0 = none) */
    int has_s, has_b, has_R, has_vera, has_vera_e;
} scute_bm_adapter;

typedef struct {
    scute_dtype dtype;        /* context dtype                                 */
    scute_dtype out_dtype;
    int d_in, d_out;
    int shared_rank;          /* 0 = no shared VeRA pair                       */
    int lowrank_launched;     /* the per-kernel plan launches the owned-term kernels */
    int vera_launched;        /* the per-kernel plan launches the VeRA kernels */
    int max_adapters;
    const scute_bm_adapter *adapters;  /* [max_adapters]                       */
    int variant;              /* SCUTE_VARIANT_* flags of the call (0: none)   */
} scute_bm_layer;

/* One call of one layer (scute_linear). */
scute_status scute_byte_model(const scute_bm_layer *layer, const int32_t *ids_host, int64_t n,
                              scute_byte_report *rep);

/* One batched call (scute_linear_batch) over n_layers (1..SCUTE_MAX_CALLS)
 * layers that read the same ids; all in one dtype.  SCUTE_ERR_UNSUPPORTED when
 * the per-kernel plan needs more than SCUTE_BM_MAX_KERNELS launches. */
scute_status scute_byte_model_batch(const scute_bm_layer *layers, int n_layers, const int32_t *ids_host,
                                    int64_t n, scute_byte_report *rep);

/* The same for layer `layer` of a context, from its registered adapters. */
scute_status scute_predict_bytes(const scute_ctx *ctx, const int32_t *ids_host, int64_t n,
                                 int layer, scute_dtype out_dtype, scute_byte_report *rep);

/* The same for a batched call of a context (only calls[i].layer is read). */
scute_status scute_predict_batch(const scute_ctx *ctx, const scute_call *calls, int n_calls,
                                 const int32_t *ids_host, int64_t n, scute_dtype out_dtype,
                                 scute_byte_report *rep);

/* Predicted time of a launch list, in microseconds:
 *     sum over launches of max(bytes / hbm_gbs, flops / tensor_tflops)
 *     + launches x launch_us.
 * With tensor_tflops <= 0 the flops term is dropped and this is the article's
 * model as it stands (bytes / bandwidth + launches x launch cost); the flops
 * term extends it to launches bound by the tensor cores (prefill GEMMs).  The
 * three constants are measured on the device, never fitted. */
scute_status scute_predict_time(const scute_byte_report *rep, double hbm_gbs, double tensor_tflops,
                                double launch_us, double *us_out);

/* ---------------------------------------------------------------- counters
 * Device kernels enqueued by this context since creation. */
int64_t scute_launch_count(const scute_ctx *ctx);

/* Kernel timing with CUDA events on the launching stream.  While enabled,
 * every launch of the hot path (the decode step; or, on the per-kernel plan,
 * the indexing, rotation, base GEMM, low-rank shrink + expand pair and the two
 * VeRA GEMMs) is bracketed by an event pair, stored in a ring of
 * `SCUTE_TIMING_SLOTS` slots in launch order and tagged with its kind
 * (SCUTE_KIND_*).  Event records made during stream capture become graph
 * nodes and are re-recorded on every replay.  Timing puts an event record
 * between launches that would otherwise overlap their start and end
 * (programmatic dependent launch), so a timed call can be slightly slower.
 * scute_timing_read synchronises the device and writes the elapsed
 * milliseconds of the first `max` used slots; scute_timing_kinds writes their
 * kinds. */
#define SCUTE_TIMING_SLOTS 256
enum {
    SCUTE_KIND_STEP = 0,         /* the batched decode step (one launch)       */
    SCUTE_KIND_INDEX = 1,        /* token indexing                             */
    SCUTE_KIND_ROTATE = 2,       /* OFT rotation / gather of the token operand */
    SCUTE_KIND_BASE_GEMM = 3,    /* base GEMM with the s / b epilogue          */
    SCUTE_KIND_LOWRANK = 4,      /* owned low-rank shrink and expand (2 launches) */
    SCUTE_KIND_VERA_SHRINK = 5,  /* VeRA shared shrink GEMM                    */
    SCUTE_KIND_VERA_EXPAND = 6,  /* VeRA shared expand GEMM                    */
    SCUTE_KIND_OFT_PASS = 7,     /* rotation as its own pass (scute_set_variant) */
    SCUTE_KIND_S_PASS = 8        /* s as its own pass (scute_set_variant)      */
};
scute_status scute_timing_enable(scute_ctx *ctx, int enable);
scute_status scute_timing_reset(scute_ctx *ctx);
scute_status scute_timing_read(scute_ctx *ctx, float *ms_out, int max, int *n_out);
scute_status scute_timing_kinds(const scute_ctx *ctx, int *kinds_out, int max, int *n_out);

/* Test hook for the failure path (no counterpart in the article).  With
 * what = SCUTE_INJECT_STALL, the context's next decode launch (bf16, n <= 128)
 * waits for a count that no CTA ever reaches: its bounded waits run out (about
 * 2 s), every CTA drains what it issued, frees TMEM and returns, and
 * scute_sync_status then reports SCUTE_ERR_TIMEOUT.  The context stays usable;
 * the hook applies to that one launch only.  Nothing traps or faults. */
#define SCUTE_INJECT_STALL 1
scute_status scute_debug_inject(scute_ctx *ctx, int what);

/* Separate-pass placements of two live slots, for validating the byte and
 * time model (article, section "Where is the cheapest place to compute the
 * remaining slots?": the model is checked there on OFT's input rotation and
 * on applying DoRA's s outside the expand).  With flags = 0 (the default) the
 * decode step applies every slot inside its one launch.  Otherwise a bf16
 * decode batch (n <= 128) of this context adds, around its step launch:
 *   SCUTE_VARIANT_OFT_PASS  one launch before the step that writes x R for
 *                           the rotated tokens (x for the others) into a
 *                           context-owned copy, which the step then reads;
 *   SCUTE_VARIANT_S_PASS    one launch after the step that multiplies the
 *                           output rows of DoRA and (IA)^3 tokens by their s,
 *                           which the step then leaves out (DoRA expanding
 *                           with B' whose s is not folded in).
 * Results stay those of the normal form up to rounding order.  Other batches
 * (fp32 contexts, more than 128 tokens) ignore the flags.  A setup call:
 * SCUTE_VARIANT_OFT_PASS allocates the rotated-copy workspace here, so do not
 * make it during stream capture.  scute_predict_batch describes the launches
 * of the flags in force. */
#define SCUTE_VARIANT_OFT_PASS 1
#define SCUTE_VARIANT_S_PASS 2
scute_status scute_set_variant(scute_ctx *ctx, int flags);

/* Test hook for the out-of-memory path (no counterpart in the article).  The
 * k-th device allocation the library makes after this call (counted over
 * every context of the process) fails as if the device were out of memory:
 * nothing is allocated for it and the call that needed it returns
 * SCUTE_ERR_OOM, having freed what it had allocated itself and leaving the
 * context as it was.  k <= 0 switches the hook off.  Host-side only: no
 * device work is involved. */
void scute_debug_fail_alloc(int k);

/* The plan of the context's last decode-step launch (the host values that
 * launch was given), so that the kernel's index arithmetic can be checked
 * against its buffers on the host.  The article has no counterpart.  Writes at
 * most `cap` int64 values to the HOST array `out`:
 *   SCUTE_PLAN_HEAD values: n_calls, n, bn (tokens per tile), stages, grid,
 *     n_units (VeRA shrink units), vs_ch (K blocks per unit), n_tiles,
 *     n_items (low-rank shrink items), rmax, t_main (main K blocks), hold,
 *     smem_bytes (before the one-CTA-per-SM floor), smem_optin,
 *     part_floats (partial-tile workspace), xs_cols and u_cols (row pitch of
 *     the token-operand and VeRA-intermediate slots), sync_ints, pre_floats
 *     (the owned low-rank rows b + v B', all call slots);
 *   then SCUTE_PLAN_CALL_FIELDS values per call: blk0, d_in, kdim, d_out,
 *     krv, rv, kblocks, vkb, n_ft, n_vt, vs_chunks, vs_unit0, tile0, lr_rmax,
 *     lr_items, lr_item0, vs_x, xs_direct;
 *   then grid + 1 values: the stream-K range bounds start[0..grid].
 * *n_out = the number of values the plan has (only the first cap written).
 * SCUTE_ERR_ARG when no decode step has been launched on the context. */
#define SCUTE_PLAN_HEAD 19
#define SCUTE_PLAN_CALL_FIELDS 18
scute_status scute_debug_step_plan(const scute_ctx *ctx, int64_t *out, int cap, int *n_out);

#ifdef __cplusplus
}
#endif
#endif /* SCUTE_H */
