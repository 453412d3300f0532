// Host runtime of libscute.so: contexts, layers, adapter registration with the
// fold rule, the per-call launch plan of the adapted linear layer, the byte
// model and the timing counters.  See include/scute.h for the contract.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ctx.h"

using namespace scute;

namespace {

scute_status fail(scute_ctx *c, scute_status s, const char *fmt, ...) {
    if (c) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(c->err, sizeof(c->err), fmt, ap);
        va_end(ap);
    }
    return s;
}

#define CU_TRY(ctx, expr)                                                                      \
    do {                                                                                       \
        cudaError_t _e = (expr);                                                               \
        if (_e != cudaSuccess) {                                                               \
            (void)cudaGetLastError();                                                          \
            if (_e == cudaErrorMemoryAllocation)                                               \
                return fail(ctx, SCUTE_ERR_OOM, "%s: %s", #expr, cudaGetErrorString(_e));      \
            return fail(ctx, SCUTE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e));         \
        }                                                                                      \
    } while (0)

// Keeps the context's device current for the duration of one API call.
struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            if (cudaSetDevice(dev) == cudaSuccess) changed = true;
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

// Test hook scute_debug_fail_alloc: while positive, counts the library's
// device allocations down; the allocation that brings it from 1 to 0 fails as
// if the device were out of memory (nothing is allocated for it).
std::atomic<int> g_fail_alloc{0};

cudaError_t dev_malloc(void **p, size_t bytes) {
    int k = g_fail_alloc.load();
    while (k > 0) {
        if (g_fail_alloc.compare_exchange_weak(k, k - 1)) {
            if (k == 1) {
                *p = nullptr;
                return cudaErrorMemoryAllocation;
            }
            break;
        }
    }
    return cudaMalloc(p, bytes);
}

bool encode_map_box(scute_ctx *c, CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, int box_rows);

bool encode_map(scute_ctx *c, CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows) {
    return encode_map_box(c, m, base, inner, rows, 64);
}

bool encode_map_box(scute_ctx *c, CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, int box_rows) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * (uint64_t)c->esz};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / c->esz), (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = c->encode(m, c->esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

scute_status grow(scute_ctx *c, void **buf, size_t *cols, size_t need_cols, size_t elem_bytes,
                  size_t rows) {
    if (need_cols <= *cols) return SCUTE_OK;
    void *p = nullptr;
    CU_TRY(c, cudaDeviceSynchronize());
    CU_TRY(c, dev_malloc(&p, need_cols * elem_bytes * rows));
    const cudaError_t e = cudaMemset(p, 0, need_cols * elem_bytes * rows);
    if (e != cudaSuccess) {
        cudaFree(p);
        CU_TRY(c, e);
    }
    if (*buf) cudaFree(*buf);
    *buf = p;
    *cols = need_cols;
    return SCUTE_OK;
}

// The decode step's owned low-rank rows b + v B': every call slot holds
// ceil(largest owned rank / 8) planes of STEP_MAX_TOKENS rows of the widest
// layer's d_out (fp32).  extra_rank: the rank of an adapter being registered.
static scute_status grow_pre(scute_ctx *c, int extra_rank) {
    if (c->dtype != SCUTE_BF16) return SCUTE_OK;   // fp32 contexts never run the decode step
    int max_dout = 0, max_rank = extra_rank;
    for (const auto &L : c->layers)
        if (L.present && L.d_out > max_dout) max_dout = L.d_out;
    for (const auto &a : c->adapters)
        if (a.used)
            for (const auto &al : a.layers)
                if (al.rank > max_rank) max_rank = al.rank;
    if (max_dout == 0 || max_rank == 0) return SCUTE_OK;
    const size_t need = (size_t)STEP_MAX_CALLS * (size_t)((max_rank + 7) / 8) * STEP_MAX_TOKENS * (size_t)max_dout;
    void *p = c->step_pre;
    const scute_status st = grow(c, &p, &c->step_pre_floats, need, sizeof(float), 1);
    c->step_pre = reinterpret_cast<float *>(p);
    return st;
}

scute_status remap_workspace(scute_ctx *c) {
    for (auto &L : c->layers) {
        if (!L.present) continue;
        if (!encode_map(c, &L.mapXs, c->xs, (uint64_t)L.kdim, (uint64_t)c->max_tokens))
            return fail(c, SCUTE_ERR_CUDA, "tensor map for the token operand failed");
        if (L.rv && !encode_map(c, &L.mapU, c->U, (uint64_t)L.krv, (uint64_t)c->max_tokens))
            return fail(c, SCUTE_ERR_CUDA, "tensor map for the VeRA intermediate failed");
    }
    return SCUTE_OK;
}

scute_status ensure_tmp(scute_ctx *c, size_t bytes) {
    if (bytes <= c->tmp_bytes) return SCUTE_OK;
    CU_TRY(c, cudaDeviceSynchronize());
    if (c->tmp) cudaFree(c->tmp);
    c->tmp = nullptr;
    c->tmp_bytes = 0;
    CU_TRY(c, dev_malloc(&c->tmp, bytes));
    c->tmp_bytes = bytes;
    return SCUTE_OK;
}

bool layer_ok(const scute_ctx *c, int layer) {
    return layer >= 0 && layer < c->max_layers && c->layers[layer].present;
}

void count_launch(scute_ctx *c, int k) { c->launches += k; }

// Timing ring (scute_timing_*): while enabled, every launch (or launch pair)
// of the hot path is bracketed by an event pair on its stream, tagged with its
// kind.  Event records made while the stream is being captured become graph
// nodes, re-recorded on every replay.
// The device address of a pinned, mapped host buffer (null for pageable
// memory, device memory, or any pointer the runtime does not know).
const void *mapped_host(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

struct TimedLaunch {
    scute_ctx *c;
    cudaStream_t st;
    int slot = -1;
    unsigned flags = cudaEventRecordDefault;
    cudaError_t begin() {
        if (!c->timing) return cudaSuccess;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(st, &cs);
        if (e != cudaSuccess) return e;
        if (cs == cudaStreamCaptureStatusActive) flags = cudaEventRecordExternal;
        slot = c->t_next;
        return cudaEventRecordWithFlags(c->ev[slot][0], st, flags);
    }
    cudaError_t end(int kind) {
        if (!c->timing || slot < 0) return cudaSuccess;
        const cudaError_t e = cudaEventRecordWithFlags(c->ev[slot][1], st, flags);
        c->ev_kind[slot] = kind;
        c->t_next = (slot + 1) % SCUTE_TIMING_SLOTS;
        if (c->t_used < SCUTE_TIMING_SLOTS) ++c->t_used;
        slot = -1;
        return e;
    }
};

}  // namespace

extern "C" {

int scute_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char *scute_last_error(const scute_ctx *ctx) { return ctx ? ctx->err : "null context"; }

scute_status scute_create(scute_ctx **out, int device, scute_dtype dtype, int max_tokens,
                          int max_adapters, int max_layers) {
    if (!out) return SCUTE_ERR_ARG;
    *out = nullptr;
    if (dtype != SCUTE_BF16 && dtype != SCUTE_FP32) return SCUTE_ERR_DTYPE;
    if (max_tokens < 1 || max_tokens > SCUTE_MAX_TOKENS || max_adapters < 1 ||
        max_adapters > SCUTE_MAX_ADAPTERS || max_layers < 1 || max_layers > (1 << 20))
        return SCUTE_ERR_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return SCUTE_ERR_NO_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return SCUTE_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return SCUTE_ERR_NO_DEVICE;  // kernels are built for sm_103a
    scute_ctx *c = new scute_ctx();
    c->err[0] = 0;
    c->device = device;
    c->dtype = dtype;
    c->esz = dtype == SCUTE_BF16 ? 2 : 4;
    c->max_tokens = max_tokens;
    c->max_adapters = max_adapters;
    c->max_layers = max_layers;
    c->num_sms = prop.multiProcessorCount;
    c->layers.resize(max_layers);
    c->adapters.resize(max_adapters);
    c->h_method.assign(max_adapters, (int8_t)-1);
    DeviceGuard dg(device);
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        delete c;
        return SCUTE_ERR_NO_DEVICE;
    }
    c->encode = reinterpret_cast<PFN_encodeTiled>(fn);
    const size_t nslots = (size_t)max_layers * max_adapters;
    bool ok = dev_malloc((void **)&c->d_slots, nslots * sizeof(Slot)) == cudaSuccess &&
              cudaMemset(c->d_slots, 0, nslots * sizeof(Slot)) == cudaSuccess &&
              dev_malloc((void **)&c->d_method, max_adapters) == cudaSuccess &&
              cudaMemset(c->d_method, 0xFF, max_adapters) == cudaSuccess &&
              dev_malloc((void **)&c->d_perm, sizeof(int) * max_tokens) == cudaSuccess &&
              dev_malloc((void **)&c->d_aid, sizeof(int) * max_tokens) == cudaSuccess &&
              dev_malloc((void **)&c->d_seg_start, sizeof(int) * (max_tokens + 1)) == cudaSuccess &&
              dev_malloc((void **)&c->d_seg_aid, sizeof(int) * max_tokens) == cudaSuccess &&
              dev_malloc((void **)&c->d_seg_unit, sizeof(int) * (max_tokens + 1)) == cudaSuccess &&
              dev_malloc((void **)&c->d_seg_tile, sizeof(int) * (max_tokens + 1)) == cudaSuccess &&
              dev_malloc((void **)&c->vs_ctr, sizeof(int) * VS_CTR_INTS) == cudaSuccess &&
              cudaMemset(c->vs_ctr, 0, sizeof(int) * VS_CTR_INTS) == cudaSuccess &&
              dev_malloc((void **)&c->d_meta, sizeof(IndexMeta)) == cudaSuccess &&
              cudaMemset(c->d_meta, 0, sizeof(IndexMeta)) == cudaSuccess &&
              dev_malloc((void **)&c->d_status, sizeof(int)) == cudaSuccess &&
              cudaMemset(c->d_status, 0, sizeof(int)) == cudaSuccess &&
              dev_malloc((void **)&c->d_err, sizeof(int)) == cudaSuccess &&
              dev_malloc((void **)&c->v_part, sizeof(float) * KS_MAX * (size_t)max_tokens * MAX_RANK) == cudaSuccess &&
              dev_malloc((void **)&c->st_ids, sizeof(int32_t) * max_tokens) == cudaSuccess &&
              dev_malloc((void **)&c->gpart, sizeof(float) * PART_WORKSPACE_FLOATS) == cudaSuccess &&
              dev_malloc((void **)&c->step_sync, sizeof(int) * STEP_SYNC_INTS) == cudaSuccess &&
              cudaMemset(c->step_sync, 0, sizeof(int) * STEP_SYNC_INTS) == cudaSuccess &&
              cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) ==
                  cudaSuccess;
    c->step_bn_max = max_tokens <= 64 ? 64 : 128;
    if (!ok) {
        scute_destroy(c);
        return SCUTE_ERR_OOM;
    }
    *out = c;
    return SCUTE_OK;
}

void scute_destroy(scute_ctx *c) {
    if (!c) return;
    DeviceGuard dg(c->device);
    cudaDeviceSynchronize();
    for (auto &L : c->layers) {
        if (L.Wt) cudaFree(L.Wt);
        if (L.Ash) cudaFree(L.Ash);
        if (L.Bsh) cudaFree(L.Bsh);
    }
    for (auto &a : c->adapters)
        if (a.storage) cudaFree(a.storage);
    void *bufs[] = {c->d_slots, c->d_method, c->d_perm, c->d_aid, c->d_seg_start, c->d_seg_aid, c->d_seg_unit, c->d_seg_tile, c->vs_ctr, c->vs_part,
                    c->d_meta, c->d_status, c->d_err, c->v_part, c->gpart, c->xs, c->U, c->st_x,
                    c->st_out, c->st_ids, c->tmp, c->step_xs, c->step_U, c->step_pre, c->step_part,
                    c->step_sync, c->step_hx, c->step_hout, c->var_x};
    for (void *p : bufs)
        if (p) cudaFree(p);
    if (c->ev_made)
        for (int i = 0; i < SCUTE_TIMING_SLOTS; ++i) {
            cudaEventDestroy(c->ev[i][0]);
            cudaEventDestroy(c->ev[i][1]);
        }
    delete c;
}

scute_status scute_add_layer(scute_ctx *c, int layer, int d_in, int d_out, const void *W) {
    if (!c || !W) return fail(c, SCUTE_ERR_ARG, "null argument");
    if (layer < 0 || layer >= c->max_layers) return fail(c, SCUTE_ERR_ARG, "layer id %d out of range", layer);
    if (c->layers[layer].present) return fail(c, SCUTE_ERR_ARG, "layer %d already exists", layer);
    if (d_in <= 0 || d_out <= 0 || d_in % 32 || d_out % 32)
        return fail(c, SCUTE_ERR_SHAPE, "d_in and d_out must be positive multiples of 32");
    DeviceGuard dg(c->device);
    const bool f32 = c->dtype == SCUTE_FP32;
    LayerRec L;
    L.present = true;
    L.d_in = d_in;
    L.d_out = d_out;
    L.kdim = f32 ? 3 * d_in : d_in;
    scute_status st = ensure_tmp(c, (size_t)d_in * d_out * c->esz);
    if (st) return st;
    CU_TRY(c, dev_malloc(&L.Wt, (size_t)d_out * L.kdim * c->esz));
    {
        cudaError_t e = cudaMemcpy(c->tmp, W, (size_t)d_in * d_out * c->esz, cudaMemcpyDefault);
        if (e == cudaSuccess) e = launch_transpose_w(f32, c->tmp, d_in, d_out, L.Wt, L.kdim, f32 ? 1 : 0, 0);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(L.Wt);
            CU_TRY(c, e);
        }
    }
    if (!encode_map(c, &L.mapW, L.Wt, (uint64_t)L.kdim, (uint64_t)d_out)) {
        cudaFree(L.Wt);
        return fail(c, SCUTE_ERR_CUDA, "tensor map for W failed");
    }
    c->layers[layer] = L;
    // workspace: token operand, host-call staging
    const size_t old_xs = c->xs_cols;
    st = grow(c, &c->xs, &c->xs_cols, (size_t)L.kdim, c->esz, c->max_tokens);
    if (!st) st = grow(c, &c->st_x, &c->st_x_cols, (size_t)d_in, c->esz, c->max_tokens);
    if (!st) st = grow(c, &c->st_out, &c->st_out_cols, (size_t)d_out, 4, c->max_tokens);
    if (!st && !f32) {
        // decode-step slots, host-call staging and partial tiles
        const size_t rows = (size_t)STEP_MAX_CALLS * STEP_MAX_TOKENS;
        st = grow(c, &c->step_xs, &c->step_xs_cols, (size_t)L.kdim, c->esz, rows);
        if (!st) st = grow(c, &c->step_hx, &c->step_hx_cols, (size_t)d_in, c->esz, rows);
        if (!st) st = grow(c, &c->step_hout, &c->step_hout_cols, (size_t)d_out, 4, rows);
        if (!st && (c->variant & VARIANT_OFT_PASS)) st = grow(c, &c->var_x, &c->var_x_cols, (size_t)d_in, c->esz, rows);
        int max_ft = 0;
        for (const auto &Lr : c->layers)
            if (Lr.present && (Lr.d_out + 127) / 128 > max_ft) max_ft = (Lr.d_out + 127) / 128;
        const int G = c->num_sms < STEP_MAX_GRID ? c->num_sms : STEP_MAX_GRID;
        const size_t slots = (size_t)2 * G + (size_t)STEP_MAX_CALLS * max_ft;
        void *pp = c->step_part;
        if (!st) st = grow(c, &pp, &c->step_part_floats, slots * 2 * 128 * c->step_bn_max, 4, 1);
        c->step_part = reinterpret_cast<float *>(pp);
        if (!st) st = grow_pre(c, 0);
    }
    if (st) {
        // the layer is not added; buffers that did grow have moved, so the
        // other layers' tensor maps are refreshed before returning
        cudaFree(c->layers[layer].Wt);
        c->layers[layer] = LayerRec();
        remap_workspace(c);
        return st;
    }
    (void)old_xs;
    return remap_workspace(c);
}

scute_status scute_set_shared(scute_ctx *c, int layer, int rank, const void *A_sh, const void *B_sh) {
    if (!c || !A_sh || !B_sh) return fail(c, SCUTE_ERR_ARG, "null argument");
    if (!layer_ok(c, layer)) return fail(c, SCUTE_ERR_ARG, "unknown layer %d", layer);
    if (rank <= 0 || rank % 32 || rank > SCUTE_MAX_SHARED_RANK)
        return fail(c, SCUTE_ERR_SHAPE, "shared rank must be a positive multiple of 32, at most %d",
                    SCUTE_MAX_SHARED_RANK);
    LayerRec &L = c->layers[layer];
    if (L.rv) return fail(c, SCUTE_ERR_ARG, "layer %d already has a shared pair", layer);
    DeviceGuard dg(c->device);
    const bool f32 = c->dtype == SCUTE_FP32;
    const int krv = f32 ? 3 * rank : rank;
    size_t big = (size_t)L.d_in * rank;
    if ((size_t)rank * L.d_out > big) big = (size_t)rank * L.d_out;
    scute_status st = ensure_tmp(c, big * c->esz);
    if (st) return st;
    void *Ash = nullptr, *Bsh = nullptr;
    {
        cudaError_t e = dev_malloc(&Ash, (size_t)rank * L.kdim * c->esz);
        if (e == cudaSuccess) e = dev_malloc(&Bsh, (size_t)L.d_out * krv * c->esz);
        if (e == cudaSuccess) e = cudaMemcpy(c->tmp, A_sh, (size_t)L.d_in * rank * c->esz, cudaMemcpyDefault);
        if (e == cudaSuccess) e = launch_transpose_w(f32, c->tmp, L.d_in, rank, Ash, L.kdim, f32 ? 1 : 0, 0);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaMemcpy(c->tmp, B_sh, (size_t)rank * L.d_out * c->esz, cudaMemcpyDefault);
        if (e == cudaSuccess) e = launch_transpose_w(f32, c->tmp, rank, L.d_out, Bsh, krv, f32 ? 1 : 0, 0);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            if (Ash) cudaFree(Ash);
            if (Bsh) cudaFree(Bsh);
            CU_TRY(c, e);
        }
    }
    if (!encode_map(c, &L.mapAsh, Ash, (uint64_t)L.kdim, (uint64_t)rank) ||
        !encode_map(c, &L.mapBsh, Bsh, (uint64_t)krv, (uint64_t)L.d_out)) {
        cudaFree(Ash);
        cudaFree(Bsh);
        return fail(c, SCUTE_ERR_CUDA, "tensor map for the shared pair failed");
    }
    // the VeRA intermediates must hold the new rank before the layer uses it
    st = grow(c, &c->U, &c->u_cols, (size_t)krv, c->esz, c->max_tokens);
    if (!st && !f32) st = grow(c, &c->step_U, &c->step_u_cols, (size_t)krv, c->esz,
                               (size_t)STEP_MAX_CALLS * STEP_MAX_TOKENS);
    if (!st && !f32) {
        // partial tiles of the tensor-core VeRA shrink (prefill-sized batches)
        void *vp = c->vs_part;
        st = grow(c, &vp, &c->vs_part_cols, (size_t)rank, sizeof(float), (size_t)VS_KS * c->max_tokens);
        c->vs_part = reinterpret_cast<float *>(vp);
    }
    if (st) {
        cudaFree(Ash);
        cudaFree(Bsh);
        remap_workspace(c);   // U may have moved
        return st;
    }
    L.Ash = Ash;
    L.Bsh = Bsh;
    L.rv = rank;
    L.krv = krv;
    return remap_workspace(c);
}

scute_status scute_register_adapter(scute_ctx *c, scute_method method, const scute_layer_tensors *t,
                                    int n_layers, int32_t *id_out) {
    if (!c || !id_out || n_layers < 0 || (n_layers > 0 && !t)) return fail(c, SCUTE_ERR_ARG, "null argument");
    if (method < SCUTE_LORA || method > SCUTE_NF) return fail(c, SCUTE_ERR_ARG, "bad method %d", (int)method);
    int id = -1;
    for (int i = 0; i < c->max_adapters; ++i)
        if (!c->adapters[i].used) { id = i; break; }
    if (id < 0) return fail(c, SCUTE_ERR_ARG, "no free adapter id (max_adapters = %d)", c->max_adapters);
    const bool f32 = c->dtype == SCUTE_FP32;
    const size_t E = c->esz;

    // ---- validate and size
    size_t total = 0, tmp_need = 0;
    std::vector<AdapterLayer> info;
    for (int i = 0; i < n_layers; ++i) {
        const scute_layer_tensors &x = t[i];
        if (!layer_ok(c, x.layer)) return fail(c, SCUTE_ERR_ARG, "unknown layer %d", x.layer);
        for (int k = 0; k < i; ++k)
            if (t[k].layer == x.layer) return fail(c, SCUTE_ERR_ARG, "layer %d listed twice", x.layer);
        const LayerRec &L = c->layers[x.layer];
        AdapterLayer al{x.layer, 0, false, false, false, false, false};
        const bool owned = x.A || x.B;
        switch (method) {
            case SCUTE_LORA:
            case SCUTE_DORA:
                if (!x.A || !x.B) return fail(c, SCUTE_ERR_ARG, "LoRA/DoRA need A and B");
                if (method == SCUTE_DORA && !x.magnitude) return fail(c, SCUTE_ERR_ARG, "DoRA needs magnitude");
                al.rank = x.rank;
                al.s = method == SCUTE_DORA;
                break;
            case SCUTE_IA3:
                if (!x.l) return fail(c, SCUTE_ERR_ARG, "(IA)^3 needs l");
                al.s = true;
                break;
            case SCUTE_VERA:
                if (!x.d) return fail(c, SCUTE_ERR_ARG, "VeRA needs d");
                if (!L.rv) return fail(c, SCUTE_ERR_ARG, "layer %d has no shared VeRA pair", x.layer);
                al.vera = true;
                al.vera_e = x.e != nullptr;
                break;
            case SCUTE_OFT:
                if (!x.R) return fail(c, SCUTE_ERR_ARG, "OFT needs R");
                al.R = true;
                break;
            case SCUTE_NF:
                if (owned && (!x.A || !x.B)) return fail(c, SCUTE_ERR_ARG, "an owned term needs A and B");
                al.rank = owned ? x.rank : 0;
                al.s = x.s != nullptr;
                al.b = x.b != nullptr;
                al.R = x.R != nullptr;
                break;
        }
        if (al.rank < 0 || ((method == SCUTE_LORA || method == SCUTE_DORA || (method == SCUTE_NF && owned)) &&
                            al.rank < 1))
            return fail(c, SCUTE_ERR_SHAPE, "rank must be positive");
        if (al.rank > SCUTE_MAX_RANK)
            return fail(c, SCUTE_ERR_UNSUPPORTED, "rank %d above %d", al.rank, SCUTE_MAX_RANK);
        if (al.s) total += align256(4 * (size_t)L.d_out);
        if (al.b) total += align256(4 * (size_t)L.d_out);
        if (al.R) total += align256((size_t)L.d_in * OFT_BLK * E) * (c->dtype == SCUTE_BF16 ? 2 : 1);
        if (al.rank) {
            total += align256((size_t)al.rank * L.d_in * E) + align256((size_t)al.rank * L.d_out * E);
            if (c->dtype == SCUTE_BF16) total += align256(sizeof(CUtensorMap));   // A' map of the shrink
            // DoRA also keeps B' without its s (read only by the separate-s-pass placement)
            if (method == SCUTE_DORA) total += align256((size_t)al.rank * L.d_out * E);
            size_t need = align256((size_t)L.d_in * al.rank * E) + align256((size_t)al.rank * L.d_out * E) +
                          3 * align256(4 * (size_t)L.d_out) + align256(4 * (size_t)al.rank);
            if (need > tmp_need) tmp_need = need;
        }
        if (al.vera) {
            total += align256(4 * (size_t)L.rv) + align256(4 * (size_t)L.d_out);
            if (align256(4 * (size_t)L.rv) > tmp_need) tmp_need = align256(4 * (size_t)L.rv);
        }
        info.push_back(al);
    }
    DeviceGuard dg(c->device);
    scute_status st = ensure_tmp(c, tmp_need ? tmp_need : 256);
    if (st) return st;
    {
        int new_rank = 0;
        for (const auto &al : info)
            if (al.rank > new_rank) new_rank = al.rank;
        st = grow_pre(c, new_rank);
        if (st) return st;
    }
    void *storage = nullptr;
    CU_TRY(c, dev_malloc(&storage, total ? total : 256));
    uint8_t *cur = reinterpret_cast<uint8_t *>(storage);
    auto take = [&](size_t bytes) {
        void *p = cur;
        cur += align256(bytes);
        return p;
    };
#define REG_TRY(expr)                                                                  \
    do {                                                                               \
        cudaError_t _e = (expr);                                                       \
        if (_e != cudaSuccess) {                                                       \
            cudaFree(storage);                                                         \
            (void)cudaGetLastError();                                                  \
            return fail(c, _e == cudaErrorMemoryAllocation ? SCUTE_ERR_OOM : SCUTE_ERR_CUDA, \
                        "%s: %s", #expr, cudaGetErrorString(_e));                      \
        }                                                                              \
    } while (0)
    REG_TRY(cudaMemset(c->d_err, 0, sizeof(int)));
    std::vector<Slot> slots((size_t)n_layers);
    for (int i = 0; i < n_layers; ++i) {
        const scute_layer_tensors &x = t[i];
        const LayerRec &L = c->layers[x.layer];
        const AdapterLayer &al = info[i];
        Slot s{};
        uint8_t *tmp = reinterpret_cast<uint8_t *>(c->tmp);
        if (al.rank) {
            void *tA = tmp;
            void *tB = tmp + align256((size_t)L.d_in * al.rank * E);
            float *tv = reinterpret_cast<float *>(tmp + align256((size_t)L.d_in * al.rank * E) +
                                                  align256((size_t)al.rank * L.d_out * E));
            float *te = tv + align256(4 * (size_t)L.d_out) / 4;
            float *tm = te + align256(4 * (size_t)L.d_out) / 4;
            float *td = tm + align256(4 * (size_t)L.d_out) / 4;
            REG_TRY(cudaMemcpy(tA, x.A, (size_t)L.d_in * al.rank * E, cudaMemcpyDefault));
            REG_TRY(cudaMemcpy(tB, x.B, (size_t)al.rank * L.d_out * E, cudaMemcpyDefault));
            const float *dvec = nullptr, *evec = nullptr, *svec = nullptr;
            if (method == SCUTE_NF && x.d) {
                REG_TRY(cudaMemcpy(td, x.d, 4 * (size_t)al.rank, cudaMemcpyDefault));
                dvec = td;
            }
            if (method == SCUTE_NF && x.e) {
                REG_TRY(cudaMemcpy(te, x.e, 4 * (size_t)L.d_out, cudaMemcpyDefault));
                evec = te;
            }
            void *Ap = take((size_t)al.rank * L.d_in * E);
            void *Bp = take((size_t)al.rank * L.d_out * E);
            if (method == SCUTE_DORA) {
                float *sp = reinterpret_cast<float *>(take(4 * (size_t)L.d_out));
                REG_TRY(cudaMemcpy(tm, x.magnitude, 4 * (size_t)L.d_out, cudaMemcpyDefault));
                REG_TRY(launch_dora_scale(f32, L.Wt, L.kdim, L.d_in, L.d_out, tA, tB, al.rank, x.c, tm, sp,
                                          c->d_err, 0));
                s.s = sp;
                svec = sp;
            }
            REG_TRY(launch_fold_A(f32, tA, L.d_in, al.rank, x.c, dvec, Ap, 0));
            REG_TRY(launch_fold_B(f32, tB, al.rank, L.d_out, evec, svec, Bp, 0));
            if (method == SCUTE_DORA) {
                void *Bu = take((size_t)al.rank * L.d_out * E);
                REG_TRY(launch_fold_B(f32, tB, al.rank, L.d_out, nullptr, nullptr, Bu, 0));
                s.Bu = Bu;
            }
            s.A = Ap;
            s.B = Bp;
            s.rank = al.rank;
            if (c->dtype == SCUTE_BF16) {
                // the tensor-core shrink reads A' through a map of its own:
                // 64 columns x the rank rounded up to 16 rows per box
                CUtensorMap hm;
                if (!encode_map_box(c, &hm, Ap, (uint64_t)L.d_in, (uint64_t)al.rank, (al.rank + 15) & ~15)) {
                    cudaFree(storage);
                    return fail(c, SCUTE_ERR_CUDA, "tensor map for A' failed");
                }
                void *mp = take(sizeof(CUtensorMap));
                REG_TRY(cudaMemcpy(mp, &hm, sizeof(CUtensorMap), cudaMemcpyHostToDevice));
                s.mapA = mp;
            }
        }
        if (method == SCUTE_IA3) {
            float *sp = reinterpret_cast<float *>(take(4 * (size_t)L.d_out));
            REG_TRY(cudaMemcpy(sp, x.l, 4 * (size_t)L.d_out, cudaMemcpyDefault));
            s.s = sp;
        }
        if (method == SCUTE_NF && x.s) {
            float *sp = reinterpret_cast<float *>(take(4 * (size_t)L.d_out));
            REG_TRY(cudaMemcpy(sp, x.s, 4 * (size_t)L.d_out, cudaMemcpyDefault));
            s.s = sp;
        }
        if (method == SCUTE_NF && x.b) {
            float *bp = reinterpret_cast<float *>(take(4 * (size_t)L.d_out));
            REG_TRY(cudaMemcpy(bp, x.b, 4 * (size_t)L.d_out, cudaMemcpyDefault));
            s.b = bp;
        }
        if (al.R) {
            void *Rp = take((size_t)L.d_in * OFT_BLK * E);
            REG_TRY(cudaMemcpy(Rp, x.R, (size_t)L.d_in * OFT_BLK * E, cudaMemcpyDefault));
            s.R = Rp;
            if (c->dtype == SCUTE_BF16) {
                // the decode step reads R by columns: keep a copy with every block transposed
                void *Rtp = take((size_t)L.d_in * OFT_BLK * E);
                REG_TRY(launch_transpose_blocks(Rp, Rtp, L.d_in / OFT_BLK, 0));
                s.Rt = Rtp;
            }
        }
        if (al.vera) {
            float *dp = reinterpret_cast<float *>(take(4 * (size_t)L.rv));
            float *ep = reinterpret_cast<float *>(take(4 * (size_t)L.d_out));
            float *td = reinterpret_cast<float *>(tmp);
            REG_TRY(cudaMemcpy(td, x.d, 4 * (size_t)L.rv, cudaMemcpyDefault));
            // the shared term's scalar c is the adapter's own: merged into its d
            // (applied as given, like every other term's c)
            REG_TRY(launch_scale_vec(td, x.c, dp, L.rv, 0));
            if (x.e) {
                REG_TRY(cudaMemcpy(ep, x.e, 4 * (size_t)L.d_out, cudaMemcpyDefault));
                s.ve = ep;
            }
            s.vd = dp;
        }
        // raw tensors in tmp are reused by the next layer: finish this one first
        REG_TRY(cudaDeviceSynchronize());
        slots[i] = s;
    }
    int herr = 0;
    REG_TRY(cudaMemcpy(&herr, c->d_err, sizeof(int), cudaMemcpyDeviceToHost));
    if (herr) {
        cudaFree(storage);
        return fail(c, SCUTE_ERR_ARG, "DoRA: a column of W + cAB has zero norm");
    }
    for (int i = 0; i < n_layers; ++i)
        REG_TRY(cudaMemcpy(c->d_slots + (size_t)t[i].layer * c->max_adapters + id, &slots[i], sizeof(Slot),
                           cudaMemcpyHostToDevice));
    const int8_t m8 = (int8_t)method;
    REG_TRY(cudaMemcpy(c->d_method + id, &m8, 1, cudaMemcpyHostToDevice));
#undef REG_TRY
    AdapterRec &a = c->adapters[id];
    a.used = true;
    a.method = method;
    a.storage = storage;
    a.layers = info;
    c->h_method[id] = m8;
    for (const auto &al : info) {
        LayerRec &L = c->layers[al.layer];
        if (al.rank) ++L.n_lr;
        if (al.vera) ++L.n_vera;
        if (al.R) ++L.n_rot;
        if (al.R && al.rank) ++L.n_rot_lr;
    }
    *id_out = id;
    return SCUTE_OK;
}

scute_status scute_unregister_adapter(scute_ctx *c, int32_t id) {
    if (!c) return SCUTE_ERR_ARG;
    if (id < 0 || id >= c->max_adapters || !c->adapters[id].used)
        return fail(c, SCUTE_ERR_ARG, "adapter %d is not registered", id);
    DeviceGuard dg(c->device);
    CU_TRY(c, cudaDeviceSynchronize());
    AdapterRec &a = c->adapters[id];
    const int8_t none = -1;
    CU_TRY(c, cudaMemcpy(c->d_method + id, &none, 1, cudaMemcpyHostToDevice));
    const Slot zero{};
    for (const auto &al : a.layers) {
        CU_TRY(c, cudaMemcpy(c->d_slots + (size_t)al.layer * c->max_adapters + id, &zero, sizeof(Slot),
                             cudaMemcpyHostToDevice));
        LayerRec &L = c->layers[al.layer];
        if (al.rank) --L.n_lr;
        if (al.vera) --L.n_vera;
        if (al.R) --L.n_rot;
        if (al.R && al.rank) --L.n_rot_lr;
    }
    CU_TRY(c, cudaFree(a.storage));
    a = AdapterRec();
    c->h_method[id] = -1;
    return SCUTE_OK;
}

static int max_owned_rank(const scute_ctx *c, int layer) {
    int r = 0;
    for (const auto &a : c->adapters)
        if (a.used)
            for (const auto &al : a.layers)
                if (al.layer == layer && al.rank > r) r = al.rank;
    return r;
}

// One decode step over n_calls layers (bf16 context, n <= STEP_MAX_TOKENS):
// argument block, stream-K ranges and workspace slots, then one cooperative
// launch.  Arguments are validated by the callers.
static scute_status step_launch(scute_ctx *c, const scute_call *calls, int nc, const int32_t *ids, int nn,
                                int out_f32, cudaStream_t st) {
    StepArgs a;
    memset(&a, 0, sizeof(a));
    const int G = c->num_sms < STEP_MAX_GRID ? c->num_sms : STEP_MAX_GRID;
    const int BN = nn <= 64 ? 64 : 128;
    if (BN > c->step_bn_max) return fail(c, SCUTE_ERR_UNSUPPORTED, "decode workspace sized for fewer tokens");
    const bool oft_pass = (c->variant & VARIANT_OFT_PASS) != 0, s_pass = (c->variant & VARIANT_S_PASS) != 0;
    int max_din = 0, max_dout = 0;
    for (int i = 0; i < nc; ++i) {
        const LayerRec &L = c->layers[calls[i].layer];
        if (L.d_in > max_din) max_din = L.d_in;
        if (L.d_out > max_dout) max_dout = L.d_out;
    }
    if (oft_pass && (size_t)max_din > c->var_x_cols)
        return fail(c, SCUTE_ERR_UNSUPPORTED, "rotated-copy workspace smaller than a layer's input");
    long long blk = 0;
    int tile = 0, item = 0, rmax = 0;
    for (int i = 0; i < nc; ++i) {
        const LayerRec &L = c->layers[calls[i].layer];
        StepCall &k = a.call[i];
        const bool vera_on = L.rv > 0 && L.n_vera > 0;
        // the rotation placed in a separate pass: the token operand is read
        // from that pass's rotated copy of x
        k.x = oft_pass ? reinterpret_cast<uint8_t *>(c->var_x) + (size_t)i * STEP_MAX_TOKENS * c->var_x_cols * c->esz
                       : calls[i].x;
        k.x0 = calls[i].x;
        k.xs = reinterpret_cast<uint8_t *>(c->step_xs) + (size_t)i * STEP_MAX_TOKENS * c->step_xs_cols * c->esz;
        k.U = vera_on ? reinterpret_cast<uint8_t *>(c->step_U) + (size_t)i * STEP_MAX_TOKENS * c->step_u_cols * c->esz
                      : nullptr;
        k.pre = c->step_pre ? c->step_pre + (size_t)i * (c->step_pre_floats / STEP_MAX_CALLS) : nullptr;
        k.out = calls[i].out;
        k.slots = c->d_slots + (size_t)calls[i].layer * c->max_adapters;
        k.Wt = L.Wt;
        k.mapW = L.mapW;
        if (!encode_map(c, &k.mapXs, k.xs, (uint64_t)L.kdim, (uint64_t)STEP_MAX_TOKENS))
            return fail(c, SCUTE_ERR_CUDA, "tensor map for the token operand failed");
        if (vera_on) {
            k.mapAsh = L.mapAsh;
            k.mapBsh = L.mapBsh;
            if (!encode_map(c, &k.mapU, k.U, (uint64_t)L.krv, (uint64_t)STEP_MAX_TOKENS))
                return fail(c, SCUTE_ERR_CUDA, "tensor map for the VeRA intermediate failed");
        }
        // Rows that nothing rotates are rows of x: a layer with no rotation
        // adapter (or whose rotation ran in its own pass) needs no token
        // operand copy at all, and its base tiles read x itself from the first
        // block on.  VeRA tokens are never rotated, so the VeRA shrink reads x
        // directly in every case and starts before x' is formed (rows of other
        // tokens are discarded by the shrink's epilogue).
        // (an injected stall keeps the wait on x', which is what it withholds)
        const bool direct = (L.n_rot == 0 || oft_pass) && c->inject != SCUTE_INJECT_STALL;
        const bool x_map = (vera_on || direct) && reinterpret_cast<uintptr_t>(k.x) % 16 == 0 &&
                           ((size_t)L.d_in * c->esz) % 16 == 0 &&
                           encode_map(c, &k.mapX, k.x, (uint64_t)L.d_in, (uint64_t)nn);
        k.vs_x = vera_on && x_map ? 1 : 0;
        k.xs_direct = direct && x_map ? 1 : 0;
        k.d_in = L.d_in;
        k.kdim = L.kdim;
        k.d_out = L.d_out;
        k.krv = L.krv;
        k.rv = L.rv;
        k.kblocks = (L.kdim + 63) / 64;
        k.vkb = vera_on ? (L.krv + 63) / 64 : 0;
        k.n_ft = (L.d_out + 127) / 128;
        k.n_vt = vera_on ? (L.rv + 127) / 128 : 0;
        k.lr_rmax = L.n_lr > 0 ? max_owned_rank(c, calls[i].layer) : 0;
        if (k.lr_rmax > rmax) rmax = k.lr_rmax;
        if (k.lr_rmax > 0 && (size_t)((k.lr_rmax + 7) / 8) * STEP_MAX_TOKENS * (size_t)L.d_out >
                                 c->step_pre_floats / STEP_MAX_CALLS)
            return fail(c, SCUTE_ERR_UNSUPPORTED, "low-rank row workspace smaller than a call needs");
        k.out_f32 = out_f32;
        k.blk0 = blk;
        blk += (long long)k.n_ft * (k.kblocks + k.vkb);
        k.tile0 = tile;
        tile += k.n_ft;
    }
    for (int i = 0; i < nc; ++i) {
        const LayerRec &L = c->layers[calls[i].layer];
        StepCall &k = a.call[i];
        k.lr_items = k.lr_rmax > 0 ? (L.n_lr < nn ? L.n_lr : nn) * ((k.lr_rmax + 7) / 8) : 0;
        k.lr_item0 = item;
        item += k.lr_items;
    }
    // VeRA shrink units: the shortest K chunk (a power of two >= 16 blocks)
    // that gives at most one unit per CTA (a unit per VeRA tile at the least)
    int vt_total = 0;
    for (int i = 0; i < nc; ++i) vt_total += a.call[i].n_vt;
    if (vt_total > G) return fail(c, SCUTE_ERR_UNSUPPORTED, "more VeRA shrink tiles (%d) than CTAs (%d)", vt_total, G);
    int ch = 16, units = 0;
    for (;;) {
        units = 0;
        for (int i = 0; i < nc; ++i) units += a.call[i].n_vt * ((a.call[i].kblocks + ch - 1) / ch);
        if (units <= G) break;
        ch *= 2;
    }
    long long t_vs = 0;
    int u = 0;
    std::vector<int> ublk(units > 0 ? units : 1, 0);
    for (int i = 0; i < nc; ++i) {
        StepCall &k = a.call[i];
        k.vs_chunks = (k.kblocks + ch - 1) / ch;
        k.vs_unit0 = u;
        for (int vt = 0; vt < k.n_vt; ++vt)
            for (int cc = 0; cc < k.vs_chunks; ++cc) {
                const int b0 = cc * ch, b1 = b0 + ch < k.kblocks ? b0 + ch : k.kblocks;
                ublk[u++] = b1 - b0;
                t_vs += b1 - b0;
            }
    }
    {
        // low-rank items are dealt with the calls of most work per item
        // (d_in + d_out) first, ties in call order
        unsigned used = 0;
        for (int o = 0; o < nc; ++o) {
            int best = 0, bw = -1;
            for (int i = 0; i < nc; ++i) {
                const int w = a.call[i].d_in + a.call[i].d_out;
                if (!((used >> i) & 1u) && w > bw) {
                    bw = w;
                    best = i;
                }
            }
            used |= 1u << best;
            a.it_call[o] = best;
            a.it_ng[o] = (a.call[best].lr_rmax + 7) / 8;
        }
    }
    // Each CTA's epilogue warps run the low-rank items dealt to it (item it to
    // CTA G - 1 - it mod G) while its stream runs, and they slow that stream:
    // an item is charged (d_in + d_out) / ITEM_FEATURES_PER_BLOCK stream blocks
    // against its CTA, counted on the host's bound of items per call (the
    // batch's own count is known only on the device).  Per-CTA timestamps on
    // the 64-token mixed batch: an item delays its CTA by about a third of its
    // own time; a gate or up item then weighs about 16 blocks.
    std::vector<long long> icost((size_t)G, 0);
    {
        long long it = 0;
        for (int o = 0; o < nc; ++o) {
            const StepCall &k = a.call[a.it_call[o]];
            const long long pen = (long long)(k.d_in + k.d_out) / ITEM_FEATURES_PER_BLOCK;
            for (int j = 0; j < k.lr_items; ++j, ++it) icost[(size_t)(G - 1 - (int)(it % G))] += pen;
        }
    }
    long long tcost = 0;
    for (int i = 0; i < G; ++i) tcost += icost[(size_t)i];
    // stream-K ranges: every CTA gets about (main + VeRA-shrink blocks + item
    // charges) / G, its VeRA unit and its items counted against its share of
    // main blocks
    const long long W = blk + t_vs + tcost;
    long long vsb = 0;
    bool mono = true;
    for (int i = 0; i <= G; ++i) {
        a.start[i] = (long long)i * W / G - vsb;
        if (i < units) vsb += ublk[i];
        if (i < G) vsb += icost[(size_t)i];
        if (i > 0 && a.start[i] < a.start[i - 1]) mono = false;
    }
    if (!mono || a.start[0] != 0 || a.start[G] != blk)
        for (int i = 0; i <= G; ++i) a.start[i] = (long long)i * blk / G;
    a.n_calls = nc;
    a.n = nn;
    a.A = c->max_adapters;
    a.bn = BN;
    a.grid = G;
    a.ids = ids;
    a.method_tab = c->d_method;
    a.status = c->d_status;
    a.part = c->step_part;
    a.sync = c->step_sync;
    a.t_main = blk;
    a.w_total = W;
    a.n_units = units;
    a.vs_ch = ch;
    a.n_tiles = tile;
    a.n_items = item;
    a.rmax = rmax;
    a.hold = c->inject == SCUTE_INJECT_STALL ? 1 : 0;
    c->inject = 0;
    int S = 8;
    while (S > 2 && step_smem_bytes(BN, S, rmax) > (size_t)c->smem_optin) --S;
    if (step_smem_bytes(BN, S, rmax) > (size_t)c->smem_optin)
        return fail(c, SCUTE_ERR_UNSUPPORTED, "decode step does not fit shared memory");
    a.stages = S;
    if ((size_t)(units + tile + G) * 2 * 128 * BN > c->step_part_floats)
        return fail(c, SCUTE_ERR_UNSUPPORTED, "partial-tile workspace too small for this batch");
    if (SY_TILE + tile > STEP_SYNC_INTS) return fail(c, SCUTE_ERR_UNSUPPORTED, "too many tiles in one batch");
    a.variant = c->variant;
    {
        // the plan as launched, for scute_debug_step_plan
        std::vector<int64_t> &P = c->last_plan;
        P.clear();
        const int64_t head[SCUTE_PLAN_HEAD] = {nc, nn, BN, S, G, units, ch, tile, item, rmax, blk, a.hold,
                                               (int64_t)step_smem_bytes(BN, S, rmax), c->smem_optin,
                                               (int64_t)c->step_part_floats, (int64_t)c->step_xs_cols,
                                               (int64_t)c->step_u_cols, STEP_SYNC_INTS,
                                               (int64_t)c->step_pre_floats};
        P.insert(P.end(), head, head + SCUTE_PLAN_HEAD);
        for (int i = 0; i < nc; ++i) {
            const StepCall &k = a.call[i];
            const int64_t f[SCUTE_PLAN_CALL_FIELDS] = {k.blk0, k.d_in, k.kdim, k.d_out, k.krv, k.rv,
                                                       k.kblocks, k.vkb, k.n_ft, k.n_vt, k.vs_chunks,
                                                       k.vs_unit0, k.tile0, k.lr_rmax, k.lr_items,
                                                       k.lr_item0, k.vs_x, k.xs_direct};
            P.insert(P.end(), f, f + SCUTE_PLAN_CALL_FIELDS);
        }
        P.insert(P.end(), a.start, a.start + G + 1);
    }
    PassArgs pa;
    memset(&pa, 0, sizeof(pa));
    pa.n_calls = nc;
    pa.n = nn;
    pa.A = c->max_adapters;
    pa.out_f32 = out_f32;
    pa.ids = ids;
    pa.method_tab = c->d_method;
    for (int i = 0; i < nc; ++i) {
        const LayerRec &L = c->layers[calls[i].layer];
        pa.call[i].x = calls[i].x;
        pa.call[i].xo = const_cast<void *>(a.call[i].x);
        pa.call[i].out = calls[i].out;
        pa.call[i].slots = a.call[i].slots;
        pa.call[i].d_in = L.d_in;
        pa.call[i].d_out = L.d_out;
    }
    TimedLaunch tl{c, st};
    cudaGetLastError();
    if (oft_pass) {
        CU_TRY(c, tl.begin());
        CU_TRY(c, launch_oft_pass(pa, max_din, st));
        CU_TRY(c, tl.end(SCUTE_KIND_OFT_PASS));
        count_launch(c, 1);
    }
    CU_TRY(c, tl.begin());
    CU_TRY(c, launch_step(a, st));
    CU_TRY(c, tl.end(SCUTE_KIND_STEP));
    count_launch(c, 1);
    if (s_pass) {
        CU_TRY(c, tl.begin());
        CU_TRY(c, launch_s_pass(pa, max_dout, st));
        CU_TRY(c, tl.end(SCUTE_KIND_S_PASS));
        count_launch(c, 1);
    }
    return SCUTE_OK;
}

scute_status scute_linear(scute_ctx *c, const void *x, const int32_t *ids, int64_t n, int layer, void *out,
                          scute_dtype out_dtype, void *stream) {
    if (!c) return SCUTE_ERR_ARG;
    if (!layer_ok(c, layer)) return fail(c, SCUTE_ERR_ARG, "unknown layer %d", layer);
    if (n < 0 || n > c->max_tokens) return fail(c, SCUTE_ERR_ARG, "n = %lld outside 0..%d", (long long)n, c->max_tokens);
    if (out_dtype != SCUTE_BF16 && out_dtype != SCUTE_FP32) return fail(c, SCUTE_ERR_DTYPE, "bad out dtype");
    if (c->dtype == SCUTE_FP32 && out_dtype != SCUTE_FP32)
        return fail(c, SCUTE_ERR_DTYPE, "an fp32 context writes fp32 output");
    if (n == 0) return SCUTE_OK;
    if (!x || !ids || !out) return fail(c, SCUTE_ERR_ARG, "null argument");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
        return fail(c, SCUTE_ERR_ARG, "x and out must be 16-byte aligned");
    DeviceGuard dg(c->device);
    const LayerRec &L = c->layers[layer];
    const bool f32 = c->dtype == SCUTE_FP32;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int nn = (int)n;
    const Slot *slots = c->d_slots + (size_t)layer * c->max_adapters;
    const int out_f32 = out_dtype == SCUTE_FP32 ? 1 : 0;
    if (!f32 && nn <= STEP_MAX_TOKENS) {
        const scute_call one = {x, layer, out};
        return step_launch(c, &one, 1, ids, nn, out_f32, st);
    }
    int k = 0;

    const int lr_rmax = L.n_lr > 0 ? max_owned_rank(c, layer) : 0;
    const bool vera_on = L.rv > 0 && L.n_vera > 0;
    // Other batches (fp32 contexts, or more than STEP_MAX_TOKENS tokens): one
    // launch per step.
    TimedLaunch tl{c, st};
    {
        // 1. token indexing
        CU_TRY(c, tl.begin());
        CU_TRY(c, launch_index(ids, nn, c->d_method, c->max_adapters, c->d_perm, c->d_aid, c->d_seg_start,
                               c->d_seg_aid, c->d_meta, c->d_status, st, c->d_seg_unit, c->d_seg_tile));
        CU_TRY(c, tl.end(SCUTE_KIND_INDEX));
        ++k;
        // 2. rotation prologue into the sorted token operand
        CU_TRY(c, tl.begin());
        CU_TRY(c, launch_gather_rotate(f32, x, L.d_in, nn, c->d_perm, c->d_aid, slots, c->xs, L.kdim, st,
                                       c->pdl));
        CU_TRY(c, tl.end(SCUTE_KIND_ROTATE));
        ++k;
    }
    const bool tok_on_p = nn > 256;
    // bf16 with tokens on the GEMM's 128-row side: the owned low-rank expand
    // runs in the base GEMM's epilogue (each out row written once), so the
    // shrink comes first
    const bool lr_fused = !f32 && tok_on_p && L.n_lr > 0;
    // owned low-rank term: units of SEG_UNIT_ROWS rows of every segment;
    // there are at most n / SEG_UNIT_ROWS + (segments) of them, and at most
    // one segment per registered adapter plus the base rows
    int reg = 0;
    for (const auto &a : c->adapters) reg += a.used ? 1 : 0;
    const int unit_bound = (nn + SEG_UNIT_ROWS - 1) / SEG_UNIT_ROWS + (reg + 1 < nn ? reg + 1 : nn);
    int lr_ks = 0;
    {
        int kchunk = 0;
        lr_ks = lowrank_ks(L.d_in, &kchunk);
    }
    // VeRA shared shrink on the tensor cores (bf16, many VeRA rows); right
    // after the tensor-core owned shrink it runs beside that launch
    const bool vs_tc = vera_on && !f32 && tok_on_p && L.rv % 64 == 0 && c->vs_part_cols >= (size_t)L.rv;
    const bool vs_after_lr = vs_tc && lr_fused && L.n_rot_lr == 0;
    // owned low-rank shrink (and, unless fused, its expand).  bf16: the shrink
    // runs on the tensor cores over the sorted token operand, which holds x
    // itself for every owned-term row unless an adapter of the layer has both
    // a rotation and an owned term
    auto owned_lowrank = [&](bool expand) -> scute_status {
        const bool tc = !f32 && L.n_rot_lr == 0;
        CU_TRY(c, tl.begin());
        if (tc) {
            LrTcArgs q;
            memset(&q, 0, sizeof(q));
            q.mapX = L.mapXs;
            q.kblocks = (L.d_in + 63) / 64;
            int kchunk = 0;
            q.ks = lowrank_ks(L.d_in, &kchunk);
            q.chunk_blocks = kchunk / 64;
            q.max_tokens = c->max_tokens;
            q.seg_start = c->d_seg_start;
            q.seg_aid = c->d_seg_aid;
            q.seg_tile = c->d_seg_tile;
            q.meta = c->d_meta;
            q.slots = slots;
            q.v_part = c->v_part;
            q.status = c->d_status;
            const int tile_bound = (nn + SEG_TILE_ROWS - 1) / SEG_TILE_ROWS + (reg + 1 < nn ? reg + 1 : nn);
            const int units = tile_bound * q.ks;
            CU_TRY(c, launch_lr_shrink_tc(q, units < c->num_sms ? units : c->num_sms, st, c->pdl,
                                          vs_after_lr && !expand));
        }
        if (!tc || expand)
            CU_TRY(c, launch_lowrank(f32, x, L.d_in, L.d_out, unit_bound, c->d_perm, c->d_seg_start, c->d_seg_aid,
                                     c->d_seg_unit, c->d_meta, slots, c->v_part, c->max_tokens, out, out_f32, st,
                                     c->pdl, lr_rmax, !tc, expand));
        CU_TRY(c, tl.end(SCUTE_KIND_LOWRANK));
        k += expand ? 2 : 1;
        return SCUTE_OK;
    };
    // 3. owned low-rank shrink, when its expand is fused into the base GEMM
    if (lr_fused) {
        const scute_status e = owned_lowrank(false);
        if (e != SCUTE_OK) return e;
    }
    // 3b. VeRA shared shrink over the VeRA rows, bf16 with many VeRA rows:
    // K-split units on the tensor cores, so that every SM streams (one CTA per
    // 128 x rank tile over all of K would leave most of them idle).  It needs
    // neither the owned shrink nor the base GEMM, so it comes before the GEMM
    if (vs_tc) {
        VsTcArgs q;
        memset(&q, 0, sizeof(q));
        q.mapX = L.mapXs;
        q.mapA = L.mapAsh;
        q.kblocks = (L.d_in + 63) / 64;
        // at most VS_KS chunks, none of them empty
        q.chunk_blocks = (q.kblocks + VS_KS - 1) / VS_KS;
        q.ks = (q.kblocks + q.chunk_blocks - 1) / q.chunk_blocks;
        q.n_nt = L.rv / 64;
        q.rv = L.rv;
        q.ldu = L.krv;
        q.max_tokens = c->max_tokens;
        q.meta = c->d_meta;
        q.aid_s = c->d_aid;
        q.slots = slots;
        q.part = c->vs_part;
        q.ctr = c->vs_ctr;
        q.U = c->U;
        q.status = c->d_status;
        q.after_lr = vs_after_lr ? 1 : 0;
        const int units = (nn + 127) / 128 * q.n_nt * q.ks;
        if (VS_CTR_TILES + (nn + 127) / 128 * q.n_nt > VS_CTR_INTS)
            return fail(c, SCUTE_ERR_UNSUPPORTED, "VeRA shrink counters too few for this batch");
        CU_TRY(c, tl.begin());
        CU_TRY(c, launch_vera_shrink_tc(q, units < c->num_sms ? units : c->num_sms, st, c->pdl));
        CU_TRY(c, tl.end(SCUTE_KIND_VERA_SHRINK));
    }
    // 4. base GEMM with the s / b (and fused owned low-rank) epilogue
    GemmArgs g;
    memset(&g, 0, sizeof(g));
    g.mapP = tok_on_p ? L.mapXs : L.mapW;
    g.mapQ = tok_on_p ? L.mapW : L.mapXs;
    g.kblocks = (L.kdim * c->esz + 127) / 128;
    g.n_feat = L.d_out;
    g.tok_on_p = tok_on_p ? 1 : 0;
    g.n_tok_host = nn;
    g.epi = EPI_BASE;
    g.out_f32 = out_f32;
    g.ld_out = L.d_out;
    g.slots = slots;
    g.perm = c->d_perm;
    g.aid_s = c->d_aid;
    g.out = out;
    g.status = c->d_status;
    if (lr_fused) {
        g.v = c->v_part;
        g.v_ld = MAX_RANK;
        g.v_ks = lr_ks;
        g.v_kstride = (long long)c->max_tokens * MAX_RANK;
        g.lr_rmax = lr_rmax;
    }
    if (!tok_on_p) {
        g.p_base = L.Wt;
        g.p_pitch = (long long)L.kdim * c->esz;
        g.p_rows = L.d_out;
    }
    GemmPlan p = plan_gemm(nn, L.d_out, g.kblocks, tok_on_p, f32, c->num_sms, g.lr_rmax);
    g.splits = p.splits;
    g.stages = p.stages;
    g.n_ft = tok_on_p ? (L.d_out + p.bn - 1) / p.bn : (L.d_out + 127) / 128;
    if (!tok_on_p && p.splits == 1 &&
        (size_t)p.stages * (128 * 128 + p.bn * 128) < (size_t)(g.vera_kb ? 2 : 1) * p.bn * 132 * 4)
        return fail(c, SCUTE_ERR_UNSUPPORTED, "the accumulator tile does not fit the pipeline buffers");
    if (!tok_on_p && p.splits > 1 && gemm_part_floats(p.grid, p.bn, g.vera_kb > 0) > PART_WORKSPACE_FLOATS)
        return fail(c, SCUTE_ERR_UNSUPPORTED, "K-split workspace too small for this launch");
    g.part = c->gpart;
    g.part_stride = (long long)p.bn * 128 * (g.vera_kb ? 2 : 1);
    CU_TRY(c, tl.begin());
    CU_TRY(c, launch_gemm(g, p, st, c->pdl));
    CU_TRY(c, tl.end(SCUTE_KIND_BASE_GEMM));
    ++k;
    // owned low-rank shrink and expand after the base GEMM (the expand adds
    // into out): fp32 contexts and the features-on-P orientation
    if (L.n_lr > 0 && !lr_fused) {
        const scute_status e = owned_lowrank(true);
        if (e != SCUTE_OK) return e;
    }
    // 5. VeRA: shared shrink then shared expand over the VeRA rows only
    if (vera_on) {
        GemmArgs v;
        memset(&v, 0, sizeof(v));
        v.mapP = tok_on_p ? L.mapXs : L.mapAsh;
        v.mapQ = tok_on_p ? L.mapAsh : L.mapXs;
        v.kblocks = g.kblocks;
        v.n_feat = L.rv;
        v.tok_on_p = g.tok_on_p;
        v.n_tok_host = nn;
        v.tok_cnt = &c->d_meta->count[RANK_VERA];
        v.tok_base = &c->d_meta->offset[RANK_VERA];
        v.sorted_base = &c->d_meta->offset[RANK_VERA];
        v.epi = EPI_VERA_D;
        v.ldu = L.krv;
        v.u_split3 = f32 ? 1 : 0;
        v.u_rank = L.rv;
        v.slots = slots;
        v.perm = c->d_perm;
        v.aid_s = c->d_aid;
        v.U = c->U;
        v.status = c->d_status;
        GemmPlan pv = plan_gemm(nn, L.rv, v.kblocks, tok_on_p, f32, c->num_sms);
        v.splits = pv.splits;
        v.stages = pv.stages;
        v.part = c->gpart;
        v.part_stride = (long long)pv.bn * 128;
        v.n_ft = tok_on_p ? (L.rv + pv.bn - 1) / pv.bn : (L.rv + 127) / 128;
        if (!vs_tc) {
            CU_TRY(c, tl.begin());
            CU_TRY(c, launch_gemm(v, pv, st, c->pdl));
            CU_TRY(c, tl.end(SCUTE_KIND_VERA_SHRINK));
        }

        GemmArgs e = v;
        e.mapP = tok_on_p ? L.mapU : L.mapBsh;
        e.mapQ = tok_on_p ? L.mapBsh : L.mapU;
        e.kblocks = (L.krv * c->esz + 127) / 128;
        e.n_feat = L.d_out;
        e.tok_base = nullptr;
        e.epi = EPI_VERA_E;
        e.out = out;
        e.out_f32 = out_f32;
        e.ld_out = L.d_out;
        e.stage_out = tok_on_p && !f32 && !out_f32 ? 1 : 0;
        GemmPlan pe = plan_gemm(nn, L.d_out, e.kblocks, tok_on_p, f32, c->num_sms, 0, e.stage_out != 0);
        e.splits = pe.splits;
        e.stages = pe.stages;
        e.part = c->gpart;
        e.part_stride = (long long)pe.bn * 128;
        e.n_ft = tok_on_p ? (L.d_out + pe.bn - 1) / pe.bn : (L.d_out + 127) / 128;
        CU_TRY(c, tl.begin());
        CU_TRY(c, launch_gemm(e, pe, st, c->pdl));
        CU_TRY(c, tl.end(SCUTE_KIND_VERA_EXPAND));
        k += 2;
    }
    count_launch(c, k);
    return SCUTE_OK;
}

scute_status scute_linear_host(scute_ctx *c, const void *x_host, const int32_t *ids_host, int64_t n, int layer,
                               void *out_host, scute_dtype out_dtype, void *stream) {
    if (!c) return SCUTE_ERR_ARG;
    if (!layer_ok(c, layer)) return fail(c, SCUTE_ERR_ARG, "unknown layer %d", layer);
    if (n < 0 || n > c->max_tokens) return fail(c, SCUTE_ERR_ARG, "n out of range");
    if (n == 0) return SCUTE_OK;
    if (!x_host || !ids_host || !out_host) return fail(c, SCUTE_ERR_ARG, "null argument");
    DeviceGuard dg(c->device);
    const LayerRec &L = c->layers[layer];
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t osz = out_dtype == SCUTE_FP32 ? 4 : 2;
    CU_TRY(c, cudaMemcpyAsync(c->st_x, x_host, (size_t)n * L.d_in * c->esz, cudaMemcpyHostToDevice, st));
    CU_TRY(c, cudaMemcpyAsync(c->st_ids, ids_host, (size_t)n * 4, cudaMemcpyHostToDevice, st));
    // a bf16 decode batch (one step launch, which only stores to out) writes
    // a pinned, mapped, 16-byte-aligned output buffer directly
    if (c->dtype != SCUTE_FP32 && n <= STEP_MAX_TOKENS && (c->variant & VARIANT_S_PASS) == 0) {
        void *dout = const_cast<void *>(mapped_host(out_host));
        if (dout && (reinterpret_cast<uintptr_t>(dout) & 15) == 0)
            return scute_linear(c, c->st_x, c->st_ids, n, layer, dout, out_dtype, stream);
    }
    scute_status s = scute_linear(c, c->st_x, c->st_ids, n, layer, c->st_out, out_dtype, stream);
    if (s) return s;
    CU_TRY(c, cudaMemcpyAsync(out_host, c->st_out, (size_t)n * L.d_out * osz, cudaMemcpyDeviceToHost, st));
    return SCUTE_OK;
}

static scute_status check_calls(scute_ctx *c, const scute_call *calls, int n_calls, int64_t n,
                                scute_dtype out_dtype, bool need_ptrs) {
    if (n_calls < 0 || n_calls > SCUTE_MAX_CALLS || (n_calls > 0 && !calls))
        return fail(c, SCUTE_ERR_ARG, "n_calls = %d outside 0..%d", n_calls, SCUTE_MAX_CALLS);
    if (n < 0 || n > c->max_tokens) return fail(c, SCUTE_ERR_ARG, "n = %lld outside 0..%d", (long long)n, c->max_tokens);
    if (out_dtype != SCUTE_BF16 && out_dtype != SCUTE_FP32) return fail(c, SCUTE_ERR_DTYPE, "bad out dtype");
    if (c->dtype == SCUTE_FP32 && out_dtype != SCUTE_FP32)
        return fail(c, SCUTE_ERR_DTYPE, "an fp32 context writes fp32 output");
    for (int i = 0; i < n_calls; ++i) {
        if (!layer_ok(c, calls[i].layer)) return fail(c, SCUTE_ERR_ARG, "call %d: unknown layer %d", i, calls[i].layer);
        if (need_ptrs && n > 0) {
            if (!calls[i].x || !calls[i].out) return fail(c, SCUTE_ERR_ARG, "call %d: null argument", i);
            if ((reinterpret_cast<uintptr_t>(calls[i].x) | reinterpret_cast<uintptr_t>(calls[i].out)) & 15)
                return fail(c, SCUTE_ERR_ARG, "call %d: x and out must be 16-byte aligned", i);
        }
    }
    return SCUTE_OK;
}

scute_status scute_linear_batch(scute_ctx *c, const scute_call *calls, int n_calls, const int32_t *ids, int64_t n,
                                scute_dtype out_dtype, void *stream) {
    if (!c) return SCUTE_ERR_ARG;
    scute_status s = check_calls(c, calls, n_calls, n, out_dtype, true);
    if (s) return s;
    if (n == 0 || n_calls == 0) return SCUTE_OK;
    if (!ids) return fail(c, SCUTE_ERR_ARG, "null argument");
    if (c->dtype == SCUTE_FP32 || n > STEP_MAX_TOKENS) {
        for (int i = 0; i < n_calls; ++i) {
            s = scute_linear(c, calls[i].x, ids, n, calls[i].layer, calls[i].out, out_dtype, stream);
            if (s) return s;
        }
        return SCUTE_OK;
    }
    DeviceGuard dg(c->device);
    return step_launch(c, calls, n_calls, ids, (int)n, out_dtype == SCUTE_FP32 ? 1 : 0,
                       reinterpret_cast<cudaStream_t>(stream));
}

scute_status scute_linear_batch_host(scute_ctx *c, const scute_call *calls, int n_calls, const int32_t *ids_host,
                                     int64_t n, scute_dtype out_dtype, void *stream) {
    if (!c) return SCUTE_ERR_ARG;
    scute_status s = check_calls(c, calls, n_calls, n, out_dtype, false);
    if (s) return s;
    if (n == 0 || n_calls == 0) return SCUTE_OK;
    if (!ids_host) return fail(c, SCUTE_ERR_ARG, "null argument");
    for (int i = 0; i < n_calls; ++i)
        if (!calls[i].x || !calls[i].out) return fail(c, SCUTE_ERR_ARG, "call %d: null argument", i);
    if (c->dtype == SCUTE_FP32 || n > STEP_MAX_TOKENS) {
        for (int i = 0; i < n_calls; ++i) {
            s = scute_linear_host(c, calls[i].x, ids_host, n, calls[i].layer, calls[i].out, out_dtype, stream);
            if (s) return s;
        }
        return SCUTE_OK;
    }
    DeviceGuard dg(c->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t osz = out_dtype == SCUTE_FP32 ? 4 : 2;
    scute_call dev[SCUTE_MAX_CALLS];
    for (int i = 0; i < n_calls; ++i) {
        dev[i].layer = calls[i].layer;
        dev[i].x = reinterpret_cast<uint8_t *>(c->step_hx) + (size_t)i * STEP_MAX_TOKENS * c->step_hx_cols * c->esz;
        dev[i].out = reinterpret_cast<uint8_t *>(c->step_hout) + (size_t)i * STEP_MAX_TOKENS * c->step_hout_cols * 4;
    }
    // Pinned, mapped, 16-byte-aligned output buffers take the step's output
    // stores directly (the step only stores to out, once per element, so
    // those writes cross to host memory while the step still streams
    // weights); not with the separate s pass, which reads out back
    bool direct_out = (c->variant & VARIANT_S_PASS) == 0;
    void *hout[SCUTE_MAX_CALLS];
    for (int i = 0; direct_out && i < n_calls; ++i) {
        hout[i] = const_cast<void *>(mapped_host(calls[i].out));
        if (!hout[i] || (reinterpret_cast<uintptr_t>(hout[i]) & 15)) direct_out = false;
    }
    if (direct_out)
        for (int i = 0; i < n_calls; ++i) dev[i].out = hout[i];
    // Pinned, mapped host buffers are moved by one gather launch before the
    // step and one scatter launch after it (the device reads and writes them
    // through their device addresses); any other host buffer, by one copy
    // each.
    static_assert(COPY_MAX_SEGS >= 2 * SCUTE_MAX_CALLS + 1, "copy segments");
    CopySegs in{}, outs{};
    bool gather = true, scatter = true;
    {
        const void *d_ids = mapped_host(ids_host);
        gather = d_ids != nullptr;
        if (gather) {
            in.src[in.n] = d_ids;
            in.dst[in.n] = c->st_ids;
            in.bytes[in.n++] = (size_t)n * 4;
        }
        for (int i = 0; i < n_calls; ++i) {
            const LayerRec &L = c->layers[calls[i].layer];
            const void *dx = gather ? mapped_host(calls[i].x) : nullptr;
            if (!dx) gather = false;
            if (gather) {
                in.src[in.n] = dx;
                in.dst[in.n] = const_cast<void *>(dev[i].x);
                in.bytes[in.n++] = (size_t)n * L.d_in * c->esz;
            }
        }
    }
    if (gather) {
        CU_TRY(c, launch_copy_segments(in, st));
        count_launch(c, 1);
    } else {
        CU_TRY(c, cudaMemcpyAsync(c->st_ids, ids_host, (size_t)n * 4, cudaMemcpyHostToDevice, st));
        for (int i = 0; i < n_calls; ++i) {
            const LayerRec &L = c->layers[calls[i].layer];
            CU_TRY(c, cudaMemcpyAsync(const_cast<void *>(dev[i].x), calls[i].x, (size_t)n * L.d_in * c->esz,
                                      cudaMemcpyHostToDevice, st));
        }
    }
    s = step_launch(c, dev, n_calls, c->st_ids, (int)n, out_dtype == SCUTE_FP32 ? 1 : 0, st);
    if (s) return s;
    if (direct_out) return SCUTE_OK;
    // the output buffers are looked up while the step runs
    for (int i = 0; scatter && i < n_calls; ++i) {
        const LayerRec &L = c->layers[calls[i].layer];
        void *dout = const_cast<void *>(mapped_host(calls[i].out));
        if (!dout) {
            scatter = false;
            break;
        }
        outs.src[outs.n] = dev[i].out;
        outs.dst[outs.n] = dout;
        outs.bytes[outs.n++] = (size_t)n * L.d_out * osz;
    }
    if (scatter) {
        CU_TRY(c, launch_copy_segments(outs, st));
        count_launch(c, 1);
    } else {
        for (int i = 0; i < n_calls; ++i) {
            const LayerRec &L = c->layers[calls[i].layer];
            CU_TRY(c, cudaMemcpyAsync(calls[i].out, dev[i].out, (size_t)n * L.d_out * osz, cudaMemcpyDeviceToHost,
                                      st));
        }
    }
    return SCUTE_OK;
}

scute_status scute_sync_status(scute_ctx *c) {
    if (!c) return SCUTE_ERR_ARG;
    DeviceGuard dg(c->device);
    CU_TRY(c, cudaDeviceSynchronize());
    int s = 0;
    CU_TRY(c, cudaMemcpy(&s, c->d_status, sizeof(int), cudaMemcpyDeviceToHost));
    CU_TRY(c, cudaMemset(c->d_status, 0, sizeof(int)));
    if (s & STATUS_TIMEOUT) return fail(c, SCUTE_ERR_TIMEOUT, "a device-side wait timed out");
    if (s & STATUS_BAD_ADAPTER) return fail(c, SCUTE_ERR_BAD_ADAPTER, "a token id named no registered adapter");
    return SCUTE_OK;
}

scute_status scute_debug_index(scute_ctx *c, const int32_t *ids, int64_t n, int32_t *perm, int32_t *aid_sorted,
                               int32_t *seg_start, int32_t *seg_aid, int32_t *counts, void *stream) {
    if (!c || (n > 0 && (!ids || !perm || !aid_sorted || !seg_aid)) || !seg_start || !counts)
        return fail(c, SCUTE_ERR_ARG, "null argument");
    if (n < 0 || n > c->max_tokens) return fail(c, SCUTE_ERR_ARG, "n out of range");
    DeviceGuard dg(c->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    CU_TRY(c, launch_index(ids, (int)n, c->d_method, c->max_adapters, c->d_perm, c->d_aid, c->d_seg_start,
                           c->d_seg_aid, c->d_meta, c->d_status, st));
    count_launch(c, 1);
    if (n > 0) {
        CU_TRY(c, cudaMemcpyAsync(perm, c->d_perm, 4 * (size_t)n, cudaMemcpyDeviceToDevice, st));
        CU_TRY(c, cudaMemcpyAsync(aid_sorted, c->d_aid, 4 * (size_t)n, cudaMemcpyDeviceToDevice, st));
        CU_TRY(c, cudaMemcpyAsync(seg_aid, c->d_seg_aid, 4 * (size_t)n, cudaMemcpyDeviceToDevice, st));
    }
    CU_TRY(c, cudaMemcpyAsync(seg_start, c->d_seg_start, 4 * (size_t)(n + 1), cudaMemcpyDeviceToDevice, st));
    CU_TRY(c, cudaMemcpyAsync(counts, c->d_meta, sizeof(IndexMeta), cudaMemcpyDeviceToDevice, st));
    return SCUTE_OK;
}

int64_t scute_launch_count(const scute_ctx *c) { return c ? c->launches : 0; }

scute_status scute_timing_enable(scute_ctx *c, int enable) {
    if (!c) return SCUTE_ERR_ARG;
    DeviceGuard dg(c->device);
    if (enable && !c->ev_made) {
        for (int i = 0; i < SCUTE_TIMING_SLOTS; ++i) {
            CU_TRY(c, cudaEventCreate(&c->ev[i][0]));
            CU_TRY(c, cudaEventCreate(&c->ev[i][1]));
        }
        c->ev_made = true;
    }
    c->timing = enable != 0;
    return SCUTE_OK;
}

scute_status scute_timing_reset(scute_ctx *c) {
    if (!c) return SCUTE_ERR_ARG;
    c->t_next = 0;
    c->t_used = 0;
    return SCUTE_OK;
}

void scute_debug_fail_alloc(int k) { g_fail_alloc.store(k > 0 ? k : 0); }

scute_status scute_set_variant(scute_ctx *c, int flags) {
    if (!c) return SCUTE_ERR_ARG;
    if (flags & ~(SCUTE_VARIANT_OFT_PASS | SCUTE_VARIANT_S_PASS)) return fail(c, SCUTE_ERR_ARG, "unknown variant %d", flags);
    if ((flags & SCUTE_VARIANT_OFT_PASS) && c->dtype == SCUTE_BF16) {
        DeviceGuard dg(c->device);
        size_t need = 0;
        for (const auto &L : c->layers)
            if (L.present && (size_t)L.d_in > need) need = (size_t)L.d_in;
        const scute_status st = grow(c, &c->var_x, &c->var_x_cols, need, c->esz,
                                     (size_t)STEP_MAX_CALLS * STEP_MAX_TOKENS);
        if (st) return st;
    }
    c->variant = flags;
    return SCUTE_OK;
}

scute_status scute_debug_inject(scute_ctx *c, int what) {
    if (!c) return SCUTE_ERR_ARG;
    if (what != 0 && what != SCUTE_INJECT_STALL) return fail(c, SCUTE_ERR_ARG, "unknown injection %d", what);
    c->inject = what;
    return SCUTE_OK;
}

scute_status scute_timing_read(scute_ctx *c, float *ms, int max, int *n_out) {
    if (!c || !ms || !n_out) return SCUTE_ERR_ARG;
    DeviceGuard dg(c->device);
    CU_TRY(c, cudaDeviceSynchronize());
    int m = c->t_used < max ? c->t_used : max;
    for (int i = 0; i < m; ++i) CU_TRY(c, cudaEventElapsedTime(&ms[i], c->ev[i][0], c->ev[i][1]));
    *n_out = m;
    return SCUTE_OK;
}

scute_status scute_debug_step_plan(const scute_ctx *c, int64_t *out, int cap, int *n_out) {
    if (!c || !n_out || cap < 0 || (cap > 0 && !out)) return SCUTE_ERR_ARG;
    if (c->last_plan.empty()) return SCUTE_ERR_ARG;
    const int m = (int)c->last_plan.size();
    for (int i = 0; i < m && i < cap; ++i) out[i] = c->last_plan[i];
    *n_out = m;
    return SCUTE_OK;
}

scute_status scute_timing_kinds(const scute_ctx *c, int *kinds, int max, int *n_out) {
    if (!c || !kinds || !n_out) return SCUTE_ERR_ARG;
    int m = c->t_used < max ? c->t_used : max;
    for (int i = 0; i < m; ++i) kinds[i] = c->ev_kind[i];
    *n_out = m;
    return SCUTE_OK;
}

}  // extern "C"
