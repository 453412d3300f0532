// Zero-parameter byte and time model of the adapted layer's calls (host
// arithmetic only).
//
// The article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA"
// (paper-daily.com, section "Where is the cheapest place to compute the
// remaining slots?") measures adapter work in bytes read and written and
// predicts added time as extra bytes / memory bandwidth + extra launches x
// launch cost, with no fitted parameter.  This file lists, for the launch plan
// the library follows, every kernel launch with the bytes it must move (each
// operand read once, each result written once; what a launch keeps to itself
// between its phases is not counted) and its floating-point operations, plus
// the call's algorithmic bytes, and turns a launch list into a predicted time.
#include <cstring>
#include <vector>

#include "ctx.h"

namespace {

void add_kernel(scute_byte_report *r, const char *name, int64_t bytes, int64_t flops) {
    const int k = r->n_kernels++;
    strncpy(r->name[k], name, sizeof(r->name[k]) - 1);
    r->name[k][sizeof(r->name[k]) - 1] = 0;
    r->bytes[k] = bytes;
    r->flops[k] = flops;
}

// What one call of one layer reads, writes and computes, by slot.
struct LayerCount {
    int64_t E, Eo, din, dout, kd, rv, krv, n;
    int64_t distinct = 0, n_lr = 0, lr_rank_rows = 0, n_v = 0, n_rot = 0, segs = 0;
    int64_t live = 0, R = 0, sb = 0, A = 0, B = 0, d = 0, e = 0;
    int64_t n_s = 0, s_pass_vec = 0;   // DoRA / (IA)^3 tokens with a live s, and their distinct s bytes
    int64_t W() const { return din * dout * E; }
    int64_t shared() const { return n_v > 0 ? (din + dout) * rv * E : 0; }
    int64_t x() const { return n * din * E; }
    int64_t out() const { return n * dout * Eo; }
    // W once, each distinct adapter's live tensors once, the shared pair once
    // when a VeRA token is present, x read, out written, ids read
    int64_t algorithmic() const { return W() + live + shared() + x() + out() + 4 * n; }
    // multiply-adds x 2 of every term of the normal form over the batch
    int64_t flops() const {
        return 2 * n * din * dout + 2 * n_rot * din * 32 + 2 * lr_rank_rows * (din + dout) +
               2 * n_v * rv * (din + dout);
    }
};

bool count_layer(const scute_bm_layer *L, const int32_t *ids, int64_t n, LayerCount &c) {
    if (!L || !L->adapters || L->max_adapters < 1 || L->d_in <= 0 || L->d_out <= 0) return false;
    const bool f32 = L->dtype == SCUTE_FP32;
    c.E = f32 ? 4 : 2;
    c.Eo = L->out_dtype == SCUTE_FP32 ? 4 : 2;
    c.din = L->d_in;
    c.dout = L->d_out;
    c.kd = f32 ? 3 * c.din : c.din;
    c.rv = L->shared_rank;
    c.krv = f32 ? 3 * c.rv : c.rv;
    c.n = n;
    std::vector<char> seen((size_t)L->max_adapters, 0);
    bool has_base = false;
    for (int64_t t = 0; t < n; ++t) {
        const int a = ids[t];
        const bool valid = a >= 0 && a < L->max_adapters && L->adapters[a].method >= 0;
        if (!valid) {
            has_base = true;
            continue;
        }
        const scute_bm_adapter &ad = L->adapters[a];
        if (ad.rank > 0) {
            ++c.n_lr;
            c.lr_rank_rows += ad.rank;
        }
        if (ad.has_vera) ++c.n_v;
        if (ad.has_R) ++c.n_rot;
        const bool sp = ad.has_s && (ad.method == SCUTE_DORA || ad.method == SCUTE_IA3);
        if (sp) ++c.n_s;
        if (seen[a]) continue;
        if (sp) c.s_pass_vec += 4 * c.dout;
        seen[a] = 1;
        ++c.distinct;
        if (ad.has_s) { c.live += 4 * c.dout; c.sb += 4 * c.dout; }
        if (ad.has_b) { c.live += 4 * c.dout; c.sb += 4 * c.dout; }
        if (ad.has_R) { c.live += 32 * c.din * c.E; c.R += 32 * c.din * c.E; }
        if (ad.rank > 0) {
            c.live += (int64_t)ad.rank * (c.din + c.dout) * c.E;
            c.A += (int64_t)ad.rank * c.din * c.E;
            c.B += (int64_t)ad.rank * c.dout * c.E;
        }
        if (ad.has_vera) {
            c.live += 4 * c.rv;
            c.d += 4 * c.rv;
            if (ad.has_vera_e) { c.live += 4 * c.dout; c.e += 4 * c.dout; }
        }
    }
    c.segs = c.distinct + (has_base ? 1 : 0);
    return true;
}

// The per-kernel plan (fp32 contexts and batches above the decode step's
// token limit): indexing, rotation into the sorted token operand, base GEMM,
// owned low-rank shrink and expand, VeRA shrink and expand GEMMs.  In bf16
// contexts with more than 256 tokens the owned shrink runs before the base
// GEMM and the owned expand inside its epilogue (the GEMM then also reads the
// partial v and each B', and writes out once); there the VeRA shrink of a
// shared rank that is a multiple of 64 (its tensor-core form) also comes
// before the base GEMM.
void per_kernel_plan(const scute_bm_layer *L, const LayerCount &c, scute_byte_report *rep) {
    const int64_t n = c.n, E = c.E, Eo = c.Eo;
    const int64_t index_out = 8 * n + 4 * (c.segs + 1) + 4 * c.segs + 88;
    const int64_t ks = scute::lowrank_ks(L->d_in, nullptr);
    const bool fused = L->lowrank_launched && L->dtype != SCUTE_FP32 && n > 256;
    add_kernel(rep, "index", 4 * n + index_out, 0);
    add_kernel(rep, "rotate", n * c.din * E + 8 * n + c.R + n * c.kd * E, 2 * c.n_rot * c.din * 32);
    const int64_t shrink_b = c.n_lr * c.din * E + c.A + ks * c.lr_rank_rows * 4;
    const int64_t shA = c.n_v > 0 ? c.rv * c.kd * E : 0;
    const int64_t shB = c.n_v > 0 ? c.dout * c.krv * E : 0;
    const int64_t vshrink_b = c.n_v * c.kd * E + shA + c.d + c.n_v * c.krv * E;
    const int64_t vshrink_f = 2 * c.n_v * c.rv * c.kd;
    const bool vs_first = L->vera_launched && L->dtype != SCUTE_FP32 && n > 256 && c.rv % 64 == 0;
    if (fused) add_kernel(rep, "lr_shrink", shrink_b, 2 * c.lr_rank_rows * c.din);
    if (vs_first) add_kernel(rep, "vera_shrink", vshrink_b, vshrink_f);
    int64_t gemm_b = c.dout * c.kd * E + n * c.kd * E + c.sb + 8 * n + n * c.dout * Eo;
    int64_t gemm_f = 2 * n * c.kd * c.dout;
    if (fused) {
        gemm_b += ks * c.lr_rank_rows * 4 + c.B;
        gemm_f += 2 * c.lr_rank_rows * c.dout;
    }
    add_kernel(rep, "base_gemm", gemm_b, gemm_f);
    if (L->lowrank_launched && !fused) {
        add_kernel(rep, "lr_shrink", shrink_b, 2 * c.lr_rank_rows * c.din);
        add_kernel(rep, "lr_expand", ks * c.lr_rank_rows * 4 + c.B + 2 * c.n_lr * c.dout * Eo,
                   2 * c.lr_rank_rows * c.dout);
    }
    if (L->vera_launched) {
        if (!vs_first) add_kernel(rep, "vera_shrink", vshrink_b, vshrink_f);
        add_kernel(rep, "vera_expand", c.n_v * c.krv * E + shB + c.e + 2 * c.n_v * c.dout * Eo,
                   2 * c.n_v * c.krv * c.dout);
    }
}

}  // namespace

extern "C" {

scute_status scute_byte_model(const scute_bm_layer *L, const int32_t *ids, int64_t n,
                              scute_byte_report *rep) {
    return scute_byte_model_batch(L, L ? 1 : 0, ids, n, rep);
}

scute_status scute_byte_model_batch(const scute_bm_layer *layers, int n_layers, const int32_t *ids, int64_t n,
                                    scute_byte_report *rep) {
    if (!layers || !rep || n_layers < 1 || n_layers > SCUTE_MAX_CALLS || n < 0 || (n > 0 && !ids))
        return SCUTE_ERR_ARG;
    memset(rep, 0, sizeof(*rep));
    std::vector<LayerCount> cs((size_t)n_layers);
    for (int i = 0; i < n_layers; ++i) {
        if (!count_layer(&layers[i], ids, n, cs[i])) return SCUTE_ERR_ARG;
        if (layers[i].dtype != layers[0].dtype) return SCUTE_ERR_ARG;
    }
    // bf16 batches of at most STEP_MAX_TOKENS tokens are one launch of the
    // decode step over every listed layer: its bytes are what crosses the
    // launch (ids once; every layer's W, live adapter tensors, shared pair, x
    // and out); the token operand, low-rank and VeRA intermediates and the
    // partial tiles stay inside it
    const bool step = layers[0].dtype != SCUTE_FP32 && n <= scute::STEP_MAX_TOKENS;
    int64_t alg = 4 * n, adapter = 0, wbytes = 0;
    for (const LayerCount &c : cs) {
        alg += c.algorithmic() - 4 * n;
        adapter += c.live + c.shared();
        wbytes += c.W();
    }
    if (step) {
        const int var = layers[0].variant;
        int64_t fl = 0, step_bytes = alg;
        for (const LayerCount &c : cs) fl += c.flops();
        if (var & SCUTE_VARIANT_OFT_PASS) {
            // x read, R of each distinct rotating adapter, the rotated copy
            // written (per layer), ids once; the step no longer reads R
            int64_t b = 4 * n, f = 0;
            for (const LayerCount &c : cs) {
                b += 2 * c.n * c.din * c.E + c.R;
                f += 2 * c.n_rot * c.din * 32;
                step_bytes -= c.R;
            }
            fl -= f;
            add_kernel(rep, "oft_pass", b, f);
        }
        int64_t sb = 4 * n, sf = 0;
        if (var & SCUTE_VARIANT_S_PASS) {
            // the DoRA and (IA)^3 rows of out read and written again, their
            // distinct s vectors, ids once; the step no longer reads those s
            for (const LayerCount &c : cs) {
                sb += 2 * c.n_s * c.dout * c.Eo + c.s_pass_vec;
                sf += c.n_s * c.dout;
                step_bytes -= c.s_pass_vec;
            }
        }
        add_kernel(rep, "step", step_bytes, fl);
        if (var & SCUTE_VARIANT_S_PASS) add_kernel(rep, "s_pass", sb, sf);
    } else {
        for (int i = 0; i < n_layers; ++i) {
            if (rep->n_kernels + 7 > SCUTE_BM_MAX_KERNELS) return SCUTE_ERR_UNSUPPORTED;
            per_kernel_plan(&layers[i], cs[i], rep);
        }
    }
    rep->algorithmic_bytes = alg;
    rep->adapter_bytes = adapter;
    rep->base_weight_bytes = wbytes;
    rep->distinct_adapters = (int32_t)cs[0].distinct;   // the same on every layer of a batch
    return SCUTE_OK;
}

scute_status scute_predict_time(const scute_byte_report *rep, double hbm_gbs, double tensor_tflops,
                                double launch_us, double *us_out) {
    if (!rep || !us_out || !(hbm_gbs > 0.0) || launch_us < 0.0 || rep->n_kernels < 0 ||
        rep->n_kernels > SCUTE_BM_MAX_KERNELS)
        return SCUTE_ERR_ARG;
    double us = 0.0;
    for (int k = 0; k < rep->n_kernels; ++k) {
        const double t_mem = (double)rep->bytes[k] / (hbm_gbs * 1e3);   // bytes / (GB/s) in us
        const double t_math = tensor_tflops > 0.0 ? (double)rep->flops[k] / (tensor_tflops * 1e6) : 0.0;
        us += t_mem > t_math ? t_mem : t_math;
    }
    *us_out = us + launch_us * rep->n_kernels;
    return SCUTE_OK;
}

static void fill_layer(const scute_ctx *c, int layer, scute_dtype out_dtype, std::vector<scute_bm_adapter> &ads,
                       scute_bm_layer &bl) {
    const LayerRec &L = c->layers[layer];
    ads.assign((size_t)c->max_adapters, scute_bm_adapter{});
    for (int a = 0; a < c->max_adapters; ++a) {
        scute_bm_adapter &b = ads[a];
        memset(&b, 0, sizeof(b));
        b.method = c->adapters[a].used ? c->adapters[a].method : -1;
        if (!c->adapters[a].used) continue;
        for (const auto &al : c->adapters[a].layers) {
            if (al.layer != layer) continue;
            b.rank = al.rank;
            b.has_s = al.s;
            b.has_b = al.b;
            b.has_R = al.R;
            b.has_vera = al.vera;
            b.has_vera_e = al.vera_e;
        }
    }
    bl.dtype = c->dtype;
    bl.out_dtype = out_dtype;
    bl.d_in = L.d_in;
    bl.d_out = L.d_out;
    bl.shared_rank = L.rv;
    bl.lowrank_launched = L.n_lr > 0;
    bl.vera_launched = L.rv > 0 && L.n_vera > 0;
    bl.max_adapters = c->max_adapters;
    bl.adapters = ads.data();
    bl.variant = c->variant;
}

scute_status scute_predict_bytes(const scute_ctx *c, const int32_t *ids, int64_t n, int layer,
                                 scute_dtype out_dtype, scute_byte_report *rep) {
    if (!c || layer < 0 || layer >= c->max_layers || !c->layers[layer].present) return SCUTE_ERR_ARG;
    std::vector<scute_bm_adapter> ads;
    scute_bm_layer bl;
    fill_layer(c, layer, out_dtype, ads, bl);
    return scute_byte_model(&bl, ids, n, rep);
}

scute_status scute_predict_batch(const scute_ctx *c, const scute_call *calls, int n_calls, const int32_t *ids,
                                 int64_t n, scute_dtype out_dtype, scute_byte_report *rep) {
    if (!c || !calls || n_calls < 1 || n_calls > SCUTE_MAX_CALLS) return SCUTE_ERR_ARG;
    std::vector<std::vector<scute_bm_adapter>> ads((size_t)n_calls);
    std::vector<scute_bm_layer> bls((size_t)n_calls);
    for (int i = 0; i < n_calls; ++i) {
        const int layer = calls[i].layer;
        if (layer < 0 || layer >= c->max_layers || !c->layers[layer].present) return SCUTE_ERR_ARG;
        fill_layer(c, layer, out_dtype, ads[i], bls[i]);
    }
    return scute_byte_model_batch(bls.data(), n_calls, ids, n, rep);
}

}  // extern "C"
