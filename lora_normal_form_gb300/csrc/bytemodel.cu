// Zero-parameter byte model of one scute_linear call (host arithmetic only).
//
// The article "Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA"
// (paper-daily.com, section "Where is the cheapest place to compute the
// remaining slots?") measures adapter work in bytes read and written and
// predicts added time as extra bytes / memory bandwidth + extra launches x
// launch cost, with no fitted parameter.  This file counts, for the launch plan
// scute_linear follows, the bytes each kernel must move (every operand read
// once, every result written once) and the call's algorithmic bytes.
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

}  // namespace

extern "C" {

scute_status scute_byte_model(const scute_bm_layer *L, const int32_t *ids, int64_t n,
                              scute_byte_report *rep) {
    if (!L || !rep || n < 0 || (n > 0 && !ids) || !L->adapters || L->max_adapters < 1 ||
        L->d_in <= 0 || L->d_out <= 0)
        return SCUTE_ERR_ARG;
    memset(rep, 0, sizeof(*rep));
    const bool f32 = L->dtype == SCUTE_FP32;
    const int64_t E = f32 ? 4 : 2;
    const int64_t Eo = L->out_dtype == SCUTE_FP32 ? 4 : 2;
    const int64_t din = L->d_in, dout = L->d_out;
    const int64_t kd = f32 ? 3 * din : din;
    const int64_t rv = L->shared_rank;
    const int64_t krv = f32 ? 3 * rv : rv;

    std::vector<char> seen((size_t)L->max_adapters, 0);
    int64_t distinct = 0, n_lr = 0, lr_rank_rows = 0, n_v = 0, n_rot = 0;
    bool has_base = false;
    int64_t live = 0, sum_R = 0, sum_sb = 0, sum_A = 0, sum_B = 0, sum_d = 0, sum_e = 0;
    for (int64_t t = 0; t < n; ++t) {
        const int a = ids[t];
        const bool valid = a >= 0 && a < L->max_adapters && L->adapters[a].method >= 0;
        if (!valid) {
            has_base = true;
            continue;
        }
        const scute_bm_adapter &ad = L->adapters[a];
        if (ad.rank > 0) {
            ++n_lr;
            lr_rank_rows += ad.rank;
        }
        if (ad.has_vera) ++n_v;
        if (ad.has_R) ++n_rot;
        if (seen[a]) continue;
        seen[a] = 1;
        ++distinct;
        if (ad.has_s) { live += 4 * dout; sum_sb += 4 * dout; }
        if (ad.has_b) { live += 4 * dout; sum_sb += 4 * dout; }
        if (ad.has_R) { live += 32 * din * E; sum_R += 32 * din * E; }
        if (ad.rank > 0) {
            live += (int64_t)ad.rank * (din + dout) * E;
            sum_A += (int64_t)ad.rank * din * E;
            sum_B += (int64_t)ad.rank * dout * E;
        }
        if (ad.has_vera) {
            live += 4 * rv;
            sum_d += 4 * rv;
            if (ad.has_vera_e) { live += 4 * dout; sum_e += 4 * dout; }
        }
    }
    const int64_t segs = distinct + (has_base ? 1 : 0);

    // bf16 calls with at most 128 tokens run the fused decode plan: one
    // prologue (indexing, rotation, both shrinks) and one GEMM whose epilogue
    // applies s, b and both expands
    const bool fused = !f32 && n <= 128;
    const int64_t index_out = 8 * n + 4 * (segs + 1) + 4 * segs + 88;
    if (fused) {
        const int64_t shA = n_v > 0 ? rv * din * E : 0;
        const int64_t shB = n_v > 0 ? dout * rv * E : 0;
        add_kernel(rep, "prep",
                   4 * n + n * din * E + sum_R + sum_A + shA + sum_d + n * kd * E + lr_rank_rows * 4 +
                       n_v * rv * E + index_out,
                   2 * n_rot * din * 32 + 2 * lr_rank_rows * din + 2 * n_v * rv * din);
        add_kernel(rep, "base_gemm",
                   dout * kd * E + n * kd * E + sum_sb + sum_B + lr_rank_rows * 4 + shB + n_v * rv * E + sum_e +
                       8 * n + n * dout * Eo,
                   2 * n * kd * dout + 2 * lr_rank_rows * dout + 2 * n_v * rv * dout);
    } else {
        add_kernel(rep, "index", 4 * n + index_out, 0);
        add_kernel(rep, "rotate", n * din * E + 8 * n + sum_R + n * kd * E, 2 * n_rot * din * 32);
        add_kernel(rep, "base_gemm", dout * kd * E + n * kd * E + sum_sb + 8 * n + n * dout * Eo,
                   2 * n * kd * dout);
        if (L->lowrank_launched) {
            const int64_t ks = scute::lowrank_ks(L->d_in, nullptr);
            add_kernel(rep, "lr_shrink", n_lr * din * E + sum_A + ks * lr_rank_rows * 4, 2 * lr_rank_rows * din);
            add_kernel(rep, "lr_expand", ks * lr_rank_rows * 4 + sum_B + 2 * n_lr * dout * Eo,
                       2 * lr_rank_rows * dout);
        }
        if (L->vera_launched) {
            const int64_t shA = n_v > 0 ? rv * kd * E : 0;
            const int64_t shB = n_v > 0 ? dout * krv * E : 0;
            add_kernel(rep, "vera_shrink", n_v * kd * E + shA + sum_d + n_v * krv * E, 2 * n_v * rv * kd);
            add_kernel(rep, "vera_expand", n_v * krv * E + shB + sum_e + 2 * n_v * dout * Eo,
                       2 * n_v * krv * dout);
        }
    }
    const int64_t shared = n_v > 0 ? (din + dout) * rv * E : 0;
    rep->base_weight_bytes = din * dout * E;
    rep->adapter_bytes = live + shared;
    rep->algorithmic_bytes = rep->base_weight_bytes + rep->adapter_bytes + n * din * E + n * dout * Eo + 4 * n;
    rep->distinct_adapters = (int32_t)distinct;
    return SCUTE_OK;
}

scute_status scute_predict_bytes(const scute_ctx *c, const int32_t *ids, int64_t n, int layer,
                                 scute_dtype out_dtype, scute_byte_report *rep) {
    if (!c || layer < 0 || layer >= c->max_layers || !c->layers[layer].present) return SCUTE_ERR_ARG;
    const LayerRec &L = c->layers[layer];
    std::vector<scute_bm_adapter> ads((size_t)c->max_adapters);
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
    scute_bm_layer bl;
    bl.dtype = c->dtype;
    bl.out_dtype = out_dtype;
    bl.d_in = L.d_in;
    bl.d_out = L.d_out;
    bl.shared_rank = L.rv;
    bl.lowrank_launched = L.n_lr > 0;
    bl.vera_launched = L.rv > 0 && L.n_vera > 0;
    bl.max_adapters = c->max_adapters;
    bl.adapters = ads.data();
    return scute_byte_model(&bl, ids, n, rep);
}

}  // extern "C"
