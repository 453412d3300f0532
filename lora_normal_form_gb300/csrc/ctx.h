// Private definition of the context object shared by the host runtime files.
#pragma once

#include <string>
#include <vector>

#include "internal.h"
#include "scute.h"

namespace scute {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct LayerRec {
    bool present = false;
    int d_in = 0, d_out = 0, kdim = 0;
    void *Wt = nullptr;  // [d_out][kdim]
    CUtensorMap mapW, mapXs;
    int rv = 0, krv = 0;
    void *Ash = nullptr;  // [rv][kdim]
    void *Bsh = nullptr;  // [d_out][krv]
    CUtensorMap mapAsh, mapBsh, mapU;
    int n_lr = 0;         // registered adapters with an owned term here
    int n_vera = 0;       // registered adapters with a VeRA term here
    int n_rot = 0;        // registered adapters with a rotation here
    int n_rot_lr = 0;     // registered adapters with both a rotation and an owned term here
};

struct AdapterLayer {
    int layer;
    int rank;      // owned rank (0 none)
    bool s, b, R, vera, vera_e;
};

struct AdapterRec {
    bool used = false;
    int method = -1;
    void *storage = nullptr;
    std::vector<AdapterLayer> layers;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace scute

using namespace scute;

struct scute_ctx {
    int device = 0;
    scute_dtype dtype = SCUTE_BF16;
    int esz = 2;
    int max_tokens = 0, max_adapters = 0, max_layers = 0;
    int num_sms = 0;
    bool pdl = true;
    std::vector<LayerRec> layers;
    std::vector<AdapterRec> adapters;
    std::vector<int8_t> h_method;
    Slot *d_slots = nullptr;
    int8_t *d_method = nullptr;
    int *d_perm = nullptr, *d_aid = nullptr, *d_seg_start = nullptr, *d_seg_aid = nullptr;
    int *d_seg_unit = nullptr;   // work units of the segmented low-rank kernels
    int *d_seg_tile = nullptr;   // 128-row tiles of the tensor-core low-rank shrink
    float *vs_part = nullptr;    // VeRA shrink partial tiles [VS_KS][max_tokens][rv] (prefill, bf16)
    size_t vs_part_cols = 0;
    int *vs_ctr = nullptr;       // VeRA shrink tile counters (VS_CTR_INTS, zero between launches)
    IndexMeta *d_meta = nullptr;
    int *d_status = nullptr;
    int *d_err = nullptr;
    float *v_part = nullptr;
    float *gpart = nullptr;      // K-split partial tiles of the GEMM
    void *xs = nullptr;
    size_t xs_cols = 0;  // elements per row the xs buffer holds
    void *U = nullptr;
    size_t u_cols = 0;
    void *st_x = nullptr, *st_out = nullptr;
    int32_t *st_ids = nullptr;
    size_t st_x_cols = 0, st_out_cols = 0;
    void *tmp = nullptr;
    size_t tmp_bytes = 0;
    // decode-step workspace: STEP_MAX_CALLS slots of STEP_MAX_TOKENS rows each
    void *step_xs = nullptr;     // token operands, slot row pitch step_xs_cols elements
    size_t step_xs_cols = 0;
    void *step_U = nullptr;      // VeRA intermediates
    size_t step_u_cols = 0;
    float *step_pre = nullptr;   // owned low-rank rows b + v B': per call slot [planes][128][d_out]
    size_t step_pre_floats = 0;  // capacity (all STEP_MAX_CALLS slots)
    float *step_part = nullptr;  // partial tiles
    size_t step_part_floats = 0;
    int *step_sync = nullptr;    // counters (STEP_SYNC_INTS, zero between launches)
    void *step_hx = nullptr;     // host-call staging of the inputs / outputs
    size_t step_hx_cols = 0;
    void *step_hout = nullptr;
    size_t step_hout_cols = 0;
    int step_bn_max = 64;
    int smem_optin = 0;
    int inject = 0;              // scute_debug_inject, consumed by the next decode launch
    int variant = 0;             // scute_set_variant: slots placed in separate passes
    std::vector<int64_t> last_plan;   // scute_debug_step_plan: the last decode launch's plan
    void *var_x = nullptr;       // rotated copies of the calls' x (separate rotation pass)
    size_t var_x_cols = 0;
    PFN_encodeTiled encode = nullptr;
    int64_t launches = 0;
    bool timing = false;
    cudaEvent_t ev[SCUTE_TIMING_SLOTS][2];
    int ev_kind[SCUTE_TIMING_SLOTS] = {};
    bool ev_made = false;
    int t_next = 0, t_used = 0;
    char err[512];
};

