// C ABI of the DFlash round (include/dflash.h): configuration guards,
// workspace layout, TMA descriptors and the launch sequence of each call.
//
// The guards check the drafter against the target (hidden size, vocabulary,
// tap layers) before any buffer is touched ("feat: DFlash2 block-diffusion
// drafter for Qwen 3.8", the config-guard commit: a checkpoint with the
// right vocabulary and layer count but another hidden size had been
// accepted).  The calls follow the round of "[RFC] DFlash", "Key
// Implementation Details": taps (Phase 1), draft, batched verify,
// first-mismatch acceptance and KV-cache rollback (Phase 3).
//
// The library never allocates device memory and never synchronises except
// in dflash_stats / dflash_check; every launch goes to the caller's stream,
// so the launches of a round can be captured in a CUDA graph.

#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/dflash.h"
#include "attention.cuh"
#include "gemm_tc.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"
#include "capi_internal.cuh"

using namespace dfl;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

#define CUDA_TRY(x)                                                                   \
    do {                                                                              \
        cudaError_t e_ = (x);                                                         \
        if (e_ != cudaSuccess)                                                        \
            return fail(DFLASH_ERR_CUDA, "%s: %s", #x, cudaGetErrorString(e_));       \
    } while (0)

#define LAUNCH_TRY(x)                                                                 \
    do {                                                                              \
        if ((x) != 0) {                                                               \
            cudaError_t e_ = cudaGetLastError();                                      \
            return fail(DFLASH_ERR_CUDA, "%s failed: %s", #x, cudaGetErrorString(e_)); \
        }                                                                             \
    } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int elem_size(int dtype) { return dtype == DFLASH_F32 ? 4 : 2; }

// positions per (layer, K|V, head) run of a cache: max_seq rounded up to a
// whole number of 64-key attention chunks
int cache_cap(const dflash_config& c) { return (c.max_seq + 63) / 64 * 64; }

int max_chunks(const dflash_config& c) { return cache_cap(c) / ATTN_CHUNK; }

// The tap commit projects the committed context rows for every draft layer
// in one GEMM over a copy of the layers' [W_k; W_v] (bf16 drafters of more
// than one layer whose [W_k; W_v] fills whole 128-row tiles).
bool ctxkv_grouped(const dflash_config& c) {
    return c.dtype == DFLASH_BF16 && c.drf_layers > 1 && (2 * c.n_kv * c.head_dim) % GEMM_BN == 0 &&
           GEMM_BN % c.head_dim == 0;
}

// ------------------------------------------------------------------ layout

struct Layout {
    size_t state, x, hn, ssq, qrot, attn, act, taps, rcos, rsin, invf, rtab, ctxkv_w, ctxkv_kn, amax, part,
        slots, counters,
        acnt, pf_x, pf_xlo, pf_y, pf_chi, pf_clo, pf_w, pp_x, pp_y, pp_hi, pp_lo, pp_ahi, pp_alo, pp_q,
        pp_thi, pp_tlo, pf_rope, pp_w, total;
};

constexpr int MAX_SMS = 256 * DFL_GEMM_CTAS_PER_SM;   // GEMM CTAs (split-K slots)

// Fewest 64-key chunks one attention split folds (build knob).
#ifndef DFL_ATTN_MIN_SPLIT
#define DFL_ATTN_MIN_SPLIT 1
#endif
constexpr int MAX_TILES = 8192;

// Dense prompt prefill of a bf16 target (every prompt row before the last
// 16-row chunk): the shapes the dense GEMM's tiles and segments cover.
bool dense_ingest_ok(const dflash_config& c);
bool dense_prefill_ok(const dflash_config& c) {
    const int qd = c.n_q * c.head_dim, kvd = c.n_kv * c.head_dim;
    return c.dtype == DFLASH_BF16 && c.tgt_layers > 0 &&
           (c.tgt_wfmt == DFLASH_BF16 || c.tgt_wfmt == DFLASH_INT4G64) &&
           (c.drf_layers == 0 || dense_ingest_ok(c)) && c.hidden % 256 == 0 && qd % 256 == 0 &&
           kvd % 256 == 0 && c.ffn % 256 == 0 && (c.head_dim == 128 || c.head_dim == 64);
}

// Window ingest on the dense tcgen05 GEMM: rows per pass, and whether the
// configuration has it (bf16 drafter, shapes the GEMM's tiles cover).
constexpr int PF_ROWS = 1024;
bool dense_ingest_ok(const dflash_config& c) {
    return c.dtype == DFLASH_BF16 && c.drf_layers > 0 && c.n_taps > 0 &&
           (c.drf_wfmt == DFLASH_BF16 || c.drf_wfmt == DFLASH_INT4G64) && c.hidden % 64 == 0 &&
           (c.n_kv * c.head_dim) % 256 == 0 && c.hidden % 4 == 0;
}

// Workspace carving.  hn holds the next GEMM's normalised input rows
// (x * w_norm, activation type) and ssq their per-128-column partial sums
// of x^2, from which the consuming GEMM derives the RMSNorm row scale.
// GEMM inputs (hn, attn, act, taps) take 4 bytes per (row, column): fp32
// rows, or the [32][width] hi/lo bf16 planes of the bf16 models.
Layout make_layout(const dflash_config& c) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    const size_t R = DFL_MAX_ROWS;
    const int es = elem_size(c.dtype);
    const int qd = c.n_q * c.head_dim;
    L.state = take(sizeof(DevState));
    L.x = take(R * c.hidden * 4);
    L.hn = take(R * c.hidden * 4);
    L.ssq = take(R * (c.hidden / 128 + 1) * 4);
    L.qrot = take(R * qd * es);
    L.attn = take(R * qd * 4);
    L.act = take(R * c.ffn * 4);
    L.taps = take(R * (size_t)(c.n_taps > 0 ? c.n_taps : 1) * c.hidden * 4);
    L.rcos = take(R * (c.head_dim / 2) * 4);
    L.rsin = take(R * (c.head_dim / 2) * 4);
    L.invf = take((c.head_dim / 2) * 8);
    // RoPE angles of every cache position: cos [cap][head_dim / 2], then sin
    L.rtab = take((size_t)2 * cache_cap(c) * (c.head_dim / 2) * 4);
    if (ctxkv_grouped(c)) {   // every draft layer's [W_k; W_v] and k-norm, one after another
        const size_t rows = (size_t)c.drf_layers * 2 * c.n_kv * c.head_dim;
        if (c.drf_wfmt == DFLASH_INT4G64) {   // codes [rows][hidden / 2], then scales [hidden / 64][rows]
            L.ctxkv_w = take(rows * (c.hidden / 2) + rows * (c.hidden / 64) * 2);
        } else {
            L.ctxkv_w = take(rows * c.hidden * 2);
        }
        L.ctxkv_kn = take((size_t)c.drf_layers * c.head_dim * 4);
    }
    L.amax = take(R * 8);
    L.part = take((size_t)max_chunks(c) * R * c.n_q * (c.head_dim + 2) * 4);
    L.slots = take((size_t)MAX_SMS * 2 * GEMM_BN * R * 4);
    L.counters = take((size_t)MAX_TILES * 4);
    L.acnt = take((size_t)2 * c.n_kv * 4);
    if (dense_ingest_ok(c)) {   // [PF_ROWS] rows: taps bf16, GEMM out fp32, context rows hi/lo bf16
        const size_t kv = (size_t)2 * c.n_kv * c.head_dim;
        L.pf_x = take((size_t)PF_ROWS * c.n_taps * c.hidden * 2);
        L.pf_xlo = take((size_t)PF_ROWS * c.n_taps * c.hidden * 2);   // lo plane of hc-mean taps
        L.pf_y = take((size_t)PF_ROWS * (kv > (size_t)c.hidden ? kv : (size_t)c.hidden) * 4);
        L.pf_chi = take((size_t)PF_ROWS * c.hidden * 2);
        L.pf_clo = take((size_t)PF_ROWS * c.hidden * 2);
        if (c.drf_wfmt == DFLASH_INT4G64)   // one layer's [W_k; W_v] dequantised to f16
            L.pf_w = take(kv * c.hidden * 2);
        L.pf_rope = take((size_t)PF_ROWS * c.head_dim * 4);   // cos, sin [PF_ROWS][head_dim / 2]
    }
    if (dense_prefill_ok(c)) {   // [PF_ROWS] rows of a dense target forward
        const size_t qd = (size_t)c.n_q * c.head_dim, kvd = (size_t)c.n_kv * c.head_dim;
        size_t ywide = qd + 2 * kvd;
        if ((size_t)2 * c.ffn > ywide) ywide = (size_t)2 * c.ffn;
        if ((size_t)c.hidden > ywide) ywide = c.hidden;
        size_t xwide = c.hidden;
        if (qd > xwide) xwide = qd;
        if ((size_t)c.ffn > xwide) xwide = c.ffn;
        L.pp_x = take((size_t)PF_ROWS * c.hidden * 4);
        L.pp_y = take((size_t)PF_ROWS * ywide * 4);
        L.pp_hi = take((size_t)PF_ROWS * xwide * 2);
        L.pp_lo = take((size_t)PF_ROWS * xwide * 2);
        L.pp_ahi = take((size_t)PF_ROWS * c.ffn * 2);   // SwiGLU output planes: W_down's input
        L.pp_alo = take((size_t)PF_ROWS * c.ffn * 2);
        L.pp_q = take((size_t)PF_ROWS * qd * 2);
        if (!L.pf_rope) L.pf_rope = take((size_t)PF_ROWS * c.head_dim * 4);
        if (c.tgt_wfmt == DFLASH_INT4G64) {   // the largest of a layer's matrices, dequantised to f16
            size_t wmax = (qd + 2 * kvd) * c.hidden;
            if ((size_t)2 * c.ffn * c.hidden > wmax) wmax = (size_t)2 * c.ffn * c.hidden;
            L.pp_w = take(wmax * 2);
        }
        if (c.drf_layers > 0) {
            L.pp_thi = take((size_t)PF_ROWS * c.n_taps * c.hidden * 2);
            L.pp_tlo = take((size_t)PF_ROWS * c.n_taps * c.hidden * 2);
        }
    }
    L.total = off;
    return L;
}

// ------------------------------------------------------------------ validation

int validate(const dflash_config* c) {
    if (!c) return fail(DFLASH_ERR_ARG, "config is NULL");
    if (c->hidden <= 0 || c->hidden % 128) return fail(DFLASH_ERR_CONFIG, "hidden %d: must be a positive multiple of 128", c->hidden);
    if (c->head_dim != 64 && c->head_dim != 128) return fail(DFLASH_ERR_CONFIG, "head_dim %d: 64 or 128", c->head_dim);
    if (c->n_q <= 0 || c->n_kv <= 0 || c->n_q % c->n_kv) return fail(DFLASH_ERR_CONFIG, "n_q %d / n_kv %d: n_q must be a multiple of n_kv", c->n_q, c->n_kv);
    if ((c->n_q / c->n_kv) * DFL_MAX_ROWS > 256) return fail(DFLASH_ERR_CONFIG, "query group too large");
    if ((c->n_q * c->head_dim) % 128 || (c->n_kv * c->head_dim) % 128) return fail(DFLASH_ERR_CONFIG, "n_q*head_dim and n_kv*head_dim must be multiples of 128");
    if (c->ffn <= 0 || c->ffn % 64) return fail(DFLASH_ERR_CONFIG, "ffn %d: multiple of 64", c->ffn);
    if (c->vocab <= 0 || c->vocab % 128) return fail(DFLASH_ERR_CONFIG, "vocab %d: multiple of 128", c->vocab);
    if (c->vocab / 128 > MAX_TILES) return fail(DFLASH_ERR_CONFIG, "vocab too large");
    if (c->block_max < 1 || c->block_max > DFLASH_MAX_BLOCK) return fail(DFLASH_ERR_CONFIG, "block_max %d: 1..16", c->block_max);
    if (c->tgt_layers < 0 || c->drf_layers < 0 || (c->tgt_layers == 0 && c->drf_layers == 0)) return fail(DFLASH_ERR_CONFIG, "need a target or a drafter");
    if (c->max_seq < 2) return fail(DFLASH_ERR_CONFIG, "max_seq %d", c->max_seq);
    if (c->window < 0) return fail(DFLASH_ERR_CONFIG, "window %d", c->window);
    if (c->dtype != DFLASH_F32 && c->dtype != DFLASH_BF16) return fail(DFLASH_ERR_CONFIG, "dtype %d: F32 or BF16", c->dtype);
    if (c->dtype == DFLASH_BF16 && c->n_q / c->n_kv > 4)
        return fail(DFLASH_ERR_CONFIG, "%d q heads per kv head: the BF16 attention takes at most 4", c->n_q / c->n_kv);
    if (c->drf_layers > 0) {
        if (c->n_taps < 1 || c->n_taps > DFLASH_MAX_TAPS) return fail(DFLASH_ERR_CONFIG, "n_taps %d: 1..8", c->n_taps);
        for (int i = 0; i < c->n_taps; ++i) {
            if (c->tap_layer[i] < 0 || (c->tgt_layers > 0 && c->tap_layer[i] >= c->tgt_layers))
                return fail(DFLASH_ERR_CONFIG, "tap layer %d out of range", c->tap_layer[i]);
            if (i > 0 && c->tap_layer[i] <= c->tap_layer[i - 1]) return fail(DFLASH_ERR_CONFIG, "tap layers must increase");
        }
    }
    auto fmt_ok = [&](int f) {
        if (c->dtype == DFLASH_F32) return f == DFLASH_F32;
        return f == DFLASH_BF16 || f == DFLASH_INT4G64;
    };
    if (c->tgt_layers > 0 && !fmt_ok(c->tgt_wfmt)) return fail(DFLASH_ERR_CONFIG, "tgt_wfmt %d not supported with dtype %d", c->tgt_wfmt, c->dtype);
    if (c->drf_layers > 0 && !fmt_ok(c->drf_wfmt)) return fail(DFLASH_ERR_CONFIG, "drf_wfmt %d not supported with dtype %d", c->drf_wfmt, c->dtype);
    if (c->adaptive_block != 0 && c->adaptive_block != 1)
        return fail(DFLASH_ERR_CONFIG, "adaptive_block %d: 0 or 1", c->adaptive_block);
    if (c->lm_wfmt != 0 && !(c->dtype == DFLASH_BF16 && c->lm_wfmt == DFLASH_INT4G64))
        return fail(DFLASH_ERR_CONFIG, "lm_wfmt %d: 0 (tied embedding) or INT4G64 with dtype BF16", c->lm_wfmt);
    const bool int4 = (c->tgt_layers > 0 && c->tgt_wfmt == DFLASH_INT4G64) ||
                      (c->drf_layers > 0 && c->drf_wfmt == DFLASH_INT4G64) ||
                      c->lm_wfmt == DFLASH_INT4G64;
    if (int4 && (c->hidden % 256 || (c->n_q * c->head_dim) % 256 || c->ffn % 256))
        return fail(DFLASH_ERR_CONFIG, "INT4 projections need hidden, n_q*head_dim and ffn to be multiples of 256");
    if (c->eos_id >= c->vocab) return fail(DFLASH_ERR_CONFIG, "eos_id %d >= vocab", c->eos_id);
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return fail(DFLASH_ERR_CONFIG, "rms_eps / rope_theta must be positive");
    return DFLASH_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ------------------------------------------------------------------ TMA maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encode() {
    if (g_encode) return DFLASH_OK;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return DFLASH_OK;
}

// 2D map over a row-major [rows][inner] matrix of es-byte elements.
int make_map_raw(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int es, uint64_t inner,
                 uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
    if (!aligned16(base)) return fail(DFLASH_ERR_ARG, "matrix %p is not 16-byte aligned", base);
    if ((inner * es) % 16) return fail(DFLASH_ERR_ARG, "row of %llu elements is not a multiple of 16 bytes", (unsigned long long)inner);
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * es};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
#ifndef DFL_L2_PROMOTION
#define DFL_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif
    CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, DFL_L2_PROMOTION,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DFLASH_OK;
}

// 128-byte swizzled boxes of [box_rows][128 bytes] over an f32/bf16/f16 matrix.
int make_map(CUtensorMap* m, const void* base, int xt, uint64_t inner, uint64_t rows,
             uint32_t box_rows) {
    const int es = xt == XT_F32 ? 4 : 2;
    CUtensorMapDataType dt = xt == XT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                           : xt == XT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return make_map_raw(m, base, dt, es, inner, rows, 128 / es, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// ------------------------------------------------------------------ plans

struct GemmPlan {
    GemmMaps maps;
    GemmArgs args;   // pointers that vary per call are patched before launch
    int wfmt, epi, xt, grid;
    double wbytes;   // weight bytes streamed per launch
    double abytes;   // algorithmic bytes per launch (weights + activations + outputs)
};

struct LayerPlans {
    GemmPlan qkv, o, gateup, down, ctxkv;
};

}  // namespace

struct dflash_ctx {
    dflash_config cfg;
    dflash_weights w;
    std::vector<dflash_layer> tgt, drf;
    Layout L;
    uint8_t* ws;
    void* kv_t;
    void* kv_d;
    int sms;
    std::vector<LayerPlans> tplan, dplan;
    GemmPlan lm, fc;
    GemmPlan ctxkv_all;   // every draft layer's context K/V in one GEMM (when grouped)
    bool ctxkv_group = false;
    AttnMaps amap_t{}, amap_d{};   // tensor-core attention maps (fp16 q and caches)
    // fused attention per model (0 target, 1 drafter): chunks per split and
    // splits of a launch (0: two-kernel form)
    int attn_split_chunks[2] = {0, 0};
    int attn_max_splits[2] = {0, 0};
    int attn_tc[2] = {0, 0};   // tcgen05 form of the fused attention
    bool dense_ingest = false;  // window ingest on the dense tcgen05 GEMM
    DenseMaps d_fc{};           // fc over the window's tap rows
    DenseMaps d_fc_hl{};        // the same over hi/lo tap rows (means of hc > 1 streams)
    std::vector<DenseMaps> d_kv;   // per draft layer: context K/V from the context rows
    bool dense_prefill = false;    // prompt rows before the last chunk on the dense GEMM
    struct PrefillLayer { DenseMaps qkv, o, gu, down; };
    std::vector<PrefillLayer> d_pp;
    DenseMaps d_fc_pp{};           // fc over the prefill's hi/lo tap rows
    CUtensorMap pp_qmap{};         // q rows of the prefill attention
    float* verify_logits = nullptr;
    float* draft_logits = nullptr;
    bool prefilled = false;
    // dflash_profile state
    bool prof = false;
    std::vector<cudaEvent_t> ev;
    size_t ev_used = 0;
    long long prof_launches = 0;
    double prof_bytes = 0, prof_wbytes = 0;

    DevState* st() const { return reinterpret_cast<DevState*>(ws + L.state); }
    template <typename T> T* buf(size_t off) const { return reinterpret_cast<T*>(ws + off); }
    // GEMM inputs: fp32, or hi/lo bf16 planes for the bf16 models
    int act_xt() const { return cfg.dtype == DFLASH_F32 ? XT_F32 : XT_BF16S; }
    // The input type of a GEMM whose weights have format f: fp32 for the
    // fp32 models, one f16 plane for INT4 weights (the codes are exact in
    // f16, and one plane halves the MMAs of the instruction-bound INT4
    // GEMM), bf16 hi/lo planes for bf16 weights.
    int gin_xt(int f) const {
        if (cfg.dtype == DFLASH_F32) return XT_F32;
        return f == DFLASH_INT4G64 ? XT_F16 : XT_BF16S;
    }
    int xt_model(bool target) const { return gin_xt(target ? cfg.tgt_wfmt : cfg.drf_wfmt); }
    int xt_lm() const { return gin_xt(cfg.lm_wfmt == DFLASH_INT4G64 ? DFLASH_INT4G64 : cfg.dtype); }
    // attention operands (q, K/V caches): fp32, or fp16 for the bf16 models
    int kv_xt() const { return cfg.dtype == DFLASH_F32 ? XT_F32 : XT_F16; }
    int wf(int f) const { return f == DFLASH_F32 ? WF_F32 : f == DFLASH_INT4G64 ? WF_INT4 : WF_BF16; }
    size_t cache_layer_stride() const {   // elements per layer (K and V)
        return (size_t)2 * cfg.n_kv * cache_cap(cfg) * cfg.head_dim;
    }
    size_t cache_kv_offset() const {      // elements from a layer's K to its V
        return (size_t)cfg.n_kv * cache_cap(cfg) * cfg.head_dim;
    }
};

namespace {

int plan_gemm(dflash_ctx* c, GemmPlan* p, int wfmt, int epi, const void* const* w, const int* rows,
              int nseg, int K, const void* x, int xt, const void* const* scales = nullptr) {
    memset(p, 0, sizeof *p);
    p->wfmt = wfmt;
    p->epi = epi;
    p->xt = xt;
    const int wxt = wfmt == WF_F32 ? XT_F32 : XT_BF16;
    const uint32_t box_rows = epi == EPI_SWIGLU ? 64 : GEMM_BN;
    int N = 0;
    for (int i = 0; i < nseg; ++i) {
        int r;
        if (wfmt == WF_INT4) {
            if (!scales || !aligned16(scales[i])) return fail(DFLASH_ERR_ARG, "INT4 scales missing or misaligned");
            if (K % 256) return fail(DFLASH_ERR_CONFIG, "INT4 reduction length %d is not a multiple of 256", K);
            r = make_map_raw(&p->maps.w[i], w[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows[i], 128,
                             box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
            if (!r)
                r = make_map_raw(&p->maps.s[i], scales[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, rows[i],
                                 K / 64, box_rows, 4, CU_TENSOR_MAP_SWIZZLE_NONE);
        } else {
            r = make_map(&p->maps.w[i], w[i], wxt, K, rows[i], box_rows);
        }
        if (r) return r;
        p->args.seg_rows[i] = rows[i];
        N += rows[i];
    }
    const uint32_t xrows = xt == XT_BF16S ? 2 * DFL_MAX_ROWS : DFL_MAX_ROWS;
    int r = make_map(&p->maps.x, x, xt == XT_BF16S ? XT_BF16 : xt, K, xrows, xrows);
    if (r) return r;
    GemmArgs& a = p->args;
    a.x_split = xt == XT_BF16S ? 1 : 0;
    a.n_seg = nseg;
    a.K = K;
    a.kb = K / (wfmt == WF_F32 ? 32 : wfmt == WF_INT4 ? 256 : 64);
    if (epi == EPI_SWIGLU) {
        a.N = rows[0];
        a.n_tiles = rows[0] / 64;
    } else {
        a.N = N;
        a.n_tiles = N / GEMM_BN;
    }
    if (a.n_tiles > MAX_TILES) return fail(DFLASH_ERR_CONFIG, "GEMM with %d tiles", a.n_tiles);
    a.slots = c->buf<float>(c->L.slots);
    a.counters = c->buf<int>(c->L.counters);
    a.st = c->st();
    const long long units = (long long)a.n_tiles * a.kb;
    const int ctas = c->sms * DFL_GEMM_CTAS_PER_SM;
    p->grid = (int)(units < ctas ? units : ctas);
    const double wes = wfmt == WF_F32 ? 4.0 : wfmt == WF_INT4 ? 0.5 : 2.0;
    const double xes = (xt == XT_F32 || xt == XT_BF16S) ? 4.0 : 2.0;
    p->wbytes = (double)N * K * wes + (wfmt == WF_INT4 ? (double)N * (K / 64) * 2 : 0.0);
    double outb = 0;
    if (epi == EPI_STORE) outb = (double)DFL_MAX_ROWS * N * 4;
    else if (epi == EPI_RESID) outb = (double)DFL_MAX_ROWS * N * (8 + xes);
    else if (epi == EPI_NORMOUT) outb = (double)DFL_MAX_ROWS * N * xes;
    else if (epi == EPI_SWIGLU) outb = (double)DFL_MAX_ROWS * a.N * xes;
    else if (epi == EPI_QKV) outb = (double)DFL_MAX_ROWS * N * xes;
    else outb = DFL_MAX_ROWS * 8.0;
    p->abytes = p->wbytes + (double)DFL_MAX_ROWS * K * xes + outb;
    return DFLASH_OK;
}

// Records a profiling event: as an event node when the stream is being
// captured into a graph, as a plain record otherwise.
cudaError_t record_event(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t r = cudaStreamIsCapturing(s, &cs);
    if (r != cudaSuccess) return r;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
               : cudaEventRecord(e, s);
}

// Where the pieces of a forward are launched.
struct Emit {
    cudaStream_t s = nullptr;
};

int run_gemm(dflash_ctx* c, const GemmPlan& p, const GemmArgs& a, Emit& em) {
    cudaStream_t s = em.s;
    const bool timed = c->prof && c->ev_used + 2 <= c->ev.size();
    if (timed) CUDA_TRY(record_event(c->ev[c->ev_used], s));
    const int e = launch_gemm(p.wfmt, p.epi, p.xt, p.maps, a, p.grid, s);
    if (e)
        return fail(DFLASH_ERR_CUDA, "GEMM launch failed (fmt %d epi %d N %d K %d grid %d): %s",
                    p.wfmt, p.epi, a.N, a.K, p.grid, cudaGetErrorString((cudaError_t)e));
    if (timed) {
        CUDA_TRY(record_event(c->ev[c->ev_used + 1], s));
        c->ev_used += 2;
        c->prof_launches += 1;
        c->prof_bytes += p.abytes;
        c->prof_wbytes += p.wbytes;
    }
    return DFLASH_OK;
}

int build_layer_plans(dflash_ctx* c, const dflash_layer& lw, int wfmt, bool draft, LayerPlans* lp) {
    const dflash_config& g = c->cfg;
    const int H = g.hidden, qd = g.n_q * g.head_dim, kvd = g.n_kv * g.head_dim;
    const int wf = c->wf(wfmt), xt = c->gin_xt(wfmt);
    const void* hn = c->ws + c->L.hn;
    const void* wqkv[3] = {lw.wq, lw.wk, lw.wv};
    const void* sqkv[3] = {lw.sq, lw.sk, lw.sv};
    const int rqkv[3] = {qd, kvd, kvd};
    int r = plan_gemm(c, &lp->qkv, wf, EPI_QKV, wqkv, rqkv, 3, H, hn, xt, sqkv);
    if (r) return r;
    const void* wo[1] = {lw.wo};
    const void* so[1] = {lw.so};
    const int ro[1] = {H};
    if ((r = plan_gemm(c, &lp->o, wf, EPI_RESID, wo, ro, 1, qd, c->ws + c->L.attn, xt, so))) return r;
    const void* wgu[2] = {lw.w_gate, lw.w_up};
    const void* sgu[2] = {lw.s_gate, lw.s_up};
    const int rgu[2] = {g.ffn, g.ffn};
    if ((r = plan_gemm(c, &lp->gateup, wf, EPI_SWIGLU, wgu, rgu, 2, H, hn, xt, sgu))) return r;
    const void* wd[1] = {lw.w_down};
    const void* sd[1] = {lw.s_down};
    if ((r = plan_gemm(c, &lp->down, wf, EPI_RESID, wd, ro, 1, g.ffn, c->ws + c->L.act, xt, sd))) return r;
    if (draft) {
        const void* wkv[2] = {lw.wk, lw.wv};
        const void* skv[2] = {lw.sk, lw.sv};
        const int rkv[2] = {kvd, kvd};
        if ((r = plan_gemm(c, &lp->ctxkv, wf, EPI_QKV, wkv, rkv, 2, H, hn, xt, skv))) return r;
    }
    return DFLASH_OK;
}

// ------------------------------------------------------------------ forward pieces

// Folded-RMSNorm input of a GEMM: the partial sums written by the producer.
void set_norm_in(const dflash_ctx* c, GemmArgs& a, bool on) {
    a.ssq_in = on ? c->buf<float>(c->L.ssq) : nullptr;
    a.ssq_parts = c->cfg.hidden / GEMM_BN;
    a.inv_width = 1.0f / (float)c->cfg.hidden;
    a.eps = c->cfg.rms_eps;
}

// Normalised-input output of a GEMM for the next folded RMSNorm, in the
// input type of the GEMM that consumes it.
void set_norm_out(const dflash_ctx* c, GemmArgs& a, const float* w_next, bool with_ssq, int xt) {
    a.xn_out = c->ws + c->L.hn;
    a.xn_type = xt;
    a.w_next = w_next;
    a.ssq_out = with_ssq ? c->buf<float>(c->L.ssq) : nullptr;
}

QkvEpi qkv_epi(const dflash_ctx* c, const dflash_layer& lw, bool target, int layer, int n_q,
               int row_sel) {
    const dflash_config& g = c->cfg;
    QkvEpi q{};
    q.n_q = n_q;
    q.n_kv = g.n_kv;
    q.hd = g.head_dim;
    q.q_norm = lw.q_norm;
    q.k_norm = lw.k_norm;
    q.rope_cos = c->buf<float>(c->L.rcos);
    q.rope_sin = c->buf<float>(c->L.rsin);
    q.q_out = c->ws + c->L.qrot;
    q.q_type = c->kv_xt();
    uint8_t* cache = reinterpret_cast<uint8_t*>(target ? c->kv_t : c->kv_d) +
                     (size_t)layer * c->cache_layer_stride() * elem_size(g.dtype);
    q.k_cache = cache;
    q.v_cache = cache + c->cache_kv_offset() * elem_size(g.dtype);
    q.c_type = c->kv_xt();
    q.cap = cache_cap(g);
    q.max_seq = g.max_seq;
    q.row_sel = row_sel;
    return q;
}

// One model's decoder layers over the forward's rows.  Per layer: q/k/v
// GEMM (folded input norm, head norms, RoPE, K/V into the cache), attention,
// o GEMM (+ residual, next folded norm), gate/up GEMM (+ SwiGLU), down GEMM
// (+ residual, next folded norm, tap copy).
int run_layers(dflash_ctx* c, bool target, Emit& em) {
    const dflash_config& g = c->cfg;
    const int H = g.hidden;
    const int xt = c->xt_model(target);   // input type of this model's GEMMs
    const int nl = target ? g.tgt_layers : g.drf_layers;
    DevState* st = c->st();
    float* x = c->buf<float>(c->L.x);
    const float* final_norm = target ? c->w.final_norm_tgt : c->w.final_norm_drf;
    for (int l = 0; l < nl; ++l) {
        const dflash_layer& lw = target ? c->tgt[l] : c->drf[l];
        const LayerPlans& lp = target ? c->tplan[l] : c->dplan[l];
        GemmArgs a = lp.qkv.args;
        set_norm_in(c, a, true);
        a.qkv = qkv_epi(c, lw, target, l, g.n_q, ROWS_FWD);
        int r = run_gemm(c, lp.qkv, a, em);
        if (r) return r;
        AttnArgs at{};
        uint8_t* cache = reinterpret_cast<uint8_t*>(target ? c->kv_t : c->kv_d) +
                         (size_t)l * c->cache_layer_stride() * elem_size(g.dtype);
        at.q = c->ws + c->L.qrot;
        at.k_cache = cache;
        at.v_cache = cache + c->cache_kv_offset() * elem_size(g.dtype);
        at.kv_type = c->kv_xt();
        at.n_q = g.n_q;
        at.n_kv = g.n_kv;
        at.head_dim = g.head_dim;
        at.cap = cache_cap(g);
        at.causal = target ? 1 : 0;
        at.window = target ? 0 : g.window;
        at.scale = 1.0f / sqrtf((float)g.head_dim);
        at.part = c->buf<float>(c->L.part);
        at.out = c->ws + c->L.attn;
        at.out_type = xt;
        at.max_chunks = max_chunks(g);
        at.st = st;
        if (g.dtype == DFLASH_BF16) {
            AttnMmaArgs am{};
            am.n_q = g.n_q;
            am.n_kv = g.n_kv;
            am.head_dim = g.head_dim;
            am.layer = l;
            am.cap = cache_cap(g);
            am.causal = at.causal;
            am.window = at.window;
            am.scale = at.scale;
            am.part = at.part;
            am.st = st;
            if (c->attn_split_chunks[target ? 0 : 1] > 0) {
                AttnFusedArgs fa{};
                fa.m = am;
                fa.split_chunks = c->attn_split_chunks[target ? 0 : 1];
                fa.max_splits = c->attn_max_splits[target ? 0 : 1];
                fa.tc = c->attn_tc[target ? 0 : 1];
                fa.out = at.out;
                fa.out_type = at.out_type;
                fa.arrive = c->buf<int>(c->L.acnt);
                fa.done = fa.arrive + g.n_kv;
                const int e = launch_attention_fused(target ? c->amap_t : c->amap_d, fa, em.s);
                if (e) return fail(DFLASH_ERR_CUDA, "attention launch: %s", cudaGetErrorString((cudaError_t)e));
            } else {
                const int e = launch_attention_mma(target ? c->amap_t : c->amap_d, am, at.max_chunks, em.s);
                if (e) return fail(DFLASH_ERR_CUDA, "attention launch: %s", cudaGetErrorString((cudaError_t)e));
                LAUNCH_TRY(launch_attention_combine(at, em.s));
            }
        } else {
            LAUNCH_TRY(launch_attention(at, em.s));
        }
        GemmArgs ao = lp.o.args;
        ao.out = x;
        ao.ldo = H;
        set_norm_out(c, ao, lw.ln_mlp, true, xt);
        GemmArgs agu = lp.gateup.args;
        set_norm_in(c, agu, true);
        agu.act = c->ws + c->L.act;
        agu.ld_act = g.ffn;
        agu.act_type = xt;
        GemmArgs ad = lp.down.args;
        ad.out = x;
        ad.ldo = H;
        const float* w_next = l + 1 < nl ? (target ? c->tgt[l + 1] : c->drf[l + 1]).ln_attn : final_norm;
        set_norm_out(c, ad, w_next, true, l + 1 < nl ? xt : c->xt_lm());
        if (target && g.drf_layers > 0) {
            for (int i = 0; i < g.n_taps; ++i)
                if (g.tap_layer[i] == l) {
                    ad.tap_out = c->ws + c->L.taps + (size_t)i * H * elem_size(g.dtype);   // column i*H
                    ad.ld_tap = g.n_taps * H;
                    ad.tap_type = c->act_xt();   // taps feed fc (bf16 weights)
                }
        }
        if ((r = run_gemm(c, lp.o, ao, em))) return r;
        if ((r = run_gemm(c, lp.gateup, agu, em))) return r;
        if ((r = run_gemm(c, lp.down, ad, em))) return r;
    }
    return DFLASH_OK;
}

// LM head over the final-norm input the last down projection wrote.
int run_lm_head(dflash_ctx* c, float* logits, Emit& em) {
    GemmArgs a = c->lm.args;
    set_norm_in(c, a, true);
    a.amax = c->buf<unsigned long long>(c->L.amax);
    a.logits = logits;
    a.ldl = c->cfg.vocab;
    return run_gemm(c, c->lm, a, em);
}

// fc -> context norm -> per draft layer k/v projection with k-norm and
// RoPE into the draft cache, for the rows the device state marks committed.
int run_ingest(dflash_ctx* c, Emit& em) {
    const dflash_config& g = c->cfg;
    GemmArgs a = c->fc.args;
    a.ldo = g.hidden;
    set_norm_out(c, a, g.ctx_norm ? c->w.ctx_norm : nullptr, g.ctx_norm != 0, c->xt_model(false));
    int r = run_gemm(c, c->fc, a, em);
    if (r) return r;
    if (c->ctxkv_group) {
        a = c->ctxkv_all.args;
        set_norm_in(c, a, g.ctx_norm != 0);
        a.qkv = qkv_epi(c, c->drf[0], false, 0, 0, ROWS_COMMIT);
        a.qkv.group = g.drf_layers;
        a.qkv.cache_stride = (long long)c->cache_layer_stride();
        a.qkv.k_norm_all = c->buf<float>(c->L.ctxkv_kn);
        return run_gemm(c, c->ctxkv_all, a, em);
    }
    for (int l = 0; l < g.drf_layers; ++l) {
        const LayerPlans& lp = c->dplan[l];
        a = lp.ctxkv.args;
        set_norm_in(c, a, g.ctx_norm != 0);
        a.qkv = qkv_epi(c, c->drf[l], false, l, 0, ROWS_COMMIT);
        if ((r = run_gemm(c, lp.ctxkv, a, em))) return r;
    }
    return DFLASH_OK;
}

// A CUDA error left pending by the caller's own earlier calls would be
// reported by our first launch check; surface it under its own name instead.
int pending_error() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(DFLASH_ERR_CUDA, "a CUDA error was pending before this call: %s",
                    cudaGetErrorString(e));
    return DFLASH_OK;
}

RowsArgs rows_args(dflash_ctx* c, int mode) {
    const dflash_config& g = c->cfg;
    RowsArgs a{};
    a.mode = mode;
    a.hidden = g.hidden;
    a.vocab = g.vocab;
    a.mask_id = g.vocab - 1;
    a.embed = g.tgt_layers > 0 || g.drf_layers > 0 ? c->w.embed : nullptr;
    a.embed_f32 = g.dtype == DFLASH_F32;
    a.x = c->buf<float>(c->L.x);
    a.rope_cos = c->buf<float>(c->L.rcos);
    a.rope_sin = c->buf<float>(c->L.rsin);
    a.head_dim = g.head_dim;
    a.rope_theta = g.rope_theta;
    rope_table(c, &a.tab_cos, &a.tab_sin, &a.tab_rows);
    a.amax = c->buf<unsigned long long>(c->L.amax);
    const bool draft = mode == FWD_DRAFT;
    a.w0 = draft ? (g.drf_layers ? c->drf[0].ln_attn : nullptr)
                 : (g.tgt_layers ? c->tgt[0].ln_attn : nullptr);
    if (!a.w0) a.embed = nullptr;   // no model runs (drafter-alone tap staging)
    a.xn = c->ws + c->L.hn;
    a.xn_type = c->xt_model(!draft);   // layer 0 of the model that runs
    a.ssq = c->buf<float>(c->L.ssq);
    a.st = c->st();
    return a;
}


// Arguments of the acceptance kernel common to every forward mode.
AcceptArgs accept_args(dflash_ctx* c, int mode) {
    const dflash_config& g = c->cfg;
    AcceptArgs aa{};
    aa.mode = mode;
    aa.amax = c->buf<unsigned long long>(c->L.amax);
    aa.block_max = g.block_max;
    aa.max_seq = g.max_seq;
    aa.eos_id = g.eos_id;
    aa.st = c->st();
    return aa;
}

}  // namespace

// Host helpers shared with the other C-ABI source files.
namespace dfl {

int report_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int make_linear_maps(GemmMaps* maps, const void* w, const void* x, int n, int k) {
    int r = get_encode();
    if (r) return r;
    memset(maps, 0, sizeof *maps);
    r = make_map(&maps->w[0], w, XT_BF16, k, n, GEMM_BN);
    if (!r) r = make_map(&maps->x, x, XT_BF16, k, DFL_MAX_ROWS, DFL_MAX_ROWS);
    return r;
}

DevState* ctx_state(const dflash_ctx* c) { return c->st(); }

void rope_table(const dflash_ctx* c, const float** cos_tab, const float** sin_tab, int* rows) {
    const int cap = cache_cap(c->cfg), half = c->cfg.head_dim / 2;
    *cos_tab = c->buf<float>(c->L.rtab);
    *sin_tab = *cos_tab + (size_t)cap * half;
    *rows = cap;
}
bool ctx_grouped_ctxkv(const dflash_ctx* c, const void** w, const float** k_norm, int* rows) {
    const dflash_config& g = c->cfg;
    if (!c->ctxkv_group || g.drf_wfmt == DFLASH_INT4G64) return false;
    *w = c->ws + c->L.ctxkv_w;
    *k_norm = c->buf<float>(c->L.ctxkv_kn);
    *rows = g.drf_layers * 2 * g.n_kv * g.head_dim;
    return true;
}
const dflash_layer* ctx_layers(const dflash_ctx* c, bool target) {
    return target ? c->tgt.data() : c->drf.data();
}
const dflash_weights& ctx_weights(const dflash_ctx* c) { return c->w; }
int encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int es, uint64_t inner,
               uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
    int r = get_encode();
    if (r) return r;
    return make_map_raw(m, base, dt, es, inner, rows, box_inner, box_rows, swz);
}

int run_linear_store(const void* w, const void* x, int n, int k, float* y, float* slots,
                     int* counters, DevState* st, void* clear, size_t clear_bytes, int32_t* err,
                     int sms, cudaStream_t s) {
    GemmMaps maps;
    int r = make_linear_maps(&maps, w, x, n, k);
    if (r) return r;
    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.N = n;
    a.K = k;
    a.n_tiles = n / GEMM_BN;
    a.kb = k / 64;
    a.seg_rows[0] = n;
    a.n_seg = 1;
    a.out = y;
    a.ldo = n;
    a.slots = slots;
    a.counters = counters;
    a.st = st;
    // the error words this call reports start at zero (and whatever else the
    // caller asked to clear: the fixed scratch's tickets)
    cudaError_t e = cudaMemsetAsync(clear, 0, clear_bytes, s);
    if (e != cudaSuccess) return report_error(DFLASH_ERR_CUDA, "scratch clear: %s", cudaGetErrorString(e));
    const long long units = (long long)a.n_tiles * a.kb;
    const int ctas = sms * DFL_GEMM_CTAS_PER_SM;
    const int grid = (int)(units < ctas ? units : ctas);
    const int le = launch_gemm(WF_BF16, EPI_STORE, XT_BF16, maps, a, grid, s);
    if (le) return report_error(DFLASH_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString((cudaError_t)le));
    // the kernel's (code, site) words, after it, into the caller's err
    e = cudaMemcpyAsync(err, &st->err, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return report_error(DFLASH_ERR_CUDA, "error-word copy: %s", cudaGetErrorString(e));
    return DFLASH_OK;
}

}  // namespace dfl

// ====================================================================== C ABI

extern "C" {

const char* dflash_last_error(void) { return g_err.c_str(); }

size_t dflash_workspace_bytes(const dflash_config* cfg) {
    if (validate(cfg)) return 0;
    return make_layout(*cfg).total;
}

size_t dflash_kv_target_bytes(const dflash_config* cfg) {
    if (validate(cfg)) return 0;
    return (size_t)cfg->tgt_layers * 2 * cfg->n_kv * cache_cap(*cfg) * cfg->head_dim * elem_size(cfg->dtype);
}

size_t dflash_kv_draft_bytes(const dflash_config* cfg) {
    if (validate(cfg)) return 0;
    return (size_t)cfg->drf_layers * 2 * cfg->n_kv * cache_cap(*cfg) * cfg->head_dim * elem_size(cfg->dtype);
}

int dflash_init(const dflash_config* cfg, const dflash_weights* w, void* kv_target, void* kv_draft,
                void* workspace, size_t workspace_bytes, dflash_ctx** out) {
    int r = validate(cfg);
    if (r) return r;
    if (!w || !out) return fail(DFLASH_ERR_ARG, "weights/out is NULL");
    *out = nullptr;
    const dflash_config& g = *cfg;
    // every weight pointer is checked before any buffer is touched
    if (!aligned16(w->embed)) return fail(DFLASH_ERR_ARG, "embed missing or misaligned");
    if (g.lm_wfmt == DFLASH_INT4G64 && (!aligned16(w->lm_head) || !aligned16(w->lm_scales)))
        return fail(DFLASH_ERR_ARG, "INT4 LM head or its scales missing or misaligned");
    if (g.tgt_layers > 0 && (!w->tgt || !w->final_norm_tgt)) return fail(DFLASH_ERR_ARG, "target weights missing");
    if (g.drf_layers > 0 && (!w->drf || !w->final_norm_drf || !aligned16(w->fc) || !w->ctx_norm))
        return fail(DFLASH_ERR_ARG, "draft weights missing");
    auto check_layer = [&](const dflash_layer& l, const char* who, int i, int fmt) -> int {
        const void* ps[7] = {l.wq, l.wk, l.wv, l.wo, l.w_gate, l.w_up, l.w_down};
        for (const void* p : ps)
            if (!aligned16(p)) return fail(DFLASH_ERR_ARG, "%s layer %d: projection missing or misaligned", who, i);
        const void* ss[7] = {l.sq, l.sk, l.sv, l.so, l.s_gate, l.s_up, l.s_down};
        if (fmt == DFLASH_INT4G64)
            for (const void* p : ss)
                if (!aligned16(p)) return fail(DFLASH_ERR_ARG, "%s layer %d: INT4 scales missing or misaligned", who, i);
        if (!l.ln_attn || !l.ln_mlp || !l.q_norm || !l.k_norm)
            return fail(DFLASH_ERR_ARG, "%s layer %d: norm weight missing", who, i);
        return DFLASH_OK;
    };
    for (int i = 0; i < g.tgt_layers; ++i) if ((r = check_layer(w->tgt[i], "target", i, g.tgt_wfmt))) return r;
    for (int i = 0; i < g.drf_layers; ++i) if ((r = check_layer(w->drf[i], "draft", i, g.drf_wfmt))) return r;
    const Layout L = make_layout(g);
    if (!workspace || workspace_bytes < L.total)
        return fail(DFLASH_ERR_ARG, "workspace %zu bytes < %zu", workspace_bytes, L.total);
    if (!aligned16(workspace)) return fail(DFLASH_ERR_ARG, "workspace misaligned");
    if (g.tgt_layers > 0 && !aligned16(kv_target)) return fail(DFLASH_ERR_ARG, "target KV cache missing");
    if (g.drf_layers > 0 && !aligned16(kv_draft)) return fail(DFLASH_ERR_ARG, "draft KV cache missing");
    if ((r = get_encode())) return r;
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    int sms = 0;
    CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (sms > 256) sms = 256;

    dflash_ctx* c = new dflash_ctx();
    c->cfg = g;
    c->w = *w;
    c->tgt.assign(w->tgt, w->tgt + g.tgt_layers);
    c->drf.assign(w->drf, w->drf + g.drf_layers);
    c->w.tgt = c->tgt.data();
    c->w.drf = c->drf.data();
    c->L = L;
    c->ws = static_cast<uint8_t*>(workspace);
    c->kv_t = kv_target;
    c->kv_d = kv_draft;
    c->sms = sms;
    c->tplan.resize(g.tgt_layers);
    c->dplan.resize(g.drf_layers);
    for (int i = 0; i < g.tgt_layers && !r; ++i) r = build_layer_plans(c, c->tgt[i], g.tgt_wfmt, false, &c->tplan[i]);
    for (int i = 0; i < g.drf_layers && !r; ++i) r = build_layer_plans(c, c->drf[i], g.drf_wfmt, true, &c->dplan[i]);
    if (!r) {
        const int re[1] = {g.vocab};
        if (g.lm_wfmt == DFLASH_INT4G64) {
            const void* wl[1] = {w->lm_head};
            const void* sl[1] = {w->lm_scales};
            r = plan_gemm(c, &c->lm, WF_INT4, EPI_ARGMAX, wl, re, 1, g.hidden, c->ws + L.hn,
                          c->xt_lm(), sl);
        } else {
            const void* we[1] = {w->embed};
            r = plan_gemm(c, &c->lm, c->wf(g.dtype), EPI_ARGMAX, we, re, 1, g.hidden, c->ws + L.hn,
                          c->xt_lm());
        }
    }
    if (!r && g.drf_layers > 0) {
        const void* wfc[1] = {w->fc};
        const int rfc[1] = {g.hidden};
        r = plan_gemm(c, &c->fc, c->wf(g.dtype), EPI_NORMOUT, wfc, rfc, 1, g.n_taps * g.hidden,
                      c->ws + L.taps, c->act_xt());
    }
    const char* cg_env = getenv("DFLASH_CTXKV_GROUP");   // "0": one context K/V GEMM per draft layer
    if (!r && ctxkv_grouped(g) && !(cg_env && cg_env[0] == '0')) {
        // the draft layers' [W_k; W_v] and k-norm weights copied one after
        // another: the tap commit streams them in one launch (the drafter's
        // own q/k/v GEMMs keep reading the caller's weights)
        // (the copy itself is made after the workspace is cleared, below)
        const bool q4 = g.drf_wfmt == DFLASH_INT4G64;
        const size_t rows = (size_t)g.drf_layers * 2 * g.n_kv * g.head_dim;
        const size_t rb = q4 ? g.hidden / 2 : (size_t)g.hidden * 2;   // bytes of one weight row
        const void* wkv[1] = {c->ws + L.ctxkv_w};
        const void* skv[1] = {c->ws + L.ctxkv_w + rows * rb};   // INT4: scales [hidden / 64][rows]
        const int rkv[1] = {(int)rows};
        r = plan_gemm(c, &c->ctxkv_all, c->wf(g.drf_wfmt), EPI_QKV, wkv, rkv, 1, g.hidden, c->ws + L.hn,
                      c->xt_model(false), q4 ? skv : nullptr);
        c->ctxkv_group = !r;
    }
    if (!r && g.dtype == DFLASH_BF16) {
        const int cap = cache_cap(g);
        const int qrows = (g.n_q / g.n_kv) * DFL_MAX_ROWS;
        r = make_map_raw(&c->amap_t.q, c->ws + L.qrot, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                         (uint64_t)g.n_q * DFL_MAX_ROWS, 64, qrows, CU_TENSOR_MAP_SWIZZLE_128B);
        if (!r)
            r = make_map_raw(&c->amap_t.q16, c->ws + L.qrot, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                             (uint64_t)g.n_q * DFL_MAX_ROWS, 64, DFL_MAX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
        c->amap_d.q = c->amap_t.q;
        c->amap_d.q16 = c->amap_t.q16;
        if (!r && g.tgt_layers > 0)
            r = make_map_raw(&c->amap_t.kv, kv_target, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                             (uint64_t)g.tgt_layers * 2 * g.n_kv * cap, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        if (!r && g.drf_layers > 0)
            r = make_map_raw(&c->amap_d.kv, kv_draft, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                             (uint64_t)g.drf_layers * 2 * g.n_kv * cap, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!r && g.dtype == DFLASH_BF16) {
        // fused attention: the splits of a kv head wait for one another, so
        // every CTA of a launch must be resident at once
        int per_sm = 0;
        const int e = attention_fused_per_sm(g.head_dim, g.n_q, g.n_kv, &per_sm);
        if (e) r = fail(DFLASH_ERR_CUDA, "attention occupancy: %s", cudaGetErrorString((cudaError_t)e));
        const int capacity = per_sm * sms;
        // chunks a forward can touch: the whole cache for the causal target,
        // the window (+ block, + a partial chunk) for the drafter
        auto model_chunks = [&](int mdl) {
            int mc = max_chunks(g);
            if (mdl == 1 && g.window > 0) {
                const int wc = (g.window + g.block_max + 63) / 64 + 1;
                if (wc < mc) mc = wc;
            }
            return mc;
        };
        for (int mdl = 0; mdl < 2 && !r && capacity > 0; ++mdl) {
            const int mc = model_chunks(mdl);
            int q = (mc * g.n_kv + capacity - 1) / capacity;
            if (q < (mc + 63) / 64) q = (mc + 63) / 64;
            if (q < DFL_ATTN_MIN_SPLIT) q = DFL_ATTN_MIN_SPLIT;
            const int smax = (mc + q - 1) / q;
            if (g.n_kv * smax <= capacity && smax <= 64) {
                c->attn_split_chunks[mdl] = q;
                c->attn_max_splits[mdl] = smax;
            }
        }
        // tcgen05 form (opt-in, DFLASH_ATTN_TC=1: measured slower than the
        // mma.sync form on the 16-row round) with splits of 1 or 2 chunks,
        // where every CTA of a launch is resident at once and the tensor
        // memory of the CTAs one SM holds fits its 512 columns
        const char* tc_env = getenv("DFLASH_ATTN_TC");
        for (int mdl = 0; mdl < 2 && !r && tc_env && tc_env[0] == '1'; ++mdl) {
            if (c->attn_split_chunks[mdl] <= 0) continue;
            const int mc = model_chunks(mdl);
            for (int nc = 1; nc <= 2 && !r; ++nc) {
                int tc_per_sm = 0, tc_cols = 0;
                const int e2 = attention_tc_per_sm(g.head_dim, nc, &tc_per_sm, &tc_cols);
                if (e2) {
                    r = fail(DFLASH_ERR_CUDA, "attention occupancy: %s", cudaGetErrorString((cudaError_t)e2));
                    break;
                }
                const int smax = (mc + nc - 1) / nc;
                if (tc_per_sm > 0 && g.n_kv * smax <= tc_per_sm * sms && smax <= 64 &&
                    tc_per_sm * tc_cols <= 512) {
                    c->attn_split_chunks[mdl] = nc;
                    c->attn_max_splits[mdl] = smax;
                    c->attn_tc[mdl] = 1;
                    break;
                }
            }
        }
    }
    // window ingest on the dense tcgen05 GEMM (DFLASH_DENSE_INGEST=0 keeps
    // the 16-row chunks through the round's kernels)
    // the tail box map of a one-segment dense weight: 160-column tiles
    auto tail_map = [&](DenseMaps& m, const void* wt, CUtensorMapDataType dt, uint64_t k, uint64_t n) {
        const int e = make_map_raw(&m.w_tail, wt, dt, 2, k, n, DT_BK, DT_WTAIL, CU_TENSOR_MAP_SWIZZLE_128B);
        m.has_tail = e ? 0 : 1;
        return e;
    };
    const char* di_env = getenv("DFLASH_DENSE_INGEST");
    if (!r && dense_ingest_ok(g) && !(di_env && di_env[0] == '0')) {
        const uint64_t K1 = (uint64_t)g.n_taps * g.hidden, kvr = (uint64_t)g.n_kv * g.head_dim;
        const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
        r = make_map_raw(&c->d_fc.x, c->ws + L.pf_x, bf, 2, K1, PF_ROWS, DT_BK, DT_BM, sw);
        if (!r) r = make_map_raw(&c->d_fc.w[0], w->fc, bf, 2, K1, g.hidden, DT_BK, DT_WBOX, sw);
        if (!r) r = tail_map(c->d_fc, w->fc, bf, K1, g.hidden);
        if (!r) {
            c->d_fc_hl = c->d_fc;
            r = make_map_raw(&c->d_fc_hl.x_lo, c->ws + L.pf_xlo, bf, 2, K1, PF_ROWS, DT_BK, DT_BM, sw);
        }
        c->d_kv.resize(g.drf_layers);
        const bool q4 = g.drf_wfmt == DFLASH_INT4G64;   // f16 operands: rows and dequantised weights
        const CUtensorMapDataType xt = q4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : bf;
        for (int l = 0; l < g.drf_layers && !r; ++l) {
            DenseMaps& m = c->d_kv[l];
            r = make_map_raw(&m.x, c->ws + L.pf_chi, xt, 2, g.hidden, PF_ROWS, DT_BK, DT_BM, sw);
            if (!r) r = make_map_raw(&m.x_lo, c->ws + L.pf_clo, xt, 2, g.hidden, PF_ROWS, DT_BK, DT_BM, sw);
            if (!r && q4)
                r = make_map_raw(&m.w[0], c->ws + L.pf_w, xt, 2, g.hidden, 2 * kvr, DT_BK, DT_WBOX, sw);
            if (!r && !q4) r = make_map_raw(&m.w[0], c->drf[l].wk, bf, 2, g.hidden, kvr, DT_BK, DT_WBOX, sw);
            if (!r && !q4) r = make_map_raw(&m.w[1], c->drf[l].wv, bf, 2, g.hidden, kvr, DT_BK, DT_WBOX, sw);
        }
        c->dense_ingest = !r;
    }
    // dense prompt prefill (DFLASH_DENSE_PREFILL=0 keeps 16-row forwards)
    const char* dp_env = getenv("DFLASH_DENSE_PREFILL");
    if (!r && dense_prefill_ok(g) && (g.drf_layers == 0 || c->dense_ingest) && !(dp_env && dp_env[0] == '0')) {
        const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
        const uint64_t qd = (uint64_t)g.n_q * g.head_dim, kvd = (uint64_t)g.n_kv * g.head_dim;
        const bool q4 = g.tgt_wfmt == DFLASH_INT4G64;   // f16 rows times exactly dequantised f16 weights
        const CUtensorMapDataType xt = q4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : bf;
        auto xmaps = [&](DenseMaps& m, uint64_t width, bool act = false) {
            uint8_t* xh = c->ws + (act ? L.pp_ahi : L.pp_hi);
            uint8_t* xl = c->ws + (act ? L.pp_alo : L.pp_lo);
            int e = make_map_raw(&m.x, xh, xt, 2, width, PF_ROWS, DT_BK, DT_BM, sw);
            if (!e) e = make_map_raw(&m.x_lo, xl, xt, 2, width, PF_ROWS, DT_BK, DT_BM, sw);
            return e;
        };
        c->d_pp.resize(g.tgt_layers);
        for (int l = 0; l < g.tgt_layers && !r && q4; ++l) {   // every layer's GEMMs read the scratch
            dflash_ctx::PrefillLayer& P = c->d_pp[l];
            uint8_t* pw = c->ws + L.pp_w;
            r = xmaps(P.qkv, g.hidden);
            if (!r) r = make_map_raw(&P.qkv.w[0], pw, xt, 2, g.hidden, qd + 2 * kvd, DT_BK, DT_WBOX, sw);
            if (!r) r = xmaps(P.o, qd);
            if (!r) r = make_map_raw(&P.o.w[0], pw, xt, 2, qd, g.hidden, DT_BK, DT_WBOX, sw);
            if (!r) r = tail_map(P.o, pw, xt, qd, g.hidden);
            if (!r) r = xmaps(P.gu, g.hidden);
            if (!r) r = make_map_raw(&P.gu.w[0], pw, xt, 2, g.hidden, 2 * (uint64_t)g.ffn, DT_BK, DT_WBOX, sw);
            if (!r) r = xmaps(P.down, g.ffn, true);
            if (!r) r = make_map_raw(&P.down.w[0], pw, xt, 2, g.ffn, g.hidden, DT_BK, DT_WBOX, sw);
            if (!r) r = tail_map(P.down, pw, xt, g.ffn, g.hidden);
        }
        for (int l = 0; l < g.tgt_layers && !r && !q4; ++l) {
            const dflash_layer& lw = c->tgt[l];
            dflash_ctx::PrefillLayer& P = c->d_pp[l];
            r = xmaps(P.qkv, g.hidden);
            if (!r) r = make_map_raw(&P.qkv.w[0], lw.wq, bf, 2, g.hidden, qd, DT_BK, DT_WBOX, sw);
            if (!r) r = make_map_raw(&P.qkv.w[1], lw.wk, bf, 2, g.hidden, kvd, DT_BK, DT_WBOX, sw);
            if (!r) r = make_map_raw(&P.qkv.w[2], lw.wv, bf, 2, g.hidden, kvd, DT_BK, DT_WBOX, sw);
            if (!r) r = xmaps(P.o, qd);
            if (!r) r = make_map_raw(&P.o.w[0], lw.wo, bf, 2, qd, g.hidden, DT_BK, DT_WBOX, sw);
            if (!r) r = tail_map(P.o, lw.wo, bf, qd, g.hidden);
            if (!r) r = xmaps(P.gu, g.hidden);
            if (!r) r = make_map_raw(&P.gu.w[0], lw.w_gate, bf, 2, g.hidden, g.ffn, DT_BK, DT_WBOX, sw);
            if (!r) r = make_map_raw(&P.gu.w[1], lw.w_up, bf, 2, g.hidden, g.ffn, DT_BK, DT_WBOX, sw);
            if (!r) r = xmaps(P.down, g.ffn, true);
            if (!r) r = make_map_raw(&P.down.w[0], lw.w_down, bf, 2, g.ffn, g.hidden, DT_BK, DT_WBOX, sw);
            if (!r) r = tail_map(P.down, lw.w_down, bf, g.ffn, g.hidden);
        }
        if (!r)
            r = make_map_raw(&c->pp_qmap, c->ws + L.pp_q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                             (uint64_t)PF_ROWS * g.n_q, 64, (g.n_q / g.n_kv) * DFL_MAX_ROWS, sw);
        if (!r && g.drf_layers > 0) {
            const uint64_t K1 = (uint64_t)g.n_taps * g.hidden;
            r = make_map_raw(&c->d_fc_pp.x, c->ws + L.pp_thi, bf, 2, K1, PF_ROWS, DT_BK, DT_BM, sw);
            if (!r) r = make_map_raw(&c->d_fc_pp.x_lo, c->ws + L.pp_tlo, bf, 2, K1, PF_ROWS, DT_BK, DT_BM, sw);
            if (!r) r = make_map_raw(&c->d_fc_pp.w[0], w->fc, bf, 2, K1, g.hidden, DT_BK, DT_WBOX, sw);
            if (!r) r = tail_map(c->d_fc_pp, w->fc, bf, K1, g.hidden);
        }
        c->dense_prefill = !r;
    }
    if (r) {
        delete c;
        return r;
    }
    cudaError_t e = cudaMemset(workspace, 0, L.total);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        delete c;
        return fail(DFLASH_ERR_CUDA, "workspace clear: %s", cudaGetErrorString(e));
    }
    if (c->ctxkv_group) {
        // the draft layers' [W_k; W_v] (INT4: codes by rows, scales by
        // columns) and k-norm weights, one layer after another: the tap
        // commit streams them in one launch (the drafter's own q/k/v GEMMs
        // keep reading the caller's weights)
        const bool q4 = g.drf_wfmt == DFLASH_INT4G64;
        const size_t kvd = (size_t)g.n_kv * g.head_dim, rows = (size_t)g.drf_layers * 2 * kvd;
        const size_t rb = q4 ? g.hidden / 2 : (size_t)g.hidden * 2;   // bytes of one weight row
        uint8_t* dst = c->ws + L.ctxkv_w;
        uint8_t* sdst = dst + rows * rb;
        for (int l = 0; l < g.drf_layers && e == cudaSuccess; ++l) {
            const void* src[2] = {c->drf[l].wk, c->drf[l].wv};
            const void* ssrc[2] = {c->drf[l].sk, c->drf[l].sv};
            for (int j = 0; j < 2 && e == cudaSuccess; ++j) {
                const size_t row0 = (2 * l + j) * kvd;
                e = cudaMemcpy(dst + row0 * rb, src[j], kvd * rb, cudaMemcpyDeviceToDevice);
                if (q4 && e == cudaSuccess)   // columns row0.. of every scale row
                    e = cudaMemcpy2D(sdst + row0 * 2, rows * 2, ssrc[j], kvd * 2, kvd * 2, g.hidden / 64,
                                     cudaMemcpyDeviceToDevice);
            }
            if (e == cudaSuccess)
                e = cudaMemcpy(c->ws + L.ctxkv_kn + (size_t)l * g.head_dim * 4, c->drf[l].k_norm,
                               (size_t)g.head_dim * 4, cudaMemcpyDeviceToDevice);
        }
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            delete c;
            return fail(DFLASH_ERR_CUDA, "context K/V weights: %s", cudaGetErrorString(e));
        }
    }
    if (g.adaptive_block) {
        const int one = 1;
        e = cudaMemcpy(&c->st()->adaptive, &one, sizeof one, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            delete c;
            return fail(DFLASH_ERR_CUDA, "state init: %s", cudaGetErrorString(e));
        }
    }
    {
        // RoPE frequencies theta^(-2i/d), in double
        std::vector<double> invf(g.head_dim / 2);
        for (int i = 0; i < g.head_dim / 2; ++i)
            invf[i] = pow((double)g.rope_theta, -2.0 * (double)i / (double)g.head_dim);
        e = cudaMemcpy(c->ws + L.invf, invf.data(), invf.size() * 8, cudaMemcpyHostToDevice);
        // the angles of every position, once: the forwards copy their rows
        // from this table instead of evaluating cos / sin in double (slow
        // on this part) every time
        const int half = g.head_dim / 2, cap = cache_cap(g);
        float* tab = c->buf<float>(L.rtab);
        if (e == cudaSuccess)
            e = (cudaError_t)launch_rope_rows(0, cap, half, c->buf<double>(L.invf), tab,
                                              tab + (size_t)cap * half, nullptr);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            delete c;
            return fail(DFLASH_ERR_CUDA, "RoPE table: %s", cudaGetErrorString(e));
        }
    }
    *out = c;
    return DFLASH_OK;
}

void dflash_destroy(dflash_ctx* ctx) {
    if (!ctx) return;
    for (cudaEvent_t e : ctx->ev) cudaEventDestroy(e);
    delete ctx;
}

int64_t dflash_launch_count(void) { return g_launches; }

int dflash_profile(dflash_ctx* c, int32_t mode, dflash_profile_t* out) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    if (mode == 1) {
        if (c->ev.empty()) {
            c->ev.resize(1 << 16);
            for (auto& e : c->ev) CUDA_TRY(cudaEventCreate(&e));
        }
        c->ev_used = 0;
        c->prof_launches = 0;
        c->prof_bytes = c->prof_wbytes = 0;
        c->prof = true;
        return DFLASH_OK;
    }
    if (mode == 0) c->prof = false;
    double ms = 0;
    for (size_t i = 0; i + 1 < c->ev_used; i += 2) {
        CUDA_TRY(cudaEventSynchronize(c->ev[i + 1]));
        float t = 0;
        CUDA_TRY(cudaEventElapsedTime(&t, c->ev[i], c->ev[i + 1]));
        ms += t;
    }
    const long long launches = c->prof_launches;
    const double bytes = c->prof_bytes, wbytes = c->prof_wbytes;
    if (out) {
        out->gemm_launches = launches;
        out->gemm_ms = ms;
        out->gemm_bytes = bytes;
        out->gemm_weight_bytes = wbytes;
    }
    return DFLASH_OK;
}

int dflash_set_logits_out(dflash_ctx* ctx, float* verify_logits, float* draft_logits) {
    if (!ctx) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    ctx->verify_logits = verify_logits;
    ctx->draft_logits = draft_logits;
    return DFLASH_OK;
}

namespace {

// The drafter's context-window ingest as dense work, PF_ROWS rows per pass
// (positions p0..p0+R-1 of the external tap rows): tap rows (bf16) -> fc on
// the dense GEMM -> context RMSNorm into hi/lo rows -> per draft layer
// [W_k; W_v] on the dense GEMM (hi + lo) -> k-norm, RoPE and the cache rows.
// bf16 drafters use bf16 rows and weights; INT4 drafters f16 rows and the
// layer's W_k, W_v dequantised exactly to f16 first (the tensor core takes
// one type for both operands).
// fc over R context rows already in place (x rows m_off .. m_off + R - 1 of
// fc's maps), then the context norm, K/V and cache rows at pos0 ...
// RoPE angles of rows pos0 .. pos0 + R - 1 of a dense pass: the rows of the
// position table, or (rows past it) the pass's own buffer filled now.
int pass_rope(dflash_ctx* c, int pos0, int R, const float** rcos, const float** rsin, cudaStream_t s) {
    const float *tc, *ts;
    int rows;
    rope_table(c, &tc, &ts, &rows);
    const int half = c->cfg.head_dim / 2;
    if (pos0 >= 0 && pos0 + R <= rows) {
        *rcos = tc + (size_t)pos0 * half;
        *rsin = ts + (size_t)pos0 * half;
        return DFLASH_OK;
    }
    float* bc = c->buf<float>(c->L.pf_rope);
    float* bs = bc + (size_t)PF_ROWS * half;
    LAUNCH_TRY(launch_rope_rows(pos0, R, half, c->buf<double>(c->L.invf), bc, bs, s));
    *rcos = bc;
    *rsin = bs;
    return DFLASH_OK;
}

int ingest_rows(dflash_ctx* c, const DenseMaps& fcm, int x_split, int m_off, int R, int pos0, cudaStream_t s) {
    const dflash_config& g = c->cfg;
    const int kvr = g.n_kv * g.head_dim;
    int* err = &c->st()->err;
    DenseArgs fa{};
    fa.M = R;
    fa.N = g.hidden;
    fa.K = g.n_taps * g.hidden;
    fa.n_seg0 = (g.hidden + DT_BN - 1) / DT_BN * DT_BN;
    fa.n_seg1 = 1 << 30;
    fa.m_off = m_off;
    fa.x_split = x_split;
    fa.y = c->buf<float>(c->L.pf_y);
    fa.ldy = g.hidden;
    fa.err = err;
    fa.w_ready = 1;   // the model's fc weights
    LAUNCH_TRY(launch_dense(fcm, fa, s));
    CtxRowsArgs ra{};
    ra.y = fa.y;
    ra.rows = R;
    ra.hidden = g.hidden;
    ra.w = g.ctx_norm ? c->w.ctx_norm : nullptr;
    ra.norm = g.ctx_norm ? 1 : 0;
    ra.eps = g.rms_eps;
    ra.c_hi = c->ws + c->L.pf_chi;
    ra.c_lo = c->ws + c->L.pf_clo;
    const bool q4 = g.drf_wfmt == DFLASH_INT4G64;
    ra.f16 = q4 ? 1 : 0;
    LAUNCH_TRY(launch_ctx_rows(ra, s));
    const float *rcos, *rsin;
    if (int e = pass_rope(c, pos0, R, &rcos, &rsin, s)) return e;
    for (int l = 0; l < g.drf_layers; ++l) {
        if (q4) {   // this layer's W_k and W_v, dequantised (exactly) to f16
            uint8_t* wq = c->ws + c->L.pf_w;
            LAUNCH_TRY(launch_dequant_int4g64_f16(static_cast<const uint8_t*>(c->drf[l].wk),
                                                  static_cast<const uint16_t*>(c->drf[l].sk), kvr, g.hidden,
                                                  wq, s));
            LAUNCH_TRY(launch_dequant_int4g64_f16(static_cast<const uint8_t*>(c->drf[l].wv),
                                                  static_cast<const uint16_t*>(c->drf[l].sv), kvr, g.hidden,
                                                  wq + (size_t)kvr * g.hidden * 2, s));
        }
        DenseArgs ka{};
        ka.M = R;
        ka.N = 2 * kvr;
        ka.K = g.hidden;
        ka.n_seg0 = q4 ? (2 * kvr + DT_BN - 1) / DT_BN * DT_BN : kvr;
        ka.n_seg1 = 1 << 30;
        ka.f16 = q4 ? 1 : 0;
        ka.x_split = 1;
        ka.y = c->buf<float>(c->L.pf_y);
        ka.ldy = 2 * kvr;
        ka.err = err;
        ka.w_ready = q4 ? 0 : 1;   // INT4: dequantised into the scratch just before
        LAUNCH_TRY(launch_dense(c->d_kv[l], ka, s));
        const QkvEpi q = qkv_epi(c, c->drf[l], false, l, 0, ROWS_COMMIT);
        CtxKvArgs ca{};
        ca.y = ka.y;
        ca.rows = R;
        ca.pos0 = pos0;
        ca.n_kv = g.n_kv;
        ca.head_dim = g.head_dim;
        ca.cap = q.cap;
        ca.max_seq = g.max_seq;
        ca.k_norm = c->drf[l].k_norm;
        ca.eps = g.rms_eps;
        ca.rope_cos = rcos;
        ca.rope_sin = rsin;
        ca.k_cache = q.k_cache;
        ca.v_cache = q.v_cache;
        ca.c_type = q.c_type;
        ca.st = c->st();
        LAUNCH_TRY(launch_ctx_kv_store(ca, s));
    }
    return DFLASH_OK;
}

int run_dense_ingest(dflash_ctx* c, const void* ext_taps, int n_ext, int hc, int commit_lo, cudaStream_t s) {
    const dflash_config& g = c->cfg;
    for (int p0 = commit_lo; p0 < n_ext; p0 += PF_ROWS) {
        const int R = n_ext - p0 < PF_ROWS ? n_ext - p0 : PF_ROWS;
        TapArgs ta{};
        for (int i = 0; i < g.n_taps; ++i)
            ta.src[i] = static_cast<const uint8_t*>(ext_taps) + ((size_t)i * n_ext + p0) * hc * g.hidden * 2;
        ta.n_layers = g.n_taps;
        ta.rows = R;
        ta.hc = hc;
        ta.hidden = g.hidden;
        ta.in_type = XT_BF16;
        ta.out = c->ws + c->L.pf_x;
        ta.out_row_stride = (long long)g.n_taps * g.hidden;
        if (hc == 1) {
            ta.out_type = XT_BF16;   // the tap rows themselves: exact in bf16
        } else {
            // the hc-stream mean carries more bits than bf16: hi/lo planes,
            // as the round's own GEMM inputs
            ta.out_type = XT_BF16S;
            ta.lo_offset = (long long)((c->L.pf_xlo - c->L.pf_x) / 2);
        }
        LAUNCH_TRY(launch_tap_reduce(ta, s));
        if (int r = ingest_rows(c, hc == 1 ? c->d_fc : c->d_fc_hl, hc == 1 ? 0 : 1, 0, R, p0, s)) return r;
    }
    return DFLASH_OK;
}

// Dense forward of prompt rows [0, P) of the target (P a multiple of 16,
// the rows before the prompt's last chunk), PF_ROWS rows per pass: per
// layer RMSNorm -> [W_q; W_k; W_v] -> q/k norms, RoPE, cache rows -> causal
// attention -> W_o -> residual + RMSNorm -> [W_gate; W_up] -> SwiGLU ->
// W_down -> residual; the tap layers' outputs of the committed rows then go
// through the dense window ingest.  The prompt's last chunk runs the round's
// 16-row forward, which also takes the LM head and sets the state.
int run_dense_prefill(dflash_ctx* c, const int32_t* tokens, int P, int commit_lo, cudaStream_t s) {
    const dflash_config& g = c->cfg;
    const int qd = g.n_q * g.head_dim, kvd = g.n_kv * g.head_dim;
    int* err = &c->st()->err;
    float* x = c->buf<float>(c->L.pp_x);
    float* y = c->buf<float>(c->L.pp_y);
    void* hi = c->ws + c->L.pp_hi;
    void* lo = c->ws + c->L.pp_lo;
    const long long tap_ld = (long long)g.n_taps * g.hidden;
    const bool q4 = g.tgt_wfmt == DFLASH_INT4G64;
    uint8_t* pw = c->ws + c->L.pp_w;
    auto deq = [&](const void* packed, const void* scales, int n, int k, size_t row_off) {
        return launch_dequant_int4g64_f16(static_cast<const uint8_t*>(packed),
                                          static_cast<const uint16_t*>(scales), n, k,
                                          pw + row_off * k * 2, s);
    };
    auto dense = [&](const DenseMaps& m, int R, int N, int K, int seg0, int seg1) {
        DenseArgs d{};
        d.M = R;
        d.N = N;
        d.K = K;
        d.n_seg0 = q4 ? 1 << 30 : seg0;   // INT4: one dequantised matrix
        d.n_seg1 = q4 ? 1 << 30 : seg1;
        d.f16 = q4 ? 1 : 0;
        d.x_split = 1;
        d.y = y;
        d.ldy = N;
        d.err = err;
        d.w_ready = q4 ? 0 : 1;   // INT4: the previous kernel dequantised them into the scratch
        return launch_dense(m, d, s);
    };
    // [W_gate; W_up] with the SwiGLU epilogue at 256-column tiles (128 gate
    // rows + the matching 128 up rows, the maps' 128-row boxes), silu(gate)
    // * up straight into W_down's input planes
    auto dense_swiglu = [&](const DenseMaps& m, int R) {
        DenseArgs d{};
        d.M = R;
        d.N = 2 * g.ffn;
        d.K = g.hidden;
        d.n_seg0 = 1 << 30;
        d.n_seg1 = 1 << 30;
        d.f16 = q4 ? 1 : 0;
        d.x_split = 1;
        d.err = err;
        d.bn = 256;
        d.swiglu = 1;
        d.up_map = q4 ? 0 : 1;          // INT4: gate then up rows in one dequantised scratch
        d.up_row = q4 ? g.ffn : 0;
        d.act_hi = c->ws + c->L.pp_ahi;
        d.act_lo = c->ws + c->L.pp_alo;
        d.act_ld = g.ffn;
        d.w_ready = q4 ? 0 : 1;
        return launch_dense(m, d, s);
    };
    for (int p0 = 0; p0 < P; p0 += PF_ROWS) {
        const int R = P - p0 < PF_ROWS ? P - p0 : PF_ROWS;
        LAUNCH_TRY(launch_embed_rows(tokens + p0, R, c->w.embed, g.hidden, g.vocab, x, c->st(), s));
        const float *rcos, *rsin;
        if (int e = pass_rope(c, p0, R, &rcos, &rsin, s)) return e;
        for (int l = 0; l <= g.tgt_layers; ++l) {
            // residual of layer l - 1's down projection, then layer l's input norm
            // (after the last layer: the final norm, whose rows nothing reads)
            ResidNormArgs rn{};
            rn.x = x;
            rn.y = l > 0 ? y : nullptr;
            rn.rows = R;
            rn.hidden = g.hidden;
            rn.w = l < g.tgt_layers ? c->tgt[l].ln_attn : c->w.final_norm_tgt;
            rn.eps = g.rms_eps;
            rn.hi = hi;
            rn.lo = lo;
            rn.f16 = q4 ? 1 : 0;
            for (int i = 0; i < g.n_taps && l > 0 && g.drf_layers > 0; ++i)
                if (g.tap_layer[i] == l - 1) {
                    rn.tap_hi = c->ws + c->L.pp_thi;
                    rn.tap_lo = c->ws + c->L.pp_tlo;
                    rn.tap_ld = tap_ld;
                    rn.tap_col = i * g.hidden;
                }
            LAUNCH_TRY(launch_resid_norm(rn, s));
            if (l == g.tgt_layers) break;
            const dflash_ctx::PrefillLayer& PL = c->d_pp[l];
            const dflash_layer& lw = c->tgt[l];
            if (q4) {
                LAUNCH_TRY(deq(lw.wq, lw.sq, qd, g.hidden, 0));
                LAUNCH_TRY(deq(lw.wk, lw.sk, kvd, g.hidden, qd));
                LAUNCH_TRY(deq(lw.wv, lw.sv, kvd, g.hidden, qd + kvd));
            }
            LAUNCH_TRY(dense(PL.qkv, R, qd + 2 * kvd, g.hidden, qd, qd + kvd));
            const QkvEpi q = qkv_epi(c, c->tgt[l], true, l, g.n_q, ROWS_FWD);
            QkvRowsArgs qa{};
            qa.y = y;
            qa.rows = R;
            qa.pos0 = p0;
            qa.n_q = g.n_q;
            qa.n_kv = g.n_kv;
            qa.head_dim = g.head_dim;
            qa.cap = q.cap;
            qa.max_seq = g.max_seq;
            qa.q_norm = c->tgt[l].q_norm;
            qa.k_norm = c->tgt[l].k_norm;
            qa.eps = g.rms_eps;
            qa.rope_cos = rcos;
            qa.rope_sin = rsin;
            qa.q_out = c->ws + c->L.pp_q;
            qa.k_cache = q.k_cache;
            qa.v_cache = q.v_cache;
            qa.c_type = q.c_type;
            qa.st = c->st();
            LAUNCH_TRY(launch_qkv_rows(qa, s));
            PrefillAttnArgs pa{};
            pa.m.n_q = g.n_q;
            pa.m.n_kv = g.n_kv;
            pa.m.head_dim = g.head_dim;
            pa.m.layer = l;
            pa.m.cap = cache_cap(g);
            pa.m.causal = 1;
            pa.m.window = 0;
            pa.m.scale = 1.0f / sqrtf((float)g.head_dim);
            pa.m.st = c->st();
            pa.rows = R;
            pa.pos0 = p0;
            pa.out_hi = hi;
            pa.out_lo = lo;
            pa.f16 = q4 ? 1 : 0;
            LAUNCH_TRY(launch_prefill_attention(c->pp_qmap, c->amap_t.kv, pa, s));
            if (q4) LAUNCH_TRY(deq(lw.wo, lw.so, g.hidden, qd, 0));
            LAUNCH_TRY(dense(PL.o, R, g.hidden, qd, (g.hidden + DT_BN - 1) / DT_BN * DT_BN, 1 << 30));
            rn = ResidNormArgs{};
            rn.x = x;
            rn.y = y;
            rn.rows = R;
            rn.hidden = g.hidden;
            rn.w = c->tgt[l].ln_mlp;
            rn.eps = g.rms_eps;
            rn.hi = hi;
            rn.lo = lo;
            rn.f16 = q4 ? 1 : 0;
            LAUNCH_TRY(launch_resid_norm(rn, s));
            if (q4) {
                LAUNCH_TRY(deq(lw.w_gate, lw.s_gate, g.ffn, g.hidden, 0));
                LAUNCH_TRY(deq(lw.w_up, lw.s_up, g.ffn, g.hidden, g.ffn));
            }
            LAUNCH_TRY(dense_swiglu(PL.gu, R));
            if (q4) LAUNCH_TRY(deq(lw.w_down, lw.s_down, g.hidden, g.ffn, 0));
            LAUNCH_TRY(dense(PL.down, R, g.hidden, g.ffn, (g.hidden + DT_BN - 1) / DT_BN * DT_BN, 1 << 30));
        }
        if (g.drf_layers > 0 && p0 + R > commit_lo) {   // the committed rows of this pass
            const int r0 = commit_lo > p0 ? commit_lo - p0 : 0;
            if (int r = ingest_rows(c, c->d_fc_pp, 1, r0, R - r0, p0 + r0, s)) return r;
        }
    }
    return DFLASH_OK;
}

}  // namespace

int dflash_prefill_taps(dflash_ctx* c, const int32_t* prompt_ids, int32_t n_prompt,
                        const void* ext_taps, int32_t n_ext, int32_t hc, int32_t first_token,
                        int32_t max_new, dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    const dflash_config& g = c->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Emit em;
    em.s = s;
    if (max_new < 1) return fail(DFLASH_ERR_ARG, "max_new %d < 1", max_new);
    if (int r0 = pending_error()) return r0;
    int r;
    if (g.tgt_layers > 0) {
        if (!prompt_ids || n_prompt < 1) return fail(DFLASH_ERR_ARG, "prompt missing");
        if (n_prompt + 1 > g.max_seq) return fail(DFLASH_ERR_CAPACITY, "prompt of %d exceeds max_seq %d", n_prompt, g.max_seq);
        const int commit_lo = g.window > 0 ? (n_prompt > g.window ? n_prompt - g.window : 0) : 0;
        int p_first = 0;
        if (c->dense_prefill && n_prompt > DFL_MAX_ROWS) {
            // every row through the dense forward (its passes also commit
            // the taps to the drafter's context); the last chunk's residual
            // rows then take the final norm into the round's LM head, which
            // gives the first token, and the acceptance sets the round state
            if ((r = run_dense_prefill(c, prompt_ids, n_prompt, commit_lo, s))) return r;
            const int p0 = (n_prompt - 1) / DFL_MAX_ROWS * DFL_MAX_ROWS, T = n_prompt - p0;
            const int pass0 = (n_prompt - 1) / PF_ROWS * PF_ROWS;   // first row of the last pass
            RowsArgs ra = rows_args(c, FWD_PREFILL);
            ra.pos0 = p0;
            ra.T = T;
            ra.tokens = prompt_ids;
            ra.embed = nullptr;
            ra.x_src = c->buf<float>(c->L.pp_x) + (size_t)(p0 - pass0) * g.hidden;
            ra.w0 = c->w.final_norm_tgt;
            ra.xn_type = c->xt_lm();   // the LM head's input, as the last layer writes it
            LAUNCH_TRY(launch_prepare_rows(ra, s));
            if ((r = run_lm_head(c, c->verify_logits, em))) return r;
            AcceptArgs aa = accept_args(c, FWD_PREFILL);
            aa.max_new = max_new;
            aa.prompt_len = n_prompt;
            LAUNCH_TRY(launch_accept(aa, s));
            p_first = n_prompt;
        }
        for (int p0 = p_first; p0 < n_prompt; p0 += DFL_MAX_ROWS) {
            const int T = n_prompt - p0 < DFL_MAX_ROWS ? n_prompt - p0 : DFL_MAX_ROWS;
            RowsArgs ra = rows_args(c, FWD_PREFILL);
            ra.pos0 = p0;
            ra.T = T;
            ra.tokens = prompt_ids;
            LAUNCH_TRY(launch_prepare_rows(ra, s));
            LAUNCH_TRY(launch_set_chunk(c->st(), p0, T, commit_lo, s));
            if ((r = run_layers(c, true, em))) return r;
            if (p0 + T == n_prompt) {
                if ((r = run_lm_head(c, c->verify_logits, em))) return r;
                AcceptArgs aa = accept_args(c, FWD_PREFILL);
                aa.max_new = max_new;
                aa.prompt_len = n_prompt;
                LAUNCH_TRY(launch_accept(aa, s));
            }
            if (g.drf_layers > 0 && p0 + T > commit_lo)
                if ((r = run_ingest(c, em))) return r;
        }
    } else {
        if (!ext_taps || n_ext < 1 || hc < 1) return fail(DFLASH_ERR_ARG, "external taps missing");
        if (n_ext + g.block_max > g.max_seq) return fail(DFLASH_ERR_CAPACITY, "%d tap rows + block exceed max_seq %d", n_ext, g.max_seq);
        if (first_token < 0 || first_token >= g.vocab) return fail(DFLASH_ERR_ARG, "first_token %d", first_token);
        if (g.hidden % 8) return fail(DFLASH_ERR_CONFIG, "hidden must be a multiple of 8");
        const int commit_lo = g.window > 0 ? (n_ext > g.window ? n_ext - g.window : 0) : 0;
        const int es = elem_size(g.dtype);
        if (c->dense_ingest) {
            if ((r = run_dense_ingest(c, ext_taps, n_ext, hc, commit_lo, s))) return r;
        } else
        for (int p0 = commit_lo / DFL_MAX_ROWS * DFL_MAX_ROWS; p0 < n_ext; p0 += DFL_MAX_ROWS) {
            const int T = n_ext - p0 < DFL_MAX_ROWS ? n_ext - p0 : DFL_MAX_ROWS;
            RowsArgs ra = rows_args(c, FWD_PREFILL);
            ra.pos0 = p0;
            ra.T = T;
            ra.embed = nullptr;
            ra.amax = nullptr;
            LAUNCH_TRY(launch_prepare_rows(ra, s));
            LAUNCH_TRY(launch_set_chunk(c->st(), p0, T, commit_lo, s));
            TapArgs ta{};
            for (int i = 0; i < g.n_taps; ++i)
                ta.src[i] = static_cast<const uint8_t*>(ext_taps) +
                            ((size_t)i * n_ext + p0) * hc * g.hidden * es;
            ta.n_layers = g.n_taps;
            ta.rows = T;
            ta.hc = hc;
            ta.hidden = g.hidden;
            ta.in_type = g.dtype == DFLASH_F32 ? XT_F32 : XT_BF16;
            ta.out = c->ws + c->L.taps;
            ta.out_type = c->act_xt();
            ta.out_row_stride = (long long)g.n_taps * g.hidden;
            LAUNCH_TRY(launch_tap_reduce(ta, s));
            if ((r = run_ingest(c, em))) return r;
        }
        LAUNCH_TRY(launch_set_ext_state(c->st(), n_ext, first_token, max_new, g.block_max, g.max_seq,
                                        g.eos_id, s));
    }
    c->prefilled = true;
    return DFLASH_OK;
}

int dflash_adopt_kv(dflash_ctx* c, int32_t n, int32_t pending_token, int32_t max_new,
                    dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    const dflash_config& g = c->cfg;
    if (n < 1 || n + 1 > g.max_seq) return fail(DFLASH_ERR_CAPACITY, "n %d outside [1, max_seq)", n);
    if (pending_token < 0 || pending_token >= g.vocab) return fail(DFLASH_ERR_ARG, "token %d", pending_token);
    if (max_new < 1) return fail(DFLASH_ERR_ARG, "max_new %d < 1", max_new);
    LAUNCH_TRY(launch_set_ext_state(c->st(), n, pending_token, max_new, g.block_max, g.max_seq,
                                    g.eos_id, reinterpret_cast<cudaStream_t>(stream)));
    c->prefilled = true;
    return DFLASH_OK;
}

int dflash_draft_block(dflash_ctx* c, int32_t* draft_ids, dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    if (int r0 = pending_error()) return r0;
    const dflash_config& g = c->cfg;
    if (g.drf_layers == 0) return fail(DFLASH_ERR_STATE, "no drafter configured");
    if (!c->prefilled) return fail(DFLASH_ERR_STATE, "draft before prefill");
    if (!draft_ids) return fail(DFLASH_ERR_ARG, "draft_ids is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Emit em;
    em.s = s;
    LAUNCH_TRY(launch_prepare_rows(rows_args(c, FWD_DRAFT), s));
    int r = run_layers(c, false, em);
    if (r) return r;
    if ((r = run_lm_head(c, c->draft_logits, em))) return r;
    AcceptArgs aa = accept_args(c, FWD_DRAFT);
    aa.draft_out = draft_ids;
    LAUNCH_TRY(launch_accept(aa, s));
    return DFLASH_OK;
}

int dflash_verify_accept(dflash_ctx* c, const int32_t* draft_ids, int32_t* tokens_out,
                         int32_t* n_emitted, dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    const dflash_config& g = c->cfg;
    if (g.tgt_layers == 0) return fail(DFLASH_ERR_STATE, "no target configured");
    if (!c->prefilled) return fail(DFLASH_ERR_STATE, "verify before prefill");
    if (!tokens_out || !n_emitted) return fail(DFLASH_ERR_ARG, "tokens_out / n_emitted is NULL");
    if (int r0 = pending_error()) return r0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int mode = draft_ids ? FWD_VERIFY : FWD_GREEDY;
    Emit em;
    em.s = s;
    RowsArgs ra = rows_args(c, mode);
    ra.tokens = draft_ids;
    LAUNCH_TRY(launch_prepare_rows(ra, s));
    int r = run_layers(c, true, em);
    if (r) return r;
    if ((r = run_lm_head(c, c->verify_logits, em))) return r;
    AcceptArgs aa = accept_args(c, mode);
    aa.draft_ids = draft_ids;
    aa.tokens_out = tokens_out;
    aa.n_emitted = n_emitted;
    LAUNCH_TRY(launch_accept(aa, s));
    if (g.drf_layers > 0)
        if ((r = run_ingest(c, em))) return r;
    return DFLASH_OK;
}

int dflash_rollback(dflash_ctx* c, int64_t new_len, int32_t token, dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    if (!c->prefilled) return fail(DFLASH_ERR_STATE, "rollback before prefill");
    if (new_len < 1 || new_len >= c->cfg.max_seq) return fail(DFLASH_ERR_ARG, "new_len %lld", (long long)new_len);
    if (token < 0 || token >= c->cfg.vocab) return fail(DFLASH_ERR_ARG, "token %d", token);
    LAUNCH_TRY(launch_rollback(c->st(), (int)new_len, token, c->cfg.block_max, c->cfg.max_seq,
                               reinterpret_cast<cudaStream_t>(stream)));
    return DFLASH_OK;
}

int dflash_stats(dflash_ctx* c, dflash_stats_t* out, dflash_stream_t stream) {
    if (!c || !out) return fail(DFLASH_ERR_ARG, "NULL argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DevState h;
    CUDA_TRY(cudaMemcpyAsync(&h, c->st(), sizeof h, cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    memset(out, 0, sizeof *out);
    out->rounds = h.rounds;
    out->emitted = h.emitted;
    for (int j = 0; j < DFLASH_MAX_BLOCK; ++j) out->accept_hist[j] = h.accept_hist[j];
    out->n = h.n;
    out->t_n = h.t_n;
    out->block_len = h.bl;
    out->generated = h.generated;
    out->max_new = h.max_new;
    out->ctx_len = h.ctx_len;
    out->finished = h.finished;
    out->last_accept = h.last_a;
    out->device_error = h.err;
    return DFLASH_OK;
}

int dflash_check(dflash_ctx* c, dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaStreamSynchronize(s));
    int err[2];
    CUDA_TRY(cudaMemcpy(err, &c->st()->err, sizeof err, cudaMemcpyDeviceToHost));
    if (err[0] == DERR_NONE) return DFLASH_OK;
    const int zero[2] = {0, 0};   // report once, then clear
    CUDA_TRY(cudaMemcpy(&c->st()->err, zero, sizeof zero, cudaMemcpyHostToDevice));
    // a kernel that gave up may have left split-K or attention counters set
    CUDA_TRY(cudaMemset(c->ws + c->L.counters, 0, (size_t)MAX_TILES * 4));
    CUDA_TRY(cudaMemset(c->ws + c->L.acnt, 0, (size_t)2 * c->cfg.n_kv * 4));
    if (err[0] == DERR_TIMEOUT) return fail(DFLASH_ERR_TIMEOUT, "bounded wait expired (site %d)", err[1]);
    return fail(DFLASH_ERR_DEVICE, "device error %d (info %d)", err[0], err[1]);
}

int dflash_attention_form(const dflash_ctx* c, int32_t model) {
    if (!c || (model != 0 && model != 1)) return fail(DFLASH_ERR_ARG, "NULL context or model %d", model);
    if (c->cfg.dtype != DFLASH_BF16 || c->attn_split_chunks[model] <= 0) return 0;
    return c->attn_tc[model] ? 2 : 1;
}

int dflash_progress(dflash_ctx* c, int32_t* out, dflash_stream_t stream) {
    if (!c || !out) return fail(DFLASH_ERR_ARG, "NULL argument");
    LAUNCH_TRY(launch_progress(c->st(), out, reinterpret_cast<cudaStream_t>(stream)));
    return DFLASH_OK;
}

int dflash_selftest_timeout(dflash_ctx* c, int64_t limit_ns, dflash_stream_t stream) {
    if (!c) return fail(DFLASH_ERR_ARG, "ctx is NULL");
    if (limit_ns < 0 || limit_ns > 2000000000LL) return fail(DFLASH_ERR_ARG, "limit %lld ns", (long long)limit_ns);
    LAUNCH_TRY(launch_selftest_wait(c->st(), (unsigned long long)limit_ns,
                                    reinterpret_cast<cudaStream_t>(stream)));
    return DFLASH_OK;
}

int dflash_tap_reduce(const void* const* layer_streams, int32_t n_layers, int32_t rows, int32_t hc,
                      int32_t hidden, float* out, dflash_stream_t stream) {
    if (!layer_streams || !out) return fail(DFLASH_ERR_ARG, "NULL argument");
    if (n_layers < 1 || n_layers > 8 || rows < 0 || hc < 1 || hidden < 8 || hidden % 8)
        return fail(DFLASH_ERR_ARG, "bad shape (layers %d rows %d hc %d hidden %d)", n_layers, rows, hc, hidden);
    if (rows == 0) return DFLASH_OK;
    TapArgs ta{};
    for (int i = 0; i < n_layers; ++i) {
        if (!aligned16(layer_streams[i])) return fail(DFLASH_ERR_ARG, "stream %d misaligned", i);
        ta.src[i] = layer_streams[i];
    }
    if (!aligned16(out)) return fail(DFLASH_ERR_ARG, "out misaligned");
    ta.n_layers = n_layers;
    ta.rows = rows;
    ta.hc = hc;
    ta.hidden = hidden;
    ta.in_type = XT_BF16;
    ta.out = out;
    ta.out_type = XT_F32;
    ta.out_row_stride = (long long)n_layers * hidden;
    LAUNCH_TRY(launch_tap_reduce(ta, reinterpret_cast<cudaStream_t>(stream)));
    return DFLASH_OK;
}

size_t dflash_linear_workspace_bytes(int32_t n, int32_t k) {
    if (n < GEMM_BN || n % GEMM_BN || k < 64 || k % 64) return 0;
    return align_up((size_t)MAX_SMS * 2 * GEMM_BN * DFL_MAX_ROWS * 4, 1024) +
           align_up((size_t)(n / GEMM_BN) * 4, 256) + align_up(sizeof(DevState), 256);
}

int dflash_linear_dense(const void* w, const void* x, const void* x_lo, int32_t m, int32_t n, int32_t k,
                        float* y, int32_t* err, dflash_stream_t stream) {
    if (!w || !x || !y || !err) return fail(DFLASH_ERR_ARG, "NULL argument");
    if (m < 1 || n < 1 || k < DT_BK || k % DT_BK)
        return fail(DFLASH_ERR_ARG, "m %d n %d k %d: m, n >= 1, k a multiple of 64", m, n, k);
    if (!aligned16(w) || !aligned16(x) || !aligned16(y) || !aligned16(err) || (x_lo && !aligned16(x_lo)))
        return fail(DFLASH_ERR_ARG, "misaligned buffer");
    if (n % 4) return fail(DFLASH_ERR_ARG, "n %d: rows of y must stay 16-byte aligned (n a multiple of 4)", n);
    if (int r0 = get_encode()) return r0;
    if (int r0 = pending_error()) return r0;
    DenseMaps maps;
    memset(&maps, 0, sizeof maps);
    int r = make_map_raw(&maps.x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, m, DT_BK, DT_BM,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r && x_lo)
        r = make_map_raw(&maps.x_lo, x_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, m, DT_BK, DT_BM,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r)
        r = make_map_raw(&maps.w[0], w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, n, DT_BK, DT_WBOX,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (r) return r;
    DenseArgs a{};
    a.M = m;
    a.N = n;
    a.K = k;
    a.n_seg0 = (n + DT_BN - 1) / DT_BN * DT_BN;
    a.n_seg1 = 1 << 30;
    a.x_split = x_lo ? 1 : 0;
    a.y = y;
    a.ldy = n;
    a.err = err;
    const int e = launch_dense(maps, a, reinterpret_cast<cudaStream_t>(stream));
    if (e) return fail(DFLASH_ERR_CUDA, "dense GEMM launch: %s", cudaGetErrorString((cudaError_t)e));
    return DFLASH_OK;
}

int dflash_linear(const void* w, const void* x, int32_t n, int32_t k, float* y, void* workspace,
                  size_t workspace_bytes, int32_t* err, dflash_stream_t stream) {
    if (!w || !x || !y || !workspace || !err) return fail(DFLASH_ERR_ARG, "NULL argument");
    const size_t need = dflash_linear_workspace_bytes(n, k);
    if (need == 0) return fail(DFLASH_ERR_ARG, "n %d k %d: n a multiple of 128, k of 64", n, k);
    if (workspace_bytes < need) return fail(DFLASH_ERR_ARG, "workspace %zu < %zu", workspace_bytes, need);
    if (!aligned16(w) || !aligned16(x) || !aligned16(y) || !aligned16(workspace) || !aligned16(err))
        return fail(DFLASH_ERR_ARG, "misaligned buffer");
    if (int r0 = get_encode()) return r0;
    if (int r0 = pending_error()) return r0;
    int dev = 0, sms = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (sms > 256) sms = 256;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DevState* st = reinterpret_cast<DevState*>(ws + need - align_up(sizeof(DevState), 256));
    return run_linear_store(
        w, x, n, k, y, reinterpret_cast<float*>(ws),
        reinterpret_cast<int*>(ws + align_up((size_t)MAX_SMS * 2 * GEMM_BN * DFL_MAX_ROWS * 4, 1024)),
        st, &st->err, 2 * sizeof(int), err, sms, reinterpret_cast<cudaStream_t>(stream));
}

int dflash_quantize_int4g64(const float* w, int32_t n, int32_t k, uint8_t* packed, uint16_t* scales,
                            dflash_stream_t stream) {
    if (!w || !packed || !scales) return fail(DFLASH_ERR_ARG, "NULL argument");
    if (n < 1 || k < 256 || k % 256) return fail(DFLASH_ERR_ARG, "n %d k %d: k must be a multiple of 256", n, k);
    LAUNCH_TRY(launch_quantize_int4g64(w, n, k, packed, scales, reinterpret_cast<cudaStream_t>(stream)));
    return DFLASH_OK;
}

}  // extern "C"
