// Several independent sequences decoded in lockstep rounds: one drafter
// forward and one target forward over all sequences' rows at once.
//
// By page: the verify costs time by its row count ("[RFC] DFlash",
// "Performance": 32 ms at T = 1 against 239 ms at T = 16 on the pages'
// hardware), and each sequence's round is the draft -> batched verify ->
// first-mismatch acceptance -> KV rollback of "Key Implementation Details",
// Phase 3.  Batching sequences is this library's extension (the pages verify
// one sequence's [1, 1 + m] rows per forward): every sequence keeps its own
// context (round state, target and draft caches, block length, budget,
// statistics) and its state evolves exactly as dflash_draft_block /
// dflash_verify_accept would move it; the sequences share the weight
// stream.
//
// Rows: sequence s owns rows 16 s .. 16 s + 15 of every activation (its
// forward's T rows first, the rest zero); with S sequences the GEMMs have
// M = 16 S rows, a real contraction at S >= 8, so they run on the dense
// tcgen05 GEMM with the activations as bf16 hi/lo planes (the round's
// precision).  A GEMM's k-split count and tile width depend on N and K only,
// and attention, norms and RoPE work row by row, so a sequence's results do
// not depend on how many sequences the batch has.

#include <cmath>
#include <cstring>
#include <vector>

#include "../../include/dflash.h"
#include "attention.cuh"
#include "capi_internal.cuh"
#include "gemm.cuh"
#include "gemm_tc.cuh"
#include "kernels.cuh"
#include "kernels_dev.cuh"

using namespace dfl;

namespace {

constexpr int BATCH_MAX_SEQ = 32;

__device__ __forceinline__ void bf16_hilo(void* hi, void* lo, size_t i, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    reinterpret_cast<__nv_bfloat16*>(hi)[i] = h;
    reinterpret_cast<__nv_bfloat16*>(lo)[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

struct BlockBar {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// ---------------------------------------------------------------- row preparation

struct BatchRowsArgs {
    int mode;                       // FWD_DRAFT | FWD_VERIFY | FWD_GREEDY
    DevState* const* sts;           // [S]
    int hidden, vocab, mask_id, head_dim, block_max;
    const int32_t* tokens;          // VERIFY: draft ids [S][block_max - 1]
    const __nv_bfloat16* embed;     // [vocab][hidden]
    const float* w0;                // input-norm weight of the model's first layer
    float eps;
    const float* tab_cos;           // RoPE angles of every cache position [tab_rows][head_dim / 2]
    const float* tab_sin;
    int tab_rows;
    float* x;                       // [R][hidden] residual
    void* hi;                       // [R][hidden] bf16: RMSNorm(x) * w0, high part
    void* lo;                       //                  ... and the rounding remainder
    float* rope_cos;                // [R][head_dim / 2]
    float* rope_sin;
    unsigned long long* amax;       // [R] argmax keys, reset
};

// One CTA of 256 threads per row r = 16 s + t: sequence s's forward
// descriptor, token, RoPE angles and argmax reset exactly as the
// single-sequence row preparation makes them, then the embedding row and
// the first layer's input RMSNorm as hi/lo planes.
__global__ void __launch_bounds__(256) batch_rows_kernel(BatchRowsArgs b) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x, sq = r >> 4, t = r & 15, tid = threadIdx.x;
    __shared__ int sh[3];
    __shared__ float s_part[8];
    const int half = b.head_dim / 2;
    RowsArgs a{};
    a.mode = b.mode;
    a.hidden = b.hidden;
    a.vocab = b.vocab;
    a.mask_id = b.mask_id;
    a.tokens = b.tokens ? b.tokens + (size_t)sq * (b.block_max - 1) : nullptr;
    a.embed = nullptr;   // the gather and the norm follow below
    a.x = b.x;
    a.rope_cos = b.rope_cos + (size_t)sq * DFL_MAX_ROWS * half;
    a.rope_sin = b.rope_sin + (size_t)sq * DFL_MAX_ROWS * half;
    a.head_dim = b.head_dim;
    a.tab_cos = b.tab_cos;
    a.tab_sin = b.tab_sin;
    a.tab_rows = b.tab_rows;
    a.amax = b.amax + (size_t)sq * DFL_MAX_ROWS;
    a.st = b.sts[sq];
    kdev::prepare_row(a, t, tid, 256, sh, BlockBar());
    __syncthreads();
    const int T = sh[0], tok = sh[2];
    float* xr = b.x + (size_t)r * b.hidden;
    float ss = 0.f;
    for (int j = tid; j < b.hidden; j += 256) {
        const float v = t < T ? __bfloat162float(b.embed[(size_t)tok * b.hidden + j]) : 0.f;
        xr[j] = v;
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += s_part[w];
    const float rstd = 1.0f / sqrtf(tot / (float)b.hidden + b.eps);
    for (int j = tid; j < b.hidden; j += 256)
        bf16_hilo(b.hi, b.lo, (size_t)r * b.hidden + j, xr[j] * b.w0[j] * rstd);
}

// ---------------------------------------------------------------- q/k/v rows

struct BatchQkvArgs {
    const float* y;                 // [R][(n_q + 2 n_kv) hd]: q heads, k heads, v heads
    int y_splits;                   // > 1: y is that many split-K slabs, summed in split order
    size_t y_slab;
    DevState* const* sts;
    int rows, n_q, n_kv, head_dim, cap, max_seq;
    const float* q_norm;
    const float* k_norm;
    float eps;
    const float* rope_cos;          // [R][hd / 2]
    const float* rope_sin;
    __half* q_out;                  // [S][n_q][16][hd]
    __half* cache;                  // every sequence's cache of the model [S][layers][2][n_kv][cap][hd]
    int n_layers, layer;
};

__device__ __forceinline__ void rope_pair(float (&v)[4], int per, const float* cs_row,
                                          const float* sn_row, int lane) {
    float cs[2], sn[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        cs[m] = m < per / 2 ? cs_row[lane + 32 * m] : 1.f;
        sn[m] = m < per / 2 ? sn_row[lane + 32 * m] : 0.f;
    }
    float o[4];
    if (per == 4) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            o[m] = v[m] * cs[m] - v[m + 2] * sn[m];
            o[m + 2] = v[m + 2] * cs[m] + v[m] * sn[m];
        }
    } else {
        o[0] = v[0] * cs[0] - v[1] * sn[0];
        o[1] = v[1] * cs[0] + v[0] * sn[0];
        o[2] = o[3] = 0.f;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = o[m];
}

// One warp per (row, head): per-head RMSNorm of q and k, RoPE at the row's
// position, q rows out, K/V rows into the row's sequence's cache (the
// formulas of the round's q/k/v epilogue).  Rows past the sequence's T
// write zero q rows and no cache rows.
__global__ void batch_qkv_rows_kernel(BatchQkvArgs a) {
    pdl_trigger();
    pdl_wait();
    const int heads = a.n_q + 2 * a.n_kv;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= a.rows * heads) return;
    const int r = warp / heads, h = warp % heads, sq = r >> 4, t = r & 15;
    DevState* st = a.sts[sq];
    const int T = st->fwd_T, pos = st->fwd_pos0 + t;
    const bool is_q = h < a.n_q, is_k = !is_q && h < a.n_q + a.n_kv;
    const int hd = a.head_dim, per = hd / 32;
    float v[4];
    const float* src = a.y + (size_t)r * heads * hd + (size_t)h * hd;
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = (m < per && t < T) ? src[lane + 32 * m] : 0.f;
    if (a.y_splits > 1 && t < T) {
        // every split's loads in flight at once, then the adds in split order
        float u[7][4];
#pragma unroll
        for (int z = 1; z < 8; ++z)
#pragma unroll
            for (int m = 0; m < 4; ++m)
                u[z - 1][m] = (z < a.y_splits && m < per) ? __ldcg(src + (size_t)z * a.y_slab + lane + 32 * m) : 0.f;
#pragma unroll
        for (int z = 1; z < 8; ++z)
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (z < a.y_splits) v[m] += u[z - 1][m];
        for (int z = 8; z < a.y_splits; ++z)
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (m < per) v[m] += __ldcg(src + (size_t)z * a.y_slab + lane + 32 * m);
    }
    if (t < T && (is_q || is_k)) {
        const float* nw = is_q ? a.q_norm : a.k_norm;
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(v[m], v[m], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)hd + a.eps);
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = m < per ? v[m] * inv * nw[lane + 32 * m] : 0.f;
        rope_pair(v, per, a.rope_cos + (size_t)r * (hd / 2), a.rope_sin + (size_t)r * (hd / 2), lane);
    }
    if (is_q) {
        __half* q = a.q_out + (((size_t)sq * a.n_q + h) * DFL_MAX_ROWS + t) * hd;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (m < per) q[lane + 32 * m] = __float2half_rn(v[m]);
        return;
    }
    if (t >= T) return;
    if (pos < 0 || pos >= a.max_seq || pos >= a.cap) {
        if (lane == 0) set_error(st, DERR_INDEX, pos);
        return;
    }
    const int kh = is_k ? h - a.n_q : h - a.n_q - a.n_kv;
    const size_t run = (((size_t)sq * a.n_layers + a.layer) * 2 + (is_k ? 0 : 1)) * a.n_kv + kh;
    __half* dst = a.cache + (run * a.cap + pos) * hd;
#pragma unroll
    for (int m = 0; m < 4; ++m)
        if (m < per) dst[lane + 32 * m] = __float2half_rn(v[m]);
}

// ---------------------------------------------------------------- acceptance

struct BatchAcceptArgs {
    int mode;
    DevState* const* sts;
    const unsigned long long* amax;   // [R]
    const int32_t* draft_ids;         // VERIFY: [S][block_max - 1]
    int32_t* draft_out;               // DRAFT: [S][block_max - 1]
    int32_t* tokens_out;              // VERIFY/GREEDY: [S][block_max]
    int32_t* n_emitted;               // [S]
    int block_max, max_seq, eos_id;
};

// One block per sequence: the single-sequence acceptance and bookkeeping on
// the sequence's own rows and state.
__global__ void batch_accept_kernel(BatchAcceptArgs b) {
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x != 0) return;
    const int sq = blockIdx.x, B = b.block_max;
    AcceptArgs a{};
    a.mode = b.mode;
    a.amax = b.amax + (size_t)sq * DFL_MAX_ROWS;
    a.draft_ids = b.draft_ids ? b.draft_ids + (size_t)sq * (B - 1) : nullptr;
    a.draft_out = b.draft_out ? b.draft_out + (size_t)sq * (B - 1) : nullptr;
    a.tokens_out = b.tokens_out ? b.tokens_out + (size_t)sq * B : nullptr;
    a.n_emitted = b.n_emitted ? b.n_emitted + sq : nullptr;
    a.block_max = B;
    a.max_seq = b.max_seq;
    a.eos_id = b.eos_id;
    a.st = b.sts[sq];
    kdev::accept_run(a);
}

// ---------------------------------------------------------------- tap commit

struct BatchCtxKvArgs {
    const float* y;                 // [R][2 n_kv hd]: K heads, then V heads
    DevState* const* sts;
    int rows, n_kv, head_dim, cap, max_seq;
    const float* k_norm;
    float eps;
    const float* rope_cos;          // [R][hd / 2] (the verify's positions)
    const float* rope_sin;
    __half* cache;                  // every sequence's draft cache [S][layers][2][n_kv][cap][hd]
    int n_layers;
    // layers layer0 .. layer0 + nl - 1: y rows hold their K and V one layer
    // after another, k_norm their weights [nl][hd]
    int layer0, nl;
};

// One warp per (row, layer, kv head, K or V): the committed rows t <
// fwd_commit of each sequence, at positions fwd_pos0 + t: k RMSNorm and
// RoPE on K, both into the sequence's draft cache (the round's tap-commit
// formulas).
__global__ void batch_ctx_kv_kernel(BatchCtxKvArgs a) {
    pdl_trigger();
    pdl_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= a.rows * a.nl * a.n_kv * 2) return;
    const int per_row = a.nl * 2 * a.n_kv;
    const int r = warp / per_row, rl = warp % per_row, li = rl / (2 * a.n_kv), rem = rl % (2 * a.n_kv);
    const int sq = r >> 4, t = r & 15;
    DevState* st = a.sts[sq];
    if (t < st->fwd_commit_r0 || t >= st->fwd_commit_r0 + st->fwd_commit) return;
    const bool is_k = rem < a.n_kv;
    const int kh = is_k ? rem : rem - a.n_kv;
    const int hd = a.head_dim, per = hd / 32;
    const int pos = st->fwd_pos0 + t;
    if (pos < 0 || pos >= a.max_seq || pos >= a.cap) {
        if (lane == 0) set_error(st, DERR_INDEX, pos);
        return;
    }
    const float* src = a.y + (size_t)r * per_row * hd + (size_t)rl * hd;
    const float* k_norm = a.k_norm + (size_t)li * hd;
    float v[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = m < per ? src[lane + 32 * m] : 0.f;
    if (is_k) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(v[m], v[m], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)hd + a.eps);
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = m < per ? v[m] * inv * k_norm[lane + 32 * m] : 0.f;
        rope_pair(v, per, a.rope_cos + (size_t)r * (hd / 2), a.rope_sin + (size_t)r * (hd / 2), lane);
    }
    const size_t run = (((size_t)sq * a.n_layers + a.layer0 + li) * 2 + (is_k ? 0 : 1)) * a.n_kv + kh;
    __half* dst = a.cache + (run * a.cap + pos) * hd;
#pragma unroll
    for (int m = 0; m < 4; ++m)
        if (m < per) dst[lane + 32 * m] = __float2half_rn(v[m]);
}

template <typename... KArgs, typename... Args>
int launch_warps(void (*kern)(KArgs...), long long warps, cudaStream_t s, Args&&... args) {
    if (warps <= 0) return 0;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    return (int)launch_k(kern, dim3(blocks), dim3(256), 0, s, std::forward<Args>(args)...);
}

}  // namespace

// ==================================================================== host

struct dflash_batch {
    dflash_config cfg;
    int S = 0, R = 0, sms = 0;
    // tile width of the projections: 128 up to 8 sequences (one row tile),
    // 256 above, so that two row tiles keep the split GEMMs in one wave; the
    // k-split counts stay those of 128-column tiles and a tensor-core
    // output element's sum over k does not depend on the tile width, so a
    // sequence's results stay the same for every S
    int bn = 128;
    std::vector<dflash_ctx*> ctx;
    uint8_t* kv_t = nullptr;
    uint8_t* kv_d = nullptr;
    // batch workspace
    DevState** sts = nullptr;
    float* x = nullptr;
    void* hi = nullptr;
    void* lo = nullptr;
    void* ahi = nullptr;   // [R][ffn] SwiGLU output planes: the down projection's input
    void* alo = nullptr;
    void* thi = nullptr;
    void* tlo = nullptr;
    float* y = nullptr;
    __half* q = nullptr;
    float* rcos = nullptr;
    float* rsin = nullptr;
    unsigned long long* amax = nullptr;
    float* part = nullptr;
    float* apart = nullptr;   // attention split partials
    int* err = nullptr;
    struct LayerMaps {
        DenseMaps qkv, o, gu, down, ctxkv;
    };
    std::vector<LayerMaps> tl, dl;
    DenseMaps lm{}, fc{};
    // the tap commit's context K/V of every draft layer in one GEMM, over the
    // first context's copy of the layers' [W_k; W_v] (when it has one)
    DenseMaps ctxkv_all{};
    bool grouped_ctxkv = false;
    const float* ctxkv_knorm = nullptr;
    CUtensorMap qmap{}, kvmap_t{}, kvmap_d{};
    float* verify_logits = nullptr;
    float* draft_logits = nullptr;
};

namespace {

size_t up1k(size_t v) { return (v + 1023) / 1024 * 1024; }

// Split count of a GEMM: at most one CTA per SM over the 128-column tiles,
// at most 8, at least two k-blocks per split.  Depends on N and K only.
int splits_for(int N, int K, int sms) {
    const int tiles = (N + 127) / 128;
    // rounded down: one CTA per SM, so a count past the SMs adds a wave
    // (rounding to nearest gave o and down 160 CTAs on 152 SMs)
    int z = sms / tiles;
    z = z < 1 ? 1 : (z > 8 ? 8 : z);
    const int kmax = (K / DT_BK) / 2;
    return z > kmax ? (kmax < 1 ? 1 : kmax) : z;
}

// Attention splits of a model: at most 5 per (kv head, sequence), each of a
// fixed number of 64-key chunks counted from the first visible chunk (from
// the cache capacity, or the drafter's window), so a row's split boundaries
// depend on its position only.
void attn_splits(const dflash_config& g, bool target, int* chunks, int* splits) {
    const int cap = (g.max_seq + 63) / 64 * 64;
    int maxc = cap / 64;
    if (!target && g.window > 0) {
        const int w = (g.window + DFL_MAX_ROWS + 63) / 64 + 1;
        if (w < maxc) maxc = w;
    }
    const int q = (maxc + 4) / 5;
    *chunks = q < 1 ? 1 : q;
    *splits = (maxc + *chunks - 1) / *chunks;
}

struct BatchLayout {
    size_t sts, x, hi, lo, ahi, alo, thi, tlo, y, q, rcos, rsin, amax, part, apart, err, total;
};

BatchLayout batch_layout(const dflash_config& g, int S, int sms) {
    const size_t R = (size_t)16 * S;
    const int H = g.hidden, qd = g.n_q * g.head_dim, kvd = g.n_kv * g.head_dim, F = g.ffn;
    const size_t wmax = (size_t)std::max(std::max(H, qd), F);
    // the grouped context K/V of the tap commit: every draft layer's K and V
    const int kv_all = g.drf_layers * 2 * kvd;
    const size_t ymax = (size_t)std::max(std::max(qd + 2 * kvd, 2 * F), std::max(H, kv_all));
    const int tw = g.drf_layers > 0 ? g.n_taps * H : 0;
    // partial tiles of the largest split GEMM the round runs
    size_t pf = 0;
    auto need = [&](int N, int K) {
        const int z = splits_for(N, K, sms);
        if (z > 1) pf = std::max(pf, dense_split_floats((int)R, N, z, 128));
    };
    need(qd + 2 * kvd, H);
    need(H, qd);
    need(2 * F, H);
    need(H, F);
    if (tw) {
        need(H, tw);
        need(2 * kvd, H);
        need(kv_all, H);
    }
    BatchLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += up1k(bytes); return at; };
    L.sts = take((size_t)S * sizeof(void*));
    L.x = take(R * H * 4);
    L.hi = take(R * wmax * 2);
    L.lo = take(R * wmax * 2);
    L.ahi = take(R * (size_t)F * 2);
    L.alo = take(R * (size_t)F * 2);
    L.thi = take(R * (size_t)(tw ? tw : 64) * 2);
    L.tlo = take(R * (size_t)(tw ? tw : 64) * 2);
    L.y = take(R * ymax * 4);
    L.q = take(R * (size_t)qd * 2);
    L.rcos = take(R * (size_t)(g.head_dim / 2) * 4);
    L.rsin = take(R * (size_t)(g.head_dim / 2) * 4);
    L.amax = take(R * 8);
    L.part = take(pf * 4 + 16);
    int ct, st, cd = 1, sd = 1;
    attn_splits(g, true, &ct, &st);
    if (g.drf_layers > 0) attn_splits(g, false, &cd, &sd);
    L.apart = take((size_t)S * std::max(st, sd) * DFL_MAX_ROWS * g.n_q * (g.head_dim + 2) * 4);
    L.err = take(256);
    L.total = o;
    return L;
}

int batch_cfg_ok(const dflash_config* c, int S) {
    if (!c) return report_error(DFLASH_ERR_ARG, "cfg is NULL");
    if (S < 1 || S > BATCH_MAX_SEQ) return report_error(DFLASH_ERR_ARG, "S %d outside [1, %d]", S, BATCH_MAX_SEQ);
    if (c->dtype != DFLASH_BF16 || c->tgt_wfmt != DFLASH_BF16 ||
        (c->drf_layers > 0 && c->drf_wfmt != DFLASH_BF16) || c->lm_wfmt != 0)
        return report_error(DFLASH_ERR_CONFIG, "the many-sequence round runs bf16 models (bf16 weights, tied LM head)");
    if (c->tgt_layers < 1) return report_error(DFLASH_ERR_CONFIG, "the many-sequence round needs a target");
    const int qd = c->n_q * c->head_dim, kvd = c->n_kv * c->head_dim;
    if ((c->head_dim != 64 && c->head_dim != 128) || qd % 256 || kvd % 256 || c->ffn % 256 ||
        c->hidden % 128 || (c->n_taps * c->hidden) % 64)
        return report_error(DFLASH_ERR_CONFIG, "shapes outside the dense GEMM's tiles (head_dim %d, q %d, kv %d, ffn %d)",
                            c->head_dim, qd, kvd, c->ffn);
    return DFLASH_OK;
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return 148;
    return sms;
}

// x planes [R][K] of a GEMM input (box 128 rows x 64) and its weight maps
int dense_maps(DenseMaps* m, const void* hi, const void* lo, int R, int K, const void* const* w, const int* rows,
               int nseg, int wbox = DT_WBOX) {
    memset(m, 0, sizeof *m);
    int r = encode_map(&m->x, hi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, R, DT_BK, DT_BM,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = encode_map(&m->x_lo, lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, R, DT_BK, DT_BM,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    for (int i = 0; i < nseg && !r; ++i)
        r = encode_map(&m->w[i], w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, rows[i], DT_BK, wbox,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    return r;
}

#define BTRY(x)                                                                                    \
    do {                                                                                           \
        if ((x) != 0) {                                                                            \
            const cudaError_t e_ = cudaGetLastError();                                             \
            return report_error(DFLASH_ERR_CUDA, "%s failed: %s", #x, cudaGetErrorString(e_));     \
        }                                                                                          \
    } while (0)

// Where a row kernel finds a dense GEMM's output: y rows, or the split-K
// slabs the row kernel sums itself (no reduce launch).
struct YView {
    const float* y;
    int splits;
    size_t slab;
};

int dense(dflash_batch* b, const DenseMaps& m, int N, int K, int seg0, int seg1, float* y,
          unsigned long long* amax, cudaStream_t s, YView* view = nullptr) {
    DenseArgs d{};
    d.M = b->R;
    d.N = N;
    d.K = K;
    d.n_seg0 = seg0;
    d.n_seg1 = seg1;
    d.x_split = 1;
    d.y = y;
    d.ldy = N;
    d.err = b->err;
    // 128-column tiles, except the LM head's argmax GEMM (1187 tiles of 128
    // at Qwen3's vocabulary, nearly 8 waves): 256 halves the tiles and with
    // them the re-reads of the activation block
    d.bn = amax ? 256 : b->bn;
    d.amax = amax;
    d.splits = amax ? 1 : splits_for(N, K, b->sms);
    d.part = b->part;
    d.w_ready = 1;   // the model's weights
    if (view) {
        size_t slab = 0, ldp = 0;
        dense_part_layout(d.M, N, d.bn, &slab, &ldp);
        if (d.splits > 1 && ldp == (size_t)N) {   // slab rows are y rows: the consumer sums them
            d.keep_parts = 1;
            *view = YView{b->part, d.splits, slab};
        } else {
            *view = YView{y, 1, 0};
        }
    }
    const int e = launch_dense(m, d, s);
    if (e) return report_error(DFLASH_ERR_CUDA, "dense GEMM (N %d K %d): %s", N, K, cudaGetErrorString((cudaError_t)e));
    return DFLASH_OK;
}

// Fused gate/up with the SwiGLU epilogue: silu(gate) * up straight into
// the down projection's input planes (ahi / alo), at the context's tile width.
int dense_swiglu(dflash_batch* b, const DenseMaps& m, int F, int K, cudaStream_t s) {
    DenseArgs d{};
    d.M = b->R;
    d.N = 2 * F;
    d.K = K;
    d.n_seg0 = 1 << 30;
    d.n_seg1 = 1 << 30;
    d.x_split = 1;
    d.err = b->err;
    d.bn = b->bn;
    d.splits = 1;
    d.swiglu = 1;
    d.up_map = 1;
    d.up_row = 0;
    d.act_hi = b->ahi;
    d.act_lo = b->alo;
    d.act_ld = F;
    d.w_ready = 1;
    const int e = launch_dense(m, d, s);
    if (e) return report_error(DFLASH_ERR_CUDA, "dense SwiGLU GEMM (F %d K %d): %s", F, K, cudaGetErrorString((cudaError_t)e));
    return DFLASH_OK;
}

// The decoder layers of one model over every sequence's rows (input norm of
// the first layer already in hi/lo); the last layer leaves the final norm
// of x in hi/lo for the LM head.  Target layers copy their outputs at the
// tap layers into thi/tlo.
int batch_layers(dflash_batch* b, bool target, cudaStream_t s) {
    const dflash_config& g = b->cfg;
    const int H = g.hidden, qd = g.n_q * g.head_dim, kvd = g.n_kv * g.head_dim, F = g.ffn;
    const int nl = target ? g.tgt_layers : g.drf_layers;
    const dflash_layer* lw = ctx_layers(b->ctx[0], target);
    const dflash_weights& w = ctx_weights(b->ctx[0]);
    const int cap = (g.max_seq + 63) / 64 * 64;
    for (int l = 0; l < nl; ++l) {
        const dflash_batch::LayerMaps& M = target ? b->tl[l] : b->dl[l];
        YView yv{};
        int r = dense(b, M.qkv, qd + 2 * kvd, H, qd, qd + kvd, b->y, nullptr, s, &yv);
        if (r) return r;
        BatchQkvArgs qa{};
        qa.y = yv.y;
        qa.y_splits = yv.splits;
        qa.y_slab = yv.slab;
        qa.sts = b->sts;
        qa.rows = b->R;
        qa.n_q = g.n_q;
        qa.n_kv = g.n_kv;
        qa.head_dim = g.head_dim;
        qa.cap = cap;
        qa.max_seq = g.max_seq;
        qa.q_norm = lw[l].q_norm;
        qa.k_norm = lw[l].k_norm;
        qa.eps = g.rms_eps;
        qa.rope_cos = b->rcos;
        qa.rope_sin = b->rsin;
        qa.q_out = b->q;
        qa.cache = reinterpret_cast<__half*>(target ? b->kv_t : b->kv_d);
        qa.n_layers = nl;
        qa.layer = l;
        BTRY(launch_warps(batch_qkv_rows_kernel, (long long)b->R * (g.n_q + 2 * g.n_kv), s, qa));
        BatchAttnArgs at{};
        at.m.n_q = g.n_q;
        at.m.n_kv = g.n_kv;
        at.m.head_dim = g.head_dim;
        at.m.layer = l;
        at.m.cap = cap;
        at.m.causal = target ? 1 : 0;
        at.m.window = target ? 0 : g.window;
        at.m.scale = 1.0f / sqrtf((float)g.head_dim);
        at.sts = b->sts;
        at.n_layers = nl;
        attn_splits(g, target, &at.split_chunks, &at.splits);
        at.part = b->apart;
        at.out_hi = b->hi;
        at.out_lo = b->lo;
        BTRY(launch_batch_attention(b->qmap, target ? b->kvmap_t : b->kvmap_d, at, b->S, s));
        if ((r = dense(b, M.o, H, qd, 1 << 30, 1 << 30, b->y, nullptr, s, &yv))) return r;
        ResidNormArgs rn{};
        rn.x = b->x;
        rn.y = yv.y;
        rn.y_splits = yv.splits;
        rn.y_slab = yv.slab;
        rn.rows = b->R;
        rn.hidden = H;
        rn.w = lw[l].ln_mlp;
        rn.eps = g.rms_eps;
        rn.hi = b->hi;
        rn.lo = b->lo;
        BTRY(launch_resid_norm(rn, s));
        if ((r = dense_swiglu(b, M.gu, F, H, s))) return r;
        if ((r = dense(b, M.down, H, F, 1 << 30, 1 << 30, b->y, nullptr, s, &yv))) return r;
        rn = ResidNormArgs{};
        rn.x = b->x;
        rn.y = yv.y;
        rn.y_splits = yv.splits;
        rn.y_slab = yv.slab;
        rn.rows = b->R;
        rn.hidden = H;
        rn.w = l + 1 < nl ? lw[l + 1].ln_attn : (target ? w.final_norm_tgt : w.final_norm_drf);
        rn.eps = g.rms_eps;
        rn.hi = b->hi;
        rn.lo = b->lo;
        if (target && g.drf_layers > 0)
            for (int i = 0; i < g.n_taps; ++i)
                if (g.tap_layer[i] == l) {
                    rn.tap_hi = b->thi;
                    rn.tap_lo = b->tlo;
                    rn.tap_ld = (long long)g.n_taps * H;
                    rn.tap_col = i * H;
                }
        BTRY(launch_resid_norm(rn, s));
    }
    return DFLASH_OK;
}

int batch_rows(dflash_batch* b, int mode, const int32_t* tokens, bool target, cudaStream_t s) {
    const dflash_config& g = b->cfg;
    BatchRowsArgs ra{};
    ra.mode = mode;
    ra.sts = b->sts;
    ra.hidden = g.hidden;
    ra.vocab = g.vocab;
    ra.mask_id = g.vocab - 1;
    ra.head_dim = g.head_dim;
    ra.block_max = g.block_max;
    ra.tokens = tokens;
    ra.embed = static_cast<const __nv_bfloat16*>(ctx_weights(b->ctx[0]).embed);
    ra.w0 = ctx_layers(b->ctx[0], target)[0].ln_attn;
    ra.eps = g.rms_eps;
    rope_table(b->ctx[0], &ra.tab_cos, &ra.tab_sin, &ra.tab_rows);
    ra.x = b->x;
    ra.hi = b->hi;
    ra.lo = b->lo;
    ra.rope_cos = b->rcos;
    ra.rope_sin = b->rsin;
    ra.amax = b->amax;
    BTRY(launch_k(batch_rows_kernel, dim3((unsigned)b->R), dim3(256), 0, s, ra));
    return DFLASH_OK;
}

int batch_accept(dflash_batch* b, int mode, const int32_t* draft_ids, int32_t* draft_out, int32_t* tokens_out,
                 int32_t* n_emitted, cudaStream_t s) {
    BatchAcceptArgs aa{};
    aa.mode = mode;
    aa.sts = b->sts;
    aa.amax = b->amax;
    aa.draft_ids = draft_ids;
    aa.draft_out = draft_out;
    aa.tokens_out = tokens_out;
    aa.n_emitted = n_emitted;
    aa.block_max = b->cfg.block_max;
    aa.max_seq = b->cfg.max_seq;
    aa.eos_id = b->cfg.eos_id;
    BTRY(launch_k(batch_accept_kernel, dim3((unsigned)b->S), dim3(32), 0, s, aa));
    return DFLASH_OK;
}

int pending() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return report_error(DFLASH_ERR_CUDA, "a CUDA error was pending before this call: %s", cudaGetErrorString(e));
    return DFLASH_OK;
}

}  // namespace

extern "C" {

size_t dflash_batch_workspace_bytes(const dflash_config* cfg, int32_t S) {
    if (batch_cfg_ok(cfg, S)) return 0;
    const size_t per = dflash_workspace_bytes(cfg);
    if (!per) return 0;
    return (size_t)S * up1k(per) + batch_layout(*cfg, S, sm_count()).total;
}

int dflash_batch_init(const dflash_config* cfg, const dflash_weights* w, int32_t S, void* kv_target,
                      void* kv_draft, void* workspace, size_t workspace_bytes, dflash_batch** out) {
    if (!out || !w || !kv_target || !workspace) return report_error(DFLASH_ERR_ARG, "NULL argument");
    *out = nullptr;
    if (int r = batch_cfg_ok(cfg, S)) return r;
    const dflash_config& g = *cfg;
    if (g.drf_layers > 0 && !kv_draft) return report_error(DFLASH_ERR_ARG, "kv_draft is NULL");
    const size_t need = dflash_batch_workspace_bytes(cfg, S);
    if (!need || workspace_bytes < need)
        return report_error(DFLASH_ERR_ARG, "workspace %zu < %zu", workspace_bytes, need);
    if (int r = pending()) return r;
    const size_t per_ws = up1k(dflash_workspace_bytes(cfg));
    const size_t per_kt = dflash_kv_target_bytes(cfg), per_kd = dflash_kv_draft_bytes(cfg);
    dflash_batch* b = new dflash_batch();
    b->cfg = g;
    b->S = S;
    b->R = 16 * S;
    b->sms = sm_count();
    b->bn = (S > 8 && g.hidden % 256 == 0) ? 256 : 128;
    b->kv_t = static_cast<uint8_t*>(kv_target);
    b->kv_d = static_cast<uint8_t*>(kv_draft);
    auto bail = [&](int r) {
        for (dflash_ctx* c : b->ctx) dflash_destroy(c);
        delete b;
        return r;
    };
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    for (int s = 0; s < S; ++s) {
        dflash_ctx* c = nullptr;
        const int r = dflash_init(cfg, w, b->kv_t + (size_t)s * per_kt,
                                  g.drf_layers > 0 ? b->kv_d + (size_t)s * per_kd : nullptr,
                                  ws + (size_t)s * per_ws, per_ws, &c);
        if (r) return bail(r);
        b->ctx.push_back(c);
    }
    const BatchLayout L = batch_layout(g, S, b->sms);
    uint8_t* bw = ws + (size_t)S * per_ws;
    b->sts = reinterpret_cast<DevState**>(bw + L.sts);
    b->x = reinterpret_cast<float*>(bw + L.x);
    b->hi = bw + L.hi;
    b->lo = bw + L.lo;
    b->ahi = bw + L.ahi;
    b->alo = bw + L.alo;
    b->thi = bw + L.thi;
    b->tlo = bw + L.tlo;
    b->y = reinterpret_cast<float*>(bw + L.y);
    b->q = reinterpret_cast<__half*>(bw + L.q);
    b->rcos = reinterpret_cast<float*>(bw + L.rcos);
    b->rsin = reinterpret_cast<float*>(bw + L.rsin);
    b->amax = reinterpret_cast<unsigned long long*>(bw + L.amax);
    b->part = reinterpret_cast<float*>(bw + L.part);
    b->apart = reinterpret_cast<float*>(bw + L.apart);
    b->err = reinterpret_cast<int*>(bw + L.err);
    std::vector<DevState*> hs(S);
    for (int s = 0; s < S; ++s) hs[s] = ctx_state(b->ctx[s]);
    if (cudaMemcpy(b->sts, hs.data(), S * sizeof(DevState*), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(b->err, 0, 8) != cudaSuccess)
        return bail(report_error(DFLASH_ERR_CUDA, "batch workspace set-up failed"));
    // tensor maps: GEMM inputs (hi/lo planes at the reduction width) and weights
    const int H = g.hidden, qd = g.n_q * g.head_dim, kvd = g.n_kv * g.head_dim, F = g.ffn, R = b->R;
    const int cap = (g.max_seq + 63) / 64 * 64;
    int r = 0;
    auto layer_maps = [&](const dflash_layer& lw, dflash_batch::LayerMaps* M, bool draft) {
        const void* wqkv[3] = {lw.wq, lw.wk, lw.wv};
        const int rqkv[3] = {qd, kvd, kvd};
        int e = dense_maps(&M->qkv, b->hi, b->lo, R, H, wqkv, rqkv, 3);
        const void* wo[1] = {lw.wo};
        const int ro[1] = {H};
        if (!e) e = dense_maps(&M->o, b->hi, b->lo, R, qd, wo, ro, 1);
        const void* wgu[2] = {lw.w_gate, lw.w_up};
        const int rgu[2] = {F, F};
        // the SwiGLU form of the dense GEMM: weight boxes of half a tile
        if (!e) e = dense_maps(&M->gu, b->hi, b->lo, R, H, wgu, rgu, 2, b->bn == 256 ? DT_WBOX : DT_SWBOX);
        const void* wd[1] = {lw.w_down};
        if (!e) e = dense_maps(&M->down, b->ahi, b->alo, R, F, wd, ro, 1);
        if (!e && draft) {
            const void* wkv[2] = {lw.wk, lw.wv};
            const int rkv[2] = {kvd, kvd};
            e = dense_maps(&M->ctxkv, b->hi, b->lo, R, H, wkv, rkv, 2);
        }
        return e;
    };
    const dflash_layer* tl = ctx_layers(b->ctx[0], true);
    const dflash_layer* dl = ctx_layers(b->ctx[0], false);
    b->tl.resize(g.tgt_layers);
    b->dl.resize(g.drf_layers);
    for (int l = 0; l < g.tgt_layers && !r; ++l) r = layer_maps(tl[l], &b->tl[l], false);
    for (int l = 0; l < g.drf_layers && !r; ++l) r = layer_maps(dl[l], &b->dl[l], true);
    const dflash_weights& wt = ctx_weights(b->ctx[0]);
    if (!r) {
        const void* we[1] = {wt.embed};
        const int rv[1] = {g.vocab};
        r = dense_maps(&b->lm, b->hi, b->lo, R, H, we, rv, 1);
    }
    if (!r && g.drf_layers > 0) {
        const void* wf[1] = {wt.fc};
        const int rf[1] = {H};
        r = dense_maps(&b->fc, b->thi, b->tlo, R, g.n_taps * H, wf, rf, 1);
    }
    const void* gw = nullptr;
    int grows = 0;
    if (!r && g.drf_layers > 0 && ctx_grouped_ctxkv(b->ctx[0], &gw, &b->ctxkv_knorm, &grows)) {
        const void* wk[1] = {gw};
        const int rk[1] = {grows};
        r = dense_maps(&b->ctxkv_all, b->hi, b->lo, R, H, wk, rk, 1);
        b->grouped_ctxkv = !r;
    }
    const int group_rows = (g.n_q / g.n_kv) * 16;
    if (!r)
        r = encode_map(&b->qmap, b->q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim, (uint64_t)R * g.n_q, 64,
                       group_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r)
        r = encode_map(&b->kvmap_t, b->kv_t, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                       (uint64_t)S * g.tgt_layers * 2 * g.n_kv * cap, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r && g.drf_layers > 0)
        r = encode_map(&b->kvmap_d, b->kv_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.head_dim,
                       (uint64_t)S * g.drf_layers * 2 * g.n_kv * cap, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r) return bail(r);
    *out = b;
    return DFLASH_OK;
}

dflash_ctx* dflash_batch_context(dflash_batch* b, int32_t s) {
    if (!b || s < 0 || s >= b->S) {
        report_error(DFLASH_ERR_ARG, "no sequence %d", s);
        return nullptr;
    }
    return b->ctx[s];
}

int dflash_batch_set_logits_out(dflash_batch* b, float* verify_logits, float* draft_logits) {
    if (!b) return report_error(DFLASH_ERR_ARG, "batch is NULL");
    b->verify_logits = verify_logits;
    b->draft_logits = draft_logits;
    return DFLASH_OK;
}

int dflash_batch_draft(dflash_batch* b, int32_t* draft_ids, dflash_stream_t stream) {
    if (!b || !draft_ids) return report_error(DFLASH_ERR_ARG, "NULL argument");
    if (b->cfg.drf_layers == 0) return report_error(DFLASH_ERR_STATE, "no drafter configured");
    if (int r = pending()) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int r = batch_rows(b, FWD_DRAFT, nullptr, false, s);
    if (!r) r = batch_layers(b, false, s);
    if (!r) r = dense(b, b->lm, b->cfg.vocab, b->cfg.hidden, 1 << 30, 1 << 30, b->draft_logits, b->amax, s);
    if (!r) r = batch_accept(b, FWD_DRAFT, nullptr, draft_ids, nullptr, nullptr, s);
    return r;
}

int dflash_batch_verify_accept(dflash_batch* b, const int32_t* draft_ids, int32_t* tokens_out,
                               int32_t* n_emitted, dflash_stream_t stream) {
    if (!b || !tokens_out || !n_emitted) return report_error(DFLASH_ERR_ARG, "NULL argument");
    if (int r = pending()) return r;
    const dflash_config& g = b->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int mode = draft_ids ? FWD_VERIFY : FWD_GREEDY;
    int r = batch_rows(b, mode, draft_ids, true, s);
    if (!r) r = batch_layers(b, true, s);
    if (!r) r = dense(b, b->lm, g.vocab, g.hidden, 1 << 30, 1 << 30, b->verify_logits, b->amax, s);
    if (!r) r = batch_accept(b, mode, draft_ids, nullptr, tokens_out, n_emitted, s);
    if (r || g.drf_layers == 0) return r;
    // tap commit: fc over the verify rows' taps, context norm, then every
    // draft layer's context K/V of each sequence's committed rows
    const int H = g.hidden, kvd = g.n_kv * g.head_dim;
    if ((r = dense(b, b->fc, H, g.n_taps * H, 1 << 30, 1 << 30, b->y, nullptr, s))) return r;
    CtxRowsArgs cr{};
    cr.y = b->y;
    cr.rows = b->R;
    cr.hidden = H;
    cr.w = ctx_weights(b->ctx[0]).ctx_norm;
    cr.norm = g.ctx_norm;
    cr.eps = g.rms_eps;
    cr.c_hi = b->hi;
    cr.c_lo = b->lo;
    BTRY(launch_ctx_rows(cr, s));
    const dflash_layer* dl = ctx_layers(b->ctx[0], false);
    const int cap = (g.max_seq + 63) / 64 * 64;
    BatchCtxKvArgs ca{};
    ca.y = b->y;
    ca.sts = b->sts;
    ca.rows = b->R;
    ca.n_kv = g.n_kv;
    ca.head_dim = g.head_dim;
    ca.cap = cap;
    ca.max_seq = g.max_seq;
    ca.eps = g.rms_eps;
    ca.rope_cos = b->rcos;
    ca.rope_sin = b->rsin;
    ca.cache = reinterpret_cast<__half*>(b->kv_d);
    ca.n_layers = g.drf_layers;
    if (b->grouped_ctxkv) {   // every layer in one GEMM over the first context's grouped weights
        const int kv_all = g.drf_layers * 2 * kvd;
        if ((r = dense(b, b->ctxkv_all, kv_all, H, 1 << 30, 1 << 30, b->y, nullptr, s))) return r;
        ca.k_norm = b->ctxkv_knorm;
        ca.layer0 = 0;
        ca.nl = g.drf_layers;
        BTRY(launch_warps(batch_ctx_kv_kernel, (long long)b->R * g.drf_layers * g.n_kv * 2, s, ca));
        return DFLASH_OK;
    }
    for (int l = 0; l < g.drf_layers; ++l) {
        if ((r = dense(b, b->dl[l].ctxkv, 2 * kvd, H, kvd, 1 << 30, b->y, nullptr, s))) return r;
        ca.k_norm = dl[l].k_norm;
        ca.layer0 = l;
        ca.nl = 1;
        BTRY(launch_warps(batch_ctx_kv_kernel, (long long)b->R * g.n_kv * 2, s, ca));
    }
    return DFLASH_OK;
}

int dflash_batch_check(dflash_batch* b, dflash_stream_t stream) {
    if (!b) return report_error(DFLASH_ERR_ARG, "batch is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return report_error(DFLASH_ERR_CUDA, "stream: %s", cudaGetErrorString(cudaGetLastError()));
    int e[2] = {0, 0};
    if (cudaMemcpy(e, b->err, sizeof e, cudaMemcpyDeviceToHost) != cudaSuccess)
        return report_error(DFLASH_ERR_CUDA, "error word read failed");
    if (e[0]) {
        const int zero[2] = {0, 0};
        cudaMemcpy(b->err, zero, sizeof zero, cudaMemcpyHostToDevice);
        return report_error(e[0] == DERR_TIMEOUT ? DFLASH_ERR_TIMEOUT : DFLASH_ERR_DEVICE,
                            "batch GEMM error %d (site %d)", e[0], e[1]);
    }
    for (dflash_ctx* c : b->ctx)
        if (int r = dflash_check(c, stream)) return r;
    return DFLASH_OK;
}

void dflash_batch_destroy(dflash_batch* b) {
    if (!b) return;
    for (dflash_ctx* c : b->ctx) dflash_destroy(c);
    delete b;
}

}  // extern "C"
