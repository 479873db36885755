// Skinny GEMM of the DFlash path: Y[t][n] = sum_k X[t][k] * W[n][k] for the
// <= 16 rows t of one forward (draft block, verify batch or prefill chunk),
// streaming the weight matrix W once from HBM.
#pragma once

#include "common.cuh"

namespace dfl {

enum WFmt : int { WF_F32 = 0, WF_BF16 = 1, WF_INT4 = 2 };
// Epilogues.  The RMSNorm that precedes a projection is folded into the
// GEMMs around it: the producer of a normalised input (RESID, NORMOUT, the
// row-preparation kernel) writes x * w_norm rounded to the GEMM input type
// plus per-128-column partial sums of x^2; the consumer (QKV, SWIGLU,
// ARGMAX) scales its rows by rstd = 1 / sqrt(sum / width + eps).
enum Epi : int {
    EPI_STORE = 0,    // fp32 store
    EPI_RESID = 1,    // x += Y; next normalised input (+ partial sums) and tap copy
    EPI_SWIGLU = 2,   // silu(rstd * gate) * (rstd * up) of paired tiles
    EPI_ARGMAX = 3,   // LM head: rstd-scaled logits, packed argmax (+ optional dump)
    EPI_QKV = 4,      // rstd, per-head q/k RMSNorm, RoPE, q out and K/V into the cache
    EPI_NORMOUT = 5,  // Y * w_norm as the next normalised input (+ partial sums)
};
// Activation element types.  XT_BF16S is a GEMM input kept to about 16
// mantissa bits as two bf16 planes of one [32][ld] buffer: row t holds
// hi = bf16(v) and row 16 + t holds lo = bf16(v - hi); the GEMM multiplies
// both planes by the same weights and sums them in fp32.
enum XType : int { XT_F32 = 0, XT_BF16 = 1, XT_F16 = 2, XT_BF16S = 3 };

// Stores v as element (t, col) of a [rows][ld] activation of type xt (for
// XT_BF16S: the hi plane at row t, the lo plane at row 16 + t).
__device__ __forceinline__ void store_act(void* base, int xt, size_t ld, int t, size_t col, float v) {
    const size_t i = (size_t)t * ld + col;
    if (xt == XT_F32) {
        reinterpret_cast<float*>(base)[i] = v;
    } else if (xt == XT_F16) {
        reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
    } else {
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        reinterpret_cast<__nv_bfloat16*>(base)[i] = hi;
        if (xt == XT_BF16S)
            reinterpret_cast<__nv_bfloat16*>(base)[i + DFL_MAX_ROWS * ld] =
                __float2bfloat16_rn(v - __bfloat162float(hi));
    }
}

constexpr int GEMM_BN = 128;        // output rows (weight rows) per tile
constexpr int GEMM_CONSUMERS = 8;   // MMA warps, 16 weight rows each
constexpr int GEMM_THREADS = (GEMM_CONSUMERS + 1) * 32;
constexpr int GEMM_STAGE_W = GEMM_BN * 128;   // bytes of the weight tile per stage

// Per weight format: a k-block is one 128-byte row of a weight tile; a
// pipeline stage holds CHUNK consecutive k-blocks of one tile, so every
// weight row is fetched CHUNK x 128 contiguous bytes at a time.
//   F32 : 32 k per k-block,  X [16][32] fp32,                1 k-block per stage, 8 stages
//   BF16: 64 k per k-block,  X [32][64] bf16 (hi/lo planes),  3 k-blocks per stage, 3 stages
//   INT4: 256 k per k-block, X 4 x [32][64] bf16, scales [4 groups][128 rows] bf16,
//         2 k-blocks per stage, 3 stages
// (an unsplit bf16 input fills only the 16 hi rows of each X slot)
// Pipeline shape, overridable at build time for tuning sweeps.
#ifndef DFL_BF16_CHUNK
#define DFL_BF16_CHUNK 3
#endif
#ifndef DFL_BF16_STAGES
#define DFL_BF16_STAGES 3
#endif
#ifndef DFL_INT4_CHUNK
#define DFL_INT4_CHUNK 2
#endif
// Ring stages the producer fills with weights before the dependency wait
// (build knob).  Each one streams while the predecessor still runs, but
// those reads also queue ahead of the predecessor's split-tile hand-offs:
// measured on an 8-layer round, 1 stage 1.424 ms, 2 stages 1.431, a full
// ring (3) 1.457.
#ifndef DFL_GEMM_PREWAIT
#define DFL_GEMM_PREWAIT 1
#endif

#ifndef DFL_INT4_STAGES
#define DFL_INT4_STAGES 3
#endif
#ifndef DFL_GEMM_CTAS_PER_SM
#define DFL_GEMM_CTAS_PER_SM 1
#endif
// Register budget: a GEMM CTA sized to share its SM with one more CTA (the
// next kernel's, under programmatic dependent launch) when set to 2.
#ifndef DFL_GEMM_MINBLOCKS
#define DFL_GEMM_MINBLOCKS DFL_GEMM_CTAS_PER_SM
#endif

template <int WF> struct GemmCfg;
template <> struct GemmCfg<0> {
    static constexpr int KBLK = 32, XB = 2048, SB = 0, CHUNK = 1, STAGES = 8;
};
template <> struct GemmCfg<1> {
    static constexpr int KBLK = 64, XB = 4096, SB = 0, CHUNK = DFL_BF16_CHUNK, STAGES = DFL_BF16_STAGES;
};
template <> struct GemmCfg<2> {
    static constexpr int KBLK = 256, XB = 16384, SB = 1024, CHUNK = DFL_INT4_CHUNK,
                         STAGES = DFL_INT4_STAGES;
};

// Per-head epilogue of the q/k/v projection (EPI_QKV).
struct QkvEpi {
    int n_q, n_kv, hd;          // heads in the tile order q.., k.., v..
    const float* q_norm;        // [hd] (unused when n_q == 0)
    const float* k_norm;        // [hd]
    const float* rope_cos;      // [16][hd/2] angles of the forward's rows
    const float* rope_sin;
    void* q_out;                // [n_q][16][hd], q_type
    int q_type;
    void* k_cache;              // layer base [n_kv][cap][hd], c_type
    void* v_cache;
    int c_type;
    int cap, max_seq;
    int row_sel;                // rows written: ROWS_FWD (the forward's) or ROWS_COMMIT
    // group > 1: the weights are `group` consecutive layers' [W_k; W_v]
    // (n_q == 0), tiles in layer order; layer l's rows go to the caches at
    // element offset l * cache_stride with k-norm weights k_norm_all + l * hd
    int group;
    long long cache_stride;
    const float* k_norm_all;    // [group][hd]
};

struct GemmArgs {
    int N;              // output width (SWIGLU: ffn)
    int K;              // reduction length
    int n_tiles;        // tiles of GEMM_BN output rows (SWIGLU: 64 outputs per tile)
    int kb;             // k-blocks per tile
    int seg_rows[3];    // rows of weight maps 0..2 (concatenated along N)
    int n_seg;
    int x_split;        // 1: the activation is XT_BF16S (the x map's box is 32 rows)
    // input row scale of a folded RMSNorm (QKV, SWIGLU, ARGMAX): NULL = 1
    const float* ssq_in;    // [ssq_parts][16] partial sums of x^2
    int ssq_parts;
    float inv_width;        // 1 / normalised width
    float eps;
    // STORE: fp32 [16][ldo];  RESID: the fp32 residual x [16][ldo]
    float* out;
    int ldo;
    // RESID / NORMOUT: next normalised input (x or Y) * w_next as xn_type
    void* xn_out;
    const float* w_next;    // NULL = ones
    float* ssq_out;         // [n_tiles][16], or NULL
    int xn_type;
    // RESID: optional raw copy of the new x (target taps)
    void* tap_out;
    int ld_tap;
    int tap_type;
    // SWIGLU: activation [16][ld_act]
    void* act;
    int ld_act;
    int act_type;
    // ARGMAX
    unsigned long long* amax;  // packed keys [16]
    float* logits;             // optional fp32 dump [16][ldl]
    int ldl;
    // QKV
    QkvEpi qkv;
    // deterministic split-K across CTAs
    float* slots;       // [grid][2][GEMM_BN * 16]
    int* counters;      // [n_tiles], zero between launches
    DevState* st;
};

struct GemmMaps {
    CUtensorMap w[3];   // weight maps (SWIGLU: 0 = gate, 1 = up)
    CUtensorMap s[3];   // INT4 scale maps, one per weight map
    CUtensorMap x;      // activation map
};

// Host: enqueue one GEMM (fmt, epilogue and activation type fixed per call).
// Returns 0 or the cudaError_t of the launch.
int launch_gemm(int wfmt, int epi, int xt, const GemmMaps& maps, const GemmArgs& args,
                int grid, cudaStream_t stream);

// Host helpers of the C ABI (defined with it): record the message returned
// by dflash_last_error and return code; build the bf16 weight and [16][k]
// activation maps of a plain y = x w^T.
int report_error(int code, const char* fmt, ...);
int make_linear_maps(GemmMaps* maps, const void* w, const void* x, int n, int k);
// The standalone y = x w^T (bf16 w [n][k], x [16][k], y fp32 [16][n]) on
// caller-chosen scratch: clears clear_bytes at clear, launches the GEMM on
// sms SMs with its split-K slots, tickets and state at slots / counters /
// st, then copies the state's (code, site) error words into err (device
// int32[2]); all on stream s.
int run_linear_store(const void* w, const void* x, int n, int k, float* y, float* slots,
                     int* counters, DevState* st, void* clear, size_t clear_bytes, int32_t* err,
                     int sms, cudaStream_t s);

}  // namespace dfl
