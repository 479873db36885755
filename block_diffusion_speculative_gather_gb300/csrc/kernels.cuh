// Launchers of the non-GEMM kernels of the DFlash round.
#pragma once

#include "common.cuh"

namespace dfl {

enum FwdMode : int { FWD_PREFILL = 0, FWD_DRAFT = 1, FWD_VERIFY = 2, FWD_GREEDY = 3 };

constexpr int ATTN_CHUNK = 64;   // keys per attention split (fixed: batch invariance)

struct RowsArgs {
    int mode;
    int hidden, vocab, mask_id;
    int pos0, T;                 // PREFILL only: chunk position and rows
    const int32_t* tokens;       // PREFILL: prompt; VERIFY: draft ids; else unused
    const void* embed;           // [vocab][hidden] (dtype)
    int embed_f32;               // 1 = fp32 embedding, 0 = bf16
    const float* x_src;          // instead of embed: the rows' residual [T][hidden] fp32
                                 // (a dense prefill's last rows, for the final norm)
    float* x;                    // fp32 [16][hidden]
    float* rope_cos;             // [16][head_dim/2]: the forward rows' angles, copied from
    float* rope_sin;             //   the position table below
    int head_dim;
    float rope_theta;
    const float* tab_cos;        // [tab_rows][head_dim/2] cos of every cache position
    const float* tab_sin;        // [tab_rows][head_dim/2] sin
    int tab_rows;
    unsigned long long* amax;    // [16] reset to 0
    // folded input norm of the first layer: xn = x * w0 and partial sums of x^2
    const float* w0;             // [hidden] ln_attn of layer 0 of the model that runs
    void* xn;                    // [16][hidden], xn_type
    int xn_type;
    float* ssq;                  // [hidden / 128][16]
    DevState* st;
};

int launch_prepare_rows(const RowsArgs& a, cudaStream_t s);

struct AttnArgs {
    const void* q;          // [n_q][16][head_dim]
    const void* k_cache;    // layer base [n_kv][cap][head_dim]
    const void* v_cache;
    int kv_type;            // XT_F32 | XT_BF16 (q has the same type)
    int n_q, n_kv, head_dim, cap;
    int causal;             // 1: key pos <= query pos (verify/prefill); 0: draft block
    int window;             // draft: context window (0 = all)
    float scale;
    float* part;            // [max_chunks][16][n_q][head_dim + 2]
    void* out;              // [16][n_q * head_dim], type out_type
    int out_type;
    int max_chunks;
    DevState* st;
};

// CUDA-core split-KV attention (the fp32 path) + the chunk-order combine.
int launch_attention(const AttnArgs& a, cudaStream_t s);
// The combine alone (after the tensor-core partial kernel).
int launch_attention_combine(const AttnArgs& a, cudaStream_t s);

struct AcceptArgs {
    int mode;               // FWD_DRAFT | FWD_VERIFY | FWD_GREEDY | FWD_PREFILL (last chunk)
    const unsigned long long* amax;
    const int32_t* draft_ids;     // VERIFY
    int32_t* draft_out;           // DRAFT: [block_max - 1]
    int32_t* tokens_out;          // VERIFY/GREEDY: [block_max]
    int32_t* n_emitted;
    int block_max, max_seq, eos_id;
    int max_new;                  // PREFILL
    int prompt_len;               // PREFILL
    int window;                   // PREFILL: tap rows committed = trailing window
    DevState* st;
};

int launch_accept(const AcceptArgs& a, cudaStream_t s);

// Prefill bookkeeping: forward descriptor of chunk (pos0, T) and the rows
// of it whose taps are committed to the draft context.
int launch_set_chunk(DevState* st, int pos0, int T, int commit_lo, cudaStream_t s);

int launch_rollback(DevState* st, int new_len, int token, int block_max, int max_seq,
                    cudaStream_t s);

// Drafter-alone prefill: state after n_ext externally supplied tap rows.
int launch_set_ext_state(DevState* st, int n_ext, int first_token, int max_new, int block_max,
                         int max_seq, int eos_id, cudaStream_t s);

struct TapArgs {
    const void* src[8];   // per tap layer: [rows][hc * hidden] (in_type)
    int n_layers, rows, hc, hidden;
    int in_type;          // XT_F32 | XT_BF16
    void* out;            // [rows][n_layers * hidden], out_type
    int out_type;
    long long out_row_stride;   // elements between output rows
    long long lo_offset;        // XT_BF16S: elements from a value to its low part (0: 16 rows below)
};

int launch_tap_reduce(const TapArgs& a, cudaStream_t s);

// Context rows of a window ingest (many rows at once): c = RMSNorm(y) * w
// (or c = y without the norm), y fp32 [rows][hidden], written as bf16 hi
// and lo planes [rows][hidden] (c = hi + lo to 16 bits).
struct CtxRowsArgs {
    const float* y;
    int rows, hidden;
    const float* w;       // [hidden] ctx norm weight; NULL with norm = 0
    int norm;
    float eps;
    void* c_hi;
    void* c_lo;
    int f16;              // 1: the planes are f16 (else bf16)
};
int launch_ctx_rows(const CtxRowsArgs& a, cudaStream_t s);

// ---- dense prompt prefill (many rows at once; the same formulas as the
// round's 16-row kernels and epilogues)

// x[r] = embedding row of tokens[r] (bf16 -> fp32); an id outside [0, vocab)
// sets the error word and gives a zero row.
int launch_embed_rows(const int32_t* tokens, int rows, const void* embed, int hidden, int vocab, float* x,
                      DevState* st, cudaStream_t s);

// x += y (y may be NULL), then RMSNorm(x) * w as bf16 hi/lo planes; with
// tap_hi, x itself (after the add) also goes to tap_hi/tap_lo rows
// [rows][tap_ld] at column tap_col.
struct ResidNormArgs {
    float* x;
    const float* y;       // [rows][hidden], or NULL (no residual add)
    // y_splits > 1: y holds that many split-K partial slabs of a dense GEMM
    // (slab z at y + z * y_slab, rows of `hidden`), summed here in split
    // order 0, 1, ... (the order of the dense GEMM's own reduce)
    int y_splits;
    size_t y_slab;
    int rows, hidden;
    const float* w;
    float eps;
    void* hi;
    void* lo;
    void* tap_hi;
    void* tap_lo;
    long long tap_ld;
    int tap_col;
    int f16;              // 1: hi/lo planes of the norm output are f16 (taps stay bf16)
};
int launch_resid_norm(const ResidNormArgs& a, cudaStream_t s);

// q/k/v rows of a dense forward: y fp32 [rows][(n_q + 2 n_kv) hd] (q heads,
// k heads, v heads) of rows at positions pos0 + r; q gets q-norm and RoPE
// and goes to q_out f16 [rows/16][n_q][16][hd]; k gets k-norm and RoPE, k
// and v go to the layer's cache rows [n_kv][cap][hd] (c_type).
struct QkvRowsArgs {
    const float* y;
    int rows, pos0, n_q, n_kv, head_dim, cap, max_seq;
    const float* q_norm;
    const float* k_norm;
    float eps;
    const float* rope_cos;  // [rows][head_dim / 2]: the rows of the RoPE position table
    const float* rope_sin;
    void* q_out;
    void* k_cache;
    void* v_cache;
    int c_type;
    DevState* st;
};
int launch_qkv_rows(const QkvRowsArgs& a, cudaStream_t s);


// RoPE table of positions pos0 .. pos0 + rows - 1: cos and sin [rows][half]
// of pos * inv_freq[i] (angle reduced and evaluated in double, rounded once
// to fp32): the position table made at init, and a dense pass's rows past
// it.
int launch_rope_rows(int pos0, int rows, int half, const double* inv_freq, float* cos_out, float* sin_out,
                     cudaStream_t s);

// INT4G64 weights [n][k] (packed [n][k/2], scales bf16 [k/64][n]) to f16
// [n][k]: code * scale has at most 11 significant bits, so the f16 value is
// exact (inside f16's normal range).
int launch_dequant_int4g64_f16(const uint8_t* packed, const uint16_t* scales, int n, int k, void* out,
                               cudaStream_t s);

// Context K/V of a window ingest for one draft layer: y fp32 [rows][2 n_kv
// hd] (K heads, then V heads) of rows at positions pos0 + r; K gets the
// per-head k RMSNorm and RoPE at its position, both go to the layer's cache
// rows ([n_kv][cap][hd], c_type) as the round's q/k/v epilogue writes them.
struct CtxKvArgs {
    const float* y;
    int rows, pos0, n_kv, head_dim, cap, max_seq;
    const float* k_norm;    // [head_dim]
    float eps;
    const float* rope_cos;  // [rows][head_dim / 2]: the rows of the RoPE position table
    const float* rope_sin;
    void* k_cache;
    void* v_cache;
    int c_type;
    DevState* st;
};
int launch_ctx_kv_store(const CtxKvArgs& a, cudaStream_t s);

int launch_selftest_wait(DevState* st, unsigned long long limit_ns, cudaStream_t s);

int launch_progress(const DevState* st, int32_t* out, cudaStream_t s);

int launch_quantize_int4g64(const float* w, int n, int k, uint8_t* packed, uint16_t* scales,
                            cudaStream_t s);

}  // namespace dfl
