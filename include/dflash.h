/*
 * dflash.h -- C ABI of the GB300 (sm_103a) DFlash block-diffusion
 * speculative-decoding round.
 *
 * One round: (1) tap ingest -- target hidden-state taps are hc-mean-reduced,
 * concatenated and fc-projected into the drafter's context K/V; (2) draft --
 * one drafter forward over the masked block [t_n, MASK x (bl-1)] attending
 * over [sliding context | bidirectional block], ending in an LM-head argmax;
 * (3) verify -- one batched target forward over the 1+m rows
 * [t_n, d_1..d_m]; (4) accept -- greedy first-mismatch acceptance, then the
 * target KV positions and the draft context are rolled back to match.
 *
 * Sources: "[RFC] DFlash" (ExecuTorch PR #20840): "DFlash Overview", "Key
 * Implementation Details" (Phase 1 taps, Phase 3 draft / verify /
 * first-mismatch acceptance / KV-cache position rollback), review
 * "Requested changes" 1 (dynamic block length), 3 (persistent draft KV
 * cache) and 6 (acceptance cases); "feat: DFlash2 block-diffusion drafter
 * for Qwen 3.8" (Mference PR #22): block attention over [sliding ctx |
 * bidirectional block], fp32 residual stream, tap staging, config guards
 * that fire before any buffer is built; "dflash: the chain verify builds
 * pipelined ..." (mlx-serve PR #937), first commit: hc-stream mean taps.
 *
 * Memory.  The library allocates nothing.  Weights, both KV caches and one
 * workspace are caller-owned device buffers (PyTorch tensors in the Python
 * binding) that the caller keeps alive until dflash_destroy().  Every
 * pointer is a DEVICE pointer unless marked (host).  Sizes come from
 * dflash_workspace_bytes / dflash_kv_target_bytes / dflash_kv_draft_bytes.
 *
 * Streams.  Every call enqueues work on the given stream and returns without
 * synchronising, except dflash_stats() and dflash_check(), which synchronise
 * that stream.  The round's state (positions, next token, block length,
 * budget, statistics) lives in device memory, so a round needs no host
 * round-trip and the launches of a round can be captured in a CUDA graph.
 * Calls on one context must not overlap on the GPU (one stream per context).
 * Every kernel is launched with programmatic dependent launch: it may be
 * scheduled while its predecessor drains and waits for it only before
 * touching memory the predecessor writes.  Environment DFLASH_PDL=0, read
 * once when the library loads, launches every kernel plainly instead (same
 * results; a latency study switch).
 *
 * Errors.  Every int-returning call returns DFLASH_OK (0) or a negative
 * DFLASH_ERR_* code and never aborts; dflash_last_error() gives a message
 * (thread-local).  Kernels never trap: an impossible index or an expired
 * bounded wait sets a device error word that dflash_check() reports.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dflash_stream_t; /* a cudaStream_t; NULL = legacy default */

enum {
    DFLASH_OK = 0,
    DFLASH_ERR_CONFIG = -1,   /* shape/format mismatch, rejected before any write */
    DFLASH_ERR_CAPACITY = -2, /* max_seq / draft context capacity exceeded */
    DFLASH_ERR_ARG = -3,      /* null pointer, size out of range, misaligned buffer */
    DFLASH_ERR_CUDA = -4,     /* a CUDA runtime/driver call or launch failed */
    DFLASH_ERR_DEVICE = -5,   /* a kernel set the device error word */
    DFLASH_ERR_TIMEOUT = -6,  /* a kernel's bounded wait expired */
    DFLASH_ERR_STATE = -7     /* call out of order (e.g. verify before prefill) */
};

enum { DFLASH_F32 = 0, DFLASH_BF16 = 1, DFLASH_INT4G64 = 2 };

#define DFLASH_MAX_TAPS 8
#define DFLASH_MAX_BLOCK 16

/* Model and run configuration (Qwen3-shaped target and drafter). */
typedef struct {
    int32_t hidden, n_q, n_kv, head_dim, ffn, vocab;   /* n_q a multiple of n_kv; with
                        * dtype BF16 at most 4 q heads per kv head (one warp of the
                        * tensor-core attention per q head), else at most 16 */
    int32_t tgt_layers;                 /* 0 = drafter alone (taps supplied by caller) */
    int32_t drf_layers;                 /* 0 = target alone */
    int32_t n_taps;                     /* tap layers; taps concatenate in this order */
    int32_t tap_layer[DFLASH_MAX_TAPS]; /* strictly increasing target layer indices */
    int32_t block_max;                  /* native block B, 1..16 */
    int32_t window;                     /* drafter context window W; 0 = whole context */
    int32_t max_seq;                    /* positions held by both caches */
    int32_t eos_id;                     /* -1 = no EOS */
    int32_t dtype;     /* DFLASH_F32 | DFLASH_BF16: embedding, fc, activations; the
                        * caches are fp32 for F32 and fp16 for BF16 */
    int32_t tgt_wfmt;  /* projection format of target layers: F32 | BF16 | INT4G64 */
    int32_t drf_wfmt;  /* projection format of draft layers: F32 | BF16 | INT4G64 */
    int32_t ctx_norm;  /* 1 = RMSNorm after fc (drafter context) */
    float rms_eps, rope_theta;
    int32_t lm_wfmt;   /* LM head: 0 = the embedding itself (tied); INT4G64 = a
                        * group-64 INT4 copy of it (dtype BF16 only; "[RFC] DFlash",
                        * "Test Plan": target and drafter both run 4-bit) */
    int32_t adaptive_block; /* 1: cap each round's block from recent acceptance:
                        * ema <- ema/2 + a/2 (a = drafts accepted, fp32, from
                        * block_max - 1), next block <= 4 rows if ema < 1.5, <= 8 if
                        * ema < 4.5, else block_max (the round policy of "dflash: the
                        * chain verify builds pipelined ...", first commit) */
} dflash_config;

/*
 * One decoder layer.  Projections use the nn.Linear layout [out][in].
 *   F32/BF16: element type as the format says.
 *   INT4G64 : packed [out][in/2] bytes read as little-endian 32-bit words,
 *             each holding 8 consecutive inputs k0..k0+7 interleaved:
 *             input k0+2j in nibble j, k0+2j+1 in nibble j+4 (j = 0..3);
 *             code = nibble - 8; the scale pointer (s*) is bf16 [in/64][out]
 *             (group-major); weight = code * scale.  Produced by
 *             dflash_quantize_int4g64().  The interleave lets one AND/OR per
 *             pair of nibbles build a bf16 pair of adjacent inputs.
 * Norm weights are fp32: ln_attn/ln_mlp [hidden], q_norm/k_norm [head_dim].
 * All matrices must be 16-byte aligned with rows a multiple of 16 bytes.
 */
typedef struct {
    const void *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
    const void *sq, *sk, *sv, *so, *s_gate, *s_up, *s_down;
    const float *ln_attn, *ln_mlp, *q_norm, *k_norm;
} dflash_layer;

typedef struct {
    const void* embed;            /* [vocab][hidden] dtype; also the tied LM head */
    const float* final_norm_tgt;  /* [hidden] */
    const float* final_norm_drf;  /* [hidden] */
    const void* fc;               /* [hidden][n_taps*hidden] dtype */
    const float* ctx_norm;        /* [hidden] */
    const dflash_layer* tgt;      /* (host) array [tgt_layers], copied by dflash_init */
    const dflash_layer* drf;      /* (host) array [drf_layers], copied by dflash_init */
    const void* lm_head;          /* lm_wfmt INT4G64: packed [vocab][hidden/2] of the
                                   * embedding (dflash_quantize_int4g64); else NULL */
    const void* lm_scales;        /* lm_wfmt INT4G64: bf16 [hidden/64][vocab]; else NULL */
} dflash_weights;

/* Round counters kept on the device (per-draft-position accept profile). */
typedef struct {
    int64_t rounds;                      /* verify_accept calls that emitted */
    int64_t emitted;                     /* tokens emitted by them */
    int64_t accept_hist[DFLASH_MAX_BLOCK]; /* [j]: rounds in which draft j+1 was accepted */
    int32_t n;          /* target KV length = position of the pending token */
    int32_t t_n;        /* pending token (emitted, not yet forwarded) */
    int32_t block_len;  /* block length of the next round */
    int32_t generated;  /* tokens emitted so far, the prefill's first included */
    int32_t max_new;    /* generation budget */
    int32_t ctx_len;    /* committed draft context rows */
    int32_t finished;   /* EOS or budget reached */
    int32_t last_accept;/* a of the last round (accepted length - 1) */
    int32_t device_error;
    int32_t pad_;
} dflash_stats_t;

typedef struct dflash_ctx dflash_ctx;

/* Bytes of the caller-owned buffers for a configuration (0 if invalid). */
size_t dflash_workspace_bytes(const dflash_config* cfg /*host*/);
/* Target KV cache: [tgt_layers][2][n_kv][cap][head_dim], cap = max_seq
 * rounded up to a multiple of 64 (whole attention chunks); elements fp32
 * when dtype is F32, fp16 (IEEE binary16) when dtype is BF16. */
size_t dflash_kv_target_bytes(const dflash_config* cfg /*host*/);
/* Draft context K/V: [drf_layers][2][n_kv][cap][head_dim] (elements as the
 * target cache), indexed
 * by absolute position (a persistent cache bounded by max_seq:
 * "[RFC] DFlash", "Requested changes" 3 and the reply "3. Draft KV cache"). */
size_t dflash_kv_draft_bytes(const dflash_config* cfg /*host*/);

/*
 * Validates cfg against the weights (hidden size, vocab, tap layers, formats,
 * divisibility) BEFORE touching any buffer ("feat: DFlash2 ..." commit: the
 * config guard fires before any buffer is built), builds the TMA
 * descriptors, zeroes the workspace's counters on the legacy stream and
 * returns a context in *out (host).  Borrowed buffers must outlive it.
 * With a bf16 model whose drafter has more than one layer it also copies
 * every draft layer's W_k, W_v (INT4: codes and scales) and k_norm into the
 * workspace: the tap commit projects
 * the committed context rows for all layers in one GEMM over that copy, so
 * a change to those weights after dflash_init reaches the drafter's own
 * forwards but not its context rows (make a new context instead).
 * Environment DFLASH_CTXKV_GROUP=0 at init runs one context K/V GEMM per
 * draft layer instead (the same rows to fp32 summation order).
 *
 * Ordering: the calls on one context must be ordered on the GPU (one stream,
 * or streams joined by events); they share the workspace.  The kernels also
 * expect the device to themselves: inside a GEMM or attention launch some
 * CTAs wait for others of the same launch, so kernels of another context or
 * stream running at the same time on the same GPU can hold the SMs those
 * waits need.  Every such wait is bounded: contention ends in
 * DFLASH_ERR_TIMEOUT from dflash_check (which also resets the counters),
 * never in a hang.
 */
int dflash_init(const dflash_config* cfg /*host*/, const dflash_weights* w /*host*/,
                void* kv_target, void* kv_draft, void* workspace, size_t workspace_bytes,
                dflash_ctx** out /*host*/);

/*
 * Starts a generation.
 * Target mode (tgt_layers > 0): prompt_ids [n_prompt] int32 (device) run
 *   through the target; K/V fill the target cache, tap rows of the trailing
 *   context window are fc-projected into the draft context ("feat: DFlash2
 *   ...": prefill stages the prompt's trailing window of tap rows), the
 *   argmax of the last row is the first generated token.  With a bf16 or
 *   INT4 target every prompt row runs as a dense forward (tcgen05 GEMMs
 *   over up to 1024 rows at a time; INT4 matrices dequantised exactly to
 *   f16 layer by layer; environment DFLASH_DENSE_PREFILL=0 at dflash_init
 *   runs 16-row chunks instead), and the rows of the last 16-row chunk go
 *   through the final norm into the round's LM head.
 * Drafter-alone mode (tgt_layers == 0): ext_taps holds n_ext tap rows as
 *   dtype [n_taps][n_ext][hc*hidden] (hc streams per tap layer, reduced by
 *   their mean); rows are positions 0..n_ext-1 and first_token is the pending
 *   token at position n_ext.  With a bf16 or INT4 drafter the window's rows
 *   are ingested on the dense tcgen05 GEMM, hc > 1 streams reduced to their
 *   mean as bf16 hi/lo rows first (DFLASH_DENSE_INGEST=0 at dflash_init:
 *   16-row chunks).
 * max_new is the generation budget (the first token counts).  Errors:
 * ARG, CAPACITY (n_prompt or n_ext + block > max_seq), STATE.
 */
int dflash_prefill_taps(dflash_ctx* ctx, const int32_t* prompt_ids, int32_t n_prompt,
                        const void* ext_taps, int32_t n_ext, int32_t hc, int32_t first_token,
                        int32_t max_new, dflash_stream_t stream);

/*
 * Adopts caches the caller filled itself (e.g. by another prefill engine):
 * the target cache, and the draft context cache if a drafter is configured,
 * hold positions [0, n) in the layouts above; the generation continues from
 * pending_token at position n with budget max_new (that token counts), as
 * dflash_prefill_taps would leave it.  Errors: CAPACITY (n + 1 > max_seq),
 * ARG.
 */
int dflash_adopt_kv(dflash_ctx* ctx, int32_t n, int32_t pending_token, int32_t max_new,
                    dflash_stream_t stream);

/*
 * One drafter forward over the block of the device-held length bl at
 * positions n..n+bl-1; writes draft_ids [block_max-1] int32 (entries
 * >= bl-1 are -1).  bl <= 1 drafts nothing ("[RFC] DFlash", "Requested
 * changes" 1: a one-token round is a target-only step).
 */
int dflash_draft_block(dflash_ctx* ctx, int32_t* draft_ids, dflash_stream_t stream);

/*
 * Verifies [t_n, draft_ids[0..bl-2]] in one target forward (draft_ids NULL:
 * plain greedy step, one row), accepts the first-mismatch prefix plus the
 * bonus token (EOS-truncated), writes tokens_out [block_max] (unused = -1)
 * and *n_emitted, rolls the target KV length to n + n_emitted, commits the
 * accepted rows' taps to the draft context and sets the next block length
 * min(B, max_new - generated, max_seq - n).  A finished context emits 0.
 */
int dflash_verify_accept(dflash_ctx* ctx, const int32_t* draft_ids, int32_t* tokens_out,
                         int32_t* n_emitted, dflash_stream_t stream);

/*
 * Rewinds the target KV length and the draft context to new_len (host),
 * 1 <= new_len <= current length; the pending token becomes
 * token_at_new_len (host).  Nothing is moved: positions >= new_len are
 * overwritten by later rounds.  ("[RFC] DFlash", "Key Implementation
 * Details": KV-cache position rollback; "feat: DFlash2 ...": continuity
 * breaks reset the drafter with positions realigned.)
 */
int dflash_rollback(dflash_ctx* ctx, int64_t new_len, int32_t token_at_new_len,
                    dflash_stream_t stream);

/* Copies the device counters and state to *out (host); synchronises stream. */
int dflash_stats(dflash_ctx* ctx, dflash_stats_t* out, dflash_stream_t stream);

/* Synchronises stream; returns DEVICE or TIMEOUT if a kernel flagged an
 * error since the last check (and clears the flag), else OK.  After TIMEOUT
 * the split-K tickets may be inconsistent: re-create the context. */
int dflash_check(dflash_ctx* ctx, dflash_stream_t stream);

/*
 * Enqueues a copy of the round state's progress words into out (device,
 * int32[4]): finished (nonzero once the generation is done), tokens
 * generated (the prefill's first included), KV length n, tokens emitted by
 * rounds.  No synchronisation, so a host loop can run many rounds from a
 * CUDA graph and read the progress once per replay (the host builds while
 * the GPU runs: "dflash: the chain verify builds pipelined ...", the chain
 * verify commit).  Errors: ARG.
 */
int dflash_progress(dflash_ctx* ctx, int32_t* out, dflash_stream_t stream);

/*
 * The attention form a context's forwards run for the target (model 0) or
 * the drafter (model 1), fixed at dflash_init from the configuration and
 * the device: 2 = split-KV on the fifth-generation tensor cores (tcgen05),
 * splits of one 64-key chunk; 1 = split-KV on mma.sync tensor cores, splits
 * of several chunks; 0 = the separate partial and combine kernels (fp32
 * models, and bf16 ones whose splits do not fit the device at once).  Form
 * 2 is opt-in: environment
 * DFLASH_ATTN_TC=1 at init (on the 16-row round it measured slower than
 * form 1).  No counterpart in the pages: an implementation choice
 * of this library.  Returns the form, or ARG for a NULL context or a model
 * other than 0 and 1.
 */
int dflash_attention_form(const dflash_ctx* ctx, int32_t model);

/* Self-test of the kernels' bounded waits: launches one warp that waits on
 * an mbarrier nothing arrives on, gives up after limit_ns (<= 2 s) and sets
 * the device error word, so that the next dflash_check returns TIMEOUT. */
int dflash_selftest_timeout(dflash_ctx* ctx, int64_t limit_ns, dflash_stream_t stream);

/*
 * Parity taps: while set (non-NULL), every target LM head (verify, and the
 * last prefill chunk) writes its fp32 logits [16][vocab] to verify_logits
 * (row i = forward row i) and every draft writes [16][vocab] to draft_logits
 * (row j = block row j); rows past the forward's length hold padding.
 * Costs one extra write of the logits; NULL switches it off.
 */
int dflash_set_logits_out(dflash_ctx* ctx, float* verify_logits, float* draft_logits);

/*
 * Kernel timing of the dominant kernel family (the weight-streaming GEMM).
 * mode 1: start -- every later GEMM launch of this context is bracketed by
 *   two CUDA events recorded on its stream (up to 1 << 15 launches; events
 *   recorded during stream capture become event nodes of the graph, so a
 *   captured round keeps timing itself on every replay);
 * mode 2: read -- synchronise the bracketed events and sum them into *out;
 * mode 0: read and stop.
 * gemm_bytes counts algorithmic bytes: weights, the 16 activation rows read
 * and the outputs written; gemm_weight_bytes the weights alone.
 */
typedef struct {
    int64_t gemm_launches;
    double gemm_ms;
    double gemm_bytes;
    double gemm_weight_bytes;
} dflash_profile_t;

int dflash_profile(dflash_ctx* ctx, int32_t mode, dflash_profile_t* out /*host*/);

/* Kernels launched by this process through the library so far. */
int64_t dflash_launch_count(void);

void dflash_destroy(dflash_ctx* ctx);
const char* dflash_last_error(void);

/* ---- several sequences in lockstep rounds ----------------------------- */

/*
 * A batch of S independent sequences (1 <= S <= 32) that share one model:
 * each sequence is a context of its own (round state, target and draft
 * caches, block length, budget, statistics), and a batched round runs one
 * drafter forward and one target forward over every sequence's rows at
 * once, so the weights stream once for all of them.  The pages verify one
 * sequence's [1, 1 + m] rows per forward ("[RFC] DFlash", "Key
 * Implementation Details", Phase 3) and note that the verify's cost follows
 * its row count ("Performance"); batching sequences is this library's
 * extension: every sequence's state moves exactly as dflash_draft_block /
 * dflash_verify_accept would move it, and its tokens are its own
 * single-sequence decode.  Sequence s owns rows 16 s .. 16 s + 15 of each
 * forward; the 16 S-row GEMMs run on the dense tcgen05 GEMM (bf16 hi/lo
 * activation planes, k-splits chosen from N and K only, 128-column tiles up
 * to 8 sequences and 256 above, which leaves each output's sum over k
 * unchanged), so a sequence's results do not depend on S.  bf16 models only (dtype, target, drafter and
 * the tied LM head bf16); head_dim 64 or 128.
 *
 * Memory (caller-owned, device): kv_target holds S consecutive target
 * caches of dflash_kv_target_bytes(cfg) each, kv_draft S draft caches of
 * dflash_kv_draft_bytes(cfg); workspace (dflash_batch_workspace_bytes, zero
 * not required) holds the S contexts' workspaces and the batch's own rows.
 * Errors: CONFIG (a configuration the batched round does not run), ARG,
 * CUDA.
 */
typedef struct dflash_batch dflash_batch;
size_t dflash_batch_workspace_bytes(const dflash_config* cfg /*host*/, int32_t S);
int dflash_batch_init(const dflash_config* cfg /*host*/, const dflash_weights* w /*host*/, int32_t S,
                      void* kv_target, void* kv_draft, void* workspace, size_t workspace_bytes,
                      dflash_batch** out /*host*/);
/* Sequence s's context, owned by the batch: start it with
 * dflash_prefill_taps (or dflash_adopt_kv), read it with dflash_stats, roll
 * it back with dflash_rollback, as any context; every such call must be
 * ordered with the batch's calls on the GPU.  NULL for s outside [0, S). */
dflash_ctx* dflash_batch_context(dflash_batch* b, int32_t s);
/* One drafter forward over every sequence's block (its device-held block
 * length, [t_n, MASK...] at its positions), writing draft_ids [S][block_max-1]
 * int32 (sequence s's ids at s * (block_max - 1); entries past its block -1). */
int dflash_batch_draft(dflash_batch* b, int32_t* draft_ids, dflash_stream_t stream);
/* One target forward over every sequence's [t_n, d_1..d_{bl-1}] (draft_ids
 * [S][block_max-1]; NULL: a one-row greedy step each), then per sequence the
 * first-mismatch acceptance, KV rollback and the commit of its accepted
 * rows' taps to its draft context: tokens_out [S][block_max] (unused -1),
 * n_emitted [S].  Finished sequences emit 0. */
int dflash_batch_verify_accept(dflash_batch* b, const int32_t* draft_ids, int32_t* tokens_out,
                               int32_t* n_emitted, dflash_stream_t stream);
/* Parity taps of the batched forwards: fp32 logits [16 S][vocab] (row
 * 16 s + t = sequence s's forward row t; rows past its T hold padding) of
 * every verify / draft while set; NULL switches it off. */
int dflash_batch_set_logits_out(dflash_batch* b, float* verify_logits, float* draft_logits);
/* Synchronises stream; reports a bounded wait of a batched GEMM that ran out
 * (TIMEOUT) or the first sequence context whose error word is set (as
 * dflash_check), clearing what it reports. */
int dflash_batch_check(dflash_batch* b, dflash_stream_t stream);
void dflash_batch_destroy(dflash_batch* b);

/* ---- standalone operations ------------------------------------------- */

/*
 * hc-stream tap reduce ("dflash: the chain verify builds pipelined ...",
 * first commit: per-token mean of the hyper-connection streams,
 * unflatten(-1, (hc, hidden)).mean(-2)): layer_streams[i] (host array of
 * n_layers device pointers) is bf16 [rows][hc*hidden] with stream s at
 * columns s*hidden..; out is fp32 [rows][n_layers*hidden], tap layer i at
 * columns i*hidden...  Streams are summed in order s = 0..hc-1 in fp32,
 * then multiplied by 1/hc.  hidden must be a multiple of 8.
 */
int dflash_tap_reduce(const void* const* layer_streams /*host array*/, int32_t n_layers,
                      int32_t rows, int32_t hc, int32_t hidden, float* out,
                      dflash_stream_t stream);

/*
 * INT4 group-64 quantiser (the INT4G64 format above) of w fp32 [n][k]:
 * per group of 64 consecutive k of one row, s = bf16(absmax / 7) (round to
 * nearest even), code = clamp(rint(w / s), -8, 7) (0 where s == 0).  The
 * scale and the division are fp32.  packed [n][k/2] bytes (interleaved
 * words), scales bf16 [k/64][n].  k must be a multiple of 256.
 */
int dflash_quantize_int4g64(const float* w, int32_t n, int32_t k, uint8_t* packed,
                            uint16_t* scales, dflash_stream_t stream);

/*
 * The round's weight-streaming GEMM as a standalone operation:
 * y[t][j] = sum_k x[t][k] * w[j][k] for the 16 rows t of x, w bf16 [n][k]
 * (nn.Linear layout), x bf16 [16][k] (rows the caller does not use are
 * zero), y fp32 [16][n].  n a multiple of 128, k a multiple of 64; every
 * buffer 16-byte aligned.  The workspace (dflash_linear_workspace_bytes)
 * holds the split-K partial tiles and tickets, then a 256-byte state block;
 * zero-fill it before its first use (every completed call leaves the
 * tickets at zero again); calls sharing a workspace must not overlap on the
 * GPU.  The result of a row depends only on that row (fixed reduction
 * order).
 * err: device int32[2].  The call clears the state's error words, and
 * after the GEMM copies them into err on the stream: {0, 0} when the GEMM
 * completed; {1, site} when one of its bounded waits ran out (2 s; the
 * owner of a split tile waiting for the other parts is site 105), in which
 * case y is incomplete and the workspace's tickets may be left nonzero --
 * zero-fill it again before the next call.  Read err after synchronising
 * the stream: the call itself returns DFLASH_OK once the work is enqueued.
 * Errors (returned): ARG, CUDA.
 */
size_t dflash_linear_workspace_bytes(int32_t n, int32_t k);
int dflash_linear(const void* w, const void* x, int32_t n, int32_t k, float* y, void* workspace,
                  size_t workspace_bytes, int32_t* err, dflash_stream_t stream);

/*
 * dflash_linear without a workspace, for callers that cannot allocate
 * device memory: code that runs inside a host framework whose allocator
 * owns the device memory, or in a latency-critical loop where cudaMalloc /
 * cudaFree would synchronise the device.  No counterpart in the paper: the
 * method itself has no such operation; this is a library convenience.
 *
 * Same operands, layout and result as dflash_linear (the same kernel and
 * launch shape), with n at most 262144 output columns; larger n returns
 * DFLASH_ERR_ARG before anything is launched.  The split-K scratch is one
 * fixed 4 MiB + 9 KiB array in the library's device memory, held by every
 * GPU that loads the library until the process exits.  The first call on a
 * device looks up that array's device address (with the device current);
 * make that first call before any stream capture, and make no call on a
 * device after a cudaDeviceReset of it (the address belongs to the module
 * loaded before the reset).  Every call on a device shares the array: each
 * clears the tickets and error words it needs on its stream first, but
 * calls that overlap on the GPU (unordered streams) race and may return
 * wrong results.  err (device int32[2], 8-byte aligned) receives the
 * GEMM's error words as in dflash_linear: {0, 0}, or {1, site} when a
 * bounded wait ran out and y is incomplete; read it after synchronising the
 * stream.  The call allocates nothing.
 */
int dflash_linear_noalloc(const void* w, const void* x, int32_t n, int32_t k, float* y,
                          int32_t* err, dflash_stream_t stream);

/*
 * Dense many-row GEMM on the fifth-generation tensor cores (tcgen05, f32
 * accumulators in tensor memory): y[m][j] = sum_i x[m][i] * w[j][i] (+ the
 * same with x_lo) for m < M, j < N.  x bf16 row-major [M][K]; x_lo a second
 * bf16 plane of x added to it (the low part of an fp32 activation split
 * into bf16 hi + lo), or NULL; w bf16 [N][K] (nn.Linear layout); y fp32
 * [M][N].  M >= 1, N >= 1, K a multiple of 64, every pointer 16-byte
 * aligned.  err: device int32[2], zero before the call; a kernel wait that
 * timed out writes 1 and a site number there (kernels never trap).  The library's
 * kernel for the dense steps of the pipeline, where the rows number in the
 * hundreds or thousands: the drafter's context-window ingest (the fc
 * re-projection of the window's tap rows and each draft layer's context
 * K/V, "[RFC] DFlash", "Requested changes" 3, the persistent draft KV
 * cache) and the target's prompt prefill (every projection of the prompt
 * rows).  The binding checks dtypes, shapes
 * and devices before the call.  Errors: ARG, CUDA.
 */
int dflash_linear_dense(const void* w, const void* x, const void* x_lo, int32_t m, int32_t n, int32_t k,
                        float* y, int32_t* err, dflash_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
