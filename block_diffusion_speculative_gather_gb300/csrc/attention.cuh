// Tensor-core split-KV attention (fp16 q and caches).
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int ATTN_KEYS = 64;   // keys per chunk; equals the fp32 path's chunk

struct AttnMaps {
    CUtensorMap q;    // q rows [n_q * 16][head_dim] (head-major, 16 rows per head), box = the group
    CUtensorMap kv;   // whole cache [layers * 2 * n_kv * cap][head_dim]
    CUtensorMap q16;  // the q rows again, box = one head's 16 rows
};

struct AttnMmaArgs {
    int n_q, n_kv, head_dim;
    int layer;        // layer index inside the cache map
    int cap;          // positions per (layer, K|V, head) run, a multiple of 64
    int causal, window;
    float scale;
    float* part;      // [max_chunks][16][n_q][head_dim + 2]
    DevState* st;
};

int launch_attention_mma(const AttnMaps& maps, const AttnMmaArgs& a, int max_chunks,
                         cudaStream_t s);

// Split-KV attention with the combine in the same kernel.  CTA (kv head,
// split) folds `split_chunks` consecutive 64-key chunks with an online
// softmax, publishes its (max, sum, output) and, once every split of its kv
// head has done so, normalises its share of the head group's (q head, row)
// outputs over the splits in split order.  The splits of a kv head wait for
// one another, so the launch must fit on the device at once: split_chunks is
// chosen per configuration so that n_kv * max_splits CTAs are resident.
struct AttnFusedArgs {
    AttnMmaArgs m;      // shapes, layer, cap, mask rule, scale, partials, state
    int split_chunks;   // chunks per split (fixed per configuration)
    int max_splits;     // grid.y
    void* out;          // [16][n_q * head_dim], out_type (hi/lo planes for XT_BF16S)
    int out_type;
    int* arrive;        // [n_kv] published splits, zero between launches
    int* done;          // [n_kv] splits done combining, zero between launches
    int tc;             // 1: tensor-core (tcgen05) form; split_chunks 1 or 2
};

int launch_attention_fused(const AttnMaps& maps, const AttnFusedArgs& f, cudaStream_t s);

// Causal attention of a dense prompt prefill: rows pos0 .. pos0 + rows - 1,
// q from q_map ([rows/16][n_q][16][hd] f16, box = one kv head's q group),
// K/V from the target cache map; one CTA per (kv head, 16-row block) folds
// every visible 64-key chunk with the online softmax of the round's
// attention and writes the normalised rows as bf16 hi/lo planes
// [rows][n_q * hd].
struct PrefillAttnArgs {
    AttnMmaArgs m;      // shapes, layer, cap, scale (causal, no window), state
    int rows, pos0;
    void* out_hi;
    void* out_lo;
    int f16;            // 1: f16 planes (else bf16)
};
int launch_prefill_attention(const CUtensorMap& q_map, const CUtensorMap& kv_map, const PrefillAttnArgs& p,
                             cudaStream_t s);
// Attention of a many-sequence round: sequence s's 16 rows (its forward's
// T rows at positions pos0 .. pos0 + T - 1, from its round state) against
// its own cache rows, causal (verify) or [window context | bidirectional
// block] (draft).  The caches of all sequences are one map
// [S][layers][2][n_kv][cap][hd] (f16); q rows [S][n_q][16][hd] (f16, box =
// one kv head's q group).  One CTA per (kv head, sequence, split) folds its
// split's 64-key chunks (split z: chunks c_lo + z q .. c_lo + (z + 1) q - 1,
// counted from the first visible chunk, q fixed per model) with the online
// softmax of the round's attention into (max, sum, output) partials
// [S][splits][16][n_q][hd + 2]; a combine kernel folds the splits in split
// order and writes the normalised rows as bf16 hi/lo planes
// [S * 16][n_q * hd] (rows past T zero).
struct BatchAttnArgs {
    AttnMmaArgs m;            // shapes, layer, cap, causal, window, scale
    DevState* const* sts;     // [S] round state of each sequence
    int n_layers;             // layers of the cache map's model
    int split_chunks;         // q: chunks per split
    int splits;               // splits per (kv head, sequence): grid.z
    float* part;              // partials
    void* out_hi;
    void* out_lo;
};
int launch_batch_attention(const CUtensorMap& q_map, const CUtensorMap& kv_map, const BatchAttnArgs& b,
                           int S, cudaStream_t s);
// Host: CTAs of the fused attention kernel one SM holds, for head_dim hd.
int attention_fused_per_sm(int hd, int n_q, int n_kv, int* out);
// Host: the same for the tcgen05 form with nc (1 or 2) chunks per split,
// and the tensor-memory columns one of its CTAs allocates.
int attention_tc_per_sm(int hd, int nc, int* out, int* tmem_cols);

}  // namespace dfl
