// Tensor-core split-KV attention (fp16 q and caches).
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int ATTN_KEYS = 64;   // keys per chunk; equals the fp32 path's chunk

struct AttnMaps {
    CUtensorMap q;    // q rows [n_q * 16][head_dim] (head-major, 16 rows per head)
    CUtensorMap kv;   // whole cache [layers * 2 * n_kv * cap][head_dim]
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

}  // namespace dfl
