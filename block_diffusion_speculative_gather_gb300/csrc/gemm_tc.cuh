// Dense many-row GEMM on the fifth-generation tensor cores (by page: the
// drafter's context ingest stages the prompt's trailing window of tap rows,
// "feat: DFlash2 block-diffusion drafter for Qwen 3.8", third commit, into
// the persistent draft KV cache of "[RFC] DFlash", "Requested changes" 3;
// and the target's prompt forward, which returns logits and tap rows,
// "[RFC] DFlash", "Key Implementation Details", Phase 1, target hidden-state
// export):
// y[m][n] = sum_k x[m][k] * w[n][k], x and w bf16 or both f16 (w in nn.Linear layout),
// y fp32, accumulated in tensor memory.  Serves the dense part of the
// round's pipeline, the drafter's context-window ingest (fc over the
// window's tap rows, then every draft layer's context K/V), where the rows
// number hundreds to thousands and the work is a real contraction.
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int DT_BM = 128;   // rows of x per CTA (tensor-memory lanes)
constexpr int DT_BN = 256;   // widest output tile (tensor-memory columns); 128 where it balances better
constexpr int DT_WBOX = 128; // rows of one weight TMA box (a 256-column tile loads two)
constexpr int DT_SWBOX = 64; // rows of a weight box of the SwiGLU form (gate and up halves)
constexpr int DT_WTAIL = 32; // rows of the tail box of a 160-column tile (128 + 32)
constexpr int DT_BK = 64;    // k per pipeline stage (one 128-byte swizzled row)

struct DenseMaps {
    CUtensorMap x;      // [M][K] bf16, box [128 rows][64]
    CUtensorMap x_lo;   // low plane of x when x_split (same shape)
    CUtensorMap w[3];   // [N_i][K] segments concatenated along n, box [128 rows][64]
    // w[0] again with a box of DT_WTAIL rows: the last rows of a 160-column
    // tile (one-segment weights); has_tail = 1 when it is set, which lets
    // the automatic tile width pick 160 columns
    CUtensorMap w_tail;
    int has_tail;
};

struct DenseArgs {
    int M, N, K;        // K a multiple of 64
    int n_seg0;         // columns of w[0] (a multiple of 256); n >= n_seg0 reads w[1] ...
    int n_seg1;         // ... up to n_seg1 (a multiple of 256, or >= N), then w[2]
    int m_off;          // rows of x to skip: output row m reads x row m_off + m
    int x_split;        // 1: x = x (hi) + x_lo, two MMAs per k step
    int f16;            // 1: x and w are f16 (else bf16); both operands always share one type
    float* y;           // [M][ldy] fp32 (argmax epilogue: optional logits dump, or NULL)
    int ldy;            // a multiple of 4
    int* err;           // device [code, site]: a wait that timed out sets it (code 0 before)
    // split-K: `splits` CTAs per output tile share its k-blocks (contiguous
    // ranges in split order); each stores its fp32 partial rows in slab z of
    // `part` ([splits][m tiles * 128][n tiles * bn]) and a reduce kernel
    // launched after the GEMM adds the slabs in split order 0, 1, ... into y
    // (so a row's result depends on N, K and `splits`, never on M or
    // timing).  Needs y, bn 128 or 256, N a multiple of 4; no argmax.
    int splits;         // 1: no split
    float* part;
    int keep_parts;     // split-K: 1 = no reduce launch; the slabs stay for
                        // a consumer that sums them itself (y unused then)
    int bn;             // tile width: 0 = chosen by wave balance (160 too where maps.has_tail
                        // and N is a multiple of 160), else 128 or 256
    // argmax epilogue (LM head): per row the packed key (orderable logit,
    // ~column) of the largest column, atomicMax into amax[row]
    unsigned long long* amax;   // NULL: the plain fp32 store
    // SwiGLU epilogue (the fused gate/up projection), tile width bn = 128
    // or 256 fixed by the caller, h = bn / 2: output tile t holds the h gate
    // rows h t.. of w[0] (columns 0..h-1) and the matching h up rows of
    // w[up_map] at row up_row + h t (columns h..bn-1), each one weight box
    // of h rows (the maps must be made with that box: DT_SWBOX rows for bn
    // 128, DT_WBOX for 256); the epilogue writes silu(gate) * up as hi/lo
    // planes act_hi / act_lo [M][act_ld] (f16 with f16 set, else bf16) at
    // columns h t..  No split, no argmax; N = 2 x the SwiGLU width, a
    // multiple of bn.
    int swiglu;
    int up_map, up_row;
    // 1: no kernel earlier in the stream writes the weights (the model's own
    // tensors), so the first stages' weight tiles may be loaded before the
    // dependency wait; 0 (e.g. a scratch the previous kernel dequantised
    // into): every load waits
    int w_ready;
    void* act_hi;
    void* act_lo;
    int act_ld;
};

// Host: partial-tile floats a split launch needs, and its ticket count.
size_t dense_split_floats(int M, int N, int splits, int bn);
// Host: where a split launch's partial rows go: slab z of `part` starts at
// z * slab floats, row m of a slab at m * ldp.
void dense_part_layout(int M, int N, int bn, size_t* slab, size_t* ldp);
int dense_tiles(int M, int N, int bn);

// Host: dynamic shared memory of the kernel (x_split or not), the launch
// (grid ceil(M/128) x ceil(N/BN), 128 threads; BN 256, or 128 where that
// saves a wave of CTAs over the SMs).  Returns 0 or a cudaError_t.
size_t dense_smem(bool split);
int launch_dense(const DenseMaps& maps, const DenseArgs& a, cudaStream_t s);

}  // namespace dfl
