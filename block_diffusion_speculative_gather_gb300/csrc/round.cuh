// Persistent round kernel: one cooperative launch runs a whole forward of
// the DFlash round (row preparation, every decoder layer's GEMMs, attention
// and combine, the LM head, the acceptance and the tap commit) as a program
// of phases separated by grid barriers, with the weight stream of the next
// GEMM running ahead across those barriers.
#pragma once

#include "attention.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace dfl {

enum PhaseKind : int { PH_PREP = 0, PH_GEMM = 1, PH_ATTN = 2, PH_COMBINE = 3, PH_ACCEPT = 4 };

// Pointers a recorded phase takes from the launch rather than from the
// recording (they change from call to call).
enum CallSlot : int { CS_NONE = 0, CS_VERIFY_LOGITS = 1, CS_DRAFT_LOGITS = 2, CS_DRAFT_IDS = 3 };

// One phase of a program, in device memory.  The tensor maps come first
// (their type carries the alignment TMA requires).
struct Phase {
    GemmMaps maps;     // PH_GEMM: weight and activation maps
    GemmArgs g;        // PH_GEMM
    AttnMmaArgs am;    // PH_ATTN
    AttnArgs ac;       // PH_COMBINE
    RowsArgs rows;     // PH_PREP
    AcceptArgs acc;    // PH_ACCEPT
    int kind;
    int sync_before;   // 1: a grid barrier separates this phase from the previous one
    int bars_before;   // grid barriers completed before this phase reads its inputs
    int epi;           // PH_GEMM epilogue
    int logits_slot;   // PH_GEMM (ARGMAX): CS_VERIFY_LOGITS, CS_DRAFT_LOGITS or CS_NONE
    int tokens_slot;   // PH_PREP: CS_DRAFT_IDS or CS_NONE
    int target;        // PH_ATTN: 1 = target cache map, 0 = draft cache map
};

// Kernel parameter of one launch.
struct RoundCall {
    const Phase* phases;       // device
    int n_phases;
    int head_dim;
    const AttnMaps* amaps;     // device, [2]: 0 draft cache, 1 target cache
    unsigned int* bar_count;   // [0] grid-barrier arrivals, [1] abort word; zero at launch
    int* counters;             // split-K tickets of every GEMM phase, zeroed by the kernel
    int n_counters;
    DevState* st;
    const int32_t* draft_ids;  // verify input
    int32_t* draft_out;        // draft output
    int32_t* tokens_out;       // verify / greedy outputs
    int32_t* n_emitted;
    float* verify_logits;      // optional logit dumps
    float* draft_logits;
    unsigned long long* phase_ns;   // optional [n_phases + 1] phase start times (ns)
};

// Shared memory: a 4-stage ring of 2 k-blocks (bf16 weight tile 16 KB + hi/lo
// activation tile 4 KB each), one attention slot, the tile accumulator.
#ifndef DFL_ROUND_STAGES
#define DFL_ROUND_STAGES 4
#endif
#ifndef DFL_ROUND_CHUNK
#define DFL_ROUND_CHUNK 2
#endif
constexpr int ROUND_STAGES = DFL_ROUND_STAGES;
constexpr int ROUND_CHUNK = DFL_ROUND_CHUNK;
constexpr int ROUND_ATTN_BYTES = 48 * 1024;

// Attention slot bytes a configuration needs (q group + K + V of one chunk).
inline int round_attn_bytes(int n_q, int n_kv, int head_dim) {
    return (head_dim / 64) * ((n_q / n_kv) * 16 + 2 * ATTN_KEYS) * 128;
}

// Host: dynamic shared memory of the kernel, cooperative launch on `grid`
// CTAs (one per SM).  Returns 0 or the cudaError_t.
size_t round_smem_bytes();
int launch_round(const RoundCall& rc, int grid, cudaStream_t s);
// Host: CTAs of the kernel that can be resident at once on this device.
int round_max_ctas(int device, int* out);

}  // namespace dfl
