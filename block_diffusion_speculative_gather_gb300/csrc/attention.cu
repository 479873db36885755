// Split-KV attention on tensor cores for the bf16 models (verify, prefill
// and the drafter's block attention).  q and the K/V caches are fp16 (11
// mantissa bits, against bf16's 8: the scores of a 36-layer stack stay
// within the logit tolerance), P is rounded to fp16 for the P V product.
//
// One CTA per (kv head, chunk of 64 keys).  TMA brings the query-head
// group's 16 rows per head ([group*16][head_dim], the q layout written by
// the q/k-norm kernel), and the chunk's K and V ([64][head_dim] each, one
// contiguous run per head in the cache) into 128-byte-swizzled shared
// memory.  Warp j owns query head j of the group: S = Q K^T and O = P V run
// on mma.sync m16n8k16 (fp16 in, fp32 accumulate) with ldmatrix fragments;
// the softmax state (max, sum, unnormalised O) of every row goes to the
// split partials, which the combine kernel folds in chunk order.  A key
// outside [lo, hi), or after the query under the causal rule, gets weight
// exactly 0, so a row's result never depends on how many rows the forward
// has (batch invariance) or on the chunks past its own causal limit.

#include "attention_dev.cuh"

namespace dfl {

namespace {

template <int HD>
__global__ void __launch_bounds__(128)
attn_mma_kernel(const __grid_constant__ AttnMaps maps, const AttnMmaArgs a) {
    constexpr int C = ATTN_KEYS;         // 64 keys per chunk
    constexpr int HALVES = HD / 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int group = a.n_q / a.n_kv;
    const int qrows = group * 16;
    uint8_t* Qs = sm;                                  // [HALVES][qrows][128 B]
    uint8_t* Ks = Qs + HALVES * qrows * 128;           // [HALVES][64][128 B]
    uint8_t* Vs = Ks + HALVES * C * 128;
    uint64_t* bar = reinterpret_cast<uint64_t*>(Vs + HALVES * C * 128);

    pdl_trigger();
    pdl_wait();
    const int kh = blockIdx.x, c = blockIdx.y;
    const int T = a.st->fwd_T, pos0 = a.st->fwd_pos0;
    const int hi = pos0 + T;
    const int lo = (!a.causal && a.window > 0) ? max(0, pos0 - a.window) : 0;
    const int k0 = c * C;
    if (T == 0 || k0 >= hi || k0 + C <= lo) return;

    const uint32_t bytes = (uint32_t)(HALVES * (qrows + 2 * C) * 128);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, bytes);
        const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + k0;
        const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + k0;
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            tma_load_2d(Qs + h * qrows * 128, &maps.q, bar, 64 * h, kh * qrows);
            tma_load_2d(Ks + h * C * 128, &maps.kv, bar, 64 * h, krow);
            tma_load_2d(Vs + h * C * 128, &maps.kv, bar, 64 * h, vrow);
        }
    }
    const bool ok = mbar_wait_bounded(bar, 0);
    if (!ok) {
        if (threadIdx.x == 0) {
            set_error(a.st, DERR_TIMEOUT, 200);
            mbar_wait_bounded(bar, 0, 100000000ull);   // let late copies land
        }
        return;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= group) return;
    adev::chunk_partials<HD>(Qs, Ks, Vs, a, qrows, group, kh, c, T, pos0, lo, hi, warp, lane);
}

}  // namespace

int launch_attention_mma(const AttnMaps& maps, const AttnMmaArgs& a, int max_chunks,
                         cudaStream_t s) {
    const int group = a.n_q / a.n_kv;
    const int halves = a.head_dim / 64;
    const size_t smem = 1024 + (size_t)halves * (group * 16 + 2 * ATTN_KEYS) * 128 + 64;
    dim3 grid(a.n_kv, max_chunks);
    if (a.head_dim == 128) {
        static bool set = false;
        if (!set) {
            const cudaError_t e = cudaFuncSetAttribute(
                attn_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
            set = true;
        }
        return (int)launch_k(attn_mma_kernel<128>, grid, dim3(128), smem, s, maps, a);
    } else if (a.head_dim == 64) {
        static bool set = false;
        if (!set) {
            const cudaError_t e = cudaFuncSetAttribute(
                attn_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
            set = true;
        }
        return (int)launch_k(attn_mma_kernel<64>, grid, dim3(128), smem, s, maps, a);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace dfl
