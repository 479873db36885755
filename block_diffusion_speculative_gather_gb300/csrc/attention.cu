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

#include "attention.cuh"

namespace dfl {

namespace {

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// Byte address of (row, 16-byte chunk) in a tile made of HD/64 swizzled
// halves of [rows][128 B] (d 0..63 in half 0, 64..127 in half 1).
template <int HD>
__device__ __forceinline__ const uint8_t* tile_at(const uint8_t* base, int rows, int row, int chunk) {
    return base + (chunk >> 3) * rows * 128 + swz128(row, chunk & 7);
}

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
    const int g = lane >> 2, cq = lane & 3;
    const int hq = kh * group + warp;

    // ---- S = Q K^T : 16 rows x 64 keys per warp
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int kd = 0; kd < HD / 16; ++kd) {
        uint32_t qa[4];
        ldsm_x4(qa, tile_at<HD>(Qs, qrows, warp * 16 + (lane & 15), 2 * kd + (lane >> 4)));
#pragma unroll
        for (int np = 0; np < 4; ++np) {    // pairs of n8 key tiles
            uint32_t kb[4];
            const int key = np * 16 + (lane & 7) + 8 * (lane >> 4);
            ldsm_x4(kb, tile_at<HD>(Ks, C, key, 2 * kd + ((lane >> 3) & 1)));
            const uint32_t b0[2] = {kb[0], kb[1]}, b1[2] = {kb[2], kb[3]};
            mma_f16_16816(s[2 * np], qa, b0);
            mma_f16_16816(s[2 * np + 1], qa, b1);
        }
    }

    // ---- mask, row max, probabilities (rows g and g + 8 are tokens t)
    float m[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = g + 8 * (e >> 1);
            const int key = k0 + nt * 8 + 2 * cq + (e & 1);
            const bool valid = t < T && key >= lo && key < hi && (!a.causal || key <= pos0 + t);
            s[nt][e] = valid ? s[nt][e] * a.scale : -INFINITY;
            m[e >> 1] = fmaxf(m[e >> 1], s[nt][e]);
        }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        m[r] = fmaxf(m[r], __shfl_xor_sync(0xffffffffu, m[r], 1));
        m[r] = fmaxf(m[r], __shfl_xor_sync(0xffffffffu, m[r], 2));
    }
    float l[2] = {0.f, 0.f};
    uint32_t pa[4][4];   // A fragments of P for the 4 k16 steps over the 64 keys
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            p[e] = s[nt][e] == -INFINITY ? 0.f : expf(s[nt][e] - m[e >> 1]);
            l[e >> 1] += p[e];
        }
        const int kk = nt >> 1, hi8 = nt & 1;
        pa[kk][0 + 2 * hi8] = pack_f16x2(p[0], p[1]);   // row g   (a0a1 / a4a5)
        pa[kk][1 + 2 * hi8] = pack_f16x2(p[2], p[3]);   // row g+8 (a2a3 / a6a7)
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }

    // ---- O = P V : 16 rows x HD
    float o[HD / 8][4];
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int dp = 0; dp < HD / 16; ++dp) {   // pairs of n8 d tiles
            uint32_t vb[4];
            const int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
            ldsm_x4_trans(vb, tile_at<HD>(Vs, C, key, 2 * dp + (lane >> 4)));
            const uint32_t b0[2] = {vb[0], vb[1]}, b1[2] = {vb[2], vb[3]};
            mma_f16_16816(o[2 * dp], pa[kk], b0);
            mma_f16_16816(o[2 * dp + 1], pa[kk], b1);
        }
    }

    // ---- partial softmax state of rows t = g, g + 8
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int t = g + 8 * r;
        float* dst = a.part + (((size_t)c * DFL_MAX_ROWS + t) * a.n_q + hq) * (HD + 2);
        if (cq == 0) {
            dst[0] = m[r];
            dst[1] = l[r];
        }
#pragma unroll
        for (int dt = 0; dt < HD / 8; ++dt) {
            dst[2 + dt * 8 + 2 * cq] = o[dt][2 * r];
            dst[2 + dt * 8 + 2 * cq + 1] = o[dt][2 * r + 1];
        }
    }
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
