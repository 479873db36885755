// Device building blocks of the tensor-core split-KV attention, shared by
// the per-launch attention kernel and the persistent round kernel.
#pragma once

#include "attention.cuh"

namespace dfl {
namespace adev {

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

// Four 8x8 b16 matrices from registers (ldmatrix fragment layout) to shared
// memory, each transposed; lane l gives the address of row l % 8 of matrix l / 8.
__device__ __forceinline__ void stsm_x4_trans(void* p, const uint32_t (&r)[4]) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
                 ::"r"(smem_u32(p)), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

// Byte address of (row, 16-byte chunk) in a tile made of HD/64 swizzled
// halves of [rows][128 B] (d 0..63 in half 0, 64..127 in half 1).
template <int HD>
__device__ __forceinline__ const uint8_t* tile_at(const uint8_t* base, int rows, int row, int chunk) {
    return base + (chunk >> 3) * rows * 128 + swz128(row, chunk & 7);
}

// Partial softmax state of one 64-key chunk (keys k0.., chunk index c) for
// q head kh * group + warp, from the tiles Qs / Ks / Vs that TMA brought
// into shared memory; rows t >= T and keys outside [lo, hi) (or after the
// query under the causal rule) weigh exactly 0.  One warp per q head.
template <int HD>
__device__ __forceinline__ void chunk_partials(const uint8_t* Qs, const uint8_t* Ks, const uint8_t* Vs,
                                               const AttnMmaArgs& a, int qrows, int group, int kh,
                                               int c, int T, int pos0, int lo, int hi, int warp,
                                               int lane) {
    constexpr int C = ATTN_KEYS;
    const int k0 = c * C;
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

// One 64-key chunk folded into a running softmax state (online softmax):
// m[r], l[r] are the running max and sum of rows g, g + 8 of q head
// kh * group + warp and o the unnormalised output.  Scores are kept in the
// base-2 domain (scaled by scale * log2 e, so p = 2^(s - m)).  A key that is
// masked for a row weighs exactly 0, and a chunk masked entirely for a row
// leaves that row's state bit-identical, so a row's result does not depend
// on how many rows the forward has.  A chunk every row sees whole (all its
// keys inside the window and before the first query) skips the mask; for a
// row that sees it whole the masked path computes the same values, and rows
// t >= T are never read.
template <int HD>
__device__ __forceinline__ void chunk_online(const uint8_t* Qs, const uint8_t* Ks, const uint8_t* Vs,
                                             const AttnMmaArgs& a, int qrows, int c, int T, int pos0,
                                             int lo, int hi, int warp, int lane, float (&m)[2],
                                             float (&l)[2], float (&o)[HD / 8][4]) {
    constexpr int C = ATTN_KEYS;
    const int k0 = c * C;
    const int g = lane >> 2, cq = lane & 3;
    const float sl2 = a.scale * 1.4426950408889634f;
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
        for (int np = 0; np < 4; ++np) {
            uint32_t kb[4];
            const int key = np * 16 + (lane & 7) + 8 * (lane >> 4);
            ldsm_x4(kb, tile_at<HD>(Ks, C, key, 2 * kd + ((lane >> 3) & 1)));
            const uint32_t b0[2] = {kb[0], kb[1]}, b1[2] = {kb[2], kb[3]};
            mma_f16_16816(s[2 * np], qa, b0);
            mma_f16_16816(s[2 * np + 1], qa, b1);
        }
    }
    const bool whole = k0 >= lo && (a.causal ? k0 + C - 1 <= pos0 : k0 + C <= hi);
    float mc[2] = {-INFINITY, -INFINITY};
    if (whole) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[nt][e] *= sl2;
                mc[e >> 1] = fmaxf(mc[e >> 1], s[nt][e]);
            }
    } else {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = g + 8 * (e >> 1);
                const int key = k0 + nt * 8 + 2 * cq + (e & 1);
                const bool valid = t < T && key >= lo && key < hi && (!a.causal || key <= pos0 + t);
                s[nt][e] = valid ? s[nt][e] * sl2 : -INFINITY;
                mc[e >> 1] = fmaxf(mc[e >> 1], s[nt][e]);
            }
    }
    float mn[2], alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        mc[r] = fmaxf(mc[r], __shfl_xor_sync(0xffffffffu, mc[r], 1));
        mc[r] = fmaxf(mc[r], __shfl_xor_sync(0xffffffffu, mc[r], 2));
        mn[r] = fmaxf(m[r], mc[r]);
        alpha[r] = (mn[r] == m[r]) ? 1.f : exp2f(m[r] - mn[r]);   // m = -inf -> 0
    }
    float ls[2] = {0.f, 0.f};
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            p[e] = (!whole && s[nt][e] == -INFINITY) ? 0.f : exp2f(s[nt][e] - mn[e >> 1]);
            ls[e >> 1] += p[e];
        }
        const int kk = nt >> 1, hi8 = nt & 1;
        pa[kk][0 + 2 * hi8] = pack_f16x2(p[0], p[1]);
        pa[kk][1 + 2 * hi8] = pack_f16x2(p[2], p[3]);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        ls[r] += __shfl_xor_sync(0xffffffffu, ls[r], 1);
        ls[r] += __shfl_xor_sync(0xffffffffu, ls[r], 2);
        l[r] = l[r] * alpha[r] + ls[r];
        m[r] = mn[r];
    }
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
        o[dt][0] *= alpha[0];
        o[dt][1] *= alpha[0];
        o[dt][2] *= alpha[1];
        o[dt][3] *= alpha[1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int dp = 0; dp < HD / 16; ++dp) {
            uint32_t vb[4];
            const int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
            ldsm_x4_trans(vb, tile_at<HD>(Vs, C, key, 2 * dp + (lane >> 4)));
            const uint32_t b0[2] = {vb[0], vb[1]}, b1[2] = {vb[2], vb[3]};
            mma_f16_16816(o[2 * dp], pa[kk], b0);
            mma_f16_16816(o[2 * dp + 1], pa[kk], b1);
        }
    }
}

}  // namespace adev
}  // namespace dfl
