// Device building blocks of the skinny weight-streaming GEMM, shared by the
// per-launch GEMM kernel and the persistent round kernel: the tensor-core
// work on one k-block of a 128-row weight tile, and the finish of a tile
// (deterministic split-K reduction across CTAs, folded-RMSNorm row scale,
// fused epilogue).  Both expect the 8 consumer warps of a CTA
// (GEMM_CONSUMERS * 32 threads, named barrier 1).
#pragma once

#include "gemm.cuh"

namespace dfl {
namespace gdev {

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(GEMM_CONSUMERS * 32) : "memory");
}

__device__ __forceinline__ long long range_start(int b, long long U, int G) {
    return (long long)b * U / G;
}

// CTA whose stream-K range holds unit u.
__device__ __forceinline__ int cta_of(long long u, long long U, int G) {
    int b = (int)((u * G) / U);
    while (b + 1 < G && range_start(b + 1, U, G) <= u) ++b;
    while (b > 0 && range_start(b, U, G) > u) --b;
    return b;
}

template <typename T>
__device__ __forceinline__ void store_as(void* base, size_t idx, float v) {
    reinterpret_cast<T*>(base)[idx] = from_f32<T>(v);
}

__device__ __forceinline__ void store_xt(void* base, int xt, size_t idx, float v) {
    if (xt == XT_F32) store_as<float>(base, idx, v);
    else if (xt == XT_BF16) store_as<__nv_bfloat16>(base, idx, v);
    else store_as<__half>(base, idx, v);
}

__device__ __forceinline__ int ld_acquire_s32(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_s32(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

// acc += (the warp's 16 weight rows of k-block tile Wt) x (activation tile
// Xt): swap-AB mma.sync with the weight rows as M and the 16 activation rows
// as two n8 tiles (rows g, g + 8 of the C fragment are weight rows, columns
// the tokens); the lo plane of a split input is multiplied by the same
// weight fragments into its own accumulators accl (four independent MMA
// chains per warp instead of two: the chains' latency, not the tensor pipe,
// bounds these MMAs), which the tile's finish adds to acc.  Sb: the INT4
// scales of the k-block.
template <int WF, int EPI>
__device__ __forceinline__ void mma_kblock(const uint8_t* Wt, const uint8_t* Xt, const uint8_t* Sb,
                                           const GemmArgs& a, int warp, int lane, float (&acc)[8],
                                           float (&accl)[8]) {
    constexpr int XB = GemmCfg<WF>::XB;
    const int g = lane >> 2, c = lane & 3;
    if (WF == WF_INT4) {
        // 4 scale groups of 64 k; inside group q a lane owns k 16c..16c+15
        // of rows r0 and r0+8 (two interleaved 32-bit words each) and the
        // same 16 k of tokens g and g+8.  INT4 consumers take one f16
        // activation plane (rows 0..15 of the tile): the codes are exact in
        // f16, so a code pair becomes an f16 pair with one mask/or and one
        // subtraction.  Each group's partial sums, in four independent
        // chains (even / odd k-steps of both token tiles), are scaled per
        // row by the group's bf16 scale in fp32 and added to the
        // accumulators.
        const int r0 = warp * 16 + g;
        const __nv_bfloat16* St = reinterpret_cast<const __nv_bfloat16*>(Sb);
        const __half2 bias = __floats2half2_rn(1032.f, 1032.f);
        // one 64-k group at a time (a rolled loop: fewer live registers and
        // a quarter of the code, which each CTA fetches cold)
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            const uint32_t off = swz128(r0, 2 * q + (c >> 1)) + 8 * (c & 1);
            const uint2 wa = *reinterpret_cast<const uint2*>(Wt + off);
            const uint2 wb = *reinterpret_cast<const uint2*>(
                Wt + swz128(r0 + 8, 2 * q + (c >> 1)) + 8 * (c & 1));
            float sa, sb;
            if (EPI == EPI_SWIGLU) {
                sa = __bfloat162float(St[(r0 >> 6) * 256 + q * 64 + (r0 & 63)]);
                sb = __bfloat162float(St[((r0 + 8) >> 6) * 256 + q * 64 + ((r0 + 8) & 63)]);
            } else {
                sa = __bfloat162float(St[q * 128 + r0]);
                sb = __bfloat162float(St[q * 128 + r0 + 8]);
            }
            uint32_t xa[8], xb[8];
            const uint8_t* Xq = Xt + q * (XB / 4);
            *reinterpret_cast<uint4*>(&xa[0]) = lds128(Xq + swz128(g, 2 * c));
            *reinterpret_cast<uint4*>(&xa[4]) = lds128(Xq + swz128(g, 2 * c + 1));
            *reinterpret_cast<uint4*>(&xb[0]) = lds128(Xq + swz128(g + 8, 2 * c));
            *reinterpret_cast<uint4*>(&xb[4]) = lds128(Xq + swz128(g + 8, 2 * c + 1));
            // dequantise: pair p_i of a word = nibbles (i, i+4) = k (2i, 2i+1).
            // An even nibble in the low mantissa bits, 0x6400 | u, is the f16
            // 1024 + u, minus 1032 the code u - 8; an odd one left in bits
            // 4..7, 0x6400 | 16 u, is 1024 + 16 u, times 1/16 minus 72 the
            // code u - 8 (one fma, no shift); all exact in f16.  One shift
            // per word instead of three.
            uint32_t pa[8], pb[8];
            const uint32_t wordsa[2] = {wa.x, wa.y}, wordsb[2] = {wb.x, wb.y};
            const __half2 sixteenth = __floats2half2_rn(0.0625f, 0.0625f);
            const __half2 bias_hi = __floats2half2_rn(-72.f, -72.f);
            auto deq_word = [&](uint32_t w, uint32_t* p) {
                const uint32_t w8 = w >> 8;
                uint32_t u0 = (w & 0x000F000Fu) | 0x64006400u;
                uint32_t u1 = (w & 0x00F000F0u) | 0x64006400u;
                uint32_t u2 = (w8 & 0x000F000Fu) | 0x64006400u;
                uint32_t u3 = (w8 & 0x00F000F0u) | 0x64006400u;
                __half2 v0 = __hsub2(*reinterpret_cast<__half2*>(&u0), bias);
                __half2 v1 = __hfma2(*reinterpret_cast<__half2*>(&u1), sixteenth, bias_hi);
                __half2 v2 = __hsub2(*reinterpret_cast<__half2*>(&u2), bias);
                __half2 v3 = __hfma2(*reinterpret_cast<__half2*>(&u3), sixteenth, bias_hi);
                p[0] = *reinterpret_cast<uint32_t*>(&v0);
                p[1] = *reinterpret_cast<uint32_t*>(&v1);
                p[2] = *reinterpret_cast<uint32_t*>(&v2);
                p[3] = *reinterpret_cast<uint32_t*>(&v3);
            };
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                deq_word(wordsa[m], pa + 4 * m);
                deq_word(wordsb[m], pb + 4 * m);
            }
            float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
            float h0[4] = {0.f, 0.f, 0.f, 0.f}, h1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t A[4] = {pa[2 * j], pb[2 * j], pa[2 * j + 1], pb[2 * j + 1]};
                const uint32_t B0[2] = {xa[2 * j], xa[2 * j + 1]};
                const uint32_t B1[2] = {xb[2 * j], xb[2 * j + 1]};
                if (j & 1) {
                    mma_f16_16816(h0, A, B0);
                    mma_f16_16816(h1, A, B1);
                } else {
                    mma_f16_16816(g0, A, B0);
                    mma_f16_16816(g1, A, B1);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                g0[e] += h0[e];
                g1[e] += h1[e];
            }
            acc[0] = fmaf(sa, g0[0], acc[0]);
            acc[1] = fmaf(sa, g0[1], acc[1]);
            acc[2] = fmaf(sb, g0[2], acc[2]);
            acc[3] = fmaf(sb, g0[3], acc[3]);
            acc[4] = fmaf(sa, g1[0], acc[4]);
            acc[5] = fmaf(sa, g1[1], acc[5]);
            acc[6] = fmaf(sb, g1[2], acc[6]);
            acc[7] = fmaf(sb, g1[3], acc[7]);
        }
        (void)accl;
    } else if (WF == WF_BF16) {
        const int r0 = warp * 16 + g;
        uint32_t ra[8], rb[8], xa[8], xb[8];
        *reinterpret_cast<uint4*>(&ra[0]) = lds128(Wt + swz128(r0, 2 * c));
        *reinterpret_cast<uint4*>(&ra[4]) = lds128(Wt + swz128(r0, 2 * c + 1));
        *reinterpret_cast<uint4*>(&rb[0]) = lds128(Wt + swz128(r0 + 8, 2 * c));
        *reinterpret_cast<uint4*>(&rb[4]) = lds128(Wt + swz128(r0 + 8, 2 * c + 1));
        *reinterpret_cast<uint4*>(&xa[0]) = lds128(Xt + swz128(g, 2 * c));
        *reinterpret_cast<uint4*>(&xa[4]) = lds128(Xt + swz128(g, 2 * c + 1));
        *reinterpret_cast<uint4*>(&xb[0]) = lds128(Xt + swz128(g + 8, 2 * c));
        *reinterpret_cast<uint4*>(&xb[4]) = lds128(Xt + swz128(g + 8, 2 * c + 1));
        float(&d0)[4] = *reinterpret_cast<float(*)[4]>(&acc[0]);
        float(&d1)[4] = *reinterpret_cast<float(*)[4]>(&acc[4]);
        float(&e0)[4] = *reinterpret_cast<float(*)[4]>(&accl[0]);
        float(&e1)[4] = *reinterpret_cast<float(*)[4]>(&accl[4]);
        uint32_t la[8], lb[8];
        if (a.x_split) {   // lo planes: tokens g, g + 8 at rows 16 + g, 24 + g
            *reinterpret_cast<uint4*>(&la[0]) = lds128(Xt + swz128(16 + g, 2 * c));
            *reinterpret_cast<uint4*>(&la[4]) = lds128(Xt + swz128(16 + g, 2 * c + 1));
            *reinterpret_cast<uint4*>(&lb[0]) = lds128(Xt + swz128(24 + g, 2 * c));
            *reinterpret_cast<uint4*>(&lb[4]) = lds128(Xt + swz128(24 + g, 2 * c + 1));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t A[4] = {ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1]};
            const uint32_t B0[2] = {xa[2 * j], xa[2 * j + 1]};
            const uint32_t B1[2] = {xb[2 * j], xb[2 * j + 1]};
            mma_bf16_16816(d0, A, B0);
            mma_bf16_16816(d1, A, B1);
            if (a.x_split) {
                const uint32_t L0[2] = {la[2 * j], la[2 * j + 1]};
                const uint32_t L1[2] = {lb[2 * j], lb[2 * j + 1]};
                mma_bf16_16816(e0, A, L0);
                mma_bf16_16816(e1, A, L1);
            }
        }
    } else {  // WF_F32: CUDA-core FMAs, k in order
        const int t = lane & 15, h = lane >> 4;
        float xv[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint4 v = lds128(Xt + swz128(t, q));
            xv[4 * q + 0] = __uint_as_float(v.x);
            xv[4 * q + 1] = __uint_as_float(v.y);
            xv[4 * q + 2] = __uint_as_float(v.z);
            xv[4 * q + 3] = __uint_as_float(v.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = warp * 16 + 8 * h + i;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = lds128(Wt + swz128(row, q));
                acc[i] = fmaf(__uint_as_float(v.x), xv[4 * q + 0], acc[i]);
                acc[i] = fmaf(__uint_as_float(v.y), xv[4 * q + 1], acc[i]);
                acc[i] = fmaf(__uint_as_float(v.z), xv[4 * q + 2], acc[i]);
                acc[i] = fmaf(__uint_as_float(v.w), xv[4 * q + 3], acc[i]);
            }
        }
    }
}

// Row scale of a folded RMSNorm, once per GEMM and CTA: rstd[t] from the
// producer's per-128-column partial sums of x^2, summed in column order
// (the same for every forward length).  Threads 0..15 load every part first
// (independent loads, one round trip) and then add them in order; s_rstd is
// read only after the next consumer barrier.
template <int EPI>
__device__ __forceinline__ void compute_rstd(const GemmArgs& a, float* s_rstd, int tid) {
    if (!(EPI == EPI_SWIGLU || EPI == EPI_ARGMAX || EPI == EPI_QKV)) return;
    if (tid >= DFL_MAX_ROWS) return;
    float r = 1.f;
    if (a.ssq_in) {
        float ss = 0.f;
        for (int p0 = 0; p0 < a.ssq_parts; p0 += 8) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = p0 + j < a.ssq_parts ? a.ssq_in[(p0 + j) * DFL_MAX_ROWS + tid] : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (p0 + j < a.ssq_parts) ss += v[j];
        }
        r = 1.0f / sqrtf(ss * a.inv_width + a.eps);
    }
    s_rstd[tid] = r;
}

// Finish of a tile whose last k-block this CTA has just accumulated.  A
// tile split across CTAs is finished by its owner, the first CTA of the
// split (it reaches the tile at the end of its range): the other CTAs
// publish their parts and go on; the owner sums the parts in CTA order and
// runs the epilogue, so a row's result never depends on timing or on the
// other rows.
template <int WF, int EPI>
__device__ __forceinline__ void finish_tile(const GemmArgs& a, int tile, const float (&acc)[8],
                                            float* ctile, volatile int* s_flags, float* s_rstd,
                                            long long U, int G, int cta, int warp, int lane,
                                            int tid) {
    const int g = lane >> 2, c = lane & 3;
    // ------------------------------------------ finish this tile
    if (WF != WF_F32) {
        // C fragment: (row g, tokens 2c,2c+1), (row g+8, tokens 2c,2c+1) per n8 tile
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t0 = nt * 8 + 2 * c, r = warp * 16 + g;
            ctile[(t0 + 0) * GEMM_BN + r] = acc[nt * 4 + 0];
            ctile[(t0 + 1) * GEMM_BN + r] = acc[nt * 4 + 1];
            ctile[(t0 + 0) * GEMM_BN + r + 8] = acc[nt * 4 + 2];
            ctile[(t0 + 1) * GEMM_BN + r + 8] = acc[nt * 4 + 3];
        }
    } else {
        const int t = lane & 15, h = lane >> 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) ctile[t * GEMM_BN + warp * 16 + 8 * h + i] = acc[i];
    }
    consumer_bar();

    const long long ts = (long long)tile * a.kb;
    const int i_first = cta_of(ts, U, G), i_last = cta_of(ts + a.kb - 1, U, G);
    const bool aborted = s_flags[0] != 0;
    bool do_epi = !aborted;
    // Epilogue operands from global memory, loaded now (independent loads,
    // in flight while the parts of a split tile are gathered) by the CTA
    // that runs the epilogue.
    float pre_x[2][4], pre_w[4];
    if ((EPI == EPI_RESID || EPI == EPI_NORMOUT) && (i_first == i_last || cta == i_first)) {
        const int n0 = tile * GEMM_BN;
#pragma unroll
        for (int i = 0; i < 4; ++i) pre_w[i] = a.w_next ? a.w_next[n0 + lane * 4 + i] : 1.f;
        if (EPI == EPI_RESID) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    pre_x[q][i] = a.out[(size_t)(warp * 2 + q) * a.ldo + n0 + lane * 4 + i];
        }
    }
    if (i_first != i_last && cta != i_first) {
        // A later part of a split tile: the tile was this CTA's first, so its
        // part goes to this CTA's slot; the tile's owner, CTA i_first (whose
        // range ends in the tile, so it reaches the tile last), is told
        // through the tile's counter and nothing here waits.
        // The barrier orders every thread's part stores before thread 0's
        // release add, and a release is cumulative over what was ordered
        // before it, so the add publishes the whole part; no thread fences
        // on its own stores (a fence per thread held all consumer warps for
        // the stores' acknowledgement, several microseconds under the full
        // weight stream, while the ring stalled behind them).
        float* mine = a.slots + (size_t)cta * 2 * (GEMM_BN * DFL_MAX_ROWS);
        for (int e = tid; e < GEMM_BN * DFL_MAX_ROWS; e += GEMM_CONSUMERS * 32)
            __stcg(mine + e, ctile[e]);
        consumer_bar();
        if (tid == 0) red_release_add_s32(&a.counters[tile], 1);
        do_epi = false;
    } else if (i_first != i_last) {
        // The owner: wait (bounded) until the other parts are published,
        // then sum all parts in CTA order, its own (still in ctile) first.
        if (tid == 0) {
            const int need = i_last - i_first;
            bool ok = ld_acquire_s32(&a.counters[tile]) >= need;
            if (!ok && !aborted) {
                const uint64_t t0 = globaltimer_ns();
                while (!(ok = ld_acquire_s32(&a.counters[tile]) >= need)) {
                    if (globaltimer_ns() - t0 > 2000000000ull) {
                        set_error(a.st, DERR_TIMEOUT, 105);
                        break;
                    }
                }
            }
            if (ok) a.counters[tile] = 0;   // ready for the next launch
            s_flags[1] = ok ? 1 : 0;
        }
        consumer_bar();
        do_epi = !aborted && s_flags[1] != 0;
        if (do_epi) {
            // Thread 0's acquire, then the barrier, order the parts' loads
            // (L2, __ldcg) after their publication for every thread.
            // Each thread owns 8 consecutive elements (two float4).
            const int e0 = tid * 8;
            float4 acc0 = *reinterpret_cast<const float4*>(ctile + e0);
            float4 acc1 = *reinterpret_cast<const float4*>(ctile + e0 + 4);
            auto part_ptr = [&](int i) {
                return reinterpret_cast<const float4*>(
                    a.slots + (size_t)i * 2 * (GEMM_BN * DFL_MAX_ROWS) + e0);
            };
            auto add4 = [](float4& x, const float4& y) {
                x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
            };
            // up to 8 parts in flight at once (a tile of a 152-CTA split has <= 8)
            for (int i0 = i_first + 1; i0 <= i_last; i0 += 8) {
                float4 va[8], vb[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (i0 + j <= i_last) {
                        va[j] = __ldcg(part_ptr(i0 + j));
                        vb[j] = __ldcg(part_ptr(i0 + j) + 1);
                    }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (i0 + j <= i_last) {
                        add4(acc0, va[j]);
                        add4(acc1, vb[j]);
                    }
            }
            *reinterpret_cast<float4*>(ctile + e0) = acc0;   // its own elements only
            *reinterpret_cast<float4*>(ctile + e0 + 4) = acc1;
            consumer_bar();
        }
    }

    if (do_epi) {
        if (EPI == EPI_STORE) {
            const int n0 = tile * GEMM_BN;
            for (int e = tid; e < GEMM_BN * DFL_MAX_ROWS; e += GEMM_CONSUMERS * 32) {
                const int t = e / GEMM_BN, r = e % GEMM_BN;
                a.out[(size_t)t * a.ldo + n0 + r] = ctile[e];
            }
        } else if (EPI == EPI_RESID || EPI == EPI_NORMOUT) {
            // warp w: tokens 2w, 2w+1; lane: 4 consecutive columns
            const int n0 = tile * GEMM_BN;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int t = warp * 2 + q;
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane * 4 + i;
                    float v = ctile[t * GEMM_BN + r];
                    if (EPI == EPI_RESID) {
                        v += pre_x[q][i];
                        a.out[(size_t)t * a.ldo + n0 + r] = v;
                        if (a.tap_out) store_act(a.tap_out, a.tap_type, a.ld_tap, t, n0 + r, v);
                    }
                    ss = fmaf(v, v, ss);
                    store_act(a.xn_out, a.xn_type, a.ldo, t, n0 + r, v * pre_w[i]);
                }
                ss = warp_sum(ss);
                if (a.ssq_out && lane == 0) a.ssq_out[tile * DFL_MAX_ROWS + t] = ss;
            }
        } else if (EPI == EPI_SWIGLU) {
            const int j0 = tile * 64;
            for (int e = tid; e < 64 * DFL_MAX_ROWS; e += GEMM_CONSUMERS * 32) {
                const int t = e / 64, r = e % 64;
                const float gt = ctile[t * GEMM_BN + r] * s_rstd[t];
                const float up = ctile[t * GEMM_BN + 64 + r] * s_rstd[t];
                const float v = gt / (1.f + expf(-gt)) * up;
                store_act(a.act, a.act_type, a.ld_act, t, j0 + r, v);
            }
        } else if (EPI == EPI_QKV) {
            // the tile is 128 / hd whole heads; item = (token, head in tile)
            const QkvEpi& qe = a.qkv;
            int r0;
            const int nrows = rows_of(a.st, qe.row_sel, &r0);
            const int pos0 = a.st->fwd_pos0;
            const int hd = qe.hd, hpt = GEMM_BN / hd, per = hd / 32;
            int tile_l = tile;               // the tile within its layer
            const float* k_norm = qe.k_norm;
            size_t lay_off = 0;              // cache element offset of the tile's layer
            if (qe.group > 1) {
                const int tpl = 2 * qe.n_kv / hpt;   // tiles per layer: [W_k; W_v]
                const int l = tile / tpl;
                tile_l = tile - l * tpl;
                k_norm = qe.k_norm_all + (size_t)l * hd;
                lay_off = (size_t)l * (size_t)qe.cache_stride;
            }
            const int h_first = tile_l * hpt;
            // head-norm weights of this lane (q and k), loaded once
            float qn[4], kn[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                qn[m] = (m < per && qe.n_q > 0) ? qe.q_norm[lane + 32 * m] : 0.f;
                kn[m] = m < per ? k_norm[lane + 32 * m] : 0.f;
            }
            for (int item = warp; item < DFL_MAX_ROWS * hpt; item += GEMM_CONSUMERS) {
                const int t = item / hpt, hi = item % hpt;
                if (t < r0 || t >= r0 + nrows) continue;
                const int h = h_first + hi;
                const bool is_q = h < qe.n_q, is_k = !is_q && h < qe.n_q + qe.n_kv;
                // rotate-half pairs element i with i + hd/2 (same lane, m + per/2)
                float cs[2], sn[2];
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    cs[m] = (m < per / 2 && (is_q || is_k)) ? qe.rope_cos[t * (hd / 2) + lane + 32 * m] : 0.f;
                    sn[m] = (m < per / 2 && (is_q || is_k)) ? qe.rope_sin[t * (hd / 2) + lane + 32 * m] : 0.f;
                }
                float v[4];
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    v[m] = m < per ? ctile[t * GEMM_BN + hi * hd + lane + 32 * m] * s_rstd[t] : 0.f;
                if (is_q || is_k) {
                    float ss = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) ss = fmaf(v[m], v[m], ss);   // v[m >= per] = 0
                    ss = warp_sum(ss);
                    const float inv = 1.0f / sqrtf(ss / (float)hd + a.eps);
#pragma unroll
                    for (int m = 0; m < 4; ++m) v[m] = v[m] * inv * (is_q ? qn[m] : kn[m]);
                    float rr[4];
                    if (per == 4) {
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            rr[m] = v[m] * cs[m] - v[m + 2] * sn[m];
                            rr[m + 2] = v[m + 2] * cs[m] + v[m] * sn[m];
                        }
                    } else {
                        rr[0] = v[0] * cs[0] - v[1] * sn[0];
                        rr[1] = v[1] * cs[0] + v[0] * sn[0];
                        rr[2] = rr[3] = 0.f;
                    }
#pragma unroll
                    for (int m = 0; m < 4; ++m) v[m] = rr[m];
                }
                if (is_q) {
                    const size_t base = ((size_t)h * DFL_MAX_ROWS + t) * hd;   // [n_q][16][hd]
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m < per) store_xt(qe.q_out, qe.q_type, base + lane + 32 * m, v[m]);
                    continue;
                }
                const int pos = pos0 + t;
                if (pos < 0 || pos >= qe.max_seq) {
                    if (lane == 0) set_error(a.st, DERR_INDEX, pos);
                    continue;
                }
                const int kh = is_k ? h - qe.n_q : h - qe.n_q - qe.n_kv;
                void* cache = is_k ? qe.k_cache : qe.v_cache;
                const size_t base = lay_off + ((size_t)kh * qe.cap + pos) * hd;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (m < per) store_xt(cache, qe.c_type, base + lane + 32 * m, v[m]);
            }
        } else {  // EPI_ARGMAX: warp w reduces tokens 2w, 2w+1
            const int n0 = tile * GEMM_BN;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int t = warp * 2 + q;
                unsigned long long best = 0ull;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane * 4 + i;
                    const float v = ctile[t * GEMM_BN + r] * s_rstd[t];
                    best = umax64(best, argmax_key(v, n0 + r));
                    if (a.logits) a.logits[(size_t)t * a.ldl + n0 + r] = v;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
                if (lane == 0) atomicMax(a.amax + t, best);
            }
        }
    }
    consumer_bar();   // ctile is rewritten by the next tile
}

}  // namespace gdev
}  // namespace dfl
