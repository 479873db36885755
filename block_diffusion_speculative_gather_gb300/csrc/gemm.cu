// Skinny weight-streaming GEMM for the <= 16 rows of one DFlash forward.
//
// Y[t][n] = sum_k X[t][k] W[n][k], W in the nn.Linear layout [N][K].  The
// rows t (block rows, verify rows or a prefill chunk) are few, so the work
// is a stream of W from HBM: one pass over W per call is the whole cost.
//
// Design (sm_103a):
//  * one persistent CTA per SM; the flattened (tile, k-block) space is split
//    into equal contiguous ranges (stream-K), so every SM streams the same
//    number of bytes whatever N and K are;
//  * a producer warp issues TMA tile loads (cp.async.bulk.tensor, 128-byte
//    swizzle) of consecutive weight tiles [128 rows x 128 B] and the
//    matching activation tiles into a shared-memory ring of stages guarded
//    by mbarriers; 8 consumer warps each own 16 weight rows;
//  * the activations of the model's own forward are two bf16 planes (hi and
//    the rounding remainder lo, rows 0..15 and 16..31 of the X tile): each
//    weight fragment is multiplied by both, so the product carries the
//    activation to about 16 mantissa bits while the weights stream once;
//  * bf16 weights: the weight rows are the M=16 side of mma.sync m16n8k16
//    (swap-AB) and the <= 16 activation rows the N side (two n8 tiles);
//    inside each 64-wide k-block every lane takes 16 consecutive k
//    (one 32-byte run per row) and the same permutation of k is applied to
//    both operands, so fragments come from plain 16-byte shared loads;
//  * fp32 weights (the tiny fp32 workload) use CUDA-core FMAs in k order;
//  * a tile whose k-range is split across CTAs is finished by the last CTA
//    to arrive (atomic ticket, no waiting), which sums the parts in a fixed
//    order: the result of a row never depends on how many rows the forward
//    has, on timing, or on the other rows (batch invariance);
//  * fused epilogues: store fp32, residual add (+ tap copy), SwiGLU of
//    paired gate/up tiles, LM-head argmax with packed 64-bit atomicMax.
//
// Every mbarrier wait is bounded; an expired wait sets the device error
// word, stops new copies and drains the copies already issued.

#include <cstdlib>

#include "gemm.cuh"

namespace dfl {

long long g_launches = 0;
bool g_pdl = [] {
    const char* e = getenv("DFLASH_PDL");
    return !(e && e[0] == '0');
}();

namespace {

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(GEMM_CONSUMERS * 32) : "memory");
}

__device__ __forceinline__ long long range_start(int b, long long U, int G) {
    return (long long)b * U / G;
}

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

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

template <int WF, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, DFL_GEMM_MINBLOCKS)
gemm_skinny_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using CFG = GemmCfg<WF>;
    constexpr int STAGES = CFG::STAGES, KBLK = CFG::KBLK, XB = CFG::XB, SB = CFG::SB;
    constexpr int CHUNK = CFG::CHUNK;
    // bytes one k-block brings: an unsplit bf16 input fills half of its X slot
    const uint32_t KB_BYTES = GEMM_STAGE_W + SB + ((WF == WF_F32 || a.x_split) ? XB : XB / 2);
    uint8_t* Ws = smem;                                        // [STAGES][CHUNK][128 x 128 B]
    uint8_t* Xs = Ws + STAGES * CHUNK * GEMM_STAGE_W;          // [STAGES][CHUNK][XB]
    uint8_t* Ss = Xs + STAGES * CHUNK * XB;                    // [STAGES][CHUNK][SB] (INT4)
    float* ctile = reinterpret_cast<float*>(Ss + STAGES * CHUNK * SB);   // [16][128]
    uint64_t* full = reinterpret_cast<uint64_t*>(ctile + DFL_MAX_ROWS * GEMM_BN);
    uint64_t* empty = full + STAGES;
    volatile int* s_flags = reinterpret_cast<volatile int*>(empty + STAGES);
    // s_flags[0]: abort, [1]: last-arriver, [2]: consumed stage count

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const long long U = (long long)a.n_tiles * a.kb;
    const long long u0 = range_start(blockIdx.x, U, G), u1 = range_start(blockIdx.x + 1, U, G);
    // k-blocks in the stage that starts at unit u: never past the tile or the range
    auto chunk_len = [&](long long u) {
        long long n = CHUNK;
        if (u1 - u < n) n = u1 - u;
        const long long to_tile_end = a.kb - (u % a.kb);
        if (to_tile_end < n) n = to_tile_end;
        return (int)n;
    };

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GEMM_CONSUMERS);
        }
        s_flags[0] = 0;
        s_flags[1] = 0;
        s_flags[2] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == GEMM_CONSUMERS) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < a.n_seg; ++i) {
                tma_prefetch_desc(&maps.w[i]);
                if (WF == WF_INT4) tma_prefetch_desc(&maps.s[i]);
            }
            tma_prefetch_desc(&maps.x);
            // weight (+ INT4 scale) tile of unit u into slot j of a stage
            auto load_w = [&](long long u, int stage, int j) {
                const int tile = (int)(u / a.kb), k = (int)(u % a.kb);
                uint8_t* wdst = Ws + (stage * CHUNK + j) * GEMM_STAGE_W;
                uint8_t* sdst = Ss + (stage * CHUNK + j) * SB;
                // weight x coordinate: elements for F32/BF16, bytes for packed INT4
                const int wx = WF == WF_INT4 ? k * 128 : k * KBLK;
                if (EPI == EPI_SWIGLU) {
                    tma_load_2d(wdst, &maps.w[0], &full[stage], wx, tile * 64);
                    tma_load_2d(wdst + 64 * 128, &maps.w[1], &full[stage], wx, tile * 64);
                    if (WF == WF_INT4) {
                        tma_load_2d(sdst, &maps.s[0], &full[stage], tile * 64, k * 4);
                        tma_load_2d(sdst + SB / 2, &maps.s[1], &full[stage], tile * 64, k * 4);
                    }
                } else {
                    int row = tile * GEMM_BN, seg = 0;
                    while (seg + 1 < a.n_seg && row >= a.seg_rows[seg]) {
                        row -= a.seg_rows[seg];
                        ++seg;
                    }
                    tma_load_2d(wdst, &maps.w[seg], &full[stage], wx, row);
                    if (WF == WF_INT4) tma_load_2d(sdst, &maps.s[seg], &full[stage], row, k * 4);
                }
            };
            // activation tile(s) of unit u into slot j of a stage
            auto load_x = [&](long long u, int stage, int j) {
                const int k = (int)(u % a.kb);
                uint8_t* xdst = Xs + (stage * CHUNK + j) * XB;
                if (WF == WF_INT4) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tma_load_2d(xdst + q * (XB / 4), &maps.x, &full[stage], k * KBLK + 64 * q, 0);
                } else {
                    tma_load_2d(xdst, &maps.x, &full[stage], k * KBLK, 0);
                }
            };
            // The weights do not depend on earlier kernels: fill the ring with
            // them before waiting for the predecessor (programmatic dependent
            // launch), then add the activation tiles.
            long long pu[STAGES];
            int pl[STAGES];
            int npre = 0;
            long long u = u0;
            while (u < u1 && npre < STAGES) {
                const int len = chunk_len(u);
                pu[npre] = u;
                pl[npre] = len;
                mbar_arrive_expect_tx(&full[npre], len * KB_BYTES);
                for (int j = 0; j < len; ++j) load_w(u + j, npre, j);
                u += len;
                ++npre;
            }
            pdl_wait();
            for (int i = 0; i < npre; ++i)
                for (int j = 0; j < pl[i]; ++j) load_x(pu[i] + j, i, j);
            long long issued = npre;
            int stage = npre % STAGES;
            uint32_t phase = npre == STAGES ? 1u : 0u;
            while (u < u1) {
                if (s_flags[0]) break;
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1u)) {
                    s_flags[0] = 1;
                    set_error(a.st, DERR_TIMEOUT, 100);
                    break;
                }
                if (s_flags[0]) break;   // consumers gave up: issue nothing more
                const int len = chunk_len(u);
                mbar_arrive_expect_tx(&full[stage], len * KB_BYTES);
                for (int j = 0; j < len; ++j) {
                    load_w(u + j, stage, j);
                    load_x(u + j, stage, j);
                }
                u += len;
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            // Wait (bounded) until the consumers have seen every issued copy
            // land; after an abort, wait (bounded) for the copies still in
            // flight so none lands after the CTA has exited.
            const uint64_t t0 = globaltimer_ns();
            while (s_flags[2] < issued && !s_flags[0]) {
                if (globaltimer_ns() - t0 > 4000000000ull) {
                    s_flags[0] = 1;
                    set_error(a.st, DERR_TIMEOUT, 102);
                    break;
                }
                __nanosleep(256);
            }
            if (s_flags[0]) {
                for (long long j = s_flags[2]; j < issued; ++j)
                    mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1),
                                      100000000ull);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    __shared__ float s_rstd[DFL_MAX_ROWS];
    pdl_wait();    // the epilogues read and write buffers of earlier kernels
    const int tid = threadIdx.x;   // 0..255
    const int g = lane >> 2, c = lane & 3;
    int stage = 0;
    uint32_t phase = 0;
    float acc[8];
    int first_tile_of_me = (int)(u0 / a.kb);

    for (long long u = u0; u < u1;) {
        const int len = chunk_len(u);
        const int tile = (int)(u / a.kb), k = (int)(u % a.kb);
        if (k == 0 || u == u0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        }
        bool ok = false;
        if (!s_flags[0]) {
            ok = mbar_wait_bounded(&full[stage], phase);
            if (!ok) {
                s_flags[0] = 1;
                set_error(a.st, DERR_TIMEOUT, 101);
            }
        }
        if (ok) {
            for (int jb = 0; jb < len; ++jb) {
            const uint8_t* Wt = Ws + (stage * CHUNK + jb) * GEMM_STAGE_W;
            const uint8_t* Xt = Xs + (stage * CHUNK + jb) * XB;
            const uint8_t* Sb = Ss + (stage * CHUNK + jb) * SB;
            if (WF == WF_INT4) {
                // 4 scale groups of 64 k; inside group q a lane owns k 16c..16c+15
                // of rows r0 and r0+8 (two interleaved 32-bit words each) and the
                // same 16 k of tokens g and g+8; the group's partial sums are
                // scaled per row in fp32 and added to the accumulators.
                const int r0 = warp * 16 + g;
                const __nv_bfloat16* St = reinterpret_cast<const __nv_bfloat16*>(Sb);
                const __nv_bfloat162 bias = __floats2bfloat162_rn(136.f, 136.f);
#pragma unroll
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
                    // dequantise: pair p_i of a word = nibbles (i, i+4) = k (2i, 2i+1)
                    uint32_t pa[8], pb[8];
                    const uint32_t wordsa[2] = {wa.x, wa.y}, wordsb[2] = {wb.x, wb.y};
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t ua = ((wordsa[m] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
                            uint32_t ub = ((wordsb[m] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
                            __nv_bfloat162 va = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&ua), bias);
                            __nv_bfloat162 vb = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&ub), bias);
                            pa[4 * m + i] = *reinterpret_cast<uint32_t*>(&va);
                            pb[4 * m + i] = *reinterpret_cast<uint32_t*>(&vb);
                        }
                    }
                    float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t A[4] = {pa[2 * j], pb[2 * j], pa[2 * j + 1], pb[2 * j + 1]};
                        const uint32_t B0[2] = {xa[2 * j], xa[2 * j + 1]};
                        const uint32_t B1[2] = {xb[2 * j], xb[2 * j + 1]};
                        mma_bf16_16816(g0, A, B0);
                        mma_bf16_16816(g1, A, B1);
                    }
                    if (a.x_split) {   // lo planes: tokens g, g + 8 at rows 16 + g, 24 + g
                        *reinterpret_cast<uint4*>(&xa[0]) = lds128(Xq + swz128(16 + g, 2 * c));
                        *reinterpret_cast<uint4*>(&xa[4]) = lds128(Xq + swz128(16 + g, 2 * c + 1));
                        *reinterpret_cast<uint4*>(&xb[0]) = lds128(Xq + swz128(24 + g, 2 * c));
                        *reinterpret_cast<uint4*>(&xb[4]) = lds128(Xq + swz128(24 + g, 2 * c + 1));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t A[4] = {pa[2 * j], pb[2 * j], pa[2 * j + 1], pb[2 * j + 1]};
                            const uint32_t B0[2] = {xa[2 * j], xa[2 * j + 1]};
                            const uint32_t B1[2] = {xb[2 * j], xb[2 * j + 1]};
                            mma_bf16_16816(g0, A, B0);
                            mma_bf16_16816(g1, A, B1);
                        }
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
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t A[4] = {ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1]};
                    const uint32_t B0[2] = {xa[2 * j], xa[2 * j + 1]};
                    const uint32_t B1[2] = {xb[2 * j], xb[2 * j + 1]};
                    mma_bf16_16816(d0, A, B0);
                    mma_bf16_16816(d1, A, B1);
                }
                if (a.x_split) {   // lo planes: tokens g, g + 8 at rows 16 + g, 24 + g
                    *reinterpret_cast<uint4*>(&xa[0]) = lds128(Xt + swz128(16 + g, 2 * c));
                    *reinterpret_cast<uint4*>(&xa[4]) = lds128(Xt + swz128(16 + g, 2 * c + 1));
                    *reinterpret_cast<uint4*>(&xb[0]) = lds128(Xt + swz128(24 + g, 2 * c));
                    *reinterpret_cast<uint4*>(&xb[4]) = lds128(Xt + swz128(24 + g, 2 * c + 1));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t A[4] = {ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1]};
                        const uint32_t B0[2] = {xa[2 * j], xa[2 * j + 1]};
                        const uint32_t B1[2] = {xb[2 * j], xb[2 * j + 1]};
                        mma_bf16_16816(d0, A, B0);
                        mma_bf16_16816(d1, A, B1);
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
            }   // k-blocks of the stage
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (tid == 0 && ok) s_flags[2] = s_flags[2] + 1;   // stages seen complete
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        u += len;

        if (!(k + len == a.kb || u == u1)) continue;

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
        if (i_first != i_last) {
            const int slot = (tile == first_tile_of_me) ? 0 : 1;
            float* mine = a.slots + ((size_t)blockIdx.x * 2 + slot) * (GEMM_BN * DFL_MAX_ROWS);
            for (int e = tid; e < GEMM_BN * DFL_MAX_ROWS; e += GEMM_CONSUMERS * 32)
                __stcg(mine + e, ctile[e]);
            __threadfence();
            consumer_bar();
            if (tid == 0) {
                int last = 0;
                if (!aborted) {
                    const int old = atomicAdd(&a.counters[tile], 1);
                    last = (old == i_last - i_first);
                }
                s_flags[1] = last;
            }
            consumer_bar();
            do_epi = s_flags[1] != 0;
            if (do_epi) {
                __threadfence();
                if (tid == 0) a.counters[tile] = 0;
                // Sum the parts in CTA order.  Each thread owns 8 consecutive
                // elements (two float4) and issues the loads of four parts at
                // a time, so the L2 round trips overlap.
                const int e0 = tid * 8;
                float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
                auto part_ptr = [&](int i) {
                    const int first_i = (int)(range_start(i, U, G) / a.kb);
                    const int si = (tile == first_i) ? 0 : 1;
                    return a.slots + ((size_t)i * 2 + si) * (GEMM_BN * DFL_MAX_ROWS) + e0;
                };
                auto add4 = [](float4& x, const float4& y) {
                    x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
                };
                int i = i_first;
                for (; i + 3 <= i_last; i += 4) {
                    const float4* p0 = reinterpret_cast<const float4*>(part_ptr(i));
                    const float4* p1 = reinterpret_cast<const float4*>(part_ptr(i + 1));
                    const float4* p2 = reinterpret_cast<const float4*>(part_ptr(i + 2));
                    const float4* p3 = reinterpret_cast<const float4*>(part_ptr(i + 3));
                    const float4 a0 = __ldcg(p0), b0 = __ldcg(p0 + 1);
                    const float4 a1 = __ldcg(p1), b1 = __ldcg(p1 + 1);
                    const float4 a2 = __ldcg(p2), b2 = __ldcg(p2 + 1);
                    const float4 a3 = __ldcg(p3), b3 = __ldcg(p3 + 1);
                    add4(acc0, a0); add4(acc1, b0);
                    add4(acc0, a1); add4(acc1, b1);
                    add4(acc0, a2); add4(acc1, b2);
                    add4(acc0, a3); add4(acc1, b3);
                }
                for (; i <= i_last; ++i) {
                    const float4* p0 = reinterpret_cast<const float4*>(part_ptr(i));
                    add4(acc0, __ldcg(p0));
                    add4(acc1, __ldcg(p0 + 1));
                }
                *reinterpret_cast<float4*>(ctile + e0) = acc0;
                *reinterpret_cast<float4*>(ctile + e0 + 4) = acc1;
                consumer_bar();
            }
        }

        // Row scale of a folded RMSNorm: rstd[t] from the partial sums, summed
        // in a fixed order (the same for every forward length).  Computed by
        // all consumer threads, before the (barrier-free) epilogue.
        if (EPI == EPI_SWIGLU || EPI == EPI_ARGMAX || EPI == EPI_QKV) {
            if (tid < DFL_MAX_ROWS) {
                float r = 1.f;
                if (a.ssq_in) {
                    float ss = 0.f;
                    for (int p = 0; p < a.ssq_parts; ++p) ss += a.ssq_in[p * DFL_MAX_ROWS + tid];
                    r = 1.0f / sqrtf(ss * a.inv_width + a.eps);
                }
                s_rstd[tid] = r;
            }
            consumer_bar();
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
                            const size_t o = (size_t)t * a.ldo + n0 + r;
                            v += a.out[o];
                            a.out[o] = v;
                            if (a.tap_out) store_act(a.tap_out, a.tap_type, a.ld_tap, t, n0 + r, v);
                        }
                        ss = fmaf(v, v, ss);
                        const float wn = a.w_next ? a.w_next[n0 + r] : 1.f;
                        store_act(a.xn_out, a.xn_type, a.ldo, t, n0 + r, v * wn);
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
                const int hd = qe.hd, hpt = GEMM_BN / hd, per = hd / 32;
                const int h_first = tile * hpt;
                for (int item = warp; item < DFL_MAX_ROWS * hpt; item += GEMM_CONSUMERS) {
                    const int t = item / hpt, hi = item % hpt;
                    if (t < r0 || t >= r0 + nrows) continue;
                    const int h = h_first + hi;
                    const bool is_q = h < qe.n_q, is_k = !is_q && h < qe.n_q + qe.n_kv;
                    float v[4];
                    for (int m = 0; m < per; ++m)
                        v[m] = ctile[t * GEMM_BN + hi * hd + lane + 32 * m] * s_rstd[t];
                    if (is_q || is_k) {
                        const float* nw = is_q ? qe.q_norm : qe.k_norm;
                        float ss = 0.f;
                        for (int m = 0; m < per; ++m) ss = fmaf(v[m], v[m], ss);
                        ss = warp_sum(ss);
                        const float inv = 1.0f / sqrtf(ss / (float)hd + a.eps);
                        for (int m = 0; m < per; ++m) v[m] = v[m] * inv * nw[lane + 32 * m];
                        // rotate-half: element i pairs with i + hd/2 (same lane, m + per/2)
                        const float* cs = qe.rope_cos + t * (hd / 2);
                        const float* sn = qe.rope_sin + t * (hd / 2);
                        float rr[4];
                        for (int m = 0; m < per / 2; ++m) {
                            const int i = lane + 32 * m;
                            rr[m] = v[m] * cs[i] - v[m + per / 2] * sn[i];
                            rr[m + per / 2] = v[m + per / 2] * cs[i] + v[m] * sn[i];
                        }
                        for (int m = 0; m < per; ++m) v[m] = rr[m];
                    }
                    if (is_q) {
                        const size_t base = ((size_t)h * DFL_MAX_ROWS + t) * hd;   // [n_q][16][hd]
                        for (int m = 0; m < per; ++m) store_xt(qe.q_out, qe.q_type, base + lane + 32 * m, v[m]);
                        continue;
                    }
                    const int pos = a.st->fwd_pos0 + t;
                    if (pos < 0 || pos >= qe.max_seq) {
                        if (lane == 0) set_error(a.st, DERR_INDEX, pos);
                        continue;
                    }
                    const int kh = is_k ? h - qe.n_q : h - qe.n_q - qe.n_kv;
                    void* cache = is_k ? qe.k_cache : qe.v_cache;
                    const size_t base = ((size_t)kh * qe.cap + pos) * hd;
                    for (int m = 0; m < per; ++m) store_xt(cache, qe.c_type, base + lane + 32 * m, v[m]);
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
}

template <int WF, int EPI>
int launch_one(const GemmMaps& maps, const GemmArgs& args, int grid, cudaStream_t stream) {
    using CFG = GemmCfg<WF>;
    constexpr size_t smem = 1024 + (size_t)CFG::STAGES * CFG::CHUNK * (GEMM_STAGE_W + CFG::XB + CFG::SB) +
                            DFL_MAX_ROWS * GEMM_BN * 4 + 2 * CFG::STAGES * 8 + 64;
    static_assert(smem <= 232448, "GEMM shared memory exceeds the per-block limit");
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<WF, EPI>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) return (int)e;
        attr_set = true;
    }
    return (int)launch_k(gemm_skinny_kernel<WF, EPI>, dim3(grid), dim3(GEMM_THREADS), smem, stream,
                         maps, args);
}

}  // namespace

int launch_gemm(int wfmt, int epi, int xt, const GemmMaps& maps, const GemmArgs& args,
                int grid, cudaStream_t stream) {
    (void)xt;
    if (wfmt == WF_BF16) {
        switch (epi) {
            case EPI_STORE: return launch_one<WF_BF16, EPI_STORE>(maps, args, grid, stream);
            case EPI_RESID: return launch_one<WF_BF16, EPI_RESID>(maps, args, grid, stream);
            case EPI_SWIGLU: return launch_one<WF_BF16, EPI_SWIGLU>(maps, args, grid, stream);
            case EPI_ARGMAX: return launch_one<WF_BF16, EPI_ARGMAX>(maps, args, grid, stream);
            case EPI_QKV: return launch_one<WF_BF16, EPI_QKV>(maps, args, grid, stream);
            case EPI_NORMOUT: return launch_one<WF_BF16, EPI_NORMOUT>(maps, args, grid, stream);
        }
    } else if (wfmt == WF_INT4) {
        switch (epi) {
            case EPI_STORE: return launch_one<WF_INT4, EPI_STORE>(maps, args, grid, stream);
            case EPI_RESID: return launch_one<WF_INT4, EPI_RESID>(maps, args, grid, stream);
            case EPI_SWIGLU: return launch_one<WF_INT4, EPI_SWIGLU>(maps, args, grid, stream);
            case EPI_QKV: return launch_one<WF_INT4, EPI_QKV>(maps, args, grid, stream);
        }
    } else if (wfmt == WF_F32) {
        switch (epi) {
            case EPI_STORE: return launch_one<WF_F32, EPI_STORE>(maps, args, grid, stream);
            case EPI_RESID: return launch_one<WF_F32, EPI_RESID>(maps, args, grid, stream);
            case EPI_SWIGLU: return launch_one<WF_F32, EPI_SWIGLU>(maps, args, grid, stream);
            case EPI_ARGMAX: return launch_one<WF_F32, EPI_ARGMAX>(maps, args, grid, stream);
            case EPI_QKV: return launch_one<WF_F32, EPI_QKV>(maps, args, grid, stream);
            case EPI_NORMOUT: return launch_one<WF_F32, EPI_NORMOUT>(maps, args, grid, stream);
        }
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace dfl
