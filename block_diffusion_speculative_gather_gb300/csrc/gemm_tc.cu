// Dense many-row GEMM on tcgen05 (see gemm_tc.cuh).
//
// One CTA per 128 x BN output tile (BN 256, or 128 where that balances
// the waves over the SMs better, or as the caller fixes it) and k-split,
// 128 threads.  Thread 0 is the TMA
// producer: a ring of k-blocks (the x tile [128][64], its low plane when
// x_split, and the w tile [256][64], bf16 or all f16, 128-byte swizzled,
// K-major).  Thread 32 issues tcgen05.mma (M 128, N BN, K 16, f32
// accumulators in BN tensor-memory columns) four times per k-block (twice
// that with the low plane) and commits each stage back to the producer
// through its "empty" mbarrier.  After the last k-block every warp reads
// its 32 tensor-memory lanes (rows) with tcgen05.ld and stores fp32 rows;
// rows past M and columns past N are not stored (TMA fills the missing x
// and w rows with zeros).  Every wait is bounded; a wait that times out
// sets the device error word, and the MMA thread still commits, so the
// tensor memory is freed only after the MMAs it issued have finished.
// Split-K (few rows: the many-sequence round): the k-blocks of a tile are
// cut into `splits` contiguous ranges in split order; each split stores its
// fp32 partial rows into its own slab, and a reduce kernel launched right
// after adds the slabs in split order (coalesced, one pass over them) --
// or, with keep_parts, the row kernel that consumes the output does -- so a
// row's result is the same whatever the number of rows.  The argmax
// epilogue (the LM head of that round) keeps per row the packed (orderable
// logit, ~column) key of its largest column and folds it into the row's key
// with atomicMax (lowest column on ties).  The SwiGLU form (the fused
// gate/up projection) loads half a tile of gate rows and the matching half
// of up rows and writes silu(gate) * up as hi/lo planes.

#include "gemm_tc.cuh"
#include "rows_dev.cuh"
#include "tc_dev.cuh"

namespace dfl {

namespace {

// Ring stages whose weight tiles may go out before the dependency wait
// (build knob; only for weights no earlier kernel writes).
#ifndef DFL_DENSE_PREWAIT
#define DFL_DENSE_PREWAIT 8
#endif

__device__ __forceinline__ void dense_error(int* err, int site) {
    if (atomicCAS(&err[0], 0, DERR_TIMEOUT) == 0) err[1] = site;
}

// Eight consecutive values as hi/lo planes from element i (16-byte
// aligned): the rounding of store_hilo, packed into one 16-byte store per
// plane.
__device__ __forceinline__ void store_hilo8(void* hi, void* lo, size_t i, const float* v, int f16) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (f16) {
            const __half a = __float2half_rn(v[2 * q]), b = __float2half_rn(v[2 * q + 1]);
            const __half la = __float2half_rn(v[2 * q] - __half2float(a));
            const __half lb = __float2half_rn(v[2 * q + 1] - __half2float(b));
            h[q] = (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
            l[q] = (uint32_t)__half_as_ushort(la) | ((uint32_t)__half_as_ushort(lb) << 16);
        } else {
            const __nv_bfloat16 a = __float2bfloat16_rn(v[2 * q]), b = __float2bfloat16_rn(v[2 * q + 1]);
            const __nv_bfloat16 la = __float2bfloat16_rn(v[2 * q] - __bfloat162float(a));
            const __nv_bfloat16 lb = __float2bfloat16_rn(v[2 * q + 1] - __bfloat162float(b));
            h[q] = (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
            l[q] = (uint32_t)__bfloat16_as_ushort(la) | ((uint32_t)__bfloat16_as_ushort(lb) << 16);
        }
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(hi) + i) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(lo) + i) = make_uint4(l[0], l[1], l[2], l[3]);
}

template <bool SPLIT, int BN>
struct DenseCfg {
    static constexpr uint32_t XB = DT_BM * 128;                    // x tile bytes (64 k)
    static constexpr uint32_t WB = BN * 128;                       // w tile bytes
    static constexpr uint32_t STAGE = (SPLIT ? 2 : 1) * XB + WB;
    static constexpr int STAGES = (int)((192u * 1024u) / STAGE);   // 192 KB of ring
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + (2 * STAGES + 1) * 8 + 16;
};

template <bool SPLIT, bool F16, int BN>
__global__ void __launch_bounds__(128, 1)
gemm_dense_kernel(const __grid_constant__ DenseMaps maps, const DenseArgs a) {
    using CFG = DenseCfg<SPLIT, BN>;
    constexpr int STAGES = CFG::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + STAGES * CFG::STAGE);
    uint64_t* empty = full + STAGES;
    uint64_t* done = empty + STAGES;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    __shared__ int s_fail;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * DT_BM, n0 = blockIdx.y * BN;
    // this CTA's k-blocks: split z of Z takes [nkb z / Z, nkb (z + 1) / Z)
    const int Z = a.splits > 1 ? a.splits : 1, z = blockIdx.z;
    const int kb_lo = (int)((long long)(a.K / DT_BK) * z / Z);
    const int nkb = (int)((long long)(a.K / DT_BK) * (z + 1) / Z) - kb_lo;
    const int seg = n0 >= a.n_seg1 ? 2 : n0 >= a.n_seg0 ? 1 : 0;
    const int wrow = n0 - (seg == 2 ? a.n_seg1 : seg == 1 ? a.n_seg0 : 0);

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
        s_fail = 0;
        tma_prefetch_desc(&maps.x);
        if (SPLIT) tma_prefetch_desc(&maps.x_lo);
        tma_prefetch_desc(&maps.w[seg]);
        if (a.swiglu) tma_prefetch_desc(&maps.w[a.up_map]);
    }
    constexpr uint32_t TCOLS = BN <= 128 ? 128u : 256u;   // a power of two >= BN
    if (warp == 1) tc::tmem_alloc(s_tmem, TCOLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *s_tmem;

    // weight tile(s) of k-block kb into its stage's w part
    auto load_w = [&](int kb, uint8_t* wst, uint64_t* bar) {
        const int kx = (kb_lo + kb) * DT_BK;
        if (a.swiglu) {   // BN / 2 gate rows, then the matching BN / 2 up rows
            constexpr int HB = BN / 2;
            const int t = n0 / BN;
            tma_load_2d(wst, &maps.w[0], bar, kx, HB * t);
            tma_load_2d(wst + HB * 128, &maps.w[a.up_map], bar, kx, a.up_row + HB * t);
        } else {
            constexpr int NB = BN / DT_WBOX, TAIL = BN % DT_WBOX;
            static_assert(TAIL == 0 || TAIL == DT_WTAIL, "tile width: whole weight boxes and one tail box");
#pragma unroll
            for (int b = 0; b < NB; ++b)
                tma_load_2d(wst + b * DT_WBOX * 128, &maps.w[seg], bar, kx, wrow + b * DT_WBOX);
            if (TAIL) tma_load_2d(wst + NB * DT_WBOX * 128, &maps.w_tail, bar, kx, wrow + NB * DT_WBOX);
        }
    };
    const int pre = nkb < STAGES ? nkb : STAGES;
    // weights no earlier kernel writes: the first stages' weight tiles (up
    // to DFL_DENSE_PREWAIT of them) go out before the dependency wait
    const int pre_w = a.w_ready ? (pre < DFL_DENSE_PREWAIT ? pre : DFL_DENSE_PREWAIT) : 0;
    auto first_w = [&](int lo, int hi) {
        for (int kb = lo; kb < hi; ++kb) {
            mbar_arrive_expect_tx(&full[kb], CFG::STAGE);
            load_w(kb, ring + kb * CFG::STAGE + (SPLIT ? 2 : 1) * CFG::XB, &full[kb]);
        }
    };
    if (threadIdx.x == 0) first_w(0, pre_w);
    pdl_wait();   // x (and without w_ready the weights) may come from the previous kernel

    if (threadIdx.x == 0) {   // ---- TMA producer
        first_w(pre_w, pre);
        for (int kb = 0; kb < pre; ++kb) {
            uint8_t* st = ring + kb * CFG::STAGE;
            const int kx = (kb_lo + kb) * DT_BK;
            tma_load_2d(st, &maps.x, &full[kb], kx, a.m_off + m0);
            if (SPLIT) tma_load_2d(st + CFG::XB, &maps.x_lo, &full[kb], kx, a.m_off + m0);
        }
        for (int kb = pre; kb < nkb; ++kb) {
            const int s = kb % STAGES;
            if (!mbar_wait_bounded(&empty[s], (uint32_t)((kb / STAGES - 1) & 1))) {
                s_fail = 1;
                dense_error(a.err, 300);
                break;
            }
            uint8_t* st = ring + s * CFG::STAGE;
            const int kx = (kb_lo + kb) * DT_BK;
            mbar_arrive_expect_tx(&full[s], CFG::STAGE);
            tma_load_2d(st, &maps.x, &full[s], kx, a.m_off + m0);
            if (SPLIT) tma_load_2d(st + CFG::XB, &maps.x_lo, &full[s], kx, a.m_off + m0);
            load_w(kb, st + (SPLIT ? 2 : 1) * CFG::XB, &full[s]);
        }
    } else if (threadIdx.x == 32) {   // ---- MMA issuer
        constexpr uint32_t ID = F16 ? tc::idesc_f16_f32(DT_BM, BN) : tc::idesc_bf16_f32(DT_BM, BN);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % STAGES;
            if (!mbar_wait_bounded(&full[s], (uint32_t)((kb / STAGES) & 1))) {
                s_fail = 1;
                dense_error(a.err, 301);
                break;
            }
            tc::fence_after_sync();
            const uint8_t* st = ring + s * CFG::STAGE;
            const uint8_t* wt = st + (SPLIT ? 2 : 1) * CFG::XB;
#pragma unroll
            for (int k = 0; k < DT_BK / 16; ++k) {
                const uint64_t bd = tc::desc_sw128(wt + 32 * k);
                tc::mma_f16(tm, tc::desc_sw128(st + 32 * k), bd, ID, (kb | k) != 0 ? 1u : 0u);
                if (SPLIT) tc::mma_f16(tm, tc::desc_sw128(st + CFG::XB + 32 * k), bd, ID, 1u);
            }
            tc::commit(&empty[s]);   // the stage is free once these MMAs are done
        }
        tc::commit(done);   // always: the epilogue (and the free) waits on it
    }
    __syncwarp();

    // ---- epilogue: warp w holds rows m0 + 32 w + lane in its tensor-memory lanes
    bool ok = mbar_wait_bounded(done, 0);
    ok = __syncthreads_and(ok) != 0;   // the barrier also orders the s_fail writes
    ok = ok && s_fail == 0;
    tc::fence_after_sync();
    const int row = m0 + 32 * warp + lane;
    if (ok && Z > 1) {
        // split z's partial rows into slab z of part ([Z][m tiles * 128][n tiles * BN]);
        // the reduce kernel that follows adds the slabs in split order
        const size_t ldp = (size_t)gridDim.y * BN;
        float* mypart = a.part + ((size_t)z * gridDim.x * DT_BM + row) * ldp + n0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tc::ld_x32(tm + ((uint32_t)(32 * warp) << 16) + 32 * c, v);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                __stcg(reinterpret_cast<float4*>(mypart + 32 * c + i),
                       make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        }
    }
    const bool last = Z == 1;
    if (ok && last && a.swiglu) {
        // columns 0..BN/2-1 gate, BN/2..BN-1 up: silu(gate) * up into the
        // hi/lo planes at columns (BN / 2) t.. of the row
        constexpr int HB = BN / 2;
        const int t = n0 / BN;
#pragma unroll 1
        for (int c = 0; c < HB / 32; ++c) {
            float g[32], u[32];
            tc::ld_x32(tm + ((uint32_t)(32 * warp) << 16) + 32 * c, g);
            tc::ld_x32(tm + ((uint32_t)(32 * warp) << 16) + HB + 32 * c, u);
            if (row < a.M) {
#pragma unroll
                for (int i = 0; i < 32; ++i) g[i] = swiglu(g[i], u[i]);
                const size_t base = (size_t)row * a.act_ld + (size_t)HB * t + 32 * c;
#pragma unroll
                for (int i = 0; i < 32; i += 8) store_hilo8(a.act_hi, a.act_lo, base + i, g + i, a.f16);
            }
        }
    } else if (ok && last) {
        unsigned long long best = 0ull;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tc::ld_x32(tm + ((uint32_t)(32 * warp) << 16) + 32 * c, v);
            const int col = n0 + 32 * c;
            if (row < a.M && col < a.N) {
                if (a.amax) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (col + i < a.N) {
                            const unsigned long long key = argmax_key(v[i], col + i);
                            best = key > best ? key : best;
                        }
                }
                if (a.y) {
                    float* dst = a.y + (size_t)row * a.ldy + col;
                    if (col + 32 <= a.N) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col + i < a.N) dst[i] = v[i];
                    }
                }
            }
        }
        if (a.amax && row < a.M) atomicMax(a.amax + row, best);
    } else if (!ok && threadIdx.x == 0 && s_fail == 0) {
        dense_error(a.err, 302);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tm, TCOLS);
}

// y = sum over the split slabs in split order (z = 0, 1, ...), four
// consecutive columns per thread: coalesced, every load of a thread in
// flight at once.
__global__ void dense_split_reduce_kernel(const float* __restrict__ part, int Z, int M, int N,
                                          size_t slab, size_t ldp, float* __restrict__ y, int ldy) {
    pdl_trigger();
    pdl_wait();
    const long long n4 = N / 4, total = (long long)M * n4;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int row = (int)(e / n4), col = (int)(e % n4) * 4;
        const float* src = part + (size_t)row * ldp + col;
        float4 v[8];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int z0 = 0; z0 < Z; z0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (z0 + j < Z) v[j] = __ldcg(reinterpret_cast<const float4*>(src + (size_t)(z0 + j) * slab));
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (z0 + j < Z) {
                    acc.x += v[j].x;
                    acc.y += v[j].y;
                    acc.z += v[j].z;
                    acc.w += v[j].w;
                }
        }
        *reinterpret_cast<float4*>(y + (size_t)row * ldy + col) = acc;
    }
}

template <bool SPLIT, bool F16, int BN>
int launch_one(const DenseMaps& maps, const DenseArgs& a, cudaStream_t s) {
    constexpr size_t smem = DenseCfg<SPLIT, BN>::SMEM;
    static_assert(smem <= 232448, "dense GEMM shared memory exceeds the per-block limit");
    static bool set = false;
    if (!set) {
        const cudaError_t e = cudaFuncSetAttribute(gemm_dense_kernel<SPLIT, F16, BN>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        set = true;
    }
    const dim3 grid((unsigned)((a.M + DT_BM - 1) / DT_BM), (unsigned)((a.N + BN - 1) / BN),
                    (unsigned)(a.splits > 1 ? a.splits : 1));
    int e = (int)launch_k(gemm_dense_kernel<SPLIT, F16, BN>, grid, dim3(128), smem, s, maps, a);
    if (e || a.splits <= 1 || a.keep_parts) return e;
    const size_t ldp = (size_t)grid.y * BN, slab = (size_t)grid.x * DT_BM * ldp;
    const long long items = (long long)a.M * (a.N / 4);
    long long blocks = (items + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    return (int)launch_k(dense_split_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                         (const float*)a.part, a.splits, a.M, a.N, slab, ldp, a.y, a.ldy);
}

template <bool SPLIT, bool F16>
int launch_bn(const DenseMaps& maps, const DenseArgs& a, cudaStream_t s) {
    // one CTA per SM; a 128-column tile costs about 0.8 of a 256-column one
    // (measured: the x tile streams once per column tile either way), so
    // the narrow tile wins only where it saves a whole wave
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            sms = 1;
    }
    if (a.bn == 128) return launch_one<SPLIT, F16, 128>(maps, a, s);
    if (a.bn == 256) return launch_one<SPLIT, F16, 256>(maps, a, s);
    const long long mt = (a.M + DT_BM - 1) / DT_BM;
    const long long w256 = (mt * ((a.N + 255) / 256) + sms - 1) / sms;
    const long long w128 = (mt * ((a.N + 127) / 128) + sms - 1) / sms;
    // a 160-column tile's stage is bound by its copies (32 KB of x planes +
    // 20 KB of weights against 64 KB for 256 columns): about 0.8 of a
    // 256-column one too; it wins where it takes a wave fewer than 128
    // columns and the same as 256 (o and down over 1024 rows: 128 tiles on
    // 152 SMs, against 160 and 80)
    if (maps.has_tail && a.N % 160 == 0 && !a.swiglu && !a.amax && a.splits <= 1) {
        const long long w160 = (mt * (a.N / 160) + sms - 1) / sms;
        if (w160 * 4 < w256 * 5 && w160 <= w128) return launch_one<SPLIT, F16, 160>(maps, a, s);
    }
    if (w128 * 4 < w256 * 5) return launch_one<SPLIT, F16, 128>(maps, a, s);
    return launch_one<SPLIT, F16, 256>(maps, a, s);
}

}  // namespace

size_t dense_split_floats(int M, int N, int splits, int bn) {
    return (size_t)dense_tiles(M, N, bn) * (size_t)(splits > 1 ? splits : 1) * DT_BM * bn;
}

int dense_tiles(int M, int N, int bn) { return ((M + DT_BM - 1) / DT_BM) * ((N + bn - 1) / bn); }

void dense_part_layout(int M, int N, int bn, size_t* slab, size_t* ldp) {
    *ldp = (size_t)((N + bn - 1) / bn) * bn;
    *slab = (size_t)((M + DT_BM - 1) / DT_BM) * DT_BM * *ldp;
}

size_t dense_smem(bool split) { return split ? DenseCfg<true, DT_BN>::SMEM : DenseCfg<false, DT_BN>::SMEM; }

int launch_dense(const DenseMaps& maps, const DenseArgs& a, cudaStream_t s) {
    const bool kept = a.splits > 1 && a.keep_parts;
    // the SwiGLU epilogue stores 8 plane elements (16 bytes) at a time
    if (a.swiglu && ((a.bn != 128 && a.bn != 256) || a.splits > 1 || a.amax || a.N % a.bn || !a.act_hi || !a.act_lo ||
                     ((reinterpret_cast<uintptr_t>(a.act_hi) | reinterpret_cast<uintptr_t>(a.act_lo)) & 15) ||
                     a.act_ld % 8 || a.act_ld < a.N / 2 || a.up_map < 0 || a.up_map > 2 || a.up_row < 0))
        return (int)cudaErrorInvalidValue;
    if (a.M < 1 || a.N < 1 || a.K < DT_BK || a.K % DT_BK || (a.y && (a.ldy < a.N || a.ldy % 4)) ||
        (!a.y && !a.amax && !kept && !a.swiglu) || a.n_seg0 % DT_BN ||
        (a.n_seg1 < a.N && (a.n_seg1 % DT_BN || a.n_seg1 < a.n_seg0)) || a.m_off < 0 ||
        (a.bn != 0 && a.bn != 128 && a.bn != 256) || a.splits > a.K / DT_BK ||
        (a.splits > 1 && (a.bn == 0 || !a.part || (!a.y && !kept) || a.amax || a.N % 4)))
        return (int)cudaErrorInvalidValue;
    if (a.f16) return a.x_split ? launch_bn<true, true>(maps, a, s) : launch_bn<false, true>(maps, a, s);
    return a.x_split ? launch_bn<true, false>(maps, a, s) : launch_bn<false, false>(maps, a, s);
}

}  // namespace dfl
