// Skinny weight-streaming GEMM for the <= 16 rows of one DFlash forward.
//
// By page: the drafter's projections stream each weight once for all the
// block's rows ("feat: DFlash2 block-diffusion drafter for Qwen 3.8", first
// commit: the multi-x BF16 GEMV; third commit: projections quantised at
// load into the multi-x INT4 format); the verify runs the 1+m rows in one
// forward ("dflash: the chain verify builds pipelined ...", fourth commit:
// the [1, 1+m] verify forward; "[RFC] DFlash", "Key Implementation Details",
// Phase 3); the residual stream stays fp32 (DFlash2 page, first commit: the
// o/down projections overflow fp16 on outlier channels).  A row's result
// never depends on how many rows the call has (the RFC author's reply, the
// aside on a quantised-matmul kernel switch at batch 6 that flipped argmaxes).
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
//  * a tile whose k-range is split across CTAs is finished by its owner,
//    the CTA whose range reaches the tile's first k-block (it gets there
//    last): the others store their parts and publish them on the tile's
//    counter without waiting, the owner waits (bounded) for them and sums
//    the parts in CTA order: the result of a row never depends on how many
//    rows the forward has, on timing, or on the other rows (batch
//    invariance);
//  * fused epilogues: store fp32, residual add (+ tap copy), SwiGLU of
//    paired gate/up tiles, LM-head argmax with packed 64-bit atomicMax.
//
// Every mbarrier wait is bounded; an expired wait sets the device error
// word, stops new copies and drains the copies already issued.

#include <cstdlib>
#include <mutex>
#include <vector>

#include "gemm_dev.cuh"

namespace dfl {

long long g_launches = 0;

void set_carveout_once(const void* kern) {
    if (DFL_SMEM_CARVEOUT < 0) return;
    static std::mutex mu;
    static std::vector<const void*> done;
    std::lock_guard<std::mutex> lock(mu);
    for (const void* k : done)
        if (k == kern) return;
    // a hint: on failure clear the error so it is not reported by a later check
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             DFL_SMEM_CARVEOUT) != cudaSuccess)
        (void)cudaGetLastError();
    done.push_back(kern);
}
bool g_pdl = [] {
    const char* e = getenv("DFLASH_PDL");
    return !(e && e[0] == '0');
}();

namespace {

// Build knob for latency studies: per-CTA %globaltimer stamps of the last
// launch (entry, weights issued, producer released, consumers released,
// first stage landed, last k-block done, tile finishes done, exit).
#ifdef DFL_GEMM_TIMESTAMPS
__device__ unsigned long long g_gemm_ts[256][8];
#define GEMM_TS(i) (g_gemm_ts[blockIdx.x & 255][(i)] = globaltimer_ns())
#else
#define GEMM_TS(i) ((void)0)
#endif

using gdev::consumer_bar;
using gdev::range_start;
using gdev::mma_kblock;
using gdev::finish_tile;

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
    if (threadIdx.x == 0) GEMM_TS(0);
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
            // The weights do not depend on earlier kernels: the first
            // DFL_GEMM_PREWAIT stages take them before waiting for the
            // predecessor (programmatic dependent launch), then their
            // activation tiles follow.
            constexpr int PRE = DFL_GEMM_PREWAIT < STAGES ? DFL_GEMM_PREWAIT : STAGES;
            long long pu[STAGES];
            int pl[STAGES];
            int npre = 0;
            long long u = u0;
            while (u < u1 && npre < PRE) {
                const int len = chunk_len(u);
                pu[npre] = u;
                pl[npre] = len;
                mbar_arrive_expect_tx(&full[npre], len * KB_BYTES);
                for (int j = 0; j < len; ++j) load_w(u + j, npre, j);
                u += len;
                ++npre;
            }
            GEMM_TS(1);
            pdl_wait();
            GEMM_TS(2);
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
    if (tid == 0) GEMM_TS(3);
    bool first_seen = false;
    gdev::compute_rstd<EPI>(a, s_rstd, tid);   // read after the first tile's barrier
    int stage = 0;
    uint32_t phase = 0;
    float acc[8], accl[8];   // hi and lo planes' accumulators, added at the tile's finish

    for (long long u = u0; u < u1;) {
        const int len = chunk_len(u);
        const int tile = (int)(u / a.kb), k = (int)(u % a.kb);
        if (k == 0 || u == u0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = accl[i] = 0.f;
        }
        bool ok = false;
        if (!s_flags[0]) {
            ok = mbar_wait_bounded(&full[stage], phase);
            if (!ok) {
                s_flags[0] = 1;
                set_error(a.st, DERR_TIMEOUT, 101);
            }
            if (tid == 0 && !first_seen) {
                first_seen = true;
                GEMM_TS(4);
            }
        }
        if (ok) {
            for (int jb = 0; jb < len; ++jb) {
            const uint8_t* Wt = Ws + (stage * CHUNK + jb) * GEMM_STAGE_W;
            const uint8_t* Xt = Xs + (stage * CHUNK + jb) * XB;
            const uint8_t* Sb = Ss + (stage * CHUNK + jb) * SB;
            mma_kblock<WF, EPI>(Wt, Xt, Sb, a, warp, lane, acc, accl);
            }   // k-blocks of the stage
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (tid == 0 && ok) s_flags[2] = s_flags[2] + 1;   // stages seen complete
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        u += len;

        if (!(k + len == a.kb || u == u1)) continue;
        if (tid == 0 && u == u1) GEMM_TS(5);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += accl[i];
        finish_tile<WF, EPI>(a, tile, acc, ctile, s_flags, s_rstd, U, G, blockIdx.x, warp, lane,
                             tid);
    }
    if (tid == 0) GEMM_TS(7);
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

#ifdef DFL_GEMM_TIMESTAMPS
extern "C" int dfl_gemm_timestamps(unsigned long long* out) {
    return (int)cudaMemcpyFromSymbol(out, g_gemm_ts, sizeof(g_gemm_ts));
}
#endif

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
            case EPI_ARGMAX: return launch_one<WF_INT4, EPI_ARGMAX>(maps, args, grid, stream);
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
