// Persistent round kernel (see round.cuh).
//
// One CTA per SM, launched cooperatively so that every CTA is resident and
// grid barriers are safe.  Warp 8 is the producer: it walks the program's
// GEMM phases in order and streams their weight tiles into a shared-memory
// ring with TMA.  Weights never depend on earlier phases, so the producer
// fills the ring with the next GEMM's tiles while the consumers are still
// finishing the current phase, running attention or waiting at a barrier;
// only the activation tiles of a GEMM wait until the barrier before it has
// completed.  Warps 0..7 are the consumers: they run every phase (GEMM
// tiles with their fused epilogues, attention chunks, the chunk combine,
// row preparation, acceptance) and meet at a grid barrier between phases.
//
// Every wait is bounded: a barrier, a ring slot or a copy that does not
// arrive in time sets the device error word and the CTA leaves the program;
// the producer waits (bounded) for the copies it issued before it exits.

#include "attention_dev.cuh"
#include "gemm_dev.cuh"
#include "kernels_dev.cuh"
#include "round.cuh"

namespace dfl {

namespace {

using gdev::consumer_bar;
using gdev::range_start;

constexpr int RXB = GemmCfg<WF_BF16>::XB;              // 4 KB: hi/lo activation tile
constexpr uint32_t RKB = GEMM_STAGE_W + RXB;            // bytes one k-block brings
constexpr int RSLOTS = ROUND_STAGES * ROUND_CHUNK;
constexpr uint64_t BARRIER_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's view of global memory (made visible by a barrier)
// before its later TMA reads of it.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

struct ConsumerBar {
    __device__ __forceinline__ void operator()() const { consumer_bar(); }
};

struct GroupBar {   // named barrier `id` over `n` threads
    int id, n;
    __device__ __forceinline__ void operator()() const {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
    }
};

// k-blocks in the ring stage that starts at unit u (never past the tile or
// the CTA's range).
__device__ __forceinline__ int chunk_len(long long u, long long u1, int kb) {
    long long n = ROUND_CHUNK;
    if (u1 - u < n) n = u1 - u;
    const long long to_tile_end = kb - (u % kb);
    if (to_tile_end < n) n = to_tile_end;
    return (int)n;
}

// Records a timeout at `site` and tells every CTA to leave the program.
__device__ __forceinline__ void abort_all(const RoundCall& rc, int site) {
    set_error(rc.st, DERR_TIMEOUT, site);
    atomicExch(rc.bar_count + 1, 1u);
}

// Waits (bounded) until `target` barrier arrivals are counted; false on
// timeout or when another CTA has aborted the program.
__device__ __forceinline__ bool wait_count(const RoundCall& rc, unsigned target) {
    if (ld_acquire_u32(rc.bar_count) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ld_acquire_u32(rc.bar_count) >= target) return true;
        if (*reinterpret_cast<volatile unsigned*>(rc.bar_count + 1) != 0) return false;
        if (globaltimer_ns() - t0 > BARRIER_LIMIT_NS) {
            abort_all(rc, 400);
            return false;
        }
    }
}

// Grid barrier of the consumer warps (256 threads of every CTA).
__device__ __forceinline__ bool grid_sync(const RoundCall& rc, unsigned target, volatile int* s_flags,
                                          int tid) {
    consumer_bar();
    if (tid == 0) {
        __threadfence();
        red_release_add_u32(rc.bar_count, 1u);
        if (!wait_count(rc, target)) s_flags[0] = 1;
        __threadfence();
    }
    consumer_bar();
    return s_flags[0] == 0;
}

// ------------------------------------------------------------------ producer

// What the producer needs of a GEMM phase, read once into registers (the
// phase itself lives in global memory, and every TMA issue is a memory
// clobber that would force its fields to be re-read).
struct ProdPhase {
    const CUtensorMap* w[3];
    const CUtensorMap* x;
    int kb, n_seg, seg0, seg1, swiglu;
};

// Weight tile of GEMM unit u into ring slot `slot`.
__device__ __forceinline__ void load_w(const ProdPhase& q, long long u, uint8_t* Ws, int slot,
                                       uint64_t* bar) {
    const int tile = (int)(u / q.kb), k = (int)(u % q.kb);
    uint8_t* wdst = Ws + slot * GEMM_STAGE_W;
    const int wx = k * 64;
    if (q.swiglu) {
        tma_load_2d(wdst, q.w[0], bar, wx, tile * 64);
        tma_load_2d(wdst + 64 * 128, q.w[1], bar, wx, tile * 64);
    } else {
        int row = tile * GEMM_BN, seg = 0;
        if (q.n_seg > 1 && row >= q.seg0) {
            row -= q.seg0;
            seg = 1;
            if (q.n_seg > 2 && row >= q.seg1) {
                row -= q.seg1;
                seg = 2;
            }
        }
        tma_load_2d(wdst, q.w[seg], bar, wx, row);
    }
}

__device__ __forceinline__ void load_x(const ProdPhase& q, long long u, uint8_t* Xs, int slot,
                                       uint64_t* bar) {
    tma_load_2d(Xs + slot * RXB, q.x, bar, (int)(u % q.kb) * 64, 0);
}

__device__ void producer(const RoundCall& rc, uint8_t* Ws, uint8_t* Xs, uint64_t* full,
                         uint64_t* empty, volatile int* s_flags) {
    const int G = gridDim.x, cta = blockIdx.x;
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    struct Pending {
        long long u;
        int len, stage;
    } pend[ROUND_STAGES];
    int npend = 0;
    for (int p = 0; p < rc.n_phases && !s_flags[0]; ++p) {
        const Phase* P = rc.phases + p;
        if (P->kind != PH_GEMM) continue;
        ProdPhase q;
        q.kb = P->g.kb;
        q.n_seg = P->g.n_seg;
        q.seg0 = P->g.seg_rows[0];
        q.seg1 = P->g.seg_rows[1];
        q.swiglu = P->epi == EPI_SWIGLU;
        for (int i = 0; i < 3; ++i) q.w[i] = &P->maps.w[i];
        q.x = &P->maps.x;
        const int kb = q.kb;
        const int n_tiles = P->g.n_tiles;
        const unsigned bars_before = (unsigned)P->bars_before;
        for (int i = 0; i < q.n_seg; ++i) tma_prefetch_desc(q.w[i]);
        tma_prefetch_desc(q.x);
        const long long U = (long long)n_tiles * kb;
        const long long u0 = range_start(cta, U, G), u1 = range_start(cta + 1, U, G);
        const unsigned target = (unsigned)G * bars_before;
        bool x_ready = ld_acquire_u32(rc.bar_count) >= target;
        if (x_ready) fence_proxy_async_global();
        auto release_pending = [&]() -> bool {
            if (!wait_count(rc, target)) return false;
            fence_proxy_async_global();
            for (int i = 0; i < npend; ++i)
                for (int j = 0; j < pend[i].len; ++j)
                    load_x(q, pend[i].u + j, Xs, pend[i].stage * ROUND_CHUNK + j,
                           &full[pend[i].stage]);
            npend = 0;
            x_ready = true;
            return true;
        };
        for (long long u = u0; u < u1;) {
            if (s_flags[0]) break;
            // every slot holds this phase's tiles waiting for their activations:
            // they can only drain once the barrier before the phase completes
            if (!x_ready && npend == ROUND_STAGES && !release_pending()) {
                s_flags[0] = 1;
                break;
            }
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u)) {
                s_flags[0] = 1;
                abort_all(rc, 401);
                break;
            }
            if (s_flags[0]) break;
            const int len = chunk_len(u, u1, kb);
            mbar_arrive_expect_tx(&full[stage], (uint32_t)len * RKB);
            for (int j = 0; j < len; ++j)
                load_w(q, u + j, Ws, stage * ROUND_CHUNK + j, &full[stage]);
            if (x_ready) {
                for (int j = 0; j < len; ++j)
                    load_x(q, u + j, Xs, stage * ROUND_CHUNK + j, &full[stage]);
            } else {
                pend[npend++] = {u, len, stage};
            }
            u += len;
            ++issued;
            if (++stage == ROUND_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!s_flags[0] && npend > 0 && !release_pending()) s_flags[0] = 1;
    }
    // Wait (bounded) until the consumers have seen every issued stage land;
    // after an abort, wait (bounded) for copies still in flight.
    const uint64_t t0 = globaltimer_ns();
    while (s_flags[2] < issued && !s_flags[0]) {
        if (globaltimer_ns() - t0 > 4000000000ull) {
            s_flags[0] = 1;
            abort_all(rc, 402);
            break;
        }
        __nanosleep(256);
    }
    if (s_flags[0]) {
        for (long long j = s_flags[2]; j < issued; ++j)
            mbar_wait_bounded(&full[j % ROUND_STAGES], (uint32_t)((j / ROUND_STAGES) & 1),
                              100000000ull);
    }
}

// ------------------------------------------------------------------ consumers

// Tile finish of one epilogue, kept out of line: the k-block loop then
// holds only its own registers.
template <int EPI>
__device__ __noinline__ void finish_out_of_line(const GemmArgs& a, int tile, const float (&acc)[8],
                                                float* ctile, volatile int* s_flags, float* s_rstd,
                                                long long U, int warp, int lane, int tid) {
    gdev::finish_tile<WF_BF16, EPI>(a, tile, acc, ctile, s_flags, s_rstd, U, gridDim.x, blockIdx.x,
                                    warp, lane, tid);
}

// One GEMM phase: the CTA's stream-K range of (tile, k-block) units.
__device__ __forceinline__ void gemm_phase(int epi, const GemmArgs& a, uint8_t* Ws, uint8_t* Xs,
                                           uint64_t* full, uint64_t* empty, float* ctile,
                                           volatile int* s_flags, float* s_rstd, int& stage,
                                           uint32_t& phase, const RoundCall& rc, int warp,
                                           int lane, int tid) {
    const int G = gridDim.x, cta = blockIdx.x;
    const long long U = (long long)a.n_tiles * a.kb;
    const long long u0 = range_start(cta, U, G), u1 = range_start(cta + 1, U, G);
    switch (epi) {   // rstd is read after the first tile's barrier
        case EPI_SWIGLU: gdev::compute_rstd<EPI_SWIGLU>(a, s_rstd, tid); break;
        case EPI_ARGMAX: gdev::compute_rstd<EPI_ARGMAX>(a, s_rstd, tid); break;
        case EPI_QKV: gdev::compute_rstd<EPI_QKV>(a, s_rstd, tid); break;
        default: break;
    }
    float acc[8], accl[8];   // hi and lo planes' accumulators, added at the tile's finish
    for (long long u = u0; u < u1;) {
        const int len = chunk_len(u, u1, a.kb);
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
                abort_all(rc, 403);
            }
        }
        if (ok) {
            for (int jb = 0; jb < len; ++jb) {
                const int slot = stage * ROUND_CHUNK + jb;
                gdev::mma_kblock<WF_BF16, EPI_STORE>(Ws + slot * GEMM_STAGE_W, Xs + slot * RXB,
                                                     nullptr, a, warp, lane, acc, accl);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (tid == 0 && ok) s_flags[2] = s_flags[2] + 1;
        if (++stage == ROUND_STAGES) {
            stage = 0;
            phase ^= 1u;
        }
        u += len;
        if (!(k + len == a.kb || u == u1)) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += accl[i];
        switch (epi) {
            case EPI_STORE:
                finish_out_of_line<EPI_STORE>(a, tile, acc, ctile, s_flags, s_rstd, U, warp, lane, tid);
                break;
            case EPI_RESID:
                finish_out_of_line<EPI_RESID>(a, tile, acc, ctile, s_flags, s_rstd, U, warp, lane, tid);
                break;
            case EPI_SWIGLU:
                finish_out_of_line<EPI_SWIGLU>(a, tile, acc, ctile, s_flags, s_rstd, U, warp, lane, tid);
                break;
            case EPI_ARGMAX:
                finish_out_of_line<EPI_ARGMAX>(a, tile, acc, ctile, s_flags, s_rstd, U, warp, lane, tid);
                break;
            case EPI_QKV:
                finish_out_of_line<EPI_QKV>(a, tile, acc, ctile, s_flags, s_rstd, U, warp, lane, tid);
                break;
            default:
                finish_out_of_line<EPI_NORMOUT>(a, tile, acc, ctile, s_flags, s_rstd, U, warp, lane, tid);
                break;
        }
    }
}

// Attention phase: (kv head, 64-key chunk) items dealt round-robin over the
// CTAs; TMA brings the q group, K and V of an item into the attention slot
// and warp j computes q head j of the group.
template <int HD>
__device__ __forceinline__ void attn_phase(const RoundCall& rc, const Phase* P, uint8_t* As,
                                           uint64_t* abar, uint32_t& aphase,
                                           volatile int* s_flags, int warp, int lane, int tid) {
    constexpr int C = ATTN_KEYS, HALVES = HD / 64;
    const AttnMmaArgs a = P->am;   // by value: read once, not after every barrier
    const AttnMaps* maps = rc.amaps + P->target;
    const int G = gridDim.x;
    const int group = a.n_q / a.n_kv, qrows = group * 16;
    uint8_t* Qs = As;
    uint8_t* Ks = Qs + HALVES * qrows * 128;
    uint8_t* Vs = Ks + HALVES * C * 128;
    const int T = a.st->fwd_T, pos0 = a.st->fwd_pos0;
    if (T == 0) return;
    const int hi = pos0 + T;
    const int lo = (!a.causal && a.window > 0) ? max(0, pos0 - a.window) : 0;
    const int c_lo = lo / C, c_hi = (hi - 1) / C, nch = c_hi - c_lo + 1;
    const int items = a.n_kv * nch;
    const uint32_t bytes = (uint32_t)(HALVES * (qrows + 2 * C) * 128);
    for (int i = blockIdx.x; i < items; i += G) {
        const int kh = i / nch, c = c_lo + i % nch;
        if (tid == 0) {
            mbar_arrive_expect_tx(abar, bytes);
            const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + c * C;
            const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + c * C;
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                tma_load_2d(Qs + h * qrows * 128, &maps->q, abar, 64 * h, kh * qrows);
                tma_load_2d(Ks + h * C * 128, &maps->kv, abar, 64 * h, krow);
                tma_load_2d(Vs + h * C * 128, &maps->kv, abar, 64 * h, vrow);
            }
        }
        const bool ok = mbar_wait_bounded(abar, aphase);
        aphase ^= 1u;
        if (!ok) {
            if (tid == 0) {
                abort_all(rc, 404);
                s_flags[0] = 1;
                mbar_wait_bounded(abar, aphase ^ 1u, 100000000ull);   // let late copies land
            }
            consumer_bar();
            return;
        }
        if (warp < group)
            adev::chunk_partials<HD>(Qs, Ks, Vs, a, qrows, group, kh, c, T, pos0, lo, hi, warp, lane);
        consumer_bar();   // the slot is refilled by the next item
    }
}

// Combine phase: (q head, row) items, HD threads per item.
template <int HD>
__device__ __forceinline__ void combine_phase(const Phase* P, uint8_t* As, int tid) {
    constexpr int NG = GEMM_CONSUMERS * 32 / HD;   // item groups per CTA
    const int gi = tid / HD, d = tid % HD;
    float* base = reinterpret_cast<float*>(As) + gi * (2 * kdev::COMBINE_MAXC + HD / 32);
    float* s_w = base;
    float* s_l = base + kdev::COMBINE_MAXC;
    float* s_red = s_l + kdev::COMBINE_MAXC;
    const AttnArgs ac = P->ac;
    const int items = ac.n_q * DFL_MAX_ROWS;
    const int stride = gridDim.x * NG;
    for (int i = blockIdx.x * NG + gi; i < items; i += stride)
        kdev::combine_item<HD>(ac, i / DFL_MAX_ROWS, i % DFL_MAX_ROWS, d, s_w, s_l, s_red,
                               GroupBar{2 + gi, HD});
}

template <int HD>
__global__ void __launch_bounds__(GEMM_THREADS, 1) round_kernel(const __grid_constant__ RoundCall rc) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* Ws = smem;                                   // [RSLOTS][16 KB]
    uint8_t* Xs = Ws + RSLOTS * GEMM_STAGE_W;              // [RSLOTS][4 KB]
    uint8_t* As = Xs + RSLOTS * RXB;                       // attention / combine slot
    float* ctile = reinterpret_cast<float*>(As + ROUND_ATTN_BYTES);   // [16][128]
    uint64_t* full = reinterpret_cast<uint64_t*>(ctile + DFL_MAX_ROWS * GEMM_BN);
    uint64_t* empty = full + ROUND_STAGES;
    uint64_t* abar = empty + ROUND_STAGES;
    volatile int* s_flags = reinterpret_cast<volatile int*>(abar + 1);
    // s_flags[0]: abort, [1]: last-arriver, [2]: consumed stages, [3..5]: row preparation
    __shared__ float s_rstd[DFL_MAX_ROWS];
    __shared__ GemmArgs s_args;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < ROUND_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GEMM_CONSUMERS);
        }
        mbar_init(abar, 1);
        for (int i = 0; i < 8; ++i) s_flags[i] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == GEMM_CONSUMERS) {
        if (lane == 0) producer(rc, Ws, Xs, full, empty, s_flags);
        return;
    }

    const int tid = threadIdx.x, cta = blockIdx.x, G = gridDim.x;
    int stage = 0;
    uint32_t phase = 0, aphase = 0;
    unsigned bars = 0;
    // split-K tickets start at zero whatever an earlier, aborted launch left
    for (int i = cta * (GEMM_CONSUMERS * 32) + tid; i < rc.n_counters; i += G * GEMM_CONSUMERS * 32)
        rc.counters[i] = 0;
    const bool stamp = rc.phase_ns != nullptr && cta == 0 && tid == 0;
    if (stamp) rc.phase_ns[0] = globaltimer_ns();
    for (int p = 0; p < rc.n_phases; ++p) {
        const Phase* P = rc.phases + p;
        if (P->sync_before) {
            ++bars;
            if (!grid_sync(rc, (unsigned)G * bars, s_flags, tid)) break;
            if (stamp) rc.phase_ns[p] = globaltimer_ns();
        }
        if (s_flags[0]) break;
        switch (P->kind) {
            case PH_PREP:
                if (cta < DFL_MAX_ROWS) {
                    RowsArgs ra = P->rows;
                    if (P->tokens_slot == CS_DRAFT_IDS) ra.tokens = rc.draft_ids;
                    kdev::prepare_row(ra, cta, tid, GEMM_CONSUMERS * 32, s_flags + 3, ConsumerBar());
                }
                break;
            case PH_GEMM: {
                if (tid == 0) {
                    GemmArgs g = P->g;
                    if (P->logits_slot == CS_VERIFY_LOGITS) g.logits = rc.verify_logits;
                    else if (P->logits_slot == CS_DRAFT_LOGITS) g.logits = rc.draft_logits;
                    s_args = g;
                }
                consumer_bar();
                gemm_phase(P->epi, s_args, Ws, Xs, full, empty, ctile, s_flags, s_rstd, stage, phase,
                           rc, warp, lane, tid);
                break;
            }
            case PH_ATTN:
                attn_phase<HD>(rc, P, As, abar, aphase, s_flags, warp, lane, tid);
                break;
            case PH_COMBINE:
                combine_phase<HD>(P, As, tid);
                break;
            case PH_ACCEPT:
                if (cta == 0 && tid == 0) {
                    AcceptArgs aa = P->acc;
                    aa.draft_ids = rc.draft_ids;
                    aa.draft_out = rc.draft_out;
                    aa.tokens_out = rc.tokens_out;
                    aa.n_emitted = rc.n_emitted;
                    kdev::accept_run(aa);
                }
                break;
        }
    }
    if (rc.phase_ns != nullptr && !s_flags[0]) {
        ++bars;
        if (grid_sync(rc, (unsigned)G * bars, s_flags, tid) && stamp)
            rc.phase_ns[rc.n_phases] = globaltimer_ns();
    }
}

constexpr size_t ROUND_SMEM = 1024 + (size_t)RSLOTS * RKB + ROUND_ATTN_BYTES +
                              DFL_MAX_ROWS * GEMM_BN * 4 + (2 * ROUND_STAGES + 1) * 8 + 64;
static_assert(ROUND_SMEM + sizeof(GemmArgs) + 64 <= 232448, "round kernel shared memory");
static_assert(2 * (2 * kdev::COMBINE_MAXC + 4) * 4 <= ROUND_ATTN_BYTES, "combine scratch");

template <int HD>
cudaError_t prepare_attrs() {
    static bool done = false;
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(round_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ROUND_SMEM);
    if (e != cudaSuccess) return e;
    done = true;
    return cudaSuccess;
}

}  // namespace

size_t round_smem_bytes() { return ROUND_SMEM; }

int round_max_ctas(int device, int* out) {
    int sms = 0, per_sm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = prepare_attrs<128>();
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, round_kernel<128>, GEMM_THREADS,
                                                          ROUND_SMEM);
    *out = e == cudaSuccess ? sms * per_sm : 0;
    return (int)e;
}

int launch_round(const RoundCall& rc, int grid, cudaStream_t s) {
    cudaError_t e = rc.head_dim == 128 ? prepare_attrs<128>() : prepare_attrs<64>();
    if (e != cudaSuccess) return (int)e;
    e = cudaMemsetAsync(rc.bar_count, 0, 2 * sizeof(unsigned), s);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = ROUND_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ++g_launches;
    if (rc.head_dim == 128) {
        set_carveout_once(reinterpret_cast<const void*>(round_kernel<128>));
        return (int)cudaLaunchKernelEx(&cfg, round_kernel<128>, rc);
    }
    set_carveout_once(reinterpret_cast<const void*>(round_kernel<64>));
    return (int)cudaLaunchKernelEx(&cfg, round_kernel<64>, rc);
}

}  // namespace dfl
