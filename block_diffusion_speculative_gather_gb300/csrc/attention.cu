// Split-KV attention on tensor cores for the bf16 models (verify, prefill
// and the drafter's block attention).
//
// What it computes, by page: the drafter's block rows attend to the sliding
// context window and to every row of their own block, with no causal order
// inside the block ("feat: DFlash2 block-diffusion drafter for Qwen 3.8",
// first commit: block attention over [sliding ctx | bidirectional block];
// "[RFC] DFlash", "Requested changes" 2: the draft block is non-causal); the
// target's verify and prefill rows attend causally over the KV cache ("[RFC]
// DFlash", "Key Implementation Details", Phase 3).  Only the valid part of a
// cache is read, never the whole buffer (the RFC author's reply, "3. Draft
// KV cache": a masked full-buffer attention cost tracked the buffer size).  q and the K/V caches are fp16 (11
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
#include "gemm.cuh"
#include "tc_dev.cuh"

namespace dfl {

namespace {

__device__ __forceinline__ int ld_acquire_s32_(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_s32_(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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
    adev::chunk_partials<HD>(Qs, Ks, Vs, a, qrows, group, kh, c, T, pos0, lo, hi, warp, lane);
}


// Second half of a split-KV attention launch: once every split of kv head
// kh has published its (max, sum) and unnormalised output into the partials
// (outputs [max_splits][16][n_q][HD], then (max, sum) [max_splits][16][n_q],
// maxima in the base-2 domain), CTA sp normalises its share of the group's
// (q head, row) pairs.  Called by all threads after their stores.
template <int HD>
__device__ __forceinline__ void exchange_combine(const AttnFusedArgs& f, int kh, int sp, int S, int T,
                                                 int group, int tid, int warp, int lane) {
    const AttnMmaArgs& a = f.m;
    const size_t osplit = (size_t)DFL_MAX_ROWS * a.n_q * HD;
    const float* Op = a.part;
    const float2* MLp = reinterpret_cast<const float2*>(a.part + (size_t)f.max_splits * osplit);
    // the barrier orders every thread's stores before thread 0's release add
    __syncthreads();
    __shared__ int s_ok;
    if (tid == 0) {
        red_release_add_s32_(&f.arrive[kh], 1);
        bool got = ld_acquire_s32_(&f.arrive[kh]) >= S;
        const uint64_t t0 = globaltimer_ns();
        while (!got) {
            got = ld_acquire_s32_(&f.arrive[kh]) >= S;
            if (!got && globaltimer_ns() - t0 > 2000000000ull) {
                set_error(a.st, DERR_TIMEOUT, 211);
                break;
            }
        }
        s_ok = got ? 1 : 0;
    }
    __syncthreads();   // thread 0's acquire orders the partial loads below
    if (!s_ok) return;

    // ---- combine: this CTA's (q head of the group, row) pairs p = sp, sp + S, ...,
    // one warp per pair.  Lane j holds split j's (and j + 32's) max and sum;
    // with M the maximum, split j weighs w_j = 2^(m_j - M), the row's sum is
    // L = sum_j w_j l_j, and lane d folds output columns 4d..4d+3 over the
    // splits in split order.  All loads of a batch are independent, so a
    // pair costs about two L2 round trips whatever S is.
    constexpr int NV = HD / 4;        // float4 columns of one output row
    constexpr int BATCH = 16;         // splits loaded per batch
    const size_t ld = (size_t)a.n_q * HD;
    const int pairs = group * DFL_MAX_ROWS;
    for (int p = sp + warp * S; p < pairs; p += 4 * S) {
        const int hq = kh * group + p / DFL_MAX_ROWS, t = p % DFL_MAX_ROWS;
        const size_t col = (size_t)hq * HD + 4 * lane;
        if (t >= T) {
            if (lane < NV)
#pragma unroll
                for (int e = 0; e < 4; ++e) store_act(f.out, f.out_type, ld, t, col + e, 0.f);
            continue;
        }
        const float2* ml = MLp + (size_t)t * a.n_q + hq;
        const size_t mls = (size_t)DFL_MAX_ROWS * a.n_q;
        const float2 ml0 = lane < S ? __ldcg(ml + lane * mls) : make_float2(-INFINITY, 0.f);
        const float2 ml1 = lane + 32 < S ? __ldcg(ml + (lane + 32) * mls) : make_float2(-INFINITY, 0.f);
        const float4* src = reinterpret_cast<const float4*>(Op + ((size_t)t * a.n_q + hq) * HD) + lane;
        const size_t sst = osplit / 4;
        float4 v[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u)
            v[u] = (u < S && lane < NV) ? __ldcg(src + u * sst) : make_float4(0.f, 0.f, 0.f, 0.f);
        float M = fmaxf(ml0.x, ml1.x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float w0 = ml0.x == -INFINITY ? 0.f : exp2f(ml0.x - M);   // maxima are base-2
        const float w1 = ml1.x == -INFINITY ? 0.f : exp2f(ml1.x - M);
        float L = fmaf(w1, ml1.y, w0 * ml0.y);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < S; j0 += BATCH) {
            float4 nv[BATCH];
            const int j1 = j0 + BATCH;
#pragma unroll
            for (int u = 0; u < BATCH; ++u)   // next batch in flight while this one folds
                nv[u] = (j1 + u < S && lane < NV) ? __ldcg(src + (size_t)(j1 + u) * sst)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int j = j0 + u;
                const float wa = __shfl_sync(0xffffffffu, w0, j & 31);
                const float wb = __shfl_sync(0xffffffffu, w1, j & 31);
                const float wj = j < 32 ? wa : wb;
                O.x = fmaf(v[u].x, wj, O.x);
                O.y = fmaf(v[u].y, wj, O.y);
                O.z = fmaf(v[u].z, wj, O.z);
                O.w = fmaf(v[u].w, wj, O.w);
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) v[u] = nv[u];
        }
        if (lane < NV) {
            const float inv = 1.f / L;
            store_act(f.out, f.out_type, ld, t, col + 0, O.x * inv);
            store_act(f.out, f.out_type, ld, t, col + 1, O.y * inv);
            store_act(f.out, f.out_type, ld, t, col + 2, O.z * inv);
            store_act(f.out, f.out_type, ld, t, col + 3, O.w * inv);
        }
    }
    // the last split of the head to finish resets the head's counters
    if (tid == 0) {
        const int old = atomicAdd(&f.done[kh], 1);
        if (old == S - 1) {
            f.arrive[kh] = 0;
            f.done[kh] = 0;
        }
    }
}

// Shared memory of the fused kernel: the q group, two K/V chunk buffers,
// mbarriers.
template <int HD>
constexpr size_t fused_smem(int qrows) {
    return 1024 + (size_t)(HD / 64) * (qrows + 4 * ATTN_KEYS) * 128 + 3 * 8 + 64;
}

template <int HD>
__global__ void __launch_bounds__(128)
attn_fused_kernel(const __grid_constant__ AttnMaps maps, const AttnFusedArgs f) {
    constexpr int C = ATTN_KEYS, HALVES = HD / 64;
    constexpr int MAXS = 64;   // splits a combine folds (host guarantees max_splits <= 64)
    const AttnMmaArgs& a = f.m;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int group = a.n_q / a.n_kv, qrows = group * 16;
    uint8_t* Qs = sm;                                   // [HALVES][qrows][128 B]
    uint8_t* KV = Qs + HALVES * qrows * 128;            // 2 x (K, V) [HALVES][64][128 B]
    constexpr int KVB = HALVES * C * 128;               // bytes of one K (or V) chunk
    uint64_t* bar = reinterpret_cast<uint64_t*>(KV + 4 * KVB);   // [0] q, [1..2] buffers

    pdl_trigger();
    const int kh = blockIdx.x, sp = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // When the first visible key is 0 (causal, or no window) a split's chunks
    // sit at fixed positions, so they can be brought into L2 while the
    // predecessor still writes this forward's rows (L2 stays coherent with
    // those writes; the copies into shared memory come after the wait).
    // Only the chunks the forward will read: the visible length comes from
    // the round state read before the wait, as a hint (the state's writer
    // may not have finished, so it may still hold the previous forward's
    // length; a stale value only changes which chunks are prefetched, and
    // boxes past the tensor are ignored).
    if (tid == 0 && (a.causal || a.window <= 0)) {
        const volatile int* vs = reinterpret_cast<const volatile int*>(a.st);
        const int hint = vs[offsetof(DevState, fwd_pos0) / 4] + vs[offsetof(DevState, fwd_T) / 4];
        const int c_last = hint > 0 ? (hint - 1) / C : 0;
        const int np = min(f.split_chunks, 2);
        for (int i = 0; i < np; ++i) {
            const int c = sp * f.split_chunks + i;
            if (c > c_last) break;
            const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + c * C;
            const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + c * C;
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                tma_prefetch_l2_2d(&maps.kv, 64 * h, krow);
                tma_prefetch_l2_2d(&maps.kv, 64 * h, vrow);
            }
        }
    }
    pdl_wait();
    const int T = a.st->fwd_T, pos0 = a.st->fwd_pos0;
    if (T == 0) return;
    const int hi = pos0 + T;
    const int lo = (!a.causal && a.window > 0) ? max(0, pos0 - a.window) : 0;
    const int c_lo = lo / C, c_hi = (hi - 1) / C;
    const int S = (c_hi - c_lo + f.split_chunks) / f.split_chunks;   // splits in use
    if (sp >= S) return;
    if (S > MAXS || S > f.max_splits) {
        if (tid == 0) set_error(a.st, DERR_INDEX, S);
        return;
    }
    const int c0 = c_lo + sp * f.split_chunks;
    const int n_my = min(f.split_chunks, c_hi + 1 - c0);

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto load_chunk = [&](int i) {   // chunk c0 + i into buffer i & 1
        uint8_t* Kb = KV + (i & 1) * 2 * KVB;
        uint8_t* Vb = Kb + KVB;
        const int c = c0 + i;
        const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + c * C;
        const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + c * C;
        mbar_arrive_expect_tx(&bar[1 + (i & 1)], 2 * KVB);
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            tma_load_2d(Kb + h * C * 128, &maps.kv, &bar[1 + (i & 1)], 64 * h, krow);
            tma_load_2d(Vb + h * C * 128, &maps.kv, &bar[1 + (i & 1)], 64 * h, vrow);
        }
    };
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], HALVES * qrows * 128);
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            tma_load_2d(Qs + h * qrows * 128, &maps.q, &bar[0], 64 * h, kh * qrows);
        load_chunk(0);
        if (n_my > 1) load_chunk(1);
    }
    // every wait is voted on by the whole CTA, so all threads leave together
    bool ok = __syncthreads_and(mbar_wait_bounded(&bar[0], 0)) != 0;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[HD / 8][4];
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    int issued = n_my > 1 ? 2 : 1;
    for (int i = 0; i < n_my && ok; ++i) {
        ok = __syncthreads_and(mbar_wait_bounded(&bar[1 + (i & 1)], (uint32_t)((i >> 1) & 1))) != 0;
        if (ok && warp < group)
            adev::chunk_online<HD>(Qs, KV + (i & 1) * 2 * KVB, KV + (i & 1) * 2 * KVB + KVB, a,
                                   qrows, c0 + i, T, pos0, lo, hi, warp, lane, m, l, o);
        __syncthreads();   // buffer i & 1 is free again
        if (ok && tid == 0 && i + 2 < n_my) {
            load_chunk(i + 2);
            ++issued;
        }
    }
    if (!ok) {
        if (tid == 0) {
            set_error(a.st, DERR_TIMEOUT, 210);
            // let copies still in flight land before the CTA exits
            mbar_wait_bounded(&bar[0], 0, 100000000ull);
            for (int i = 0; i < issued; ++i)
                mbar_wait_bounded(&bar[1 + (i & 1)], (uint32_t)((i >> 1) & 1), 100000000ull);
        }
        return;
    }

    // ---- publish this split's (max, sum) and unnormalised output of rows g, g + 8
    // partials: outputs [max_splits][16][n_q][HD], then (max, sum) [max_splits][16][n_q]
    const size_t osplit = (size_t)DFL_MAX_ROWS * a.n_q * HD;
    float* Op = a.part;
    float2* MLp = reinterpret_cast<float2*>(a.part + (size_t)f.max_splits * osplit);
    if (warp < group) {
        const int g = lane >> 2, cq = lane & 3, hq = kh * group + warp;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int t = g + 8 * r;
            float* dst = Op + sp * osplit + ((size_t)t * a.n_q + hq) * HD + 2 * cq;
            if (cq == 0) MLp[((size_t)sp * DFL_MAX_ROWS + t) * a.n_q + hq] = make_float2(m[r], l[r]);
#pragma unroll
            for (int dt = 0; dt < HD / 8; ++dt)
                *reinterpret_cast<float2*>(dst + dt * 8) = make_float2(o[dt][2 * r], o[dt][2 * r + 1]);
        }
    }
    exchange_combine<HD>(f, kh, sp, S, T, group, tid, warp, lane);
}

// Tensor-core (tcgen05) form of the fused attention for splits of NC = 1 or
// 2 consecutive 64-key chunks (KEYS = 64 NC keys).  TMA brings each q
// head's 16 rows to tile rows 32h..32h+15 (so the score row of q head h,
// token t lands in tensor-memory lane 32h + t and warp h owns head h), and
// the split's K and V.  One thread issues S = Q K^T (M 128, N KEYS) into
// tensor memory while the CTA transposes V into a K-major tile; each thread
// of a real row then reads its scores, masks, takes the row max and the
// base-2 exponentials in registers, and writes its f16 probabilities as the
// A tile of O = P V (M 128, N head_dim, K KEYS), which the tensor core
// accumulates in f32.  The rows' (max, sum, unnormalised output) are
// published like the mma.sync form's and combined the same way.  A kernel
// that allocates tensor memory holds one CTA per SM here, so a launch has
// at most one CTA per SM and NC = 2 serves the longer caches.
template <int HD, int NC>
constexpr size_t tc_smem() {
    // Q [HD/64][128 rows][128 B], V and K [HD/64][KEYS][128 B] each,
    // V^T [NC][HD][128 B]; P [NC][128][128 B] over K (as large for head_dim
    // 128, twice as large for 64), barriers and the tensor-memory address
    constexpr size_t q = (size_t)(HD / 64) * 128 * 128, kv = (size_t)(HD / 64) * NC * ATTN_KEYS * 128;
    constexpr size_t vt = (size_t)NC * HD * 128, pk = (size_t)NC * 128 * 128;
    return 1024 + q + kv + vt + (kv > pk ? kv : pk) + 3 * 8 + 8 + 64;
}
template <int HD, int NC>
constexpr uint32_t tc_cols() {   // S (KEYS columns) + O (HD), rounded up to a power of two
    return NC * ATTN_KEYS + HD <= 128 ? 128u : NC * ATTN_KEYS + HD <= 256 ? 256u : 512u;
}

template <int HD, int NC>
__global__ void __launch_bounds__(128)
attn_tc_kernel(const __grid_constant__ AttnMaps maps, const AttnFusedArgs f) {
    constexpr int C = ATTN_KEYS, HALVES = HD / 64, KEYS = NC * C;
    constexpr int MAXS = 64;
    constexpr uint32_t TCOLS = tc_cols<HD, NC>();
    const AttnMmaArgs& a = f.m;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int KVH = KEYS * 128;            // bytes of one 64-column half of K (or V)
    uint8_t* Qs = sm;                          // [HALVES][128 rows][128 B]
    uint8_t* Vs = Qs + HALVES * 128 * 128;     // [HALVES][KEYS][128 B]
    uint8_t* Vt = Vs + HALVES * KVH;           // [NC][HD][128 B]: V^T, 64 keys per 128-byte row
    uint8_t* Ks = Vt + NC * HD * 128;          // [HALVES][KEYS][128 B]
    uint8_t* Ps = Ks;                          // [NC][128 rows][128 B] over K once S is done
    constexpr int KP = HALVES * KVH > NC * 128 * 128 ? HALVES * KVH : NC * 128 * 128;
    uint64_t* bar = reinterpret_cast<uint64_t*>(Ks + KP);   // [0] loads, [1] S, [2] O
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 3);

    pdl_trigger();
    const int kh = blockIdx.x, sp = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    if (tid == 0 && (a.causal || a.window <= 0)) {   // the split's chunks sit at fixed positions
        // only chunks the forward reads (visible length from the state, a
        // hint read before the wait, as in attn_fused_kernel)
        const volatile int* vs = reinterpret_cast<const volatile int*>(a.st);
        const int hint = vs[offsetof(DevState, fwd_pos0) / 4] + vs[offsetof(DevState, fwd_T) / 4];
        const int c_last = hint > 0 ? (hint - 1) / C : 0;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            if (sp * NC + j > c_last) break;
            const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + (sp * NC + j) * C;
            const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + (sp * NC + j) * C;
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                tma_prefetch_l2_2d(&maps.kv, 64 * h, krow);
                tma_prefetch_l2_2d(&maps.kv, 64 * h, vrow);
            }
        }
    }
    pdl_wait();
    const int T = a.st->fwd_T, pos0 = a.st->fwd_pos0;
    if (T == 0) return;
    const int hi = pos0 + T;
    const int lo = (!a.causal && a.window > 0) ? max(0, pos0 - a.window) : 0;
    const int c_lo = lo / C, c_hi = (hi - 1) / C;
    const int S = (c_hi - c_lo + NC) / NC;   // splits in use
    if (sp >= S) return;
    if (S > MAXS || S > f.max_splits) {
        if (tid == 0) set_error(a.st, DERR_INDEX, S);
        return;
    }
    const int k0 = (c_lo + sp * NC) * C;   // first key of the split
    const int group = a.n_q / a.n_kv;

    // the loads first, so the tensor-memory allocation overlaps them
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar[0], HALVES * (group * 16 + 2 * KEYS) * 128);
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            for (int q = 0; q < group; ++q)
                tma_load_2d(Qs + h * 128 * 128 + q * 32 * 128, &maps.q16, &bar[0], 64 * h,
                            (kh * group + q) * 16);
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + k0 + j * C;
                const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + k0 + j * C;
                tma_load_2d(Ks + h * KVH + j * C * 128, &maps.kv, &bar[0], 64 * h, krow);
                tma_load_2d(Vs + h * KVH + j * C * 128, &maps.kv, &bar[0], 64 * h, vrow);
            }
        }
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(s_tmem, TCOLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *s_tmem;
    // every wait is voted on by the whole CTA, so all threads leave together
    bool ok = __syncthreads_and(mbar_wait_bounded(&bar[0], 0)) != 0;
    const bool s_issued = ok;
    if (ok && tid == 0) {   // S = Q K^T while the CTA transposes V
        tc::fence_after_sync();
        constexpr uint32_t IS = tc::idesc_f16_f32(128, KEYS);
#pragma unroll
        for (int kd = 0; kd < HD / 16; ++kd) {
            const int h = kd >> 2, ko = (kd & 3) * 32;
            tc::mma_f16(tm, tc::desc_sw128(Qs + h * 128 * 128 + ko), tc::desc_sw128(Ks + h * KVH + ko), IS,
                        kd > 0 ? 1u : 0u);
        }
        tc::commit(&bar[1]);
    }
    if (ok) {   // V^T by 8x8 transposes: ldmatrix a [keys][d] block, store it as [d][keys]
        const int r8 = lane & 7, m = lane >> 3;
#pragma unroll 1
        for (int o = warp; o < NC * HALVES * 16; o += 4) {
            const int j = o / (HALVES * 16), h = (o / 16) % HALVES;
            const int kb = (o & 15) >> 1, db = ((o & 1) << 2) + m;   // key block, d block of matrix m
            const int key = 8 * kb + r8, d = 64 * h + 8 * db + r8;
            uint32_t r[4];
            adev::ldsm_x4(r, Vs + h * KVH + j * C * 128 + key * 128 + ((db ^ (key & 7)) << 4));
            adev::stsm_x4_trans(Vt + j * HD * 128 + d * 128 + ((kb ^ (d & 7)) << 4), r);
        }
    }
    tc::fence_async_smem();   // V^T visible to the tensor core
    if (ok) ok = __syncthreads_and(mbar_wait_bounded(&bar[1], 0)) != 0;
    tc::fence_after_sync();

    // ---- softmax of this thread's score row (q head `warp`, token `lane`),
    // 32 scores at a time: the row max first, then the probabilities
    const bool mine = warp < group && lane < 16;
    float m_r = -INFINITY, l_r = 0.f;
    if (ok && warp < group) {
        const uint32_t trow = tm + ((uint32_t)(warp * 32) << 16);
        const int t = lane;
        const float sl2 = a.scale * 1.4426950408889634f;
        const int kmax = a.causal ? min(hi - 1, pos0 + t) : hi - 1;
        const bool whole = t < T && k0 >= lo && k0 + KEYS - 1 <= kmax;
        // scaled, masked scores of keys k0 + 32 b + j.  The load is warp-wide;
        // lanes 16..31 hold the tile's padding rows (never-written shared
        // memory, any bit pattern) and do no arithmetic on them.
        auto scores = [&](int b, float (&sv)[32]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sv[j] *= sl2;
            if (!whole) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int key = k0 + 32 * b + j;
                    if (!(t < T && key >= lo && key <= kmax)) sv[j] = -INFINITY;
                }
            }
        };
        float mx = -INFINITY, sum = 0.f;
#pragma unroll 1
        for (int b = 0; b < KEYS / 32; ++b) {
            float sv[32];
            tc::ld_x32(trow + 32 * b, sv);
            if (mine) {
                scores(b, sv);
#pragma unroll
                for (int j = 0; j < 32; ++j) mx = fmaxf(mx, sv[j]);
            }
        }
#pragma unroll 1
        for (int b = 0; b < KEYS / 32; ++b) {
            float sv[32];
            tc::ld_x32(trow + 32 * b, sv);
            if (mine) {   // keys 32b.. : chunk b/2 of P, 16-byte groups 4(b&1)..4(b&1)+3
                scores(b, sv);
#pragma unroll
                for (int j = 0; j < 32; ++j) sv[j] = sv[j] == -INFINITY ? 0.f : exp2f(sv[j] - mx);
#pragma unroll
                for (int j = 0; j < 32; ++j) sum += sv[j];
                uint8_t* prow = Ps + (b >> 1) * 128 * 128 + tid * 128;
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    const int kc = 4 * (b & 1) + g4;
                    *reinterpret_cast<uint4*>(prow + ((kc ^ (tid & 7)) << 4)) = make_uint4(
                        pack_f16x2(sv[8 * g4 + 0], sv[8 * g4 + 1]), pack_f16x2(sv[8 * g4 + 2], sv[8 * g4 + 3]),
                        pack_f16x2(sv[8 * g4 + 4], sv[8 * g4 + 5]), pack_f16x2(sv[8 * g4 + 6], sv[8 * g4 + 7]));
                }
            }
        }
        m_r = mx;
        l_r = sum;
    }
    tc::fence_async_smem();   // P visible to the tensor core
    tc::fence_before_sync();
    __syncthreads();
    const bool o_issued = ok;
    if (ok && tid == 0) {   // O = P V
        tc::fence_after_sync();
        constexpr uint32_t IO = tc::idesc_f16_f32(128, HD);
#pragma unroll
        for (int kk = 0; kk < KEYS / 16; ++kk) {
            const int j = kk >> 2, ko = (kk & 3) * 32;
            tc::mma_f16(tm + KEYS, tc::desc_sw128(Ps + j * 128 * 128 + ko),
                        tc::desc_sw128(Vt + j * HD * 128 + ko), IO, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bar[2]);
    }
    if (ok) ok = __syncthreads_and(mbar_wait_bounded(&bar[2], 0)) != 0;
    tc::fence_after_sync();

    // ---- publish (max, sum) and the unnormalised output row
    const size_t osplit = (size_t)DFL_MAX_ROWS * a.n_q * HD;
    float* Op = a.part;
    float2* MLp = reinterpret_cast<float2*>(a.part + (size_t)f.max_splits * osplit);
    if (ok && warp < group) {
        const int t = lane, hq = kh * group + warp;
        float* dst = Op + sp * osplit + ((size_t)t * a.n_q + hq) * HD;
        const uint32_t trow = tm + ((uint32_t)(warp * 32) << 16) + KEYS;
#pragma unroll 1
        for (int q = 0; q < HD / 32; ++q) {
            float v[32];
            tc::ld_x32(trow + 32 * q, v);
            if (mine)
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(dst + 32 * q + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
        if (mine) MLp[((size_t)sp * DFL_MAX_ROWS + t) * a.n_q + hq] = make_float2(m_r, l_r);
    }
    if (!ok) {   // copies and MMAs still in flight finish before tensor memory is freed
        if (tid == 0) set_error(a.st, DERR_TIMEOUT, 212);
        mbar_wait_bounded(&bar[0], 0, 100000000ull);
        if (s_issued) mbar_wait_bounded(&bar[1], 0, 100000000ull);
        if (o_issued) mbar_wait_bounded(&bar[2], 0, 100000000ull);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TCOLS);
    if (!ok) return;
    exchange_combine<HD>(f, kh, sp, S, T, group, tid, warp, lane);
}

struct PrefillMaps {
    CUtensorMap q, kv;
};

template <int HD>
__global__ void __launch_bounds__(128)
prefill_attn_kernel(const __grid_constant__ PrefillMaps maps, const PrefillAttnArgs p) {
    constexpr int C = ATTN_KEYS, HALVES = HD / 64;
    const AttnMmaArgs& a = p.m;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int group = a.n_q / a.n_kv, qrows = group * 16;
    uint8_t* Qs = sm;                                   // [HALVES][qrows][128 B]
    uint8_t* KV = Qs + HALVES * qrows * 128;            // 2 x (K, V) [HALVES][64][128 B]
    constexpr int KVB = HALVES * C * 128;
    uint64_t* bar = reinterpret_cast<uint64_t*>(KV + 4 * KVB);   // [0] q, [1..2] buffers

    pdl_trigger();
    pdl_wait();
    // row blocks in decreasing order: under the causal mask block z folds
    // about z / 4 + 1 chunks, and the blocks that start first should be
    // the longest ones, so that the short ones fill the tail of the launch
    const int kh = blockIdx.x, z = gridDim.y - 1 - blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int T = min(16, p.rows - 16 * z);
    if (T <= 0) return;
    const int pos0 = p.pos0 + 16 * z, hi = pos0 + T;
    const int n_my = (hi - 1) / C + 1;   // chunks 0 .. (hi - 1) / 64

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto load_chunk = [&](int i) {   // chunk i into buffer i & 1
        uint8_t* Kb = KV + (i & 1) * 2 * KVB;
        uint8_t* Vb = Kb + KVB;
        const int krow = ((a.layer * 2 + 0) * a.n_kv + kh) * a.cap + i * C;
        const int vrow = ((a.layer * 2 + 1) * a.n_kv + kh) * a.cap + i * C;
        mbar_arrive_expect_tx(&bar[1 + (i & 1)], 2 * KVB);
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            tma_load_2d(Kb + h * C * 128, &maps.kv, &bar[1 + (i & 1)], 64 * h, krow);
            tma_load_2d(Vb + h * C * 128, &maps.kv, &bar[1 + (i & 1)], 64 * h, vrow);
        }
    };
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], HALVES * qrows * 128);
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            tma_load_2d(Qs + h * qrows * 128, &maps.q, &bar[0], 64 * h, (z * a.n_q + kh * group) * 16);
        load_chunk(0);
        if (n_my > 1) load_chunk(1);
    }
    bool ok = __syncthreads_and(mbar_wait_bounded(&bar[0], 0)) != 0;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[HD / 8][4];
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    int issued = n_my > 1 ? 2 : 1;
    for (int i = 0; i < n_my && ok; ++i) {
        ok = __syncthreads_and(mbar_wait_bounded(&bar[1 + (i & 1)], (uint32_t)((i >> 1) & 1))) != 0;
        if (ok && warp < group)
            adev::chunk_online<HD>(Qs, KV + (i & 1) * 2 * KVB, KV + (i & 1) * 2 * KVB + KVB, a, qrows, i, T,
                                   pos0, 0, hi, warp, lane, m, l, o);
        __syncthreads();   // buffer i & 1 is free again
        if (ok && tid == 0 && i + 2 < n_my) {
            load_chunk(i + 2);
            ++issued;
        }
    }
    if (!ok) {
        if (tid == 0) {
            set_error(a.st, DERR_TIMEOUT, 220);
            mbar_wait_bounded(&bar[0], 0, 100000000ull);
            for (int i = 0; i < issued; ++i)
                mbar_wait_bounded(&bar[1 + (i & 1)], (uint32_t)((i >> 1) & 1), 100000000ull);
        }
        return;
    }
    if (warp < group) {
        const int g = lane >> 2, cq = lane & 3, hq = kh * group + warp;
        const size_t ld = (size_t)a.n_q * HD;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int t = g + 8 * r;
            if (t >= T) continue;
            const float inv = 1.f / l[r];
            const size_t row = (size_t)(16 * z + t) * ld + (size_t)hq * HD + 2 * cq;
#pragma unroll
            for (int dt = 0; dt < HD / 8; ++dt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float v = o[dt][2 * r + e] * inv;
                    if (p.f16) {
                        const __half h = __float2half_rn(v);
                        reinterpret_cast<__half*>(p.out_hi)[row + dt * 8 + e] = h;
                        reinterpret_cast<__half*>(p.out_lo)[row + dt * 8 + e] = __float2half_rn(v - __half2float(h));
                    } else {
                        const __nv_bfloat16 h = __float2bfloat16_rn(v);
                        reinterpret_cast<__nv_bfloat16*>(p.out_hi)[row + dt * 8 + e] = h;
                        reinterpret_cast<__nv_bfloat16*>(p.out_lo)[row + dt * 8 + e] =
                            __float2bfloat16_rn(v - __bfloat162float(h));
                    }
                }
        }
    }
}

template <int HD>
__global__ void __launch_bounds__(128)
batch_attn_kernel(const __grid_constant__ PrefillMaps maps, const BatchAttnArgs b) {
    constexpr int C = ATTN_KEYS, HALVES = HD / 64;
    const AttnMmaArgs& a = b.m;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int group = a.n_q / a.n_kv, qrows = group * 16;
    uint8_t* Qs = sm;                                   // [HALVES][qrows][128 B]
    uint8_t* KV = Qs + HALVES * qrows * 128;            // 2 x (K, V) [HALVES][64][128 B]
    constexpr int KVB = HALVES * C * 128;
    uint64_t* bar = reinterpret_cast<uint64_t*>(KV + 4 * KVB);   // [0] q, [1..2] buffers

    pdl_trigger();
    pdl_wait();
    const int kh = blockIdx.x, sq = blockIdx.y, z = blockIdx.z, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    DevState* st = b.sts[sq];
    const int T = st->fwd_T, pos0 = st->fwd_pos0;
    const int hi = pos0 + T;
    const int lo = (!a.causal && a.window > 0) ? max(0, pos0 - a.window) : 0;
    const int c_lo = lo / C, c_hi = (hi - 1) / C;
    const int c0 = c_lo + z * b.split_chunks;
    const int n_my = T > 0 ? max(0, min(b.split_chunks, c_hi + 1 - c0)) : 0;
    // partials of this split: (max, sum, unnormalised output) per (row, q head)
    float* pbase = b.part + ((size_t)(sq * b.splits + z) * DFL_MAX_ROWS) * a.n_q * (HD + 2);
    if (n_my == 0) {   // nothing visible in this split: an empty partial
        for (int e = tid; e < DFL_MAX_ROWS * group; e += blockDim.x) {
            const int t = e / group, hq = kh * group + e % group;
            float* pp = pbase + ((size_t)t * a.n_q + hq) * (HD + 2);
            pp[0] = -INFINITY;
            pp[1] = 0.f;
        }
        return;
    }
    const int layer_row = (sq * b.n_layers + a.layer) * 2;   // K run of this layer in the map

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto load_chunk = [&](int i) {   // chunk c0 + i into buffer i & 1
        uint8_t* Kb = KV + (i & 1) * 2 * KVB;
        uint8_t* Vb = Kb + KVB;
        const int c = c0 + i;
        const int krow = ((layer_row + 0) * a.n_kv + kh) * a.cap + c * C;
        const int vrow = ((layer_row + 1) * a.n_kv + kh) * a.cap + c * C;
        mbar_arrive_expect_tx(&bar[1 + (i & 1)], 2 * KVB);
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
            tma_load_2d(Kb + h * C * 128, &maps.kv, &bar[1 + (i & 1)], 64 * h, krow);
            tma_load_2d(Vb + h * C * 128, &maps.kv, &bar[1 + (i & 1)], 64 * h, vrow);
        }
    };
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], HALVES * qrows * 128);
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            tma_load_2d(Qs + h * qrows * 128, &maps.q, &bar[0], 64 * h, (sq * a.n_q + kh * group) * 16);
        load_chunk(0);
        if (n_my > 1) load_chunk(1);
    }
    bool ok = __syncthreads_and(mbar_wait_bounded(&bar[0], 0)) != 0;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[HD / 8][4];
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    int issued = n_my > 1 ? 2 : 1;
    for (int i = 0; i < n_my && ok; ++i) {
        ok = __syncthreads_and(mbar_wait_bounded(&bar[1 + (i & 1)], (uint32_t)((i >> 1) & 1))) != 0;
        if (ok && warp < group)
            adev::chunk_online<HD>(Qs, KV + (i & 1) * 2 * KVB, KV + (i & 1) * 2 * KVB + KVB, a, qrows,
                                   c0 + i, T, pos0, lo, hi, warp, lane, m, l, o);
        __syncthreads();   // buffer i & 1 is free again
        if (ok && tid == 0 && i + 2 < n_my) {
            load_chunk(i + 2);
            ++issued;
        }
    }
    if (!ok) {
        if (tid == 0) {
            set_error(st, DERR_TIMEOUT, 230);
            mbar_wait_bounded(&bar[0], 0, 100000000ull);
            for (int i = 0; i < issued; ++i)
                mbar_wait_bounded(&bar[1 + (i & 1)], (uint32_t)((i >> 1) & 1), 100000000ull);
        }
        return;
    }
    if (warp < group) {
        const int g = lane >> 2, cq = lane & 3, hq = kh * group + warp;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int t = g + 8 * r;
            float* pp = pbase + ((size_t)t * a.n_q + hq) * (HD + 2);
            if (cq == 0) {
                pp[0] = m[r];   // base-2 domain
                pp[1] = l[r];
            }
#pragma unroll
            for (int dt = 0; dt < HD / 8; ++dt)
#pragma unroll
                for (int e = 0; e < 2; ++e) pp[2 + dt * 8 + 2 * cq + e] = o[dt][2 * r + e];
        }
    }
}

// One warp per (sequence, row, q head): folds the splits' partials in split
// order (base-2 maxima) and writes the normalised row as bf16 hi/lo (zero
// for rows past the sequence's T).
template <int HD>
__global__ void batch_attn_combine_kernel(const BatchAttnArgs b, int S) {
    pdl_trigger();
    pdl_wait();
    const AttnMmaArgs& a = b.m;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= S * DFL_MAX_ROWS * a.n_q) return;
    const int sq = warp / (DFL_MAX_ROWS * a.n_q), rem = warp % (DFL_MAX_ROWS * a.n_q);
    const int t = rem / a.n_q, hq = rem % a.n_q;
    const int T = b.sts[sq]->fwd_T;
    const size_t ld = (size_t)a.n_q * HD;
    const size_t obase = (size_t)(16 * sq + t) * ld + (size_t)hq * HD;
    float out[HD / 32];
#pragma unroll
    for (int j = 0; j < HD / 32; ++j) out[j] = 0.f;
    if (t < T) {
        const size_t pstride = (size_t)DFL_MAX_ROWS * a.n_q * (HD + 2);
        const float* p0 = b.part + ((size_t)sq * b.splits * DFL_MAX_ROWS + t) * a.n_q * (HD + 2) +
                          (size_t)hq * (HD + 2);
        float M = -INFINITY;
        for (int zz = 0; zz < b.splits; ++zz) M = fmaxf(M, p0[zz * pstride]);
        float L = 0.f;
        for (int zz = 0; zz < b.splits; ++zz) {
            const float mz = p0[zz * pstride];
            const float w = mz == -INFINITY ? 0.f : exp2f(mz - M);
            L = fmaf(p0[zz * pstride + 1], w, L);
#pragma unroll
            for (int j = 0; j < HD / 32; ++j)
                out[j] = fmaf(w == 0.f ? 0.f : p0[zz * pstride + 2 + lane + 32 * j], w, out[j]);
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int j = 0; j < HD / 32; ++j) out[j] *= inv;
    }
#pragma unroll
    for (int j = 0; j < HD / 32; ++j) {
        const float v = out[j];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        reinterpret_cast<__nv_bfloat16*>(b.out_hi)[obase + lane + 32 * j] = h;
        reinterpret_cast<__nv_bfloat16*>(b.out_lo)[obase + lane + 32 * j] =
            __float2bfloat16_rn(v - __bfloat162float(h));
    }
}

template <int HD>
int launch_batch_hd(const CUtensorMap& q_map, const CUtensorMap& kv_map, const BatchAttnArgs& b, int S,
                    cudaStream_t s) {
    const int qrows = (b.m.n_q / b.m.n_kv) * 16;
    const size_t smem = 1024 + (size_t)(HD / 64) * (qrows + 4 * ATTN_KEYS) * 128 + 3 * 8 + 64;
    static bool set = false;
    if (!set) {
        const cudaError_t e = cudaFuncSetAttribute(batch_attn_kernel<HD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        set = true;
    }
    PrefillMaps maps;
    maps.q = q_map;
    maps.kv = kv_map;
    int e = (int)launch_k(batch_attn_kernel<HD>, dim3((unsigned)b.m.n_kv, (unsigned)S, (unsigned)b.splits),
                          dim3(128), smem, s, maps, b);
    if (e) return e;
    const long long warps = (long long)S * DFL_MAX_ROWS * b.m.n_q;
    return (int)launch_k(batch_attn_combine_kernel<HD>, dim3((unsigned)((warps * 32 + 255) / 256)), dim3(256), 0,
                         s, b, S);
}

template <int HD>
int launch_prefill_hd(const CUtensorMap& q_map, const CUtensorMap& kv_map, const PrefillAttnArgs& p,
                      cudaStream_t s) {
    const int qrows = (p.m.n_q / p.m.n_kv) * 16;
    const size_t smem = 1024 + (size_t)(HD / 64) * (qrows + 4 * ATTN_KEYS) * 128 + 3 * 8 + 64;
    static bool set = false;
    if (!set) {
        const cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel<HD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        set = true;
    }
    PrefillMaps maps;
    maps.q = q_map;
    maps.kv = kv_map;
    return (int)launch_k(prefill_attn_kernel<HD>, dim3((unsigned)p.m.n_kv, (unsigned)((p.rows + 15) / 16)),
                         dim3(128), smem, s, maps, p);
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


template <int HD, int NC>
int launch_tc(const AttnMaps& maps, const AttnFusedArgs& f, cudaStream_t s) {
    constexpr size_t smem = tc_smem<HD, NC>();
    static bool set = false;
    if (!set) {
        const cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, NC>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        set = true;
    }
    return (int)launch_k(attn_tc_kernel<HD, NC>, dim3(f.m.n_kv, f.max_splits), dim3(128), smem, s, maps, f);
}

template <int HD, int NC>
int tc_per_sm(int* out, int* tmem_cols) {
    *tmem_cols = (int)tc_cols<HD, NC>();
    set_carveout_once(reinterpret_cast<const void*>(attn_tc_kernel<HD, NC>));
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc_smem<HD, NC>());
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, attn_tc_kernel<HD, NC>, 128, tc_smem<HD, NC>());
    return (int)e;
}

template <int HD>
int launch_fused_hd(const AttnMaps& maps, const AttnFusedArgs& f, cudaStream_t s) {
    const int qrows = (f.m.n_q / f.m.n_kv) * 16;
    const size_t smem = fused_smem<HD>(qrows);
    static bool set = false;
    if (!set) {
        const cudaError_t e = cudaFuncSetAttribute(attn_fused_kernel<HD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        set = true;
    }
    if (f.tc) {
        if (f.split_chunks == 1) return launch_tc<HD, 1>(maps, f, s);
        if (f.split_chunks == 2) return launch_tc<HD, 2>(maps, f, s);
        return (int)cudaErrorInvalidValue;
    }
    return (int)launch_k(attn_fused_kernel<HD>, dim3(f.m.n_kv, f.max_splits), dim3(128), smem, s, maps, f);
}

int launch_prefill_attention(const CUtensorMap& q_map, const CUtensorMap& kv_map, const PrefillAttnArgs& p,
                             cudaStream_t s) {
    if (p.rows < 1) return 0;
    if (p.m.head_dim == 128) return launch_prefill_hd<128>(q_map, kv_map, p, s);
    if (p.m.head_dim == 64) return launch_prefill_hd<64>(q_map, kv_map, p, s);
    return (int)cudaErrorInvalidValue;
}

int launch_batch_attention(const CUtensorMap& q_map, const CUtensorMap& kv_map, const BatchAttnArgs& b,
                           int S, cudaStream_t s) {
    if (b.m.head_dim == 128) return launch_batch_hd<128>(q_map, kv_map, b, S, s);
    if (b.m.head_dim == 64) return launch_batch_hd<64>(q_map, kv_map, b, S, s);
    return (int)cudaErrorInvalidValue;
}

int launch_attention_fused(const AttnMaps& maps, const AttnFusedArgs& f, cudaStream_t s) {
    if (f.m.head_dim == 128) return launch_fused_hd<128>(maps, f, s);
    if (f.m.head_dim == 64) return launch_fused_hd<64>(maps, f, s);
    return (int)cudaErrorInvalidValue;
}

int attention_fused_per_sm(int hd, int n_q, int n_kv, int* out) {
    const int qrows = (n_q / n_kv) * 16;
    *out = 0;
    cudaError_t e;
    if (hd == 128) {
        const size_t smem = fused_smem<128>(qrows);
        set_carveout_once(reinterpret_cast<const void*>(attn_fused_kernel<128>));
        e = cudaFuncSetAttribute(attn_fused_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, attn_fused_kernel<128>, 128, smem);
    } else {
        const size_t smem = fused_smem<64>(qrows);
        set_carveout_once(reinterpret_cast<const void*>(attn_fused_kernel<64>));
        e = cudaFuncSetAttribute(attn_fused_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, attn_fused_kernel<64>, 128, smem);
    }
    return (int)e;
}

int attention_tc_per_sm(int hd, int nc, int* out, int* tmem_cols) {
    *out = 0;
    if (nc == 1) return hd == 128 ? tc_per_sm<128, 1>(out, tmem_cols) : tc_per_sm<64, 1>(out, tmem_cols);
    if (nc == 2) return hd == 128 ? tc_per_sm<128, 2>(out, tmem_cols) : tc_per_sm<64, 2>(out, tmem_cols);
    return (int)cudaErrorInvalidValue;
}

}  // namespace dfl
