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
#include "gemm.cuh"

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
    if (tid == 0 && (a.causal || a.window <= 0)) {
        const int np = min(f.split_chunks, 2);
        for (int i = 0; i < np; ++i) {
            const int c = sp * f.split_chunks + i;
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
    return (int)launch_k(attn_fused_kernel<HD>, dim3(f.m.n_kv, f.max_splits), dim3(128), smem, s, maps, f);
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
        e = cudaFuncSetAttribute(attn_fused_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, attn_fused_kernel<128>, 128, smem);
    } else {
        const size_t smem = fused_smem<64>(qrows);
        e = cudaFuncSetAttribute(attn_fused_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, attn_fused_kernel<64>, 128, smem);
    }
    return (int)e;
}

}  // namespace dfl
