// Shared device helpers of the DFlash sm_103a library: error word, device
// round state, mbarrier / TMA / mma.sync inline PTX, small math.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DFL_MAX_ROWS 16  // rows of one forward (block_max and prefill chunk)

// Device error word values (first error wins).
enum : int {
    DERR_NONE = 0,
    DERR_TIMEOUT = 1,   // a bounded mbarrier wait expired
    DERR_INDEX = 2,     // an index outside its buffer was requested and skipped
    DERR_TOKEN = 3,     // a token id outside [0, vocab)
};

// Round state held in device memory (one per context).
struct DevState {
    int n;           // target KV length = position of the pending token
    int t_n;         // pending token
    int bl;          // block length of the next round
    int generated;   // tokens emitted so far (the prefill's first included)
    int max_new;     // generation budget
    int ctx_len;     // committed draft context rows
    int finished;
    int last_a;
    int err;         // device error word
    int err_info;
    // descriptor of the forward in flight
    int fwd_pos0;    // position of row 0
    int fwd_T;       // rows in this forward
    int fwd_commit;  // rows whose taps are committed to the draft context ...
    int fwd_commit_r0;  // ... starting at this row of the forward
    int draft_bl;    // block length the last draft used
    int pad_;
    long long rounds, emitted;
    long long accept_hist[16];
    float acc_ema;   // adaptive block: running average of accepted drafts
    int adaptive;    // 1: the next block is capped from acc_ema
};

#include <utility>

namespace dfl {
// Rows a kernel writes: the forward's rows, or the rows committed to the
// draft context (both at absolute position fwd_pos0 + row).
enum RowSel : int { ROWS_FWD = 0, ROWS_COMMIT = 1 };

// Kernels launched through the library by this process (host counter).
extern long long g_launches;
// Programmatic dependent launch on (default) or off (environment DFLASH_PDL=0).
extern bool g_pdl;

// Launches a kernel on stream s with programmatic stream serialisation: the
// kernel may be scheduled while its predecessor drains; every kernel of the
// library calls pdl_wait() before it touches memory a predecessor writes.
// Shared-memory carveout every kernel of the library asks for (percent of
// the unified L1/shared array; -1 leaves the choice to the driver).  One
// value for all kernels keeps the SMs from reconfiguring the split between
// consecutive kernels of a round.
#ifndef DFL_SMEM_CARVEOUT
#define DFL_SMEM_CARVEOUT 100
#endif
void set_carveout_once(const void* kern);

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args&&... args) {
    set_carveout_once(reinterpret_cast<const void*>(kern));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ++g_launches;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
}  // namespace dfl

// Programmatic dependent launch: let the next kernel be scheduled now /
// wait until every predecessor has finished and its writes are visible.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

namespace dfl {
// Row range [*r0, *r0 + n) a kernel with row selection `sel` works on.
__device__ __forceinline__ int rows_of(const DevState* st, int sel, int* r0) {
    if (sel == ROWS_COMMIT) {
        *r0 = st->fwd_commit_r0;
        return st->fwd_commit;
    }
    *r0 = 0;
    return st->fwd_T;
}
}  // namespace dfl

// Block length cap of the next round: the native block, or with the
// adaptive policy 4 / 8 / 16 rows (3 / 7 / 15 drafts) from the running
// average of accepted drafts (< 1.5, < 4.5, else).
__device__ __forceinline__ int block_cap(const DevState* st, int B) {
    if (!st->adaptive) return B;
    const float e = st->acc_ema;
    const int cap = e < 1.5f ? 4 : (e < 4.5f ? 8 : 16);
    return cap < B ? cap : B;
}

__device__ __forceinline__ void set_error(DevState* st, int code, int info) {
    if (atomicCAS(&st->err, 0, code) == 0) st->err_info = info;
}

// ------------------------------------------------------------------ math

__device__ __forceinline__ float warp_sum(float v) {
    // butterfly: the same fixed order on every call
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger int).
__device__ __forceinline__ uint32_t float_orderable(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Packed argmax key: (orderable logit << 32) | (0xFFFFFFFF - index):
// atomicMax keeps the largest logit and, among equal logits, the lowest index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    return ((unsigned long long)float_orderable(v) << 32) |
           (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
    return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after `limit_ns` of wall time and returns false.
// No wait in this library is unbounded.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(dst)), "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// L2 prefetch of a 2-D tile (no shared memory, no completion to wait for)
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];"
                 ::"l"((uint64_t)map), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// 1D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------ mma.sync

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// 16-byte shared-memory load.
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// Byte offset of logical 16-byte chunk `chunk` (0..7) of row `row` inside a
// tile written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (128-byte rows, the
// pattern repeating every 8 rows; the tile base is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
