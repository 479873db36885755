// Device helpers shared by the row kernels and the dense GEMM's epilogues.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace dfl {

// v as a hi/lo pair of planes: hi = v rounded, lo = the rounding remainder
// rounded (bf16, or f16 with f16 set), element i of each plane.
__device__ __forceinline__ void store_hilo(void* hi, void* lo, size_t i, float v, int f16 = 0) {
    if (f16) {
        const __half h = __float2half_rn(v);
        reinterpret_cast<__half*>(hi)[i] = h;
        reinterpret_cast<__half*>(lo)[i] = __float2half_rn(v - __half2float(h));
        return;
    }
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    reinterpret_cast<__nv_bfloat16*>(hi)[i] = h;
    reinterpret_cast<__nv_bfloat16*>(lo)[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// SwiGLU of one gate / up pair, in the order every path computes it.
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.f + expf(-g)) * u; }

}  // namespace dfl
