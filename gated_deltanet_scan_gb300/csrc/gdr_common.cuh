// Small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

__device__ __forceinline__ float load_in(const void *p, size_t i, int is_bf16) {
    if (is_bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return reinterpret_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_out(void *p, size_t i, float x, int is_bf16) {
    if (is_bf16)
        reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float *>(p)[i] = x;
}

// Sequence bounds: packed by cu_seqlens, or fixed-length blocks.
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int fixed_len, int s, int64_t &t0,
                                           int64_t &t1) {
    if (cu) {
        t0 = cu[s];
        t1 = cu[s + 1];
    } else {
        t0 = (int64_t)s * fixed_len;
        t1 = t0 + fixed_len;
    }
}

// The epsilon of the fused q/k L2 normalisation (inside the square root).
constexpr float kL2NormEps = 1e-6f;

// 1 / sqrt(sum x^2 + eps) from a sum of squares.
__device__ __forceinline__ float l2norm_scale(float sumsq) { return rsqrtf(sumsq + kL2NormEps); }

// beta from its input: the value itself, or sigmoid of a logit.
__device__ __forceinline__ float beta_of(float b, int logits) { return logits ? 1.f / (1.f + __expf(-b)) : b; }

// silu(z) = z sigmoid(z), the gate of the output RMSNorm.
__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace gdr
