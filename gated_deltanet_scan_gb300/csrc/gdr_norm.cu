// Gated RMSNorm of the rule's outputs, the step right after the rule: per
// (token, V head) row of d values,
//     y = w * o / sqrt(mean(o^2) + eps) * silu(z),   silu(z) = z sigmoid(z),
// with one weight per channel.  The Qwen3.5-9B NPU model card ("fp16 precision
// of the DeltaNet output") places a gated RMSNorm right after the rule; the
// Candle PR's bug log ("Bug 7") gives its epsilon, 1e-6.  The gate's form,
// silu(z), is not on the pages (a reading).
//
// One warp per row (d / 32 values per lane, vector loads), grid-stride over the
// rows: a pass that reads o and z once and writes y once (HBM-bound).
#include <cuda_bf16.h>

#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

template <int D>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(int64_t rows, const void *o, int o_bf16, const void *z,
                                                            int z_bf16, const float *__restrict__ w, float eps,
                                                            void *y, int y_bf16) {
    constexpr int PER = D / 32;  // values per lane
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    float wv[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) wv[i] = w[lane * PER + i];
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const size_t base = (size_t)r * D + lane * PER;
        float ov[PER], zv[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            ov[i] = load_in(o, base + i, o_bf16);
            zv[i] = load_in(z, base + i, z_bf16);
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) ss = fmaf(ov[i], ov[i], ss);
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / D + eps);
#pragma unroll
        for (int i = 0; i < PER; ++i) store_out(y, base + i, wv[i] * ov[i] * inv * silu(zv[i]), y_bf16);
    }
}

}  // namespace

cudaError_t launch_gated_rmsnorm(int64_t rows, int d, const void *o, int o_bf16, const void *z, int z_bf16,
                                 const float *w, float eps, void *y, int y_bf16, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    int64_t blocks64 = (rows + 7) / 8;
    if (blocks64 > 152 * 16) blocks64 = 152 * 16;
    const unsigned blocks = (unsigned)blocks64;
    switch (d) {
        case 32: gated_rmsnorm_kernel<32><<<blocks, 256, 0, s>>>(rows, o, o_bf16, z, z_bf16, w, eps, y, y_bf16); break;
        case 64: gated_rmsnorm_kernel<64><<<blocks, 256, 0, s>>>(rows, o, o_bf16, z, z_bf16, w, eps, y, y_bf16); break;
        case 128: gated_rmsnorm_kernel<128><<<blocks, 256, 0, s>>>(rows, o, o_bf16, z, z_bf16, w, eps, y, y_bf16); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdr
