// Gated RMSNorm of the rule's outputs, the step right after the rule: per
// (token, V head) row of d values,
//     y = w * o / sqrt(mean(o^2) + eps) * silu(z),   silu(z) = z sigmoid(z),
// with one weight per channel.  The Qwen3.5-9B NPU model card ("fp16 precision
// of the DeltaNet output") places a gated RMSNorm right after the rule; the
// Candle PR's bug log ("Bug 7") gives its epsilon, 1e-6.  The gate's form,
// silu(z), is not on the pages (a reading).
//
// One warp per row (d / 32 consecutive values per lane, one vector access each
// for o, z and y), two rows in flight per warp, grid-stride over the rows: a pass
// that reads o and z once and writes y once (HBM-bound).
#include <cuda_bf16.h>

#include "gdr_common.cuh"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {
namespace {

using tc::pack_bf16x2;

// PER consecutive values of a row, fp32 or bf16, in one vector access per lane
// where PER x the element size is 8 or 16 bytes.
template <int PER>
__device__ __forceinline__ void load_row(const void *p, size_t i, int is_bf16, float (&v)[PER]) {
    if (is_bf16) {
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(p) + i;
        if constexpr (PER == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(b);
            v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
            v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) v[j] = __bfloat162float(b[j]);
        }
    } else {
        const float *f = reinterpret_cast<const float *>(p) + i;
        if constexpr (PER == 4) {
            const float4 u = *reinterpret_cast<const float4 *>(f);
            v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        } else if constexpr (PER == 2) {
            const float2 u = *reinterpret_cast<const float2 *>(f);
            v[0] = u.x; v[1] = u.y;
        } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) v[j] = f[j];
        }
    }
}
template <int PER>
__device__ __forceinline__ void store_row(void *p, size_t i, int is_bf16, const float (&v)[PER]) {
    if (is_bf16) {
        __nv_bfloat16 *b = reinterpret_cast<__nv_bfloat16 *>(p) + i;
        if constexpr (PER == 4) {
            *reinterpret_cast<uint2 *>(b) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) b[j] = __float2bfloat16_rn(v[j]);
        }
    } else {
        float *f = reinterpret_cast<float *>(p) + i;
        if constexpr (PER == 4) {
            *reinterpret_cast<float4 *>(f) = make_float4(v[0], v[1], v[2], v[3]);
        } else if constexpr (PER == 2) {
            *reinterpret_cast<float2 *>(f) = make_float2(v[0], v[1]);
        } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) f[j] = v[j];
        }
    }
}

// One warp per row, NR rows in flight per warp and step (every row's loads are
// issued before any is reduced), grid-stride over the rows; lane l holds a row's
// values l * PER .. + PER - 1.
template <int D>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(int64_t rows, const void *o, int o_bf16, const void *z,
                                                            int z_bf16, const float *__restrict__ w, float eps,
                                                            void *y, int y_bf16) {
    constexpr int PER = D / 32;  // values per lane
    constexpr int NR = 2;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    float wv[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) wv[i] = w[lane * PER + i];
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += NR * warps) {
        float ov[NR][PER], zv[NR][PER];
#pragma unroll
        for (int h = 0; h < NR; ++h) {
            const int64_t rh = r + h * warps;  // warp-uniform
            if (rh < rows) {
                load_row<PER>(o, (size_t)rh * D + lane * PER, o_bf16, ov[h]);
                load_row<PER>(z, (size_t)rh * D + lane * PER, z_bf16, zv[h]);
            }
        }
#pragma unroll
        for (int h = 0; h < NR; ++h) {
            const int64_t rh = r + h * warps;
            if (rh >= rows) break;
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < PER; ++i) ss = fmaf(ov[h][i], ov[h][i], ss);
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss / D + eps);
            float yv[PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) yv[i] = wv[i] * ov[h][i] * inv * silu(zv[h][i]);
            store_row<PER>(y, (size_t)rh * D + lane * PER, y_bf16, yv);
        }
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
