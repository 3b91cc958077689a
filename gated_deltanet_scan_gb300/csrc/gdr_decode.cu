// Batched decode step: one token per sequence, the state streamed through once.
//
// Math (the 1-token matrix form on the Qwen3.5-9B NPU model card, "How it
// works"): with d = exp(g), y = S^T k, z = S^T q, delta = beta (v - d y):
//     o = scale (d z + (q.k) delta),      S' = d S + k delta^T.
//
// Design.  The op is bound by HBM: each (sequence, V head) reads and writes its
// d x d fp32 state once (128 KiB for d = 128) and touches only ~1 KiB of
// q/k/v/o.  One 256-thread block owns one (sequence, V head).  Lane l of every
// warp owns the same d/32 adjacent columns; warp w owns d/8 rows, so each warp
// load is one fully coalesced 512-byte row slab (float4 per lane at d = 128).
// The slab stays in registers: partial S^T k and S^T q over the warp's rows go
// through shared memory once to reduce over the 8 warps, then every thread
// forms delta for its columns and writes d S + k delta^T straight from its
// registers.  Loads and stores carry streaming (evict-first) hints because the
// state is touched exactly once per step.
#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int D>
struct Vec;
template <>
struct Vec<32> {
    using T = float;
    static __device__ __forceinline__ void split(const T &v, float *f) { f[0] = v; }
    static __device__ __forceinline__ T pack(const float *f) { return f[0]; }
};
template <>
struct Vec<64> {
    using T = float2;
    static __device__ __forceinline__ void split(const T &v, float *f) {
        f[0] = v.x;
        f[1] = v.y;
    }
    static __device__ __forceinline__ T pack(const float *f) { return make_float2(f[0], f[1]); }
};
template <>
struct Vec<128> {
    using T = float4;
    static __device__ __forceinline__ void split(const T &v, float *f) {
        f[0] = v.x;
        f[1] = v.y;
        f[2] = v.z;
        f[3] = v.w;
    }
    static __device__ __forceinline__ T pack(const float *f) {
        return make_float4(f[0], f[1], f[2], f[3]);
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(Args a) {
    constexpr int CPL = D / 32;     // columns per lane
    constexpr int RPW = D / kWarps;  // rows per warp
    using V = Vec<D>;
    using VT = typename V::T;

    __shared__ float sk[D], sq[D];
    __shared__ float red[2][kWarps][D];
    __shared__ float s_qk;

    const int bh = blockIdx.x;
    const int b = bh / a.h_v, h = bh - b * a.h_v;
    const int hq = h / (a.h_v / a.h_qk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = lane * CPL;

    // Issue the state loads first: they are the only HBM-heavy traffic.
    VT *S = reinterpret_cast<VT *>(a.state + ((size_t)b * a.h_v + h) * D * D);
    VT sv[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) sv[r] = __ldcs(&S[(size_t)(warp * RPW + r) * (D / CPL) + lane]);

    const size_t qk_off = ((size_t)b * a.h_qk + hq) * D;
    for (int i = threadIdx.x; i < D; i += kThreads) {
        sk[i] = load_in(a.k, qk_off + i, a.in_bf16);
        sq[i] = load_in(a.q, qk_off + i, a.in_bf16);
    }
    const size_t vh = (size_t)b * a.h_v + h;
    const float dgate = __expf(a.g[vh]);
    const float bt = a.beta[vh];
    float vv[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) vv[c] = load_in(a.v, vh * D + col0 + c, a.in_bf16);
    __syncthreads();

    float y[CPL], z[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) y[c] = z[c] = 0.f;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        float f[CPL];
        V::split(sv[r], f);
        const float kr = sk[warp * RPW + r], qr = sq[warp * RPW + r];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            y[c] = fmaf(f[c], kr, y[c]);
            z[c] = fmaf(f[c], qr, z[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        red[0][warp][col0 + c] = y[c];
        red[1][warp][col0 + c] = z[c];
    }
    if (warp == 0) {
        float p = 0.f;
        for (int i = lane; i < D; i += 32) p = fmaf(sk[i], sq[i], p);
        p = warp_sum(p);
        if (lane == 0) s_qk = p;
    }
    __syncthreads();

    float delta[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        float yt = 0.f, zt = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            yt += red[0][w][col0 + c];
            zt += red[1][w][col0 + c];
        }
        delta[c] = bt * (vv[c] - dgate * yt);
        z[c] = zt;
    }
    if (warp == 0) {
        const float qk = s_qk;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            store_out(a.o, vh * D + col0 + c, a.scale * fmaf(dgate, z[c], qk * delta[c]), a.out_bf16);
    }

#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        float f[CPL];
        V::split(sv[r], f);
        const float kr = sk[warp * RPW + r];
#pragma unroll
        for (int c = 0; c < CPL; ++c) f[c] = fmaf(dgate, f[c], kr * delta[c]);
        __stcs(&S[(size_t)(warp * RPW + r) * (D / CPL) + lane], V::pack(f));
    }
}

}  // namespace

cudaError_t launch_decode(const Args &a, cudaStream_t s) {
    const unsigned blocks = (unsigned)a.n_seqs * (unsigned)a.h_v;
    if (blocks == 0) return cudaSuccess;
    switch (a.d) {
        case 32: decode_kernel<32><<<blocks, kThreads, 0, s>>>(a); break;
        case 64: decode_kernel<64><<<blocks, kThreads, 0, s>>>(a); break;
        case 128: decode_kernel<128><<<blocks, kThreads, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdr
