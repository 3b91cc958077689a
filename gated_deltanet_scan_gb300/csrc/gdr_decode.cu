// Batched decode step: one token per sequence, the state streamed through once.
//
// Math (the 1-token matrix form on the Qwen3.5-9B NPU model card, "How it
// works"): with d = exp(g), y = S^T k, z = S^T q, delta = beta (v - d y):
//     o = scale (d z + (q.k) delta),      S' = d S + k delta^T.
//
// Design.  The op is bound by HBM: each (sequence, V head) reads and writes its
// d x d fp32 state once (128 KiB for d = 128) and touches only ~1 KiB of
// q/k/v/o.  One 256-thread block owns one (sequence, V head).  One thread
// brings the whole state into shared memory with bulk asynchronous copies
// completed on an mbarrier, so a block holds no state in registers (about 40
// of them) and three blocks fit on an SM (3 x 64 KiB in flight at d = 128):
// the SM keeps more bytes moving than with the state held in registers, which
// matters most when the step shares the GPU with other work.  Thread t owns
// column quad t % (d/4) of every (256 / (d/4))-th row: a warp reads whole rows
// from shared memory, conflict free.  The partial S^T k and S^T q of its rows
// go through shared memory once to reduce over the row groups; then every
// thread forms delta for its columns, re-reads its rows and writes d S + k
// delta^T straight to HBM with streaming (evict-first) stores.  The wait on
// the copies is bounded: on timeout the block records GDR_ERR_DEVICE_TIMEOUT
// and leaves the state as it was.
#include "gdr_common.cuh"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr long long kWaitLimit = 4000000000LL;  // SM clocks (about 2 s)

template <int D>
struct DecShape {
    static constexpr int Q4 = D / 4;            // column quads per row
    static constexpr int RSTEP = kThreads / Q4;  // row groups (rows between a thread's rows)
    static constexpr int NR = D / RSTEP;         // rows per thread
    static constexpr uint32_t SBYTES = D * D * 4;
    static constexpr uint32_t NCOPY = SBYTES > 16384 ? SBYTES / 16384 : 1;  // bulk copies of <= 16 KiB
    static constexpr uint32_t CBYTES = SBYTES / NCOPY;
    // dynamic shared memory: state, then one partial-sum table (y, then z), then the mbarrier
    static constexpr uint32_t OFF_RED = SBYTES;
    static constexpr uint32_t OFF_BAR = OFF_RED + RSTEP * D * 4;
    static constexpr uint32_t SMEM = OFF_BAR + 16;
};

template <int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(Args a, int32_t *err) {
    using Sh = DecShape<D>;
    extern __shared__ __align__(128) uint8_t dsm[];
    float4 *sS = reinterpret_cast<float4 *>(dsm);
    float *red = reinterpret_cast<float *>(dsm + Sh::OFF_RED);  // [RSTEP][D]
    const uint32_t bar = smem_u32(dsm + Sh::OFF_BAR);
    __shared__ float sk[D], sq[D];
    __shared__ float s_qk, s_rk, s_rq;

    const int bh = blockIdx.x;
    const int b = bh / a.h_v, h = bh - b * a.h_v;
    const int hq = h / (a.h_v / a.h_qk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cq = tid % Sh::Q4, rg = tid / Sh::Q4;

    float *S = a.state + (size_t)bh * D * D;
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, Sh::SBYTES);
#pragma unroll
        for (uint32_t i = 0; i < Sh::NCOPY; ++i)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(dsm) + i * Sh::CBYTES),
                "l"(reinterpret_cast<uint64_t>(S) + i * Sh::CBYTES), "r"(Sh::CBYTES), "r"(bar)
                : "memory");
    }
    const size_t qk_off = ((size_t)b * a.h_qk + hq) * D;
    for (int i = tid; i < D; i += kThreads) {
        sk[i] = load_in(a.k, qk_off + i, a.in_bf16);
        sq[i] = load_in(a.q, qk_off + i, a.in_bf16);
    }
    const size_t vh = (size_t)b * a.h_v + h;
    const float dgate = __expf(a.g[vh]);
    const float bt = beta_of(a.beta[vh], a.beta_logits);
    float vv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) vv[c] = load_in(a.v, vh * D + 4 * cq + c, a.in_bf16);
    // the gated RMSNorm's gate and weights for the output row (row group 0), loaded
    // with the other vectors, off the path after the reductions
    float gz[4] = {0.f, 0.f, 0.f, 0.f}, gw[4] = {0.f, 0.f, 0.f, 0.f};
    if (a.norm_z && rg == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            gz[c] = silu(load_in(a.norm_z, vh * D + 4 * cq + c, a.in_bf16));
            gw[c] = a.norm_w[4 * cq + c];
        }
    }
    __syncthreads();  // the mbarrier is initialised, sk and sq are written
    if (a.qk_norm && warp < 2) {
        // fused L2 normalisation: per-row scales of k (warp 0) and q (warp 1)
        const float *x = warp == 0 ? sk : sq;
        float ss = 0.f;
        for (int i = lane; i < D; i += 32) ss = fmaf(x[i], x[i], ss);
        ss = warp_sum(ss);
        if (lane == 0) (warp == 0 ? s_rk : s_rq) = l2norm_scale(ss);
    }
    const bool ok = mbar_wait_bounded(bar, 0, kWaitLimit);
    if (!__syncthreads_and(ok)) {
        // leave the state untouched; let the copies land before the block's shared memory is released
        if (tid == 0) {
            atomicCAS(err, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
            mbar_wait_bounded(bar, 0, kWaitLimit / 8);
        }
        __syncthreads();
        return;
    }

    // partial y = S^T k and z = S^T q over this thread's rows, for its 4 columns
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f), z = y;
#pragma unroll
    for (int i = 0; i < Sh::NR; ++i) {
        const int r = rg + i * Sh::RSTEP;
        const float4 sv = sS[r * Sh::Q4 + cq];
        const float kr = sk[r], qr = sq[r];
        y.x = fmaf(sv.x, kr, y.x);
        y.y = fmaf(sv.y, kr, y.y);
        y.z = fmaf(sv.z, kr, y.z);
        y.w = fmaf(sv.w, kr, y.w);
        z.x = fmaf(sv.x, qr, z.x);
        z.y = fmaf(sv.y, qr, z.y);
        z.z = fmaf(sv.z, qr, z.z);
        z.w = fmaf(sv.w, qr, z.w);
    }
    // sum the row groups' partials: y first, then z through the same table
    *reinterpret_cast<float4 *>(red + rg * D + 4 * cq) = y;
    if (warp == 0) {
        float pq = 0.f;
        for (int i = lane; i < D; i += 32) pq = fmaf(sk[i], sq[i], pq);
        pq = warp_sum(pq);
        if (lane == 0) s_qk = pq;
    }
    __syncthreads();
    // with the fused normalisation the sums above used the raw k and q: scale them
    const float rk = a.qk_norm ? s_rk : 1.f, rq = a.qk_norm ? s_rq : 1.f;
    float delta[4], zt[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float ys = 0.f;
#pragma unroll 8
        for (int w = 0; w < Sh::RSTEP; ++w) ys += red[w * D + 4 * cq + c];
        delta[c] = bt * (vv[c] - dgate * rk * ys);
    }
    __syncthreads();
    *reinterpret_cast<float4 *>(red + rg * D + 4 * cq) = z;
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float zs = 0.f;
#pragma unroll 8
        for (int w = 0; w < Sh::RSTEP; ++w) zs += red[w * D + 4 * cq + c];
        zt[c] = rq * zs;
    }
    if (rg == 0) {
        // row group 0 (lanes 0 .. D/4 - 1 of warp 0) holds the whole output row
        const float qk = s_qk * rq * rk;
        float ov[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) ov[c] = a.scale * fmaf(dgate, zt[c], qk * delta[c]);
        if (a.norm_z) {
            // gated RMSNorm of the row, fused: y = w o / sqrt(mean(o^2) + eps) silu(z)
            constexpr unsigned kMask = Sh::Q4 == 32 ? 0xffffffffu : ((1u << Sh::Q4) - 1u);
            float ss = ov[0] * ov[0] + ov[1] * ov[1] + ov[2] * ov[2] + ov[3] * ov[3];
#pragma unroll
            for (int off = Sh::Q4 / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(kMask, ss, off);
            const float inv = rsqrtf(ss / D + a.norm_eps);
#pragma unroll
            for (int c = 0; c < 4; ++c) ov[c] = gw[c] * ov[c] * inv * gz[c];
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) store_out(a.o, vh * D + 4 * cq + c, ov[c], a.out_bf16);
    }

    // S' = d S + k delta^T, from shared memory straight to HBM
    float4 *Sg = reinterpret_cast<float4 *>(S);
#pragma unroll
    for (int i = 0; i < Sh::NR; ++i) {
        const int r = rg + i * Sh::RSTEP;
        const float4 sv = sS[r * Sh::Q4 + cq];
        const float kr = rk * sk[r];
        const float4 nv = make_float4(fmaf(dgate, sv.x, kr * delta[0]), fmaf(dgate, sv.y, kr * delta[1]),
                                      fmaf(dgate, sv.z, kr * delta[2]), fmaf(dgate, sv.w, kr * delta[3]));
        __stcs(&Sg[r * Sh::Q4 + cq], nv);
    }
}

template <int D>
cudaError_t launch_d(const Args &a, int32_t *err, unsigned blocks, cudaStream_t s, bool overlap) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)DecShape<D>::SMEM);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = DecShape<D>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = overlap ? &attr : nullptr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_kernel<D>, a, err);
}

}  // namespace

cudaError_t launch_decode(const Args &a, int32_t *err, cudaStream_t s, bool overlap) {
    const unsigned blocks = (unsigned)a.n_seqs * (unsigned)a.h_v;
    if (blocks == 0) return cudaSuccess;
    switch (a.d) {
        case 32: return launch_d<32>(a, err, blocks, s, overlap);
        case 64: return launch_d<64>(a, err, blocks, s, overlap);
        case 128: return launch_d<128>(a, err, blocks, s, overlap);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdr
