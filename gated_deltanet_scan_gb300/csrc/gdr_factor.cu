// State-independent factors of the chunked prefill, computed for every chunk at
// once (no chunk depends on another): one CTA per (chunk, QK head) writes, for
// each V head that reads this QK head, the chunk's gates, T = (I + N)^-1 and
// P T into the factor workspace (layout in gdr_factor_layout.h).
//
// Per chunk (the chunkwise-parallel form of the Qwen3.5-9B NPU model card,
// "How it works"; forward substitution for the unit triangular factor as in
// the Candle PR's "Chunked GatedDeltaNet Scan"; log-space masking from its
// "Float32 overflow fix"):
//   G   = inclusive running sum of g over the chunk (padding rows: g = beta = 0)
//   [K Kᵀ; Q Kᵀ] = [K; Q] Kᵀ                    one M=128 tcgen05 MMA group, exact
//                                               bf16 products, fp32 accumulation
//   N   = diag(beta) (K Kᵀ ⊙ exp(G_t - G_j))_{j<t}
//   P   =            (Q Kᵀ ⊙ exp(G_t - G_j))_{j<=t}
//         (the exponent is formed only on the kept triangle, so it never overflows)
//   T   = (I + N)^-1            fp32 on the CUDA cores: the four 16x16 diagonal
//                               blocks by forward substitution, then two block-
//                               doubling levels T21 = -T22 N21 T11 (16 -> 32 -> 64)
//   P T                         fp32 on the CUDA cores, blockwise lower triangular
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdr_common.cuh"
#include "gdr_factor_layout.h"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {
namespace {

using namespace tc;

constexpr int C = fac::C;
constexpr int NT = 256;
constexpr int SROW = 68;  // fp32 row stride of the 64 x 64 scratch matrices (floats)
constexpr int XROW = 34;  // row stride of the block-doubling partial products

// Shared memory, bytes from a 1024-byte aligned base.  The [K; Q] tile is only
// read by the Gram MMA; once that has completed, N and P overwrite it.
constexpr uint32_t MAT_BYTES = 64 * SROW * 4;           // 17408
constexpr uint32_t OFF_KQ = 0;                          // 32 KB, [K rows 0-63; Q rows 64-127] x 2 K-halves
constexpr uint32_t OFF_N = 0;                           // N, later P T
constexpr uint32_t OFF_P = MAT_BYTES;
constexpr uint32_t OFF_T = 2 * MAT_BYTES;
constexpr uint32_t OFF_X = 3 * MAT_BYTES;               // [32][XROW]
constexpr uint32_t OFF_GATES = OFF_X + 32 * XROW * 4;   // G log2(e), beta, exp(G): 3 x 64 floats
constexpr uint32_t OFF_SCAN = OFF_GATES + 768;
constexpr uint32_t OFF_BARS = OFF_SCAN + 16;            // 2 mbarriers
constexpr uint32_t OFF_TMEM = OFF_BARS + 16;
constexpr uint32_t SMEM_USED = OFF_TMEM + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(2 * MAT_BYTES >= 32768, "N and P cover the K/Q tile");
static_assert(OFF_GATES % 16 == 0 && OFF_BARS % 8 == 0, "alignment");

constexpr uint32_t TM_COLS = 64;  // [K Kᵀ; Q Kᵀ], 128 lanes x 64 fp32 columns
constexpr uint32_t IDESC_G1 = idesc_bf16_f32(128, 64, 0, 0);
constexpr long long kWaitLimit = 4000000000LL;
constexpr float kLog2e = 1.4426950408889634f;

struct FacParams {
    int h_qk, h_v, n_seqs;
    int64_t t_total;
    const int32_t *cu_seqlens;
    const float *g, *beta;
    float *ws;
    int32_t *err;
};

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// T = (I + N)^-1 for strictly lower N; both fp32 [64][SROW].  Entries of T above
// the 16-block diagonal are left unwritten; everything on or below it is final.
__device__ void unit_lower_inverse(const float *N, float *T, float *X, int tid) {
    // diagonal 16 x 16 blocks: column jj of block I by right-looking substitution
    if (tid < 64) {
        const int I = tid >> 4, jj = tid & 15, base = 16 * I;
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) col[r] = (r == jj) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 15; ++m) {
#pragma unroll
            for (int r = m + 1; r < 16; ++r) col[r] = fmaf(-N[(base + r) * SROW + base + m], col[m], col[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(base + r) * SROW + base + jj] = col[r];
    }
    __syncthreads();
    // level 1: T_{I,I-1} = -T_II (N_{I,I-1} T_{I-1,I-1}) for I = 1 and 3
    {
        const int blk = tid >> 7, I = 2 * blk + 1, J = I - 1, r = (tid >> 3) & 15, cc = (tid & 7) * 2;
        const float *nr = N + (16 * I + r) * SROW + 16 * J;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float2 tv = *reinterpret_cast<const float2 *>(T + (16 * J + m) * SROW + 16 * J + cc);
            a0 = fmaf(nr[m], tv.x, a0);
            a1 = fmaf(nr[m], tv.y, a1);
        }
        *reinterpret_cast<float2 *>(X + (16 * blk + r) * XROW + cc) = make_float2(a0, a1);
    }
    __syncthreads();
    {
        const int blk = tid >> 7, I = 2 * blk + 1, J = I - 1, r = (tid >> 3) & 15, cc = (tid & 7) * 2;
        const float *tr = T + (16 * I + r) * SROW + 16 * I;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float2 xv = *reinterpret_cast<const float2 *>(X + (16 * blk + m) * XROW + cc);
            a0 = fmaf(tr[m], xv.x, a0);
            a1 = fmaf(tr[m], xv.y, a1);
        }
        *reinterpret_cast<float2 *>(T + (16 * I + r) * SROW + 16 * J + cc) = make_float2(-a0, -a1);
    }
    __syncthreads();
    // level 2: T[32:64, 0:32] = -T[32:64, 32:64] (N[32:64, 0:32] T[0:32, 0:32]), 2 x 2 per thread
    const int r0 = (tid >> 4) * 2, c0 = (tid & 15) * 2;
    {
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        const float *n0 = N + (32 + r0) * SROW, *n1 = n0 + SROW;
        for (int m = c0; m < 32; ++m) {  // T[0:32, 0:32] is lower: rows m >= c0 only
            const float2 tv = *reinterpret_cast<const float2 *>(T + m * SROW + c0);
            const float u0 = n0[m], u1 = n1[m];
            a00 = fmaf(u0, tv.x, a00);
            a01 = fmaf(u0, tv.y, a01);
            a10 = fmaf(u1, tv.x, a10);
            a11 = fmaf(u1, tv.y, a11);
        }
        *reinterpret_cast<float2 *>(X + r0 * XROW + c0) = make_float2(a00, a01);
        *reinterpret_cast<float2 *>(X + (r0 + 1) * XROW + c0) = make_float2(a10, a11);
    }
    __syncthreads();
    {
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        const float *t0 = T + (32 + r0) * SROW + 32, *t1 = t0 + SROW;
        for (int m = 0; m <= r0 + 1; ++m) {  // T[32:64, 32:64] is lower: columns m <= row
            const float2 xv = *reinterpret_cast<const float2 *>(X + m * XROW + c0);
            const float u0 = t0[m], u1 = t1[m];
            a00 = fmaf(u0, xv.x, a00);
            a01 = fmaf(u0, xv.y, a01);
            a10 = fmaf(u1, xv.x, a10);
            a11 = fmaf(u1, xv.y, a11);
        }
        *reinterpret_cast<float2 *>(T + (32 + r0) * SROW + c0) = make_float2(-a00, -a01);
        *reinterpret_cast<float2 *>(T + (33 + r0) * SROW + c0) = make_float2(-a10, -a11);
    }
    __syncthreads();
}

// PT = P T for lower-triangular P and T (fp32 [64][SROW]); only blocks on or
// below the 16-block diagonal are formed.  The ten blocks are split into four
// groups of equal work (counted in 16x16x16 products: block (I, J) costs
// I - J + 1), one group per 64 threads, 2 x 2 outputs per thread per block.
__device__ void lower_product(const float *P, const float *T, float *PT, int tid) {
    const int gp = tid >> 6, ti = tid & 63, rr = (ti >> 3) * 2, cc = (ti & 7) * 2;
    // (I, J) pairs per group: {30, 00}, {20, 10}, {31, 21}, {32, 11, 22, 33}
    const uint32_t blocks = gp == 0 ? 0x0030u : gp == 1 ? 0x1020u : gp == 2 ? 0x2131u : 0x33221132u;
    const int nb = gp == 3 ? 4 : 2;
    for (int b = 0; b < nb; ++b) {
        const uint32_t code = (blocks >> (8 * b)) & 0xFFu;
        const int I = (int)(code >> 4), J = (int)(code & 15u);
        const int row = 16 * I + rr, col = 16 * J + cc;
        const float *p0 = P + row * SROW, *p1 = p0 + SROW;
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        // T rows m >= col (T lower), P columns m <= row + 1 (P lower)
        for (int m = col; m <= row + 1; ++m) {
            const float2 tv = *reinterpret_cast<const float2 *>(T + m * SROW + col);
            const float u0 = p0[m], u1 = p1[m];
            a00 = fmaf(u0, tv.x, a00);
            a01 = fmaf(u0, tv.y, a01);
            a10 = fmaf(u1, tv.x, a10);
            a11 = fmaf(u1, tv.y, a11);
        }
        *reinterpret_cast<float2 *>(PT + row * SROW + col) = make_float2(a00, a01);
        *reinterpret_cast<float2 *>(PT + (row + 1) * SROW + col) = make_float2(a10, a11);
    }
}

// Packs the lower triangle of a [64][SROW] matrix (rows in 8-float chunks up to
// the diagonal chunk) into `dst`.  Four threads per row, float4 stores.
__device__ __forceinline__ void store_packed(const float *M, float *dst, int tid) {
    const int t = tid >> 2, nch = (t >> 3) + 1;
    float *row = dst + fac::tri8_base(t);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int f = (tid & 3) + 4 * i;  // float4 index in the row: chunk f / 2, half f % 2
        if ((f >> 1) < nch)
            *reinterpret_cast<float4 *>(row + 4 * f) = *reinterpret_cast<const float4 *>(M + t * SROW + 4 * f);
    }
}

__global__ void __launch_bounds__(NT) factor_kernel(const __grid_constant__ CUtensorMap tmK,
                                                    const __grid_constant__ CUtensorMap tmQ, FacParams p) {
    const int64_t slot = blockIdx.x;
    const int hq = blockIdx.y;
    // the sequence whose chunk this slot holds: the last s with slot_base(s) <= slot
    int lo = 0, hi = p.n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (fac::slot_base(p.cu_seqlens[mid], mid) <= slot)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int64_t ts0 = p.cu_seqlens[lo], ts1 = p.cu_seqlens[lo + 1];
    const int64_t c = slot - fac::slot_base(ts0, lo);
    if (ts0 < 0 || ts1 < ts0 || ts1 > p.t_total) {
        if (threadIdx.x == 0) atomicCAS(p.err, 0, (int32_t)GDR_ERR_INVALID_ARG);
        return;
    }
    if (c < 0 || c * C >= ts1 - ts0) return;  // a slot between sequences: nothing to do
    const int64_t t0 = ts0 + c * C;
    const int L = (int)((ts1 - t0) < C ? (ts1 - t0) : C);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *sG = reinterpret_cast<float *>(sm + OFF_GATES), *sB = sG + 64, *sE = sG + 128;
    float *sScan = reinterpret_cast<float *>(sm + OFF_SCAN);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
    const uint32_t bar_tma = sb + OFF_BARS, bar_mma = sb + OFF_BARS + 8;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, 32768);
        tma_load_3d(sb + OFF_KQ, &tmK, bar_tma, 0, hq, (int)t0);
        tma_load_3d(sb + OFF_KQ + 16384, &tmK, bar_tma, 64, hq, (int)t0);
        tma_load_3d(sb + OFF_KQ + 8192, &tmQ, bar_tma, 0, hq, (int)t0);
        tma_load_3d(sb + OFF_KQ + 16384 + 8192, &tmQ, bar_tma, 64, hq, (int)t0);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    // Gram products [K Kᵀ; Q Kᵀ] into TMEM (lane = row, column = key token)
    bool ok = true;
    if (tid == 0) {
        ok = mbar_wait_bounded(bar_tma, 0, kWaitLimit);
        if (ok) {
            tc_fence_after_sync();
            const uint64_t a0 = smem_desc_sw128(sb + OFF_KQ, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t a = desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32);
                mma_bf16(tmem, a, a, IDESC_G1, ks > 0);
            }
            mma_commit(bar_mma);
        }
    }
    ok = ok && mbar_wait_bounded(bar_mma, 0, kWaitLimit);
    if (!ok) atomicCAS(p.err, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
    if (!__syncthreads_and(ok)) {
        // let the tile load land before this CTA's shared memory is released
        if (tid == 0) mbar_wait_bounded(bar_tma, 0, kWaitLimit / 8);
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, TM_COLS);
        return;
    }
    tc_fence_after_sync();

    float *N = reinterpret_cast<float *>(sm + OFF_N), *P = reinterpret_cast<float *>(sm + OFF_P);
    float *T = reinterpret_cast<float *>(sm + OFF_T), *X = reinterpret_cast<float *>(sm + OFF_X);
    const int grp = p.h_v / p.h_qk;
    for (int hh = 0; hh < grp; ++hh) {
        const int h = hq * grp + hh;
        // gates: G = running sum of g (kept as G log2(e) so each decay is one exp2)
        float gl = 0.f;
        if (tid < C) {
            float b = 0.f;
            if (tid < L) {
                const size_t i = (size_t)(t0 + tid) * p.h_v + h;
                gl = p.g[i] * kLog2e;
                b = p.beta[i];
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, gl, o);
                if (lane >= o) gl += u;
            }
            if (lane == 31) sScan[warp] = gl;
            sB[tid] = b;
        }
        __syncthreads();
        if (tid < C) {
            if (tid >= 32) gl += sScan[0];
            sG[tid] = gl;
            sE[tid] = fast_exp2(gl);
        }
        __syncthreads();
        // N (rows 0-63 of the Gram tile) and P (rows 64-127), masked in log space
        {
            const int q4 = warp & 3, half = warp >> 2;
            const int row = 32 * q4 + lane, t = row & 63;
            float a[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + 32 * half, a);
            const float Gt = sG[t];
            const bool is_n = row < 64;
            const float w = is_n ? sB[t] : 1.f;
            const int lim = is_n ? t : t + 1;  // keep j < t (N) or j <= t (P)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int jj = 32 * half + j;
                a[j] = (jj < lim) ? w * fast_exp2(Gt - sG[jj]) * a[j] : 0.f;
            }
            float *dst = (is_n ? N : P) + t * SROW + 32 * half;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(dst + j) = make_float4(a[j], a[j + 1], a[j + 2], a[j + 3]);
        }
        tc_fence_before_sync();
        __syncthreads();
        unit_lower_inverse(N, T, X, tid);  // ends with a barrier; N is free afterwards
        lower_product(P, T, N, tid);       // P T into N's space
        __syncthreads();
        float *slot_out = p.ws + ((size_t)slot * p.h_v + h) * fac::SLOT_FLOATS;
        store_packed(T, slot_out + fac::OFF_T, tid);
        store_packed(N, slot_out + fac::OFF_PT, tid);
        if (tid < 48) {
            const int a = tid >> 4, e = (tid & 15) * 4;  // G, beta, exp(G): 16 float4 each
            *reinterpret_cast<float4 *>(slot_out + fac::OFF_G + 64 * a + e) =
                *reinterpret_cast<const float4 *>(sG + 64 * a + e);
        }
        __syncthreads();  // scratch and gates are reused by the next V head
    }
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

cudaError_t launch_factors(const Args &a, float *ws, int32_t *err, cudaStream_t s) {
    CUtensorMap tmK, tmQ;
    if (!encode_bf16_3d(&tmK, a.k, 128, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_3d(&tmQ, a.q, 128, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(factor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    FacParams p;
    p.h_qk = a.h_qk;
    p.h_v = a.h_v;
    p.n_seqs = a.n_seqs;
    p.t_total = a.t_total;
    p.cu_seqlens = a.cu_seqlens;
    p.g = a.g;
    p.beta = a.beta;
    p.ws = ws;
    p.err = err;
    const int64_t slots = fac::n_slots(a.t_total, a.n_seqs);
    dim3 grid((unsigned)slots, (unsigned)a.h_qk);
    factor_kernel<<<grid, NT, SMEM_BYTES, s>>>(tmK, tmQ, p);
    return cudaGetLastError();
}

}  // namespace gdr
