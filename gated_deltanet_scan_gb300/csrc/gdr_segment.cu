// Two-level (segment-parallel) prefill: the chunks of each sequence are cut into
// P segments whose chunk scans run side by side instead of one after another.
//
// Over a segment the recurrence is affine in the state it starts from, X: after
// its tokens the state is Phi X + B, and each of its outputs is
// o_t = o0_t + X^T m_t.  This follows from the closed form of the state after a
// chunk on the Qwen3.5-9B NPU model card ("How it works": S_T = exp(G_T) S0 +
// K^T diag(exp(G_T - G)) D, with D affine in S0), applied chunk after chunk.
// (B, o0) is the segment's run from X = 0 with its values; (Phi, m) its run from
// X = I with every value zero (Phi is that run's final state, m its outputs).
// So one launch of the chunk scan walks segment 0 from the real state and, beside
// it, both runs of every later segment; then, per segment in order,
//     X_{p+1} = Phi_p X_p + B_p                      (combine_kernel)
// gives every segment's start, and a last pass forms the later segments'
// outputs o_t = o0_t + X_p^T m_t (fixup_kernel).  The final X is the state after
// the sequence.
//
// Scratch (inside the caller's workspace, after the factor slots):
//   Phi[P-1], B[P-1], X[P-1]  fp32 [n_seqs][h_v][d][d]   (X[j] = start of segment j+1)
//   XT[P-1]   per (sequence, V head) X[j]^T as bf16 hi and lo tensor-core operand
//             tiles (64 KB; see xt_offset)
//   O0, M     fp32 [t_total][h_v][d]     (rows of segments >= 1 only)
#include <cuda_bf16.h>

#include "gdr_factor_layout.h"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {
namespace {

constexpr int D = 128;
using namespace tc;

__device__ __forceinline__ uint64_t desc_add_bytes(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// A 128 x 128 bf16 tensor-core operand, K-major with 128-byte swizzled rows: two
// 16 KB halves (columns 0-63, 64-127), 16-byte chunk j of row r of a half at
// r * 128 + 16 (j ^ (r % 8)).  The fix-up's operands are pairs of such tiles
// (the bf16 hi and lo parts of an fp32 matrix): hi at 0, lo at 32 KB.
__host__ __device__ constexpr uint32_t kt_chunk_offset(int r, int j) {  // j: 16-byte chunk 0..15 of row r
    return (uint32_t)((j >> 3) * 16384 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}
constexpr uint32_t KT_BYTES = 32768, KT_PAIR = 2 * KT_BYTES;

// bf16 hi and lo words of (x0, x1): hi = the top 16 bits of each, lo = bf16(x - hi); x0 low.
__device__ __forceinline__ void hilo_word(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t a = __float_as_uint(x0), b = __float_as_uint(x1);
    hi = __byte_perm(a, b, 0x7632);
    __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(a & 0xFFFF0000u), x1 - __uint_as_float(b & 0xFFFF0000u));
    lo = *reinterpret_cast<uint32_t *>(&l);
}
// Eight consecutive fp32 values as one 16-byte chunk of the hi tile and one of the lo tile.
__device__ __forceinline__ void store_hilo_chunk(uint8_t *pair, uint32_t off, const float *x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) hilo_word(x[2 * i], x[2 * i + 1], h[i], l[i]);
    *reinterpret_cast<uint4 *>(pair + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(pair + KT_BYTES + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Phi = I and B = 0 for every (segment >= 1, sequence, V head): the start states
// of the transition and offset runs.
__global__ void segment_init_kernel(float4 *__restrict__ phi, float4 *__restrict__ b, size_t n_mats) {
    const size_t n4 = n_mats * (D * D / 4);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const int e = (int)(i % (D * D / 4)) * 4;  // first element of the quad in its matrix
        const int row = e / D, col = e % D;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row >= col && row < col + 4) (&v.x)[row - col] = 1.f;
        phi[i] = v;
        b[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned); all of a
// thread's copies are in flight until cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Every segment's start, for one (sequence, V head) and 4 state columns per
// block: X_{p+1} = Phi_p X_p + B_p for p = 1 .. P-1 in order.  The columns are
// independent (X_{p+1}'s columns depend only on the same columns of X_p), so each
// block walks all steps for its 16 columns with X in shared memory; Phi_{p+1}
// is copied in (asynchronously, rows padded to 132 floats) while step p
// computes.  X_1 is the state segment 0 left in `state`: it is saved to
// xseg[0]; X_p goes to xseg[p-1], and the last, X_P, back to `state`.
constexpr int CMB_COLS = 4, PHI_LD = D + 4;
constexpr int CMB_SMEM = (2 * D * PHI_LD + 2 * D * CMB_COLS) * (int)sizeof(float);
struct CombineParams {
    int P;
    size_t seg_stride;  // floats between one segment's matrices and the next's
    const float *phi, *b;
    float *state, *xseg;
    uint8_t *xt;        // XT[p-1]: X_p^T operand tiles for the fix-up, KT_PAIR bytes per matrix
};
__global__ void __launch_bounds__(256) combine_kernel(CombineParams c) {
    extern __shared__ __align__(16) float csm[];
    // two Phi buffers [D][PHI_LD], then two X buffers [D][CMB_COLS]
    auto ph = [&](int i) { return csm + i * D * PHI_LD; };
    auto xs = [&](int i) { return csm + 2 * D * PHI_LD + i * D * CMB_COLS; };
    const size_t mat = (size_t)blockIdx.x * D * D;
    const int c0 = blockIdx.y * CMB_COLS;
    const int tid = threadIdx.x;
    auto load_phi = [&](int p, float *dst) {  // Phi_p (p >= 1) into dst
        const float *src = c.phi + (size_t)(p - 1) * c.seg_stride + mat;
#pragma unroll 4
        for (int i = tid; i < D * D / 4; i += 256) {
            const int r = i / (D / 4), q4 = i % (D / 4);
            cp_async16(dst + r * PHI_LD + 4 * q4, src + (size_t)r * D + 4 * q4);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // X_1 (this block's columns of the state) and Phi_1
    for (int i = tid; i < D * CMB_COLS / 4; i += 256) {
        const int r = i / (CMB_COLS / 4), q4 = i % (CMB_COLS / 4);
        const float4 v = *reinterpret_cast<const float4 *>(c.state + mat + (size_t)r * D + c0 + 4 * q4);
        reinterpret_cast<float4 *>(xs(0))[i] = v;
        *reinterpret_cast<float4 *>(c.xseg + mat + (size_t)r * D + c0 + 4 * q4) = v;
    }
    load_phi(1, ph(0));
    // X_p^T as the fix-up's B operand: rows = this block's 4 columns of X_p, 128 k
    // each, hi and lo (thread t < 128: column c0 + t / 16, k = 8 (t % 16) .. + 7)
    auto write_tiles = [&](const float *xsm, int p) {
        if (tid >= CMB_COLS * 16) return;
        const int nl = tid >> 4, j = tid & 15;
        float x8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x8[i] = xsm[(8 * j + i) * CMB_COLS + nl];
        store_hilo_chunk(c.xt + ((size_t)(p - 1) * (c.seg_stride / (D * D)) + blockIdx.x) * KT_PAIR,
                         kt_chunk_offset(c0 + nl, j), x8);
    };
    const int r = tid >> 1, cc = (tid & 1) * 2;  // row r, 2 of the 4 columns
    for (int p = 1; p < c.P; ++p) {
        const int cur = (p - 1) & 1;
        if (p + 1 < c.P) {
            load_phi(p + 1, ph(cur ^ 1));
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // Phi_p has landed
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();  // Phi_p and X_p visible to every thread
        if (p == 1) write_tiles(xs(0), 1);
        const float *bb = c.b + (size_t)(p - 1) * c.seg_stride + mat + (size_t)r * D + c0 + cc;
        float acc[2];
        {
            const float2 v = *reinterpret_cast<const float2 *>(bb);
            acc[0] = v.x;
            acc[1] = v.y;
        }
        const float *pr = ph(cur) + r * PHI_LD;
        const float *xin = xs(cur);
#pragma unroll 4
        for (int k4 = 0; k4 < D / 4; ++k4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(pr + 4 * k4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float2 x0 = *reinterpret_cast<const float2 *>(xin + (4 * k4 + kk) * CMB_COLS + cc);
                acc[0] = fmaf(av[kk], x0.x, acc[0]);
                acc[1] = fmaf(av[kk], x0.y, acc[1]);
            }
        }
        // X_{p+1}: to shared memory for the next step, and to xseg[p] (or the state)
        float *xo = xs(cur ^ 1) + r * CMB_COLS + cc;
        *reinterpret_cast<float2 *>(xo) = make_float2(acc[0], acc[1]);
        float *g = (p == c.P - 1 ? c.state : c.xseg + (size_t)p * c.seg_stride) + mat + (size_t)r * D + c0 + cc;
        *reinterpret_cast<float2 *>(g) = make_float2(acc[0], acc[1]);
        __syncthreads();  // every thread is done with Phi_p and X_p before they are overwritten
        if (p + 1 < c.P) write_tiles(xs(cur ^ 1), p + 1);
    }
}

// o_t = o0_t + X_p^T m_t for the tokens of segments >= 1, on tcgen05: a CTA
// covers up to 128 tokens (two chunks) of one segment of one sequence and one V
// head, the 128 x 128 product of those tokens' maps M (rows) and X_p.  The
// combine kernel left X_p^T as bf16 hi and lo K-major tiles (bulk-copied in);
// the CTA splits its rows of M into hi and lo tiles itself; three products
// (hi hi + hi lo + lo hi, fp32 accumulation in TMEM: 2^-16 relative, as the
// chunk scan's state products), 8 k-steps of M = 128, N = 128 MMAs each; thread
// t then adds its TMEM row to o0 and stores o.
struct FixParams {
    int h_v, n_seqs, P, out_bf16;
    int cuts[9];    // chunk cuts: segment p is chunks [cuts[p], cuts[p+1])
    int tiles[9];   // first CTA (blockIdx.x) of segment p's 128-token tiles, p >= 1; tiles[P] = total
    const int32_t *cu_seqlens;
    const uint8_t *xt;  // XT[p-1], KT_PAIR bytes per (sequence, V head)
    const float *o0, *m;
    void *o;
    int32_t *err;
};

// Shared memory: the A and B tile pairs, an fp32 staging row per thread (its row
// of M, later of o0, brought in by cp.async with every copy in flight at once),
// then 2 mbarriers and the TMEM address.
constexpr int STAGE_LD = D + 4;  // staging row stride (floats): conflict-free 16-byte reads of a row per thread
constexpr uint32_t FIX_A = 0, FIX_B = KT_PAIR, FIX_STAGE = 2 * KT_PAIR, FIX_BARS = FIX_STAGE + 128 * STAGE_LD * 4;
constexpr int FIX_SMEM = (int)(FIX_BARS + 32 + 1024);
constexpr uint32_t IDESC_FIX = idesc_bf16_f32(128, 128, 0, 0);
constexpr long long kFixWait = 4000000000LL;  // SM clocks (about 2 s)

__global__ void __launch_bounds__(128, 1) fixup_kernel(FixParams p) {
    extern __shared__ uint8_t fsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(fsm_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t bar_x = sb + FIX_BARS, bar_mma = sb + FIX_BARS + 8;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + FIX_BARS + 16);
    const int bx = (int)blockIdx.x;
    int seg = 1;  // the segment of this CTA's tile (static indices: the tables stay in the parameter space)
#pragma unroll
    for (int q = 2; q < 9; ++q)
        if (q < p.P && bx >= p.tiles[q]) seg = q;
    int cseg_lo = 0, cseg_hi = 0, tile0 = 0;  // the segment's chunks [cseg_lo, cseg_hi), its first tile
#pragma unroll
    for (int q = 1; q < 9; ++q)
        if (q == seg) {
            cseg_lo = p.cuts[q];
            tile0 = p.tiles[q];
        }
#pragma unroll
    for (int q = 2; q < 9; ++q)
        if (q == seg + 1) cseg_hi = p.cuts[q];
    const int c0 = cseg_lo + 2 * (bx - tile0);  // first chunk of the tile
    const int s = (int)blockIdx.y / p.h_v, h = (int)blockIdx.y % p.h_v;
    const int64_t ts = p.cu_seqlens[s], te = p.cu_seqlens[s + 1];
    const int64_t t0 = ts + (int64_t)c0 * 64;
    int64_t tend = ts + (int64_t)cseg_hi * 64;
    if (tend > te) tend = te;
    if (t0 >= tend) return;  // past this sequence's end in this segment (or an empty sequence)
    const int ntok = (int)((tend - t0) < 128 ? (tend - t0) : 128);
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        mbar_init(bar_x, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        const uint8_t *src = p.xt + ((size_t)(seg - 1) * p.n_seqs * p.h_v + blockIdx.y) * KT_PAIR;
        mbar_arrive_expect_tx(bar_x, KT_PAIR);
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) bulk_load(sb + FIX_B + i * 16384u, src + i * 16384u, 16384u, bar_x);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), 128);
        tmem_relinquish();
    }
    // The tile's rows of M, staged by cp.async (warp w: rows 32 w .. + 31, one whole
    // 512-byte row per instruction), as hi and lo A tiles (rows past the tile's tokens:
    // zero); then its rows of o0 into the same staging rows.  Thread tid reads and
    // writes staging row tid only, which its own warp brought in.
    const int lane = tid & 31;
    float *stage_all = reinterpret_cast<float *>(sm + FIX_STAGE);
    float *stage = stage_all + tid * STAGE_LD;
    auto grow = [&](int r) { return ((size_t)(t0 + r) * p.h_v + h) * D; };
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
        const int r = 32 * warp + i;
        if (r < ntok) cp_async16(stage_all + r * STAGE_LD + 4 * lane, p.m + grow(r) + 4 * lane);
    }
    cp_async_wait_all();
    __syncwarp();
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        float x8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (tid < ntok) {
            const float4 a = *reinterpret_cast<const float4 *>(stage + 8 * j);
            const float4 b = *reinterpret_cast<const float4 *>(stage + 8 * j + 4);
            x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w;
            x8[4] = b.x; x8[5] = b.y; x8[6] = b.z; x8[7] = b.w;
        }
        store_hilo_chunk(sm + FIX_A, kt_chunk_offset(tid, j), x8);
    }
    __syncwarp();  // every lane is done with the rows of M before o0 replaces them
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {  // o0, read in the epilogue; lands while the MMAs run
        const int r = 32 * warp + i;
        if (r < ntok) cp_async16(stage_all + r * STAGE_LD + 4 * lane, p.o0 + grow(r) + 4 * lane);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    bool ok = true;
    if (tid == 0) {
        ok = mbar_wait_bounded(bar_x, 0, kFixWait);
        if (ok) {
            tc_fence_after_sync();
            const uint64_t ah = smem_desc_sw128(sb + FIX_A, 16, 1024), al = desc_add_bytes(ah, KT_BYTES);
            const uint64_t bh = smem_desc_sw128(sb + FIX_B, 16, 1024), bl = desc_add_bytes(bh, KT_BYTES);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32);
                mma_bf16(tmem, desc_add_bytes(ah, off), desc_add_bytes(bh, off), IDESC_FIX, ks > 0);
                mma_bf16(tmem, desc_add_bytes(ah, off), desc_add_bytes(bl, off), IDESC_FIX, 1);
                mma_bf16(tmem, desc_add_bytes(al, off), desc_add_bytes(bh, off), IDESC_FIX, 1);
            }
            mma_commit(bar_mma);
        } else {
            atomicCAS(p.err, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
        }
        *reinterpret_cast<volatile int *>(tmem_holder + 1) = ok ? 1 : 0;
    }
    __syncthreads();
    const bool issued = *reinterpret_cast<volatile int *>(tmem_holder + 1) != 0;
    bool done = issued && mbar_wait_bounded(bar_mma, 0, kFixWait);
    if (issued && !done) atomicCAS(p.err, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
    if (done) {
        tc_fence_after_sync();
        // thread t: TMEM lane t, the tile's token row t; o = o0 + M X written back into
        // the staging row, then the warp stores its rows whole (one row per instruction)
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();  // the warp's rows of o0 have landed
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            float acc[32];
            tmem_ld32(lane_addr + 32 * q, acc);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                float4 *b = reinterpret_cast<float4 *>(stage + 32 * q + e);
                const float4 v = *b;
                *b = make_float4(v.x + acc[e], v.y + acc[e + 1], v.z + acc[e + 2], v.w + acc[e + 3]);
            }
        }
        __syncwarp();
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * warp + i;
            if (r < ntok) {
                const float4 y = *reinterpret_cast<const float4 *>(stage_all + r * STAGE_LD + 4 * lane);
                if (p.out_bf16) {
                    __nv_bfloat162 v0 = __floats2bfloat162_rn(y.x, y.y), v1 = __floats2bfloat162_rn(y.z, y.w);
                    uint2 pk;
                    pk.x = *reinterpret_cast<uint32_t *>(&v0);
                    pk.y = *reinterpret_cast<uint32_t *>(&v1);
                    *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + grow(r) + 4 * lane) = pk;
                } else {
                    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + grow(r) + 4 * lane) = y;
                }
            }
        }
    } else if (tid == 0 && !issued) {
        mbar_wait_bounded(bar_x, 0, kFixWait / 8);  // let the tile copy land before the memory is released
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy of this thread still in flight
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 128);
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

SegLayout segment_layout(int64_t factor_bytes, int n_seqs, int h_v, int64_t t_total, int P) {
    SegLayout L;
    const size_t mats = (size_t)(P - 1) * n_seqs * h_v * D * D * sizeof(float);
    const size_t rows = (size_t)t_total * h_v * D * sizeof(float);
    L.phi = align256((size_t)factor_bytes);
    L.b = L.phi + align256(mats);
    L.x = L.b + align256(mats);
    L.xt = L.x + align256(mats);  // one KT_PAIR (64 KB, the size of an fp32 state) per matrix
    L.o0 = L.xt + align256(mats);
    L.m = L.o0 + align256(rows);
    L.total = L.m + align256(rows);
    return L;
}

int segment_cut(int64_t n_chunks, int P, int p) { return (int)((n_chunks * p) / P); }

cudaError_t launch_segmented(const Args &a, int P, uint8_t *ws, const SegLayout &L, int32_t *err, cudaStream_t s) {
    const int64_t n_ch = (a.t_total + 63) / 64;
    float *phi = reinterpret_cast<float *>(ws + L.phi);
    float *bb = reinterpret_cast<float *>(ws + L.b);
    float *xseg = reinterpret_cast<float *>(ws + L.x);
    float *o0 = reinterpret_cast<float *>(ws + L.o0);
    float *m = reinterpret_cast<float *>(ws + L.m);
    uint8_t *xt = ws + L.xt;
    const size_t per_seg = (size_t)a.n_seqs * a.h_v;  // matrices per segment
    const size_t mat_floats = (size_t)D * D;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (configured_device != dev) {
        e0 = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CMB_SMEM);
        if (e0 == cudaSuccess)
            e0 = cudaFuncSetAttribute(fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FIX_SMEM);
        if (e0 != cudaSuccess) return e0;
        configured_device = dev;
    }
    // 1. start states of the transition (I) and offset (0) runs
    {
        const size_t n4 = (size_t)(P - 1) * per_seg * (mat_floats / 4);
        unsigned blocks = (unsigned)((n4 + 255) / 256);
        if (blocks > 152u * 8u) blocks = 152u * 8u;
        segment_init_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<float4 *>(phi), reinterpret_cast<float4 *>(bb),
                                                     (size_t)(P - 1) * per_seg);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // 2. the factors of every chunk, 3. every segment's runs in one scan launch
    cudaError_t e = launch_factors(a, reinterpret_cast<float *>(ws), err, s, false);
    if (e != cudaSuccess) return e;
    TcRun runs[kMaxTcRuns];
    int n_runs = 0;
    runs[n_runs++] = TcRun{segment_cut(n_ch, P, 0), segment_cut(n_ch, P, 1), a.out_bf16, 0, a.state, a.o};
    for (int p = 1; p < P; ++p) {
        const int lo = segment_cut(n_ch, P, p), hi = segment_cut(n_ch, P, p + 1);
        runs[n_runs++] = TcRun{lo, hi, 0, 0, bb + (size_t)(p - 1) * per_seg * mat_floats, o0};
        runs[n_runs++] = TcRun{lo, hi, 0, 1, phi + (size_t)(p - 1) * per_seg * mat_floats, m};
    }
    e = launch_prefill_tc_runs(a, runs, n_runs, reinterpret_cast<float *>(ws), s, true);
    if (e != cudaSuccess) return e;
    // 4. every segment's start (X_1 is the state segment 0 left in `state`)
    {
        CombineParams cp;
        cp.P = P;
        cp.seg_stride = per_seg * mat_floats;
        cp.phi = phi;
        cp.b = bb;
        cp.state = a.state;
        cp.xseg = xseg;
        cp.xt = xt;
        combine_kernel<<<dim3((unsigned)per_seg, D / CMB_COLS), 256, CMB_SMEM, s>>>(cp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // 5. outputs of segments >= 1
    FixParams fp = {};
    fp.h_v = a.h_v;
    fp.n_seqs = a.n_seqs;
    fp.P = P;
    fp.out_bf16 = a.out_bf16;
    for (int p = 0; p <= P; ++p) fp.cuts[p] = segment_cut(n_ch, P, p);
    fp.cu_seqlens = a.cu_seqlens;
    fp.xt = xt;
    fp.o0 = o0;
    fp.m = m;
    fp.o = a.o;
    fp.err = err;
    int n_tiles = 0;  // 128-token tiles of segments >= 1, segment by segment
    for (int p = 1; p < P; ++p) {
        fp.tiles[p] = n_tiles;
        n_tiles += (fp.cuts[p + 1] - fp.cuts[p] + 1) / 2;
    }
    fp.tiles[P] = n_tiles;
    if (n_tiles <= 0) return cudaSuccess;
    fixup_kernel<<<dim3((unsigned)n_tiles, (unsigned)per_seg), 128, FIX_SMEM, s>>>(fp);
    return cudaGetLastError();
}

}  // namespace gdr
