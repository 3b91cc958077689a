// Chunked prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Shapes: d_k = d_v = 128, 64-token chunks, bf16 q/k/v, fp32 state, fp32 or
// bf16 output.  A cluster of four CTAs owns one (sequence, V head); CTA r of
// the cluster owns state columns [32 r, 32 r + 32) and walks the sequence's
// chunks in order, keeping its 128 x 32 block of the state on chip for the
// whole sequence (fp32 in registers, bf16 hi/lo copies in shared memory as
// MMA operands).
//
// Per chunk (the chunkwise-parallel form of the Qwen3.5-9B NPU model card,
// "How it works"; forward substitution for the unit triangular factor as in
// the Candle PR's chunked scan; log-space masking from its overflow fix):
//   G   = inclusive running sum of g over the chunk (padding rows: g = beta = 0)
//   G1  [K Kᵀ; Q Kᵀ] = [K; Q] Kᵀ                         (M=128 MMA, exact bf16)
//   N   = diag(beta) (K Kᵀ ⊙ exp(G_t - G_j))_{j<t},  P = (Q Kᵀ ⊙ exp(G_t - G_j))_{j<=t}
//         (the exponent is only formed on the kept triangle, so it is <= 0)
//   T   = (I + N)^-1   (16x16 forward substitution, then two block-doubling levels)
//   MPT PT = P T                                          (M=64 MMA, hi/lo)
//   MMA1 [K S; Q S] = [K; Q] S                            (S as bf16 hi + lo)
//   R   = diag(beta) (V - diag(e^G) K S)
//   MMA2 [D; P D] = [T; PT] R                             (hi/lo on both sides)
//   O   = scale (diag(e^G) Q S + P D)
//   MMA3 Y = Kᵀ D~,  D~ = diag(exp(G_C - G)) D            (D~ as hi + lo)
//   S  <- exp(G_C) S + Y
// which is D = (I + N)^-1 diag(beta)(V - diag(e^G) K S0), O = diag(e^G) Q S0 + P D,
// S_C = e^{G_C} S0 + Kᵀ diag(e^{G_C - G}) D written as products on the tensor
// cores.  The bf16 hi/lo split (x = hi + lo, both bf16) keeps every product
// that feeds the state within ~2^-16 relative; K, Q and V are exact in bf16.
//
// Warp roles (512 threads).  Warps 0-7, the "chain", run the state-dependent
// MMA1 -> MMA2 -> MMA3 sequence of chunk c; warp w owns TMEM lanes
// 32 (w % 4) .. + 31 and state columns 16 (w / 4) .. + 15 of the CTA's 32.
// Warps 8-15, "stage 1", prepare the state-independent factors.  The four
// CTAs of a cluster take turns: CTA r prepares chunks r, r+4, r+8, ... (gates,
// Gram MMA, N and P, triangular inverse, P T), stages [T; PT] and the gates
// in one of two buffers, and bulk-copies them into the three peers' shared
// memory, completing on each peer's mbarrier.  Chains signal a buffer free
// to the CTA that fills it next.  Every mbarrier wait is bounded: on timeout
// a thread records GDR_ERR_DEVICE_TIMEOUT in the device error word and its
// role stops; the peers time out on their own waits, and every CTA meets the
// final cluster barrier, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdr_common.cuh"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {

static __device__ int32_t g_device_error;

namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NCL = 4;         // CTAs per cluster (column blocks of one V head)
constexpr int BV = D / NCL;    // 32 state columns per CTA
constexpr int NCHAIN = 256;    // warps 0-7
constexpr int NS1 = 256;       // warps 8-15
constexpr int NTHREADS = NCHAIN + NS1;
constexpr int SROW = 68;  // fp32 scratch row stride in floats (bank-conflict-free float4 rows)
constexpr int XROW = 33;  // level-2 partial product row stride
constexpr uint32_t BAR_CHAIN = 1, BAR_S1 = 2;  // named barrier ids
constexpr int ROLE_CHAIN = 0, ROLE_S1 = 1;

// Shared memory map, bytes from a 1024-byte aligned base.
constexpr uint32_t KQ_BYTES = 32768;  // [kb=0: K rows 0-63, Q rows 64-127][kb=1: same], 128-B rows
constexpr uint32_t V_BYTES = 4096;    // V tile: 64 tokens x 32 columns, 64-B rows
constexpr uint32_t OFF_KQ = 0;        // two ring buffers
constexpr uint32_t OFF_V = 2 * KQ_BYTES;  // two ring buffers
constexpr uint32_t ATP_BYTES = 32768;     // [T; PT] hi (16 KB) + lo (16 KB), K-major 128 x 64 bf16
constexpr uint32_t OFF_ATP = OFF_V + 2 * V_BYTES;  // two buffers (chunk parity)
constexpr uint32_t OFF_S_HI = OFF_ATP + 2 * ATP_BYTES;  // state block, MN-major 128 (k) x 32 (n), 64-B rows
constexpr uint32_t OFF_S_LO = OFF_S_HI + 8192;
constexpr uint32_t OFF_RD_HI = OFF_S_LO + 8192;  // R, then D~: MN-major 64 (k = token) x 32 (n)
constexpr uint32_t OFF_RD_LO = OFF_RD_HI + 4096;
constexpr uint32_t OFF_P_HI = OFF_RD_LO + 4096;  // P as K-major 64 x 64 bf16 (A of the PT MMA)
constexpr uint32_t OFF_P_LO = OFF_P_HI + 8192;
constexpr uint32_t SCR_MAT = 64 * SROW * 4;      // fp32 [64][SROW]
// Stage 1's own K/Q tile for the Gram MMA; once that MMA has completed the
// region holds the fp32 scratch N, T and X.
constexpr uint32_t OFF_S1 = OFF_P_LO + 8192;
constexpr uint32_t OFF_N = OFF_S1;
constexpr uint32_t OFF_T = OFF_N + SCR_MAT;
constexpr uint32_t OFF_X = OFF_T + SCR_MAT;  // partial products: [32][XROW] fp32
constexpr uint32_t S1_BYTES = 40960;
constexpr uint32_t OFF_SMALL = OFF_S1 + S1_BYTES;
constexpr uint32_t SM_GATES = OFF_SMALL;         // float [2 buffers][3][64]: G log2(e), beta, e^G
constexpr uint32_t SM_SCAN = OFF_SMALL + 1536;   // float[4]
constexpr uint32_t SM_BARS = OFF_SMALL + 1600;   // 8 x uint64
constexpr uint32_t SM_TMEM = OFF_SMALL + 1664;   // uint32
constexpr uint32_t SM_ABORT = OFF_SMALL + 1672;  // int32[2], one per role
constexpr uint32_t SM_GPRIV = OFF_SMALL + 2048;  // float[3][64]: stage 1's own copy of the gates
constexpr uint32_t SMEM_USED = OFF_SMALL + 3072;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_X + 32 * XROW * 4 <= OFF_S1 + S1_BYTES && KQ_BYTES <= S1_BYTES, "stage-1 region");
static_assert(OFF_ATP % 1024 == 0 && OFF_S_HI % 1024 == 0 && OFF_RD_HI % 1024 == 0 && OFF_P_HI % 1024 == 0 &&
                  OFF_S1 % 1024 == 0 && OFF_V % 1024 == 0,
              "operand tiles must be 1 KB aligned");

// mbarriers
constexpr int B_TMA0 = 0, B_MMA_CHAIN = 2, B_MMA_S1 = 3, B_ATP_FULL0 = 4, B_ATP_FREE = 6, B_TMA_S1 = 7;
constexpr int NBARS = 8;

// TMEM columns (fp32 accumulators).
constexpr uint32_t TM_G1 = 0;    // [K Kᵀ; Q Kᵀ]   128 x 64 (stage 1, lane = row)
constexpr uint32_t TM_PT = 64;   // P T            64 x 64  (stage 1, M=64 layout)
constexpr uint32_t TM_KS = 128;  // [K S; Q S]     128 x 32 (chain)
constexpr uint32_t TM_DP = 160;  // [D; P D]       128 x 32 (chain)
constexpr uint32_t TM_Y = 192;   // Kᵀ D~          128 x 32 (chain)
constexpr uint32_t TM_COLS = 256;

constexpr uint32_t TMA_BYTES = 2 * 16384 + V_BYTES;      // K + Q (two 64-column halves each) + V
constexpr uint32_t GATE_BYTES = 192 * 4;
constexpr uint32_t ATP_COPY_BYTES = ATP_BYTES + GATE_BYTES;
constexpr long long kWaitLimit = 4000000000LL;  // SM clocks (about 2 s)
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t IDESC_G1 = idesc_bf16_f32(128, 64, 0, 0);  // A K-major, B K-major
constexpr uint32_t IDESC_PT = idesc_bf16_f32(64, 64, 0, 1);   // A K-major (P), B MN-major (T)
constexpr uint32_t IDESC_KS = idesc_bf16_f32(128, BV, 0, 1);  // A K-major, B MN-major
constexpr uint32_t IDESC_DP = idesc_bf16_f32(128, BV, 0, 1);
constexpr uint32_t IDESC_Y = idesc_bf16_f32(128, BV, 1, 1);   // A MN-major (Kᵀ), B MN-major

struct TcParams {
    int h_qk, h_v, out_bf16;
    float scale;
    const int32_t *cu_seqlens;
    const float *g, *beta;
    float *state;
    void *o;
};

struct Ctx {
    uint8_t *sm;
    uint32_t sbase;
    uint32_t tmem;
    volatile int *abort_flag;
    uint32_t rank;  // rank in the cluster = column block
    __device__ uint32_t bar(int i) const { return sbase + SM_BARS + 8 * i; }
    __device__ float *gates(int buf) const { return reinterpret_cast<float *>(sm + SM_GATES) + buf * 192; }
    __device__ uint32_t atp_hi(int buf) const { return OFF_ATP + buf * ATP_BYTES; }
    __device__ uint32_t atp_lo(int buf) const { return OFF_ATP + buf * ATP_BYTES + 16384; }
};

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

__device__ __forceinline__ void role_sync(int role) {
    if (role == ROLE_CHAIN)
        named_sync(BAR_CHAIN, NCHAIN);
    else
        named_sync(BAR_S1, NS1);
}

// Bounded wait shared by all threads of one role.  A thread whose wait times
// out records the error and raises its role's abort flag; the role barrier
// that follows makes every thread of the role read the same flag, so the role
// leaves its loop together and never strands a sibling at a later barrier.
// Each role reads only its own flag.
__device__ __forceinline__ bool role_wait(const Ctx &x, uint32_t bar, uint32_t parity, int role) {
    if (!mbar_wait_bounded(bar, parity, kWaitLimit)) {
        x.abort_flag[role] = 1;
        atomicCAS(&g_device_error, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
    }
    role_sync(role);
    return x.abort_flag[role] == 0;
}

__device__ __forceinline__ void issue_chunk_loads(const Ctx &x, int buf, int tok, int hq, int h,
                                                  const CUtensorMap *tmK, const CUtensorMap *tmQ,
                                                  const CUtensorMap *tmV) {
    const uint32_t bar = x.bar(B_TMA0 + buf);
    mbar_arrive_expect_tx(bar, TMA_BYTES);
    const uint32_t kq = x.sbase + OFF_KQ + buf * KQ_BYTES;
    tma_load_3d(kq, tmK, bar, 0, hq, tok);
    tma_load_3d(kq + 16384, tmK, bar, 64, hq, tok);
    tma_load_3d(kq + 8192, tmQ, bar, 0, hq, tok);
    tma_load_3d(kq + 16384 + 8192, tmQ, bar, 64, hq, tok);
    tma_load_3d(x.sbase + OFF_V + buf * V_BYTES, tmV, bar, (int)x.rank * BV, h, tok);
}

// Stage 1's copy of the chunk's K and Q (for the Gram MMA only).
__device__ __forceinline__ void issue_s1_loads(const Ctx &x, int tok, int hq, const CUtensorMap *tmK,
                                               const CUtensorMap *tmQ) {
    const uint32_t bar = x.bar(B_TMA_S1);
    mbar_arrive_expect_tx(bar, 2 * 16384);
    const uint32_t kq = x.sbase + OFF_S1;
    tma_load_3d(kq, tmK, bar, 0, hq, tok);
    tma_load_3d(kq + 16384, tmK, bar, 64, hq, tok);
    tma_load_3d(kq + 8192, tmQ, bar, 0, hq, tok);
    tma_load_3d(kq + 16384 + 8192, tmQ, bar, 64, hq, tok);
}

// 32 values as chunks [4 half, 4 half + 4) of row `row` of a 128-B hi/lo tile pair.
__device__ __forceinline__ void store_half_hilo(uint8_t *hi, uint8_t *lo, int row, int half, const float *x) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) store_hilo_chunk(hi, lo, row, 4 * half + ch, x + 8 * ch);
}
// 16 values as chunks [2 half, 2 half + 2) of row `row` of a 64-B hi/lo tile pair.
__device__ __forceinline__ void store_quarter_hilo64(uint8_t *hi, uint8_t *lo, int row, int half, const float *x) {
    store_hilo_chunk64(hi, lo, row, 2 * half, x);
    store_hilo_chunk64(hi, lo, row, 2 * half + 1, x + 8);
}

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
    return tmem + ((uint32_t)((warp & 3) * 32) << 16);
}

// ================================ stage 1 ===========================================
// T = (I + N)^-1 for strictly lower N (fp32 scratch, row stride SROW);
// s = stage-1 thread index (0..255).  Ends with a role barrier.
__device__ void unit_lower_inverse(uint8_t *sm, int s) {
    const float *N = reinterpret_cast<const float *>(sm + OFF_N);
    float *T = reinterpret_cast<float *>(sm + OFF_T);
    float *X = reinterpret_cast<float *>(sm + OFF_X);
    if (s < 64) {
        // 16 x 16 diagonal blocks by forward substitution, one column per thread
        const int base = (s >> 4) * 16, jj = s & 15;
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a0 = (r == jj) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                if (m < r && m >= jj) {
                    const float nv = N[(base + r) * SROW + base + m];
                    if (m & 1)
                        a1 = fmaf(-nv, col[m], a1);
                    else
                        a0 = fmaf(-nv, col[m], a0);
                }
            }
            col[r] = a0 + a1;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(base + r) * SROW + base + jj] = col[r];
    } else {
        // everything above the 16-block diagonal is zero
        for (int e = s - 64; e < 6 * 256; e += NS1 - 64) {
            const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            const int I = b < 3 ? 0 : (b < 5 ? 1 : 2);
            const int J = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
            T[(16 * I + r) * SROW + 16 * J + cc] = 0.f;
        }
    }
    named_sync(BAR_S1, NS1);
    // level 1: T_{I,I-1} = -T_II (N_{I,I-1} T_{I-1,I-1}) for I = 1, 3; two entries per thread
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int e = s + NS1 * k, blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
        const int I = 2 * blk + 1, J = I - 1;
        const float *nr = N + (16 * I + r) * SROW + 16 * J;
        const float *tc = T + (16 * J) * SROW + 16 * J + cc;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 2) {
            a0 = fmaf(nr[m], tc[m * SROW], a0);
            a1 = fmaf(nr[m + 1], tc[(m + 1) * SROW], a1);
        }
        X[(16 * blk + r) * XROW + cc] = a0 + a1;
    }
    named_sync(BAR_S1, NS1);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int e = s + NS1 * k, blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
        const int I = 2 * blk + 1;
        const float *tr = T + (16 * I + r) * SROW + 16 * I;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 2) {
            a0 = fmaf(tr[m], X[(16 * blk + m) * XROW + cc], a0);
            a1 = fmaf(tr[m + 1], X[(16 * blk + m + 1) * XROW + cc], a1);
        }
        T[(16 * I + r) * SROW + 16 * (I - 1) + cc] = -(a0 + a1);
    }
    named_sync(BAR_S1, NS1);
    // level 2: T[32:64, 0:32] = -T[32:64, 32:64] (N[32:64, 0:32] T[0:32, 0:32]);
    // each thread a 2 x 2 tile of the 32 x 32 block
    const int r0 = (s >> 4) * 2, c0 = (s & 15) * 2;
    {
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        const float *n0 = N + (32 + r0) * SROW, *n1 = n0 + SROW;
#pragma unroll 8
        for (int m = c0; m < 32; ++m) {  // T[0:32, 0:32] is lower: rows m >= c0 only
            const float2 tv = *reinterpret_cast<const float2 *>(T + m * SROW + c0);
            const float u0 = n0[m], u1 = n1[m];
            a00 = fmaf(u0, tv.x, a00);
            a01 = fmaf(u0, tv.y, a01);
            a10 = fmaf(u1, tv.x, a10);
            a11 = fmaf(u1, tv.y, a11);
        }
        X[r0 * XROW + c0] = a00;
        X[r0 * XROW + c0 + 1] = a01;
        X[(r0 + 1) * XROW + c0] = a10;
        X[(r0 + 1) * XROW + c0 + 1] = a11;
    }
    named_sync(BAR_S1, NS1);
    {
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        const float *t0 = T + (32 + r0) * SROW + 32, *t1 = t0 + SROW;
#pragma unroll 8
        for (int m = 0; m <= r0 + 1; ++m) {  // T[32:64, 32:64] is lower: columns m <= row
            const float x0 = X[m * XROW + c0], x1 = X[m * XROW + c0 + 1];
            const float u0 = t0[m], u1 = t1[m];
            a00 = fmaf(u0, x0, a00);
            a01 = fmaf(u0, x1, a01);
            a10 = fmaf(u1, x0, a10);
            a11 = fmaf(u1, x1, a11);
        }
        *reinterpret_cast<float2 *>(T + (32 + r0) * SROW + c0) = make_float2(-a00, -a01);
        *reinterpret_cast<float2 *>(T + (33 + r0) * SROW + c0) = make_float2(-a10, -a11);
    }
    named_sync(BAR_S1, NS1);
}

__device__ void stage1_role(const Ctx &x, const TcParams &p, int64_t t0, int64_t t1, int nchunks, int h, int hq,
                            const CUtensorMap *tmK, const CUtensorMap *tmQ, const int tid) {
    const int s = tid - NCHAIN;  // 0..255
    const int warp = tid >> 5, lane = tid & 31;
    const int half = (s >> 5) >> 2;  // column half of this warp's TMEM reads
    const uint32_t tmem = x.tmem;
    float *sScan = reinterpret_cast<float *>(x.sm + SM_SCAN);
    float *gp = reinterpret_cast<float *>(x.sm + SM_GPRIV);
    const int first = (int)x.rank;

    // gates of this role's next chunk, loaded one turn ahead (threads s < 64)
    float g_next = 0.f, b_next = 0.f;
    if (s < C && first < nchunks && t0 + (int64_t)first * C + s < t1) {
        g_next = p.g[(size_t)(t0 + (int64_t)first * C + s) * p.h_v + h];
        b_next = p.beta[(size_t)(t0 + (int64_t)first * C + s) * p.h_v + h];
    }
    if (s == 0 && first < nchunks) issue_s1_loads(x, (int)(t0 + (int64_t)first * C), hq, tmK, tmQ);
    int turn = 0;
    for (int c = first; c < nchunks; c += NCL, ++turn) {
        const int buf = c & 1;
        const int64_t c0 = t0 + (int64_t)c * C;
        float gt = g_next, bt = b_next;
        if (s < C) {
            g_next = b_next = 0.f;
            if (c0 + NCL * C + s < t1) {
                g_next = p.g[(size_t)(c0 + NCL * C + s) * p.h_v + h];
                b_next = p.beta[(size_t)(c0 + NCL * C + s) * p.h_v + h];
            }
        }
        // this turn's K and Q tile
        if (!role_wait(x, x.bar(B_TMA_S1), (uint32_t)turn & 1u, ROLE_S1)) break;

        // Gram products of the chunk: [K Kᵀ; Q Kᵀ] into TMEM
        if (s == 0) {
            tc_fence_after_sync();  // the previous turn's reads of these TMEM columns are done
            const uint64_t a0 = smem_desc_sw128(x.sbase + OFF_S1, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t a = desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32);
                mma_bf16(tmem + TM_G1, a, a, IDESC_G1, ks > 0);
            }
            mma_commit(x.bar(B_MMA_S1));
        }
        // gates: G = inclusive running sum of g, kept as G log2(e) so every decay is one
        // ex2 (padding rows: g = 0, beta = 0)
        gt *= kLog2e;
        if (s < C) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, gt, o);
                if (lane >= o) gt += u;
            }
            if (lane == 31) sScan[s >> 5] = gt;
            gp[64 + s] = bt;
        }
        named_sync(BAR_S1, NS1);
        if (s < C) {
            if (s >= 32) gt += sScan[0];
            gp[s] = gt;
            gp[128 + s] = fast_exp2(gt);
        }
        if (!role_wait(x, x.bar(B_MMA_S1), 0u, ROLE_S1)) break;  // also publishes the gates
        tc_fence_after_sync();
        {
            // row = lane quarter of this warp; columns [32 half, 32 half + 32)
            const int row = ((warp & 3) << 5) + lane;
            float a[32];
            tmem_ld32(lane_base(tmem, warp) + TM_G1 + 32 * half, a);
            const int t = row & 63;
            const float Gt = gp[t];
            const bool is_n = row < 64;
            const float w = is_n ? gp[64 + t] : 1.f;
            const int lim = is_n ? t : t + 1;  // keep j < t (N) or j <= t (P)
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 gj = *reinterpret_cast<const float4 *>(gp + 32 * half + j);
                const float gv[4] = {gj.x, gj.y, gj.z, gj.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int jj = 32 * half + j + e;
                    a[j + e] = (jj < lim) ? w * fast_exp2(Gt - gv[e]) * a[j + e] : 0.f;
                }
            }
            if (is_n) {
                float *dst = reinterpret_cast<float *>(x.sm + OFF_N) + t * SROW + 32 * half;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(a[j], a[j + 1], a[j + 2], a[j + 3]);
            } else {
                store_half_hilo(x.sm + OFF_P_HI, x.sm + OFF_P_LO, t, half, a);
            }
        }
        tc_fence_before_sync();
        named_sync(BAR_S1, NS1);
        unit_lower_inverse(x.sm, s);

        // this parity's [T; PT] buffers are free once every chain finished MMA2 of chunk c-2
        if (c >= 2 && !role_wait(x, x.bar(B_ATP_FREE), (uint32_t)((c - 2) >> 2) & 1u, ROLE_S1)) break;
        {
            // T rows as the top half of [T; PT] (also the B operand of the PT product), and the gates
            const int row = s >> 2, cp = s & 3;
            const float *src = reinterpret_cast<const float *>(x.sm + OFF_T) + row * SROW + 16 * cp;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const float4 u = *reinterpret_cast<const float4 *>(src + 8 * ch);
                const float4 v = *reinterpret_cast<const float4 *>(src + 8 * ch + 4);
                const float xv[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
                store_hilo_chunk(x.sm + x.atp_hi(buf), x.sm + x.atp_lo(buf), row, 2 * cp + ch, xv);
            }
            if (s < 192) x.gates(buf)[s] = gp[s];
        }
        fence_proxy_async_smem();
        named_sync(BAR_S1, NS1);
        // the scratch is spent: fetch the next turn's K and Q into it
        if (s == 0 && c + NCL < nchunks) issue_s1_loads(x, (int)(c0 + NCL * C), hq, tmK, tmQ);
        // PT = P T  (M = 64)
        if (s == 0) {
            tc_fence_after_sync();
            const uint64_t ah0 = smem_desc_sw128(x.sbase + OFF_P_HI, 16, 1024);
            const uint64_t al0 = smem_desc_sw128(x.sbase + OFF_P_LO, 16, 1024);
            const uint64_t bh0 = smem_desc_sw128(x.sbase + x.atp_hi(buf), 16, 1024);
            const uint64_t bl0 = smem_desc_sw128(x.sbase + x.atp_lo(buf), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ah = desc_add(ah0, ks * 32), al = desc_add(al0, ks * 32);
                const uint64_t bh = desc_add(bh0, ks * 2048), bl = desc_add(bl0, ks * 2048);
                mma_bf16(tmem + TM_PT, ah, bh, IDESC_PT, ks > 0);
                mma_bf16(tmem + TM_PT, al, bh, IDESC_PT, 1);
                mma_bf16(tmem + TM_PT, ah, bl, IDESC_PT, 1);
            }
            mma_commit(x.bar(B_MMA_S1));
        }
        if (!role_wait(x, x.bar(B_MMA_S1), 1u, ROLE_S1)) break;
        tc_fence_after_sync();
        {
            // M = 64 accumulator: row i sits in lane 32 (i / 16) + i % 16
            float a[32];
            tmem_ld32(lane_base(tmem, warp) + TM_PT + 32 * half, a);
            if (lane < 16)
                store_half_hilo(x.sm + x.atp_hi(buf), x.sm + x.atp_lo(buf), 64 + 16 * (warp & 3) + lane, half, a);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_sync(BAR_S1, NS1);
        if (s == 0) {
            // local chain: [T; PT] and gates are in place; each peer: one bulk copy of both
            mbar_arrive(x.bar(B_ATP_FULL0 + buf));
            const uint32_t goff = SM_GATES + (uint32_t)buf * GATE_BYTES;
#pragma unroll
            for (uint32_t d = 1; d < NCL; ++d) {
                const uint32_t peer = map_to_rank(x.sbase, (x.rank + d) % NCL);
                const uint32_t full = peer + SM_BARS + 8 * (B_ATP_FULL0 + buf);
                mbar_arrive_expect_tx_cluster(full, ATP_COPY_BYTES);
                bulk_copy_to_peer(peer + x.atp_hi(buf), x.sbase + x.atp_hi(buf), ATP_BYTES, full);
                bulk_copy_to_peer(peer + goff, x.sbase + goff, GATE_BYTES, full);
            }
        }
    }
}

// ================================= chain ============================================
__device__ void chain_role(const Ctx &x, const TcParams &p, int64_t t0, int64_t t1, int nchunks, int h, int hq,
                           float *Sr, const CUtensorMap *tmK, const CUtensorMap *tmQ, const CUtensorMap *tmV,
                           const int tid, bool &ok) {
    const int warp = tid >> 5, lane = tid & 31;
    const int hc = warp >> 2;                    // column half: columns [16 hc, 16 hc + 16) of the CTA's 32
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane = state row (d_k index) / chunk row
    const int t = row & 63;
    const uint32_t lb = lane_base(x.tmem, warp);
    const uint32_t tmem = x.tmem;
    const int cb = (int)x.rank;
    // descriptor bases (start addresses advance per MMA)
    const uint64_t dS_hi = smem_desc(x.sbase + OFF_S_HI, 8192, 512, kSwizzle64);
    const uint64_t dS_lo = smem_desc(x.sbase + OFF_S_LO, 8192, 512, kSwizzle64);
    const uint64_t dRD_hi = smem_desc(x.sbase + OFF_RD_HI, 4096, 512, kSwizzle64);
    const uint64_t dRD_lo = smem_desc(x.sbase + OFF_RD_LO, 4096, 512, kSwizzle64);
    uint32_t mma_phase = 0;
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        const int64_t c0 = t0 + (int64_t)c * C;
        const int L = (int)((t1 - c0) < C ? (t1 - c0) : C);
        const uint32_t kq = x.sbase + OFF_KQ + buf * KQ_BYTES;
        if (!role_wait(x, x.bar(B_TMA0 + buf), (uint32_t)(c >> 1) & 1u, ROLE_CHAIN)) break;

        // ---- MMA1: [K S; Q S] = [K; Q] (S_hi + S_lo) --------------------------------
        if (tid == 0) {
            tc_fence_after_sync();
            const uint64_t a0 = smem_desc_sw128(kq, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t a = desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32);
                mma_bf16(tmem + TM_KS, a, desc_add(dS_hi, ks * 1024), IDESC_KS, ks > 0);
                mma_bf16(tmem + TM_KS, a, desc_add(dS_lo, ks * 1024), IDESC_KS, 1);
            }
            mma_commit(x.bar(B_MMA_CHAIN));
        }
        // stage 1 of this chunk: gates and [T; PT]
        if (!role_wait(x, x.bar(B_ATP_FULL0 + buf), (uint32_t)(c >> 1) & 1u, ROLE_CHAIN)) break;
        const float *gts = x.gates(buf);
        const float Gt = gts[t], bt = gts[64 + t], egt = gts[128 + t];
        const float eGC = gts[128 + C - 1], GC = gts[C - 1];
        if (!role_wait(x, x.bar(B_MMA_CHAIN), mma_phase, ROLE_CHAIN)) break;
        mma_phase ^= 1;
        tc_fence_after_sync();
        float qse[16];  // rows 64-127: e^G Q S for this thread's columns, kept for the output
        {
            float a[16];
            tmem_ld16(lb + TM_KS + 16 * hc, a);
            if (row < 64) {
                // R = beta (V - e^G K S), staged as the hi/lo MN-major B operand of MMA2
                const uint8_t *vt = x.sm + OFF_V + buf * V_BYTES;
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    float v[8], r[8];
                    load_bf16_chunk64(vt, t, 2 * hc + ch, v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = bt * (v[e] - egt * a[ch * 8 + e]);
                    store_hilo_chunk64(x.sm + OFF_RD_HI, x.sm + OFF_RD_LO, t, 2 * hc + ch, r);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) qse[j] = egt * a[j];
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_sync(BAR_CHAIN, NCHAIN);

        // ---- MMA2: [D; P D] = [T; PT] R ---------------------------------------------
        if (tid == 0) {
            tc_fence_after_sync();
            const uint64_t ah0 = smem_desc_sw128(x.sbase + x.atp_hi(buf), 16, 1024);
            const uint64_t al0 = smem_desc_sw128(x.sbase + x.atp_lo(buf), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ah = desc_add(ah0, ks * 32), al = desc_add(al0, ks * 32);
                const uint64_t bh = desc_add(dRD_hi, ks * 1024), bl = desc_add(dRD_lo, ks * 1024);
                mma_bf16(tmem + TM_DP, ah, bh, IDESC_DP, ks > 0);
                mma_bf16(tmem + TM_DP, al, bh, IDESC_DP, 1);
                mma_bf16(tmem + TM_DP, ah, bl, IDESC_DP, 1);
            }
            mma_commit(x.bar(B_MMA_CHAIN));
        }
        if (!role_wait(x, x.bar(B_MMA_CHAIN), mma_phase, ROLE_CHAIN)) break;
        mma_phase ^= 1;
        tc_fence_after_sync();
        if (tid == 0) {
            // this parity's [T; PT] may be overwritten: tell the CTA that fills it next (chunk c+2)
            mbar_arrive_cluster(map_to_rank(x.bar(B_ATP_FREE), (uint32_t)(c + 2) % NCL));
        }
        {
            float dd[16];
            tmem_ld16(lb + TM_DP + 16 * hc, dd);
            if (row < 64) {
                // D~ = exp(G_C - G_t) D, staged as the hi/lo MN-major B operand of MMA3
                const float sc = fast_exp2(GC - Gt);
#pragma unroll
                for (int j = 0; j < 16; ++j) dd[j] *= sc;
                store_quarter_hilo64(x.sm + OFF_RD_HI, x.sm + OFF_RD_LO, t, hc, dd);
            } else if (t < L) {
                // O = scale (e^G Q S + P D) for the chunk's real rows
                const size_t off = ((size_t)(c0 + t) * p.h_v + h) * D + cb * BV + 16 * hc;
                if (p.out_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + off);
#pragma unroll
                    for (int j = 0; j < 16; j += 8) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = p.scale * (qse[j + e] + dd[j + e]);
                        dst[j / 8] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + off);
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        dst[j / 4] = make_float4(p.scale * (qse[j] + dd[j]), p.scale * (qse[j + 1] + dd[j + 1]),
                                                 p.scale * (qse[j + 2] + dd[j + 2]),
                                                 p.scale * (qse[j + 3] + dd[j + 3]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_sync(BAR_CHAIN, NCHAIN);

        // ---- MMA3: Y = Kᵀ (D~_hi + D~_lo) ---------------------------------------------
        if (tid == 0) {
            tc_fence_after_sync();
            const uint64_t a0 = smem_desc_sw128(kq, 16384, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = desc_add(a0, ks * 2048);
                mma_bf16(tmem + TM_Y, a, desc_add(dRD_hi, ks * 1024), IDESC_Y, ks > 0);
                mma_bf16(tmem + TM_Y, a, desc_add(dRD_lo, ks * 1024), IDESC_Y, 1);
            }
            mma_commit(x.bar(B_MMA_CHAIN));
        }
        if (!role_wait(x, x.bar(B_MMA_CHAIN), mma_phase, ROLE_CHAIN)) break;
        mma_phase ^= 1;
        tc_fence_after_sync();
        // chunk c's tiles are no longer read: fetch chunk c+2 into them
        if (tid == 0 && c + 2 < nchunks) {
            fence_proxy_async_smem();
            issue_chunk_loads(x, buf, (int)(c0 + 2 * C), hq, h, tmK, tmQ, tmV);
        }
        {
            float y[16];
            tmem_ld16(lb + TM_Y + 16 * hc, y);
#pragma unroll
            for (int j = 0; j < 16; ++j) Sr[j] = fmaf(eGC, Sr[j], y[j]);
            store_quarter_hilo64(x.sm + OFF_S_HI, x.sm + OFF_S_LO, row, hc, Sr);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_sync(BAR_CHAIN, NCHAIN);
    }
    ok = (x.abort_flag[ROLE_CHAIN] == 0);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmV, TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    Ctx x;
    x.sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    x.sbase = smem_u32(x.sm);
    x.abort_flag = reinterpret_cast<volatile int *>(x.sm + SM_ABORT);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(x.sm + SM_TMEM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    x.rank = cluster_rank();
    const int h = (blockIdx.x / NCL) % p.h_v;
    const int s = (blockIdx.x / NCL) / p.h_v;
    const int hq = h / (p.h_v / p.h_qk);
    const int64_t t0 = p.cu_seqlens[s], t1 = p.cu_seqlens[s + 1];
    const int nchunks = (int)((t1 - t0 + C - 1) / C);

    if (tid == 0) {
        for (int i = 0; i < NBARS; ++i) mbar_init(x.bar(i), i == B_ATP_FREE ? NCL : 1);
        x.abort_flag[0] = 0;
        x.abort_flag[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    // chain thread: row `srow` (a d_k index), columns [16 hc, 16 hc + 16) of the CTA's block
    const int srow = ((warp & 3) << 5) + lane, hc = (warp >> 2) & 1;
    float Sr[16];
    float *Sg = p.state + (((size_t)s * p.h_v + h) * D + srow) * D + x.rank * BV + 16 * hc;
    if (tid < NCHAIN) {
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(Sg + j);
            Sr[j] = v.x;
            Sr[j + 1] = v.y;
            Sr[j + 2] = v.z;
            Sr[j + 3] = v.w;
        }
        store_quarter_hilo64(x.sm + OFF_S_HI, x.sm + OFF_S_LO, srow, hc, Sr);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    cluster_sync();  // every CTA's barriers are initialised before any remote arrive
    tc_fence_after_sync();
    x.tmem = *tmem_holder;

    if (tid == 0) {
        if (nchunks > 0) issue_chunk_loads(x, 0, (int)t0, hq, h, &tmK, &tmQ, &tmV);
        if (nchunks > 1) issue_chunk_loads(x, 1, (int)(t0 + C), hq, h, &tmK, &tmQ, &tmV);
    }

    bool ok = true;
    if (tid < NCHAIN)
        chain_role(x, p, t0, t1, nchunks, h, hq, Sr, &tmK, &tmQ, &tmV, tid, ok);
    else
        stage1_role(x, p, t0, t1, nchunks, h, hq, &tmK, &tmQ, tid);

    if (tid < NCHAIN) {
        if (ok) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(Sg + j) = make_float4(Sr[j], Sr[j + 1], Sr[j + 2], Sr[j + 3]);
        } else if (tid == 0) {
            // let any outstanding tile load land before the CTA's shared memory is released
            for (int b = 0; b < 2; ++b) {
                mbar_wait_bounded(x.bar(B_TMA0 + b), 0, kWaitLimit / 8);
                mbar_wait_bounded(x.bar(B_TMA0 + b), 1, kWaitLimit / 8);
            }
        }
    }
    tc_fence_before_sync();
    cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(x.tmem, TM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// bf16 tensor [d2][d1][d0] (d0 contiguous), box {box0, 1, 64}.
bool encode_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                    CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {box0, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_tc(const Args &a, cudaStream_t s) {
    if (a.n_seqs == 0 || a.t_total == 0) return cudaSuccess;  // every sequence empty: state unchanged
    CUtensorMap tmK, tmQ, tmV;
    if (!encode_bf16_3d(&tmK, a.k, D, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_3d(&tmQ, a.q, D, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_3d(&tmV, a.v, D, (uint64_t)a.h_v, (uint64_t)a.t_total, BV, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    TcParams p;
    p.h_qk = a.h_qk;
    p.h_v = a.h_v;
    p.out_bf16 = a.out_bf16;
    p.scale = a.scale;
    p.cu_seqlens = a.cu_seqlens;
    p.g = a.g;
    p.beta = a.beta;
    p.state = a.state;
    p.o = a.o;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.n_seqs * (unsigned)a.h_v * (unsigned)NCL);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NCL;  // the four column blocks of one V head
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel, tmK, tmQ, tmV, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t read_clear_device_error(cudaStream_t s, int32_t *code) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    int32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    *code = v;
    return e;
}

}  // namespace gdr
