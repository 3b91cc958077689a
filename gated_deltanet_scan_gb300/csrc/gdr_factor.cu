// State-independent factors of the chunked prefill, computed for every chunk at
// once (no chunk depends on another).  One CTA per (chunk, V head) writes the
// chunk's gates, T = (I + N)^-1 and P T into the factor workspace (layout in
// gdr_factor_layout.h).
//
// What is stored is ready for the chunk scan's products: Tw = diag(exp(G_C - G)) T
// diag(beta) and PTw = P T diag(beta) (G_C = G of the chunk's last row), so
// that Tw (V - diag(e^G) K S) is the decay-weighted correction D~ the state
// update needs and PTw (V - diag(e^G) K S) the intra-chunk part of the output.
//
// For the chunk scan's lookahead it also writes, per (chunk c >= 1, QK head), the
// state-independent product X = [K; Q]_c K_{c-1}ᵀ as an fp16 operand tile
// (layout in gdr_factor_layout.h): the CTA of the first V head of the QK head's
// group computes it with the Gram and writes it at the end, staged in the then
// free scratch and stored by one bulk copy.
//
// Per chunk (the chunkwise-parallel form of the Qwen3.5-9B NPU model card,
// "How it works"; forward substitution for the unit triangular factor as in
// the Candle PR's "Chunked GatedDeltaNet Scan"; log-space masking from its
// "Float32 overflow fix"):
//   G   = inclusive running sum of g over the chunk (padding rows: g = beta = 0)
//   [K Kᵀ; Q Kᵀ] = [K; Q] Kᵀ      one M=128 tcgen05 MMA group, exact bf16 products,
//                                 fp32 accumulation in TMEM
//   N   = diag(beta) (K Kᵀ ⊙ exp(G_t - G_j))_{j<t}
//   P   =            (Q Kᵀ ⊙ exp(G_t - G_j))_{j<=t}
//         (the exponent is formed only on the kept triangle, so it never overflows)
//   T   = (I + N)^-1  blockwise forward substitution on 16 x 16 blocks:
//         T_II = (I + N_II)^-1                    (CUDA cores, column by column)
//         T_IJ = -T_II sum_{K=J}^{I-1} N_IK T_KJ  (I > J, by block diagonals)
//   P T   (P T)_IJ = sum_{K=J}^{I} P_IK T_KJ
// The block products run on warp-level bf16 tensor-core MMAs (m16n8k16) with
// each fp32 operand split into bf16 hi + lo (x = hi + lo to ~2^-16) and three
// products hi*hi + hi*lo + lo*hi accumulated in fp32.  Two warps solve for T,
// all four form P T.  Off-diagonal blocks of T are formed transposed, T_IJᵀ = -X_IJᵀ T_IIᵀ,
// so that X_IJᵀ comes straight out of one MMA's accumulators as the left
// operand of the next.
// Tw, PTw and X leave the kernel as fp16 MMA operand tiles (round to nearest,
// 2^-11 relative): the chunk scan multiplies them by fp16 R and D~ in one
// tensor-core pass each.
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
constexpr int NT = 128;  // four warps: one TMEM lane quadrant each

// A 16 x 16 block in shared memory as 16 rows of 8 pairs; pair p of row r holds
// hi(x[r][2p]), hi(x[r][2p+1]) in one word and the matching lo parts in the
// next.  Rows are 96 bytes apart, which keeps the 8-byte fragment loads of a
// warp free of bank conflicts.
constexpr int ROW_B = 96;
constexpr int BLK_B = 16 * ROW_B;  // 1536
__host__ __device__ constexpr int bi(int I, int J) { return I * (I + 1) / 2 + J; }  // lower block index, I >= J

// Scratch (bytes).  NB: the off-diagonal blocks of N (slots bi(I, J) - I, the
// diagonal slots left out); ND: the four diagonal blocks of N in fp32; PB: the
// ten lower blocks of P; TT: the blocks of Tᵀ on and above the diagonal, block
// (J, K) in slot bi(K, J); TD: the four diagonal blocks of T, row-major (for
// T_IIᵀ as a right operand).
__host__ __device__ constexpr int nbi(int I, int J) { return bi(I, J) - I; }  // I > J
constexpr int OFF_NB = 0;
constexpr int OFF_ND = OFF_NB + 6 * BLK_B;
constexpr int OFF_PB = OFF_ND + 4 * 1024;
constexpr int OFF_TT = OFF_PB + 10 * BLK_B;
constexpr int OFF_TD = OFF_TT + 10 * BLK_B;
constexpr int HEAD_B = OFF_TD + 4 * BLK_B;  // 50176

// Shared memory, bytes from a 1024-byte aligned base.  The K/Q tile and the
// previous chunk's K tile are only read by the Gram and X MMAs; once those have
// completed, the scratch overwrites them.
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_KP = 32768;  // K of the previous chunk: two 8 KB d_k halves
// G log2(e), beta, exp(G), exp(G_C - G): 4 x 64 fp32; with the fused L2 norm also
// 1 / |k| and 1 / |q| (2 x 64 more)
constexpr uint32_t OFF_GATES = HEAD_B;
__host__ __device__ constexpr uint32_t gates_bytes(bool qkn) { return qkn ? 1536u : 1024u; }
__host__ __device__ constexpr uint32_t off_bars(bool qkn) { return OFF_GATES + gates_bytes(qkn); }  // 2 mbarriers
__host__ __device__ constexpr uint32_t off_tmem(bool qkn) { return off_bars(qkn) + 16; }
__host__ __device__ constexpr uint32_t smem_bytes(bool qkn) { return off_tmem(qkn) + 16 + 1024; }
static_assert(OFF_KP + 16384 <= HEAD_B, "K/Q and previous K tiles fit under the scratch");
static_assert(OFF_GATES % 16 == 0 && off_bars(false) % 8 == 0 && off_bars(true) % 8 == 0 && HEAD_B % 16 == 0,
              "alignment");

constexpr uint32_t TM_COLS = 128;  // the 128 x 64 fp32 Gram tile, then X
constexpr uint32_t IDESC_G1 = idesc_bf16_f32(128, 64, 0, 0);
constexpr long long kWaitLimit = 4000000000LL;
constexpr float kLog2e = 1.4426950408889634f;

struct FacParams {
    int h_qk, h_v, n_seqs;
    int c_lo, c_hi;    // chunks of each sequence to process
    int64_t slot_lo;   // first slot of the launch (blockIdx.x = 0)
    int64_t t_total;
    const int32_t *cu_seqlens;
    const float *g, *beta;
    uint8_t *ws;  // factor slots
    uint8_t *xs;  // X tiles (fac::x_region_offset bytes into the workspace)
    int32_t *err;
};

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// (hi, lo) words of the pair (x0, x1): hi = top 16 bits of each, lo = bf16(x - hi).
__device__ __forceinline__ uint2 hl_pair(float x0, float x1) {
    const uint32_t a = __float_as_uint(x0), b = __float_as_uint(x1);
    const uint32_t h = __byte_perm(a, b, 0x7632);
    const uint32_t l = pack_bf16x2(x0 - __uint_as_float(a & 0xFFFF0000u), x1 - __uint_as_float(b & 0xFFFF0000u));
    return make_uint2(h, l);
}
__device__ __forceinline__ uint2 ld_pair(const uint8_t *blk, int r, int p) {
    return *reinterpret_cast<const uint2 *>(blk + r * ROW_B + p * 8);
}
__device__ __forceinline__ void st_pair(uint8_t *blk, int r, int p, uint2 v) {
    *reinterpret_cast<uint2 *>(blk + r * ROW_B + p * 8) = v;
}
// Elements (r, j), (r, j + 1) (j even) of the slot's fp16 operand tile.
__device__ __forceinline__ void st_tile_pair(uint8_t *slot, int r, int j, float x0, float x1) {
    *reinterpret_cast<uint32_t *>(slot + fac::OFF_T + fac::sw128_elem(r, j)) = pack_f16x2(x0, x1);
}

// Fragments of mma.m16n8k16 (row.col, bf16): lane = 4 g + c.
struct FragA {
    uint32_t hi[4], lo[4];
};
// A = X (16 x 16) from a block of row-major X.
__device__ __forceinline__ FragA ld_a(const uint8_t *blk, int g, int c) {
    const uint2 v0 = ld_pair(blk, g, c), v1 = ld_pair(blk, g + 8, c), v2 = ld_pair(blk, g, c + 4),
                v3 = ld_pair(blk, g + 8, c + 4);
    FragA f;
    f.hi[0] = v0.x;
    f.hi[1] = v1.x;
    f.hi[2] = v2.x;
    f.hi[3] = v3.x;
    f.lo[0] = v0.y;
    f.lo[1] = v1.y;
    f.lo[2] = v2.y;
    f.lo[3] = v3.y;
    return f;
}
// A from the two n8 accumulator halves of a previous product (scaled by `sign`).
__device__ __forceinline__ FragA a_from_acc(const float *d0, const float *d1, float sign) {
    const uint2 v0 = hl_pair(sign * d0[0], sign * d0[1]), v1 = hl_pair(sign * d0[2], sign * d0[3]);
    const uint2 v2 = hl_pair(sign * d1[0], sign * d1[1]), v3 = hl_pair(sign * d1[2], sign * d1[3]);
    FragA f;
    f.hi[0] = v0.x;
    f.hi[1] = v1.x;
    f.hi[2] = v2.x;
    f.hi[3] = v3.x;
    f.lo[0] = v0.y;
    f.lo[1] = v1.y;
    f.lo[2] = v2.y;
    f.lo[3] = v3.y;
    return f;
}

__device__ __forceinline__ void mma16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d[h] += A * B for both n8 halves h, where B = Yᵀ and Y is a row-major block:
// three bf16 products per half (hi hi + hi lo + lo hi).
__device__ __forceinline__ void mma_acc(float (*d)[4], const FragA &a, const uint8_t *yblk, int g, int c) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint2 b0 = ld_pair(yblk, 8 * h + g, c), b1 = ld_pair(yblk, 8 * h + g, c + 4);
        mma16816(d[h], a.hi, b0.x, b1.x);
        mma16816(d[h], a.hi, b0.y, b1.y);
        mma16816(d[h], a.lo, b0.x, b1.x);
    }
}
__device__ __forceinline__ void zero_acc(float (*d)[4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[h][i] = 0.f;
}

// Gates of V head h for the chunk's 64 rows, by one warp (lane owns rows lane
// and lane + 32): G = running sum of g in log2 units, beta, exp(G).  The raw
// g and beta are loaded first (as early as possible), the scan done later.
__device__ __forceinline__ void chunk_gates(float g0, float g1, float b0, float b1, float *gates, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, g0, o), u1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) {
            g0 += u0;
            g1 += u1;
        }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    gates[lane] = g0;
    gates[lane + 32] = g1;
    gates[64 + lane] = b0;
    gates[64 + lane + 32] = b1;
    gates[128 + lane] = fast_exp2(g0);
    gates[128 + lane + 32] = fast_exp2(g1);
    const float gc = __shfl_sync(0xffffffffu, g1, 31);  // G of the chunk's last row
    gates[192 + lane] = fast_exp2(gc - g0);
    gates[192 + lane + 32] = fast_exp2(gc - g1);
}

// The head's T from its N blocks, by the CTA's four warps wi (named barrier
// `bar`): warps 0-1 invert the diagonal blocks, then each block diagonal's
// blocks go one per warp (3, 2, 1).  Every block of Tw is stored to the slot's
// operand tiles (rows 0-63) as soon as it is formed, adjacent columns paired
// across lanes.
__device__ __forceinline__ void solve_t(uint8_t *hs, const float *gates, uint8_t *slot, int wi, int lane, uint32_t bar) {
    const int g = lane >> 2, c = lane & 3;
    const float *bw = gates + 64, *rw = gates + 192;  // column weights beta, row weights exp(G_C - G)
    // ---- diagonal blocks: warps 0-1 two each, lanes 0-15 / 16-31 one block, lane = column
    if (wi < 2) {
        const int I = 2 * wi + (lane >> 4), jj = lane & 15;
        const float *nd = reinterpret_cast<const float *>(hs + OFF_ND) + 256 * I;
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) col[r] = (r == jj) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 15; ++m) {
#pragma unroll
            for (int r = m + 1; r < 16; ++r) col[r] = fmaf(-nd[16 * r + m], col[m], col[r]);
        }
        // Tᵀ_II row jj is column jj of T_II
        uint8_t *tt = hs + OFF_TT + BLK_B * bi(I, I);
#pragma unroll
        for (int q = 0; q < 8; ++q) st_pair(tt, jj, q, hl_pair(col[2 * q], col[2 * q + 1]));
        // T_II row-major: lanes jj (even) and jj + 1 form the pairs of every row
        uint8_t *td = hs + OFF_TD + BLK_B * I;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float nb = __shfl_down_sync(0xffffffffu, col[r], 1);
            if ((jj & 1) == 0) st_pair(td, r, jj >> 1, hl_pair(col[r], nb));
        }
        // Tw: row 16 I + r, columns 16 I + jj, + 1 (jj even; 8-column chunks up to
        // the diagonal one, the rest of the row is zero-filled separately)
        const float bj = bw[16 * I + jj];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int rg = 16 * I + r, cg = 16 * I + jj;
            const float v = col[r] * bj * rw[rg];
            const float vn = __shfl_down_sync(0xffffffffu, v, 1);
            if ((jj & 1) == 0 && (cg >> 3) <= (rg >> 3)) st_tile_pair(slot, rg, cg, v, vn);
        }
    }
    named_sync(bar, NT);
    // ---- off-diagonal blocks by diagonals d = 1 (3 blocks), 2 (2), 3 (1), one per warp:
    // X_IJᵀ = sum_K Tᵀ(J, K) N_IKᵀ, then T_IJᵀ = -X_IJᵀ T_IIᵀ
    for (int d = 1; d <= 3; ++d) {
        if (wi + d <= 3) {
            const int J = wi;
            const int I = J + d;
            float x[2][4];
            zero_acc(x);
            for (int K = J; K < I; ++K)
                mma_acc(x, ld_a(hs + OFF_TT + BLK_B * bi(K, J), g, c), hs + OFF_NB + BLK_B * nbi(I, K), g, c);
            float t[2][4];
            zero_acc(t);
            mma_acc(t, a_from_acc(x[0], x[1], -1.f), hs + OFF_TD + BLK_B * I, g, c);
            // Tᵀ(J, I): rows g, g + 8; pairs 4 h + c
            uint8_t *tt = hs + OFF_TT + BLK_B * bi(I, J);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                st_pair(tt, g, 4 * h + c, hl_pair(t[h][0], t[h][1]));
                st_pair(tt, g + 8, 4 * h + c, hl_pair(t[h][2], t[h][3]));
            }
            // Tw: Tᵀ(J, I)[m][n] = T[16 I + n][16 J + m]; columns 16 J + g, + 1 paired
            // with the lane of g + 1 (lane + 4)
            const float b0 = bw[16 * J + g], b8 = bw[16 * J + g + 8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = 8 * h + 2 * c, r0 = 16 * I + n;
                const float w0 = rw[r0], w1 = rw[r0 + 1];
                const float v[4] = {t[h][0] * b0 * w0, t[h][1] * b0 * w1, t[h][2] * b8 * w0, t[h][3] * b8 * w1};
                float vn[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) vn[i] = __shfl_down_sync(0xffffffffu, v[i], 4);
                if ((g & 1) == 0) {
                    st_tile_pair(slot, r0, 16 * J + g, v[0], vn[0]);
                    st_tile_pair(slot, r0 + 1, 16 * J + g, v[1], vn[1]);
                    st_tile_pair(slot, r0, 16 * J + g + 8, v[2], vn[2]);
                    st_tile_pair(slot, r0 + 1, 16 * J + g + 8, v[3], vn[3]);
                }
            }
        }
        if (d < 3) named_sync(bar, NT);
    }
}

// The head's P T from P and Tᵀ blocks, by the four warps w: block (I, J), I >= J,
// costs I - J + 1 products; the groups {30, 00}, {20, 10}, {31, 21},
// {32, 11, 22, 33} cost five each.
__device__ __forceinline__ void solve_pt(const uint8_t *hs, const float *gates, uint8_t *slot, int w, int lane) {
    const int g = lane >> 2, c = lane & 3;
    const float *bw = gates + 64;  // column weights beta
    const uint32_t blocks = w == 0 ? 0x0030u : w == 1 ? 0x1020u : w == 2 ? 0x2131u : 0x33221132u;
    const int nblk = w == 3 ? 4 : 2;
    for (int b = 0; b < nblk; ++b) {
        const uint32_t code = (blocks >> (8 * b)) & 0xFFu;
        const int I = (int)(code >> 4), J = (int)(code & 15u);
        float acc[2][4];
        zero_acc(acc);
        for (int K = J; K <= I; ++K)
            mma_acc(acc, ld_a(hs + OFF_PB + BLK_B * bi(I, K), g, c), hs + OFF_TT + BLK_B * bi(K, J), g, c);
        // rows 16 I + g (+ 8); columns 16 J + 8 h + 2 c, + 1 (kept chunks only), times beta
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int cg = 16 * J + 8 * h + 2 * c;
            const float b0 = bw[cg], b1 = bw[cg + 1];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int rg = 16 * I + g + 8 * hr;
                if ((cg >> 3) <= (rg >> 3))
                    st_tile_pair(slot, 64 + rg, cg, acc[h][2 * hr] * b0, acc[h][2 * hr + 1] * b1);
            }
        }
    }
}

// Row `row` (a TMEM lane this warp may read) of X from TMEM columns 64-127 into
// a shared-memory image of the fp16 X tile (128-byte swizzled) at `img`.
__device__ __forceinline__ void stage_x_row(uint32_t tmem, int warp, int row, uint8_t *img) {
    uint8_t *xt = img + (size_t)row * 128;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
        float v[32];
        tmem_ld32(lane_addr + 64 + 32 * hf, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float *w = v + 8 * q;
            const uint32_t off = (uint32_t)((((4 * hf + q) ^ (row & 7)) & 7) << 4);
            *reinterpret_cast<uint4 *>(xt + off) = make_uint4(pack_f16x2(w[0], w[1]), pack_f16x2(w[2], w[3]),
                                                              pack_f16x2(w[4], w[5]), pack_f16x2(w[6], w[7]));
        }
    }
}

// QKN: the fused q/k L2 normalisation; BL: beta from logits (compile-time, so the
// default kernel carries no code for either).
template <bool QKN, bool BL>
__device__ __forceinline__ void factor_body(const CUtensorMap &tmK, const CUtensorMap &tmQ, const FacParams &p) {
    // a chunk scan queued behind this launch as a programmatic dependent may start
    // its prologue now; it waits for this grid before it reads the workspace
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t slot = p.slot_lo + blockIdx.x;
    const int h = blockIdx.y, hq = h / (p.h_v / p.h_qk);
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
    if (c < p.c_lo || c >= p.c_hi) return;     // a chunk outside this launch's range
    const int64_t t0 = ts0 + c * C;
    const int L = (int)((ts1 - t0) < C ? (ts1 - t0) : C);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *gates = reinterpret_cast<float *>(sm + OFF_GATES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + off_tmem(QKN));
    const uint32_t bar_tma = sb + off_bars(QKN), bar_mma = sb + off_bars(QKN) + 8;

    // raw gates first (warp 0): their latency overlaps the tile load
    float rg0 = 0.f, rg1 = 0.f, rb0 = 0.f, rb1 = 0.f;
    if (warp == 0) {
        if (lane < L) {
            const size_t i = (size_t)(t0 + lane) * p.h_v + h;
            rg0 = p.g[i] * kLog2e;
            rb0 = beta_of(p.beta[i], BL);
        }
        if (lane + 32 < L) {
            const size_t i = (size_t)(t0 + lane + 32) * p.h_v + h;
            rg1 = p.g[i] * kLog2e;
            rb1 = beta_of(p.beta[i], BL);
        }
    }
    // X writer: the first V head of the QK head's group; the first chunk of a
    // sequence has no X
    const bool want_x = c >= 1 && h % (p.h_v / p.h_qk) == 0;
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, want_x ? 49152u : 32768u);
        tma_load_3d(sb + OFF_KQ, &tmK, bar_tma, 0, hq, (int)t0);
        tma_load_3d(sb + OFF_KQ + 16384, &tmK, bar_tma, 64, hq, (int)t0);
        tma_load_3d(sb + OFF_KQ + 8192, &tmQ, bar_tma, 0, hq, (int)t0);
        tma_load_3d(sb + OFF_KQ + 16384 + 8192, &tmQ, bar_tma, 64, hq, (int)t0);
        if (want_x) {
            tma_load_3d(sb + OFF_KP, &tmK, bar_tma, 0, hq, (int)(t0 - C));
            tma_load_3d(sb + OFF_KP + 8192, &tmK, bar_tma, 64, hq, (int)(t0 - C));
        }
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    if (warp == 0) chunk_gates(rg0, rg1, rb0, rb1, gates, lane);

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
            if (want_x) {
                // X = [K; Q] K_prevᵀ into TMEM columns 64-127
                const uint64_t b0 = smem_desc_sw128(sb + OFF_KP, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tmem + 64, desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32),
                             desc_add(b0, (ks >> 2) * 8192 + (ks & 3) * 32), IDESC_G1, ks > 0);
            }
            mma_commit(bar_mma);
        }
    }
    if (QKN && ok && tid >= 64) {
        // fused L2 normalisation of the Q rows, while the Gram MMAs run (they only read
        // the tile too): thread i takes row i of the [K; Q] tile (both d_k halves; the
        // order of the sum does not matter).  Thread i starts at 16-byte piece i % 8 of
        // the row, so that a warp's loads spread over the banks (the same piece of 32
        // rows would hit one bank group).  (The K rows' norms are the Gram's diagonal.)
        ok = mbar_wait_bounded(bar_tma, 0, kWaitLimit);  // the tile's bytes are visible to this thread
        float ss = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const int ch = (c8 + tid) & 7;
                const uint4 wv = *reinterpret_cast<const uint4 *>(sm + OFF_KQ + 16384 * hf + 128 * tid + 16 * ch);
                const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float lo = __uint_as_float(w4[u] << 16), hi = __uint_as_float(w4[u] & 0xFFFF0000u);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
            }
        gates[256 + tid] = l2norm_scale(ss);  // rows 64-127: 1 / |q_t|
    }
    ok = ok && mbar_wait_bounded(bar_mma, 0, kWaitLimit);
    if (QKN && warp < 2) {
        // the K rows' norms: |k_t|^2 = (K Kᵀ)[t][t], the Gram's diagonal in TMEM (lane t,
        // column t: warp w reads columns 32 w .. + 31 of its lanes)
        tc_fence_after_sync();
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * warp, v);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) ss = (e == lane) ? v[e] : ss;
        if (ok) gates[256 + tid] = l2norm_scale(ss);  // rows 0-63: 1 / |k_t|
    }
    if (!ok) atomicCAS(p.err, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
    if (!__syncthreads_and(ok)) {  // also publishes the gates and the row scales
        // let the tile load land before this CTA's shared memory is released
        if (tid == 0) mbar_wait_bounded(bar_tma, 0, kWaitLimit / 8);
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, TM_COLS);
        return;
    }
    tc_fence_after_sync();

    // N (K rows, lanes 0-63) and P (Q rows, lanes 64-127), masked in log space,
    // 16 Gram columns at a time into blocks
    {
        const int row = 32 * warp + lane, t = row & 63, I = t >> 4, r16 = t & 15;
        const bool is_n = row < 64;
        const float Gt = gates[t];
        // row weight beta_t (N) or 1 (P), times the row's L2 scale with the fused normalisation
        const float w = QKN ? (is_n ? gates[64 + t] : 1.f) * gates[256 + row] : (is_n ? gates[64 + t] : 1.f);
        const int lim = is_n ? t : t + 1;  // keep j < t (N) or j <= t (P)
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            float v[16];
            tmem_ld16(lane_addr + 16 * J, v);
            if (J > I) continue;
            if constexpr (QKN) {  // column scales 1 / |k_j|
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] *= gates[256 + 16 * J + e];
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = 16 * J + e;
                v[e] = (j < lim) ? w * fast_exp2(Gt - gates[j]) * v[e] : 0.f;
            }
            if (is_n && J == I) {
                float *nd = reinterpret_cast<float *>(sm + OFF_ND) + 256 * I + 16 * r16;
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4 *>(nd + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            } else {
                uint8_t *blk = sm + (is_n ? OFF_NB + BLK_B * nbi(I, J) : OFF_PB + BLK_B * bi(I, J));
#pragma unroll
                for (int q = 0; q < 8; ++q) st_pair(blk, r16, q, hl_pair(v[2 * q], v[2 * q + 1]));
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    uint8_t *slot_out = p.ws + ((size_t)slot * p.h_v + h) * fac::SLOT_BYTES;
    uint8_t *xtile = p.xs + ((size_t)slot * p.h_qk + hq) * fac::X_BYTES;
    if (warp >= 2) {
        // while warps 0-1 invert the diagonal blocks: exp(G), and the zero 8-column
        // chunks right of each row's diagonal chunk (thread i of warps 2-3: rows i
        // of Tw and 64 + i of PTw)
        if (warp == 2) {
            float *eg = reinterpret_cast<float *>(slot_out + fac::OFF_EG);
            eg[lane] = gates[128 + lane];
            eg[lane + 32] = gates[160 + lane];
            if constexpr (QKN) {  // the row scales for the chunk scan: 1 / |k| (64), then 1 / |q| (64)
                float *rs = reinterpret_cast<float *>(slot_out + fac::OFF_RK);
#pragma unroll
                for (int i = 0; i < 4; ++i) rs[lane + 32 * i] = gates[256 + lane + 32 * i];
            }
        }
        const int t = tid - 64;
        for (int k = (t >> 3) + 1; k < 8; ++k) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint32_t off = fac::sw128_elem(t + 64 * m, 8 * k);
                *reinterpret_cast<uint4 *>(slot_out + fac::OFF_T + off) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    solve_t(sm, gates, slot_out, warp, lane, 1);
    __syncthreads();
    solve_pt(sm, gates, slot_out, warp, lane);
    if (want_x) {
        // X through the free scratch: each thread stages its row, then one bulk
        // store writes the 16 KB tile (rows of 16-byte pieces at 128-byte
        // strides, stored from registers, were the slowest part of the kernel)
        __syncthreads();  // every warp is done with the scratch
        stage_x_row(tmem, warp, tid, sm);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             reinterpret_cast<uint64_t>(xtile)),
                         "r"(sb), "r"((uint32_t)fac::X_BYTES)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // before the CTA's memory is released
        }
    }
    tc_fence_before_sync();
    __syncthreads();  // every TMEM read is done before the columns are freed
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// One kernel per option set (the default one first).
__global__ void __launch_bounds__(NT, 4) factor_kernel(const __grid_constant__ CUtensorMap tmK,
                                                       const __grid_constant__ CUtensorMap tmQ, FacParams p) {
    factor_body<false, false>(tmK, tmQ, p);
}
__global__ void __launch_bounds__(NT, 4) factor_kernel_beta_logits(const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmQ,
                                                                   FacParams p) {
    factor_body<false, true>(tmK, tmQ, p);
}
__global__ void __launch_bounds__(NT, 4) factor_kernel_qk_l2norm(const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmQ,
                                                                 FacParams p) {
    factor_body<true, false>(tmK, tmQ, p);
}
__global__ void __launch_bounds__(NT, 4) factor_kernel_qk_l2norm_beta_logits(const __grid_constant__ CUtensorMap tmK,
                                                                             const __grid_constant__ CUtensorMap tmQ,
                                                                             FacParams p) {
    factor_body<true, true>(tmK, tmQ, p);
}

}  // namespace

cudaError_t launch_factors(const Args &a, float *ws, int32_t *err, cudaStream_t s, bool overlap) {
    CUtensorMap tmK, tmQ;
    if (!encode_bf16_3d(&tmK, a.k, 128, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_3d(&tmQ, a.q, 128, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(factor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes(false));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(factor_kernel_beta_logits, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes(false));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(factor_kernel_qk_l2norm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes(true));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(factor_kernel_qk_l2norm_beta_logits, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes(true));
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
    p.ws = reinterpret_cast<uint8_t *>(ws);
    p.xs = reinterpret_cast<uint8_t *>(ws) + fac::x_region_offset(fac::n_slots(a.t_total, a.n_seqs), a.h_v);
    p.err = err;
    p.c_lo = a.c_lo;
    p.c_hi = a.c_hi;
    // one sequence: chunk c is slot c, so the launch covers exactly its range;
    // packed sequences: every slot, each CTA checks its chunk against the range
    int64_t slot_lo = 0, slot_hi = fac::n_slots(a.t_total, a.n_seqs);
    if (a.n_seqs == 1) {
        slot_lo = a.c_lo;
        if ((int64_t)a.c_hi < slot_hi) slot_hi = a.c_hi;
    }
    if (slot_hi <= slot_lo) return cudaSuccess;
    p.slot_lo = slot_lo;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(slot_hi - slot_lo), (unsigned)a.h_v);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem_bytes(a.qk_norm != 0);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = overlap ? &attr : nullptr;
    cfg.numAttrs = overlap ? 1 : 0;
    auto kern = a.qk_norm ? (a.beta_logits ? factor_kernel_qk_l2norm_beta_logits : factor_kernel_qk_l2norm)
                          : (a.beta_logits ? factor_kernel_beta_logits : factor_kernel);
    return cudaLaunchKernelEx(&cfg, kern, tmK, tmQ, p);
}

}  // namespace gdr
