// The speculative-verify block: one chunk of up to 16 tokens per sequence from
// its current state, with a snapshot of that state (the prompt-lookup loop of
// the Qwen3.5-9B NPU model card, "New in v2").  bf16 q/k/v; fp32 inputs take
// the CUDA-core chunk kernel instead.
//
// Math (the chunkwise-parallel form on the same card, "How it works"), for the
// block's tokens t < 16 with G the inclusive running sum of g:
//     N_tj = beta_t e^{G_t - G_j} k_t . k_j   (j < t)     P_tj = e^{G_t - G_j} q_t . k_j   (j <= t)
//     R    = diag(beta) (V - diag(e^G) K S)                D = (I + N)^-1 R
//     O    = scale (diag(e^G) Q S + P D)                   S' = e^{G_C} S + K^T diag(e^{G_C - G}) D
// The exponent G_t - G_j is formed only on the kept triangle.  Rows past n_tok
// are padding (k = q = v = 0, g = 0, beta = 0).
//
// Design: the op is a chain of small dependent steps, so the kernel is built
// for latency.  A block of 256 threads owns (sequence, V head, 16 state
// columns): 8 blocks per head at d = 128.  Every global read is issued at the
// start with cp.async (the state slice, the bf16 K, Q and V tiles; g and beta
// as plain loads), one wait.  The products with d-long inner dimensions run on
// warp-level bf16 tensor-core MMAs (m16n8k16, fp32 accumulation): the 8 warps
// take one 16 x 8 output tile each of [K; Q] S (the state split into bf16 hi
// and lo halves, so the products keep 2^-16 relative precision) and of the
// Gram [K; Q] K^T (exact: bf16 products).  D comes from a right-looking
// forward substitution on one warp (one column per lane; T is never formed),
// then O on all threads and S' on tensor cores again (K^T diag(w) D, D split
// into hi and lo), added to e^{G_C} S and stored.
#include "gdr_common.cuh"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {
namespace {

using tc::pack_bf16x2;
using tc::smem_u32;

constexpr int C = 16;       // tokens per block
constexpr int BV = 16;      // state columns per block
constexpr int NT = 256;     // threads
constexpr int LD = BV + 4;  // fp32 row stride of the small tiles (conflict-free fragment reads)

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// d += A B, A 16 x 16 and B 16 x 8 in bf16, d in fp32 (lane = 4 g + c holds
// rows g, g + 8 and columns 2c, 2c + 1 of the 16 x 8 tile).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// bf16 hi and lo words of the pair (x0, x1): hi = the top 16 bits, lo = bf16(x - hi).
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t a = __float_as_uint(x0), b = __float_as_uint(x1);
    hi = __byte_perm(a, b, 0x7632);
    lo = pack_bf16x2(x0 - __uint_as_float(a & 0xFFFF0000u), x1 - __uint_as_float(b & 0xFFFF0000u));
}
__device__ __forceinline__ float bf16_at(const uint8_t *row, int i) {
    return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(row)[i] << 16);
}

template <int D>
struct VShape {
    static constexpr int KB = D * 2 + 16;  // bytes per K / Q row in shared memory (padded for ldmatrix)
    static constexpr int KSTEPS = D / 16;
};

template <int D>
__global__ void __launch_bounds__(NT) verify_kernel(Args a) {
    using Sh = VShape<D>;
    __shared__ __align__(128) uint8_t sK[C * Sh::KB];
    __shared__ __align__(128) uint8_t sQ[C * Sh::KB];
    __shared__ __align__(16) float sS[D * LD];      // the block's 16 columns of the state
    __shared__ __align__(16) uint8_t sV[C * BV * 2];
    __shared__ __align__(16) float sKS[C * LD], sQS[C * LD], sGk[C * LD], sGq[C * LD];
    __shared__ __align__(16) float sNT[C * LD];     // N transposed: sNT[j][t] = N_tj
    __shared__ __align__(16) float sP[C * LD], sR[C * LD], sD[C * LD];
    __shared__ float sG[C], sB[C], sRQ[C], sW[C];

    constexpr int ncb = D / BV;
    const int cb = blockIdx.x % ncb;
    const int h = (blockIdx.x / ncb) % a.h_v;
    const int s = blockIdx.x / (ncb * a.h_v);
    const int hq = h / (a.h_v / a.h_qk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tok = a.fixed_len;
    const size_t row0 = (size_t)s * n_tok;
    const int c0 = cb * BV;
    float *Sg = a.state + ((size_t)s * a.h_v + h) * D * D;

    // ---- every global read, issued at once -------------------------------------
    for (int e = tid; e < D * (BV / 4); e += NT) {  // state rows: 4 x 16 B each
        const int r = e >> 2, q4 = e & 3;
        cp_async16(&sS[r * LD + 4 * q4], Sg + (size_t)r * D + c0 + 4 * q4);
    }
    {
        const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k);
        const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q);
        constexpr int PER_ROW = D / 8;  // 16-byte pieces of a row
        for (int e = tid; e < C * PER_ROW; e += NT) {
            const int t = e / PER_ROW, i = e - t * PER_ROW;
            uint8_t *dk = sK + t * Sh::KB + 16 * i, *dq = sQ + t * Sh::KB + 16 * i;
            if (t < n_tok) {
                const size_t off = ((row0 + t) * a.h_qk + hq) * D + 8 * i;
                cp_async16(dk, kg + off);
                cp_async16(dq, qg + off);
            } else {
                *reinterpret_cast<uint4 *>(dk) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(dq) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (tid < 2 * C) {  // V: two 16-byte pieces per token row
            const int t = tid >> 1, i = tid & 1;
            uint8_t *dv = sV + t * (BV * 2) + 16 * i;
            if (t < n_tok)
                cp_async16(dv, reinterpret_cast<const __nv_bfloat16 *>(a.v) + ((row0 + t) * a.h_v + h) * D + c0 + 8 * i);
            else
                *reinterpret_cast<uint4 *>(dv) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (warp == 0) {
        // gates: G inclusive running sum of g, beta (padding rows: g = 0, beta = 0)
        float gt = 0.f, bt = 0.f;
        if (lane < n_tok) {
            gt = a.g[(row0 + lane) * a.h_v + h];
            bt = beta_of(a.beta[(row0 + lane) * a.h_v + h], a.beta_logits);
        }
#pragma unroll
        for (int o = 1; o < C; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, gt, o);
            if (lane >= o) gt += u;
        }
        if (lane < C) {
            sG[lane] = gt;
            sB[lane] = bt;
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- the snapshot, straight from shared memory ---------------------------------
    {
        float *Sn = a.snapshot + ((size_t)s * a.h_v + h) * D * D;
        for (int e = tid; e < D * (BV / 4); e += NT) {
            const int r = e >> 2, q4 = e & 3;
            *reinterpret_cast<float4 *>(Sn + (size_t)r * D + c0 + 4 * q4) =
                *reinterpret_cast<const float4 *>(&sS[r * LD + 4 * q4]);
        }
    }

    // ---- [K; Q] S and [K; Q] K^T: one 16 x 8 output tile per warp -----------------
    const int g8 = lane >> 2, c4 = lane & 3;
    {
        const int m = warp >> 2, n = warp & 3;
        const uint8_t *A = m ? sQ : sK;
        // ldmatrix row addresses of the A fragment: lanes 8i..8i+7 give matrix i
        const int arow = ((lane >> 3) & 1) * 8 + (lane & 7), acol = (lane >> 4) * 8;
        const uint32_t a_addr = smem_u32(A + arow * Sh::KB + acol * 2);
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
        if (n < 2) {
            // S columns 8n .. 8n + 7 of the block, as the B operand in hi and lo halves
            const float *Sb = sS + 8 * n + g8;
#pragma unroll
            for (int ks = 0; ks < Sh::KSTEPS; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(a_addr + ks * 32, a0, a1, a2, a3);
                const int r = 16 * ks + 2 * c4;
                uint32_t h0, l0, h1, l1;
                split_pair(Sb[r * LD], Sb[(r + 1) * LD], h0, l0);
                split_pair(Sb[(r + 8) * LD], Sb[(r + 9) * LD], h1, l1);
                mma_bf16(acc, a0, a1, a2, a3, h0, h1);
                mma_bf16(acc2, a0, a1, a2, a3, l0, l1);
            }
        } else {
            // key tokens 8(n - 2) .. + 7: B = K^T, read as K rows
            const int j0 = 8 * (n - 2);
            const uint32_t b_addr = smem_u32(sK + (j0 + (lane & 7)) * Sh::KB + ((lane >> 3) & 1) * 16);
#pragma unroll
            for (int ks = 0; ks < Sh::KSTEPS; ++ks) {
                uint32_t a0, a1, a2, a3, b0, b1;
                ldsm_x4(a_addr + ks * 32, a0, a1, a2, a3);
                ldsm_x2(b_addr + ks * 32, b0, b1);
                mma_bf16((ks & 1) ? acc2 : acc, a0, a1, a2, a3, b0, b1);
            }
        }
        float *out = n < 2 ? (m ? sQS : sKS) + 8 * n : (m ? sGq : sGk) + 8 * (n - 2);
        *reinterpret_cast<float2 *>(out + g8 * LD + 2 * c4) = make_float2(acc[0] + acc2[0], acc[1] + acc2[1]);
        *reinterpret_cast<float2 *>(out + (g8 + 8) * LD + 2 * c4) = make_float2(acc[2] + acc2[2], acc[3] + acc2[3]);
    }
    if (a.qk_norm) {
        // fused L2 normalisation: |q_t| from the raw tile (|k_t| is the Gram's diagonal)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = 2 * warp + i;
            float ss = 0.f;
            for (int x = lane; x < D; x += 32) {
                const float v = bf16_at(sQ + t * Sh::KB, x);
                ss = fmaf(v, v, ss);
            }
            ss = warp_sum(ss);
            if (lane == 0) sRQ[t] = l2norm_scale(ss);
        }
    }
    __syncthreads();

    // ---- masks, R and the Q S term: thread (t, c) ------------------------------------
    const int t = tid >> 4, c = tid & 15;
    float qs_term;
    {
        const float Gt = sG[t], Gc = sG[c], bt = sB[t];
        const float rk_t = a.qk_norm ? l2norm_scale(sGk[t * LD + t]) : 1.f;
        const float rk_c = a.qk_norm ? l2norm_scale(sGk[c * LD + c]) : 1.f;
        const float rq_t = a.qk_norm ? sRQ[t] : 1.f;
        const float dec = c <= t ? __expf(Gt - Gc) : 0.f;  // exponent <= 0 on the kept triangle
        sNT[c * LD + t] = c < t ? bt * dec * rk_t * rk_c * sGk[t * LD + c] : 0.f;
        sP[t * LD + c] = dec * rq_t * rk_c * sGq[t * LD + c];
        const float eg = __expf(Gt);
        const float vv = bf16_at(sV + t * (BV * 2), c);
        sR[t * LD + c] = bt * (vv - eg * rk_t * sKS[t * LD + c]);
        qs_term = eg * rq_t * sQS[t * LD + c];
        if (c == 0) sW[t] = rk_t * __expf(sG[C - 1] - Gt);  // weight of token t in S'
    }
    __syncthreads();

    // ---- D = (I + N)^-1 R: right-looking forward substitution, lane = column --------
    if (warp == 0) {
        const int col = lane & 15;
        float x[C];
#pragma unroll
        for (int i = 0; i < C; ++i) x[i] = sR[i * LD + col];
#pragma unroll
        for (int j = 0; j < C - 1; ++j) {
            const float xj = x[j];
#pragma unroll
            for (int q = (j + 1) / 4; q < C / 4; ++q) {
                const float4 nt = *reinterpret_cast<const float4 *>(&sNT[j * LD + 4 * q]);
                if (4 * q + 0 > j) x[4 * q + 0] = fmaf(-nt.x, xj, x[4 * q + 0]);
                if (4 * q + 1 > j) x[4 * q + 1] = fmaf(-nt.y, xj, x[4 * q + 1]);
                if (4 * q + 2 > j) x[4 * q + 2] = fmaf(-nt.z, xj, x[4 * q + 2]);
                if (4 * q + 3 > j) x[4 * q + 3] = fmaf(-nt.w, xj, x[4 * q + 3]);
            }
        }
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < C; ++i) sD[i * LD + col] = x[i];
            if (a.deltas) {
#pragma unroll
                for (int i = 0; i < C; ++i)
                    if (i < n_tok) a.deltas[((row0 + i) * a.h_v + h) * D + c0 + col] = x[i];
            }
        }
    }
    __syncthreads();

    // ---- O = scale (e^G Q S + P D) ------------------------------------------------------
    if (t < n_tok) {
        float o = qs_term;
#pragma unroll
        for (int q = 0; q < C / 4; ++q) {
            const float4 p4 = *reinterpret_cast<const float4 *>(&sP[t * LD + 4 * q]);
            o = fmaf(p4.x, sD[(4 * q + 0) * LD + c], o);
            o = fmaf(p4.y, sD[(4 * q + 1) * LD + c], o);
            o = fmaf(p4.z, sD[(4 * q + 2) * LD + c], o);
            o = fmaf(p4.w, sD[(4 * q + 3) * LD + c], o);
        }
        store_out(a.o, ((row0 + t) * a.h_v + h) * D + c0 + c, a.scale * o, a.out_bf16);
    }

    // ---- S' = e^{G_C} S + K^T diag(w) D: warp w takes state rows 16w .. 16w + 15 --------
    if (warp < D / 16) {
        const int r0 = 16 * warp;
        // A = K^T (rows r, columns t) from the K tile by transposed ldmatrix:
        // matrix i of lanes 8i..8i+7: token rows 8(i >> 1) + (lane & 7), state rows r0 + 8(i & 1)
        const uint32_t at_addr =
            smem_u32(sK + (8 * (lane >> 4) + (lane & 7)) * Sh::KB + (r0 + 8 * ((lane >> 3) & 1)) * 2);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(at_addr, a0, a1, a2, a3);
        const float eC = __expf(sG[C - 1]);
        const float w0 = sW[2 * c4], w1 = sW[2 * c4 + 1], w8 = sW[2 * c4 + 8], w9 = sW[2 * c4 + 9];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = 8 * nt + g8;
            uint32_t h0, l0, h1, l1;
            split_pair(w0 * sD[(2 * c4) * LD + col], w1 * sD[(2 * c4 + 1) * LD + col], h0, l0);
            split_pair(w8 * sD[(2 * c4 + 8) * LD + col], w9 * sD[(2 * c4 + 9) * LD + col], h1, l1);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16(acc, a0, a1, a2, a3, h0, h1);
            mma_bf16(acc, a0, a1, a2, a3, l0, l1);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = r0 + g8 + 8 * hh, cc = 8 * nt + 2 * c4;
                const float2 sv = *reinterpret_cast<const float2 *>(&sS[r * LD + cc]);
                *reinterpret_cast<float2 *>(Sg + (size_t)r * D + c0 + cc) =
                    make_float2(fmaf(eC, sv.x, acc[2 * hh]), fmaf(eC, sv.y, acc[2 * hh + 1]));
            }
        }
    }
}

}  // namespace

cudaError_t launch_verify(const Args &a, cudaStream_t s) {
    if (a.n_seqs == 0) return cudaSuccess;
    if (!a.in_bf16 || a.fixed_len < 1 || a.fixed_len > C) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)a.n_seqs * (unsigned)a.h_v * (unsigned)(a.d / BV);
    switch (a.d) {
        case 32: verify_kernel<32><<<blocks, NT, 0, s>>>(a); break;
        case 64: verify_kernel<64><<<blocks, NT, 0, s>>>(a); break;
        case 128: verify_kernel<128><<<blocks, NT, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdr
