// Chunked gated delta rule on CUDA cores, 16-token chunks.
//
// Serves the speculative-verify block (one 16-token chunk from a snapshotted
// state) and every prefill shape the tensor-core kernel does not cover
// (d = 32 or 64, fp32 inputs, chunk 16).
//
// Per chunk of C = 16 tokens (the chunkwise-parallel form on the Qwen3.5-9B
// NPU model card, "How it works"), with G the running sum of g in the chunk:
//     N_tj = beta_t exp(G_t - G_j) (k_t . k_j)    j < t
//     P_tj =        exp(G_t - G_j) (q_t . k_j)    j <= t
//     D    = (I + N)^-1 diag(beta) (V - diag(e^G) K S)
//     O    = scale (diag(e^G) Q S + P D)
//     S   <- e^{G_C} S + K^T diag(e^{G_C - G}) D
// The exponent G_t - G_j is only formed on the lower triangle (the Candle PR's
// log-space masking), so strong decays cannot overflow.  Tail rows past the
// end of a sequence are padding (g = 0, beta = 0, k = q = v = 0).
//
// Mapping.  A block owns (sequence, V head, 32 state columns).  Warp p owns
// d/SPLIT state rows, lane j one column; the rows sit in registers for the
// whole sequence.  K and Q tiles are staged in shared memory and read as
// warp-wide broadcasts, so S^T k needs no shuffles: only the SPLIT partial sums
// of K S and Q S go through shared memory once per chunk (K S, then Q S, in one
// buffer).  Every warp holds the chunk's D column, so warp p stores the outputs
// and corrections of the tokens t = p mod SPLIT.
#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int C = 16;
constexpr int BV = 32;

template <int D>
struct CcShape {
    static constexpr int SPLIT = D / 16;  // warps per block (row groups of 16 rows)
    static constexpr int RPT = D / SPLIT;  // rows per thread
};

template <int D>
__global__ void __launch_bounds__(32 * CcShape<D>::SPLIT) chunk_cc_kernel(Args a) {
    constexpr int SPLIT = CcShape<D>::SPLIT;
    constexpr int RPT = CcShape<D>::RPT;
    constexpr int NT = 32 * SPLIT;

    __shared__ float sK[C][D + 1];
    __shared__ float sQ[C][D + 1];
    __shared__ float sG[C], sB[C];
    __shared__ float sN[C][C + 1];  // strictly lower part of N, later T = (I+N)^-1
    __shared__ float sP[C][C + 1];
    __shared__ float sT[C][C + 1];
    __shared__ float red[SPLIT][C][BV];

    const int ncb = D / BV;
    const int cb = blockIdx.x % ncb;
    const int h = (blockIdx.x / ncb) % a.h_v;
    const int s = blockIdx.x / (ncb * a.h_v);
    const int hq = h / (a.h_v / a.h_qk);
    const int p = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = cb * BV + lane;
    const int row0 = p * RPT;

    int64_t t0, t1;
    seq_bounds(a.cu_seqlens, a.fixed_len, s, t0, t1);

    float *Sg = a.state + ((size_t)s * a.h_v + h) * D * D;
    float sreg[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) sreg[r] = Sg[(size_t)(row0 + r) * D + col];
    if (a.snapshot) {
        float *Sn = a.snapshot + ((size_t)s * a.h_v + h) * D * D;
#pragma unroll
        for (int r = 0; r < RPT; ++r) Sn[(size_t)(row0 + r) * D + col] = sreg[r];
    }

    for (int64_t c0 = t0; c0 < t1; c0 += C) {
        const int L = (int)((t1 - c0) < C ? (t1 - c0) : C);
        __syncthreads();  // previous chunk's readers of shared tiles are done
        for (int e = threadIdx.x; e < C * D; e += NT) {
            const int t = e / D, i = e - t * D;
            float kv = 0.f, qv = 0.f;
            if (t < L) {
                const size_t off = ((size_t)(c0 + t) * a.h_qk + hq) * D + i;
                kv = load_in(a.k, off, a.in_bf16);
                qv = load_in(a.q, off, a.in_bf16);
            }
            sK[t][i] = kv;
            sQ[t][i] = qv;
        }
        if (threadIdx.x < 32) {
            // inclusive running sum of g over the chunk (padding: g = 0, beta = 0)
            float gt = 0.f, bt = 0.f;
            if (lane < L) {
                gt = a.g[(size_t)(c0 + lane) * a.h_v + h];
                bt = a.beta[(size_t)(c0 + lane) * a.h_v + h];
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, gt, o);
                if (lane >= o) gt += u;
            }
            if (lane < C) {
                sG[lane] = gt;
                sB[lane] = bt;
            }
        }
        __syncthreads();

        // Gram products for the chunk: N (strict lower, beta and decay applied), P (lower).
        for (int e = threadIdx.x; e < C * C; e += NT) {
            const int t = e / C, j = e - t * C;
            float nk = 0.f, pq = 0.f;
            if (j <= t) {
                float dk = 0.f, dq = 0.f;
#pragma unroll 8
                for (int i = 0; i < D; ++i) {
                    dk = fmaf(sK[t][i], sK[j][i], dk);
                    dq = fmaf(sQ[t][i], sK[j][i], dq);
                }
                const float decay = __expf(sG[t] - sG[j]);  // exponent <= 0 on this triangle
                pq = decay * dq;
                if (j < t) nk = sB[t] * decay * dk;
            }
            sN[t][j] = nk;
            sP[t][j] = pq;
        }
        __syncthreads();

        // T = (I + N)^-1 by forward substitution, one column per lane.
        if (threadIdx.x < C) {
            const int j = threadIdx.x;
            float tcol[C];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float acc = (t == j) ? 1.f : 0.f;
                if (t > j) {
#pragma unroll
                    for (int m = 0; m < C; ++m)
                        if (m >= j && m < t) acc = fmaf(-sN[t][m], tcol[m], acc);
                }
                tcol[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < C; ++t) sT[t][j] = tcol[t];
        }

        // Partial K S and Q S over this warp's rows, for this lane's column.
        float ks[C], qs[C];
#pragma unroll
        for (int t = 0; t < C; ++t) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                x = fmaf(sK[t][row0 + r], sreg[r], x);
                y = fmaf(sQ[t][row0 + r], sreg[r], y);
            }
            ks[t] = x;
            qs[t] = y;
        }
        // sum the SPLIT partials: K S first, then Q S through the same buffer
#pragma unroll
        for (int t = 0; t < C; ++t) red[p][t][lane] = ks[t];
        __syncthreads();
#pragma unroll
        for (int t = 0; t < C; ++t) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < SPLIT; ++w) x += red[w][t][lane];
            ks[t] = x;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < C; ++t) red[p][t][lane] = qs[t];
        __syncthreads();
#pragma unroll
        for (int t = 0; t < C; ++t) {
            float y = 0.f;
#pragma unroll
            for (int w = 0; w < SPLIT; ++w) y += red[w][t][lane];
            qs[t] = y;
        }

        // R = diag(beta)(V - diag(e^G) K S);  D = T R;  O = scale (e^G Q S + P D).
        float dcol[C];
        {
            float rr[C];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float vt = 0.f;
                if (t < L) vt = load_in(a.v, ((size_t)(c0 + t) * a.h_v + h) * D + col, a.in_bf16);
                rr[t] = sB[t] * (vt - __expf(sG[t]) * ks[t]);
            }
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m <= t; ++m) acc = fmaf(sT[t][m], rr[m], acc);
                dcol[t] = acc;
            }
        }
        if (a.deltas) {  // the corrections u_t of the chunk's real rows
#pragma unroll
            for (int t = 0; t < C; ++t)
                if (t < L && t % SPLIT == p) a.deltas[((size_t)(c0 + t) * a.h_v + h) * D + col] = dcol[t];
        }
        {
#pragma unroll
            for (int t = 0; t < C; ++t) {
                if (t < L && t % SPLIT == p) {
                    float acc = __expf(sG[t]) * qs[t];
#pragma unroll
                    for (int m = 0; m <= t; ++m) acc = fmaf(sP[t][m], dcol[m], acc);
                    store_out(a.o, ((size_t)(c0 + t) * a.h_v + h) * D + col, a.scale * acc, a.out_bf16);
                }
            }
        }

        // S <- e^{G_C} S + K^T diag(e^{G_C - G}) D
        const float gl = sG[C - 1];
#pragma unroll
        for (int t = 0; t < C; ++t) dcol[t] *= __expf(gl - sG[t]);
        const float eC = __expf(gl);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            float acc = eC * sreg[r];
#pragma unroll
            for (int t = 0; t < C; ++t) acc = fmaf(sK[t][row0 + r], dcol[t], acc);
            sreg[r] = acc;
        }
    }

#pragma unroll
    for (int r = 0; r < RPT; ++r) Sg[(size_t)(row0 + r) * D + col] = sreg[r];
}

}  // namespace

cudaError_t launch_chunk_cc(const Args &a, cudaStream_t s) {
    if (a.n_seqs == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)a.n_seqs * (unsigned)a.h_v * (unsigned)(a.d / BV);
    switch (a.d) {
        case 32: chunk_cc_kernel<32><<<blocks, 32 * CcShape<32>::SPLIT, 0, s>>>(a); break;
        case 64: chunk_cc_kernel<64><<<blocks, 32 * CcShape<64>::SPLIT, 0, s>>>(a); break;
        case 128: chunk_cc_kernel<128><<<blocks, 32 * CcShape<128>::SPLIT, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdr
