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

    constexpr int KSTR = D + 4;  // tile row stride: rows stay 16-byte aligned for float4 reads
    __shared__ __align__(16) float sK[C][KSTR];
    __shared__ __align__(16) float sQ[C][KSTR];
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
        // this lane's column of V for the chunk, requested before anything else
        float vpre[C];
#pragma unroll
        for (int t = 0; t < C; ++t)
            vpre[t] = (t < L) ? load_in(a.v, ((size_t)(c0 + t) * a.h_v + h) * D + col, a.in_bf16) : 0.f;
        // K and Q tiles, 16 bytes per load (8 bf16 or 4 fp32 values)
        if (a.in_bf16) {
#pragma unroll
            for (int e = threadIdx.x; e < C * D / 8; e += NT) {
                const int t = (8 * e) / D, i = (8 * e) % D;
                uint4 kw = make_uint4(0u, 0u, 0u, 0u), qw = kw;
                if (t < L) {
                    const size_t off = ((size_t)(c0 + t) * a.h_qk + hq) * D + i;
                    kw = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.k) + off);
                    qw = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.q) + off);
                }
                const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w}, qq[4] = {qw.x, qw.y, qw.z, qw.w};
                float kf[8], qf[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    kf[2 * u] = __uint_as_float(kk[u] << 16);
                    kf[2 * u + 1] = __uint_as_float(kk[u] & 0xFFFF0000u);
                    qf[2 * u] = __uint_as_float(qq[u] << 16);
                    qf[2 * u + 1] = __uint_as_float(qq[u] & 0xFFFF0000u);
                }
                *reinterpret_cast<float4 *>(&sK[t][i]) = make_float4(kf[0], kf[1], kf[2], kf[3]);
                *reinterpret_cast<float4 *>(&sK[t][i + 4]) = make_float4(kf[4], kf[5], kf[6], kf[7]);
                *reinterpret_cast<float4 *>(&sQ[t][i]) = make_float4(qf[0], qf[1], qf[2], qf[3]);
                *reinterpret_cast<float4 *>(&sQ[t][i + 4]) = make_float4(qf[4], qf[5], qf[6], qf[7]);
            }
        } else {
#pragma unroll
            for (int e = threadIdx.x; e < C * D / 4; e += NT) {
                const int t = (4 * e) / D, i = (4 * e) % D;
                float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), qv = kv;
                if (t < L) {
                    const size_t off = ((size_t)(c0 + t) * a.h_qk + hq) * D + i;
                    kv = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.k) + off);
                    qv = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.q) + off);
                }
                *reinterpret_cast<float4 *>(&sK[t][i]) = kv;
                *reinterpret_cast<float4 *>(&sQ[t][i]) = qv;
            }
        }
        if (threadIdx.x < 32) {
            // inclusive running sum of g over the chunk (padding: g = 0, beta = 0)
            float gt = 0.f, bt = 0.f;
            if (lane < L) {
                gt = a.g[(size_t)(c0 + lane) * a.h_v + h];
                bt = beta_of(a.beta[(size_t)(c0 + lane) * a.h_v + h], a.beta_logits);
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
        if (a.qk_norm) {
            // fused L2 normalisation of the chunk's k and q rows, in place (a
            // padding row is zero and stays zero)
            for (int rr = p; rr < 2 * C; rr += SPLIT) {
                float *row = rr < C ? sK[rr] : sQ[rr - C];
                float ss = 0.f;
                for (int i = lane; i < D; i += 32) ss = fmaf(row[i], row[i], ss);
                const float sc = l2norm_scale(warp_sum(ss));
                for (int i = lane; i < D; i += 32) row[i] *= sc;
            }
            __syncthreads();
        }

        // Gram products for the chunk: N (strict lower, beta and decay applied), P (lower).
        for (int e = threadIdx.x; e < C * C; e += NT) {
            const int t = e / C, j = e - t * C;
            float nk = 0.f, pq = 0.f;
            if (j <= t) {
                float dk = 0.f, dq = 0.f;
#pragma unroll 8
                for (int i = 0; i < D; i += 4) {
                    const float4 kt = *reinterpret_cast<const float4 *>(&sK[t][i]);
                    const float4 kj = *reinterpret_cast<const float4 *>(&sK[j][i]);
                    const float4 qt = *reinterpret_cast<const float4 *>(&sQ[t][i]);
                    dk = fmaf(kt.x, kj.x, fmaf(kt.y, kj.y, fmaf(kt.z, kj.z, fmaf(kt.w, kj.w, dk))));
                    dq = fmaf(qt.x, kj.x, fmaf(qt.y, kj.y, fmaf(qt.z, kj.z, fmaf(qt.w, kj.w, dq))));
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
            for (int r = 0; r < RPT; r += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sK[t][row0 + r]);
                const float4 q4 = *reinterpret_cast<const float4 *>(&sQ[t][row0 + r]);
                x = fmaf(k4.x, sreg[r], fmaf(k4.y, sreg[r + 1], fmaf(k4.z, sreg[r + 2], fmaf(k4.w, sreg[r + 3], x))));
                y = fmaf(q4.x, sreg[r], fmaf(q4.y, sreg[r + 1], fmaf(q4.z, sreg[r + 2], fmaf(q4.w, sreg[r + 3], y))));
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
            for (int t = 0; t < C; ++t) rr[t] = sB[t] * (vpre[t] - __expf(sG[t]) * ks[t]);
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
        for (int r = 0; r < RPT; ++r) sreg[r] *= eC;
#pragma unroll
        for (int t = 0; t < C; ++t) {
#pragma unroll
            for (int r = 0; r < RPT; r += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sK[t][row0 + r]);
                sreg[r] = fmaf(k4.x, dcol[t], sreg[r]);
                sreg[r + 1] = fmaf(k4.y, dcol[t], sreg[r + 1]);
                sreg[r + 2] = fmaf(k4.z, dcol[t], sreg[r + 2]);
                sreg[r + 3] = fmaf(k4.w, dcol[t], sreg[r + 3]);
            }
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
