// Verify commit: the state after the accepted prefix of a speculative-verify
// block, formed from the block's cached corrections in one pass over the states.
//
// Unrolling S_t = e^{g_t} S_{t-1} + k_t u_t^T over the a accepted tokens of the
// block (the closed form of the state after a chunk on the Qwen3.5-9B NPU model
// card, "How it works", taken at row a - 1):
//     S_a = e^{G_a} S_0 + sum_{j < a} e^{G_a - G_j} k_j u_j^T,
// G_j the running sum of g inside the block (inclusive), G_a = G_{a-1}.  The
// corrections u_j = beta_j (v_j - e^{g_j} S_{j-1}^T k_j) of the first a tokens
// depend on no later token, so the ones the verify block computed for all
// n_tok tokens serve every prefix: this replaces restoring the snapshot and
// re-feeding the accepted tokens.
//
// Mapping.  One block of 256 threads per (sequence, V head, eighth of the state
// rows), so even one sequence spreads over 8 H_v blocks (verify block + commit:
// 9.3 us with 4, 8.8 us with 8, 10.3 us with 16, where every block reloads all
// n_tok corrections of its columns for fewer rows).  Thread t owns
// column quad t % (D/4) of rows t / (D/4) + k (256 / (D/4)), k < D / 4 / (256 /
// (D/4)): every load of its rows is issued before any arithmetic, and its quad
// of the weighted corrections e^{G_a - G_j} u_j stays in registers; the
// accepted K rows sit in shared memory.
#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int NT = 256;
constexpr int MAXTOK = 16;
constexpr int NPART = 8;  // blocks per (sequence, V head), each a slice of the state rows

template <int D>
__global__ void __launch_bounds__(NT) commit_kernel(Args a, int32_t *err) {
    constexpr int Q4 = D / 4;              // column quads per row
    constexpr int RSTEP = NT / Q4;         // rows between a thread's rows
    constexpr int ROWS = D / NPART;       // rows per block
    constexpr int NR = ROWS / RSTEP;       // rows per thread (0 when RSTEP > ROWS, D < 128: see below)
    static_assert(D % NPART == 0, "row slices");
    __shared__ float sK[MAXTOK][ROWS];     // the block's rows of k_j for the accepted tokens, fp32
    __shared__ float sW[MAXTOK];           // e^{G_a - G_j} (times 1 / |k_j| with the fused L2 norm)
    __shared__ float sEa;                  // e^{G_a}

    const int part = blockIdx.x % NPART;
    const int h = (blockIdx.x / NPART) % a.h_v, s = blockIdx.x / (NPART * a.h_v);
    const int hq = h / (a.h_v / a.h_qk);
    const int n_tok = a.fixed_len;
    // every load is issued before the accepted count is known: the block's rows of
    // the snapshot, all n_tok corrections, k rows and gates (the count only masks them)
    const int acc_in = a.accepted[s];
    const int rbase = part * ROWS;
    const size_t row0 = (size_t)s * n_tok;  // the block's first token row of this sequence
    const int cq = threadIdx.x % Q4, r0 = threadIdx.x / Q4;
    const size_t sbase = ((size_t)s * a.h_v + h) * D * D;
    const float4 *src = reinterpret_cast<const float4 *>(a.snapshot_in + sbase);
    float4 *dst = reinterpret_cast<float4 *>(a.state + sbase);
    constexpr int NRT = NR > 0 ? NR : 1;
    float4 x[NRT];
#pragma unroll
    for (int k = 0; k < NRT; ++k) {
        const int r = rbase + r0 + k * RSTEP;
        x[k] = (r0 + k * RSTEP < ROWS) ? src[r * Q4 + cq] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 u[MAXTOK];
#pragma unroll
    for (int j = 0; j < MAXTOK; ++j) {
        u[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < n_tok) u[j] = *reinterpret_cast<const float4 *>(a.deltas + ((row0 + j) * a.h_v + h) * D + 4 * cq);
    }
    float graw = 0.f;
    if (threadIdx.x < 32 && threadIdx.x < n_tok) graw = a.g[(row0 + threadIdx.x) * a.h_v + h];
    for (int e = threadIdx.x; e < n_tok * ROWS; e += NT) {
        const int j = e / ROWS, i = e - j * ROWS;
        sK[j][i] = load_in(a.k, ((row0 + j) * a.h_qk + hq) * D + rbase + i, a.in_bf16);
    }
    if (acc_in < 0 || acc_in > n_tok) {  // leave the state as it is and report
        if (threadIdx.x == 0 && part == 0) atomicCAS(err, 0, (int32_t)GDR_ERR_INVALID_ARG);
        return;
    }
    const int acc = acc_in;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float gj = lane < acc ? graw : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, gj, o);
            if (lane >= o) gj += t;
        }
        const float Ga = __shfl_sync(0xffffffffu, gj, acc > 0 ? acc - 1 : 0);
        if (lane < MAXTOK) sW[lane] = (lane < acc) ? __expf(Ga - gj) : 0.f;  // exponent <= 0 for g <= 0
        if (lane == 0) sEa = acc > 0 ? __expf(Ga) : 1.f;
    }
    __syncthreads();
    if (a.qk_norm) {
        // fused L2 normalisation: k_j u_j^T uses k_j / |k_j|; the whole row's norm
        // folds into the token's weight (warp w takes tokens w, w + 8)
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int j = warp; j < acc; j += NT / 32) {
            float ss = 0.f;
            for (int i = lane; i < D; i += 32) {
                const float x = load_in(a.k, ((row0 + j) * a.h_qk + hq) * D + i, a.in_bf16);
                ss = fmaf(x, x, ss);
            }
            ss = warp_sum(ss);
            if (lane == 0) sW[j] *= l2norm_scale(ss);
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < MAXTOK; ++j) {
        const float w = sW[j];
        u[j] = make_float4(w * u[j].x, w * u[j].y, w * u[j].z, w * u[j].w);
    }
    const float ea = sEa;
#pragma unroll
    for (int k = 0; k < NRT; ++k) {
        const int rl = r0 + k * RSTEP;  // row within the block's slice
        if (rl >= ROWS) continue;
        float4 y = make_float4(ea * x[k].x, ea * x[k].y, ea * x[k].z, ea * x[k].w);
#pragma unroll
        for (int j = 0; j < MAXTOK; ++j) {
            if (j < acc) {
                const float kr = sK[j][rl];
                y.x = fmaf(kr, u[j].x, y.x);
                y.y = fmaf(kr, u[j].y, y.y);
                y.z = fmaf(kr, u[j].z, y.z);
                y.w = fmaf(kr, u[j].w, y.w);
            }
        }
        dst[(rbase + rl) * Q4 + cq] = y;
    }
}

}  // namespace

cudaError_t launch_commit(const Args &a, int32_t *err, cudaStream_t s) {
    if (a.n_seqs == 0) return cudaSuccess;
    if (a.fixed_len < 0 || a.fixed_len > MAXTOK || !err) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)a.n_seqs * (unsigned)a.h_v * (unsigned)NPART;
    switch (a.d) {
        case 32: commit_kernel<32><<<blocks, NT, 0, s>>>(a, err); break;
        case 64: commit_kernel<64><<<blocks, NT, 0, s>>>(a, err); break;
        case 128: commit_kernel<128><<<blocks, NT, 0, s>>>(a, err); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdr
