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
// Scratch (fp32, inside the caller's workspace, after the factor slots):
//   Phi[P-1], B[P-1], X[P-1]  [n_seqs][h_v][d][d]   (X[j] = start of segment j+1)
//   O0, M                     [t_total][h_v][d]     (rows of segments >= 1 only)
#include <cuda_bf16.h>

#include "gdr_factor_layout.h"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int D = 128;

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

// out = phi * in + b for one (sequence, V head) and 32 columns per block; with
// `save`, `in` is also copied there.  `in` and `out` may be the same array: a
// block reads its 32 columns of `in` completely before writing them.
constexpr int CMB_COLS = 32;
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ phi, const float *__restrict__ b,
                                                      const float *in, float *out, float *save) {
    __shared__ float xs[D][CMB_COLS];
    const size_t mat = (size_t)blockIdx.x * D * D;
    const int c0 = blockIdx.y * CMB_COLS;
    const int tid = threadIdx.x;
    for (int i = tid; i < D * CMB_COLS; i += 256) {
        const int r = i / CMB_COLS, c = i % CMB_COLS;
        const float x = in[mat + (size_t)r * D + c0 + c];
        xs[r][c] = x;
        if (save) save[mat + (size_t)r * D + c0 + c] = x;
    }
    __syncthreads();
    // thread: row r, 16 of the 32 columns
    const int r = tid >> 1, cc = (tid & 1) * 16;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = b[mat + (size_t)r * D + c0 + cc + j];
    const float *pr = phi + mat + (size_t)r * D;
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
        const float a = __ldg(pr + k);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = fmaf(a, xs[k][cc + j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) out[mat + (size_t)r * D + c0 + cc + j] = acc[j];
}

// o_t = o0_t + X_p^T m_t for the tokens of segments >= 1.  A block covers 32
// tokens of one chunk (one segment) of one sequence, one V head and 64 of the
// output columns; X_p's 64 columns and the 32 rows of m sit in shared memory.
struct FixParams {
    int h_v, n_seqs, P, out_bf16;
    int cuts[9];  // chunk cuts: segment p is chunks [cuts[p], cuts[p+1])
    const int32_t *cu_seqlens;
    const float *xseg;  // X[p-1] = start of segment p, [n_seqs][h_v][d][d]
    const float *o0, *m;
    void *o;
};

constexpr int FIX_TOK = 32, FIX_COLS = 64;
__global__ void __launch_bounds__(256) fixup_kernel(FixParams p) {
    extern __shared__ float fsm[];
    float *xs = fsm;                    // [D][FIX_COLS]
    float *ms = fsm + D * FIX_COLS;     // [FIX_TOK][D]
    const int c = p.cuts[1] + (int)blockIdx.x / 2;     // chunk index within the sequence
    const int sub = (int)blockIdx.x % 2;               // which 32 tokens of the chunk
    const int s = (int)blockIdx.y / p.h_v, h = (int)blockIdx.y % p.h_v;
    const int col0 = (int)blockIdx.z * FIX_COLS;
    int seg = 1;
    while (seg + 1 < p.P && c >= p.cuts[seg + 1]) ++seg;
    const int64_t ts = p.cu_seqlens[s], te = p.cu_seqlens[s + 1];
    const int64_t t0 = ts + (int64_t)c * 64 + FIX_TOK * sub;
    if (t0 >= te) return;  // past this sequence's end (or an empty sequence)
    const int ntok = (int)((te - t0) < FIX_TOK ? (te - t0) : FIX_TOK);
    const float *X = p.xseg + (((size_t)(seg - 1) * p.n_seqs + s) * p.h_v + h) * D * D;
    const int tid = threadIdx.x;
    for (int i = tid; i < D * FIX_COLS / 4; i += 256) {
        const int r = i / (FIX_COLS / 4), q4 = i % (FIX_COLS / 4);
        reinterpret_cast<float4 *>(xs)[i] = *reinterpret_cast<const float4 *>(X + (size_t)r * D + col0 + 4 * q4);
    }
    for (int i = tid; i < FIX_TOK * D / 4; i += 256) {
        const int tr = i / (D / 4), q4 = i % (D / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tr < ntok) v = *reinterpret_cast<const float4 *>(p.m + ((size_t)(t0 + tr) * p.h_v + h) * D + 4 * q4);
        reinterpret_cast<float4 *>(ms)[i] = v;
    }
    __syncthreads();
    // thread: token row tr, 8 consecutive columns
    const int tr = tid >> 3, cc = (tid & 7) * 8;
    if (tr >= ntok) return;
    const size_t orow = ((size_t)(t0 + tr) * p.h_v + h) * D + col0 + cc;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = p.o0[orow + j];
    const float *mr = ms + tr * D;
#pragma unroll 4
    for (int i = 0; i < D; ++i) {
        const float mi = mr[i];
        const float *xr = xs + i * FIX_COLS + cc;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(mi, xr[j], acc[j]);
    }
    if (p.out_bf16) {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.o) + orow;
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = __float2bfloat16_rn(acc[j]);
    } else {
        float *dst = reinterpret_cast<float *>(p.o) + orow;
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = acc[j];
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
    L.o0 = L.x + align256(mats);
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
    const size_t per_seg = (size_t)a.n_seqs * a.h_v;  // matrices per segment
    const size_t mat_floats = (size_t)D * D;
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
    // 4. segment starts, in order: X_1 is the state segment 0 left in `state`
    for (int p = 1; p < P; ++p) {
        const float *in = p == 1 ? a.state : xseg + (size_t)(p - 1) * per_seg * mat_floats;
        float *out = p == P - 1 ? a.state : xseg + (size_t)p * per_seg * mat_floats;
        float *save = p == 1 ? xseg : nullptr;
        combine_kernel<<<dim3((unsigned)per_seg, D / CMB_COLS), 256, 0, s>>>(
            phi + (size_t)(p - 1) * per_seg * mat_floats, bb + (size_t)(p - 1) * per_seg * mat_floats, in, out,
            save);
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
    fp.xseg = xseg;
    fp.o0 = o0;
    fp.m = m;
    fp.o = a.o;
    const int fix_chunks = (int)(n_ch - fp.cuts[1]);
    if (fix_chunks <= 0) return cudaSuccess;
    const int smem = (D * FIX_COLS + FIX_TOK * D) * (int)sizeof(float);
    static int configured_device = -1;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    fixup_kernel<<<dim3((unsigned)fix_chunks * 2, (unsigned)per_seg, D / FIX_COLS), 256, smem, s>>>(fp);
    return cudaGetLastError();
}

}  // namespace gdr
