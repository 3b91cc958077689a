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

// 16-byte asynchronous copy global -> shared (both 16-byte aligned); all of a
// thread's copies are in flight until cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Every segment's start, for one (sequence, V head) and 16 state columns per
// block: X_{p+1} = Phi_p X_p + B_p for p = 1 .. P-1 in order.  The columns are
// independent (X_{p+1}'s columns depend only on the same columns of X_p), so each
// block walks all steps for its 16 columns with X in shared memory; Phi_{p+1}
// is copied in (asynchronously, rows padded to 132 floats) while step p
// computes.  X_1 is the state segment 0 left in `state`: it is saved to
// xseg[0]; X_p goes to xseg[p-1], and the last, X_P, back to `state`.
constexpr int CMB_COLS = 16, PHI_LD = D + 4;
constexpr int CMB_SMEM = (2 * D * PHI_LD + 2 * D * CMB_COLS) * (int)sizeof(float);
struct CombineParams {
    int P;
    size_t seg_stride;  // floats between one segment's matrices and the next's
    const float *phi, *b;
    float *state, *xseg;
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
    const int r = tid >> 1, cc = (tid & 1) * 8;  // row r, 8 of the 16 columns
    for (int p = 1; p < c.P; ++p) {
        const int cur = (p - 1) & 1;
        if (p + 1 < c.P) {
            load_phi(p + 1, ph(cur ^ 1));
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // Phi_p has landed
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();  // Phi_p and X_p visible to every thread
        const float *bb = c.b + (size_t)(p - 1) * c.seg_stride + mat + (size_t)r * D + c0 + cc;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; j += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(bb + j);
            acc[j] = v.x;
            acc[j + 1] = v.y;
            acc[j + 2] = v.z;
            acc[j + 3] = v.w;
        }
        const float *pr = ph(cur) + r * PHI_LD;
        const float *xin = xs(cur);
#pragma unroll 4
        for (int k4 = 0; k4 < D / 4; ++k4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(pr + 4 * k4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 x0 = *reinterpret_cast<const float4 *>(xin + (4 * k4 + kk) * CMB_COLS + cc);
                const float4 x1 = *reinterpret_cast<const float4 *>(xin + (4 * k4 + kk) * CMB_COLS + cc + 4);
                acc[0] = fmaf(av[kk], x0.x, acc[0]);
                acc[1] = fmaf(av[kk], x0.y, acc[1]);
                acc[2] = fmaf(av[kk], x0.z, acc[2]);
                acc[3] = fmaf(av[kk], x0.w, acc[3]);
                acc[4] = fmaf(av[kk], x1.x, acc[4]);
                acc[5] = fmaf(av[kk], x1.y, acc[5]);
                acc[6] = fmaf(av[kk], x1.z, acc[6]);
                acc[7] = fmaf(av[kk], x1.w, acc[7]);
            }
        }
        // X_{p+1}: to shared memory for the next step, and to xseg[p] (or the state)
        float *xo = xs(cur ^ 1) + r * CMB_COLS + cc;
        *reinterpret_cast<float4 *>(xo) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(xo + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        float *g = (p == c.P - 1 ? c.state : c.xseg + (size_t)p * c.seg_stride) + mat + (size_t)r * D + c0 + cc;
        *reinterpret_cast<float4 *>(g) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(g + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        __syncthreads();  // every thread is done with Phi_p and X_p before they are overwritten
    }
}

// o_t = o0_t + X_p^T m_t for the tokens of segments >= 1.  A block covers one
// chunk (64 tokens, one segment) of one sequence and one V head: the 64 x 128
// tile of (64 x 128) m times (128 x 128) X_p.  Both operands are staged in
// shared memory by asynchronous copies (m's rows padded to 132 floats); each of
// the 128 threads keeps an 8-token x 8-column tile of the result in registers
// and walks the 128 terms four at a time.
struct FixParams {
    int h_v, n_seqs, P, out_bf16;
    int cuts[9];  // chunk cuts: segment p is chunks [cuts[p], cuts[p+1])
    const int32_t *cu_seqlens;
    const float *xseg;  // X[p-1] = start of segment p, [n_seqs][h_v][d][d]
    const float *o0, *m;
    void *o;
};

constexpr int FIX_TOK = 64, M_LD = D + 4, X_LD = D + 4;
constexpr int FIX_SMEM = (FIX_TOK * M_LD + D * X_LD) * (int)sizeof(float);

// bf16 hi and lo words of the pair (x0, x1): hi = the top 16 bits of each, lo =
// bf16(x - hi); x0 in the low half.
__device__ __forceinline__ void hilo2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t a = __float_as_uint(x0), b = __float_as_uint(x1);
    hi = __byte_perm(a, b, 0x7632);
    __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(a & 0xFFFF0000u), x1 - __uint_as_float(b & 0xFFFF0000u));
    lo = *reinterpret_cast<uint32_t *>(&l);
}
// d += A B for one 16 x 8 tile (m16n8k16, bf16 operands, fp32 accumulation;
// lane = 4 g + c holds rows g, g + 8 and columns 2c, 2c + 1 of d).
__device__ __forceinline__ void mma_bf16x(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One block per (64-token chunk of a later segment, sequence x V head): the
// chunk's maps m (64 x d_k) and its segment's start state X (d_k x d_v) staged in
// shared memory by cp.async, then O = o0 + M X on warp-level bf16 tensor-core
// MMAs, each fp32 operand split into bf16 hi + lo parts and three products
// (hi hi + hi lo + lo hi) accumulated in fp32: 2^-16 relative precision, as the
// chunk scan's state products.  Warp w takes tokens 32 (w & 1) .. + 31 and
// columns 64 (w >> 1) .. + 63.
__global__ void __launch_bounds__(128, 2) fixup_kernel(FixParams p) {
    extern __shared__ __align__(16) float fsm[];
    float *ms = fsm;                    // [FIX_TOK][M_LD]
    float *xs = fsm + FIX_TOK * M_LD;   // [D][X_LD]
    const int c = p.cuts[1] + (int)blockIdx.x;      // chunk index within the sequence
    const int s = (int)blockIdx.y / p.h_v, h = (int)blockIdx.y % p.h_v;
    int seg = 1;  // the segment of chunk c (static indices: the cuts stay in the parameter space)
#pragma unroll
    for (int q = 2; q < 9; ++q)
        if (q < p.P && c >= p.cuts[q]) seg = q;
    const int64_t ts = p.cu_seqlens[s], te = p.cu_seqlens[s + 1];
    const int64_t t0 = ts + (int64_t)c * 64;
    if (t0 >= te) return;  // past this sequence's end (or an empty sequence)
    const int ntok = (int)((te - t0) < FIX_TOK ? (te - t0) : FIX_TOK);
    const float *X = p.xseg + (((size_t)(seg - 1) * p.n_seqs + s) * p.h_v + h) * D * D;
    const int tid = threadIdx.x;
#pragma unroll 4
    for (int i = tid; i < D * D / 4; i += 128) {
        const int r = i / (D / 4), q4 = i % (D / 4);
        cp_async16(xs + r * X_LD + 4 * q4, X + (size_t)r * D + 4 * q4);
    }
#pragma unroll 4
    for (int i = tid; i < FIX_TOK * (D / 4); i += 128) {
        const int t = i / (D / 4), q4 = i % (D / 4);
        if (t < ntok)
            cp_async16(ms + t * M_LD + 4 * q4, p.m + ((size_t)(t0 + t) * p.h_v + h) * D + 4 * q4);
        else
            *reinterpret_cast<float4 *>(ms + t * M_LD + 4 * q4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    cp_async_wait_all();
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, cc = lane & 3;
    const int tb = 32 * (warp & 1), nb = 64 * (warp >> 1);
    float acc[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll 1
    for (int k0 = 0; k0 < D; k0 += 16) {
        uint32_t ah[2][4], al[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const float *mr = ms + (tb + 16 * mt + g) * M_LD + k0 + 2 * cc;
            const float2 v0 = *reinterpret_cast<const float2 *>(mr);
            const float2 v1 = *reinterpret_cast<const float2 *>(mr + 8 * M_LD);
            const float2 v2 = *reinterpret_cast<const float2 *>(mr + 8);
            const float2 v3 = *reinterpret_cast<const float2 *>(mr + 8 * M_LD + 8);
            hilo2(v0.x, v0.y, ah[mt][0], al[mt][0]);
            hilo2(v1.x, v1.y, ah[mt][1], al[mt][1]);
            hilo2(v2.x, v2.y, ah[mt][2], al[mt][2]);
            hilo2(v3.x, v3.y, ah[mt][3], al[mt][3]);
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float *xr = xs + (k0 + 2 * cc) * X_LD + nb + 8 * nt + g;
            uint32_t b0h, b0l, b1h, b1l;
            hilo2(xr[0], xr[X_LD], b0h, b0l);
            hilo2(xr[8 * X_LD], xr[9 * X_LD], b1h, b1l);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                mma_bf16x(acc[mt][nt], ah[mt], b0h, b1h);
                mma_bf16x(acc[mt][nt], ah[mt], b0l, b1l);
                mma_bf16x(acc[mt][nt], al[mt], b0h, b1h);
            }
        }
    }
    // o = o0 + acc: rows tb + 16 mt + g (+ 8), columns nb + 8 nt + 2 cc (+ 1)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int t = tb + 16 * mt + g + 8 * hh;
            if (t >= ntok) continue;
            const size_t orow = ((size_t)(t0 + t) * p.h_v + h) * D;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int col = nb + 8 * nt + 2 * cc;
                const float2 b = *reinterpret_cast<const float2 *>(p.o0 + orow + col);
                const float y0 = b.x + acc[mt][nt][2 * hh], y1 = b.y + acc[mt][nt][2 * hh + 1];
                if (p.out_bf16) {
                    __nv_bfloat162 v = __floats2bfloat162_rn(y0, y1);
                    *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + orow + col) = v;
                } else {
                    *reinterpret_cast<float2 *>(reinterpret_cast<float *>(p.o) + orow + col) = make_float2(y0, y1);
                }
            }
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
    fp.xseg = xseg;
    fp.o0 = o0;
    fp.m = m;
    fp.o = a.o;
    const int fix_chunks = (int)(n_ch - fp.cuts[1]);
    if (fix_chunks <= 0) return cudaSuccess;
    fixup_kernel<<<dim3((unsigned)fix_chunks, (unsigned)per_seg), 128, FIX_SMEM, s>>>(fp);
    return cudaGetLastError();
}

}  // namespace gdr
