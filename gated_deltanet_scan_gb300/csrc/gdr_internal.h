// Internal launch interface shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdr.h"

namespace gdr {

// Everything one launch needs, already validated on the host.
struct Args {
    int h_qk, h_v, d;        // d = d_k = d_v
    int in_bf16, out_bf16;   // 1 when the tensor is bf16, 0 for fp32
    float scale;
    int qk_norm;             // GDR_FLAG_QK_L2NORM: rows of q and k scaled by 1 / sqrt(sum x^2 + 1e-6)
    int beta_logits;         // GDR_FLAG_BETA_LOGITS: beta = sigmoid(beta input)
    // gated RMSNorm of the outputs (decode epilogue): when norm_z is set, o receives
    // y = w * o / sqrt(mean(o^2) + norm_eps) * silu(z) instead of o
    const void *norm_z;      // [rows][H_v][d_v], in_dtype
    const float *norm_w;     // [d_v]
    float norm_eps;
    int n_seqs;
    const int32_t *cu_seqlens;  // device; nullptr => sequence s is [s*fixed_len, (s+1)*fixed_len)
    int fixed_len;
    int64_t t_total;
    const void *q, *k, *v;
    const float *g, *beta;
    float *state;
    float *snapshot;  // optional copy of the incoming state (verify block)
    void *o;
    float *deltas;              // optional per-token corrections u_t (verify block), fp32 like v
    const int32_t *accepted;    // verify commit: accepted tokens per sequence (device)
    const float *snapshot_in;   // verify commit: the state before the block
    // tensor-core prefill: only chunks [c_lo, c_hi) of each sequence (0, INT32_MAX: all of them)
    int c_lo, c_hi;
};

// `overlap`: launch as a programmatic dependent of the kernel before it on `s`.
cudaError_t launch_decode(const Args &a, int32_t *err, cudaStream_t s, bool overlap);
cudaError_t launch_chunk_cc(const Args &a, cudaStream_t s);
// The verify block on tensor cores (gdr_verify.cu): bf16 inputs, 1 <= fixed_len <= 16 tokens.
cudaError_t launch_verify(const Args &a, cudaStream_t s);
// Tensor-core prefill in two launches: the per-chunk factors of every chunk
// into `ws` (fac::n_slots(t_total, n_seqs) * h_v slots), then the chunk scan.
// `overlap`: launch as a programmatic dependent of the kernel before it on `s`
// (it may start once every CTA of that kernel runs; it must not read its results).
cudaError_t launch_factors(const Args &a, float *ws, int32_t *err, cudaStream_t s, bool overlap);
// `overlap`: launch as a programmatic dependent of the factor launch just before
// it on `s` (its prologue overlaps that grid; it reads the workspace only after
// griddepcontrol.wait).  Only directly after the factor launch whose slots it
// reads: the kernel waits for nothing else.
// `dec` (optional): one decode step of another batch (dec->n_seqs sequences, one
// token each, dims as `a`) carried by `dec_blocks` extra blocks of the same
// launch, on the SMs the scan leaves free.
cudaError_t launch_prefill_tc(const Args &a, const float *ws, cudaStream_t s, bool overlap, const Args *dec = nullptr,
                              int dec_blocks = 0);

// One run of the chunk scan: chunks [c_lo, c_hi) of every sequence from and into
// `state` ([n_seqs][h_v][128][128] fp32), outputs to `o` (bf16 when out_bf16),
// values taken as zero when v_zero.  The tensor-core launch below walks up to
// kMaxTcRuns runs side by side; every run reads the same factor workspace.
constexpr int kMaxTcRuns = 16;
struct TcRun {
    int c_lo, c_hi;
    int out_bf16, v_zero;
    float *state;
    void *o;
};
cudaError_t launch_prefill_tc_runs(const Args &a, const TcRun *runs, int n_runs, const float *ws, cudaStream_t s,
                                   bool overlap,
                                   const Args *dec = nullptr, int dec_blocks = 0);
cudaError_t launch_copy_f32(const float *src, float *dst, size_t n, cudaStream_t s);
// y = w * o / sqrt(mean(o^2) + eps) * silu(z) for `rows` rows of d values (gdr_norm.cu).
cudaError_t launch_gated_rmsnorm(int64_t rows, int d, const void *o, int o_bf16, const void *z, int z_bf16,
                                 const float *w, float eps, void *y, int y_bf16, cudaStream_t s);

// Two-level prefill (gdr_segment.cu): byte offsets of its fp32 scratch inside the
// workspace, after the factor_bytes of the factor slots and X tiles.
struct SegLayout {
    size_t phi, b, x, xt, o0, m, total;
};
SegLayout segment_layout(int64_t factor_bytes, int n_seqs, int h_v, int64_t t_total, int P);
// First chunk of segment p of P over n_chunks chunks (p = P gives n_chunks).
int segment_cut(int64_t n_chunks, int P, int p);
// Factors, one scan launch over every segment's runs, the combine of the segment
// starts and the later segments' outputs, all on `s`; `ws` holds L.total bytes.
cudaError_t launch_segmented(const Args &a, int P, uint8_t *ws, const SegLayout &L, int32_t *err, cudaStream_t s);
// Verify commit: state = e^{G_a} snapshot + sum_{j<a} e^{G_a - G_j} k_j u_j^T per (sequence, V head).
cudaError_t launch_commit(const Args &a, int32_t *err, cudaStream_t s);

// bf16 tensor [d2][d1][d0] (d0 contiguous) as a TMA map with box {box0, 1, 64}.
bool encode_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                    CUtensorMapSwizzle swizzle);

// Device address of the error word (nullptr if it cannot be resolved).
int32_t *device_error_word();

// Synchronises `s`, then reads and clears the device error word.
cudaError_t read_clear_device_error(cudaStream_t s, int32_t *code);

}  // namespace gdr
