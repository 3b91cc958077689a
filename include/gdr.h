/*
 * gdr.h -- C ABI of the gated delta rule library (sm_103a, one GPU).
 *
 * The method.  For every sequence and V head h the library runs
 *
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   o_t = scale * S_t^T q_t
 *
 * ("Qwen3.5-9B: Giai ma kien truc Gated DeltaNet", section "Gated DeltaNet";
 * step order as in the per-token Loop of the Qwen3.5-9B NPU model card,
 * section "How it works": decay, recall S^T k, delta correction, read-out).
 * The gate is passed as g_t = log(alpha_t) <= 0 (a decay; the Candle PR's
 * "Bug 1" records that the raw value is already negative).  Each QK head feeds
 * H_v / H_qk consecutive V heads: V head h reads q and k from QK head
 * h / (H_v / H_qk) (for Qwen3.5-9B, 16 QK heads each shared by 2 of 32 V heads).
 *
 * Conventions for every entry point
 *   - Memory.  Every tensor pointer is a DEVICE pointer allocated by the caller;
 *     the library allocates nothing and keeps no pointer after the call returns.
 *     Pointers must be 16-byte aligned.  Scratch memory, where a path needs
 *     it, is passed in by the caller (see gdr_prefill_workspace_bytes).
 *   - Layouts (row-major, token-major, sequences packed back to back):
 *         q, k   [T_total][H_qk][d_k]        in_dtype  (bf16 or fp32)
 *         v      [T_total][H_v][d_v]         in_dtype
 *         o      [T_total][H_v][d_v]         out_dtype (fp32 or bf16)
 *         g, beta[T_total][H_v]              fp32  (g = log alpha)
 *         state  [n_seqs][H_v][d_k][d_v]     fp32, d_v contiguous
 *   - Ordering.  Calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and ordered like any other work on that stream.
 *   - Errors.  Arguments are checked on the host before anything is launched:
 *     GDR_ERR_INVALID_ARG (null or misaligned pointer, bad count, H_v not a
 *     multiple of H_qk, verify longer than 16 tokens, ...) or GDR_ERR_UNSUPPORTED
 *     (a head size, chunk or dtype with no compiled kernel).  GDR_ERR_CUDA means
 *     a launch failed.  Kernels that wait on asynchronous copies give up after a
 *     bounded number of polls and record GDR_ERR_DEVICE_TIMEOUT in a device
 *     error word that gdr_device_error() reads; they never spin forever.
 *   - Aliasing.  `state` is updated in place.  `o` must not overlap any input.
 *
 * Supported shapes: d_k == d_v in {32, 64, 128}; chunk in {16, 64}; any H_qk,
 * H_v with H_v % H_qk == 0.  The chunk is a tiling choice, not part of the
 * result: d_k = d_v = 128 with bf16 inputs and chunk 64 runs the tensor-core
 * (tcgen05) prefill, which needs a caller-provided workspace
 * (gdr_prefill_workspace_bytes); every other shape runs the CUDA-core chunk
 * kernel with 16-token chunks and needs none.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDR_ABI_VERSION 9

/* Same object as cudaStream_t; declared here so callers need no CUDA header. */
typedef struct CUstream_st *gdr_stream_t;

typedef enum gdr_status {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = 1,
    GDR_ERR_UNSUPPORTED = 2,
    GDR_ERR_CUDA = 3,
    GDR_ERR_DEVICE_TIMEOUT = 4
} gdr_status;

typedef enum gdr_dtype { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;

typedef struct gdr_dims {
    int32_t h_qk;      /* QK heads */
    int32_t h_v;       /* V heads; a multiple of h_qk */
    int32_t d_k;       /* key/query head size */
    int32_t d_v;       /* value head size (== d_k) */
    int32_t chunk;     /* 16 or 64 tokens per chunk */
    int32_t in_dtype;  /* gdr_dtype of q, k, v */
    int32_t out_dtype; /* gdr_dtype of o */
    float scale;       /* multiplies every output; 1.0 reproduces o_t = S_t^T q_t */
    int32_t flags;     /* GDR_FLAG_* below, or 0 */
} gdr_dims;

/*
 * Steps on either side of the rule, fused into every kernel (gdr_dims.flags):
 *   GDR_FLAG_QK_L2NORM    q and k are passed raw; every (token, QK head) row x is
 *                         used as x / sqrt(sum_i x_i^2 + 1e-6).  The workloads of
 *                         the pages feed L2-normalised q and k to the rule; the
 *                         pages give no epsilon for it (1e-6 inside the square
 *                         root is this library's reading).  The kernels apply it
 *                         as per-row scales of the exact bf16/fp32 products, in
 *                         fp32, so the normalised values are never rounded to the
 *                         input type.
 *   GDR_FLAG_BETA_LOGITS  beta holds logits b; the rule uses beta = 1 / (1 + exp(-b))
 *                         (the workloads draw beta = sigmoid(N(0, 1))).
 * The gated RMSNorm after the rule is gdr_gated_rmsnorm (and is fused into
 * gdr_decode_step_gated).  No flag changes a layout or a size.
 */
#define GDR_FLAG_QK_L2NORM 1
#define GDR_FLAG_BETA_LOGITS 2

/* GDR_ABI_VERSION of the loaded library. */
int32_t gdr_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *gdr_status_string(gdr_status status);

/*
 * Bytes of device workspace gdr_prefill_chunked needs for this problem: 0 when
 * the CUDA-core path runs (or for an empty problem), otherwise, for each of
 * P = ceil(t_total / 64) + n_seqs chunk positions, one 17,152-byte slot of
 * per-chunk factors per V head (T and P T as an fp16 MMA operand tile, the
 * chunk's exp(G), and room for the row scales of the fused q/k L2 norm), then, from the next 1 KiB boundary, one 16 KiB fp16 tile
 * per QK head of X = [K; Q]_c K_{c-1}^T (the next chunk's keys and queries
 * against this chunk's keys), rounded up to 256 bytes:
 * roundup(roundup(P * h_v * 17152, 1024) + P * h_qk * 16384, 256).
 * Host-only, never fails (invalid dims: 0).
 */
size_t gdr_prefill_workspace_bytes(const gdr_dims *dims, int32_t n_seqs, int64_t t_total);

/*
 * Chunked prefill over packed variable-length sequences.
 *
 * Computes, for every sequence s in [0, n_seqs) with tokens
 * [cu_seqlens[s], cu_seqlens[s+1]) and every V head, the outputs o_t of all its
 * tokens and the state after its last token, starting from state[s] (S0).
 * It uses the chunkwise-parallel form of the Qwen3.5-9B NPU model card
 * ("How it works": N, D = (I+N)^-1 diag(beta)(V - diag(e^G) K S0), O and S_T
 * with G the running sum of g inside a chunk), solving the unit lower
 * triangular system by forward substitution as in the Candle PR's
 * "Chunked GatedDeltaNet Scan" section, carrying the state from chunk to
 * chunk, and masking the upper triangle of G_t - G_j in log space before exp
 * (the PR's "Float32 overflow fix").  Chunks start at each sequence start; a
 * tail chunk is treated as padded with g = 0, beta = 0 rows (the model card's
 * token_valid padding), which leaves the state as after the last real token;
 * padded rows are never written.
 *
 * On the tensor-core path the call is two launches on `stream`: the
 * state-independent factors of every chunk (gates, (I+N)^-1, P (I+N)^-1, and
 * X = [K; Q]_c K_{c-1}^T) into `workspace`, then the chunk-to-chunk scan that
 * reads them.  When the scan leaves at least 16 SMs free and the factors of all
 * chunks need at least two waves of the GPU (e.g. one Qwen3.5-9B sequence of
 * 2.5K tokens or more), the call is four launches instead: factors and scan of
 * the first ~73% of the chunks, the remaining factors as a programmatic
 * dependent launch that runs on the free SMs beside that scan, then the scan of
 * the remaining chunks.  The workspace holds nothing between calls.
 *
 *   dims        shapes, dtypes, chunk, scale (host pointer, read during the call)
 *   n_seqs      number of sequences (>= 0; 0 is a no-op)
 *   cu_seqlens  DEVICE int32 [n_seqs + 1], non-decreasing, cu_seqlens[0] == 0,
 *               cu_seqlens[n_seqs] == t_total (empty sequences allowed: their
 *               state is left unchanged).  Entries outside [0, t_total] make
 *               the kernels skip those sequences and record
 *               GDR_ERR_INVALID_ARG in the device error word.
 *   t_total     total tokens (host value, sizes the launch)
 *   q, k, v, g, beta   inputs (layouts above)
 *   state       in: S0 per sequence; out: state after the last token
 *   o           out: outputs of every token
 *   workspace   DEVICE scratch of at least gdr_prefill_workspace_bytes(dims,
 *               n_seqs, t_total) bytes, 16-byte aligned, owned by the caller,
 *               not overlapping any other argument, not used by other work on
 *               other streams until this call's work on `stream` is done.  May
 *               be NULL when that size is 0.  Too small or misaligned:
 *               GDR_ERR_INVALID_ARG before anything is launched.
 *
 * Precision on the tensor-core path: the state is carried in fp32 and every
 * state-sized product keeps ~2^-16 relative precision (bf16 hi/lo operand
 * splits); the chunk-sized products with the factors (the correction D, the
 * intra-chunk output part and X D~) take fp16 operands with fp32
 * accumulation.  Their data-scaled operands (V - e^G K S and the correction D)
 * are multiplied by a power of two chosen per scan CTA from its first chunk's
 * values and its initial state (largest magnitude brought to [8, 16)), so the
 * result's relative accuracy does not depend on the data's scale (tested from
 * 2^-20 to 2^16 times unit-RMS values).  Data that grows by more than ~4000x
 * over a sequence beyond its first chunk and initial state would approach the
 * fp16 maximum.
 */
gdr_status gdr_prefill_chunked(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens,
                               int64_t t_total, const void *q, const void *k, const void *v,
                               const float *g, const float *beta, float *state, void *o,
                               void *workspace, size_t workspace_bytes, gdr_stream_t stream);

/*
 * gdr_prefill_chunked without a caller workspace and without any allocation:
 * the scratch is one fixed device array inside the library (its size is
 * gdr_prefill_static_workspace_capacity(), 64 MiB), whose device address is
 * looked up on every call.  Problems whose gdr_prefill_workspace_bytes()
 * exceed it return GDR_ERR_UNSUPPORTED before anything is launched.  With
 * Qwen3.5-9B heads (16 QK, 32 V) one chunk position takes 811,008 bytes, so
 * the array holds 82 positions: one sequence of up to 5,184 tokens, and one
 * position less per further sequence (two sequences: 5,120 tokens in all;
 * eight: 4,736).  All calls on a device share that array, so calls on
 * different streams must not overlap (order them on one stream, or
 * synchronise); everything else, arguments and results, is as in
 * gdr_prefill_chunked.
 */
gdr_status gdr_prefill_chunked_static(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens,
                                      int64_t t_total, const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float *state, void *o,
                                      gdr_stream_t stream);

/* Bytes of the fixed scratch array used by gdr_prefill_chunked_static. */
size_t gdr_prefill_static_workspace_capacity(void);

/*
 * Two-level (segment-parallel) prefill: the same result as gdr_prefill_chunked,
 * for problems with few (sequence, V head) pairs and long sequences, where one
 * chain of chunks per head would leave most of the GPU idle.
 *
 * The chunks of every sequence are cut into n_segments consecutive segments
 * (segment p: chunks [floor(n p / P), floor(n (p+1) / P)) of the
 * n = ceil(t_total / 64) chunk positions; a sequence shorter than that has only
 * its first segments).  Over a segment the recurrence is affine in the state it
 * starts from, X: the state after it is Phi X + B and each output
 * o_t = o0_t + X^T m_t, which follows from the closed form of the state after
 * a chunk on the Qwen3.5-9B NPU model card ("How it works": S_T = exp(G_T) S0 +
 * K^T diag(exp(G_T - G)) D, with D affine in S0), applied chunk after chunk.
 * So one chunk-scan launch walks segment 0 from the real state and, beside it,
 * every later segment twice: from X = 0 with its values (B, o0) and from X = I
 * with zero values (Phi, and the output maps m).  A short sequential combine
 * X_{p+1} = Phi_p X_p + B_p (fp32) then gives every segment's start state, and a
 * last pass writes the later segments' outputs.  The chain a head walks is
 * ~1/P of its chunks, at the cost of ~2x the chunk work for segments >= 1.
 *
 *   n_segments  1..8 (GDR_ERR_INVALID_ARG otherwise); more than there are chunk
 *               positions means one per chunk; 1 runs gdr_prefill_chunked's
 *               two-launch form.  With 2 or more segments n_seqs * H_v must not
 *               exceed 65535 (GDR_ERR_UNSUPPORTED, nothing launched).  gdr_prefill_segments_hint() gives the value
 *               the library would pick on the current device.
 *   workspace   DEVICE scratch of at least gdr_prefill_segmented_workspace_bytes
 *               bytes, 16-byte aligned, as for gdr_prefill_chunked.
 * Only the tensor-core shapes (d_k = d_v = 128, bf16 inputs, chunk 64) are
 * supported (GDR_ERR_UNSUPPORTED otherwise).  Every other argument, the
 * precision and the errors are as in gdr_prefill_chunked; the later segments'
 * outputs and the final state are sums of a few more fp32 products, so they
 * differ from gdr_prefill_chunked's by rounding only.
 */
gdr_status gdr_prefill_segmented(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens, int64_t t_total,
                                 const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 float *state, void *o, int32_t n_segments, void *workspace, size_t workspace_bytes,
                                 gdr_stream_t stream);

/*
 * Bytes of workspace gdr_prefill_segmented needs: gdr_prefill_workspace_bytes,
 * then, 256-byte aligned, per segment after the first four state-sized blocks
 * per (sequence, V head) (Phi, B and the start state in fp32, d_k * d_v floats
 * each, and the start state's transpose as bf16 hi and lo tensor-core operand
 * tiles, the same size), and two fp32 arrays shaped like o ([t_total][H_v][d_v])
 * for o0 and m.  Host-only;
 * equals gdr_prefill_workspace_bytes when n_segments is 1 (or the problem has one
 * chunk position).
 */
size_t gdr_prefill_segmented_workspace_bytes(const gdr_dims *dims, int32_t n_seqs, int64_t t_total,
                                             int32_t n_segments);

/*
 * The number of segments gdr_prefill_segmented should use on the current device
 * (1: use gdr_prefill_chunked).  It is the largest P <= 8 for which all
 * 2P - 1 runs of the scan launch (n_seqs * H_v * 4 CTAs of one SM each) fit on
 * the GPU at once and every segment keeps at least 8 chunks: e.g. 5 for one
 * 16K-token sequence of 4 V heads on a 152-SM GB300, 1 for 32 V heads.
 */
int32_t gdr_prefill_segments_hint(const gdr_dims *dims, int32_t n_seqs, int64_t t_total);

/*
 * One decode step for `batch` independent sequences (one token each).
 *
 * For each sequence b and V head h, with S = state[b][h] and d = exp(g):
 *     y = S^T k,  z = S^T q,  delta = beta (v - d y),
 *     o = scale (d z + (q . k) delta),  S <- d S + k delta^T   (in place)
 * which is the 1-token matrix form of the Qwen3.5-9B NPU model card
 * ("How it works": [q;k]^T S in one product, o = d q^T S + (q.k) delta,
 * S' = d S + k delta^T).  The state is read once and written once.
 *
 *   q, k [batch][H_qk][d_k]; v, o [batch][H_v][d_v]; g, beta [batch][H_v];
 *   state [batch][H_v][d_k][d_v] (in/out).
 */
gdr_status gdr_decode_step(const gdr_dims *dims, int32_t batch, const void *q, const void *k,
                           const void *v, const float *g, const float *beta, float *state, void *o,
                           gdr_stream_t stream);

/*
 * gdr_decode_step launched as a programmatic dependent of the kernel before it
 * on `stream`: it may start as soon as every CTA of that kernel is running,
 * instead of after it completes, and use the SMs that kernel leaves free.  This
 * is how a serving loop overlaps the decode step of some sequences with a long
 * prefill of another: queued right after gdr_prefill_chunked, it starts beside
 * the prefill's last chunk-scan launch (which occupies 4 SMs per V head).
 *
 * Contract: the step starts without waiting for the kernel immediately before
 * it on `stream`, nor for any kernel that was still running when that kernel
 * started (a kernel launched as a programmatic dependent starts before its own
 * predecessor has finished: gdr_prefill_chunked's chunk scan is one, of the
 * prefill's factor launch).  None of those kernels may write the step's q, k,
 * v, g, beta, state or o, or read its state or o.  Work that had completed
 * before all of them started is visible to the step.  After gdr_prefill_chunked
 * this holds whenever the decode step's tensors do not overlap the prefill's.
 * Arguments, results and errors are as in gdr_decode_step; later work on
 * `stream` is ordered after the step as usual.  Callers that cannot guarantee
 * the contract use gdr_decode_step.
 */
gdr_status gdr_decode_step_overlapped(const gdr_dims *dims, int32_t batch, const void *q, const void *k,
                                      const void *v, const float *g, const float *beta, float *state,
                                      void *o, gdr_stream_t stream);

/*
 * A prefill and one decode step of another batch in the same chunk-scan launch:
 * the continuous batching of prefill chunks and decode steps (the mixed batch of
 * serving; the prefill-to-decode handoff of a sequence is two calls, since a
 * decode step reads the state its prefill leaves).  The prefill is exactly
 * gdr_prefill_chunked(dims, n_seqs, cu_seqlens, t_total, q, k, v, g, beta,
 * state, o, workspace, workspace_bytes, stream), launches and results alike,
 * except that its last chunk-scan launch carries extra blocks on the SMs the
 * scan leaves free (one per free SM, at least one), which walk the decode
 * batch's (sequence, V head) pairs with the arithmetic of gdr_decode_step:
 * do_ and dstate come out bit-identical to gdr_decode_step(dims, dec_batch, dq,
 * dk, dv, dg, dbeta, dstate, d_o, stream).  The decode tensors have the
 * decode layouts (dq, dk [dec_batch][H_qk][d_k]; dv, d_o [dec_batch][H_v][d_v];
 * dg, dbeta [dec_batch][H_v]; dstate [dec_batch][H_v][d_k][d_v]) and must not
 * overlap the prefill's.  Only the tensor-core prefill shapes (bf16 inputs,
 * d_k = 128, chunk 64) have this launch (else GDR_ERR_UNSUPPORTED, nothing
 * launched); the gated output norm is not offered here.  dec_batch = 0 is
 * gdr_prefill_chunked; t_total = 0 is gdr_decode_step.  Errors: as
 * gdr_prefill_chunked, plus GDR_ERR_INVALID_ARG for a null or unaligned
 * decode tensor or dstate == state; device-side wait timeouts of the decode
 * blocks are reported as GDR_ERR_DEVICE_TIMEOUT through gdr_device_error.
 */
gdr_status gdr_prefill_with_decode(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens, int64_t t_total,
                                   const void *q, const void *k, const void *v, const float *g, const float *beta,
                                   float *state, void *o, void *workspace, size_t workspace_bytes, int32_t dec_batch,
                                   const void *dq, const void *dk, const void *dv, const float *dg, const float *dbeta,
                                   float *dstate, void *d_o, gdr_stream_t stream);

/*
 * gdr_decode_step with the gated RMSNorm after the rule fused into it: instead of
 * o, y = weight * o / sqrt(mean(o^2) + eps) * silu(z) is written for every
 * (sequence, V head) row of d_v outputs (the norm described at
 * gdr_gated_rmsnorm).  z [batch][H_v][d_v] in in_dtype, weight [d_v] fp32, y
 * [batch][H_v][d_v] in out_dtype; o itself is not stored.  Arguments and errors
 * otherwise as gdr_decode_step (GDR_ERR_INVALID_ARG also for a null or
 * misaligned z or weight, or a negative eps).
 */
gdr_status gdr_decode_step_gated(const gdr_dims *dims, int32_t batch, const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float *state, const void *z, const float *weight,
                                 float eps, void *y, gdr_stream_t stream);

/*
 * Gated RMSNorm of the rule's outputs, the step right after the rule: for each
 * of n_rows rows of d_v values (a (token, V head) row of o),
 *     y = weight * o / sqrt(mean(o^2) + eps) * silu(z),   silu(z) = z / (1 + exp(-z)),
 * one weight per channel.  The Qwen3.5-9B NPU model card ("fp16 precision of the
 * DeltaNet output") has a gated RMSNorm right after the rule; the Candle PR's
 * bug log ("Bug 7") gives its epsilon, 1e-6.  The form of the gate, silu(z), is
 * not on the pages: it is this library's reading.
 *   o      [n_rows][d_v] in dims->out_dtype (as gdr_prefill_chunked / gdr_verify_block wrote it)
 *   z      [n_rows][d_v] in dims->in_dtype
 *   weight [d_v] fp32;  y [n_rows][d_v] in dims->out_dtype (may be o)
 * One read of o and z and one write of y (HBM-bound).  GDR_ERR_INVALID_ARG for a
 * null or misaligned pointer, a negative n_rows or eps.
 */
gdr_status gdr_gated_rmsnorm(const gdr_dims *dims, int64_t n_rows, const void *o, const void *z, const float *weight,
                             float eps, void *y, gdr_stream_t stream);

/*
 * Speculative-verify block: n_tok <= 16 draft tokens per sequence in one pass.
 *
 * Copies state[s] to snapshot[s] (the state before the block), then runs the
 * n_tok tokens of every sequence from that state as one chunk, writing all
 * n_tok outputs and leaving the state after the whole block in state[s].
 * This is the model card's prompt-lookup decoding ("New in v2": the DeltaNet
 * state cannot be rewound, so it is snapshotted before the 16-token check and
 * the accepted tokens are re-fed).  After choosing how many tokens a_s to
 * accept, the caller either
 *   - restores the snapshot (gdr_state_restore) and re-feeds the a_s accepted
 *     tokens with gdr_prefill_chunked (lengths a_s, zero allowed), or
 *   - passes `deltas` here and commits with gdr_verify_commit, which needs no
 *     re-feed (one pass over the states).
 *
 *   q, k [n_seqs * n_tok][H_qk][d_k]; v, o [n_seqs * n_tok][H_v][d_v];
 *   g, beta [n_seqs * n_tok][H_v]; state, snapshot [n_seqs][H_v][d_k][d_v].
 *   snapshot must not overlap state.
 *   deltas: NULL, or fp32 [n_seqs * n_tok][H_v][d_v] that receives each draft
 *     token's correction u_t = beta_t (v_t - e^{g_t} S_{t-1}^T k_t), where
 *     S_{t-1} is the state just before token t inside the block.
 * With bf16 inputs the products with d-long inner dimensions run on warp-level
 * tensor-core MMAs, the state split into bf16 hi and lo halves (2^-16
 * relative, fp32 accumulation); fp32 inputs run on CUDA cores in fp32.
 * n_tok = 0 writes the snapshot and leaves the state as it is.
 */
gdr_status gdr_verify_block(const gdr_dims *dims, int32_t n_seqs, int32_t n_tok, const void *q,
                            const void *k, const void *v, const float *g, const float *beta,
                            float *state, float *snapshot, void *o, float *deltas, gdr_stream_t stream);

/*
 * Commits the accepted prefix of a verify block from its cached corrections,
 * instead of restoring the snapshot and re-feeding the accepted tokens.
 *
 * For sequence s with a = accepted[s] accepted tokens (rows s * n_tok + j,
 * j < a, of the block), writes the state after those a tokens:
 *     state[s] = e^{G_a} snapshot[s] + sum_{j < a} e^{G_a - G_j} k_j u_j^T,
 * with G_j = g_0 + ... + g_j (within the block), G_a = G_{a-1} (G_a = 0 and
 * state[s] = snapshot[s] when a = 0), u_j the corrections the block wrote to
 * `deltas`.  This unrolls the recurrence over the prefix (the model card's
 * closed form of S_T after a chunk, "How it works", taken at row a - 1): the
 * corrections of the first a tokens do not depend on later tokens, so they
 * are valid for every prefix.
 *
 *   accepted: device int32 [n_seqs], each in [0, n_tok].  A value outside
 *     that range leaves state[s] as it is and records GDR_ERR_INVALID_ARG in
 *     the device error word (see gdr_device_error).
 *   k, g, deltas: the block's tensors, as passed to gdr_verify_block.
 *   snapshot (in), state (out): [n_seqs][H_v][d_k][d_v]; must not overlap.
 */
gdr_status gdr_verify_commit(const gdr_dims *dims, int32_t n_seqs, int32_t n_tok, const int32_t *accepted,
                             const void *k, const float *g, const float *deltas, const float *snapshot,
                             float *state, gdr_stream_t stream);

/* Copy n_seqs states (H_v * d_k * d_v floats each) from `state` to `snapshot`. */
gdr_status gdr_state_snapshot(const gdr_dims *dims, int32_t n_seqs, const float *state,
                              float *snapshot, gdr_stream_t stream);

/* Copy n_seqs states back from `snapshot` to `state` (undo a verify block). */
gdr_status gdr_state_restore(const gdr_dims *dims, int32_t n_seqs, const float *snapshot,
                             float *state, gdr_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  *code receives GDR_OK or the first error a kernel recorded
 * (GDR_ERR_DEVICE_TIMEOUT when a bounded wait gave up).  Returns GDR_ERR_CUDA if
 * the synchronisation itself fails.
 */
gdr_status gdr_device_error(gdr_stream_t stream, int32_t *code);

/*
 * Self-test of the failure reporting every kernel uses: launches one block on
 * `stream` that waits, with the kernels' bounded mbarrier wait, on a barrier
 * nothing ever arrives on, for at most limit_cycles SM clocks (1 .. 2^31); the
 * wait gives up and records GDR_ERR_DEVICE_TIMEOUT in the device error word
 * (read it with gdr_device_error).  Nothing else is touched and the context
 * stays usable.  Returns GDR_ERR_INVALID_ARG for a limit out of range,
 * GDR_ERR_CUDA if the launch fails.
 */
gdr_status gdr_selftest_wait_timeout(int64_t limit_cycles, gdr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
