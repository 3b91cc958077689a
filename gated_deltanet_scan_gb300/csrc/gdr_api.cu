// C-ABI entry points: argument checks on the host, then the launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "gdr_factor_layout.h"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {
namespace {

// Scratch of gdr_prefill_chunked_static: one fixed device array, never allocated
// at run time.  Its device address (a host-side name of it is not one) is
// looked up in the current device's context on every call: nothing is cached, so
// a reset device or a new context, or concurrent first calls from several host
// threads, need no care; the lookup costs little next to the launches.
constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

void *static_workspace() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
    return p;
}

__global__ void copy_f32_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n4) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
        __stcs(&dst[i], __ldcs(&src[i]));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One thread waits, with the bounded wait of the kernels, on an mbarrier that
// nothing arrives on, gives up after `limit` SM clocks and records the timeout.
__global__ void wait_timeout_kernel(int32_t *err, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait_bounded(b, 0u, limit))
        atomicCAS(err, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
}

gdr_status check_dims(const gdr_dims *d) {
    if (!d) return GDR_ERR_INVALID_ARG;
    if (d->h_qk <= 0 || d->h_v <= 0 || d->h_v % d->h_qk != 0) return GDR_ERR_INVALID_ARG;
    if (d->d_k <= 0 || d->d_v <= 0) return GDR_ERR_INVALID_ARG;
    if (d->in_dtype != GDR_F32 && d->in_dtype != GDR_BF16) return GDR_ERR_INVALID_ARG;
    if (d->out_dtype != GDR_F32 && d->out_dtype != GDR_BF16) return GDR_ERR_INVALID_ARG;
    if (d->chunk != 16 && d->chunk != 64) return GDR_ERR_UNSUPPORTED;
    if (d->d_k != d->d_v) return GDR_ERR_UNSUPPORTED;
    if (d->d_k != 32 && d->d_k != 64 && d->d_k != 128) return GDR_ERR_UNSUPPORTED;
    if (d->flags & ~(GDR_FLAG_QK_L2NORM | GDR_FLAG_BETA_LOGITS)) return GDR_ERR_INVALID_ARG;
    return GDR_OK;
}

Args make_args(const gdr_dims *d) {
    Args a{};
    a.h_qk = d->h_qk;
    a.h_v = d->h_v;
    a.d = d->d_k;
    a.in_bf16 = d->in_dtype == GDR_BF16;
    a.out_bf16 = d->out_dtype == GDR_BF16;
    a.scale = d->scale;
    a.qk_norm = (d->flags & GDR_FLAG_QK_L2NORM) != 0;
    a.beta_logits = (d->flags & GDR_FLAG_BETA_LOGITS) != 0;
    a.c_lo = 0;
    a.c_hi = INT_MAX;
    return a;
}

bool tensors_ok(const void *q, const void *k, const void *v, const float *g, const float *beta,
                const float *state, const void *o) {
    const void *ps[] = {q, k, v, g, beta, state, o};
    for (const void *p : ps)
        if (!p || !aligned16(p)) return false;
    return true;
}

gdr_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA; }

bool use_tensor_core_prefill(const gdr_dims *d) {
    return d->chunk == 64 && d->d_k == 128 && d->in_dtype == GDR_BF16;
}

// Chunk at which a prefill is split into two parts, or 0 (no split).  The
// chunk scan runs n_seqs * h_v * 4 CTAs of one SM each; when that leaves at
// least 16 SMs free and the factor kernel (4 CTAs per SM) needs at least two
// waves, the factors of chunks [m, n) are computed on those SMs while the scan
// walks chunks [0, m).  (With one wave or less the first factor launch would
// take as long as the whole one, and the extra scan launch only costs time:
// T = 1024 at 32 V heads measured 80 us split against 74 us whole.)  Both kernels'
// costs grow with the chunks they handle; measured at h_v = 32 with 24 free
// SMs (T = 16384, a sweep of the split chunk), the prefill is fastest with
// about 73% of the chunks in the first part (m = 175-195 of 256: 0.647 ms,
// against 0.655 ms at 60% and 0.687 ms unsplit): m / n = r / (1 + r) with
// r = c h_v / F for F free SMs.  With the faster chunk scan of later versions
// c = 2.2 (m = 191) measured 0.489 ms against 0.492-0.493 ms for c = 1.8, 2.0
// and 2.5.
int split_chunk(const gdr_dims *d, int32_t n_seqs, int64_t t_total) {
    static int sms_of[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (sms_of[dev] == 0 && cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    const int64_t nch = (t_total + 63) / 64;
    const int64_t chain_ctas = (int64_t)n_seqs * d->h_v * 4;
    const int64_t free_sms = sms_of[dev] - chain_ctas;
    if (nch * d->h_v < 8LL * sms_of[dev] || free_sms < 16) return 0;
    const double r = 2.2 * d->h_v / (double)free_sms;
    int64_t m = (int64_t)std::ceil(r / (1.0 + r) * (double)nch);
    if (m < 1) m = 1;
    if (m > nch - 1) m = nch - 1;
    return (int)m;
}

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// Segments of the two-level prefill for this problem on the current device.  Its
// scan launch runs 2P - 1 runs of n_seqs * h_v * 4 CTAs (one SM each); it pays
// when they all fit on the GPU at once, so the segments' chains walk side by
// side: P is the largest value up to 8 for which they do and every segment keeps
// at least 8 chunks, else 1 (one chain per head, the ordinary prefill).
int segments_hint(const gdr_dims *d, int32_t n_seqs, int64_t t_total) {
    if (!use_tensor_core_prefill(d) || n_seqs <= 0 || t_total <= 0) return 1;
    const int sms = device_sms();
    const int64_t n_ch = (t_total + 63) / 64;
    const int64_t per_run = (int64_t)n_seqs * d->h_v * 4;
    int best = 1;
    for (int P = 2; P <= 8; ++P)
        if (per_run * (2 * P - 1) <= sms && n_ch >= 8LL * P) best = P;
    return best;
}

// The tensor-core prefill on `s`: factors, then the chunk scan (a programmatic
// dependent of the factor launch), or, split at
// chunk m (see split_chunk): factors [0, m), scan [0, m), factors [m, n) as a
// programmatic dependent launch (it starts once every CTA of the scan is
// running, on the SMs they leave free, and reads nothing the scan writes),
// then scan [m, n) from the state the first part left.
cudaError_t prefill_tc(const gdr_dims *dims, const Args &a, float *ws, int32_t *err, cudaStream_t s,
                       bool allow_split, const Args *dec = nullptr) {
    const int m = allow_split ? split_chunk(dims, a.n_seqs, a.t_total) : 0;
    // decode blocks of a mixed launch: eight (sequence, V head) pairs each, so that
    // the hardware places them on the SMs the scan leaves free and, once its CTAs
    // finish, on every SM
    int dec_blocks = 0;
    if (dec) dec_blocks = (int)std::max<int64_t>(1, ((int64_t)dec->n_seqs * dec->h_v + 7) / 8);
    if (m == 0) {
        // the scan's prologue overlaps the factor grid's last wave (T = 1024: 73 -> 67 us)
        cudaError_t e = launch_factors(a, ws, err, s, false);
        if (e != cudaSuccess) return e;
        return launch_prefill_tc(a, ws, s, true, dec, dec_blocks);
    }
    Args a1 = a, a2 = a;
    a1.c_hi = m;
    a2.c_lo = m;
    // the first scan is an ordinary launch here: as a programmatic dependent it would
    // let the second factor launch start while the first one still runs (T = 16384
    // measured 0.72 ms against 0.64 ms)
    cudaError_t e = launch_factors(a1, ws, err, s, false);
    if (e == cudaSuccess) e = launch_prefill_tc(a1, ws, s, false);
    if (e == cudaSuccess) e = launch_factors(a2, ws, err, s, true);
    // an ordinary launch: it reads the state the first scan writes
    if (e == cudaSuccess) e = launch_prefill_tc(a2, ws, s, false, dec, dec_blocks);
    return e;
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" {

int32_t gdr_abi_version(void) { return GDR_ABI_VERSION; }

const char *gdr_status_string(gdr_status st) {
    switch (st) {
        case GDR_OK: return "GDR_OK";
        case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG: invalid argument";
        case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: shape, chunk or dtype not compiled";
        case GDR_ERR_CUDA: return "GDR_ERR_CUDA: a CUDA launch or synchronisation failed";
        case GDR_ERR_DEVICE_TIMEOUT: return "GDR_ERR_DEVICE_TIMEOUT: a device-side wait gave up";
    }
    return "unknown gdr_status";
}

size_t gdr_prefill_workspace_bytes(const gdr_dims *dims, int32_t n_seqs, int64_t t_total) {
    if (check_dims(dims) != GDR_OK || n_seqs <= 0 || t_total <= 0 || !use_tensor_core_prefill(dims)) return 0;
    const size_t bytes = (size_t)fac::workspace_bytes(fac::n_slots(t_total, n_seqs), dims->h_v, dims->h_qk);
    return (bytes + 255) & ~(size_t)255;
}

}  // extern "C"

namespace gdr {
namespace {

gdr_status prefill(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens, int64_t t_total,
                   const void *q, const void *k, const void *v, const float *g, const float *beta,
                   float *state, void *o, void *workspace, size_t workspace_bytes, gdr_stream_t stream,
                   bool allow_split, const Args *dec = nullptr) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_seqs < 0 || t_total < 0) return GDR_ERR_INVALID_ARG;
    if (n_seqs == 0) return t_total == 0 ? GDR_OK : GDR_ERR_INVALID_ARG;
    if (!cu_seqlens || !aligned16(cu_seqlens) || !state || !aligned16(state)) return GDR_ERR_INVALID_ARG;
    if (t_total > 0 && !tensors_ok(q, k, v, g, beta, state, o)) return GDR_ERR_INVALID_ARG;
    if (t_total > ((int64_t)1 << 31) - 1) return GDR_ERR_UNSUPPORTED;
    const size_t need = gdr_prefill_workspace_bytes(dims, n_seqs, t_total);
    if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need)) return GDR_ERR_INVALID_ARG;
    Args a = make_args(dims);
    a.n_seqs = n_seqs;
    a.cu_seqlens = cu_seqlens;
    a.fixed_len = 0;
    a.t_total = t_total;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.snapshot = nullptr;
    a.o = o;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (t_total == 0) {  // every sequence empty: states unchanged
        if (!dec) return GDR_OK;
        int32_t *err = device_error_word();
        if (!err) return GDR_ERR_CUDA;
        return from_cuda(launch_decode(*dec, err, s, false));
    }
    if (use_tensor_core_prefill(dims)) {
        int32_t *err = device_error_word();
        if (!err) return GDR_ERR_CUDA;
        return from_cuda(prefill_tc(dims, a, static_cast<float *>(workspace), err, s, allow_split, dec));
    }
    if (dec) return GDR_ERR_UNSUPPORTED;
    return from_cuda(launch_chunk_cc(a, s));
}

}  // namespace
}  // namespace gdr

extern "C" {

gdr_status gdr_prefill_chunked(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens,
                               int64_t t_total, const void *q, const void *k, const void *v,
                               const float *g, const float *beta, float *state, void *o,
                               void *workspace, size_t workspace_bytes, gdr_stream_t stream) {
    return prefill(dims, n_seqs, cu_seqlens, t_total, q, k, v, g, beta, state, o, workspace, workspace_bytes,
                   stream, true);
}

size_t gdr_prefill_static_workspace_capacity(void) { return kStaticWorkspaceBytes; }

int32_t gdr_prefill_segments_hint(const gdr_dims *dims, int32_t n_seqs, int64_t t_total) {
    if (check_dims(dims) != GDR_OK) return 1;
    return segments_hint(dims, n_seqs, t_total);
}

size_t gdr_prefill_segmented_workspace_bytes(const gdr_dims *dims, int32_t n_seqs, int64_t t_total,
                                             int32_t n_segments) {
    const size_t factor_bytes = gdr_prefill_workspace_bytes(dims, n_seqs, t_total);
    if (factor_bytes == 0 || n_segments < 1 || n_segments > 8) return factor_bytes;
    const int64_t n_ch = (t_total + 63) / 64;
    const int P = (int)(n_segments < n_ch ? n_segments : n_ch);
    if (P <= 1) return factor_bytes;
    return segment_layout((int64_t)factor_bytes, n_seqs, dims->h_v, t_total, P).total;
}

gdr_status gdr_prefill_segmented(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens, int64_t t_total,
                                 const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 float *state, void *o, int32_t n_segments, void *workspace, size_t workspace_bytes,
                                 gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_segments < 1 || n_segments > 8) return GDR_ERR_INVALID_ARG;
    if (!use_tensor_core_prefill(dims)) return GDR_ERR_UNSUPPORTED;
    const int64_t n_ch = (t_total + 63) / 64;
    const int P = (int)(n_segments < n_ch ? n_segments : n_ch);
    if (P <= 1)  // one segment: the ordinary two-launch prefill
        return prefill(dims, n_seqs, cu_seqlens, t_total, q, k, v, g, beta, state, o, workspace, workspace_bytes,
                       stream, false);
    if (n_seqs < 0 || t_total < 0) return GDR_ERR_INVALID_ARG;
    if (n_seqs == 0) return t_total == 0 ? GDR_OK : GDR_ERR_INVALID_ARG;
    if (!cu_seqlens || !aligned16(cu_seqlens) || !tensors_ok(q, k, v, g, beta, state, o)) return GDR_ERR_INVALID_ARG;
    if (t_total > ((int64_t)1 << 31) - 1) return GDR_ERR_UNSUPPORTED;
    // the combine and fix-up grids index (sequence, V head) pairs in one grid dimension
    if ((int64_t)n_seqs * dims->h_v > 65535) return GDR_ERR_UNSUPPORTED;
    const size_t need = gdr_prefill_segmented_workspace_bytes(dims, n_seqs, t_total, n_segments);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return GDR_ERR_INVALID_ARG;
    const SegLayout L = segment_layout((int64_t)gdr_prefill_workspace_bytes(dims, n_seqs, t_total), n_seqs,
                                       dims->h_v, t_total, P);
    Args a = make_args(dims);
    a.n_seqs = n_seqs;
    a.cu_seqlens = cu_seqlens;
    a.fixed_len = 0;
    a.t_total = t_total;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.snapshot = nullptr;
    a.o = o;
    int32_t *err = device_error_word();
    if (!err) return GDR_ERR_CUDA;
    return from_cuda(launch_segmented(a, P, static_cast<uint8_t *>(workspace), L, err,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

gdr_status gdr_prefill_chunked_static(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens,
                                      int64_t t_total, const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float *state, void *o,
                                      gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_seqs < 0 || t_total < 0) return GDR_ERR_INVALID_ARG;
    const size_t need = gdr_prefill_workspace_bytes(dims, n_seqs, t_total);
    if (need > kStaticWorkspaceBytes) return GDR_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (need > 0) {
        ws = static_workspace();
        if (!ws) return GDR_ERR_CUDA;
    }
    return prefill(dims, n_seqs, cu_seqlens, t_total, q, k, v, g, beta, state, o, ws, need, stream, false);
}

gdr_status gdr_prefill_with_decode(const gdr_dims *dims, int32_t n_seqs, const int32_t *cu_seqlens, int64_t t_total,
                                   const void *q, const void *k, const void *v, const float *g, const float *beta,
                                   float *state, void *o, void *workspace, size_t workspace_bytes, int32_t dec_batch,
                                   const void *dq, const void *dk, const void *dv, const float *dg, const float *dbeta,
                                   float *dstate, void *d_o, gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (!use_tensor_core_prefill(dims)) return GDR_ERR_UNSUPPORTED;
    if (dec_batch < 0) return GDR_ERR_INVALID_ARG;
    if (dec_batch == 0)
        return prefill(dims, n_seqs, cu_seqlens, t_total, q, k, v, g, beta, state, o, workspace, workspace_bytes,
                       stream, true);
    if (!tensors_ok(dq, dk, dv, dg, dbeta, dstate, d_o) || dstate == state) return GDR_ERR_INVALID_ARG;
    Args d = make_args(dims);
    d.n_seqs = dec_batch;
    d.cu_seqlens = nullptr;
    d.fixed_len = 1;
    d.t_total = dec_batch;
    d.q = dq;
    d.k = dk;
    d.v = dv;
    d.g = dg;
    d.beta = dbeta;
    d.state = dstate;
    d.snapshot = nullptr;
    d.o = d_o;
    return prefill(dims, n_seqs, cu_seqlens, t_total, q, k, v, g, beta, state, o, workspace, workspace_bytes, stream,
                   true, &d);
}

}  // extern "C"

namespace gdr {
namespace {

gdr_status decode(const gdr_dims *dims, int32_t batch, const void *q, const void *k, const void *v,
                  const float *g, const float *beta, float *state, void *o, gdr_stream_t stream, bool overlap,
                  const void *norm_z = nullptr, const float *norm_w = nullptr, float norm_eps = 0.f) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (batch < 0) return GDR_ERR_INVALID_ARG;
    if (batch == 0) return GDR_OK;
    if (!tensors_ok(q, k, v, g, beta, state, o)) return GDR_ERR_INVALID_ARG;
    Args a = make_args(dims);
    a.n_seqs = batch;
    a.cu_seqlens = nullptr;
    a.fixed_len = 1;
    a.t_total = batch;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.snapshot = nullptr;
    a.o = o;
    a.norm_z = norm_z;
    a.norm_w = norm_w;
    a.norm_eps = norm_eps;
    int32_t *err = device_error_word();
    if (!err) return GDR_ERR_CUDA;
    return from_cuda(launch_decode(a, err, reinterpret_cast<cudaStream_t>(stream), overlap));
}

}  // namespace
}  // namespace gdr

extern "C" {

gdr_status gdr_decode_step(const gdr_dims *dims, int32_t batch, const void *q, const void *k,
                           const void *v, const float *g, const float *beta, float *state, void *o,
                           gdr_stream_t stream) {
    return decode(dims, batch, q, k, v, g, beta, state, o, stream, false);
}

gdr_status gdr_decode_step_overlapped(const gdr_dims *dims, int32_t batch, const void *q, const void *k,
                                      const void *v, const float *g, const float *beta, float *state,
                                      void *o, gdr_stream_t stream) {
    return decode(dims, batch, q, k, v, g, beta, state, o, stream, true);
}

gdr_status gdr_decode_step_gated(const gdr_dims *dims, int32_t batch, const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float *state, const void *z, const float *weight,
                                 float eps, void *y, gdr_stream_t stream) {
    if (!z || !weight || !aligned16(z) || !aligned16(weight) || !(eps >= 0.f)) return GDR_ERR_INVALID_ARG;
    return decode(dims, batch, q, k, v, g, beta, state, y, stream, false, z, weight, eps);
}

gdr_status gdr_gated_rmsnorm(const gdr_dims *dims, int64_t n_rows, const void *o, const void *z, const float *weight,
                             float eps, void *y, gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_rows < 0 || !(eps >= 0.f)) return GDR_ERR_INVALID_ARG;
    if (n_rows == 0) return GDR_OK;
    const void *ps[] = {o, z, weight, y};
    for (const void *p : ps)
        if (!p || !aligned16(p)) return GDR_ERR_INVALID_ARG;
    return from_cuda(launch_gated_rmsnorm(n_rows, dims->d_v, o, dims->out_dtype == GDR_BF16, z,
                                          dims->in_dtype == GDR_BF16, weight, eps, y, dims->out_dtype == GDR_BF16,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

gdr_status gdr_verify_block(const gdr_dims *dims, int32_t n_seqs, int32_t n_tok, const void *q,
                            const void *k, const void *v, const float *g, const float *beta,
                            float *state, float *snapshot, void *o, float *deltas, gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_seqs < 0 || n_tok < 0 || n_tok > 16) return GDR_ERR_INVALID_ARG;
    if (n_seqs == 0) return GDR_OK;
    if (!snapshot || !aligned16(snapshot) || !state || !aligned16(state)) return GDR_ERR_INVALID_ARG;
    if (snapshot == state) return GDR_ERR_INVALID_ARG;
    if (n_tok > 0 && !tensors_ok(q, k, v, g, beta, state, o)) return GDR_ERR_INVALID_ARG;
    if (deltas && !aligned16(deltas)) return GDR_ERR_INVALID_ARG;
    Args a = make_args(dims);
    a.n_seqs = n_seqs;
    a.cu_seqlens = nullptr;
    a.fixed_len = n_tok;
    a.deltas = deltas;
    a.t_total = (int64_t)n_seqs * n_tok;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.snapshot = snapshot;
    a.o = o;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (n_tok == 0) {  // no tokens: the snapshot only, the state stays as it is
        const size_t n = (size_t)n_seqs * dims->h_v * dims->d_k * dims->d_v;
        return from_cuda(launch_copy_f32(state, snapshot, n, cs));
    }
    if (a.in_bf16) return from_cuda(launch_verify(a, cs));
    return from_cuda(launch_chunk_cc(a, cs));
}

gdr_status gdr_verify_commit(const gdr_dims *dims, int32_t n_seqs, int32_t n_tok, const int32_t *accepted,
                             const void *k, const float *g, const float *deltas, const float *snapshot,
                             float *state, gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_seqs < 0 || n_tok < 0 || n_tok > 16) return GDR_ERR_INVALID_ARG;
    if (n_seqs == 0) return GDR_OK;
    if (!accepted || !snapshot || !state || !aligned16(snapshot) || !aligned16(state) || snapshot == state)
        return GDR_ERR_INVALID_ARG;
    if (n_tok > 0 && (!k || !g || !deltas || !aligned16(k) || !aligned16(g) || !aligned16(deltas)))
        return GDR_ERR_INVALID_ARG;
    int32_t *err = device_error_word();
    if (!err) return GDR_ERR_CUDA;
    Args a = make_args(dims);
    a.n_seqs = n_seqs;
    a.fixed_len = n_tok;
    a.k = k;
    a.g = g;
    a.deltas = const_cast<float *>(deltas);
    a.accepted = accepted;
    a.snapshot_in = snapshot;
    a.state = state;
    return from_cuda(launch_commit(a, err, reinterpret_cast<cudaStream_t>(stream)));
}

static gdr_status copy_states(const gdr_dims *dims, int32_t n_seqs, const float *src, float *dst,
                              gdr_stream_t stream) {
    gdr_status st = check_dims(dims);
    if (st != GDR_OK) return st;
    if (n_seqs < 0) return GDR_ERR_INVALID_ARG;
    if (n_seqs == 0) return GDR_OK;
    if (!src || !dst || !aligned16(src) || !aligned16(dst) || src == dst) return GDR_ERR_INVALID_ARG;
    const size_t n = (size_t)n_seqs * dims->h_v * dims->d_k * dims->d_v;
    return from_cuda(launch_copy_f32(src, dst, n, reinterpret_cast<cudaStream_t>(stream)));
}

gdr_status gdr_state_snapshot(const gdr_dims *dims, int32_t n_seqs, const float *state,
                              float *snapshot, gdr_stream_t stream) {
    return copy_states(dims, n_seqs, state, snapshot, stream);
}

gdr_status gdr_state_restore(const gdr_dims *dims, int32_t n_seqs, const float *snapshot,
                             float *state, gdr_stream_t stream) {
    return copy_states(dims, n_seqs, snapshot, state, stream);
}

gdr_status gdr_device_error(gdr_stream_t stream, int32_t *code) {
    if (!code) return GDR_ERR_INVALID_ARG;
    return from_cuda(read_clear_device_error(reinterpret_cast<cudaStream_t>(stream), code));
}

gdr_status gdr_selftest_wait_timeout(int64_t limit_cycles, gdr_stream_t stream) {
    if (limit_cycles < 1 || limit_cycles > ((int64_t)1 << 31)) return GDR_ERR_INVALID_ARG;
    int32_t *err = device_error_word();
    if (!err) return GDR_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, (long long)limit_cycles);
    return from_cuda(cudaGetLastError());
}

}  // extern "C"

namespace gdr {

cudaError_t launch_copy_f32(const float *src, float *dst, size_t n, cudaStream_t s) {
    // n is a multiple of 4: every state holds d_k * d_v floats with d in {32, 64, 128}.
    const size_t n4 = n / 4;
    const unsigned threads = 256;
    unsigned blocks = (unsigned)((n4 + threads - 1) / threads);
    if (blocks > 152u * 16u) blocks = 152u * 16u;
    copy_f32_kernel<<<blocks, threads, 0, s>>>(reinterpret_cast<const float4 *>(src),
                                                reinterpret_cast<float4 *>(dst), n4);
    return cudaGetLastError();
}

}  // namespace gdr
