// Internal launch interface shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdr.h"

namespace gdr {

// Everything one launch needs, already validated on the host.
struct Args {
    int h_qk, h_v, d;        // d = d_k = d_v
    int in_bf16, out_bf16;   // 1 when the tensor is bf16, 0 for fp32
    float scale;
    int n_seqs;
    const int32_t *cu_seqlens;  // device; nullptr => sequence s is [s*fixed_len, (s+1)*fixed_len)
    int fixed_len;
    int64_t t_total;
    const void *q, *k, *v;
    const float *g, *beta;
    float *state;
    float *snapshot;  // optional copy of the incoming state (verify block)
    void *o;
};

cudaError_t launch_decode(const Args &a, cudaStream_t s);
cudaError_t launch_chunk_cc(const Args &a, cudaStream_t s);
cudaError_t launch_prefill_tc(const Args &a, cudaStream_t s);
cudaError_t launch_copy_f32(const float *src, float *dst, size_t n, cudaStream_t s);

// Synchronises `s`, then reads and clears the device error word.
cudaError_t read_clear_device_error(cudaStream_t s, int32_t *code);

}  // namespace gdr
