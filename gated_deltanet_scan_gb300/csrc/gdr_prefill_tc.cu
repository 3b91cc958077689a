// Tensor-core (tcgen05) chunked prefill -- placeholder until the kernel lands.
#include "gdr_internal.h"

namespace gdr {

static __device__ int32_t g_device_error;

cudaError_t launch_prefill_tc(const Args &a, cudaStream_t s) { return launch_chunk_cc(a, s); }

cudaError_t read_clear_device_error(cudaStream_t s, int32_t *code) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    int32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    *code = v;
    return e;
}

}  // namespace gdr
