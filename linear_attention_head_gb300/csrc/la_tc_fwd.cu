// la_tc_fwd.cu -- tensor-core (tcgen05) forward-type sweep (placeholder until
// the tcgen05 kernel lands: every request goes to the CUDA-core kernels).
#include "la_internal.h"

namespace la {
namespace {
__device__ int g_tc_error;
}

bool tc_forward_supported(const SweepArgs &) { return false; }

cudaError_t tc_forward_sweep(const SweepArgs &, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t tc_read_and_clear_error(cudaStream_t s, int *err)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(err, g_tc_error, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace la
