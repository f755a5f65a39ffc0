// la_noalloc.cu -- la_fwd_noalloc: the forward pass for callers that cannot
// allocate device memory at the point of the call.
//
// la_fwd needs scratch device memory only for packed sequences: the
// longest-first schedule (one int32 per sequence) that its kernels read.  It
// takes that scratch from the caller.  Some callers have no device memory to
// give: a process whose device memory is all owned by another allocator that
// hands out no scratch buffers, or a code path where a cudaMalloc is not
// allowed because it would synchronize the device.  For them this entry point
// keeps the schedule in a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (LA_FWD_NOALLOC_MAX_SEQS int32) until the process exits.
// In host code its name is only a host-side stand-in, so its device address
// is looked up with cudaGetSymbolAddress once per device, with that device
// current, on the first packed call made on that device, and kept for the
// rest of the process (a cudaDeviceReset would make it stale, so the header
// tells callers not to use this entry point after one).  Only the schedule
// goes into the array: the workspace size passed on is the schedule's own,
// so la_fwd never places the sequence split's states there.

#include <cstdio>
#include <mutex>

#include "../../include/la.h"
#include "la_internal.h"

namespace {

static __device__ __align__(256) int32_t g_noalloc_schedule[LA_FWD_NOALLOC_MAX_SEQS];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void *g_schedule_addr[kMaxDevices] = {};

// Device address of g_noalloc_schedule on the current device (looked up once).
la_status schedule_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        la::set_last_error("la_fwd_noalloc: cudaGetDevice failed");
        return LA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        la::set_last_error("la_fwd_noalloc: device ordinal out of range");
        return LA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_schedule_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_schedule);
        if (e != cudaSuccess || !p) {
            la::set_last_error("la_fwd_noalloc: cudaGetSymbolAddress of the schedule array failed");
            return LA_ERR_CUDA;
        }
        g_schedule_addr[dev] = p;
    }
    *out = g_schedule_addr[dev];
    return LA_OK;
}

}  // namespace

extern "C" la_status la_fwd_noalloc(const la_dims *dims, int32_t dtype, const void *q,
                                    const void *k, const void *v, const float *g_gamma,
                                    float scale, const float *initial_state, int32_t reverse,
                                    const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                    void *o, float *final_state, void *stream)
{
    void *ws = nullptr;
    size_t ws_bytes = 0;
    if (cu_seqlens) {
        if (dims && dims->num_seqs > LA_FWD_NOALLOC_MAX_SEQS) {
            char msg[160];
            snprintf(msg, sizeof(msg),
                     "la_fwd_noalloc: %d packed sequences, at most %d are supported "
                     "(use la_fwd with a workspace)",
                     dims->num_seqs, LA_FWD_NOALLOC_MAX_SEQS);
            la::set_last_error(msg);
            return LA_ERR_UNSUPPORTED;
        }
        la_status st = schedule_address(&ws);
        if (st != LA_OK)
            return st;
        ws_bytes = la_workspace_size(dims ? dims->num_seqs : 0);
    }
    // The schedule overwrites the first num_seqs entries on every call and the
    // kernels read only those, so nothing has to be cleared beforehand.
    return la_fwd(dims, dtype, q, k, v, g_gamma, scale, initial_state, reverse, cu_seqlens,
                  cu_seqlens_host, o, final_state, ws, ws_bytes, stream);
}
