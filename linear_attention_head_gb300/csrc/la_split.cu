// la_split.cu -- the state scan of the sequence split.
//
// When a call has too few (sequence, head) pairs to occupy the GPU, every
// long sequence is cut into segments that run as separate packed sequences
// (the OpenNLPLab/lightning-attention README lists a parallel version of the
// method under Todo; this is one form of it, exchanging one state per
// segment).  Both sweep shapes carry a state whose
// value after a segment is an affine function of its value before it:
//     after = gamma^L * before + F,
// F being the segment's result from a zero state (L = its length).  So a
// first pass computes F for every segment (zero initial states, all segments
// in parallel), this scan turns the F into each segment's true initial state
// and the sequence's final state, and a second pass runs every segment again
// from its initial state.  With the gated form's per-key gate the segment's
// decay is a diagonal, exp(lam) per key channel (the sum of the log-decays
// over the segment), on the state's rows or columns: still elementwise.
// The scan is elementwise in the state, so one
// thread owns one state element of one (sequence, head) and walks that
// sequence's segments in visiting order.

#include <cstdint>

#include "la_internal.h"

namespace la {
namespace {

__global__ void __launch_bounds__(256) split_scan_kernel(SplitScanArgs a)
{
    const int64_t de = (int64_t)a.D * a.E;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int h = blockIdx.y, n = blockIdx.z;
    if (idx >= de)
        return;
    const int64_t r = idx / a.E, c = idx % a.E;
    const int64_t user = ((int64_t)n * a.H + h) * de;
    float carry = a.start.p ? a.start.p[user + r * a.start.rs + c * a.start.cs] : 0.f;
    const float g = a.g[h];
    const int first = a.seq_first[n], count = a.seq_first[n + 1] - first;
    const int64_t lw = a.lam_cols ? a.E : a.D, li = a.lam_cols ? c : r;
    // eight segments' contributions and decays loaded together, then the
    // carries formed in visiting order and stored
    constexpr int BATCH = 8;
    for (int j0 = 0; j0 < count; j0 += BATCH) {
        float f[BATCH], dec[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            f[u] = 0.f;
            dec[u] = 1.f;
            if (j0 + u < count) {
                const int seg = first + (a.descending ? count - 1 - (j0 + u) : j0 + u);
                f[u] = a.W[((int64_t)seg * a.H + h) * de + idx];
                const int len = a.seg_cu[seg + 1] - a.seg_cu[seg];
                dec[u] = a.lam ? a.lam[((int64_t)seg * a.H + h) * lw + li] : g * (float)len;
            }
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            if (j0 + u < count) {
                const int seg = first + (a.descending ? count - 1 - (j0 + u) : j0 + u);
                a.W[((int64_t)seg * a.H + h) * de + idx] = carry;   // the segment's initial state
                carry = fmaf(expf(dec[u]), carry, f[u]);
            }
        }
    }
    if (a.fin.p)
        a.fin.p[user + r * a.fin.rs + c * a.fin.cs] = carry;
}

}  // namespace

cudaError_t split_scan(const SplitScanArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0)
        return cudaSuccess;
    if (a.N > 65535 || a.H > 65535)
        return cudaErrorNotSupported;
    const int64_t de = (int64_t)a.D * a.E;
    dim3 grid((unsigned)((de + 255) / 256), (unsigned)a.H, (unsigned)a.N);
    split_scan_kernel<<<grid, 256, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
