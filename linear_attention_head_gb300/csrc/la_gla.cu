// la_gla.cu -- gradient of the per-key gate (the GLA form of the recurrence).
//
// With a gate g_t (a log-decay per key channel, ejkernel `recurrent`'s
// GLA-style gate) the state is S_t = diag(exp(g_gamma + g_t)) S_{t-1} + k_t v_t^T.
// Writing G_t for the cumulative log-decay up to token t (processing order),
// the output depends on G through q_t exp(G_t) and k_u exp(-G_u) only, and
// the final state through an extra factor exp(G_L).  Hence, per key channel,
//     dL/dG_t = q_t dq_t - k_t dk_t   (+ sum_e F dF at the last token),
// and since g_w enters every G_t with t >= w,
//     dg_w = sum over t at or after w (processing order) of dL/dG_t.
// dq and dk are the backward pass's gradients, F the final state and dF its
// upstream gradient.  Two kernels: per block of DG_TB tokens the sum of
// q dq - k dk per channel, then the reverse running sum inside each block
// starting from the later blocks' sums and the final-state term.
// dq and dk come in fp32, as the sweeps computed them: dg adds up T terms,
// and rounding each gradient to bf16 first would add an independent error of
// about 2^-9 of the term to each, a random walk that grows with T while dg,
// bounded by the decay, does not (0.013-0.015 of max|dg| at T = 300, 0.022
// at 2000 and 0.04-0.05 at 8192 on the test inputs).  The bf16 copies are
// written here.

#include <cstdint>

#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

template <typename T> __device__ __forceinline__ float ldt(const T *p);
template <> __device__ __forceinline__ float ldt<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ldt<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void stt(T *p, float x);
template <> __device__ __forceinline__ void stt<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void stt<__nv_bfloat16>(__nv_bfloat16 *p, float x)
{
    *p = __float2bfloat16_rn(x);
}

struct Seq {
    int64_t row, bos, len;
};

__device__ __forceinline__ Seq seq_of(const GateGradArgs &a, int n)
{
    Seq s;
    if (a.cu) {
        s.row = 0;
        s.bos = a.cu[n];
        s.len = (int64_t)a.cu[n + 1] - a.cu[n];
    } else {
        s.row = n;
        s.bos = 0;
        s.len = a.T;
    }
    return s;
}

// q dq - k dk at processing position p, channel c of query head h (k of
// its key head h / khd, dk this query head's part); COPY: also writes the
// token-dtype dq, dk there (each when its pointer is set)
template <typename T, bool COPY>
__device__ __forceinline__ float term(const GateGradArgs &a, const Seq &s, int h, int64_t p, int c)
{
    const int64_t t = s.bos + (a.reverse ? s.len - 1 - p : p);
    const int64_t off = s.row * a.sb + t * a.st + (int64_t)h * a.sh + c;
    const int64_t ko = s.row * a.ksb + t * a.kst + c;
    const int64_t fo = s.row * a.fsb + t * a.fst + (int64_t)h * a.fsh + c;
    const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k);
    const float dq = a.dqf[fo], dk = a.dkf[fo];
    if (COPY) {
        if (a.dq)
            stt(static_cast<T *>(a.dq) + off, dq);
        if (a.dk)
            stt(static_cast<T *>(a.dk) + ko + (int64_t)h * a.ksh, dk);
    }
    return ldt(q + off) * dq - ldt(k + ko + (int64_t)(h / a.khd) * a.ksh) * dk;
}

template <typename T> __global__ void __launch_bounds__(256) block_sums(GateGradArgs a)
{
    const int j = blockIdx.x, h = blockIdx.y, n = blockIdx.z, c = threadIdx.x;
    const Seq s = seq_of(a, n);
    const int64_t p0 = (int64_t)j * DG_TB;
    if (c >= a.D || p0 >= s.len)
        return;
    const int64_t p1 = s.len - p0 < DG_TB ? s.len : p0 + DG_TB;
    if (a.flags && !a.flags[(int64_t)n * a.H + h])
        return;   // done by the chunked form
    float acc = 0.f;
    for (int64_t p = p0; p < p1; ++p)
        acc += term<T, false>(a, s, h, p, c);
    a.bsum[(((int64_t)n * a.H + h) * a.nblk + j) * a.D + c] = acc;
}

template <typename T> __global__ void __launch_bounds__(256) block_scan(GateGradArgs a)
{
    const int j = blockIdx.x, h = blockIdx.y, n = blockIdx.z, c = threadIdx.x;
    const Seq s = seq_of(a, n);
    const int64_t p0 = (int64_t)j * DG_TB;
    if (c >= a.D || p0 >= s.len)
        return;
    const int64_t p1 = s.len - p0 < DG_TB ? s.len : p0 + DG_TB;
    if (a.flags && !a.flags[(int64_t)n * a.H + h])
        return;   // done by the chunked form
    // the final-state term: sum_e F[c][e] dF[c][e]; F is stored transposed
    const int64_t sidx = ((int64_t)n * a.H + h) * (int64_t)a.D * a.E;
    float acc = 0.f;
    if (a.dF && a.Ft)
        for (int e = 0; e < a.E; ++e)
            acc += a.Ft[sidx + (int64_t)e * a.D + c] * a.dF[sidx + (int64_t)c * a.E + e];
    const int nb = (int)((s.len + DG_TB - 1) / DG_TB);
    const float *bs = a.bsum + ((int64_t)n * a.H + h) * a.nblk * a.D + c;
    for (int jj = j + 1; jj < nb; ++jj)
        acc += bs[(int64_t)jj * a.D];
    for (int64_t p = p1 - 1; p >= p0; --p) {
        acc += (a.dq || a.dk) ? term<T, true>(a, s, h, p, c) : term<T, false>(a, s, h, p, c);
        const int64_t t = s.bos + (a.reverse ? s.len - 1 - p : p);
        a.dg[s.row * a.gsb + t * a.gst + (int64_t)h * a.gsh + c] = acc;
    }
}

// One thread per (sequence, head, channel): the offsets of the sequence's
// segments, walked from the one processed last (whose offset is the final
// state's term) to the one processed first.
__global__ void __launch_bounds__(256) split_dg_offsets(SplitDgArgs a)
{
    const int n = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
    if (c >= a.D)
        return;
    float carry = 0.f;
    if (a.dF && a.Ft) {
        const int64_t sidx = ((int64_t)n * a.H + h) * (int64_t)a.D * a.E;
        for (int e = 0; e < a.E; ++e)
            carry += a.Ft[sidx + (int64_t)e * a.D + c] * a.dF[sidx + (int64_t)c * a.E + e];
    }
    const int first = a.seq_first[n], count = a.seq_first[n + 1] - first;
    for (int j = 0; j < count; ++j) {
        // processing order: ascending segments going forward, descending in
        // reverse; walked here from the last processed
        const int seg = first + (a.reverse ? j : count - 1 - j);
        const int64_t sh = (int64_t)seg * a.H + h;
        a.off[sh * a.D + c] = carry;
        float tot = 0.f;
        if (a.flags[sh]) {
            const int64_t len = (int64_t)a.seg_cu[seg + 1] - a.seg_cu[seg];
            const int nb = (int)((len + DG_TB - 1) / DG_TB);
            for (int b = 0; b < nb && b < a.nblk; ++b)
                tot += a.bsum[(sh * a.nblk + b) * a.D + c];
        } else {
            tot = a.segtot[sh * a.D + c];
        }
        carry += tot;
    }
}

// Grid (segment, head, slice of DG_TB tokens); thread = channel, one token
// at a time (any strides).
__global__ void __launch_bounds__(256) split_dg_add(SplitDgArgs a)
{
    const int seg = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
    if (c >= a.D)
        return;
    const int64_t t0 = a.seg_cu[seg] + (int64_t)blockIdx.z * DG_TB, t1 = a.seg_cu[seg + 1];
    if (t0 >= t1)
        return;
    const float o = a.off[((int64_t)seg * a.H + h) * a.D + c];
    float *p = a.dg + (int64_t)h * a.gsh + c;
    const int64_t te = t1 - t0 < DG_TB ? t1 : t0 + DG_TB;
#pragma unroll 8
    for (int64_t t = t0; t < te; ++t)
        p[t * a.gst] += o;
}

// The same with four channels per thread (16-byte aligned rows, D % 4 == 0):
// thread (token lane, channel quad) walks the slice's tokens DG_TB / TL at a
// time apart.
constexpr int TL = 4;   // token lanes per CTA
__global__ void __launch_bounds__(256) split_dg_add4(SplitDgArgs a)
{
    const int seg = blockIdx.x, h = blockIdx.y;
    const int D4 = a.D / 4, q = (int)threadIdx.x % D4, lane = (int)threadIdx.x / D4;
    if (lane >= TL)
        return;
    const int64_t t0 = a.seg_cu[seg] + (int64_t)blockIdx.z * DG_TB, t1 = a.seg_cu[seg + 1];
    if (t0 >= t1)
        return;
    const float4 o =
        *reinterpret_cast<const float4 *>(a.off + ((int64_t)seg * a.H + h) * a.D + 4 * q);
    float *p = a.dg + (int64_t)h * a.gsh + 4 * q;
    const int64_t te = t1 - t0 < DG_TB ? t1 : t0 + DG_TB;
#pragma unroll 4
    for (int64_t t = t0 + lane; t < te; t += TL) {
        float4 *x = reinterpret_cast<float4 *>(p + t * a.gst);
        float4 v = *x;
        v.x += o.x;
        v.y += o.y;
        v.z += o.z;
        v.w += o.w;
        *x = v;
    }
}

}  // namespace

cudaError_t split_dg(const SplitDgArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.NS == 0 || a.H == 0)
        return cudaSuccess;
    if (a.D > 256 || a.N > 65535 || a.NS > 0x7fffffff || a.H > 65535)
        return cudaErrorNotSupported;
    const int threads = (a.D + 31) / 32 * 32;
    split_dg_offsets<<<dim3((unsigned)a.N, (unsigned)a.H), threads, 0, s>>>(a);
    note_launch();
    // the longest segment's tokens in DG_TB slices
    const int64_t slices = (a.max_seg_len + DG_TB - 1) / DG_TB;
    if (slices < 1 || slices > 65535)
        return cudaErrorNotSupported;
    const dim3 grid((unsigned)a.NS, (unsigned)a.H, (unsigned)slices);
    const bool vec = a.D % 4 == 0 && a.D / 4 * TL <= 256 && a.gst % 4 == 0 && a.gsh % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(a.dg) & 15) == 0;
    if (vec)
        split_dg_add4<<<grid, a.D / 4 * TL, 0, s>>>(a);
    else
        split_dg_add<<<grid, threads, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t gate_grad(const GateGradArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0 || a.nblk == 0)
        return cudaSuccess;
    if (a.D > 256 || a.N > 65535 || a.H > 65535 || a.nblk > 0x7fffffff || a.khd < 1)
        return cudaErrorNotSupported;
    dim3 grid((unsigned)a.nblk, (unsigned)a.H, (unsigned)a.N);
    const int threads = (a.D + 31) / 32 * 32;
    if (a.bf16) {
        block_sums<__nv_bfloat16><<<grid, threads, 0, s>>>(a);
        note_launch();
        block_scan<__nv_bfloat16><<<grid, threads, 0, s>>>(a);
    } else {
        block_sums<float><<<grid, threads, 0, s>>>(a);
        note_launch();
        block_scan<float><<<grid, threads, 0, s>>>(a);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
