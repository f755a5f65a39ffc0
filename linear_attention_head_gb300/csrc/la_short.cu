// la_short.cu -- token-by-token kernels for short sequences: decoding a few
// new tokens against a carried state, or any call whose longest sequence has
// at most SHORT_MAX_T tokens.
//
// They run the recurrence itself (ejkernel `recurrent` docstring, "The core
// update") one token at a time instead of the chunked form, because a chunk
// of 128 tokens holding 1..16 valid ones costs the chunked kernels' whole
// pipeline fill for almost no work.  One CTA per (sequence, head, 32 value
// columns); the sequence's tokens are copied into shared memory first, then
// each thread carries 16 rows of one value column of the fp32 state in
// registers (read once, written once) and runs, per token,
//   forward-type:  S <- gamma S + k_t v_t^T,  out_t = s q_t^T S
//   backward-type: G <- G + s q_t w_t^T,      out_t = G^T k_t,  G <- gamma G
// (the two shapes of la_internal.h, visited in the same token order as the
// chunked kernels).  A column's dot product over its D rows is summed over
// its row groups with lane shuffles; the token loop has no barrier.  fp32
// arithmetic for both token dtypes.

#include <cstdint>

#include <cuda_bf16.h>
#include "la_internal.h"

namespace la {
namespace {

constexpr int KW = 32;   // value columns per CTA
constexpr int RP = 16;   // state rows per thread
constexpr int MAXG = 16; // D <= 256: at most 16 row groups

template <typename T> __device__ __forceinline__ float ld_tok(const T *p);
template <> __device__ __forceinline__ float ld_tok<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld_tok<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st_tok(T *p, float x);
template <> __device__ __forceinline__ void st_tok<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void st_tok<__nv_bfloat16>(__nv_bfloat16 *p, float x)
{
    *p = __float2bfloat16_rn(x);
}

// Threads per CTA: 32 value columns x G row groups of RP state rows each,
// G = D/RP rounded up to a power of two (1 .. 16).
__host__ __device__ inline int short_groups(int D)
{
    int g = 1;
    while (RP * g < D)
        g *= 2;
    return g;
}

// Dynamic shared memory (floats): q and k of every token [max_len][20 G]
// (row group g at offset 20 g: the groups that a quarter warp reads at once
// fall in different banks; rows past D zero), and the CTA's 32 value columns
// of every token [max_len][32].
__host__ __device__ inline size_t short_smem_bytes(int max_len, int D)
{
    return ((size_t)2 * max_len * 20 * short_groups(D) + (size_t)max_len * KW) * sizeof(float);
}

template <typename T, bool BWD>
__global__ void __launch_bounds__(KW * MAXG) short_kernel(SweepArgs a)
{
    const int etiles = (a.E + KW - 1) / KW;
    const int e0 = (int)(blockIdx.x % etiles) * KW;
    const int h = (int)((blockIdx.x / etiles) % a.H);
    const int n = (int)(blockIdx.x / ((unsigned)etiles * a.H));
    const int D = a.D, G = short_groups(D), DP = RP * G, DPP = 20 * G;
    // thread = (column c, row group g) with g in the low bits, so that the
    // G partial dot products of a column sit in neighbouring lanes
    const int g = threadIdx.x & (G - 1), c = threadIdx.x / G;
    const int r0 = RP * g;
    const bool col_ok = e0 + c < a.E;
    extern __shared__ float sh[];

    int64_t row, bos, len;
    if (a.cu) {
        row = 0;
        bos = a.cu[n];
        len = (int64_t)a.cu[n + 1] - a.cu[n];
    } else {
        row = n;
        bos = 0;
        len = a.T;
    }
    const int L = (int)len;   // <= max_len <= SHORT_MAX_T
    float *qs = sh;
    float *ks = qs + (size_t)a.max_len * DPP;
    float *ws = ks + (size_t)a.max_len * DPP;
    // forward-type visits tokens in processing order, backward-type against it
    const bool flip = (a.reverse != 0) != BWD;
    auto token = [&](int u) { return bos + (flip ? len - 1 - u : u); };

    const float gam = expf(a.g[h]);
    const float scale = a.scale;
    const int64_t sbase = ((int64_t)n * a.H + h) * (int64_t)D * a.E;
    // S[j] = state(r0 + j, e0 + c); these loads are in flight while the
    // tokens are copied below
    float S[RP];
#pragma unroll
    for (int j = 0; j < RP; ++j)
        S[j] = a.s_in.p && col_ok && r0 + j < D
                   ? a.s_in.p[sbase + (int64_t)(r0 + j) * a.s_in.rs + (int64_t)(e0 + c) * a.s_in.cs]
                   : 0.f;
    // every token of the sequence into shared memory, in visiting order; the
    // loads of a thread are issued PF at a time before any is used, so the
    // copy pays a few memory latencies instead of one per element
    constexpr int PF = 8;
    const int nqk = L * DP, nthr = blockDim.x;
    for (int base = threadIdx.x; base < nqk; base += PF * nthr) {
        float xq[PF], xk[PF];
#pragma unroll
        for (int i = 0; i < PF; ++i) {
            const int idx = base + i * nthr, u = idx / DP, k = idx % DP;
            xq[i] = xk[i] = 0.f;
            if (idx < nqk && k < D) {
                const int64_t t = token(u);
                xq[i] = ld_tok(reinterpret_cast<const T *>(a.q.p) + row * a.q.sb + t * a.q.st +
                               (int64_t)(h / a.q.hdiv) * a.q.sh + k);
                xk[i] = ld_tok(reinterpret_cast<const T *>(a.k.p) + row * a.k.sb + t * a.k.st +
                               (int64_t)(h / a.k.hdiv) * a.k.sh + k);
            }
        }
#pragma unroll
        for (int i = 0; i < PF; ++i) {
            const int idx = base + i * nthr, u = idx / DP, k = idx % DP;
            if (idx < nqk) {
                qs[u * DPP + k + 4 * (k / RP)] = xq[i];
                ks[u * DPP + k + 4 * (k / RP)] = xk[i];
            }
        }
    }
    const int nw = L * KW;
    for (int base = threadIdx.x; base < nw; base += PF * nthr) {
        float xw[PF];
#pragma unroll
        for (int i = 0; i < PF; ++i) {
            const int idx = base + i * nthr, u = idx / KW, k = idx % KW;
            xw[i] = 0.f;
            if (idx < nw && e0 + k < a.E)
                xw[i] = ld_tok(reinterpret_cast<const T *>(a.v.p) + row * a.v.sb +
                               token(u) * a.v.st + (int64_t)(h / a.v.hdiv) * a.v.sh + e0 + k);
        }
#pragma unroll
        for (int i = 0; i < PF; ++i) {
            const int idx = base + i * nthr;
            if (idx < nw)
                ws[idx] = xw[i];
        }
    }

    __syncthreads();

    for (int u = 0; u < L; ++u) {
        const float4 *q4 = reinterpret_cast<const float4 *>(qs + u * DPP + 20 * g);
        const float4 *k4 = reinterpret_cast<const float4 *>(ks + u * DPP + 20 * g);
        const float w = ws[u * KW + c];
        float dot[4] = {0.f, 0.f, 0.f, 0.f};   // four chains, summed at the end
#pragma unroll
        for (int j4 = 0; j4 < RP / 4; ++j4) {
            const float4 xq = q4[j4], xk = k4[j4];
            const float qv[4] = {xq.x, xq.y, xq.z, xq.w};
            const float kv[4] = {xk.x, xk.y, xk.z, xk.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float &x = S[4 * j4 + i];
                if (!BWD) {
                    x = fmaf(kv[i], w, gam * x);
                    dot[i] = fmaf(qv[i], x, dot[i]);
                } else {
                    x = fmaf(scale * qv[i], w, x);
                    dot[i] = fmaf(kv[i], x, dot[i]);
                    x *= gam;
                }
            }
        }
        float dsum = (dot[0] + dot[1]) + (dot[2] + dot[3]);
        for (int off = 1; off < G; off <<= 1)
            dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
        if (g == 0 && col_ok) {
            T *op = reinterpret_cast<T *>(a.out.p) + row * a.out.sb + token(u) * a.out.st +
                    (int64_t)h * a.out.sh;
            st_tok(op + e0 + c, BWD ? dsum : scale * dsum);
        }
    }

    if (a.s_out.p && col_ok) {
#pragma unroll
        for (int j = 0; j < RP; ++j)
            if (r0 + j < D)
                a.s_out.p[sbase + (int64_t)(r0 + j) * a.s_out.rs + (int64_t)(e0 + c) * a.s_out.cs] =
                    S[j];
    }
}

template <typename K> cudaError_t launch_one(K kernel, const SweepArgs &a, cudaStream_t s)
{
    const size_t smem = short_smem_bytes((int)a.max_len, a.D);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int64_t blocks = (int64_t)a.N * a.H * ((a.E + KW - 1) / KW);
    const int threads = KW * short_groups(a.D);
    kernel<<<(unsigned)blocks, threads, smem, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

template <bool BWD> cudaError_t launch_short(const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0)
        return cudaSuccess;
    if (a.D < 1 || a.D > RP * MAXG || a.max_len < 0 || a.max_len > SHORT_MAX_T)
        return cudaErrorNotSupported;
    if ((int64_t)a.N * a.H * ((a.E + KW - 1) / KW) > 0x7fffffff)
        return cudaErrorNotSupported;
    return a.bf16 ? launch_one(short_kernel<__nv_bfloat16, BWD>, a, s)
                  : launch_one(short_kernel<float, BWD>, a, s);
}

}  // namespace

cudaError_t short_forward_sweep(const SweepArgs &a, cudaStream_t s)
{
    return launch_short<false>(a, s);
}

cudaError_t short_backward_sweep(const SweepArgs &a, cudaStream_t s)
{
    return launch_short<true>(a, s);
}

}  // namespace la
