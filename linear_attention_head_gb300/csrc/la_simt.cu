// la_simt.cu -- CUDA-core chunked kernels for decayed causal linear attention.
//
// These handle every case the tensor-core kernels do not: fp32 token tensors
// (where a 1e-4 relative bound rules out bf16/tf32 tensor-core operands), head
// dims the tensor-core kernels do not take, and unaligned layouts.  They
// evaluate the chunked (Lightning Attention-2) form in fp32 FFMA: per chunk of
// SC tokens an intra-chunk decay-masked score block and an inter-chunk carried
// state (the state-update formula of the ejkernel `recurrent` docstring,
// unrolled over a chunk).
//
// One CTA owns one (sequence, head, value-tile); the state tile (D x SET fp32)
// stays in shared memory for the whole sequence.  The score block is
// recomputed by each value tile (cheap next to the state work for these
// fallback sizes).  The chunk's three loops are register-blocked: thread t
// takes row t / 8 of a 32-row block and the 8 columns t % 8 + 8 m (m < 8) of
// the 64-column value tile (scores: 4 adjacent keys), so each shared-memory
// row value it loads feeds 4 or 8 independent accumulators; one accumulator
// per thread left every loop waiting on the previous load and FMA.

#include <cuda_bf16.h>
#include "la_internal.h"

namespace la {
namespace {

constexpr int SC = 32;    // tokens per chunk
constexpr int SET = 64;   // value channels per CTA
constexpr int SNT = 256;  // threads per CTA

template <typename T> __device__ __forceinline__ float ldf(const T *p);
template <> __device__ __forceinline__ float ldf<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void stf(T *p, float x);
template <> __device__ __forceinline__ void stf<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, float x)
{
    *p = __float2bfloat16_rn(x);
}

struct Seq {
    int64_t row, bos, len;
};

__device__ __forceinline__ Seq seq_of(const SweepArgs &a, int n)
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

template <typename T>
__device__ __forceinline__ const T *tok(const Tok &t, int64_t row, int64_t tkn, int h)
{
    return reinterpret_cast<const T *>(t.p) + row * t.sb + tkn * t.st +
           (int64_t)(h / t.hdiv) * t.sh;
}
template <typename T>
__device__ __forceinline__ T *tok(const TokOut &t, int64_t row, int64_t tkn, int h)
{
    return reinterpret_cast<T *>(t.p) + row * t.sb + tkn * t.st + (int64_t)h * t.sh;
}

// Shared-memory carve-up (floats): Qs[SC][D+1], Ks[SC][D+1], Vs[SC][SET+1],
// Ss[D][SET], Ps[SC][SC+1], pw[SC+1].
__host__ __device__ inline size_t simt_smem_floats(int D)
{
    return (size_t)2 * SC * (D + 1) + (size_t)SC * (SET + 1) + (size_t)D * SET +
           (size_t)SC * (SC + 1) + (SC + 1);
}

__device__ __forceinline__ int chunk_len(int64_t len, int64_t t0)
{
    return (int)(len - t0 < SC ? len - t0 : SC);
}

// Loads the chunk rows [t0, t0+Lc) of q, k (all D) and of the third tensor's
// value tile [e0, e0+ew) into shared memory as fp32; rows >= Lc are zeroed.
// Each thread issues its loads in batches of 8 before storing any, so that a
// chunk waits for a few global-memory round trips instead of one per element.
template <typename T>
__device__ void load_chunk(const SweepArgs &a, const Seq &sq, int h, int64_t t0, int Lc,
                           int e0, int ew, float *Qs, float *Ks, float *Vs, int DP)
{
    const int D = a.D;
    constexpr int LB = 8;
    for (int base = threadIdx.x; base < SC * D; base += LB * SNT) {
        float qv[LB], kv[LB];
#pragma unroll
        for (int u = 0; u < LB; ++u) {
            const int idx = base + u * SNT, i = idx / D, c = idx % D;
            qv[u] = kv[u] = 0.f;
            if (idx < SC * D && i < Lc) {
                qv[u] = ldf(tok<T>(a.q, sq.row, sq.bos + t0 + i, h) + c);
                kv[u] = ldf(tok<T>(a.k, sq.row, sq.bos + t0 + i, h) + c);
            }
        }
#pragma unroll
        for (int u = 0; u < LB; ++u) {
            const int idx = base + u * SNT, i = idx / D, c = idx % D;
            if (idx < SC * D) {
                Qs[i * DP + c] = qv[u];
                Ks[i * DP + c] = kv[u];
            }
        }
    }
    for (int base = threadIdx.x; base < SC * SET; base += LB * SNT) {
        float vv[LB];
#pragma unroll
        for (int u = 0; u < LB; ++u) {
            const int idx = base + u * SNT, i = idx / SET, c = idx % SET;
            vv[u] = 0.f;
            if (idx < SC * SET && i < Lc && c < ew)
                vv[u] = ldf(tok<T>(a.v, sq.row, sq.bos + t0 + i, h) + e0 + c);
        }
#pragma unroll
        for (int u = 0; u < LB; ++u) {
            const int idx = base + u * SNT, i = idx / SET, c = idx % SET;
            if (idx < SC * SET)
                Vs[i * (SET + 1) + c] = vv[u];
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(SNT) simt_forward_kernel(SweepArgs a)
{
    const int n = a.order ? a.order[blockIdx.x] : (int)blockIdx.x;
    const int h = blockIdx.y, e0 = blockIdx.z * SET;
    const int D = a.D, DP = D + 1, ew = min(SET, a.E - e0);
    const Seq sq = seq_of(a, n);
    extern __shared__ float sm[];
    float *Qs = sm;
    float *Ks = Qs + SC * DP;
    float *Vs = Ks + SC * DP;
    float *Ss = Vs + SC * (SET + 1);
    float *Ps = Ss + D * SET;
    float *pw = Ps + SC * (SC + 1);
    const float g = a.g[h];
    const int64_t sbase = ((int64_t)n * a.H + h) * (int64_t)a.D * a.E;

    for (int idx = threadIdx.x; idx < D * SET; idx += SNT) {
        const int r = idx / SET, c = idx % SET;
        float x = 0.f;
        if (a.s_in.p && c < ew)
            x = a.s_in.p[sbase + r * a.s_in.rs + (e0 + c) * a.s_in.cs];
        Ss[idx] = x;
    }
    if (threadIdx.x <= SC)
        pw[threadIdx.x] = threadIdx.x == 0 ? 1.f : expf(g * (float)threadIdx.x);

    const int64_t nc = (sq.len + SC - 1) / SC;
    for (int64_t cc = 0; cc < nc; ++cc) {
        const int64_t c = a.reverse ? nc - 1 - cc : cc;
        const int64_t t0 = c * SC;
        const int Lc = chunk_len(sq.len, t0);
        __syncthreads();
        load_chunk<T>(a, sq, h, t0, Lc, e0, ew, Qs, Ks, Vs, DP);
        __syncthreads();
        // decay-masked scores P[i][j] = s (q_i . k_j) gamma^(p(i)-p(j)), p(j) <= p(i):
        // row i = t / 8, keys 4 (t % 8) .. + 3
        {
            const int i = threadIdx.x >> 3, j0 = 4 * (threadIdx.x & 7);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c2 = 0; c2 < D; ++c2) {
                const float qv = Qs[i * DP + c2];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    acc[u] = fmaf(qv, Ks[(j0 + u) * DP + c2], acc[u]);
            }
            const int pi = a.reverse ? Lc - 1 - i : i;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u, pj = a.reverse ? Lc - 1 - j : j;
                Ps[i * (SC + 1) + j] =
                    i < Lc && j < Lc && pj <= pi ? a.scale * acc[u] * pw[pi - pj] : 0.f;
            }
        }
        __syncthreads();
        // out_i = sum_j P[i][j] v_j + s gamma^(p(i)+1) q_i^T S: row i = t / 8,
        // columns t % 8 + 8 m
        {
            const int i = threadIdx.x >> 3, b0 = threadIdx.x & 7;
            float intra[8], inter[8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
                intra[m] = inter[m] = 0.f;
            for (int j = 0; j < SC; ++j) {
                const float pv = Ps[i * (SC + 1) + j];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    intra[m] = fmaf(pv, Vs[j * (SET + 1) + b0 + 8 * m], intra[m]);
            }
            for (int r = 0; r < D; ++r) {
                const float qv = Qs[i * DP + r];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    inter[m] = fmaf(qv, Ss[r * SET + b0 + 8 * m], inter[m]);
            }
            if (i < Lc) {
                const int pi = a.reverse ? Lc - 1 - i : i;
                const float f = a.scale * pw[pi + 1];
                T *orow = tok<T>(a.out, sq.row, sq.bos + t0 + i, h) + e0;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (b0 + 8 * m < ew)
                        stf(orow + b0 + 8 * m, intra[m] + f * inter[m]);
            }
        }
        __syncthreads();
        // S = gamma^Lc S + sum_j gamma^(Lc-1-p(j)) k_j v_j^T: rows t / 8 + 32 rr,
        // columns t % 8 + 8 m
        for (int r = threadIdx.x >> 3; r < D; r += SNT / 8) {
            const int b0 = threadIdx.x & 7;
            float acc[8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
                acc[m] = 0.f;
            for (int j = 0; j < Lc; ++j) {
                const int pj = a.reverse ? Lc - 1 - j : j;
                const float kv = pw[Lc - 1 - pj] * Ks[j * DP + r];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    acc[m] = fmaf(kv, Vs[j * (SET + 1) + b0 + 8 * m], acc[m]);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                float *sp = Ss + r * SET + b0 + 8 * m;
                *sp = fmaf(pw[Lc], *sp, acc[m]);
            }
        }
    }
    __syncthreads();
    if (a.s_out.p) {
        for (int idx = threadIdx.x; idx < D * SET; idx += SNT) {
            const int r = idx / SET, c = idx % SET;
            if (c < ew)
                a.s_out.p[sbase + r * a.s_out.rs + (e0 + c) * a.s_out.cs] = Ss[idx];
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(SNT) simt_backward_kernel(SweepArgs a)
{
    const int n = a.order ? a.order[blockIdx.x] : (int)blockIdx.x;
    const int h = blockIdx.y, e0 = blockIdx.z * SET;
    const int D = a.D, DP = D + 1, ew = min(SET, a.E - e0);
    const Seq sq = seq_of(a, n);
    extern __shared__ float sm[];
    float *Qs = sm;
    float *Ks = Qs + SC * DP;
    float *Ws = Ks + SC * DP;           // the upstream-gradient tile (do)
    float *Gs = Ws + SC * (SET + 1);    // dL/dS tile
    float *Ps = Gs + D * SET;           // Ps[j][i]: weight of token i on token j
    float *pw = Ps + SC * (SC + 1);
    const float g = a.g[h];
    const int64_t sbase = ((int64_t)n * a.H + h) * (int64_t)a.D * a.E;

    for (int idx = threadIdx.x; idx < D * SET; idx += SNT) {
        const int r = idx / SET, c = idx % SET;
        float x = 0.f;
        if (a.s_in.p && c < ew)
            x = a.s_in.p[sbase + r * a.s_in.rs + (e0 + c) * a.s_in.cs];
        Gs[idx] = x;
    }
    if (threadIdx.x <= SC)
        pw[threadIdx.x] = threadIdx.x == 0 ? 1.f : expf(g * (float)threadIdx.x);

    const int64_t nc = (sq.len + SC - 1) / SC;
    for (int64_t cc = 0; cc < nc; ++cc) {
        // against processing order
        const int64_t c = a.reverse ? cc : nc - 1 - cc;
        const int64_t t0 = c * SC;
        const int Lc = chunk_len(sq.len, t0);
        __syncthreads();
        load_chunk<T>(a, sq, h, t0, Lc, e0, ew, Qs, Ks, Ws, DP);
        __syncthreads();
        // Ps[j][i] = s (q_i . k_j) gamma^(p(i)-p(j)), p(j) <= p(i): key row
        // j = t / 8, queries 4 (t % 8) .. + 3
        {
            const int j = threadIdx.x >> 3, i0 = 4 * (threadIdx.x & 7);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c2 = 0; c2 < D; ++c2) {
                const float kv = Ks[j * DP + c2];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    acc[u] = fmaf(Qs[(i0 + u) * DP + c2], kv, acc[u]);
            }
            const int pj = a.reverse ? Lc - 1 - j : j;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u, pi = a.reverse ? Lc - 1 - i : i;
                Ps[j * (SC + 1) + i] =
                    i < Lc && j < Lc && pj <= pi ? a.scale * acc[u] * pw[pi - pj] : 0.f;
            }
        }
        __syncthreads();
        // out_j = sum_i P[j][i] w_i + gamma^(Lc-1-p(j)) G^T k_j: row j = t / 8,
        // columns t % 8 + 8 m
        {
            const int j = threadIdx.x >> 3, b0 = threadIdx.x & 7;
            float intra[8], inter[8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
                intra[m] = inter[m] = 0.f;
            for (int i = 0; i < SC; ++i) {
                const float pv = Ps[j * (SC + 1) + i];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    intra[m] = fmaf(pv, Ws[i * (SET + 1) + b0 + 8 * m], intra[m]);
            }
            for (int r = 0; r < D; ++r) {
                const float kv = Ks[j * DP + r];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    inter[m] = fmaf(kv, Gs[r * SET + b0 + 8 * m], inter[m]);
            }
            if (j < Lc) {
                const int pj = a.reverse ? Lc - 1 - j : j;
                const float f = pw[Lc - 1 - pj];
                T *orow = tok<T>(a.out, sq.row, sq.bos + t0 + j, h) + e0;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (b0 + 8 * m < ew)
                        stf(orow + b0 + 8 * m, intra[m] + f * inter[m]);
            }
        }
        __syncthreads();
        // G = gamma^Lc G + s sum_i gamma^(p(i)+1) q_i w_i^T: rows t / 8 + 32 rr,
        // columns t % 8 + 8 m
        for (int r = threadIdx.x >> 3; r < D; r += SNT / 8) {
            const int b0 = threadIdx.x & 7;
            float acc[8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
                acc[m] = 0.f;
            for (int i = 0; i < Lc; ++i) {
                const int pi = a.reverse ? Lc - 1 - i : i;
                const float qv = pw[pi + 1] * Qs[i * DP + r];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    acc[m] = fmaf(qv, Ws[i * (SET + 1) + b0 + 8 * m], acc[m]);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                float *gp = Gs + r * SET + b0 + 8 * m;
                *gp = fmaf(pw[Lc], *gp, a.scale * acc[m]);
            }
        }
    }
    __syncthreads();
    if (a.s_out.p) {
        for (int idx = threadIdx.x; idx < D * SET; idx += SNT) {
            const int r = idx / SET, c = idx % SET;
            if (c < ew)
                a.s_out.p[sbase + r * a.s_out.rs + (e0 + c) * a.s_out.cs] = Gs[idx];
        }
    }
}

template <typename K>
cudaError_t launch(K kernel, const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0)
        return cudaSuccess;
    const size_t smem = simt_smem_floats(a.D) * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess)
        return err;
    dim3 grid(a.N, a.H, (a.E + SET - 1) / SET);
    kernel<<<grid, SNT, smem, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t simt_forward_sweep(const SweepArgs &a, cudaStream_t s)
{
    return a.bf16 ? launch(simt_forward_kernel<__nv_bfloat16>, a, s)
                  : launch(simt_forward_kernel<float>, a, s);
}

cudaError_t simt_backward_sweep(const SweepArgs &a, cudaStream_t s)
{
    return a.bf16 ? launch(simt_backward_kernel<__nv_bfloat16>, a, s)
                  : launch(simt_backward_kernel<float>, a, s);
}

}  // namespace la
