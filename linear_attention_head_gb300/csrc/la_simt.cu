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
// fallback sizes).

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
template <typename T>
__device__ void load_chunk(const SweepArgs &a, const Seq &sq, int h, int64_t t0, int Lc,
                           int e0, int ew, float *Qs, float *Ks, float *Vs, int DP)
{
    const int D = a.D;
    for (int idx = threadIdx.x; idx < SC * D; idx += SNT) {
        const int i = idx / D, c = idx % D;
        float qv = 0.f, kv = 0.f;
        if (i < Lc) {
            qv = ldf(tok<T>(a.q, sq.row, sq.bos + t0 + i, h) + c);
            kv = ldf(tok<T>(a.k, sq.row, sq.bos + t0 + i, h) + c);
        }
        Qs[i * DP + c] = qv;
        Ks[i * DP + c] = kv;
    }
    for (int idx = threadIdx.x; idx < SC * SET; idx += SNT) {
        const int i = idx / SET, c = idx % SET;
        float vv = 0.f;
        if (i < Lc && c < ew)
            vv = ldf(tok<T>(a.v, sq.row, sq.bos + t0 + i, h) + e0 + c);
        Vs[i * (SET + 1) + c] = vv;
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
        // decay-masked scores P[i][j] = s (q_i . k_j) gamma^(p(i)-p(j)), p(j) <= p(i)
        for (int idx = threadIdx.x; idx < SC * SC; idx += SNT) {
            const int i = idx / SC, j = idx % SC;
            const int pi = a.reverse ? Lc - 1 - i : i, pj = a.reverse ? Lc - 1 - j : j;
            float val = 0.f;
            if (i < Lc && j < Lc && pj <= pi) {
                float acc = 0.f;
                for (int c2 = 0; c2 < D; ++c2)
                    acc = fmaf(Qs[i * DP + c2], Ks[j * DP + c2], acc);
                val = a.scale * acc * pw[pi - pj];
            }
            Ps[i * (SC + 1) + j] = val;
        }
        __syncthreads();
        // out_i = sum_j P[i][j] v_j + s gamma^(p(i)+1) q_i^T S
        for (int idx = threadIdx.x; idx < SC * SET; idx += SNT) {
            const int i = idx / SET, b = idx % SET;
            if (i >= Lc || b >= ew)
                continue;
            float intra = 0.f, inter = 0.f;
            for (int j = 0; j < SC; ++j)
                intra = fmaf(Ps[i * (SC + 1) + j], Vs[j * (SET + 1) + b], intra);
            for (int r = 0; r < D; ++r)
                inter = fmaf(Qs[i * DP + r], Ss[r * SET + b], inter);
            const int pi = a.reverse ? Lc - 1 - i : i;
            stf(tok<T>(a.out, sq.row, sq.bos + t0 + i, h) + e0 + b,
                intra + a.scale * pw[pi + 1] * inter);
        }
        __syncthreads();
        // S = gamma^Lc S + sum_j gamma^(Lc-1-p(j)) k_j v_j^T
        for (int idx = threadIdx.x; idx < D * SET; idx += SNT) {
            const int r = idx / SET, b = idx % SET;
            float acc = 0.f;
            for (int j = 0; j < Lc; ++j) {
                const int pj = a.reverse ? Lc - 1 - j : j;
                acc = fmaf(pw[Lc - 1 - pj] * Ks[j * DP + r], Vs[j * (SET + 1) + b], acc);
            }
            Ss[idx] = fmaf(pw[Lc], Ss[idx], acc);
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
        for (int idx = threadIdx.x; idx < SC * SC; idx += SNT) {
            const int j = idx / SC, i = idx % SC;
            const int pi = a.reverse ? Lc - 1 - i : i, pj = a.reverse ? Lc - 1 - j : j;
            float val = 0.f;
            if (i < Lc && j < Lc && pj <= pi) {
                float acc = 0.f;
                for (int c2 = 0; c2 < D; ++c2)
                    acc = fmaf(Qs[i * DP + c2], Ks[j * DP + c2], acc);
                val = a.scale * acc * pw[pi - pj];
            }
            Ps[j * (SC + 1) + i] = val;
        }
        __syncthreads();
        // out_j = sum_i P[j][i] w_i + gamma^(Lc-1-p(j)) G^T k_j
        for (int idx = threadIdx.x; idx < SC * SET; idx += SNT) {
            const int j = idx / SET, b = idx % SET;
            if (j >= Lc || b >= ew)
                continue;
            float intra = 0.f, inter = 0.f;
            for (int i = 0; i < SC; ++i)
                intra = fmaf(Ps[j * (SC + 1) + i], Ws[i * (SET + 1) + b], intra);
            for (int r = 0; r < D; ++r)
                inter = fmaf(Ks[j * DP + r], Gs[r * SET + b], inter);
            const int pj = a.reverse ? Lc - 1 - j : j;
            stf(tok<T>(a.out, sq.row, sq.bos + t0 + j, h) + e0 + b,
                intra + pw[Lc - 1 - pj] * inter);
        }
        __syncthreads();
        // G = gamma^Lc G + s sum_i gamma^(p(i)+1) q_i w_i^T
        for (int idx = threadIdx.x; idx < D * SET; idx += SNT) {
            const int r = idx / SET, b = idx % SET;
            float acc = 0.f;
            for (int i = 0; i < Lc; ++i) {
                const int pi = a.reverse ? Lc - 1 - i : i;
                acc = fmaf(pw[pi + 1] * Qs[i * DP + r], Ws[i * (SET + 1) + b], acc);
            }
            Gs[idx] = fmaf(pw[Lc], Gs[idx], a.scale * acc);
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
