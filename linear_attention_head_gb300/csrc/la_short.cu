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

constexpr int TB = 16;   // tokens per shared-memory block

// Dynamic shared memory (floats) for one block of TB tokens: q, k and the
// row-gate decays [TB][20 G] (row group g at offset 20 g, so that the groups
// a quarter warp reads at once fall in different banks; rows past D zero),
// the CTA's 32 value columns [TB][32] and column-gate decays [TB][32].
// gate < 0: the synchronous path (no raw buffers).
__host__ __device__ inline size_t short_smem_bytes(int D, int esz, int gate)
{
    const size_t layout = ((size_t)3 * TB * 20 * short_groups(D) + (size_t)2 * TB * KW) * 4;
    if (gate < 0)
        return layout;
    // double-buffered raw rows of the asynchronous path: q, k, v tile, gate
    const size_t raw = (size_t)2 * TB * ((size_t)2 * D * esz + (size_t)KW * esz +
                                         (gate == 1 ? (size_t)D * 4 : 0) +
                                         (gate == 2 ? (size_t)KW * 4 : 0));
    return layout + raw;
}

// GATE: 0 the head's decay only, 1 per-row gate (state rows are key
// channels), 2 per-column gate (state columns are key channels).
template <typename T, bool BWD, int GATE, bool ASYNC>
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
    float *qs = sh;
    float *ks = qs + TB * DPP;
    float *as = ks + TB * DPP;   // row-gate decays
    float *ws = as + TB * DPP;
    float *acs = ws + TB * KW;   // column-gate decays
    // forward-type visits tokens in processing order, backward-type against it
    const bool flip = (a.reverse != 0) != BWD;
    auto token = [&](int64_t u) { return bos + (flip ? len - 1 - u : u); };

    const float gh = a.g[h];
    const float gam = expf(gh);
    const float scale = a.scale;
    const int64_t sbase = ((int64_t)n * a.H + h) * (int64_t)D * a.E;
    // token rows of this (sequence, head): key/value heads may be shared
    const T *qb = reinterpret_cast<const T *>(a.q.p) + row * a.q.sb +
                  (int64_t)(h / a.q.hdiv) * a.q.sh;
    const T *kb = reinterpret_cast<const T *>(a.k.p) + row * a.k.sb +
                  (int64_t)(h / a.k.hdiv) * a.k.sh;
    const T *vb = reinterpret_cast<const T *>(a.v.p) + row * a.v.sb +
                  (int64_t)(h / a.v.hdiv) * a.v.sh;
    const float *gb = GATE ? a.gate.p + row * a.gate.sb + (int64_t)h * a.gate.sh : nullptr;
    T *ob = reinterpret_cast<T *>(a.out.p) + row * a.out.sb + (int64_t)h * a.out.sh;

    // S[j] = state(r0 + j, e0 + c); these loads are in flight while the
    // first tokens are copied below
    float S[RP];
#pragma unroll
    for (int j = 0; j < RP; ++j)
        S[j] = a.s_in.p && col_ok && r0 + j < D
                   ? a.s_in.p[sbase + (int64_t)(r0 + j) * a.s_in.rs + (int64_t)(e0 + c) * a.s_in.cs]
                   : 0.f;

    constexpr int PF = 4;
    const int nthr = blockDim.x;

    // one block of Lb tokens from b0 on, copied synchronously into the
    // compute layout; each thread issues PF loads before using any
    auto load_sync = [&](int64_t b0, int Lb) {
        const int nqk = Lb * DP;
        for (int base = threadIdx.x; base < nqk; base += PF * nthr) {
            float xq[PF], xk[PF], xa[PF];
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr, u = idx / DP, k = idx % DP;
                xq[i] = xk[i] = 0.f;
                xa[i] = 1.f;
                if (idx < nqk && k < D) {
                    const int64_t t = token(b0 + u);
                    xq[i] = ld_tok(qb + t * a.q.st + k);
                    xk[i] = ld_tok(kb + t * a.k.st + k);
                    if (GATE == 1)
                        xa[i] = gb[t * a.gate.st + k];
                }
            }
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr, u = idx / DP, k = idx % DP;
                if (idx < nqk) {
                    const int at = u * DPP + k + 4 * (k / RP);
                    qs[at] = xq[i];
                    ks[at] = xk[i];
                    if (GATE == 1)
                        as[at] = k < D ? expf(gh + xa[i]) : 1.f;
                }
            }
        }
        const int nw = Lb * KW;
        for (int base = threadIdx.x; base < nw; base += PF * nthr) {
            float xw[PF], xg[PF];
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr, u = idx / KW, k = idx % KW;
                xw[i] = 0.f;
                xg[i] = 0.f;
                if (idx < nw && e0 + k < a.E) {
                    const int64_t t = token(b0 + u);
                    xw[i] = ld_tok(vb + t * a.v.st + e0 + k);
                    if (GATE == 2)
                        xg[i] = gb[t * a.gate.st + e0 + k];
                }
            }
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr;
                if (idx < nw) {
                    ws[idx] = xw[i];
                    if (GATE == 2)
                        acs[idx] = expf(gh + xg[i]);
                }
            }
        }
    };
    // the per-token recurrence over one block in the compute layout; the
    // partial dot products of four tokens are summed over the row groups
    // together, so that their shuffles overlap
    auto compute = [&](int64_t b0, int Lb) {
        for (int u0 = 0; u0 < Lb; u0 += 4) {
            float pend[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int u = u0 + i;
                if (u >= Lb)
                    break;
                const float4 *q4 = reinterpret_cast<const float4 *>(qs + u * DPP + 20 * g);
                const float4 *k4 = reinterpret_cast<const float4 *>(ks + u * DPP + 20 * g);
                const float4 *a4 = reinterpret_cast<const float4 *>(as + u * DPP + 20 * g);
                const float w = ws[u * KW + c];
                const float ac = GATE == 2 ? acs[u * KW + c] : gam;
                float dot[4] = {0.f, 0.f, 0.f, 0.f};   // four chains, summed at the end
#pragma unroll
                for (int j4 = 0; j4 < RP / 4; ++j4) {
                    const float4 xq = q4[j4], xk = k4[j4];
                    const float qv[4] = {xq.x, xq.y, xq.z, xq.w};
                    const float kv[4] = {xk.x, xk.y, xk.z, xk.w};
                    float dv[4] = {ac, ac, ac, ac};
                    if (GATE == 1) {
                        const float4 xa = a4[j4];
                        dv[0] = xa.x;
                        dv[1] = xa.y;
                        dv[2] = xa.z;
                        dv[3] = xa.w;
                    }
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        float &x = S[4 * j4 + m];
                        if (!BWD) {
                            x = fmaf(kv[m], w, dv[m] * x);
                            dot[m] = fmaf(qv[m], x, dot[m]);
                        } else {
                            x = fmaf(scale * qv[m], w, x);
                            dot[m] = fmaf(kv[m], x, dot[m]);
                            x *= dv[m];
                        }
                    }
                }
                pend[i] = (dot[0] + dot[1]) + (dot[2] + dot[3]);
            }
            for (int off = 1; off < G; off <<= 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    pend[i] += __shfl_xor_sync(0xffffffffu, pend[i], off);
            }
            if (g == 0 && col_ok) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (u0 + i < Lb)
                        st_tok(ob + token(b0 + u0 + i) * a.out.st + e0 + c,
                               BWD ? pend[i] : scale * pend[i]);
            }
        }
    };

    // ASYNC (chosen on the host when every row is 16-byte aligned and the
    // sequences span more than one block): double-buffered asynchronous
    // copies (16-byte cp.async) of the raw rows, the next block's loads in
    // flight while this block is converted and computed.
    const int esz = (int)sizeof(T);
    if (!ASYNC) {
        for (int64_t b0 = 0; b0 < len; b0 += TB) {
            const int Lb = (int)(len - b0 < TB ? len - b0 : TB);
            load_sync(b0, Lb);
            __syncthreads();
            compute(b0, Lb);
            __syncthreads();   // the next block overwrites the buffers
        }
    } else {
        // raw double buffers after the compute layout
        T *rq = reinterpret_cast<T *>(acs + TB * KW);
        T *rk = rq + 2 * TB * D;
        T *rv = rk + 2 * TB * D;
        float *rg = reinterpret_cast<float *>(rv + 2 * TB * KW);   // row gate [2][TB][D]
        float *rgc = rg + (GATE == 1 ? 2 * TB * D : 0);            // column gate [2][TB][KW]
        const int cq = D * esz / 16, cv = KW * esz / 16, cgr = D / 4, cgc = KW / 4;
        auto issue = [&](int64_t b0, int Lb, int buf) {
            const int per = cq * 2 + cv + (GATE == 1 ? cgr : 0) + (GATE == 2 ? cgc : 0);
            for (int idx = threadIdx.x; idx < Lb * per; idx += nthr) {
                const int u = idx / per;
                int r = idx % per;
                const int64_t t = token(b0 + u);
                const void *src;
                void *dst;
                if (r < cq) {
                    src = qb + t * a.q.st + r * (16 / esz);
                    dst = rq + ((size_t)buf * TB + u) * D + r * (16 / esz);
                } else if ((r -= cq) < cq) {
                    src = kb + t * a.k.st + r * (16 / esz);
                    dst = rk + ((size_t)buf * TB + u) * D + r * (16 / esz);
                } else if ((r -= cq) < cv) {
                    src = vb + t * a.v.st + e0 + r * (16 / esz);
                    dst = rv + ((size_t)buf * TB + u) * KW + r * (16 / esz);
                } else if (GATE == 1) {
                    r -= cv;
                    src = gb + t * a.gate.st + 4 * r;
                    dst = rg + ((size_t)buf * TB + u) * D + 4 * r;
                } else {
                    r -= cv;
                    src = gb + t * a.gate.st + e0 + 4 * r;
                    dst = rgc + ((size_t)buf * TB + u) * KW + 4 * r;
                }
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                             "l"(src)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        auto convert = [&](int Lb, int buf) {
            for (int idx = threadIdx.x; idx < Lb * DP; idx += nthr) {
                const int u = idx / DP, k = idx % DP;
                const int at = u * DPP + k + 4 * (k / RP);
                const size_t rr = ((size_t)buf * TB + u) * D + k;
                qs[at] = k < D ? ld_tok(rq + rr) : 0.f;
                ks[at] = k < D ? ld_tok(rk + rr) : 0.f;
                if (GATE == 1)
                    as[at] = k < D ? expf(gh + rg[rr]) : 1.f;
            }
            for (int idx = threadIdx.x; idx < Lb * KW; idx += nthr) {
                const size_t rr = (size_t)buf * TB * KW + idx;
                ws[idx] = ld_tok(rv + rr);
                if (GATE == 2)
                    acs[idx] = expf(gh + rgc[rr]);
            }
        };
        int it = 0;
        if (len > 0)
            issue(0, (int)(len < TB ? len : TB), 0);
        for (int64_t b0 = 0; b0 < len; b0 += TB, ++it) {
            const int Lb = (int)(len - b0 < TB ? len - b0 : TB);
            if (b0 + TB < len) {
                issue(b0 + TB, (int)(len - b0 - TB < TB ? len - b0 - TB : TB), (it + 1) & 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            __syncthreads();   // every thread's copies of this block landed
            convert(Lb, it & 1);
            __syncthreads();
            compute(b0, Lb);
        }
        __syncthreads();
    }

    if (a.s_out.p && col_ok) {
#pragma unroll
        for (int j = 0; j < RP; ++j)
            if (r0 + j < D)
                a.s_out.p[sbase + (int64_t)(r0 + j) * a.s_out.rs + (int64_t)(e0 + c) * a.s_out.cs] =
                    S[j];
    }
}

template <typename K>
cudaError_t launch_one(K kernel, const SweepArgs &a, cudaStream_t s, int gate, bool async)
{
    const size_t smem = short_smem_bytes(a.D, a.bf16 ? 2 : 4, async ? gate : -1);
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

// Rows of every tensor 16-byte aligned (base, strides, widths) and value tiles
// full: the copies can be 16-byte cp.async.
bool rows_aligned(const SweepArgs &a, int esz)
{
    auto ok = [&](const void *p, int64_t sb, int64_t st, int64_t sh, int64_t es) {
        return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && (sb * es) % 16 == 0 &&
               (st * es) % 16 == 0 && (sh * es) % 16 == 0;
    };
    bool r = ok(a.q.p, a.q.sb, a.q.st, a.q.sh, esz) && ok(a.k.p, a.k.sb, a.k.st, a.k.sh, esz) &&
             ok(a.v.p, a.v.sb, a.v.st, a.v.sh, esz) && (a.D * esz) % 16 == 0 && a.E % KW == 0;
    if (a.gate.p)
        r = r && ok(a.gate.p, a.gate.sb, a.gate.st, a.gate.sh, 4) && a.D % 4 == 0;
    return r;
}

template <typename T, bool BWD, bool ASYNC>
cudaError_t launch_async(const SweepArgs &a, cudaStream_t s)
{
    if (!a.gate.p)
        return launch_one(short_kernel<T, BWD, 0, ASYNC>, a, s, 0, ASYNC);
    return a.gate.cols ? launch_one(short_kernel<T, BWD, 2, ASYNC>, a, s, 2, ASYNC)
                       : launch_one(short_kernel<T, BWD, 1, ASYNC>, a, s, 1, ASYNC);
}

template <typename T, bool BWD> cudaError_t launch_gate(const SweepArgs &a, cudaStream_t s)
{
    if (a.max_len > TB && rows_aligned(a, (int)sizeof(T)))
        return launch_async<T, BWD, true>(a, s);
    return launch_async<T, BWD, false>(a, s);
}

template <bool BWD> cudaError_t launch_short(const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0)
        return cudaSuccess;
    if (a.D < 1 || a.D > RP * MAXG)
        return cudaErrorNotSupported;
    if ((int64_t)a.N * a.H * ((a.E + KW - 1) / KW) > 0x7fffffff)
        return cudaErrorNotSupported;
    return a.bf16 ? launch_gate<__nv_bfloat16, BWD>(a, s) : launch_gate<float, BWD>(a, s);
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
