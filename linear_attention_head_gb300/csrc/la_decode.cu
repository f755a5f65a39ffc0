// la_decode.cu -- decoding up to 16 new tokens per (sequence, head) against a
// carried fp32 state (bf16 tokens, 128 key channels, value width a multiple
// of 16 up to 128, forward-type, no gate): the tokens as one chunk of the
// chunked form, its three small contractions on the tensor cores.
//
// With the entering state S0 (D x E) and the tokens in processing order
// t = 0 .. L-1 (ejkernel `recurrent` docstring, "The core update"; the
// Lightning Attention-2 paper's intra/inter split for one block):
//     o_t = s gamma^(t+1) q_t S0 + sum_{u <= t} s gamma^(t-u) (q_t . k_u) v_u
//     S   = gamma^L S0 + sum_u (gamma^(L-1-u) k_u)^T v_u
// gamma = exp(g[h]).  One CTA per (sequence, head), warp w owns value columns
// 16 w .. 16 w + 15.  The state goes from global memory straight into the
// accumulator fragments of the update (fp32, read once, written once), so no
// shared-memory staging of the 64 KB block: every warp computes
//     P  = q k^T                 (16 x 16, K = 128: 16 MMAs), masked and
//                                 scaled by s gamma^(t-u) in registers
//     Oi = q S0                  (16 x 16, K = 128: 16 MMAs; S0 as bf16 from
//                                 its own fragments through a per-warp tile)
//     Oa = P V                   (16 x 16, K = 16: 2 MMAs)
//     o  = s gamma^(t+1) Oi + Oa
//     S  = gamma^L S0 + K^T V    (128 x 16, K = 16: 16 MMAs accumulating on
//                                 the fp32 state fragments)
// with mma.sync m16n8k16 (bf16 operands, fp32 accumulators).  The operands
// rounded to bf16 are the ones the chunked kernels round too: the state in
// the inter term, the decayed keys, the scores.  The work per block is about
// 50 MMAs and a few hundred instructions per warp, against some 4000 for the
// token loop: the kernel is bound by the state's 2 x D E x 4 bytes.  Its CTAs
// prefetch the state of the CTA one resident wave ahead into L2.

#include <cstdint>

#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int DC_D = 128;        // key channels
constexpr int DC_T = 16;         // tokens of the chunk (MMA rows)
constexpr int DC_RS = 128 + 8;   // q, k, v row stride in shared memory (bf16): 272 bytes
constexpr int DC_KS = DC_T + 8;  // K^T table and state tile row stride (bf16): 48 bytes

__device__ __forceinline__ uint32_t su32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(su32(p)));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(su32(p)));
}
// d += a b: m16n8k16, A row-major bf16, B column-major bf16, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t bf2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Shared memory: q, k [DC_T][DC_RS], v [DC_T][DC_RS], K^T [DC_D][DC_KS], one
// bf16 state tile [DC_D][DC_KS] per warp, the key decays [DC_T] (fp32).
size_t decode_smem_bytes(int warps)
{
    return (size_t)3 * DC_T * DC_RS * 2 + (size_t)DC_D * DC_KS * 2 +
           (size_t)warps * DC_D * DC_KS * 2 + DC_T * 4;
}

__global__ void __launch_bounds__(256, 2) decode_mma_kernel(SweepArgs a)
{
    extern __shared__ __align__(128) uint8_t dsm[];
    const int E = a.E, nw = E / 16;
    __nv_bfloat16 *sq = reinterpret_cast<__nv_bfloat16 *>(dsm);
    __nv_bfloat16 *sk = sq + DC_T * DC_RS;
    __nv_bfloat16 *sv = sk + DC_T * DC_RS;
    __nv_bfloat16 *skt = sv + DC_T * DC_RS;
    __nv_bfloat16 *stile = skt + DC_D * DC_KS;
    float *fk = reinterpret_cast<float *>(stile + nw * DC_D * DC_KS);

    const int h = (int)(blockIdx.x % (unsigned)a.H), n = (int)(blockIdx.x / (unsigned)a.H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;   // fragment row group, column pair
    const int e0 = 16 * warp;
    const int nthr = nw * 32;
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
    const int L = (int)len;
    const float gm = a.g[h], scale = a.scale;
    const int64_t sbase = ((int64_t)n * a.H + h) * (int64_t)DC_D * E;

    // the state of the CTA one resident wave ahead, into L2
    if (tid == 0 && a.s_in.p && a.prefetch_ctas > 0) {
        const int64_t ahead = (int64_t)blockIdx.x + a.prefetch_ctas;
        if (ahead < (int64_t)gridDim.x)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                             a.s_in.p + ahead * (int64_t)DC_D * E),
                         "r"((uint32_t)(DC_D * E * 4))
                         : "memory");
    }

    // 1. this warp's 16 state columns, all rows, as accumulator fragments:
    //    tile (i, j) holds rows 16 i + gq (+ 8), columns e0 + 8 j + 2 cq (+ 1)
    float S[8][2][4];
    if (a.s_in.p) {
        const float *sp = a.s_in.p + sbase + e0 + 2 * cq;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 x0 = *reinterpret_cast<const float2 *>(sp + (16 * i + gq) * E + 8 * j);
                const float2 x1 =
                    *reinterpret_cast<const float2 *>(sp + (16 * i + gq + 8) * E + 8 * j);
                S[i][j][0] = x0.x;
                S[i][j][1] = x0.y;
                S[i][j][2] = x1.x;
                S[i][j][3] = x1.y;
            }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    S[i][j][x] = 0.f;
    }

    // 2. the tokens in processing order, rows past L zero
    {
        const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(a.q.p) + row * a.q.sb +
                                  (int64_t)(h / a.q.hdiv) * a.q.sh;
        const __nv_bfloat16 *kp = static_cast<const __nv_bfloat16 *>(a.k.p) + row * a.k.sb +
                                  (int64_t)(h / a.k.hdiv) * a.k.sh;
        const __nv_bfloat16 *vp = static_cast<const __nv_bfloat16 *>(a.v.p) + row * a.v.sb +
                                  (int64_t)(h / a.v.hdiv) * a.v.sh;
        for (int i = tid; i < 2 * DC_T * (DC_D / 8); i += nthr) {
            const int which = i / (DC_T * (DC_D / 8)), u = (i / (DC_D / 8)) % DC_T,
                      p = i % (DC_D / 8);
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (u < L) {
                const int64_t t = bos + (a.reverse ? L - 1 - u : u);
                x = *reinterpret_cast<const uint4 *>(which ? kp + t * a.k.st + 8 * p
                                                           : qp + t * a.q.st + 8 * p);
            }
            *reinterpret_cast<uint4 *>((which ? sk : sq) + u * DC_RS + 8 * p) = x;
        }
        for (int i = tid; i < DC_T * (E / 8); i += nthr) {
            const int u = i / (E / 8), p = i % (E / 8);
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (u < L) {
                const int64_t t = bos + (a.reverse ? L - 1 - u : u);
                x = *reinterpret_cast<const uint4 *>(vp + t * a.v.st + 8 * p);
            }
            *reinterpret_cast<uint4 *>(sv + u * DC_RS + 8 * p) = x;
        }
        if (tid < DC_T)
            fk[tid] = tid < L ? expf(gm * (float)(L - 1 - tid)) : 0.f;
    }
    __syncthreads();
    // K^T [d][u] = gamma^(L-1-u) k_u[d] (bf16); zero past L.  This warp's
    // state tile as bf16 [d][e - e0], the B operand of the inter term.
    for (int i = tid; i < 2 * DC_D; i += nthr) {
        const int d = i >> 1, u0 = 8 * (i & 1);
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            w[p] = bf2(__bfloat162float(sk[(u0 + 2 * p) * DC_RS + d]) * fk[u0 + 2 * p],
                       __bfloat162float(sk[(u0 + 2 * p + 1) * DC_RS + d]) * fk[u0 + 2 * p + 1]);
        *reinterpret_cast<uint4 *>(skt + d * DC_KS + u0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __nv_bfloat16 *st = stile + warp * DC_D * DC_KS;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int d = 16 * i + gq, e = 8 * j + 2 * cq;
            *reinterpret_cast<uint32_t *>(st + d * DC_KS + e) = bf2(S[i][j][0], S[i][j][1]);
            *reinterpret_cast<uint32_t *>(st + (d + 8) * DC_KS + e) = bf2(S[i][j][2], S[i][j][3]);
        }
    __syncthreads();

    // ldmatrix row addresses of this lane: A / K^T (rows r, k contiguous),
    // B from n-rows (k contiguous), B from k-rows (n contiguous)
    const int ar = (lane & 7) + 8 * ((lane >> 3) & 1), ac = 8 * (lane >> 4);
    const int bnr = (lane & 7) + 8 * (lane >> 4), bnc = 8 * ((lane >> 3) & 1);

    // 3. P = q k^T and Oi = q S0 over the 128 key channels
    float Pc[2][4], Oi[2][4], Oa[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x)
            Pc[j][x] = Oi[j][x] = Oa[j][x] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DC_D / 16; ++kk) {
        uint32_t qa[4], kb[4], sb[4];
        ldsm4(qa, sq + ar * DC_RS + 16 * kk + ac);
        ldsm4(kb, sk + bnr * DC_RS + 16 * kk + bnc);
        ldsm4t(sb, st + (16 * kk + ar) * DC_KS + ac);
        mma_bf16(Pc[0], qa, kb[0], kb[1]);
        mma_bf16(Pc[1], qa, kb[2], kb[3]);
        mma_bf16(Oi[0], qa, sb[0], sb[1]);
        mma_bf16(Oi[1], qa, sb[2], sb[3]);
    }
    // scores s gamma^(t-u) q_t . k_u for u <= t, zero above the diagonal;
    // their accumulator fragments are the A operand of P V
    uint32_t pa[4];
    {
        float p[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int t = gq + 8 * (x >> 1), u = 8 * j + 2 * cq + (x & 1);
                p[j][x] = u <= t ? Pc[j][x] * scale * expf(gm * (float)(t - u)) : 0.f;
            }
        pa[0] = bf2(p[0][0], p[0][1]);
        pa[1] = bf2(p[0][2], p[0][3]);
        pa[2] = bf2(p[1][0], p[1][1]);
        pa[3] = bf2(p[1][2], p[1][3]);
    }
    // V (tokens x this warp's columns), the B operand of P V and of the update
    uint32_t vb[4];
    ldsm4t(vb, sv + ar * DC_RS + e0 + ac);
    mma_bf16(Oa[0], pa, vb[0], vb[1]);
    mma_bf16(Oa[1], pa, vb[2], vb[3]);

    // 4. o_t = s gamma^(t+1) Oi + Oa for t < L
    {
        __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(a.out.p) + row * a.out.sb +
                            (int64_t)h * a.out.sh + e0 + 2 * cq;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int t = gq + 8 * hf;
            if (t < L) {
                const float f = scale * expf(gm * (float)(t + 1));
                __nv_bfloat16 *orow = ob + (bos + (a.reverse ? L - 1 - t : t)) * a.out.st;
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    *reinterpret_cast<uint32_t *>(orow + 8 * j) =
                        bf2(fmaf(f, Oi[j][2 * hf], Oa[j][2 * hf]),
                            fmaf(f, Oi[j][2 * hf + 1], Oa[j][2 * hf + 1]));
            }
        }
    }

    // 5. S = gamma^L S0 + K^T V, accumulated on the fp32 fragments, and out
    const float gl = expf(gm * (float)L);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t ka[4];
        ldsm4(ka, skt + (16 * i + ar) * DC_KS + ac);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int x = 0; x < 4; ++x)
                S[i][j][x] *= gl;
            mma_bf16(S[i][j], ka, vb[2 * j], vb[2 * j + 1]);
        }
    }
    if (a.s_out.p) {
        float *sp = a.s_out.p + sbase + e0 + 2 * cq;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                *reinterpret_cast<float2 *>(sp + (16 * i + gq) * E + 8 * j) =
                    make_float2(S[i][j][0], S[i][j][1]);
                *reinterpret_cast<float2 *>(sp + (16 * i + gq + 8) * E + 8 * j) =
                    make_float2(S[i][j][2], S[i][j][3]);
            }
    }
}

bool rows16(const void *p, int64_t sb, int64_t st, int64_t sh)
{
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && sb % 8 == 0 && st % 8 == 0 &&
           sh % 8 == 0;
}

}  // namespace

cudaError_t decode_chunk_sweep(const SweepArgs &a, cudaStream_t s)
{
    auto state_ok = [&](const float *p, int64_t rs, int64_t cs) {
        return !p || ((reinterpret_cast<uintptr_t>(p) & 15) == 0 && rs == a.E && cs == 1);
    };
    if (!a.bf16 || a.D != DC_D || a.E < 16 || a.E > 128 || a.E % 16 || a.max_len > DC_T ||
        a.gate.p || a.gla_flags || a.out_f32 || !state_ok(a.s_in.p, a.s_in.rs, a.s_in.cs) ||
        !state_ok(a.s_out.p, a.s_out.rs, a.s_out.cs) ||
        !rows16(a.q.p, a.q.sb, a.q.st, a.q.sh) || !rows16(a.k.p, a.k.sb, a.k.st, a.k.sh) ||
        !rows16(a.v.p, a.v.sb, a.v.st, a.v.sh) || !rows16(a.out.p, a.out.sb, a.out.st, a.out.sh))
        return cudaErrorNotSupported;
    const int64_t blocks = (int64_t)a.N * a.H;
    if (blocks == 0)
        return cudaSuccess;
    if (blocks > 0x7fffffff)
        return cudaErrorNotSupported;
    const int warps = a.E / 16;
    const size_t smem = decode_smem_bytes(warps);
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int dev = 0, sms = 0, per_sm = 0;
    if (e == cudaSuccess)
        e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mma_kernel, warps * 32,
                                                          smem);
    if (e != cudaSuccess)
        return e;
    SweepArgs b = a;
    b.prefetch_ctas = (int64_t)per_sm * sms;
    decode_mma_kernel<<<(unsigned)blocks, warps * 32, smem, s>>>(b);
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
