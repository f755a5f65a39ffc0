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
// token loop: the kernel is bound by the state's 2 x D E x 4 bytes.
//
// Two launch forms of the same arithmetic:
//   decode_mma_kernel     one CTA per (sequence, head); the state straight
//                         from global memory into the fragments, the state
//                         of the CTA one resident wave ahead prefetched
//                         into L2.
//   decode_stream_kernel  at least two blocks per SM (E a multiple of 64):
//                         one persistent CTA per SM, whose copy thread moves
//                         each block's state and token rows into a ring of
//                         two shared-memory slots by TMA (128-byte swizzled
//                         boxes: no bank conflicts in the fragment loads),
//                         and each finished state back out, while the
//                         compute warps work on the other slot.
//                         Waits on the ring are bounded (2 s): on expiry the
//                         CTA records LA_ERR_TIMEOUT, drains its copies and
//                         returns.

#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

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

// ---- ring of the streamed form ------------------------------------------------
__device__ int g_decode_error;   // LA_ERR_TIMEOUT once a wait of the streamed form ran out
constexpr uint64_t DC_WAIT_NS = 2000000000ull;
constexpr int DC_ERR_TIMEOUT = 4;

__device__ __forceinline__ void mbar_init1(uint64_t *bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(su32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: false when the CTA is aborting or this wait ran out.
__device__ __forceinline__ bool dwait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_test(bar, parity))
        return true;
    const uint64_t t0 = now_ns();
    for (;;) {
        if (mbar_test(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (now_ns() - t0 > DC_WAIT_NS) {
            *abort_flag = 1;
            atomicExch(&g_decode_error, DC_ERR_TIMEOUT);
            return false;
        }
    }
}
// Bounded wait that ignores the abort flag (draining this CTA's own copies).
__device__ __forceinline__ void ddrain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = now_ns();
    while (!mbar_test(bar, parity))
        if (now_ns() - t0 > DC_WAIT_NS) {
            atomicExch(&g_decode_error, DC_ERR_TIMEOUT);
            return;
        }
}
__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_done()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// barrier 1 over the compute threads
__device__ __forceinline__ void comp_sync(int n)
{
    asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory");
}
// AND of ok over the compute threads (barrier 2)
__device__ __forceinline__ bool comp_and(bool ok, int n)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.and.pred p, 2, %2, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"(ok ? 1u : 0u), "r"(n)
                 : "memory");
    return r != 0;
}
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// ---- streamed form -------------------------------------------------------------
// The ring's tiles are moved by TMA: each block's state as E/32 boxes of
// [128 rows][32 floats] and its q, k, v rows as boxes of [16 tokens][64
// channels], all with the 128-byte swizzle (16-byte chunk c of row r at
// c ^ (r & 7)), so that the fragment loads meet no bank conflicts; the new
// state goes back by E/32 box stores.  Rows are in token order: in reverse
// mode the processing index of row i < L is L - 1 - i.
constexpr int DS_NS = 2;                          // ring slots
constexpr int DS_SBOX = DC_D * 32 * 4;            // one state box: 16 KB
constexpr int DS_TBOX = DC_T * 64 * 2;            // one token box: 2 KB
constexpr int DS_STATE = 4 * DS_SBOX;             // state of up to 128 columns
constexpr int DS_TOK = 2 * DS_TBOX;               // one token tensor: 128 channels
constexpr int DS_SLOT = DS_STATE + 3 * DS_TOK;    // state, q, k, v

struct DecodeParams {
    CUtensorMap ms_in, ms_out, mq, mk, mv;
    SweepArgs a;
};

// byte offsets inside a state / token tile
__device__ __forceinline__ uint32_t st_off(int r, int c)
{
    return (uint32_t)((c >> 5) * DS_SBOX + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) +
                      (c & 3) * 4);
}
__device__ __forceinline__ uint32_t tk_off(int r, int c)
{
    return (uint32_t)((c >> 6) * DS_TBOX + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                      (c & 7) * 2);
}
__device__ __forceinline__ void tma_in_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int x,
                                          int y)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
                 "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_in_4d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                          int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(su32(dst)),
                 "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(c0), "r"(c1), "r"(c2),
                 "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void tma_out_2d(const CUtensorMap *m, const void *src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(su32(src)), "r"(x), "r"(y)
                 : "memory");
}

// Shared memory of the streamed form: the ring (1024-byte aligned slots),
// the K^T table, the key decays, the barriers and the abort word, plus the
// alignment slack.
size_t decode_stream_smem_bytes()
{
    return (size_t)DS_NS * DS_SLOT + (size_t)DC_D * DC_KS * 2 + DC_T * 4 + 2 * DS_NS * 8 + 16 +
           1024;
}

__global__ void __launch_bounds__(9 * 32, 1) decode_stream_kernel(const __grid_constant__ DecodeParams P)
{
    extern __shared__ __align__(1024) uint8_t dsm_raw[];
    uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const SweepArgs &a = P.a;
    const int E = a.E, nw = E / 16, ncomp = nw * 32;
    __nv_bfloat16 *skt = reinterpret_cast<__nv_bfloat16 *>(dsm + DS_NS * DS_SLOT);
    float *fk = reinterpret_cast<float *>(skt + DC_D * DC_KS);
    uint64_t *full = reinterpret_cast<uint64_t *>(fk + DC_T);
    uint64_t *done = full + DS_NS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(done + DS_NS);
    const int heads = a.N * a.H;
    const int tid = threadIdx.x;
    const bool has_in = a.s_in.p != nullptr, has_out = a.s_out.p != nullptr;
    auto state_of = [&](int b) { return dsm + b * DS_SLOT; };
    auto tok_of = [&](int b, int which) { return dsm + b * DS_SLOT + DS_STATE + which * DS_TOK; };
    auto seq = [&](int hn, int64_t &row, int64_t &bos, int64_t &len) {
        const int n = hn / a.H;
        if (a.cu) {
            row = 0;
            bos = a.cu[n];
            len = (int64_t)a.cu[n + 1] - a.cu[n];
        } else {
            row = n;
            bos = 0;
            len = a.T;
        }
    };
    if (tid == 0) {
        for (int i = 0; i < DS_NS; ++i) {
            mbar_init1(&full[i]);
            mbar_init1(&done[i]);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (tid >= ncomp) {
        // ---- copy warp (one thread) ----
        if (tid != ncomp)
            return;
        // diagnostic (la_debug_withhold_next_handoff): the first block is
        // never copied, so the compute warps' bounded wait on it runs out
        const int skip = a.withhold_handoff ? 1 : 0;
        auto store_state = [&](int lj) {
            const uint8_t *src = state_of(lj % DS_NS);
            const int y = (blockIdx.x + lj * (int)gridDim.x) * DC_D;
            for (int b = 0; b < E / 32; ++b)
                tma_out_2d(&P.ms_out, src + b * DS_SBOX, 32 * b, y);
            bulk_commit();
        };
        int li = 0;
        bool ok = true;
        for (int hn = blockIdx.x; hn < heads; hn += gridDim.x, ++li) {
            const int buf = li % DS_NS;
            if (li < skip)
                continue;
            if (li >= DS_NS) {
                // the block DS_NS back has left this slot: store its state
                ok = dwait(&done[buf], ((li - DS_NS) / DS_NS) & 1, abort_flag);
                if (!ok)
                    break;
                if (has_out) {
                    store_state(li - DS_NS);
                    bulk_wait_read();   // before the slot is refilled
                }
            }
            int64_t row, bos, len;
            seq(hn, row, bos, len);
            const int L = (int)len, h = hn % a.H;
            const uint32_t tx = (has_in ? (uint32_t)(E / 32 * DS_SBOX) : 0u) +
                                (L > 0 ? (uint32_t)(2 * DS_TOK + E / 64 * DS_TBOX) : 0u);
            if (tx)
                mbar_expect(&full[buf], tx);
            else
                mbar_arrive1(&full[buf]);
            if (has_in)
                for (int b = 0; b < E / 32; ++b)
                    tma_in_2d(state_of(buf) + b * DS_SBOX, &P.ms_in, &full[buf], 32 * b, hn * DC_D);
            if (L > 0) {
                for (int b = 0; b < 2; ++b) {
                    tma_in_4d(tok_of(buf, 0) + b * DS_TBOX, &P.mq, &full[buf], 64 * b,
                              h / a.q.hdiv, (int)bos, (int)row);
                    tma_in_4d(tok_of(buf, 1) + b * DS_TBOX, &P.mk, &full[buf], 64 * b,
                              h / a.k.hdiv, (int)bos, (int)row);
                }
                for (int b = 0; b < E / 64; ++b)
                    tma_in_4d(tok_of(buf, 2) + b * DS_TBOX, &P.mv, &full[buf], 64 * b,
                              h / a.v.hdiv, (int)bos, (int)row);
            }
        }
        const int issued = li;
        if (ok) {
            // the last blocks' states
            for (int lj = issued > DS_NS ? issued - DS_NS : skip; lj < issued; ++lj) {
                if (!dwait(&done[lj % DS_NS], (lj / DS_NS) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                if (has_out)
                    store_state(lj);
            }
        }
        if (!ok) {
            // no copy into this CTA's shared memory may outlive it
            for (int lj = issued - DS_NS > skip ? issued - DS_NS : skip; lj < issued; ++lj)
                ddrain(&full[lj % DS_NS], (lj / DS_NS) & 1);
        }
        bulk_wait_done();
        return;
    }

    // ---- compute warps ----
    const int warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int e0 = 16 * warp;
    const int ar = (lane & 7) + 8 * ((lane >> 3) & 1), ac = 8 * (lane >> 4);
    const int bnr = (lane & 7) + 8 * (lane >> 4), bnc = 8 * ((lane >> 3) & 1);
    int li = 0;
    for (int hn = blockIdx.x; hn < heads; hn += gridDim.x, ++li) {
        const int buf = li % DS_NS;
        if (!comp_and(dwait(&full[buf], (li / DS_NS) & 1, abort_flag), ncomp))
            break;
        int64_t row, bos, len;
        seq(hn, row, bos, len);
        const int L = (int)len, h = hn % a.H;
        const bool rev = a.reverse != 0;
        const float gm = a.g[h], scale = a.scale;
        uint8_t *sq = tok_of(buf, 0), *sk = tok_of(buf, 1), *sv = tok_of(buf, 2);
        uint8_t *sb = state_of(buf);
        // token rows past L (another sequence's, or never loaded): zero
        for (int i = tid; i < (DC_T - L) * 8 * (4 + E / 64); i += ncomp) {
            const int w = i / ((DC_T - L) * 8), u = L + (i / 8) % (DC_T - L), c16 = i % 8;
            uint8_t *t = w < 2 ? sq + w * DS_TBOX : w < 4 ? sk + (w - 2) * DS_TBOX
                                                          : sv + (w - 4) * DS_TBOX;
            *reinterpret_cast<uint4 *>(t + u * 128 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        // gamma^(L-1-p) for the key of row u (p its processing index)
        if (tid < DC_T)
            fk[tid] = tid < L ? expf(gm * (float)(L - 1 - (rev ? L - 1 - tid : tid))) : 0.f;
        comp_sync(ncomp);
        for (int i = tid; i < 2 * DC_D; i += ncomp) {
            const int d = i >> 1, u0 = 8 * (i & 1);
            uint32_t w[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float k0 = __bfloat162float(
                    *reinterpret_cast<const __nv_bfloat16 *>(sk + tk_off(u0 + 2 * p, d)));
                const float k1 = __bfloat162float(
                    *reinterpret_cast<const __nv_bfloat16 *>(sk + tk_off(u0 + 2 * p + 1, d)));
                w[p] = bf2(k0 * fk[u0 + 2 * p], k1 * fk[u0 + 2 * p + 1]);
            }
            *reinterpret_cast<uint4 *>(skt + d * DC_KS + u0) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        comp_sync(ncomp);

        // P = q k^T and Oi = q S0 (S0's B fragments as bf16 from the fp32 tile)
        float Pc[2][4], Oi[2][4], Oa[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int x = 0; x < 4; ++x)
                Pc[j][x] = Oi[j][x] = Oa[j][x] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DC_D / 16; ++kk) {
            uint32_t qa[4], kb[4];
            ldsm4(qa, sq + tk_off(ar, 16 * kk + ac));
            ldsm4(kb, sk + tk_off(bnr, 16 * kk + bnc));
            mma_bf16(Pc[0], qa, kb[0], kb[1]);
            mma_bf16(Pc[1], qa, kb[2], kb[3]);
            if (has_in) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int r = 16 * kk + 2 * cq, c = e0 + 8 * j + gq;
                    auto f = [&](int rr) {
                        return *reinterpret_cast<const float *>(sb + st_off(rr, c));
                    };
                    mma_bf16(Oi[j], qa, bf2(f(r), f(r + 1)), bf2(f(r + 8), f(r + 9)));
                }
            }
        }
        uint32_t pa[4];
        {
            float p[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int t = gq + 8 * (x >> 1), u = 8 * j + 2 * cq + (x & 1);
                    const int pt = rev ? L - 1 - t : t, pu = rev ? L - 1 - u : u;
                    p[j][x] = t < L && u < L && pu <= pt
                                  ? Pc[j][x] * scale * expf(gm * (float)(pt - pu))
                                  : 0.f;
                }
            pa[0] = bf2(p[0][0], p[0][1]);
            pa[1] = bf2(p[0][2], p[0][3]);
            pa[2] = bf2(p[1][0], p[1][1]);
            pa[3] = bf2(p[1][2], p[1][3]);
        }
        uint32_t vb[4];
        ldsm4t(vb, sv + tk_off(ar, e0 + ac));
        mma_bf16(Oa[0], pa, vb[0], vb[1]);
        mma_bf16(Oa[1], pa, vb[2], vb[3]);
        {
            __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(a.out.p) + row * a.out.sb +
                                (int64_t)h * a.out.sh + e0 + 2 * cq;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = gq + 8 * hf;
                if (t < L) {
                    const int pt = rev ? L - 1 - t : t;
                    const float f = scale * expf(gm * (float)(pt + 1));
                    __nv_bfloat16 *orow = ob + (bos + t) * a.out.st;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        *reinterpret_cast<uint32_t *>(orow + 8 * j) =
                            bf2(fmaf(f, Oi[j][2 * hf], Oa[j][2 * hf]),
                                fmaf(f, Oi[j][2 * hf + 1], Oa[j][2 * hf + 1]));
                }
            }
        }
        // S = gamma^L S0 + K^T V on this warp's columns, back into the slot
        const float gl = expf(gm * (float)L);
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
            uint32_t ka[4];
            ldsm4(ka, skt + (16 * i + ar) * DC_KS + ac);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = 16 * i + gq, c = e0 + 8 * j + 2 * cq;
                float2 *p0 = reinterpret_cast<float2 *>(sb + st_off(r, c));
                float2 *p1 = reinterpret_cast<float2 *>(sb + st_off(r + 8, c));
                float cc[4] = {0.f, 0.f, 0.f, 0.f};
                if (has_in) {
                    const float2 x0 = *p0, x1 = *p1;
                    cc[0] = gl * x0.x;
                    cc[1] = gl * x0.y;
                    cc[2] = gl * x1.x;
                    cc[3] = gl * x1.y;
                }
                mma_bf16(cc, ka, vb[2 * j], vb[2 * j + 1]);
                *p0 = make_float2(cc[0], cc[1]);
                *p1 = make_float2(cc[2], cc[3]);
            }
        }
        fence_async_smem();   // the new state, visible to the tensor stores
        comp_sync(ncomp);
        if (tid == 0)
            mbar_arrive1(&done[buf]);
    }
}

// 4-D token map {channel, head, token, batch}: box {64, 1, 16, 1}, 128-byte
// swizzle; 2-D state map {column, row} over all blocks: box {32, 128}.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
bool token_map(CUtensorMap *m, const Tok &t, int X, const SweepArgs &a)
{
    auto fn = encode_tiled();
    if (!fn)
        return false;
    const int heads = a.H / t.hdiv;
    const int64_t sh = heads == 1 ? X : t.sh, st = t.st, sb = a.B == 1 ? t.st * a.T : t.sb;
    if (sh <= 0 || st <= 0 || sb <= 0)
        return false;
    cuuint64_t dims[4] = {(cuuint64_t)X, (cuuint64_t)heads, (cuuint64_t)a.T, (cuuint64_t)a.B};
    cuuint64_t strides[3] = {(cuuint64_t)(sh * 2), (cuuint64_t)(st * 2), (cuuint64_t)(sb * 2)};
    cuuint32_t box[4] = {64, 1, DC_T, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(t.p), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool state_map(CUtensorMap *m, const float *p, int E, int64_t rows)
{
    auto fn = encode_tiled();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)E * 4};
    cuuint32_t box[2] = {32, DC_D};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool rows16(const void *p, int64_t sb, int64_t st, int64_t sh)
{
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && sb % 8 == 0 && st % 8 == 0 &&
           sh % 8 == 0;
}

}  // namespace

cudaError_t decode_chunk_sweep(const SweepArgs &a, cudaStream_t s, bool *streamed)
{
    if (streamed)
        *streamed = false;
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
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    DecodeParams dp;
    if (blocks >= 2 * (int64_t)sms && a.E % 64 == 0 &&
        token_map(&dp.mq, a.q, DC_D, a) && token_map(&dp.mk, a.k, DC_D, a) &&
        token_map(&dp.mv, a.v, a.E, a) &&
        (!a.s_in.p || state_map(&dp.ms_in, a.s_in.p, a.E, blocks * DC_D)) &&
        (!a.s_out.p || state_map(&dp.ms_out, a.s_out.p, a.E, blocks * DC_D))) {
        // the streamed form: one persistent CTA per SM
        if (!a.s_in.p)
            dp.ms_in = dp.mq;   // not used
        if (!a.s_out.p)
            dp.ms_out = dp.mq;
        dp.a = a;
        const size_t smem = decode_stream_smem_bytes();
        e = cudaFuncSetAttribute(decode_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess)
            return e;
        decode_stream_kernel<<<(unsigned)sms, warps * 32 + 32, smem, s>>>(dp);
        note_launch();
        if (streamed)
            *streamed = true;
        return cudaGetLastError();
    }
    const size_t smem = decode_smem_bytes(warps);
    e = cudaFuncSetAttribute(decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    int per_sm = 0;
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

cudaError_t decode_read_and_clear_error(cudaStream_t s, int *err)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(err, g_decode_error, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof(int), 0,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace la
