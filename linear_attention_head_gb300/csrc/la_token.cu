// la_token.cu -- token-by-token kernels: decoding a few new tokens against a
// carried state, any call whose longest sequence has at most SHORT_MAX_T
// tokens, and every call with a per-key gate (any length).
//
// They run the recurrence itself (ejkernel `recurrent` docstring, "The core
// update") one token at a time instead of the chunked form:
//   forward-type:  S <- A_t S + k_t v_t^T,   out_t = s q_t^T S
//   backward-type: G <- G + s q_t w_t^T,     out_t = G^T k_t,   G <- A_t G
// (the two sweep shapes of la_internal.h, visited in the same token order as
// the chunked kernels), where A_t is the decay exp(g[h]) -- times exp(gate)
// per state row or per state column when a gate is given.
//
// Thread layout.  A thread carries a 16-row x 4-column block of the fp32
// state in registers for the whole sequence: rows 16 rg .. 16 rg + 15 and
// the four adjacent columns of its column quad.  A warp holds RGN row groups
// x QW quads (RGN x QW = 32, RGN the smallest power of two with 16 RGN >= D),
// i.e. every row of 4 QW columns, so
//   * the state is read and written once, in 16-byte pieces, and the QW lanes
//     of a row group cover 16 QW contiguous bytes of a state row;
//   * a column's dot product over the rows is summed inside the warp: a
//     reduce-scatter over the row-group lanes (halves of the quad first).
// Each row is updated with packed f32x2 arithmetic on the column pairs.  The
// per-row factors (q, k, row decay) come from shared-memory tables that hold
// every value twice, so that one 16-byte load yields the pairs of two rows.
// Tokens pass through shared memory TB at a time (16-byte cp.async copies,
// double-buffered, when every row is 16-byte aligned); warps share nothing
// else, and the token loop has no barrier inside a block.

#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace {

constexpr int RP = 16;    // state rows per thread
constexpr int TB = 16;    // tokens per shared-memory block
constexpr int MAXW = 8;   // warps per CTA
// floats per (token, row group) in the paired row tables for RP rows per
// thread: the 2 RP values and a pad that puts the row groups a quarter warp
// reads at once in different banks
__host__ __device__ constexpr int pair_stride(int rp) { return 2 * rp + (rp == 16 ? 8 : 4); }

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

// Packed two-lane fp32 arithmetic (round to nearest) on 64-bit register
// pairs: a pair of floats is carried as one 64-bit value, so that the
// operands of the packed instructions are always aligned register pairs.
typedef unsigned long long f2;
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 pack2(float lo, float hi)
{
    f2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float2 unpack2(f2 x)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
    return r;
}

__device__ __forceinline__ float &comp(float4 &v, int c)
{
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// CTA shape for widths D (state rows) and E (state columns).
struct Shape {
    int rgn;     // row groups per warp (power of two, 16 rgn >= D)
    int qw;      // column quads per warp (32 / rgn)
    int wc;      // columns per warp (4 qw)
    int wpc;     // warps per CTA
    int cw;      // columns per CTA (wpc wc)
    int tiles;   // CTAs per (sequence, head)
};

__host__ __device__ inline Shape token_shape(int D, int E, int rp)
{
    Shape s;
    s.rgn = 1;
    while (rp * s.rgn < D)
        s.rgn *= 2;
    s.qw = 32 / s.rgn;
    s.wc = 4 * s.qw;
    const int need = (E + s.wc - 1) / s.wc;
    s.wpc = need < MAXW ? need : MAXW;
    s.cw = s.wpc * s.wc;
    s.tiles = (E + s.cw - 1) / s.cw;
    return s;
}

// tokens per shared-memory block for a call whose longest sequence is max_len
__host__ __device__ inline int token_block(int64_t max_len)
{
    return max_len >= TB ? TB : (max_len < 1 ? 1 : (int)max_len);
}

// Dynamic shared memory of one CTA: the paired row tables q, k (and the row
// decays for a row gate) [tbe][rgn][SK], the value columns (and column
// decays for a column gate) [tbe][cw]; for the asynchronous path two raw
// buffers of tbe token rows: q, k [D], the value tile [cw] (token dtype) and
// the gate's row [D] or tile [cw] (fp32).
__host__ __device__ inline size_t token_smem_bytes(const Shape &s, int rp, int D, int tbe,
                                                   int esz, int gate, bool async)
{
    const size_t tab = (size_t)tbe * s.rgn * pair_stride(rp);
    size_t f = tab * (gate == 1 ? 3 : 2) + (size_t)tbe * s.cw * (gate == 2 ? 2 : 1);
    size_t b = f * 4;
    if (async)
        b += (size_t)2 * tbe * ((size_t)2 * D * esz + (size_t)s.cw * esz +
                                (gate == 1 ? (size_t)D * 4 : 0) + (gate == 2 ? (size_t)s.cw * 4 : 0));
    return b;
}

// GATE: 0 the head's decay only, 1 per-row gate, 2 per-column gate.
struct CtaSync {
    __device__ void operator()() const { __syncthreads(); }
};
// barrier 1 over the first `count` threads of the CTA
struct NamedSync {
    int count;
    __device__ void operator()() const { asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory"); }
};

// The tokens of (sequence n, head h) for the state block of thread tid (of
// nthr, column tile `tile`), carried in S01 / S23: staging through `sh` and
// the recurrence.  Sync is a barrier over the nthr threads.  SHORTC (calls
// of at most SHORT_MAX_T tokens): one token at a time; otherwise batches of
// four tokens whose row-group sums overlap.
// Raw token rows of one short sequence already in shared memory, in
// processing order: q, k [u][D], the value tile [u][cw] (token dtype) and the
// row gate [u][D] (fp32); q == nullptr when the rows are to be fetched.
struct RawRows {
    const void *q = nullptr, *k = nullptr, *v = nullptr;
    const float *g = nullptr;
};

template <typename T, bool BWD, int GATE, bool ASYNC, bool SHORTC, typename Sync>
__device__ __forceinline__ void token_loop(const SweepArgs &a, const Shape &sp, int n, int h,
                                           int tile, int tid, int nthr, float *sh,
                                           f2 (&S01)[RP], f2 (&S23)[RP], Sync sync,
                                           RawRows pre = RawRows())
{
    constexpr int SK = pair_stride(RP);
    const int D = a.D, E = a.E;
    const int warp = tid >> 5, lane = tid & 31;
    const int qd = lane & (sp.qw - 1), rg = lane / sp.qw;
    const int cb = tile * sp.cw;                 // the CTA's first column
    const int cl = warp * sp.wc + 4 * qd;        // the thread's quad within the CTA's columns
    const int c0 = cb + cl;                      // ... and in the state
    const int tbe = token_block(a.max_len);

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
    const int tab = tbe * sp.rgn * SK;
    float *qs = sh;
    float *ks = qs + tab;
    float *as = ks + tab;                               // row decays (GATE 1)
    float *vs = as + (GATE == 1 ? tab : 0);
    float *acs = vs + tbe * sp.cw;                      // column decays (GATE 2)
    // forward-type visits tokens in processing order, backward-type against it
    const bool flip = (a.reverse != 0) != BWD;
    auto token = [&](int64_t u) { return bos + (flip ? len - 1 - u : u); };

    const float gh = a.g[h];
    const float gam = expf(gh);
    const float scale = a.scale;
    // token rows of this (sequence, head): key/value heads may be shared
    const T *qb = reinterpret_cast<const T *>(a.q.p) + row * a.q.sb +
                  (int64_t)(h / a.q.hdiv) * a.q.sh;
    const T *kb = reinterpret_cast<const T *>(a.k.p) + row * a.k.sb +
                  (int64_t)(h / a.k.hdiv) * a.k.sh;
    const T *vb = reinterpret_cast<const T *>(a.v.p) + row * a.v.sb +
                  (int64_t)(h / a.v.hdiv) * a.v.sh;
    const float *gb = GATE ? a.gate.p + row * a.gate.sb + (int64_t)h * a.gate.sh : nullptr;
    // output rows: the token dtype, or fp32 when a bf16 call asks for it
    const int64_t ob = row * a.out.sb + (int64_t)h * a.out.sh;
    auto put = [&](int64_t off, float x) {
        if (sizeof(T) == 2 && a.out_f32)
            static_cast<float *>(a.out.p)[ob + off] = x;
        else
            st_tok(static_cast<T *>(a.out.p) + ob + off, x);
    };

    // ---- staging: one block of Lb tokens into the compute layout -------------
    // paired row tables: (token u, row r) at (u rgn + r / 16) SK + 2 (r % 16),
    // twice; rows past D hold zero (decay one)
    const int RR = RP * sp.rgn;
    auto put_row = [&](int u, int r, float xq, float xk, float xa) {
        const int at = (u * sp.rgn + r / RP) * SK + 2 * (r % RP);
        if (BWD)
            xq *= scale;
        *reinterpret_cast<float2 *>(qs + at) = make_float2(xq, xq);
        *reinterpret_cast<float2 *>(ks + at) = make_float2(xk, xk);
        if (GATE == 1)
            *reinterpret_cast<float2 *>(as + at) = make_float2(xa, xa);
    };
    constexpr int PF = 8;
    auto load_sync = [&](int64_t b0, int Lb) {
        const int nr = Lb * RR;
        for (int base = tid; base < nr; base += PF * nthr) {
            float xq[PF], xk[PF], xa[PF];
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr, u = idx / RR, r = idx % RR;
                xq[i] = xk[i] = 0.f;
                xa[i] = 0.f;
                if (idx < nr && r < D) {
                    const int64_t t = token(b0 + u);
                    xq[i] = ld_tok(qb + t * a.q.st + r);
                    xk[i] = ld_tok(kb + t * a.k.st + r);
                    if (GATE == 1)
                        xa[i] = gb[t * a.gate.st + r];
                }
            }
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr, u = idx / RR, r = idx % RR;
                if (idx < nr)
                    put_row(u, r, xq[i], xk[i], GATE == 1 && r < D ? expf(gh + xa[i]) : 1.f);
            }
        }
        const int nv = Lb * sp.cw;
        for (int base = tid; base < nv; base += PF * nthr) {
            float xv[PF], xg[PF];
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr, u = idx / sp.cw, c = idx % sp.cw;
                xv[i] = 0.f;
                xg[i] = 0.f;
                if (idx < nv && cb + c < E) {
                    const int64_t t = token(b0 + u);
                    xv[i] = ld_tok(vb + t * a.v.st + cb + c);
                    if (GATE == 2)
                        xg[i] = gb[t * a.gate.st + cb + c];
                }
            }
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int idx = base + i * nthr;
                if (idx < nv) {
                    vs[idx] = xv[i];
                    if (GATE == 2)
                        acs[idx] = expf(gh + xg[i]);
                }
            }
        }
    };

    // ---- the recurrence over one staged block --------------------------------
    // Per token a thread forms the partial dot products of its four columns
    // over its 16 rows; those of four tokens are then summed over the warp's
    // row groups together, so that their shuffles overlap.
    const bool bA = (rg & 1) != 0, bB = (rg & 2) != 0;
    const f2 gg = pack2(gam, gam);
    const float sc = BWD ? 1.f : scale;
    // NT tokens from u0 on (NT = 4: a full batch, 1: the tail of a block)
    auto process = [&](auto ntc, int64_t b0, int u0) {
        constexpr int NT = decltype(ntc)::value;
        // after the exchange over the first row-group bit each lane keeps two
        // columns of the quad: 2 bA, 2 bA + 1 (hv; all four, hv and hw, when
        // rgn = 1)
        float2 hv[NT], hw[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int u = u0 + i;
            // (row 2p, row 2p + 1) pairs of q, k and the row decays
            const int at = (u * sp.rgn + rg) * SK;
            const ulonglong2 *q2 = reinterpret_cast<const ulonglong2 *>(qs + at);
            const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(ks + at);
            const ulonglong2 *a2 = reinterpret_cast<const ulonglong2 *>(as + at);
            const ulonglong2 w = *reinterpret_cast<const ulonglong2 *>(vs + u * sp.cw + cl);
            f2 c01 = gg, c23 = gg;   // column decays
            if (GATE == 2) {
                const ulonglong2 ac = *reinterpret_cast<const ulonglong2 *>(acs + u * sp.cw + cl);
                c01 = ac.x;
                c23 = ac.y;
            }
            f2 e01 = 0ull, e23 = 0ull, o01 = 0ull, o23 = 0ull;
#pragma unroll
            for (int p = 0; p < RP / 2; ++p) {
                const ulonglong2 qq = q2[p], kk = k2[p];
                ulonglong2 aa;
                if (GATE == 1)
                    aa = a2[p];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int j = 2 * p + half;
                    const f2 qp = half ? qq.y : qq.x, kp = half ? kk.y : kk.x;
                    f2 d01 = c01, d23 = c23;
                    if (GATE == 1)
                        d01 = d23 = half ? aa.y : aa.x;
                    f2 &x01 = half ? o01 : e01, &x23 = half ? o23 : e23;
                    if (!BWD) {
                        S01[j] = fma2(S01[j], d01, mul2(kp, w.x));
                        S23[j] = fma2(S23[j], d23, mul2(kp, w.y));
                        x01 = fma2(qp, S01[j], x01);
                        x23 = fma2(qp, S23[j], x23);
                    } else {
                        S01[j] = fma2(qp, w.x, S01[j]);
                        S23[j] = fma2(qp, w.y, S23[j]);
                        x01 = fma2(kp, S01[j], x01);
                        x23 = fma2(kp, S23[j], x23);
                        S01[j] = mul2(S01[j], d01);
                        S23[j] = mul2(S23[j], d23);
                    }
                }
            }
            const float2 p01 = unpack2(add2(e01, o01)), p23 = unpack2(add2(e23, o23));
            if (sp.rgn == 1) {
                hv[i] = p01;
                hw[i] = p23;
            } else {
                const float2 keep = bA ? p23 : p01, send = bA ? p01 : p23;
                hv[i].x = keep.x + __shfl_xor_sync(0xffffffffu, send.x, sp.qw);
                hv[i].y = keep.y + __shfl_xor_sync(0xffffffffu, send.y, sp.qw);
            }
        }
        if (sp.rgn == 1) {
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int64_t op = token(b0 + u0 + i) * a.out.st + c0;
                const float x[4] = {hv[i].x, hv[i].y, hw[i].x, hw[i].y};
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c0 + c < E)
                        put(op + c, sc * x[c]);
            }
            return;
        }
        if (sp.rgn == 2) {
            const int c = c0 + (bA ? 2 : 0);
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int64_t op = token(b0 + u0 + i) * a.out.st;
                if (c < E)
                    put(op + c, sc * hv[i].x);
                if (c + 1 < E)
                    put(op + c + 1, sc * hv[i].y);
            }
            return;
        }
        // one column per lane over the second bit, then plain sums
        float val[NT];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const float keep = bB ? hv[i].y : hv[i].x;
            const float send = bB ? hv[i].x : hv[i].y;
            val[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * sp.qw);
        }
        for (int off = 4 * sp.qw; off < 32; off <<= 1) {
#pragma unroll
            for (int i = 0; i < NT; ++i)
                val[i] += __shfl_xor_sync(0xffffffffu, val[i], off);
        }
        const int c = c0 + (bA ? 2 : 0) + (bB ? 1 : 0);
        if (rg < 4 && c < E) {
#pragma unroll
            for (int i = 0; i < NT; ++i)
                put(token(b0 + u0 + i) * a.out.st + c, sc * val[i]);
        }
    };
    auto compute = [&](int64_t b0, int Lb) {
        int u0 = 0;
        for (; !SHORTC && u0 + 4 <= Lb; u0 += 4)
            process(std::integral_constant<int, 4>(), b0, u0);
        for (; u0 < Lb; ++u0)
            process(std::integral_constant<int, 1>(), b0, u0);
    };

    if (pre.q) {
        // the whole (short) sequence is in shared memory already
        const T *pq = static_cast<const T *>(pre.q), *pk = static_cast<const T *>(pre.k);
        const T *pv = static_cast<const T *>(pre.v);
        const int Lb = (int)len;
        for (int idx = tid; idx < Lb * RR; idx += nthr) {
            const int u = idx / RR, r = idx % RR;
            const bool ok = r < D;
            put_row(u, r, ok ? ld_tok(pq + u * D + r) : 0.f, ok ? ld_tok(pk + u * D + r) : 0.f,
                    GATE == 1 && ok ? expf(gh + pre.g[u * D + r]) : 1.f);
        }
        for (int idx = tid; idx < Lb * sp.cw; idx += nthr) {
            const int u = idx / sp.cw, c = idx % sp.cw;
            vs[idx] = cb + c < E ? ld_tok(pv + u * sp.cw + c) : 0.f;
        }
        sync();
        compute(0, Lb);
        sync();   // the tables are free again
        return;
    }
    // ASYNC (chosen on the host when every row is 16-byte aligned):
    // double-buffered 16-byte cp.async copies of the raw rows, the next
    // block's copies in flight while this block is converted and computed.
    if (!ASYNC) {
        for (int64_t b0 = 0; b0 < len; b0 += tbe) {
            const int Lb = (int)(len - b0 < tbe ? len - b0 : tbe);
            load_sync(b0, Lb);
            sync();
            compute(b0, Lb);
            sync();   // the next block overwrites the tables
        }
    } else {
        const int esz = (int)sizeof(T);
        T *rq = reinterpret_cast<T *>(acs + (GATE == 2 ? tbe * sp.cw : 0));
        T *rk = rq + 2 * tbe * D;
        T *rv = rk + 2 * tbe * D;
        float *rgt = reinterpret_cast<float *>(rv + 2 * tbe * sp.cw);   // gate rows or tiles
        const int gw = GATE == 1 ? D : sp.cw;                            // gate floats per token
        const int ecols = E - cb < sp.cw ? E - cb : sp.cw;               // valid columns here
        const int cq = D * esz / 16, cv = ecols * esz / 16;
        const int cg = GATE == 1 ? D / 4 : (GATE == 2 ? ecols / 4 : 0);
        auto issue = [&](int64_t b0, int Lb, int buf) {
            const int per = 2 * cq + cv + cg;
            for (int idx = tid; idx < Lb * per; idx += nthr) {
                const int u = idx / per;
                int r = idx % per;
                const int64_t t = token(b0 + u);
                const void *src;
                void *dst;
                if (r < cq) {
                    src = qb + t * a.q.st + r * (16 / esz);
                    dst = rq + ((size_t)buf * tbe + u) * D + r * (16 / esz);
                } else if ((r -= cq) < cq) {
                    src = kb + t * a.k.st + r * (16 / esz);
                    dst = rk + ((size_t)buf * tbe + u) * D + r * (16 / esz);
                } else if ((r -= cq) < cv) {
                    src = vb + t * a.v.st + cb + r * (16 / esz);
                    dst = rv + ((size_t)buf * tbe + u) * sp.cw + r * (16 / esz);
                } else {
                    r -= cv;
                    src = gb + t * a.gate.st + (GATE == 2 ? cb : 0) + 4 * r;
                    dst = rgt + ((size_t)buf * tbe + u) * gw + 4 * r;
                }
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                             "l"(src)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        auto convert = [&](int Lb, int buf) {
            for (int idx = tid; idx < Lb * RR; idx += nthr) {
                const int u = idx / RR, r = idx % RR;
                const size_t rr = ((size_t)buf * tbe + u) * D + r;
                const bool ok = r < D;
                put_row(u, r, ok ? ld_tok(rq + rr) : 0.f, ok ? ld_tok(rk + rr) : 0.f,
                        GATE == 1 && ok ? expf(gh + rgt[((size_t)buf * tbe + u) * gw + r]) : 1.f);
            }
            for (int idx = tid; idx < Lb * sp.cw; idx += nthr) {
                const int u = idx / sp.cw, c = idx % sp.cw;
                const bool ok = c < ecols;
                vs[idx] = ok ? ld_tok(rv + ((size_t)buf * tbe + u) * sp.cw + c) : 0.f;
                if (GATE == 2)
                    acs[idx] = ok ? expf(gh + rgt[((size_t)buf * tbe + u) * gw + c]) : 1.f;
            }
        };
        int it = 0;
        if (len > 0)
            issue(0, (int)(len < tbe ? len : tbe), 0);
        for (int64_t b0 = 0; b0 < len; b0 += tbe, ++it) {
            const int Lb = (int)(len - b0 < tbe ? len - b0 : tbe);
            if (b0 + tbe < len) {
                issue(b0 + tbe, (int)(len - b0 - tbe < tbe ? len - b0 - tbe : tbe), (it + 1) & 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            sync();   // every thread's copies of this block landed
            convert(Lb, it & 1);
            sync();
            compute(b0, Lb);
            sync();   // the tables and this raw buffer are free again
        }
    }

}

// One CTA per (sequence, head, column tile).  SHORTC: fits two CTAs per SM
// (128 registers), twice the state loads in flight; otherwise one CTA per SM.
template <typename T, bool BWD, int GATE, bool ASYNC, bool SHORTC>
__global__ void __launch_bounds__(MAXW * 32, SHORTC ? 2 : 1) token_kernel(SweepArgs a)
{
    const int D = a.D, E = a.E;
    const Shape sp = token_shape(D, E, RP);
    const int tile = (int)(blockIdx.x % sp.tiles);
    const int h = (int)((blockIdx.x / sp.tiles) % a.H);
    const int n = (int)(blockIdx.x / ((unsigned)sp.tiles * a.H));
    // gated form: only the (sequence, head) pairs the chunked form left over
    if (a.gla_flags && a.gla_flags[(int64_t)n * a.H + h] != a.gla_flag_run)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qd = lane & (sp.qw - 1), rg = lane / sp.qw;
    const int c0 = tile * sp.cw + warp * sp.wc + 4 * qd;
    const int r0 = RP * rg;
    const int64_t sbase = ((int64_t)n * a.H + h) * (int64_t)D * E;
    extern __shared__ __align__(16) float sh[];

    // ---- the state block: S[j] = state(r0 + j, c0 .. c0 + 3) ----------------
    // Loaded as 16-byte pieces along whichever state axis is contiguous,
    // element by element otherwise; these loads are in flight while the first
    // tokens are copied below.
    // the state as column pairs: S01[j] = columns c0, c0 + 1 of row r0 + j,
    // S23[j] = columns c0 + 2, c0 + 3
    f2 S01[RP], S23[RP];
    {
        const float *p = a.s_in.p;
        // bulk prefetches of whole (sequence, head) state blocks into L2 when
        // they are contiguous: this CTA's own, and the one of the CTA that
        // starts a resident wave later, so that its loads find the state in
        // L2 instead of each waiting a full trip to HBM
        if (threadIdx.x == 0 && p && (reinterpret_cast<uintptr_t>(p) & 15) == 0 &&
            ((a.s_in.cs == 1 && a.s_in.rs == E) || (a.s_in.rs == 1 && a.s_in.cs == D)) &&
            ((int64_t)D * E) % 4 == 0) {
            const uint32_t bytes = (uint32_t)((int64_t)D * E * 4);
            if (tile == 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + sbase),
                             "r"(bytes)
                             : "memory");
            const int64_t ahead = (int64_t)blockIdx.x + a.prefetch_ctas;
            if (a.prefetch_ctas > 0 && ahead < (int64_t)gridDim.x && ahead % sp.tiles == 0) {
                const int64_t hn = ahead / sp.tiles;   // (sequence, head) of that CTA
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 p + hn * (int64_t)D * E),
                             "r"(bytes)
                             : "memory");
            }
        }
        const int64_t rs = a.s_in.rs, cs = a.s_in.cs;
        const bool al = p && (reinterpret_cast<uintptr_t>(p) & 15) == 0;
        if (p && al && cs == 1 && rs % 4 == 0 && E % 4 == 0) {
            // straight into the column pairs: nothing waits on these loads
            // before the first token needs the state
#pragma unroll
            for (int j = 0; j < RP; ++j) {
                ulonglong2 x = make_ulonglong2(0ull, 0ull);
                if (c0 < E && r0 + j < D)
                    x = *reinterpret_cast<const ulonglong2 *>(p + sbase + (int64_t)(r0 + j) * rs + c0);
                S01[j] = x.x;
                S23[j] = x.y;
            }
        } else {
            float4 S[RP];
            if (p && al && rs == 1 && cs % 4 == 0 && D % 4 == 0) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j4 = 0; j4 < RP / 4; ++j4) {
                        const float4 x = c0 + c < E && r0 + 4 * j4 < D
                                             ? *reinterpret_cast<const float4 *>(
                                                   p + sbase + (int64_t)(c0 + c) * cs + r0 + 4 * j4)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                        comp(S[4 * j4 + 0], c) = x.x;
                        comp(S[4 * j4 + 1], c) = x.y;
                        comp(S[4 * j4 + 2], c) = x.z;
                        comp(S[4 * j4 + 3], c) = x.w;
                    }
            } else {
#pragma unroll
                for (int j = 0; j < RP; ++j)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        comp(S[j], c) = p && c0 + c < E && r0 + j < D
                                            ? p[sbase + (int64_t)(r0 + j) * rs +
                                                (int64_t)(c0 + c) * cs]
                                            : 0.f;
            }
#pragma unroll
            for (int j = 0; j < RP; ++j) {
                S01[j] = pack2(S[j].x, S[j].y);
                S23[j] = pack2(S[j].z, S[j].w);
            }
        }
    }

    token_loop<T, BWD, GATE, ASYNC, SHORTC>(a, sp, n, h, tile, threadIdx.x, blockDim.x, sh, S01,
                                            S23, CtaSync());

    // ---- the state block out --------------------------------------------------
    float4 S[RP];
#pragma unroll
    for (int j = 0; j < RP; ++j) {
        const float2 lo = unpack2(S01[j]), hi = unpack2(S23[j]);
        S[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    float *p = a.s_out.p;
    if (p) {
        const int64_t rs = a.s_out.rs, cs = a.s_out.cs;
        const bool al = (reinterpret_cast<uintptr_t>(p) & 15) == 0;
        if (al && cs == 1 && rs % 4 == 0 && E % 4 == 0) {
            if (c0 < E) {
#pragma unroll
                for (int j = 0; j < RP; ++j)
                    if (r0 + j < D)
                        *reinterpret_cast<float4 *>(p + sbase + (int64_t)(r0 + j) * rs + c0) = S[j];
            }
        } else if (al && rs == 1 && cs % 4 == 0 && D % 4 == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j4 = 0; j4 < RP / 4; ++j4)
                    if (c0 + c < E && r0 + 4 * j4 < D)
                        *reinterpret_cast<float4 *>(p + sbase + (int64_t)(c0 + c) * cs + r0 +
                                                    4 * j4) =
                            make_float4(comp(S[4 * j4 + 0], c), comp(S[4 * j4 + 1], c),
                                        comp(S[4 * j4 + 2], c), comp(S[4 * j4 + 3], c));
        } else {
#pragma unroll
            for (int j = 0; j < RP; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c0 + c < E && r0 + j < D)
                        p[sbase + (int64_t)(r0 + j) * rs + (int64_t)(c0 + c) * cs] = comp(S[j], c);
        }
    }
}

// ---- streamed decode ----------------------------------------------------------
// Forward-type calls of at most SHORT_MAX_T tokens with whole (sequence,
// head) state blocks contiguous ([D][E] rows, E a multiple of 4) and one
// column tile: one
// persistent CTA per SM walks the (sequence, head) blocks.  A copy warp moves
// each fp32 state block (D E 4 bytes) into a ring of NS shared-memory buffers
// by one 1-D bulk copy and back out by one bulk store, so that NS - 1 blocks
// are in flight while the compute warps, which hold only the block they work
// on, run the tokens.  Waits on the ring are bounded (2 s); on expiry the CTA
// records LA_ERR_TIMEOUT, drains its copies and returns.  Blocks of up to
// STREAM_MAX_T tokens run token by token, longer ones (up to TB tokens, no
// gate) as one chunk of the chunked form (chunk_decode).

// Longest call that the streamed kernel runs token by token: beyond it one CTA
// per SM is compute-bound on the token loop.
constexpr int STREAM_MAX_T = 4;

__device__ int g_token_error;
constexpr uint64_t TOK_WAIT_NS = 2000000000ull;
constexpr int TOK_ERR_TIMEOUT = 4;

__device__ __forceinline__ void bulk_load_1d(void *dst, const void *src, uint32_t bytes,
                                             uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(sm100::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(sm100::smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_store_1d(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(sm100::smem_u32(src)), "r"(bytes)
                 : "memory");
}
// every committed bulk store of this thread complete (written)
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Bounded wait: false when the CTA is aborting or this wait ran out.
__device__ __forceinline__ bool tok_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (sm100::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = sm100::globaltimer_ns();
    for (;;) {
        if (sm100::mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (sm100::globaltimer_ns() - t0 > TOK_WAIT_NS) {
            *abort_flag = 1;
            atomicExch(&g_token_error, TOK_ERR_TIMEOUT);
            return false;
        }
    }
}
// Bounded wait that ignores the abort flag (draining this CTA's own copies).
__device__ __forceinline__ void tok_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = sm100::globaltimer_ns();
    while (!sm100::mbar_try_wait(bar, parity))
        if (sm100::globaltimer_ns() - t0 > TOK_WAIT_NS) {
            atomicExch(&g_token_error, TOK_ERR_TIMEOUT);
            return;
        }
}
// AND of `ok` over the first `count` threads (barrier 2)
__device__ __forceinline__ bool named_and(bool ok, int count)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.and.pred p, 2, %2, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"(ok ? 1u : 0u), "r"(count)
                 : "memory");
    return r != 0;
}

// Shared memory (floats) of the chunk form's tables: q and k rows as paired
// row tables [TB][rgn][SK], the scores [TB][TB].
__host__ __device__ inline size_t chunk_table_floats(int rgn)
{
    return (size_t)2 * TB * rgn * pair_stride(RP) + TB * TB;
}

// Bytes of one raw token slot of the streamed kernel: q, k rows [tbe][D] and
// value rows [tbe][cw] of the token dtype, row gates [tbe][D] fp32.
__host__ __device__ inline size_t stream_slot_bytes(const Shape &sp, int D, int tbe, int esz,
                                                    int gate)
{
    return ((size_t)tbe * ((size_t)2 * D * esz + (size_t)sp.cw * esz +
                           (gate == 1 ? (size_t)D * 4 : 0)) + 15) / 16 * 16;
}
// Shared memory of the streamed kernel: NS state buffers, NS raw token slots,
// 2 NS barriers, the abort word (16 bytes), then the token tables (of the
// token loop, or of the chunk form).
__host__ __device__ inline size_t stream_smem_bytes(const Shape &sp, int D, int E, int tbe,
                                                    int esz, int gate, int ns, bool chunk)
{
    return (size_t)ns * D * E * 4 + (size_t)ns * stream_slot_bytes(sp, D, tbe, esz, gate) +
           (size_t)2 * ns * 8 + 16 +
           (chunk ? chunk_table_floats(sp.rgn) * 4
                  : token_smem_bytes(sp, RP, D, tbe, 4, gate, false));
}

__device__ __forceinline__ f2 shfl_xor2(f2 x, int m)
{
    const float2 v = unpack2(x);
    return pack2(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m));
}
// eight consecutive token values (16-byte aligned) as fp32
template <typename T> __device__ __forceinline__ void ld8(const T *p, float (&x)[8]);
template <> __device__ __forceinline__ void ld8<float>(const float *p, float (&x)[8])
{
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
template <> __device__ __forceinline__ void ld8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&x)[8])
{
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
// four consecutive token values (8-byte aligned for bf16, 16 for fp32)
template <typename T> __device__ __forceinline__ float4 ld4(const T *p);
template <> __device__ __forceinline__ float4 ld4<float>(const float *p)
{
    return *reinterpret_cast<const float4 *>(p);
}
template <> __device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// One (sequence, head) block of L <= TB tokens as one chunk of the chunked
// form (forward-type, the head's decay gamma = exp(g[h]) only), for the
// streamed kernel: with the entering state S0 and processing index t,
//   o_t = s gamma^(t+1) q_t S0 + s sum_{u <= t} gamma^(t-u) (q_t . k_u) v_u,
//   S   = gamma^L S0 + sum_u gamma^(L-1-u) k_u^T v_u,
// the recurrence summed in closed form (ejkernel `recurrent` docstring, "The
// core update"; the Lightning Attention-2 paper's intra/inter split for one
// block).  Each thread keeps its 16-row x 4-column state block in registers
// (the layout of token_loop): the inter term for all L tokens is one pass
// over its rows (fp32 pairs from the paired q table, 2 L FMA2 per row), then
// a reduce-scatter over the RGN row-group lanes leaves each lane the sums of
// its share of the tokens; the update is one more pass (paired k table).  The
// token loop's reduction and state pass per token become one reduction per
// group of 8 (or 16) tokens and one state pass per block.  All arithmetic fp32.  Raw rows (processing
// order): q, k [L][D], v [L][cw] of the token dtype, 16-byte aligned.
template <typename T, int RGN>
__device__ __forceinline__ void chunk_decode(const SweepArgs &a, const Shape &sp, int n, int h,
                                             int tid, int ncomp, float *tab, f2 (&S01)[RP],
                                             f2 (&S23)[RP], const T *rq, const T *rk,
                                             const T *rv)
{
    constexpr int QW = 32 / RGN, SK = pair_stride(RP);
    const int D = a.D, E = a.E;
    const int warp = tid >> 5, lane = tid & 31;
    const int qd = lane & (QW - 1), rg = lane / QW;
    const int c0 = warp * sp.wc + 4 * qd;
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
    const float g = a.g[h], scale = a.scale;
    float *QQ = tab;                      // s gamma^(t+1) q_t, paired rows
    float *KK = QQ + TB * RGN * SK;       // gamma^(L-1-u) k_u, paired rows
    float *P = KK + TB * RGN * SK;        // [t][u]: s gamma^(t-u) q_t . k_u, u <= t
    for (int i = tid; i < L * RGN * RP; i += ncomp) {
        const int t = i / (RGN * RP), r = i % (RGN * RP);
        float qv = 0.f, kv = 0.f;
        if (r < D) {
            qv = ld_tok(rq + t * D + r) * scale * expf(g * (float)(t + 1));
            kv = ld_tok(rk + t * D + r) * expf(g * (float)(L - 1 - t));
        }
        const int at = (t * RGN + r / RP) * SK + 2 * (r % RP);
        *reinterpret_cast<float2 *>(QQ + at) = make_float2(qv, qv);
        *reinterpret_cast<float2 *>(KK + at) = make_float2(kv, kv);
    }
    for (int i = tid; i < TB * TB; i += ncomp) {
        const int t = i / TB, u = i % TB;
        float sc = 0.f;
        if (u <= t && t < L) {
            // pieces of 8 channels, started at piece u: the 16 lanes of a
            // half warp read 16 different k rows in different banks
            const int np = D / 8;
            float acc = 0.f;
            for (int p = 0, pc = u % np; p < np; ++p, pc = pc + 1 == np ? 0 : pc + 1) {
                float xq[8], xk[8];
                ld8(rq + t * D + 8 * pc, xq);
                ld8(rk + u * D + 8 * pc, xk);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc = fmaf(xq[e], xk[e], acc);
            }
            sc = acc * scale * expf(g * (float)(t - u));
        }
        P[i] = sc;
    }
    NamedSync{ncomp}();

    // Tokens in groups of TG (8, or 16 for 16 row groups: the live sums stay
    // at 4 TG registers).  Inter term: A[t] = (s gamma^(t+1) q_t) . S0 over
    // this thread's rows; then a reduce-scatter over the row-group lanes
    // (lane bits of rg, highest first) leaves the lane of row group rg the
    // tokens t0 + rg TPG .. t0 + rg TPG + TPG - 1, summed over all rows, in
    // A[0 .. TPG - 1]; then the intra term and the output.
    constexpr int TG = RGN > 8 ? TB : 8, TPG = TG / RGN;
    constexpr int LEVELS = RGN >= 16 ? 4 : RGN >= 8 ? 3 : RGN >= 4 ? 2 : RGN >= 2 ? 1 : 0;
    T *ob = static_cast<T *>(a.out.p) + row * a.out.sb + (int64_t)h * a.out.sh + c0;
#pragma unroll 1
    for (int t0 = 0; t0 < L; t0 += TG) {
        f2 A01[TG], A23[TG];
#pragma unroll
        for (int k = 0; k < TG; ++k) {
            A01[k] = 0ull;
            A23[k] = 0ull;
            if (t0 + k < L) {
                const float *qp = QQ + ((t0 + k) * RGN + rg) * SK;
#pragma unroll
                for (int j = 0; j < RP; j += 2) {
                    const ulonglong2 w = *reinterpret_cast<const ulonglong2 *>(qp + 2 * j);
                    A01[k] = fma2(w.x, S01[j], A01[k]);
                    A23[k] = fma2(w.x, S23[j], A23[k]);
                    A01[k] = fma2(w.y, S01[j + 1], A01[k]);
                    A23[k] = fma2(w.y, S23[j + 1], A23[k]);
                }
            }
        }
#pragma unroll
        for (int l = 0; l < LEVELS; ++l) {
            const int lv = RGN >> (l + 1), half = TG >> (l + 1);
            const bool hi = (rg & lv) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const f2 k01 = hi ? A01[i + half] : A01[i], s01 = hi ? A01[i] : A01[i + half];
                const f2 k23 = hi ? A23[i + half] : A23[i], s23 = hi ? A23[i] : A23[i + half];
                A01[i] = add2(k01, shfl_xor2(s01, lv * QW));
                A23[i] = add2(k23, shfl_xor2(s23, lv * QW));
            }
        }
        if (c0 < E) {
#pragma unroll
            for (int k = 0; k < TPG; ++k) {
                const int t = t0 + rg * TPG + k;
                if (t >= L)
                    break;
                const float2 i01 = unpack2(A01[k]), i23 = unpack2(A23[k]);
                float o0 = i01.x, o1 = i01.y, o2 = i23.x, o3 = i23.y;
                for (int u = 0; u <= t; ++u) {
                    const float pr = P[t * TB + u];
                    const float4 v4 = ld4(rv + u * sp.cw + c0);
                    o0 = fmaf(pr, v4.x, o0);
                    o1 = fmaf(pr, v4.y, o1);
                    o2 = fmaf(pr, v4.z, o2);
                    o3 = fmaf(pr, v4.w, o3);
                }
                T *op = ob + (bos + (a.reverse ? L - 1 - t : t)) * a.out.st;
                st_tok(op, o0);
                st_tok(op + 1, o1);
                st_tok(op + 2, o2);
                st_tok(op + 3, o3);
            }
        }
    }
    // the state: gamma^L S0 + sum_u (gamma^(L-1-u) k_u)^T v_u
    const float gl = expf(g * (float)L);
    const f2 gl2 = pack2(gl, gl);
#pragma unroll
    for (int j = 0; j < RP; ++j) {
        S01[j] = mul2(S01[j], gl2);
        S23[j] = mul2(S23[j], gl2);
    }
    if (c0 < E) {
#pragma unroll 2
        for (int u = 0; u < L; ++u) {
            const float4 v4 = ld4(rv + u * sp.cw + c0);
            const f2 v01 = pack2(v4.x, v4.y), v23 = pack2(v4.z, v4.w);
            const float *kp = KK + (u * RGN + rg) * SK;
#pragma unroll
            for (int j = 0; j < RP; j += 2) {
                const ulonglong2 w = *reinterpret_cast<const ulonglong2 *>(kp + 2 * j);
                S01[j] = fma2(w.x, v01, S01[j]);
                S23[j] = fma2(w.x, v23, S23[j]);
                S01[j + 1] = fma2(w.y, v01, S01[j + 1]);
                S23[j + 1] = fma2(w.y, v23, S23[j + 1]);
            }
        }
    }
}

// CRGN > 0: the blocks run as one chunk each (chunk_decode, CRGN row groups)
// instead of token by token.
template <typename T, int GATE, int CRGN = 0>
__global__ void __launch_bounds__(MAXW * 32 + 32, 1) stream_kernel(SweepArgs a, int ns)
{
    const int D = a.D, E = a.E;
    const Shape sp = token_shape(D, E, RP);   // one column tile
    const int ncomp = sp.wpc * 32;            // compute threads; the copy warp follows
    const int heads = a.N * a.H;
    const int64_t SE = (int64_t)D * E;
    const uint32_t sbytes = (uint32_t)(SE * 4);
    const int tbe = token_block(a.max_len);
    const int esz = (int)sizeof(T);
    const size_t slot = stream_slot_bytes(sp, D, tbe, esz, GATE);
    extern __shared__ __align__(128) float sh[];
    float *sbuf = sh;
    uint8_t *raw = reinterpret_cast<uint8_t *>(sbuf + ns * SE);
    uint64_t *full = reinterpret_cast<uint64_t *>(raw + ns * slot);
    uint64_t *done = full + ns;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(done + ns);
    float *tok = reinterpret_cast<float *>(done + ns) + 4;
    const int tid = threadIdx.x;
    const bool has_in = a.s_in.p != nullptr, has_out = a.s_out.p != nullptr;
    // raw rows of slot b: q, k [tbe][D], v [tbe][cw], gate [tbe][D]
    auto slot_q = [&](int b) { return reinterpret_cast<T *>(raw + b * slot); };
    auto slot_k = [&](int b) { return slot_q(b) + tbe * D; };
    auto slot_v = [&](int b) { return slot_k(b) + tbe * D; };
    auto slot_g = [&](int b) { return reinterpret_cast<float *>(slot_v(b) + tbe * sp.cw); };
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
        for (int i = 0; i < ns; ++i) {
            sm100::mbar_init(&full[i], 1);
            sm100::mbar_init(&done[i], 1);
        }
        *abort_flag = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();

    if (tid >= ncomp) {
        // ---- copy warp ----
        const int lane = tid - ncomp;
        // diagnostic (la_debug_withhold_next_handoff): the first block is
        // never copied, so the compute warps' bounded wait on it runs out
        const int skip = a.withhold_handoff ? 1 : 0;
        int li = 0;
        bool ok = true;
        for (int hn = blockIdx.x; hn < heads; hn += gridDim.x, ++li) {
            const int buf = li % ns;
            if (li < skip)
                continue;
            if (lane == 0 && li >= ns) {
                // the block ns heads back has left this buffer: store it
                ok = tok_wait(&done[buf], ((li - ns) / ns) & 1, abort_flag);
                if (ok && has_out) {
                    bulk_store_1d(a.s_out.p + (int64_t)(hn - ns * (int)gridDim.x) * SE,
                                  sbuf + buf * SE, sbytes);
                    sm100::bulk_commit_group();
                    sm100::bulk_wait_read_all();   // before the buffer is refilled
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            int64_t row, bos, len;
            seq(hn, row, bos, len);
            const int h = hn % a.H;
            const uint32_t rowb = (uint32_t)(2 * D * esz + E * esz + (GATE == 1 ? D * 4 : 0));
            const uint32_t tx = (has_in ? sbytes : 0u) + (uint32_t)len * rowb;
            if (lane == 0) {
                if (tx)
                    sm100::mbar_arrive_expect_tx(&full[buf], tx);
                else
                    sm100::mbar_arrive(&full[buf]);
                if (has_in)
                    bulk_load_1d(sbuf + buf * SE, a.s_in.p + (int64_t)hn * SE, sbytes, &full[buf]);
            }
            __syncwarp();
            // token rows in processing order (forward-type: reversed when reverse)
            const int nrow = (int)len * (GATE == 1 ? 4 : 3);
            for (int i = lane; i < nrow; i += 32) {
                const int u = i / (GATE == 1 ? 4 : 3), kind = i % (GATE == 1 ? 4 : 3);
                const int64_t t = bos + (a.reverse ? len - 1 - u : u);
                if (kind == 0)
                    bulk_load_1d(slot_q(buf) + u * D,
                                 reinterpret_cast<const T *>(a.q.p) + row * a.q.sb + t * a.q.st +
                                     (int64_t)(h / a.q.hdiv) * a.q.sh,
                                 (uint32_t)(D * esz), &full[buf]);
                else if (kind == 1)
                    bulk_load_1d(slot_k(buf) + u * D,
                                 reinterpret_cast<const T *>(a.k.p) + row * a.k.sb + t * a.k.st +
                                     (int64_t)(h / a.k.hdiv) * a.k.sh,
                                 (uint32_t)(D * esz), &full[buf]);
                else if (kind == 2)
                    bulk_load_1d(slot_v(buf) + u * sp.cw,
                                 reinterpret_cast<const T *>(a.v.p) + row * a.v.sb + t * a.v.st +
                                     (int64_t)(h / a.v.hdiv) * a.v.sh,
                                 (uint32_t)(E * esz), &full[buf]);
                else
                    bulk_load_1d(slot_g(buf) + u * D,
                                 a.gate.p + row * a.gate.sb + t * a.gate.st +
                                     (int64_t)h * a.gate.sh,
                                 (uint32_t)(D * 4), &full[buf]);
            }
            __syncwarp();
        }
        if (lane != 0)
            return;
        const int issued = li;
        if (ok) {
            // the last blocks
            for (int lj = issued > ns ? issued - ns : 0; lj < issued; ++lj) {
                const int buf = lj % ns;
                if (!tok_wait(&done[buf], (lj / ns) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                if (has_out)
                    bulk_store_1d(a.s_out.p + (int64_t)(blockIdx.x + lj * (int)gridDim.x) * SE,
                                  sbuf + buf * SE, sbytes);
            }
            if (has_out)
                sm100::bulk_commit_group();
        }
        if (!ok) {
            // no copy into this CTA's shared memory may outlive it
            for (int lj = issued - ns > skip ? issued - ns : skip; lj < issued; ++lj)
                tok_drain(&full[lj % ns], (lj / ns) & 1);
        }
        bulk_wait_all();
        return;
    }

    // ---- compute warps ----
    const int warp = tid >> 5, lane = tid & 31;
    const int qd = lane & (sp.qw - 1), rg = lane / sp.qw;
    const int c0 = warp * sp.wc + 4 * qd;
    const int r0 = RP * rg;
    int li = 0;
    for (int hn = blockIdx.x; hn < heads; hn += gridDim.x, ++li) {
        const int buf = li % ns;
        float *sb = sbuf + buf * SE;
        if (!named_and(tok_wait(&full[buf], (li / ns) & 1, abort_flag), ncomp))
            break;
        f2 S01[RP], S23[RP];
#pragma unroll
        for (int j = 0; j < RP; ++j) {
            ulonglong2 x = make_ulonglong2(0ull, 0ull);
            if (has_in && c0 < E && r0 + j < D)
                x = *reinterpret_cast<const ulonglong2 *>(sb + (int64_t)(r0 + j) * E + c0);
            S01[j] = x.x;
            S23[j] = x.y;
        }
        if constexpr (CRGN > 0) {
            chunk_decode<T, CRGN>(a, sp, hn / a.H, hn % a.H, tid, ncomp, tok, S01, S23,
                                  slot_q(buf), slot_k(buf), slot_v(buf));
        } else {
            RawRows pre;
            pre.q = slot_q(buf);
            pre.k = slot_k(buf);
            pre.v = slot_v(buf);
            pre.g = slot_g(buf);
            token_loop<T, false, GATE, false, true>(a, sp, hn / a.H, hn % a.H, 0, tid, ncomp, tok,
                                                   S01, S23, NamedSync{ncomp}, pre);
        }
        if (has_out && c0 < E) {
#pragma unroll
            for (int j = 0; j < RP; ++j)
                if (r0 + j < D)
                    *reinterpret_cast<ulonglong2 *>(sb + (int64_t)(r0 + j) * E + c0) =
                        make_ulonglong2(S01[j], S23[j]);
        }
        sm100::fence_proxy_async_smem();   // the writes, visible to the bulk store
        NamedSync{ncomp}();
        if (tid == 0)
            sm100::mbar_arrive(&done[buf]);
    }
}

// Rows of every tensor 16-byte aligned (base, strides, widths): the copies
// can be 16-byte cp.async.
bool rows_aligned(const SweepArgs &a, int esz)
{
    auto ok = [&](const void *p, int64_t sb, int64_t st, int64_t sh, int64_t es) {
        return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && (sb * es) % 16 == 0 &&
               (st * es) % 16 == 0 && (sh * es) % 16 == 0;
    };
    bool r = ok(a.q.p, a.q.sb, a.q.st, a.q.sh, esz) && ok(a.k.p, a.k.sb, a.k.st, a.k.sh, esz) &&
             ok(a.v.p, a.v.sb, a.v.st, a.v.sh, esz) && (a.D * esz) % 16 == 0 &&
             (a.E * esz) % 16 == 0;
    if (a.gate.p)
        r = r && ok(a.gate.p, a.gate.sb, a.gate.st, a.gate.sh, 4) && a.D % 4 == 0 && a.E % 4 == 0;
    return r;
}

template <typename K>
cudaError_t launch_one(K kernel, const SweepArgs &a0, cudaStream_t s, int gate, bool async)
{
    SweepArgs a = a0;
    const Shape sp = token_shape(a.D, a.E, 16);
    const size_t smem =
        token_smem_bytes(sp, 16, a.D, token_block(a.max_len), a.bf16 ? 2 : 4, gate, async);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    // CTAs resident at once: the distance of the L2 prefetch ahead
    int per_sm = 0, dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, sp.wpc * 32, smem);
    if (e != cudaSuccess)
        return e;
    a.prefetch_ctas = (int64_t)per_sm * sms;
    const int64_t blocks = (int64_t)a.N * a.H * sp.tiles;
    kernel<<<(unsigned)blocks, sp.wpc * 32, smem, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

template <typename T, bool BWD, bool ASYNC, bool SHORTC>
cudaError_t launch_gate(const SweepArgs &a, cudaStream_t s)
{
    if (!a.gate.p)
        return launch_one(token_kernel<T, BWD, 0, ASYNC, SHORTC>, a, s, 0, ASYNC);
    return a.gate.cols ? launch_one(token_kernel<T, BWD, 2, ASYNC, SHORTC>, a, s, 2, ASYNC)
                       : launch_one(token_kernel<T, BWD, 1, ASYNC, SHORTC>, a, s, 1, ASYNC);
}

template <typename T, bool BWD, bool SHORTC>
cudaError_t launch_rows(const SweepArgs &a, cudaStream_t s)
{
    return rows_aligned(a, (int)sizeof(T)) ? launch_gate<T, BWD, true, SHORTC>(a, s)
                                           : launch_gate<T, BWD, false, SHORTC>(a, s);
}

// The streamed decode kernel when the call qualifies (forward-type, short,
// no gate or a row gate, contiguous 16-byte aligned state blocks, one column
// tile, at least two ring buffers in shared memory, more blocks than SMs);
// cudaErrorNotSupported otherwise.
template <typename T> cudaError_t try_stream(const SweepArgs &a, cudaStream_t s)
{
    const Shape sp = token_shape(a.D, a.E, RP);
    auto state_ok = [&](const float *p, int64_t rs, int64_t cs) {
        return !p || ((reinterpret_cast<uintptr_t>(p) & 15) == 0 && rs == a.E && cs == 1);
    };
    const int esz = (int)sizeof(T);
    // up to STREAM_MAX_T tokens token by token; up to TB tokens (no gate, key
    // width a multiple of 8) as one chunk
    const bool chunk = a.max_len > STREAM_MAX_T;
    if (a.max_len > TB || (chunk && (a.gate.p || a.D % 8)) || a.gate.cols || a.gla_flags ||
        a.out_f32 || sp.tiles != 1 || a.E % 4 || !state_ok(a.s_in.p, a.s_in.rs, a.s_in.cs) ||
        !state_ok(a.s_out.p, a.s_out.rs, a.s_out.cs) || !rows_aligned(a, esz))
        return cudaErrorNotSupported;
    int dev = 0, sms = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    const int64_t heads = (int64_t)a.N * a.H;
    if (heads < 2 * (int64_t)sms || heads > 0x7fffffff)
        return cudaErrorNotSupported;
    const int gate = a.gate.p ? 1 : 0, tbe = token_block(a.max_len);
    int ns = 3;
    while (ns >= 2 && stream_smem_bytes(sp, a.D, a.E, tbe, esz, gate, ns, chunk) > (size_t)optin)
        --ns;
    if (ns < 2)
        return cudaErrorNotSupported;
    const size_t smem = stream_smem_bytes(sp, a.D, a.E, tbe, esz, gate, ns, chunk);
    auto kernel = gate ? stream_kernel<T, 1> : stream_kernel<T, 0>;
    if (chunk) {
        switch (sp.rgn) {
        case 1: kernel = stream_kernel<T, 0, 1>; break;
        case 2: kernel = stream_kernel<T, 0, 2>; break;
        case 4: kernel = stream_kernel<T, 0, 4>; break;
        case 8: kernel = stream_kernel<T, 0, 8>; break;
        case 16: kernel = stream_kernel<T, 0, 16>; break;
        default: return cudaErrorNotSupported;
        }
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kernel<<<(unsigned)sms, sp.wpc * 32 + 32, smem, s>>>(a, ns);
    note_launch();
    return cudaGetLastError();
}

template <bool BWD> cudaError_t launch_token(const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0)
        return cudaSuccess;

    if (a.D < 1 || a.D > 256 || a.E < 1)
        return cudaErrorNotSupported;
    if ((int64_t)a.N * a.H * token_shape(a.D, a.E, 16).tiles > 0x7fffffff)
        return cudaErrorNotSupported;
    const bool shortc = a.max_len <= SHORT_MAX_T;
    if (a.bf16)
        return shortc ? launch_rows<__nv_bfloat16, BWD, true>(a, s)
                      : launch_rows<__nv_bfloat16, BWD, false>(a, s);
    return shortc ? launch_rows<float, BWD, true>(a, s) : launch_rows<float, BWD, false>(a, s);
}

}  // namespace

cudaError_t short_forward_sweep(const SweepArgs &a, cudaStream_t s, bool *streamed)
{
    if (streamed)
        *streamed = false;
    // more than STREAM_MAX_T tokens: one chunk on the tensor cores where it
    // applies
    if (a.max_len > STREAM_MAX_T) {
        const cudaError_t e = decode_chunk_sweep(a, s, streamed);
        if (e != cudaErrorNotSupported)
            return e;
    }
    if (a.N != 0 && a.H != 0 && a.D >= 1 && a.D <= 256 && a.E >= 1) {
        const cudaError_t e = a.bf16 ? try_stream<__nv_bfloat16>(a, s) : try_stream<float>(a, s);
        if (e != cudaErrorNotSupported) {
            if (streamed)
                *streamed = e == cudaSuccess;
            return e;
        }
    }
    return launch_token<false>(a, s);
}

cudaError_t short_backward_sweep(const SweepArgs &a, cudaStream_t s)
{
    return launch_token<true>(a, s);
}

cudaError_t token_read_and_clear_error(cudaStream_t s, int *err)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(err, g_token_error, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_token_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                    s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace la
