// la_gla_prep.cu -- operands of the chunked tensor-core form of the gated
// recurrence (the per-key gate of ejkernel `recurrent`, GLA-style).
//
// With a gate, token t decays state row a by exp(l_t[a]), l_t = g_gamma[h] +
// g_t[a].  Inside a chunk of up to 128 tokens, in processing order, let b_t be
// the running sum of l over the chunk's tokens up to and including t, B the
// sum over the whole chunk, and S the state entering the chunk.  Then
//     o_t  = s [ (q_t exp(b_t)) . S  +  sum_{u <= t} (q_t exp(b_t - b_u) . k_u) v_u ]
//     S'   = diag(exp(B)) S + sum_u (k_u exp(B - b_u))^T v_u
// (products per key channel).  With a reference r (the middle of the range of
// b over the chunk, raised to -LIM if lower), every factor splits into two
// that stay within exp(+-LIM) when all |b_t - r| <= LIM and |r| <= LIM:
//     q~_t = q_t exp(b_t - r),   k~_u = k_u exp(r - b_u),
//     o_t  = s [ q~_t . (diag(exp(r)) S) + sum_{u <= t} (q~_t . k~_u) v_u ]
//     S'   = diag(exp(B - r)) [ diag(exp(r)) S + sum_u k~_u^T v_u ]
// so the tensor-core sweep runs on q~, k~ with a plain causal mask and scales
// state rows by exp(r) and exp(B - r).  This kernel writes q~, k~ (bf16, dense
// [rows][T][H][D]), exp(r) and exp(B - r) per chunk, and flags every
// (sequence, head) with a chunk outside the range; those run the token-by-
// token kernels instead.  Chunks are cut from the start of each sequence, as
// the sweep cuts them, in either direction.
//
// The backward runs its three sweeps on the same operands and yields
// dq~ = dq exp(r - b) and dk~ = dk exp(b - r) in fp32; a second kernel
// recomputes b and r, turns them into dq and dk (token dtype) and forms the
// gate's gradient, for every (sequence, head) not flagged:
//     dg_w = sum over t at or after w (processing order) of q_t dq_t - k_t dk_t
//            + sum_e F dF,
// each term as q~ dq~ - k~ dk~ in fp32 (the bf16 operands and their own
// gradients): gla_undo_kernel walks each sequence's chunks against the
// processing order, carrying the later chunks' sum.

#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int PC = 128;   // tokens per chunk (the tensor-core sweep's chunk)

template <typename T> struct Pair;
template <> struct Pair<float> {
    static __device__ __forceinline__ float2 load(const float *p)
    {
        return *reinterpret_cast<const float2 *>(p);
    }
    static __device__ __forceinline__ void store(float *p, float2 v)
    {
        *reinterpret_cast<float2 *>(p) = v;
    }
};
template <> struct Pair<__nv_bfloat16> {
    static __device__ __forceinline__ float2 load(const __nv_bfloat16 *p)
    {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float2 v)
    {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __float22bfloat162_rn(v);
    }
};

// One CTA per (chunk position, head, sequence); thread (channel pair cp,
// group grp) takes channels 2 cp, 2 cp + 1 over the chunk's processing
// indices PT grp .. PT grp + PT - 1.  Its gates are read once, all in flight
// together, and their running sums stay in registers; the groups' totals are
// combined through shared memory.  The factors exp(b - r), exp(r - b) use the
// fast exponential: they are rounded to bf16 with their operands anyway.
// KSEP: k has strides (or a head divisor) of its own; otherwise k is read at
// q's offsets.
constexpr int PG = 4, PT = PC / PG;   // token groups per chunk, tokens per group
template <typename T, bool KSEP>
__global__ void __launch_bounds__(PG * 64, 2) gla_prep_kernel(GlaPrepArgs a)
{
    const int pc = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int cp = threadIdx.x & 63, grp = threadIdx.x >> 6, c = 2 * cp;
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
    const int64_t t0 = (int64_t)pc * PC;
    if (t0 >= len)
        return;
    const int Lc = (int)(len - t0 < PC ? len - t0 : PC);
    const int p0 = PT * grp;
    const int np = Lc - p0 < 0 ? 0 : (Lc - p0 < PT ? Lc - p0 : PT);   // this group's tokens
    const float gh = a.g_gamma[h];
    // token of processing index p0 + j: tb + j ts
    const int64_t tb = bos + t0 + (np == 0 ? 0 : (a.reverse ? Lc - 1 - p0 : p0));
    const int64_t ts = a.reverse ? -1 : 1;

    // The operands' q, k rows into L2 while the gates are summed: the lane
    // that starts each 128-byte line of a warp's channels asks for it.
    {
        const int esz = (int)sizeof(T);
        if ((c * esz) % 128 == 0) {
            const int64_t qo = row * a.sb + (int64_t)h * a.sh + c;
            const char *qr = reinterpret_cast<const char *>(static_cast<const T *>(a.q) + qo);
            if (KSEP) {
                const char *kr = reinterpret_cast<const char *>(
                    static_cast<const T *>(a.k) + row * a.ksb + (int64_t)(h / a.khd) * a.ksh + c);
                for (int j = 0; j < np; ++j) {
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(qr + (tb + j * ts) * a.st * esz));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + (tb + j * ts) * a.kst * esz));
                }
            } else {
                const char *kr = reinterpret_cast<const char *>(static_cast<const T *>(a.k) + qo);
                for (int j = 0; j < np; ++j) {
                    const int64_t off = (tb + j * ts) * a.st * esz;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(qr + off));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + off));
                }
            }
        }
    }

    // pass 1: this group's gates and their running sums (constant past its end)
    float2 b[PT];
    {
        const float *gp = a.g + row * a.gsb + (int64_t)h * a.gsh + c + tb * a.gst;
        const int64_t gstep = ts * a.gst;
#pragma unroll
        for (int j = 0; j < PT; ++j) {
            b[j] = make_float2(0.f, 0.f);
            if (j < np) {
                const float2 x = *reinterpret_cast<const float2 *>(gp + j * gstep);
                b[j] = make_float2(gh + x.x, gh + x.y);
            }
        }
    }
    float2 lo = make_float2(INFINITY, INFINITY), hi = make_float2(-INFINITY, -INFINITY);
#pragma unroll
    for (int j = 0; j < PT; ++j) {
        if (j > 0) {
            b[j].x += b[j - 1].x;
            b[j].y += b[j - 1].y;
        }
        if (j < np) {
            lo = make_float2(fminf(lo.x, b[j].x), fminf(lo.y, b[j].y));
            hi = make_float2(fmaxf(hi.x, b[j].x), fmaxf(hi.y, b[j].y));
        }
    }
    __shared__ float2 tot[PG][64], los[PG][64], his[PG][64];
    tot[grp][cp] = b[PT - 1];
    __syncthreads();
    float2 off = make_float2(0.f, 0.f), B = off;   // the sums entering this group; the totals
#pragma unroll
    for (int k = 0; k < PG; ++k) {
        const float2 x = tot[k][cp];
        if (k < grp) {
            off.x += x.x;
            off.y += x.y;
        }
        B.x += x.x;
        B.y += x.y;
    }
    los[grp][cp] = make_float2(lo.x + off.x, lo.y + off.y);
    his[grp][cp] = make_float2(hi.x + off.x, hi.y + off.y);
    __syncthreads();
    float2 LO = los[0][cp], HI = his[0][cp];
#pragma unroll
    for (int k = 1; k < PG; ++k) {
        LO = make_float2(fminf(LO.x, los[k][cp].x), fminf(LO.y, los[k][cp].y));
        HI = make_float2(fmaxf(HI.x, his[k][cp].x), fmaxf(HI.y, his[k][cp].y));
    }
    const float2 r = make_float2(fmaxf(0.5f * (LO.x + HI.x), -a.lim),
                                 fmaxf(0.5f * (LO.y + HI.y), -a.lim));
    const bool okx = HI.x - r.x <= a.lim && r.x - LO.x <= a.lim && r.x <= a.lim;
    const bool oky = HI.y - r.y <= a.lim && r.y - LO.y <= a.lim && r.y <= a.lim;
    if (grp == 0) {
        if (!(okx && oky))
            atomicOr(a.flags + (int64_t)n * a.H + h, 1);
        const int64_t vi = (((int64_t)n * a.H + h) * a.ncmax + pc) * a.D + c;
        *reinterpret_cast<float2 *>(a.er + vi) =
            make_float2(okx ? expf(r.x) : 0.f, oky ? expf(r.y) : 0.f);
        *reinterpret_cast<float2 *>(a.u + vi) =
            make_float2(okx ? expf(B.x - r.x) : 0.f, oky ? expf(B.y - r.y) : 0.f);
        if (a.btot)
            *reinterpret_cast<float2 *>(a.btot + vi) = B;
    }

    // pass 2: q~ = q exp(b - r), k~ = k exp(r - b); zeros when out of range
    const T *qp = static_cast<const T *>(a.q) + row * a.sb + (int64_t)h * a.sh + c + tb * a.st;
    const T *kp = KSEP ? static_cast<const T *>(a.k) + row * a.ksb +
                             (int64_t)(h / a.khd) * a.ksh + c + tb * a.kst
                       : static_cast<const T *>(a.k) + row * a.sb + (int64_t)h * a.sh + c +
                             tb * a.st;
    const int64_t dst = (int64_t)a.H * a.D;   // token stride of the dense outputs
    __nv_bfloat162 *xq = reinterpret_cast<__nv_bfloat162 *>(
        static_cast<__nv_bfloat16 *>(a.xq) + ((int64_t)row * a.T * a.H + h) * a.D + c + tb * dst);
    __nv_bfloat162 *yk = reinterpret_cast<__nv_bfloat162 *>(
        static_cast<__nv_bfloat16 *>(a.yk) + ((int64_t)row * a.T * a.H + h) * a.D + c + tb * dst);
    const int64_t istep = ts * a.st, kstep = KSEP ? ts * a.kst : istep, ostep = ts * dst / 2;
    const float2 sh0 = make_float2(off.x - r.x, off.y - r.y);
    // eight tokens' q, k pairs loaded together (indices clamped into the
    // group), then scaled and stored
    constexpr int PB = 8;
#pragma unroll
    for (int j0 = 0; j0 < PT; j0 += PB) {
        float2 qv[PB], kv[PB];
#pragma unroll
        for (int jj = 0; jj < PB; ++jj) {
            const int j = j0 + jj;
            const int jl = j < np ? j : (np > 0 ? np - 1 : 0);
            qv[jj] = Pair<T>::load(qp + jl * istep);
            kv[jj] = Pair<T>::load(kp + jl * kstep);
        }
#pragma unroll
        for (int jj = 0; jj < PB; ++jj) {
            const int j = j0 + jj;
            if (j < np) {
                const float ex = b[j].x + sh0.x, ey = b[j].y + sh0.y;   // b - r
                const float2 x = make_float2(okx ? qv[jj].x * __expf(ex) : 0.f,
                                             oky ? qv[jj].y * __expf(ey) : 0.f);
                const float2 y = make_float2(okx ? kv[jj].x * __expf(-ex) : 0.f,
                                             oky ? kv[jj].y * __expf(-ey) : 0.f);
                xq[j * ostep] = __float22bfloat162_rn(x);
                yk[j * ostep] = __float22bfloat162_rn(y);
            }
        }
    }
}

// dq~, dk~ -> dq, dk and the gate's gradient, one CTA per (group of 16
// channels, head, sequence) walking the sequence's chunks against the
// processing order, so that the sum of the terms of every later chunk (and
// the final state's term) is carried in registers and dg is written once.
// Thread (channel pair cp, token group grp) takes processing indices
// 8 grp .. 8 grp + 7 of each chunk.  b and r are recomputed from the gates
// as the pre-pass formed them (the same definitions; the sums grouped
// differently, so they may differ in the last bits: dq and dk take their
// factor exp(b - r) from them, dg does not).
// DKM: where dk goes -- 0 at q's offsets (k shares q's strides), 1 at k's
// own strides, 2 to a.dk32 in fp32, in place of dk~ (grouped key/value heads).
constexpr int UG = 16, UT = PC / UG, UCP = 8;   // token groups, tokens per group, channel pairs
template <typename T, int DKM>
__global__ void __launch_bounds__(UG * UCP, 4) gla_undo_kernel(GlaPrepArgs a)
{
    const int cg = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int cp = threadIdx.x % UCP, grp = threadIdx.x / UCP;
    const int c = 2 * (UCP * cg + cp);
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
    const int64_t hv = (int64_t)n * a.H + h;
    if (a.flags[hv] || c >= a.D)
        return;   // computed token by token
    const bool rev = a.reverse != 0;
    const float gh = a.g_gamma[h];
    const int nc = (int)((len + PC - 1) / PC);
    __shared__ float2 s_tot[UG][UCP], s_lo[UG][UCP], s_hi[UG][UCP], s_tm[UG][UCP];
    __shared__ float2 s_fdf[UCP];
    // the final state's term, sum_e F[c][e] dF[c][e] (F stored transposed)
    if (grp == 0) {
        float2 f = make_float2(0.f, 0.f);
        if (a.dF) {
            const float *Ft = a.Ft + hv * a.D * a.E, *dF = a.dF + hv * a.D * a.E;
            for (int e = 0; e < a.E; ++e) {
                const float2 fe = *reinterpret_cast<const float2 *>(Ft + (int64_t)e * a.D + c);
                f.x += fe.x * dF[(int64_t)c * a.E + e];
                f.y += fe.y * dF[(int64_t)(c + 1) * a.E + e];
            }
        }
        s_fdf[cp] = f;
    }
    __syncthreads();
    float2 carry = s_fdf[cp];   // the terms after the current chunk, plus F dF
    const int64_t dst = (int64_t)a.H * a.D;   // token stride of the dense tensors
    for (int k = 0; k < nc; ++k) {
        // chunks cut from the sequence's start; visited against the
        // processing order (forward: last chunk first)
        const int pc = rev ? k : nc - 1 - k;
        const int64_t t0 = (int64_t)pc * PC;
        const int Lc = (int)(len - t0 < PC ? len - t0 : PC);
        const int p0 = UT * grp;
        const int np = Lc - p0 < 0 ? 0 : (Lc - p0 < UT ? Lc - p0 : UT);
        // token of processing index p0 + j: tb + j ts
        const int64_t tb = bos + t0 + (np == 0 ? 0 : (rev ? Lc - 1 - p0 : p0));
        const int64_t ts = rev ? -1 : 1;
        const float *gp = a.g + row * a.gsb + (int64_t)h * a.gsh + c + tb * a.gst;
        const int64_t qo = row * a.sb + (int64_t)h * a.sh + c + tb * a.st;
        const int64_t fo = ((int64_t)row * a.T * a.H + h) * a.D + c + tb * dst;
        float2 b[UT], dqv[UT], dkv[UT], qv[UT], kv[UT];
#pragma unroll
        for (int j = 0; j < UT; ++j) {
            const int jl = j < np ? j : (np > 0 ? np - 1 : 0);
            const float2 x = *reinterpret_cast<const float2 *>(gp + jl * ts * a.gst);
            b[j] = j < np ? make_float2(gh + x.x, gh + x.y) : make_float2(0.f, 0.f);
            dqv[j] = *reinterpret_cast<const float2 *>(a.dqf + fo + jl * ts * dst);
            dkv[j] = *reinterpret_cast<const float2 *>(a.dkf + fo + jl * ts * dst);
            qv[j] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(
                static_cast<const __nv_bfloat16 *>(a.xq) + fo + jl * ts * dst));
            kv[j] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(
                static_cast<const __nv_bfloat16 *>(a.yk) + fo + jl * ts * dst));
        }
        // running sums of the log-decays from the chunk's first processed token
        float2 lo = make_float2(INFINITY, INFINITY), hi = make_float2(-INFINITY, -INFINITY);
#pragma unroll
        for (int j = 0; j < UT; ++j) {
            if (j > 0) {
                b[j].x += b[j - 1].x;
                b[j].y += b[j - 1].y;
            }
            if (j < np) {
                lo = make_float2(fminf(lo.x, b[j].x), fminf(lo.y, b[j].y));
                hi = make_float2(fmaxf(hi.x, b[j].x), fmaxf(hi.y, b[j].y));
            }
        }
        s_tot[grp][cp] = b[UT - 1];
        __syncthreads();
        float2 off = make_float2(0.f, 0.f);   // the sums entering this group
#pragma unroll
        for (int q = 0; q < UG; ++q)
            if (q < grp) {
                off.x += s_tot[q][cp].x;
                off.y += s_tot[q][cp].y;
            }
        s_lo[grp][cp] = make_float2(lo.x + off.x, lo.y + off.y);
        s_hi[grp][cp] = make_float2(hi.x + off.x, hi.y + off.y);
        __syncthreads();
        float2 LO = s_lo[0][cp], HI = s_hi[0][cp];
#pragma unroll
        for (int q = 1; q < UG; ++q) {
            LO = make_float2(fminf(LO.x, s_lo[q][cp].x), fminf(LO.y, s_lo[q][cp].y));
            HI = make_float2(fmaxf(HI.x, s_hi[q][cp].x), fmaxf(HI.y, s_hi[q][cp].y));
        }
        const float2 r = make_float2(fmaxf(0.5f * (LO.x + HI.x), -a.lim),
                                     fmaxf(0.5f * (LO.y + HI.y), -a.lim));
        const float2 sh0 = make_float2(off.x - r.x, off.y - r.y);
        // dq, dk, and the terms q~ dq~ - k~ dk~ (the rounded operands and
        // their own gradients) into b[]
        T *dqp = static_cast<T *>(a.dq) + qo;
        T *dkp = DKM == 2   ? nullptr
                 : DKM == 1 ? static_cast<T *>(a.dk) + row * a.ksb + (int64_t)h * a.ksh + c +
                                  tb * a.kst
                            : static_cast<T *>(a.dk) + qo;
        float2 gt = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < UT; ++j) {
            float2 tm = make_float2(0.f, 0.f);
            if (j < np) {
                const float ex = b[j].x + sh0.x, ey = b[j].y + sh0.y;   // b - r
                Pair<T>::store(dqp + j * ts * a.st,
                               make_float2(dqv[j].x * __expf(ex), dqv[j].y * __expf(ey)));
                const float2 dkj = make_float2(dkv[j].x * __expf(-ex), dkv[j].y * __expf(-ey));
                if (DKM == 2)   // this thread read dk~ here above: overwritten in place
                    *reinterpret_cast<float2 *>(a.dk32 + fo + j * ts * dst) = dkj;
                else
                    Pair<T>::store(dkp + j * ts * (DKM == 1 ? a.kst : a.st), dkj);
                tm = make_float2(qv[j].x * dqv[j].x - kv[j].x * dkv[j].x,
                                 qv[j].y * dqv[j].y - kv[j].y * dkv[j].y);
            }
            b[j] = tm;
            gt.x += tm.x;
            gt.y += tm.y;
        }
        __syncthreads();   // every thread is done with s_tot, s_lo, s_hi
        s_tm[grp][cp] = gt;
        __syncthreads();
        // dg = carry + the later groups' totals + this group's terms at or
        // after each token
        float2 acc = carry, tot = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < UG; ++q) {
            const float2 x = s_tm[q][cp];
            if (q > grp) {
                acc.x += x.x;
                acc.y += x.y;
            }
            tot.x += x.x;
            tot.y += x.y;
        }
        float *dgp = a.dg + row * a.gsb + (int64_t)h * a.gsh + c + tb * a.gst;
#pragma unroll
        for (int j = UT - 1; j >= 0; --j) {
            acc.x += b[j].x;
            acc.y += b[j].y;
            if (j < np)
                *reinterpret_cast<float2 *>(dgp + j * ts * a.gst) = acc;
        }
        carry.x += tot.x;
        carry.y += tot.y;
        __syncthreads();   // s_tm read by all before the next chunk writes it
    }
    if (a.segtot && grp == 0)
        *reinterpret_cast<float2 *>(a.segtot + hv * a.D + c) = carry;
}

// One CTA per (segment, head), one thread per key channel: the segment's
// chunk totals summed in chunk order.
__global__ void __launch_bounds__(256) seg_decay_kernel(SegDecayArgs a)
{
    const int seg = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
    if (c >= a.D)
        return;
    const int64_t len = (int64_t)a.seg_cu[seg + 1] - a.seg_cu[seg];
    const int nc = (int)((len + PC - 1) / PC);
    const float *bp = a.btot + ((int64_t)seg * a.H + h) * a.ncmax * a.D + c;
    float acc = 0.f;
    for (int pc = 0; pc < nc && pc < a.ncmax; ++pc)
        acc += bp[(int64_t)pc * a.D];
    a.lam[((int64_t)seg * a.H + h) * a.D + c] = acc;
}

}  // namespace

cudaError_t gla_segment_decay(const SegDecayArgs &a, cudaStream_t s)
{
    if (a.NS == 0 || a.H == 0)
        return cudaSuccess;
    if (a.D > 256 || a.H > 65535)
        return cudaErrorNotSupported;
    seg_decay_kernel<<<dim3((unsigned)a.NS, (unsigned)a.H), (a.D + 31) / 32 * 32, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t gla_prepare(const GlaPrepArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0 || a.ncmax == 0)
        return cudaSuccess;
    if (a.D != 128 || a.N > 65535 || a.H > 65535 || a.ncmax > 0x7fffffff || a.khd < 1)
        return cudaErrorNotSupported;
    dim3 grid((unsigned)a.ncmax, (unsigned)a.H, (unsigned)a.N);
    const int threads = PG * 64;
    const bool ksep = a.khd != 1 || a.ksb != a.sb || a.kst != a.st || a.ksh != a.sh;
    if (a.bf16 && ksep)
        gla_prep_kernel<__nv_bfloat16, true><<<grid, threads, 0, s>>>(a);
    else if (a.bf16)
        gla_prep_kernel<__nv_bfloat16, false><<<grid, threads, 0, s>>>(a);
    else if (ksep)
        gla_prep_kernel<float, true><<<grid, threads, 0, s>>>(a);
    else
        gla_prep_kernel<float, false><<<grid, threads, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t gla_undo(const GlaPrepArgs &a, cudaStream_t s)
{
    if (a.N == 0 || a.H == 0 || a.ncmax == 0)
        return cudaSuccess;
    if (a.D != 128 || a.N > 65535 || a.H > 65535)
        return cudaErrorNotSupported;
    dim3 grid((unsigned)(a.D / (2 * UCP)), (unsigned)a.H, (unsigned)a.N);
    const int dkm = a.dk32 ? 2 : (a.ksb != a.sb || a.kst != a.st || a.ksh != a.sh) ? 1 : 0;
    auto launch = [&](auto kern) { kern<<<grid, UG * UCP, 0, s>>>(a); };
    if (a.bf16)
        dkm == 2   ? launch(gla_undo_kernel<__nv_bfloat16, 2>)
        : dkm == 1 ? launch(gla_undo_kernel<__nv_bfloat16, 1>)
                   : launch(gla_undo_kernel<__nv_bfloat16, 0>);
    else
        dkm == 2   ? launch(gla_undo_kernel<float, 2>)
        : dkm == 1 ? launch(gla_undo_kernel<float, 1>)
                   : launch(gla_undo_kernel<float, 0>);
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
