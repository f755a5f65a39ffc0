// la_tc_sweep.cu -- tensor-core (tcgen05 + TMEM + TMA) sweeps (both shapes) for
// bf16 tokens, key width D = 128, value width E in {64, 128}.
//
// Chunked form of the decayed recurrence (Lightning Attention-2, as named in
// the OpenNLPLab/lightning-attention README; the recurrence itself is the
// ejkernel `recurrent` docstring's "core update"), per (sequence, head), chunk
// of C = 128 tokens with valid length Lc, positions p in processing order:
//     P      = s * (Q K^T) .* M,  M_ij = gamma^(p(i)-p(j)) if p(j) <= p(i), else 0
//     O      = P V  +  diag(s * gamma^(p(i)+1)) (Q S_bf16)
//     S     <- gamma^Lc S + (diag(gamma^(Lc-1-p(j))) K)^T V        (fp32 master)
// Every decay factor is gamma^m with m >= 0, so nothing overflows.
//
// One CTA per (sequence, head); 10 warps:
//   warp 0      TMA producer: Q, K, V chunk boxes (128-byte swizzle) into a
//               2-stage ring
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2..9  epilogue: warp w owns TMEM lanes 32*(w%4).. (rows) and column
//               half (w-2)/4; it turns scores into bf16 P (written back into
//               TMEM as the A operand of P V), scales its K row by the decay
//               in place, combines and stores o, and keeps its 64 columns of
//               the fp32 state S in registers, rewriting the bf16 copy that
//               the next chunk's Q S reads.
// TMEM (512 columns): scores / P [0,128), Q S [128,256), P V [256,384),
// K^T V [384,512).
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises a shared
// abort flag, records LA_ERR_TIMEOUT in a device word, drains its own copies
// and MMAs, frees TMEM and returns.

#include <climits>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

__device__ int g_tc_error;

constexpr int TC_C = 128;        // tokens per chunk (MMA M and the P V K-extent)
constexpr int TC_D = 128;        // key width
constexpr int TC_NST = 2;        // TMA ring stages
constexpr int TC_THREADS = 320;
constexpr int TC_EPI = 256;      // epilogue threads
constexpr uint64_t TC_WAIT_NS = 2000000000ull;
constexpr int TC_ERR_TIMEOUT = 4;
constexpr uint32_t TM_SC = 0, TM_OI = 128, TM_OA = 256, TM_DS = 384, TM_COLS = 512;

template <int E> struct TcLayout {
    static constexpr int QB = TC_C * TC_D * 2;
    static constexpr int KB = TC_C * TC_D * 2;
    static constexpr int VB = TC_C * E * 2;
    static constexpr int STAGE = QB + KB + VB;
    static constexpr int SOFF = TC_NST * STAGE;       // bf16 copy of S, [E/64][D][64]
    static constexpr int SB = TC_D * E * 2;
    static constexpr int MOFF = SOFF + SB;
    static constexpr int NBAR = 2 * TC_NST + 7;
    static constexpr int PWOFF = MOFF + NBAR * 8;
    static constexpr int SLOTOFF = PWOFF + (TC_C + 1) * 4;
    static constexpr int ABORTOFF = SLOTOFF + 4;
    static constexpr int BYTES = ABORTOFF + 4;
    static constexpr int DYN = BYTES + 1024;           // slack for 1024-byte alignment
};

struct TcParams {
    CUtensorMap mq, mk, mv;
    SweepArgs a;
};

// Bounded wait: false when the CTA is aborting or this wait ran out.
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > TC_WAIT_NS) {
            *abort_flag = 1;
            atomicExch(&g_tc_error, TC_ERR_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > TC_WAIT_NS) {
            atomicExch(&g_tc_error, TC_ERR_TIMEOUT);
            return;
        }
}

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ void epi_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(TC_EPI) : "memory");
}

// 16 bytes = 8 bf16 scaled by f, in place.
__device__ __forceinline__ uint4 scale8(uint4 v, float f)
{
    v.x = pack_bf16x2(bf16lo(v.x) * f, bf16hi(v.x) * f);
    v.y = pack_bf16x2(bf16lo(v.y) * f, bf16hi(v.y) * f);
    v.z = pack_bf16x2(bf16lo(v.z) * f, bf16hi(v.z) * f);
    v.w = pack_bf16x2(bf16lo(v.w) * f, bf16hi(v.w) * f);
    return v;
}

// Writes 64 fp32 values as one 128-byte row of a 128B-swizzled bf16 tile.
__device__ __forceinline__ void store_row_sw128(uint8_t *row_base, int row, const float *x)
{
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
        uint4 v;
        v.x = pack_bf16x2(x[8 * c16 + 0], x[8 * c16 + 1]);
        v.y = pack_bf16x2(x[8 * c16 + 2], x[8 * c16 + 3]);
        v.z = pack_bf16x2(x[8 * c16 + 4], x[8 * c16 + 5]);
        v.w = pack_bf16x2(x[8 * c16 + 6], x[8 * c16 + 7]);
        *reinterpret_cast<uint4 *>(row_base + ((c16 ^ (row & 7)) << 4)) = v;
    }
}

template <int E, bool BWD>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_sweep_kernel(const __grid_constant__ TcParams P)
{
    using L = TcLayout<E>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const SweepArgs &a = P.a;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::MOFF);
    uint64_t *full = bars, *empty = bars + TC_NST;
    uint64_t *sc_full = bars + 2 * TC_NST, *p_ready = sc_full + 1, *o_full = sc_full + 2,
             *o_free = sc_full + 3, *ds_full = sc_full + 4, *s_ready = sc_full + 5,
             *drain = sc_full + 6;
    float *pw = reinterpret_cast<float *>(sm + L::PWOFF);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::SLOTOFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::ABORTOFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x / a.H, h = blockIdx.x % a.H;
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
    const int nc = (int)((len + TC_C - 1) / TC_C);

    if (threadIdx.x == 0) {
        for (int i = 0; i < TC_NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(sc_full, 1);
        mbar_init(p_ready, TC_EPI);
        mbar_init(o_full, 1);
        mbar_init(o_free, TC_EPI);
        mbar_init(ds_full, 1);
        mbar_init(s_ready, TC_EPI);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&P.mq);
        prefetch_tmap(&P.mk);
        prefetch_tmap(&P.mv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nc; ++c) {
                const int s = c % TC_NST;
                if (c >= TC_NST && !bwait(&empty[s], ((c / TC_NST) - 1) & 1, abort_flag))
                    break;
                const int cidx = (a.reverse != 0) != BWD ? nc - 1 - c : c;
                const int t0 = (int)(bos + (int64_t)cidx * TC_C);
                uint8_t *st = sm + s * L::STAGE;
                mbar_arrive_expect_tx(&full[s], L::STAGE);
#pragma unroll
                for (int b = 0; b < TC_D / 64; ++b)
                    tma_load_4d(st + b * (TC_C * 128), &P.mq, &full[s], 64 * b, h, t0, (int)row);
#pragma unroll
                for (int b = 0; b < TC_D / 64; ++b)
                    tma_load_4d(st + L::QB + b * (TC_C * 128), &P.mk, &full[s], 64 * b, h, t0,
                                (int)row);
#pragma unroll
                for (int b = 0; b < E / 64; ++b)
                    tma_load_4d(st + L::QB + L::KB + b * (TC_C * 128), &P.mv, &full[s], 64 * b, h,
                                t0, (int)row);
                ++issued;
            }
            // every copy this thread issued has landed before the CTA may exit
            for (int c = issued > TC_NST ? issued - TC_NST : 0; c < issued; ++c)
                drain_wait(&full[c % TC_NST], (c / TC_NST) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_qs = idesc_bf16_f32(128, E, 0, 1);
            const uint32_t id_kv = idesc_bf16_f32(128, E, 1, 1);
            const uint32_t sbase = smem_u32(sm);
            bool any = false;
            for (int c = 0; c < nc; ++c) {
                const int s = c % TC_NST;
                const uint32_t qa = sbase + s * L::STAGE, ka = qa + L::QB, va = ka + L::KB;
                const uint32_t sa = sbase + L::SOFF;
                if (!bwait(&full[s], (c / TC_NST) & 1, abort_flag))
                    break;
                if (c > 0 && !bwait(o_full, (c - 1) & 1, abort_flag))   // P of c-1 consumed
                    break;
                tc_fence_after();
                // scores = Q K^T  (both K-major, K = D)
#pragma unroll
                for (int kk = 0; kk < TC_D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TM_SC, sdesc_sw128(qa + off, 16, 1024),
                           sdesc_sw128(ka + off, 16, 1024), id_qk, kk > 0);
                }
                mma_commit(sc_full);
                any = true;
                if (!bwait(s_ready, c & 1, abort_flag))
                    break;
                if (c > 0 && !bwait(o_free, (c - 1) & 1, abort_flag))
                    break;
                tc_fence_after();
                // Q S_bf16  (S: MN-major, N = E, K = D)
#pragma unroll
                for (int kk = 0; kk < TC_D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TM_OI, sdesc_sw128(qa + off, 16, 1024),
                           sdesc_sw128(sa + kk * 2048, TC_D * 128, 1024), id_qs, kk > 0);
                }
                if (!bwait(p_ready, c & 1, abort_flag))
                    break;
                tc_fence_after();
                // P V  (P from TMEM, V: MN-major, K = C tokens)
#pragma unroll
                for (int kk = 0; kk < TC_C / 16; ++kk)
                    mma_ts(tm + TM_OA, tm + TM_SC + (kk >> 2) * 64 + (kk & 3) * 8,
                           sdesc_sw128(va + kk * 2048, TC_C * 128, 1024), id_qs, kk > 0);
                mma_commit(o_full);
                // (Lambda K)^T V  (both MN-major, M = D, K = C tokens)
#pragma unroll
                for (int kk = 0; kk < TC_C / 16; ++kk)
                    mma_ss(tm + TM_DS, sdesc_sw128(ka + kk * 2048, TC_C * 128, 1024),
                           sdesc_sw128(va + kk * 2048, TC_C * 128, 1024), id_kv, kk > 0);
                mma_commit(ds_full);
                mma_commit(&empty[s]);
            }
            if (any) {   // every MMA has finished before TMEM is released
                mma_commit(drain);
                drain_wait(drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int et = threadIdx.x - 64;
        const int q = warp & 3, hh = (warp - 2) >> 2;
        const int i = 32 * q + lane;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const float g = a.g[h];
        const float scale = a.scale;
        const bool rev = a.reverse != 0;
        const bool flip = rev != BWD;   // mask / chunk order direction
        const bool cols = hh < E / 64;
        for (int m = et; m <= TC_C; m += TC_EPI)
            pw[m] = m == 0 ? 1.f : expf(g * (float)m);
        epi_bar_sync();

        const int64_t sb = ((int64_t)n * a.H + h) * (int64_t)a.D * a.E;
        uint8_t *srow = sm + L::SOFF + hh * (TC_D * 128) + i * 128;
        float S[64];
#pragma unroll
        for (int k = 0; k < 64; ++k)
            S[k] = (cols && a.s_in.p) ? a.s_in.p[sb + i * a.s_in.rs + (64 * hh + k) * a.s_in.cs]
                                      : 0.f;
        if (cols) {
            store_row_sw128(srow, i, S);
            fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(s_ready);

        __nv_bfloat16 *obase = reinterpret_cast<__nv_bfloat16 *>(a.out.p) + row * a.out.sb +
                               (int64_t)h * a.out.sh + 64 * hh;
        bool ok = true;
        for (int c = 0; c < nc && ok; ++c) {
            const int s = c % TC_NST;
            const int cidx = flip ? nc - 1 - c : c;
            const int64_t tc0 = (int64_t)cidx * TC_C;
            const int Lc = (int)(len - tc0 < TC_C ? len - tc0 : TC_C);

            // (a) decay-masked P (bf16, back into TMEM) and Lambda_k K in place
            ok = warp_all(bwait(&full[s], (c / TC_NST) & 1, abort_flag));
            if (ok)
                ok = warp_all(bwait(sc_full, c & 1, abort_flag));
            if (!ok)
                break;
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                uint32_t r[16], pk[8];
                tmem_ld16(tm + lane_off + TM_SC + 64 * hh + 16 * part, r);
#pragma unroll
                for (int jj = 0; jj < 16; jj += 2) {
                    const int j = 64 * hh + 16 * part + jj;
                    const int d0 = flip ? j - i : i - j, d1 = flip ? d0 + 1 : d0 - 1;
                    const bool k0 = d0 >= 0 && (flip ? j : i) < Lc;
                    const bool k1 = d1 >= 0 && (flip ? j + 1 : i) < Lc;
                    const float v0 = k0 ? scale * __uint_as_float(r[jj]) * pw[k0 ? d0 : 0] : 0.f;
                    const float v1 = k1 ? scale * __uint_as_float(r[jj + 1]) * pw[k1 ? d1 : 0] : 0.f;
                    pk[jj / 2] = pack_bf16x2(v0, v1);
                }
                // P for keys [64hh + 16part, +16) -> 8 packed columns inside this
                // thread's own (already read) score columns
                tmem_st8(tm + lane_off + TM_SC + 64 * hh + 8 * part, pk);
            }
            {
                // column factor: gamma^(Lc-1-p(i)) forward, gamma^(p(i)+1) backward
                const float lk = i >= Lc ? 0.f
                                 : BWD ? (rev ? pw[Lc - i] : pw[i + 1])
                                       : (rev ? pw[i] : pw[Lc - 1 - i]);
                uint8_t *krow = sm + s * L::STAGE + L::QB + hh * (TC_C * 128) + i * 128;
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                    uint4 *p = reinterpret_cast<uint4 *>(krow + ((c16 ^ (i & 7)) << 4));
                    *p = scale8(*p, lk);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_ready);

            // (b) o = P V + s gamma^(p(i)+1) Q S
            ok = warp_all(bwait(o_full, c & 1, abort_flag));
            if (!ok)
                break;
            tc_fence_after();
            if (cols) {
                // row factor: s*gamma^(p(i)+1) forward, gamma^(Lc-1-p(i)) backward
                const float lq = i >= Lc ? 0.f
                                 : BWD ? (rev ? pw[i] : pw[Lc - 1 - i])
                                       : scale * (rev ? pw[Lc - i] : pw[i + 1]);
                __nv_bfloat16 *orow = obase + (bos + tc0 + i) * a.out.st;
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t ra[16], ri[16];
                    tmem_ld16(tm + lane_off + TM_OA + 64 * hh + 16 * part, ra);
                    tmem_ld16(tm + lane_off + TM_OI + 64 * hh + 16 * part, ri);
                    if (i < Lc) {
                        uint32_t w[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            w[u] = pack_bf16x2(
                                fmaf(lq, __uint_as_float(ri[2 * u]), __uint_as_float(ra[2 * u])),
                                fmaf(lq, __uint_as_float(ri[2 * u + 1]),
                                     __uint_as_float(ra[2 * u + 1])));
                        *reinterpret_cast<uint4 *>(orow + 16 * part) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(orow + 16 * part + 8) =
                            make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(o_free);

            // (c) S = gamma^Lc S + (Lambda_k K)^T V; refresh the bf16 copy
            ok = warp_all(bwait(ds_full, c & 1, abort_flag));
            if (!ok)
                break;
            tc_fence_after();
            if (cols) {
                const float gl = pw[Lc];
                const float ds_scale = BWD ? scale : 1.f;
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t r[16];
                    tmem_ld16(tm + lane_off + TM_DS + 64 * hh + 16 * part, r);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        S[16 * part + k] = fmaf(gl, S[16 * part + k], ds_scale * __uint_as_float(r[k]));
                }
                store_row_sw128(srow, i, S);
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(s_ready);
        }
        if (ok && cols && a.s_out.p && !*abort_flag) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
                a.s_out.p[sb + i * a.s_out.rs + (64 * hh + k) * a.s_out.cs] = S[k];
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, TM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

bool aligned_tok(const void *p, int64_t sb, int64_t st, int64_t sh)
{
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && sb % 8 == 0 && st % 8 == 0 &&
           sh % 8 == 0;
}

// 4-D map {channel, head, token, batch} with a {64, 1, 128, 1} box, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *p, int X, const SweepArgs &a, int64_t sb, int64_t st,
              int64_t sh)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const int64_t lim = (int64_t)1 << 39;
    // a dimension of extent 1 never moves, any legal stride will do
    if (a.H == 1)
        sh = X;
    if (a.B == 1)
        sb = st * (int64_t)a.T;
    if (sh <= 0 || st <= 0 || sb <= 0 || sh >= lim || st >= lim || sb >= lim)
        return false;
    cuuint64_t dims[4] = {(cuuint64_t)X, (cuuint64_t)a.H, (cuuint64_t)a.T, (cuuint64_t)a.B};
    cuuint64_t strides[3] = {(cuuint64_t)sh * 2, (cuuint64_t)st * 2, (cuuint64_t)sb * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)TC_C, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tile roles: X rows (scores = X Y^T, inter term X S), Y columns (scaled in
// place for the state update), Z values.  Forward: (X, Y, Z) = (q, k, v);
// backward: (k, q, w).
template <int E, bool BWD> cudaError_t launch_tc(const SweepArgs &a, cudaStream_t s)
{
    TcParams p;
    const Tok &x = BWD ? a.k : a.q, &y = BWD ? a.q : a.k;
    if (!make_map(&p.mq, x.p, TC_D, a, x.sb, x.st, x.sh) ||
        !make_map(&p.mk, y.p, TC_D, a, y.sb, y.st, y.sh) ||
        !make_map(&p.mv, a.v.p, E, a, a.v.sb, a.v.st, a.v.sh))
        return cudaErrorNotSupported;
    p.a = a;
    auto kern = tc_sweep_kernel<E, BWD>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           TcLayout<E>::DYN);
    if (err != cudaSuccess)
        return err;
    kern<<<(unsigned)((int64_t)a.N * a.H), TC_THREADS, TcLayout<E>::DYN, s>>>(p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool tc_sweep_supported(const SweepArgs &a)
{
    if (!a.bf16 || a.D != TC_D || (a.E != 64 && a.E != 128) || a.T < 1 || a.B < 1)
        return false;
    if ((int64_t)a.N * a.H > INT_MAX)
        return false;
    return aligned_tok(a.q.p, a.q.sb, a.q.st, a.q.sh) &&
           aligned_tok(a.k.p, a.k.sb, a.k.st, a.k.sh) &&
           aligned_tok(a.v.p, a.v.sb, a.v.st, a.v.sh) &&
           aligned_tok(a.out.p, a.out.sb, a.out.st, a.out.sh);
}

cudaError_t tc_forward_sweep(const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0)
        return cudaSuccess;
    return a.E == 128 ? launch_tc<128, false>(a, s) : launch_tc<64, false>(a, s);
}

cudaError_t tc_backward_sweep(const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0)
        return cudaSuccess;
    return a.E == 128 ? launch_tc<128, true>(a, s) : launch_tc<64, true>(a, s);
}

cudaError_t tc_read_and_clear_error(cudaStream_t s, int *err)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(err, g_tc_error, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace la
