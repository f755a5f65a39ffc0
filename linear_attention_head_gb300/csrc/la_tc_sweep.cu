// la_tc_sweep.cu -- tensor-core (tcgen05 + TMEM + TMA) sweeps (both shapes) for
// bf16 tokens, key width D = 128, value width E in {64, 128}.
//
// Chunked form of the decayed recurrence (Lightning Attention-2, as named in
// the OpenNLPLab/lightning-attention README; the recurrence itself is the
// ejkernel `recurrent` docstring's "core update").  Per (sequence, head) and
// chunk of C = 128 tokens with valid length Lc and positions p(.) in
// processing order, with three 128-token tiles X, Y, Z:
//     P   = s * (X Y^T) .* M           M_rc = gamma^|p(r)-p(c)| on one side
//     O   = P Z + diag(lrow) (X S_bf16)
//     S  <- gamma^Lc S + (diag(lcol) Y)^T Z                  (fp32, in TMEM)
//   forward  (X, Y, Z) = (q, k, v):   keep p(c) <= p(r), lrow = s*gamma^(p(r)+1),
//                                     lcol = gamma^(Lc-1-p(c))
//   backward (X, Y, Z) = (k, q, do):  keep p(c) >= p(r), lrow = gamma^(Lc-1-p(r)),
//                                     lcol = s*gamma^(p(c)+1), chunks in
//                                     reverse processing order (dv; dk swaps
//                                     the tensors' roles on the host)
// Every decay factor is gamma^m with m >= 0, so nothing overflows.
//
// One CTA per (sequence, head); 18 warps:
//   warp 0        TMA producer: X, Y, Z boxes (128-byte swizzle), 2-stage ring
//   warp 1        TMEM allocator; one thread issues every tcgen05.mma
//   warps 2..9    P group: warp w owns TMEM lanes 32*(w%4).. and key half
//                 (w-2)/4 of the scores; writes bf16 P back into TMEM (the A
//                 operand of P Z) and scales its Y row in place by lcol
//   warps 10..13  S group: one thread per state row; turns the state around
//                 each chunk: S -> bf16 copy (B operand of the next X S) and
//                 S * gamma^Lc(next) back into TMEM, where the next update
//                 accumulates
//   warps 14..17  O group: one thread per token row; o = P Z + lrow * X S,
//                 written as bf16 into the Z tile of the finished stage and
//                 sent out with TMA stores, one per warp and 64-column block
//                 (the last chunk of a packed sequence, whose tile would
//                 overrun into the next sequence, is stored row by row)
// TMEM (512 columns): scores/P [0,128), X S [128,256), P Z [256,384),
// S [384,512) (value columns: E of them).  MMA order per chunk: scores and
// X S as soon as the tiles land; then, once P is written, the state update
// and P Z.  A ring stage is held only from landing to that last MMA, which is
// what bounds the memory pipeline with two 96 KB stages.  The X and Y slots of
// a stage are released by the state update (the last MMA reading them), the
// Z slot once the output tile staged in it has been stored; the next chunk's
// scores need only X and Y.
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises a shared
// abort flag and records LA_ERR_TIMEOUT in a device word, drains its own
// copies and MMAs, frees TMEM and returns.

#include <climits>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

namespace la {
namespace {

constexpr int TC_THREADS = 576;  // 18 warps
constexpr int TC_PG = 256;       // P group threads (warps 2..9)
constexpr int TC_SG = 128;       // S group threads (warps 10..13)
constexpr int TC_OG = 128;       // O group threads (warps 14..17)
constexpr uint32_t TM_SC = 0, TM_COLS = 512;

// Shared memory and TMEM of one CTA with key width D and a tile of E value
// columns.  Tiles are [channel block of 64][C rows][128 bytes], 128-byte
// swizzled.  The Y slot is padded to a multiple of 128 channels with zero
// blocks (written once, never loaded), so the state update is always M = 128
// MMAs: state rows past D only ever receive zeros and are never read.  The
// state occupies NP = YPAD / 128 TMEM pieces of E columns.
template <int D, int E> struct TcLayout {
    static constexpr int YPAD = (D + 127) / 128 * 128;
    static constexpr int NP = YPAD / 128;              // 128-row state pieces
    static constexpr int NST = D <= 128 ? 2 : 1;       // TMA ring stages
    static constexpr int XB = TC_C * D * 2;
    static constexpr int YB = TC_C * YPAD * 2;
    static constexpr int YLB = TC_C * D * 2;           // bytes of Y loaded per chunk
    static constexpr int ZB = TC_C * E * 2;
    static constexpr int STAGE = XB + YB + ZB;
    static constexpr int SOFF = NST * STAGE;           // bf16 copy of S, [E/64][D][64]
    static constexpr int SB = D * E * 2;
    static constexpr int MOFF = SOFF + SB;
    static constexpr int NBAR = 4 * NST + 12;
    // TMEM columns: scores [0,128), X S, P Z, then the state pieces
    static constexpr uint32_t TM_OI = 128, TM_OA = 128 + E, TM_S = 128 + 2 * E;
    static_assert(TM_S + NP * E <= TM_COLS, "TMEM columns");
    static constexpr int PWOFF = MOFF + NBAR * 8;
    static constexpr int CFOFF = (PWOFF + (TC_C + 1) * 4 + 15) / 16 * 16;   // 32 column factors
    static constexpr int DTOFF = CFOFF + 32 * 4;                            // 64 diagonal factors
    static constexpr int COLNOFF = DTOFF + 64 * 4;                        // 128 column factors (gated)
    static constexpr int SLOTOFF = COLNOFF + 128 * 4;
    static constexpr int ABORTOFF = SLOTOFF + 4;
    static constexpr int BYTES = ABORTOFF + 4;
    static constexpr int DYN = BYTES + 1024;           // slack for 1024-byte alignment
    static_assert(DYN <= 232448, "shared memory per CTA");
};

struct TcParams {
    CUtensorMap mx, my, mz, mo;
    int dx, dy, dz;   // head divisors of the X, Y, Z tensors (grouped key/value heads)
    SweepArgs a;
};

__device__ __forceinline__ void epi_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(TC_PG + TC_SG + TC_OG) : "memory");
}

// The gated form's P block: the decay is inside the operands, so P is the
// scaled scores under the causal mask alone.  Masked scores may be infinite
// (the operands' factors are only bounded on the causal side), so they are
// replaced, never multiplied.  kind: 0 masked block, 1 visible, 2 diagonal.
__device__ __forceinline__ void p_block_gated(uint32_t (&r)[32], int kind, float scale, bool flip,
                                              int lane)
{
    if (kind == 0) {
#pragma unroll
        for (int m = 0; m < 16; ++m)
            r[2 * m] = 0u;
    } else {
        const float2 ss = make_float2(scale, scale);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            float2 v = mul_f32x2(
                make_float2(__uint_as_float(r[2 * m]), __uint_as_float(r[2 * m + 1])), ss);
            if (kind == 2) {
                const int j0 = 2 * m, j1 = 2 * m + 1;
                if (flip ? j0 < lane : j0 > lane)
                    v.x = 0.f;
                if (flip ? j1 < lane : j1 > lane)
                    v.y = 0.f;
            }
            r[2 * m] = pack_bf16x2(v.x, v.y);
        }
    }
}

// One 128-byte row of a tile set to zero.
__device__ __forceinline__ void zero_row(uint8_t *row_base)
{
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4 *>(row_base + (c16 << 4)) = make_uint4(0u, 0u, 0u, 0u);
}

// GLA (gated form, on operands rescaled by la_gla_prep.cu): plain causal P,
// no decay factor on Y (backward-type: Y times s), the inter term scaled by
// s (forward-type) or 1; the state scaled after each chunk's update by the
// chunk's factor and the next chunk's -- exp(B - r) then exp(r) going
// forward, exp(r) then exp(B - r) going backward -- on its rows (GLA 1: the
// gated key channels are the state's rows) or columns (GLA 2).  GLA 2 gives
// dq~ or dk~, which the gate's gradient needs unrounded: its output is fp32.
// SO (state only): the sweep's final states alone (the sequence split's first
// pass): Y and Z are loaded, the state update runs, X, the scores, P Z, the
// inter term and the output are skipped.
// D: key width (X and Y channels); E: the value columns of one CTA, a tile of
// the a.E columns (a.E / E CTAs per (sequence, head), adjacent in the grid so
// that their X and Y reads meet in L2).
template <int D, int E, bool BWD, int GLA, bool SO = false>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_sweep_kernel(const __grid_constant__ TcParams P)
{
    static_assert(D % 64 == 0 && D <= 256 && (E == 64 || E == 128), "tile shape");
    // the gated form has 128 key channels: the state's rows (GLA 1) or its
    // columns (GLA 2, whose rows are the 64 or 128 value channels)
    static_assert(GLA == 0 || (GLA == 1 ? D == 128 : E == 128), "gated key channels");
    using L = TcLayout<D, E>;
    constexpr int NST = L::NST;
    constexpr uint32_t TM_OI = L::TM_OI, TM_OA = L::TM_OA, TM_S = L::TM_S;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const SweepArgs &a = P.a;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::MOFF);
    // full: the stage's X and Y tiles landed; zfull: its Z tile landed;
    // empty: its X and Y slots are free (the state update, the chunk's last
    // MMA reading them, is done); zfree: its Z slot is free (every O warp has
    // stored its rows of the output tile, staged there, out of it)
    uint64_t *full = bars, *empty = bars + NST, *zfull = bars + 2 * NST,
             *zfree = bars + 3 * NST;
    uint64_t *sc_full = bars + 4 * NST;      // scores of the chunk are in TMEM
    uint64_t *pv_done = sc_full + 1;         // P consumed (scores columns free)
    uint64_t *p_ready = sc_full + 2;         // P written, Y scaled
    uint64_t *s_ready = sc_full + 3;         // bf16 S written, TMEM S pre-scaled
    uint64_t *o_free = sc_full + 4;          // both O accumulators read
    uint64_t *ds_full = sc_full + 5;         // state update (and X S) done
    uint64_t *o_full = sc_full + 6;          // P Z (and X S) done
    uint64_t *drain = sc_full + 7;
    float *pw = reinterpret_cast<float *>(sm + L::PWOFF);
    float *cf = reinterpret_cast<float *>(sm + L::CFOFF);
    float *dt = reinterpret_cast<float *>(sm + L::DTOFF);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::SLOTOFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::ABORTOFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&zfull[i], 1);
            mbar_init(&zfree[i], TC_OG / 32);
        }
        mbar_init(sc_full, 1);
        mbar_init(pv_done, 1);
        mbar_init(p_ready, TC_PG);
        mbar_init(s_ready, TC_SG);
        mbar_init(o_free, TC_OG);
        mbar_init(ds_full, 1);
        mbar_init(o_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&P.mx);
        prefetch_tmap(&P.my);
        prefetch_tmap(&P.mz);
        prefetch_tmap(&P.mo);
    }
    if (L::YPAD > D) {
        // zero blocks padding each stage's Y slot to whole 128-channel pieces
        // (never loaded; the MMAs read them through the async proxy)
        constexpr int PADB = (L::YPAD - D) * TC_C * 2;
        for (int st = 0; st < NST; ++st)
            for (int o = 16 * threadIdx.x; o < PADB; o += 16 * TC_THREADS)
                if (LA_OK_AT(L::YLB + o + 16 <= L::YB, 1))
                    *reinterpret_cast<uint4 *>(sm + st * L::STAGE + L::XB + L::YLB + o) =
                        make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    // The set-up above touches only this CTA's shared memory, its TMEM and the
    // kernel parameters, so it overlaps the end of the stream's previous
    // kernel; global memory is read and written only after that kernel is done.
    grid_dep_wait();
    grid_dep_launch_dependents();

    // work item: the rank-th sequence of the schedule (longest first when an
    // order is given), one head and one tile of E value columns per CTA
    const int net = a.E / E;
    const int et = (int)(blockIdx.x % (unsigned)net);
    const int pair = (int)(blockIdx.x / (unsigned)net);
    const int rank = pair / a.H, h = pair % a.H;
    const int e0 = et * E;   // first value column of this CTA
    const int n = a.order ? a.order[rank] : rank;
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
    // gated form: (sequence, head) pairs whose gates are out of range run
    // token by token instead
    if (GLA && a.gla_flags && a.gla_flags[(int64_t)n * a.H + h] != a.gla_flag_run) {
        if (warp == 1)
            tmem_dealloc(tm, TM_COLS);
        return;
    }
    const int nc = (int)((len + TC_C - 1) / TC_C);
    const bool rev = a.reverse != 0;
    const bool flip = rev != BWD;   // chunk order and mask direction
    // first token and valid length of the chunk processed c-th
    auto chunk_t0 = [&](int c) { return (int64_t)(flip ? nc - 1 - c : c) * TC_C; };
    auto chunk_len = [&](int c) {
        const int64_t t0 = chunk_t0(c);
        return (int)(len - t0 < TC_C ? len - t0 : TC_C);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // head coordinate of each tile (key/value heads may be shared)
            const int hx = h / P.dx, hy = h / P.dy, hz = h / P.dz;
            int issued = 0;
            for (int c = 0; c < nc; ++c) {
                const int s = c % NST;
                const uint32_t ph = ((c / NST) - 1) & 1;
                if (c >= NST && !bwait(&empty[s], ph, abort_flag))
                    break;
                const int t0 = (int)(bos + chunk_t0(c));
                uint8_t *st = sm + s * L::STAGE;
                if (!LA_OK_AT(t0 >= 0 && t0 < a.T && e0 + E <= a.E, 21))
                    break;
                if (SO) {
                    // Y and Z, both free once the chunk's state update is done
                    mbar_arrive_expect_tx(&full[s], L::YLB + L::ZB);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_4d(st + L::XB + b * (TC_C * 128), &P.my, &full[s], 64 * b, hy, t0,
                                    (int)row);
#pragma unroll
                    for (int b = 0; b < E / 64; ++b)
                        tma_load_4d(st + L::XB + L::YB + b * (TC_C * 128), &P.mz, &full[s],
                                    64 * b + e0, hz, t0, (int)row);
                    ++issued;
                    continue;
                }
                // X and Y first: their slots are free once the chunk's state
                // update is done and the next scores need them; the Z slot
                // only once the output tile staged in it has left
                mbar_arrive_expect_tx(&full[s], L::XB + L::YLB);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_4d(st + b * (TC_C * 128), &P.mx, &full[s], 64 * b, hx, t0, (int)row);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_4d(st + L::XB + b * (TC_C * 128), &P.my, &full[s], 64 * b, hy, t0,
                                (int)row);
                // Z is copied even when this wait gives up, so that the drain
                // below sees the stage complete
                const bool zok = c < NST || bwait(&zfree[s], ph, abort_flag);
                mbar_arrive_expect_tx(&zfull[s], L::ZB);
#pragma unroll
                for (int b = 0; b < E / 64; ++b)
                    tma_load_4d(st + L::XB + L::YB + b * (TC_C * 128), &P.mz, &zfull[s],
                                64 * b + e0, hz, t0, (int)row);
                ++issued;
                if (!zok)
                    break;
            }
            // every copy this thread issued has landed before the CTA may exit
            for (int c = issued > NST ? issued - NST : 0; c < issued; ++c) {
                drain_wait(&full[c % NST], (c / NST) & 1);
                if (!SO)
                    drain_wait(&zfull[c % NST], (c / NST) & 1);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_xy = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_xz = idesc_bf16_f32(128, E, 0, 1);
            const uint32_t id_yz = idesc_bf16_f32(128, E, 1, 1);
            const uint32_t sbase = smem_u32(sm);
            const uint32_t sa = sbase + L::SOFF;
            bool any = false;
            // S (piece pc: state rows 128 pc ..) += (lcol Y)^T Z  (both MN-major,
            // M = 128 channels of Y, K = C tokens): the recurrence
            auto state_update = [&](uint32_t ya, uint32_t za) {
#pragma unroll
                for (int pc = 0; pc < L::NP; ++pc)
#pragma unroll
                    for (int kk = 0; kk < TC_C / 16; ++kk)
                        mma_ss(tm + TM_S + pc * E,
                               sdesc_sw128(ya + pc * 2 * (TC_C * 128) + kk * 2048, TC_C * 128,
                                           1024),
                               sdesc_sw128(za + kk * 2048, TC_C * 128, 1024), id_yz, 1);
            };
            for (int c = 0; c < nc; ++c) {
                const int s = c % NST;
                const uint32_t xa = sbase + s * L::STAGE, ya = xa + L::XB, za = ya + L::YB;
                if (!LA_OK_AT(za + L::ZB <= sbase + (uint32_t)L::SOFF &&
                                  sa + (uint32_t)L::SB <= sbase + (uint32_t)L::MOFF,
                              12))
                    break;
                if (!bwait(&full[s], (c / NST) & 1, abort_flag))
                    break;
                if (SO) {
                    // the state update alone, once the state is pre-scaled
                    // and Y scaled
                    if (!bwait(s_ready, c & 1, abort_flag) || !bwait(p_ready, c & 1, abort_flag))
                        break;
                    tc_fence_after();
                    state_update(ya, za);
                    mma_commit(ds_full);
                    mma_commit(&empty[s]);
                    any = true;
                    continue;
                }
                if (c > 0 && !bwait(pv_done, (c - 1) & 1, abort_flag))
                    break;
                tc_fence_after();
                // scores = X Y^T  (both K-major, K = D)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TM_SC, sdesc_sw128(xa + off, 16, 1024),
                           sdesc_sw128(ya + off, 16, 1024), id_xy, kk > 0);
                }
                mma_commit(sc_full);
                any = true;
                // X S_bf16  (S: MN-major, N = E, K = D): needs this chunk's state
                // copy and the previous chunk's O read
                if (!bwait(s_ready, c & 1, abort_flag))
                    break;
                if (c > 0 && !bwait(o_free, (c - 1) & 1, abort_flag))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TM_OI, sdesc_sw128(xa + off, 16, 1024),
                           sdesc_sw128(sa + kk * 2048, D * 128, 1024), id_xz, kk > 0);
                }
                if (!bwait(p_ready, c & 1, abort_flag))
                    break;
                if (!bwait(&zfull[s], (c / NST) & 1, abort_flag))
                    break;
                tc_fence_after();
                state_update(ya, za);
                mma_commit(ds_full);
                mma_commit(&empty[s]);   // X and Y have been read for the last time
                // P Z  (P from TMEM, Z: MN-major, K = C tokens)
#pragma unroll
                for (int kk = 0; kk < TC_C / 16; ++kk)
                    mma_ts(tm + TM_OA, tm + TM_SC + (kk >> 2) * 64 + (kk & 3) * 8,
                           sdesc_sw128(za + kk * 2048, TC_C * 128, 1024), id_xz, kk > 0);
                mma_commit(o_full);
                mma_commit(pv_done);
            }
            if (any) {   // every MMA has finished before TMEM is released
                mma_commit(drain);
                drain_wait(drain, 0);
            }
        }
        __syncwarp();
    } else {
        const int et = threadIdx.x - 64;
        const float g = a.g[h];
        const float scale = a.scale;
        for (int m = et; m <= TC_C; m += TC_PG + TC_SG + TC_OG)
            pw[m] = m == 0 ? 1.f : expf(g * (float)m);
        if (et < 32) {   // column factors of the off-diagonal blocks
            const int m = flip ? et : 31 - et;
            cf[et] = m == 0 ? 1.f : expf(g * (float)m);
        } else if (et < 96) {   // diagonal blocks, index jj - lane + 31
            const int u = et - 32;
            const int m = flip ? u - 31 : 31 - u;
            dt[u] = m < 0 || u > 62 ? 0.f : (m == 0 ? scale : scale * expf(g * (float)m));
        }
        epi_bar_sync();
        const int q = warp & 3;
        const int i = 32 * q + lane;   // TMEM lane = tile row
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;

        if (warp < 10) {
            // ------------------------------------------------------- P group
            const int hh = (warp - 2) >> 2;
            const int j0 = 64 * hh;
            // row i of every loaded 64-channel block of Y scaled in place
            // (the two halves of the group take alternate blocks)
            auto scale_y = [&](int s, float f) {
#pragma unroll
                for (int b = hh; b < D / 64; b += 2)
                    if (LA_OK_AT(b * (TC_C * 128) + i * 128 + 128 <= L::YLB && s < NST, 7))
                        scale_row_sw128(sm + s * L::STAGE + L::XB + b * (TC_C * 128) + i * 128, i,
                                        f);
            };
            for (int c = 0; c < nc; ++c) {
                const int s = c % NST;
                const int Lc = chunk_len(c);
                if (!LA_OK_AT(Lc >= 1 && Lc <= TC_C, 5))
                    break;
                bool ok = warp_all(bwait(&full[s], (c / NST) & 1, abort_flag));
                if (ok && !SO)
                    ok = warp_all(bwait(sc_full, c & 1, abort_flag));
                // state only: no scores hold this group in step with the MMA
                // issuer, so it waits for the previous state update, else it
                // could complete p_ready twice before the issuer's wait on it
                // and the parity of that wait would read the wrong phase
                if (ok && SO && c > 0)
                    ok = warp_all(bwait(ds_full, (c - 1) & 1, abort_flag));
                if (!ok)
                    break;
                tc_fence_after();
                if (SO) {
                    if (GLA) {
                        // Y carries its factors (backward-type: times s);
                        // rows past the sequence's end cleared, as below
                        uint8_t *yrow = sm + s * L::STAGE + L::XB + hh * (TC_C * 128) + i * 128;
                        if (i >= Lc)
                            zero_row(yrow);
                        else if (BWD)
                            scale_row_sw128(yrow, i, scale);
                    } else {
                        // column factor for the state update, applied to row i of Y
                        float lc = 0.f;
                        if (i < Lc) {
                            const int pi = rev ? Lc - 1 - i : i;
                            lc = BWD ? scale * pw[pi + 1] : pw[Lc - 1 - pi];
                        }
                        scale_y(s, lc);
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(p_ready);
                    continue;
                }
                uint32_t ra[32], rb[32];
                const uint32_t col = tm + lane_off + TM_SC + j0;
                // block kinds are warp-uniform: 0 zero, 1 rank one, 2 diagonal
                const int b0 = 2 * hh, b1 = b0 + 1;
                const int k0 = b0 == q ? 2 : ((flip ? b0 > q : b0 < q) ? 1 : 0);
                const int k1 = b1 == q ? 2 : ((flip ? b1 > q : b1 < q) ? 1 : 0);
                tmem_ld32_issue(col, ra);
                tmem_ld32_issue(col + 32, rb);
                tmem_wait_ld(ra, rb);
                if (GLA) {
                    p_block_gated(ra, k0, scale, flip, lane);
                    p_block_gated(rb, k1, scale, flip, lane);
                } else {
                    const int ix0 = flip ? 32 * (b0 - q) - lane : 32 * (q - b0) + lane - 31;
                    const int ix1 = flip ? 32 * (b1 - q) - lane : 32 * (q - b1) + lane - 31;
                    const float rf0 =
                        k0 == 1 && LA_OK_AT(ix0 >= 0 && ix0 <= TC_C, 3) ? scale * pw[ix0] : 0.f;
                    const float rf1 =
                        k1 == 1 && LA_OK_AT(ix1 >= 0 && ix1 <= TC_C, 3) ? scale * pw[ix1] : 0.f;
                    p_block_full(ra, k0, rf0, cf, dt, lane);
                    p_block_full(rb, k1, rf1, cf, dt, lane);
                }
                if (Lc < TC_C) {
                    // the sequence ends inside this chunk: rows past the end
                    // (forward order) or keys past it (reverse order) are zero
                    if (!flip) {
                        if (i >= Lc) {
#pragma unroll
                            for (int m = 0; m < 16; ++m)
                                ra[2 * m] = rb[2 * m] = 0u;
                        }
                    } else {
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const int ja = j0 + 2 * m, jb = j0 + 32 + 2 * m;
                            ra[2 * m] &= (ja < Lc ? 0xffffu : 0u) | (ja + 1 < Lc ? 0xffff0000u : 0u);
                            rb[2 * m] &= (jb < Lc ? 0xffffu : 0u) | (jb + 1 < Lc ? 0xffff0000u : 0u);
                        }
                    }
                }
                // P for the keys of this half: 32 packed columns inside the
                // thread's own (already read) score columns
                tmem_st16_even_issue(col, ra);
                tmem_st16_even_issue(col + 16, rb);
                tmem_wait_st();
                if (GLA) {
                    // Y carries its factors already (backward-type: times s);
                    // rows past the sequence's end (the next packed
                    // sequence's, or zero fill) are cleared
                    uint8_t *yrow = sm + s * L::STAGE + L::XB + hh * (TC_C * 128) + i * 128;
                    if (i >= Lc)
                        zero_row(yrow);
                    else if (BWD)
                        scale_row_sw128(yrow, i, scale);
                } else {
                    // column factor for the state update, applied to row i of Y
                    float lc = 0.f;
                    if (i < Lc) {
                        const int pi = rev ? Lc - 1 - i : i;
                        lc = BWD ? scale * pw[pi + 1] : pw[Lc - 1 - pi];
                    }
                    scale_y(s, lc);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                if (!(a.withhold_handoff && c == 0))   // diagnostic: let the MMA wait run out
                    mbar_arrive(p_ready);
            }
        } else if (warp < 14) {
            // ------------------------------------------------------- S group
            const int64_t sb = ((int64_t)n * a.H + h) * (int64_t)a.D * a.E;
            // thread i holds row r = 128 pc + i of state piece pc (TMEM lane i,
            // columns TM_S + pc E ..) for every r < D; rows past D are padding
            // that only ever receives zeros and is never read.  Whether a row
            // exists is warp-uniform (D is a multiple of 64).
            auto srow = [&](int pc) { return 128 * pc + i; };
            auto sbf = [&](int pc) { return sm + L::SOFF + srow(pc) * 128; };
            auto stm = [&](int pc) { return tm + lane_off + TM_S + pc * E; };
            // initial state: bf16 copy and gamma^L0-scaled fp32 in TMEM (an
            // empty sequence passes it straight to the final state)
            // gated form: factors of chunk position pc for key channel i (the
            // state's row i, or column i), [N][H][ncmax][128]; vo the chunk's
            // own factor, vn the next chunk's (also the initial state's)
            const int64_t vrow = ((int64_t)n * a.H + h) * a.gla_ncmax;
            auto vidx = [&](int cpos) { return (vrow + cpos) * 128 + i; };
            const float *vo = BWD ? a.gla_er : a.gla_u, *vn = BWD ? a.gla_u : a.gla_er;
            // GLA 2: this step's per-column factors, shared by the S group:
            // the chunk's own (colf) and the next chunk's (coln)
            float *colf = pw;
            float *coln = reinterpret_cast<float *>(sm + L::COLNOFF);
            auto sg_sync = [] { asm volatile("bar.sync 2, %0;" ::"n"(TC_SG) : "memory"); };
            // the state tensors' extent (element offsets of both corners of
            // this CTA's rows and columns must fall inside it)
            const int64_t s_total = (int64_t)a.N * a.H * a.D * a.E;
            auto s_ok = [&](int64_t rs, int64_t cs, int r) {
                const int64_t lo = sb + r * rs + (int64_t)e0 * cs;
                const int64_t hi = lo + (int64_t)(E - 1) * cs;
                return lo >= 0 && hi < s_total;
            };
            const bool in_ok = !a.s_in.p || LA_OK_AT(s_ok(a.s_in.rs, a.s_in.cs, D - 1), 15);
            const bool out_ok = !a.s_out.p || LA_OK_AT(s_ok(a.s_out.rs, a.s_out.cs, D - 1), 16);
            if (!LA_OK_AT((L::NP - 1) * 128 + 127 < L::YPAD &&
                              (D - 1) * 128 + (E / 64 - 1) * (D * 128) + 128 <= L::SB,
                          9) ||
                !in_ok || !out_ok) {
                // nothing below is safe: leave the state alone (the MMA
                // issuer's s_ready wait runs out and the kernel stops)
            } else if (nc == 0) {
#pragma unroll 1
                for (int pc = 0; pc < L::NP; ++pc)
                    if (srow(pc) < D)
                        state_copy(a.s_in, a.s_out, sb, srow(pc), e0, E);
            } else if (GLA == 1) {
                const float f0 = vn[vidx(flip ? nc - 1 : 0)];
                state_in(a.s_in, sb, i, e0, E, sbf(0), D * 128, stm(0), f0, f0);
            } else if (GLA == 2) {
                if (i < E)
                    colf[i] = vn[vidx(flip ? nc - 1 : 0)];
                sg_sync();
                if (i < D)   // rows past D (64 value channels) are padding
                    state_in(a.s_in, sb, i, e0, E, sbf(0), D * 128, stm(0), 1.f, 1.f, colf);
            } else {
#pragma unroll 1
                for (int pc = 0; pc < L::NP; ++pc)
                    if (srow(pc) < D)
                        state_in(a.s_in, sb, srow(pc), e0, E, sbf(pc), D * 128, stm(pc),
                                 pw[chunk_len(0)], 1.f);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(s_ready);
            for (int c = 0; c < nc; ++c) {
                const bool last = c + 1 == nc;
                // out = fo x (last chunk); else the copy and TMEM get ft x
                // (gated form) or x and gn x
                // gated form: the chunk's factor fo, then the next chunk's fn,
                // applied one after the other (their product can underflow
                // where each step stays in range)
                float fo = 1.f, fn = 1.f, ft = last ? 1.f : pw[chunk_len(c + 1)];
                if (GLA) {
                    fo = GLA == 1 || i < E ? vo[vidx(flip ? nc - 1 - c : c)] : 1.f;
                    if (!last)
                        fn = GLA == 1 || i < E ? vn[vidx(flip ? nc - 2 - c : c + 1)] : 1.f;
                }
                if (GLA == 2) {
                    // one decision for the whole S group: its barriers below
                    // must not be left by some warps only
                    uint32_t all;
                    asm volatile("{\n\t.reg .pred p, q;\n\t"
                                 "setp.ne.u32 q, %1, 0;\n\t"
                                 "bar.red.and.pred p, 3, %2, q;\n\t"
                                 "selp.u32 %0, 1, 0, p;\n\t}"
                                 : "=r"(all)
                                 : "r"(bwait(ds_full, c & 1, abort_flag) ? 1u : 0u), "n"(TC_SG)
                                 : "memory");
                    if (!all)
                        break;
                    if (i < E) {
                        colf[i] = fo;
                        coln[i] = fn;
                    }
                    sg_sync();
                } else if (!warp_all(bwait(ds_full, c & 1, abort_flag))) {
                    break;
                }
                tc_fence_after();
                const float gn = ft;
#pragma unroll 1
                for (int pc = 0; pc < L::NP; ++pc) {
                    if (srow(pc) >= D)
                        continue;
                    const int r = srow(pc);
#pragma unroll 1
                    for (int eb = 0; eb < E / 64; ++eb) {
                        uint32_t ra[32], rb[32];
                        tmem_ld32_issue(stm(pc) + 64 * eb, ra);
                        tmem_ld32_issue(stm(pc) + 64 * eb + 32, rb);
                        tmem_wait_ld(ra, rb);
                        if (last) {
                            if (a.s_out.p && out_ok && !*abort_flag) {
                                float *dst = a.s_out.p + sb + r * a.s_out.rs +
                                             (int64_t)(e0 + 64 * eb) * a.s_out.cs;
#pragma unroll
                                for (int k = 0; k < 32; ++k) {
                                    const float f0 = GLA == 2 ? colf[64 * eb + k] : fo;
                                    const float f1 = GLA == 2 ? colf[64 * eb + 32 + k] : fo;
                                    ra[k] = __float_as_uint(f0 * __uint_as_float(ra[k]));
                                    rb[k] = __float_as_uint(f1 * __uint_as_float(rb[k]));
                                }
                                if (a.s_out.cs == 1 &&
                                    (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                                    // contiguous row: 16-byte stores
#pragma unroll
                                    for (int k4 = 0; k4 < 8; ++k4) {
                                        *reinterpret_cast<uint4 *>(dst + 4 * k4) =
                                            make_uint4(ra[4 * k4], ra[4 * k4 + 1], ra[4 * k4 + 2],
                                                       ra[4 * k4 + 3]);
                                        *reinterpret_cast<uint4 *>(dst + 32 + 4 * k4) =
                                            make_uint4(rb[4 * k4], rb[4 * k4 + 1], rb[4 * k4 + 2],
                                                       rb[4 * k4 + 3]);
                                    }
                                } else {
#pragma unroll
                                    for (int k = 0; k < 32; ++k) {
                                        dst[k * a.s_out.cs] = __uint_as_float(ra[k]);
                                        dst[(k + 32) * a.s_out.cs] = __uint_as_float(rb[k]);
                                    }
                                }
                            }
                            continue;
                        }
                        if (!GLA && !SO &&
                            LA_OK_AT(r * 128 + eb * (D * 128) + 128 <= L::SB, 8))
                            store_row_sw128(sbf(pc) + eb * (D * 128), r, ra, rb);
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            if (GLA) {
                                const float o0 = GLA == 2 ? colf[64 * eb + k] : fo;
                                const float o1 = GLA == 2 ? colf[64 * eb + 32 + k] : fo;
                                const float n0 = GLA == 2 ? coln[64 * eb + k] : fn;
                                const float n1 = GLA == 2 ? coln[64 * eb + 32 + k] : fn;
                                ra[k] = __float_as_uint(n0 * (o0 * __uint_as_float(ra[k])));
                                rb[k] = __float_as_uint(n1 * (o1 * __uint_as_float(rb[k])));
                            } else {
                                ra[k] = __float_as_uint(gn * __uint_as_float(ra[k]));
                                rb[k] = __float_as_uint(gn * __uint_as_float(rb[k]));
                            }
                        }
                        if (GLA && LA_OK_AT(r * 128 + eb * (D * 128) + 128 <= L::SB, 8))
                            store_row_sw128(sbf(pc) + eb * (D * 128), r, ra, rb);
                        tmem_st32_issue(stm(pc) + 64 * eb, ra);
                        tmem_st32_issue(stm(pc) + 64 * eb + 32, rb);
                        tmem_wait_st();
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(s_ready);
            }
        } else {
            // ------------------------------------------------------- O group
            __nv_bfloat16 *obase = reinterpret_cast<__nv_bfloat16 *>(a.out.p) + row * a.out.sb +
                                   (int64_t)h * a.out.sh + e0;
            for (int c = 0; c < (SO ? 0 : nc); ++c) {
                const int s = c % NST;
                const int Lc = chunk_len(c);
                if (!warp_all(bwait(o_full, c & 1, abort_flag)))
                    break;
                tc_fence_after();
                float lr = 0.f;
                if (i < Lc) {
                    const int pi = rev ? Lc - 1 - i : i;
                    lr = GLA ? (BWD ? 1.f : scale) : (BWD ? pw[Lc - 1 - pi] : scale * pw[pi + 1]);
                }
                // a tile store may run past the end of a dense sequence (the
                // copy clips it) but not into the next packed sequence
                const bool tile = Lc == TC_C || !a.cu;
                // GLA 2 (dq~ or dk~, which the gate's gradient takes
                // unrounded): fp32 tiles, two 32-column parts at a time
                // through the Z slot; a packed sequence's last chunk row by
                // row from the registers
                const bool f32tile = GLA == 2 && tile;
                uint8_t *otile = sm + s * L::STAGE + L::XB + L::YB;   // Z slot, free once P Z is done
                __nv_bfloat16 *orow = obase + (bos + chunk_t0(c) + i) * a.out.st;
#pragma unroll 1
                for (int part = 0; part < E / 32; ++part) {
                    uint32_t ra[32], ri[32];
                    tmem_ld32_issue(tm + lane_off + TM_OA + 32 * part, ra);
                    tmem_ld32_issue(tm + lane_off + TM_OI + 32 * part, ri);
                    tmem_wait_ld(ra, ri);
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        ra[k] = __float_as_uint(
                            fmaf(lr, __uint_as_float(ri[k]), __uint_as_float(ra[k])));
                    if (f32tile && part == E / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive(o_free);   // both accumulators read
                    }
                    if (f32tile) {
                        if (LA_OK_AT((part & 1) * (TC_C * 128) + i * 128 + 128 <= L::ZB, 23))
                            store_row_f32_sw128(otile + (part & 1) * (TC_C * 128) + i * 128, i,
                                                ra);
                        if (part & 1) {
                            // this warp's 32 rows of both parts, once the
                            // copy engine can see them; the slot is written
                            // again only after the copy has read it
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0 && LA_OK_AT(bos + chunk_t0(c) + 32 * q >= 0 &&
                                                          bos + chunk_t0(c) < a.T &&
                                                          e0 + E <= a.E,
                                                      24)) {
#pragma unroll
                                for (int pp = 0; pp < 2; ++pp)
                                    tma_store_4d(&P.mo, otile + pp * (TC_C * 128) + q * 32 * 128,
                                                 32 * (part - 1 + pp) + e0, h,
                                                 (int)(bos + chunk_t0(c)) + 32 * q, (int)row);
                                bulk_commit_group();
                                bulk_wait_read_all();
                            }
                            __syncwarp();
                        }
                    } else if (GLA == 2) {
                        if (i < Lc && LA_OK_AT(bos + chunk_t0(c) + i < a.T, 22)) {
                            float4 *frow = reinterpret_cast<float4 *>(
                                static_cast<float *>(a.out.p) + row * a.out.sb +
                                (int64_t)h * a.out.sh + (bos + chunk_t0(c) + i) * a.out.st + e0 +
                                32 * part);
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                frow[k] = make_float4(
                                    __uint_as_float(ra[4 * k]), __uint_as_float(ra[4 * k + 1]),
                                    __uint_as_float(ra[4 * k + 2]), __uint_as_float(ra[4 * k + 3]));
                        }
                    } else if (LA_OK_AT((part >> 1) * (TC_C * 128) + i * 128 + 128 <= L::ZB, 11)) {
                        store_half_row_sw128(otile + (part >> 1) * (TC_C * 128) + i * 128, i,
                                             part & 1, ra);
                    }
                }
                if (!f32tile) {
                    tc_fence_before();
                    mbar_arrive(o_free);   // both accumulators read
                }
                if (GLA == 2) {
                    // written above
                } else if (tile) {
                    // each warp sends its own 32 rows once they are visible to
                    // the copy engine
                    fence_proxy_async_smem();
                    __syncwarp();
                    // a store may start past a dense sequence's end (the copy
                    // clips it), never before the tensor's start
                    if (lane == 0 && LA_OK_AT(bos + chunk_t0(c) + 32 * q >= 0 &&
                                                  bos + chunk_t0(c) < a.T && e0 + E <= a.E,
                                              19)) {
#pragma unroll
                        for (int b = 0; b < E / 64; ++b)
                            tma_store_4d(&P.mo, otile + b * (TC_C * 128) + q * 32 * 128, 64 * b + e0,
                                         h, (int)(bos + chunk_t0(c)) + 32 * q, (int)row);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                } else if (i < Lc && LA_OK_AT(bos + chunk_t0(c) + i < a.T, 18)) {
                    // row by row: this thread's own row, back out of the tile
#pragma unroll 1
                    for (int c16 = 0; c16 < E / 8; ++c16)
                        *reinterpret_cast<uint4 *>(orow + 8 * c16) = *reinterpret_cast<const uint4 *>(
                            otile + (c16 >> 3) * (TC_C * 128) + i * 128 + (((c16 & 7) ^ (i & 7)) << 4));
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&zfree[s]);   // this warp's rows of the Z slot may be refilled
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, TM_COLS);
    }
}

// Tile roles: X rows (scores = X Y^T, inter term X S), Y columns (scaled in
// place for the state update), Z values.  Forward: (X, Y, Z) = (q, k, v);
// backward: (k, q, w).  D = a.D; E is the value tile of one CTA (a.E / E
// CTAs per (sequence, head)).
template <int D, int E, bool BWD, int GLA, bool SO = false>
cudaError_t launch_tc(const SweepArgs &a, cudaStream_t s, const Tok *xyz = nullptr)
{
    if (a.D != D || a.E % E != 0)
        return cudaErrorNotSupported;
    TcParams p;
    // tile roles; the gated form names its three operands itself
    const Tok x = xyz ? xyz[0] : (BWD ? a.k : a.q), y = xyz ? xyz[1] : (BWD ? a.q : a.k);
    const Tok z = xyz ? xyz[2] : a.v;
    // state only: no X, no output (their maps are not used)
    if ((!SO && !make_map(&p.mx, x.p, D, a, x.sb, x.st, x.sh, TC_C, x.hdiv)) ||
        !make_map(&p.my, y.p, D, a, y.sb, y.st, y.sh, TC_C, y.hdiv) ||
        !make_map(&p.mz, z.p, a.E, a, z.sb, z.st, z.sh, TC_C, z.hdiv) ||
        (!SO && GLA != 2 && !make_map(&p.mo, a.out.p, a.E, a, a.out.sb, a.out.st, a.out.sh, 32)))
        return cudaErrorNotSupported;
    if (SO)
        p.mx = p.mo = p.my;
    if (GLA == 2 && !SO) {
        // fp32 output: 32-column tiles, or 16-byte row writes
        if ((reinterpret_cast<uintptr_t>(a.out.p) & 15) || a.out.sb % 4 || a.out.st % 4 ||
            a.out.sh % 4 ||
            !make_map(&p.mo, a.out.p, a.E, a, a.out.sb, a.out.st, a.out.sh, 32, 1, true))
            return cudaErrorNotSupported;
    }
    p.a = a;
    p.dx = x.hdiv;
    p.dy = y.hdiv;
    p.dz = z.hdiv;
    auto kern = tc_sweep_kernel<D, E, BWD, GLA, SO>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           TcLayout<D, E>::DYN);
    if (err != cudaSuccess)
        return err;
    // programmatic dependent launch: the CTAs may be scheduled, and run their
    // set-up, while the stream's previous kernel drains (the kernel waits for
    // it before touching global memory)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)a.N * a.H * (a.E / E)));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = TcLayout<D, E>::DYN;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kern, p);
    note_launch();
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

}  // namespace

// Value columns per CTA for key width D and a.E value columns: 128 where the
// state (D <= 128 rows) leaves TMEM room for it, else 64.
int tc_value_tile(int D, int E) { return D <= 128 && E % 128 == 0 ? 128 : 64; }

bool tc_sweep_supported(const SweepArgs &a)
{
    if (!a.bf16 || a.T < 1 || a.B < 1)
        return false;
    if ((a.D != 64 && a.D != 128 && a.D != 192 && a.D != 256) || a.E % 64 != 0 || a.E < 64 ||
        a.E > 256)
        return false;
    if ((int64_t)a.N * a.H * (a.E / tc_value_tile(a.D, a.E)) > INT_MAX)
        return false;
    return aligned_tok(a.q.p, a.q.sb, a.q.st, a.q.sh) &&
           aligned_tok(a.k.p, a.k.sb, a.k.st, a.k.sh) &&
           aligned_tok(a.v.p, a.v.sb, a.v.st, a.v.sh) &&
           aligned_tok(a.out.p, a.out.sb, a.out.st, a.out.sh);
}

namespace {
template <bool BWD> cudaError_t tc_sweep(const SweepArgs &a, cudaStream_t s)
{
    if (a.N == 0)
        return cudaSuccess;
    const bool wide = tc_value_tile(a.D, a.E) == 128;
    switch (a.D) {
    case 64:
        return wide ? launch_tc<64, 128, BWD, 0>(a, s) : launch_tc<64, 64, BWD, 0>(a, s);
    case 128:
        return wide ? launch_tc<128, 128, BWD, 0>(a, s) : launch_tc<128, 64, BWD, 0>(a, s);
    case 192:
        return launch_tc<192, 64, BWD, 0>(a, s);
    case 256:
        return launch_tc<256, 64, BWD, 0>(a, s);
    default:
        return cudaErrorNotSupported;
    }
}
}  // namespace

cudaError_t tc_forward_sweep(const SweepArgs &a, cudaStream_t s) { return tc_sweep<false>(a, s); }

cudaError_t tc_backward_sweep(const SweepArgs &a, cudaStream_t s) { return tc_sweep<true>(a, s); }

cudaError_t tc_gla_sweep(const SweepArgs &a, bool bwd, bool cols, const Tok &x, const Tok &y,
                         const Tok &z, cudaStream_t s, bool so)
{
    if (a.N == 0)
        return cudaSuccess;
    const Tok xyz[3] = {x, y, z};
    // one CTA per (sequence, head) with the 128 key channels as the state's
    // rows (D = 128, E in {64, 128}) or columns (E = 128, D in {64, 128})
    // state only: the forward-type sweeps (rows and columns) and the
    // backward-type one with gated rows (the split's first passes)
    if (cols) {
        if (a.E != 128 || (a.D != 64 && a.D != 128) || (so && bwd))
            return cudaErrorNotSupported;
        if (bwd)
            return a.D == 128 ? launch_tc<128, 128, true, 2>(a, s, xyz)
                              : launch_tc<64, 128, true, 2>(a, s, xyz);
        if (so)
            return a.D == 128 ? launch_tc<128, 128, false, 2, true>(a, s, xyz)
                              : launch_tc<64, 128, false, 2, true>(a, s, xyz);
        return a.D == 128 ? launch_tc<128, 128, false, 2>(a, s, xyz)
                          : launch_tc<64, 128, false, 2>(a, s, xyz);
    }
    if (a.D != 128 || (a.E != 64 && a.E != 128))
        return cudaErrorNotSupported;
    if (so)
        return bwd ? (a.E == 128 ? launch_tc<128, 128, true, 1, true>(a, s, xyz)
                                 : launch_tc<128, 64, true, 1, true>(a, s, xyz))
                   : (a.E == 128 ? launch_tc<128, 128, false, 1, true>(a, s, xyz)
                                 : launch_tc<128, 64, false, 1, true>(a, s, xyz));
    if (bwd)
        return a.E == 128 ? launch_tc<128, 128, true, 1>(a, s, xyz)
                          : launch_tc<128, 64, true, 1>(a, s, xyz);
    return a.E == 128 ? launch_tc<128, 128, false, 1>(a, s, xyz)
                      : launch_tc<128, 64, false, 1>(a, s, xyz);
}

cudaError_t tc_state_sweep(const SweepArgs &a, bool bwd, cudaStream_t s)
{
    if (a.N == 0)
        return cudaSuccess;
    // the state-only mode is built for 128 key channels and one value tile;
    // other shapes run the full sweep instead (the caller's fallback)
    if (a.D != 128 || (a.E != 64 && a.E != 128))
        return cudaErrorNotSupported;
    if (bwd)
        return a.E == 128 ? launch_tc<128, 128, true, 0, true>(a, s)
                          : launch_tc<128, 64, true, 0, true>(a, s);
    return a.E == 128 ? launch_tc<128, 128, false, 0, true>(a, s)
                      : launch_tc<128, 64, false, 0, true>(a, s);
}

cudaError_t tc_read_and_clear_error(cudaStream_t s, int *err)
{
    return read_and_clear_error_word(s, err);
}

}  // namespace la
