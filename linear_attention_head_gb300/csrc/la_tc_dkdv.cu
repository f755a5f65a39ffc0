// la_tc_dkdv.cu -- the backward pass's key and value gradients in one sweep
// (tcgen05 + TMEM + TMA) for bf16 tokens with d = e = 128.
//
// The gradient of the recurrence (the custom VJP of ejkernel `recurrent`,
// `_recurrent_bwd`, upstream grads (do, dfinal_state)) in the chunked form of
// Lightning Attention-2.  Per (sequence, head) the chunks of C = 128 tokens
// are visited against the processing order, carrying G = dL/dS (d x e, fp32,
// in TMEM) from d_final_state.  With Lc the chunk's valid length, p(.) the
// positions in processing order, s the scale and M_ji = gamma^(p(i)-p(j))
// where p(i) >= p(j) (else 0):
//     P1 = s (K Q^T) .* M            P2 = s (V dO^T) .* M
//     dV = P1 dO + diag(lk) K G       dK = P2 Q + diag(lk) V G^T
//     G <- gamma^Lc G + Q^T diag(lq) dO
// with lk_j = gamma^(Lc-1-p(j)) and lq_i = s gamma^(p(i)+1); d_initial_state
// is G after the chunk processed first.  These are the two backward-type
// sweeps of the two-pass form (dv, and dk with the roles swapped) in one
// pass: q, k, v and do are read once, dk and dv written once, G carried once.
// Every decay factor is gamma^m with m >= 0.
//
// One CTA per (sequence, head); 18 warps:
//   warp 0        TMA producer: the chunk's k, q, v, do tiles (128 tokens x
//                 128 channels, 128-byte swizzle) in that order, through a
//                 ring of six 32 KB slots (the k and v tiles always land in
//                 even slots, q and do in odd ones)
//   warp 1        TMEM allocator; one thread issues every tcgen05.mma
//   warps 2..9    P group: P1, then P2, from the scores in TMEM, packed as
//                 bf16 side by side in the columns of K Q^T (the A operands
//                 of P1 dO and P2 Q)
//   warps 10..13  S group: scales the k rows by lk and then the do rows by lq
//                 in place, each after the MMAs that read them unscaled, and
//                 turns G around each chunk (bf16 copy in shared memory,
//                 G * gamma^Lc of the next chunk back into TMEM)
//   warps 14..17  O group: scales the v rows by lk, then takes dV and dK from
//                 TMEM to bf16, staged in the slots of the chunk's k and v
//                 tiles and sent out by TMA stores
// TMEM (512 columns): K Q^T [0,128) -> P1 [0,64) and P2 [64,128); V dO^T
// [128,256), which dK takes once P2 is packed; dV [256,384); G [384,512).
// MMA order per chunk: K Q^T, V dO^T; dV = (lk K) G + P1 dO; dK = (lk V) G^T
// + P2 Q; G += Q^T (lq dO), after which the q and do slots are free.  The k
// and v slots are freed by the O group once the gradients staged there have
// been stored.  The next chunk's K Q^T needs only this chunk's MMAs done with
// P1 and P2, its V dO^T the dK columns read out of TMEM.  The v and do tiles
// of a chunk, loaded last, are first prefetched into L2 when its k tile is
// requested, a chunk ahead.
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises a shared
// abort flag and records LA_ERR_TIMEOUT in this file's device word, drains
// its own copies and MMAs, frees TMEM and returns.

#include <climits>
#include <cstdint>

#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

namespace la {
namespace {

constexpr int DK_D = 128;          // key width = value width
constexpr int DK_THREADS = 576;    // 18 warps
constexpr int DK_PG = 256;         // P group threads (warps 2..9)
constexpr int DK_SG = 128;         // S group threads (warps 10..13)
constexpr int DK_OG = 128;         // O group threads (warps 14..17)
constexpr int DK_NSLOT = 6;        // tile slots of the ring
constexpr int DK_TILE = TC_C * DK_D * 2;
constexpr uint32_t TS1 = 0, TP2 = 64, TS2 = 128, TK = 128, TV = 256, TG = 384, TCOLS = 512;

struct DkLayout {
    static constexpr int GOFF = DK_NSLOT * DK_TILE;      // bf16 copy of G, [E/64][D][64]
    static constexpr int MOFF = GOFF + DK_D * DK_D * 2;
    static constexpr int NBAR = 2 * DK_NSLOT + 14;
    static constexpr int PWOFF = MOFF + NBAR * 8;
    static constexpr int CFOFF = (PWOFF + (TC_C + 1) * 4 + 15) / 16 * 16;   // 32 column factors
    static constexpr int DTOFF = CFOFF + 32 * 4;                            // 64 diagonal factors
    static constexpr int SLOTOFF = DTOFF + 64 * 4;
    static constexpr int ABORTOFF = SLOTOFF + 4;
    static constexpr int BYTES = ABORTOFF + 4;
    static constexpr int DYN = BYTES + 1024;   // slack for 1024-byte alignment
    static_assert(DYN <= 232448, "shared memory per CTA");
};

struct DkParams {
    CUtensorMap mq, mk, mv, mdo, mdk, mdv;
    int dk_div, dv_div;   // head divisors of k and v (grouped key/value heads)
    SweepArgs a;          // a.out = dv; s_in = dL/dfinal (D x E), s_out = dL/dinitial
    TokOut dk;
};

// All consumer warps (P, S, O groups), once, after the decay tables.
__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(DK_PG + DK_SG + DK_OG) : "memory");
}
// The P group between reading its scores and packing P over them.
__device__ __forceinline__ void pg_sync()
{
    asm volatile("bar.sync 2, %0;" ::"n"(DK_PG) : "memory");
}
// One decision for the whole P group: true when `ok` holds on every thread
// (its named barriers after this must not be left by some warps only).
__device__ __forceinline__ bool pg_all(bool ok)
{
    uint32_t all;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.and.pred p, 2, %2, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(all)
                 : "r"(ok ? 1u : 0u), "n"(DK_PG)
                 : "memory");
    return all != 0;
}

// Two bf16 products in one instruction (round to nearest even).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Row i of both 64-channel blocks of the 128B-swizzled tile at t, times f, in
// place: the factor is rounded to bf16 once and each product to bf16 (as an
// in-place scaling of a bf16 tile must be); each block's eight 16-byte chunks
// are all loaded before any is stored.
__device__ __forceinline__ void scale_tile_row(uint8_t *t, int i, float f)
{
    if (!LA_OK_AT(i >= 0 && i < TC_C, 101))
        return;
    const uint32_t f2 = pack_bf16x2(f, f);
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
        uint8_t *rowp = t + b * (TC_C * 128) + i * 128;
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = *reinterpret_cast<const uint4 *>(rowp + ((k ^ (i & 7)) << 4));
#pragma unroll
        for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4 *>(rowp + ((k ^ (i & 7)) << 4)) =
                make_uint4(mul_bf16x2(v[k].x, f2), mul_bf16x2(v[k].y, f2), mul_bf16x2(v[k].z, f2),
                           mul_bf16x2(v[k].w, f2));
    }
}

__global__ void __launch_bounds__(DK_THREADS, 1) tc_dkdv_kernel(const __grid_constant__ DkParams P)
{
    using L = DkLayout;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const SweepArgs &a = P.a;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::MOFF);
    // full[s]: the tile in slot s landed; empty[s]: slot s may be refilled
    uint64_t *full = bars, *empty = bars + DK_NSLOT;
    uint64_t *sc1_full = bars + 2 * DK_NSLOT;   // K Q^T in TMEM
    uint64_t *sc2_full = sc1_full + 1;          // V dO^T in TMEM
    uint64_t *p1_ready = sc1_full + 2;          // P1 packed
    uint64_t *p2_ready = sc1_full + 3;          // P2 packed
    uint64_t *k_scaled = sc1_full + 4;          // k rows times lk
    uint64_t *v_scaled = sc1_full + 5;          // v rows times lk
    uint64_t *do_scaled = sc1_full + 6;         // do rows times lq
    uint64_t *s_ready = sc1_full + 7;           // G copy written, TMEM G pre-scaled
    uint64_t *dv_full = sc1_full + 8;           // dV done (and both scores)
    uint64_t *dk_full = sc1_full + 9;           // dK done
    uint64_t *g_done = sc1_full + 10;           // the G update done (the chunk's last MMA)
    uint64_t *dv_drained = sc1_full + 11;       // dV read out of TMEM
    uint64_t *dk_drained = sc1_full + 12;       // dK read out of TMEM
    uint64_t *drain = sc1_full + 13;
    float *pw = reinterpret_cast<float *>(sm + L::PWOFF);
    float *cf = reinterpret_cast<float *>(sm + L::CFOFF);
    float *dt = reinterpret_cast<float *>(sm + L::DTOFF);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::SLOTOFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::ABORTOFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < DK_NSLOT; ++i) {
            mbar_init(&full[i], 1);
            // even slots (k, v) are freed by the four O warps, odd ones (q,
            // do) by an MMA commit
            mbar_init(&empty[i], (i & 1) ? 1 : DK_OG / 32);
        }
        mbar_init(sc1_full, 1);
        mbar_init(sc2_full, 1);
        mbar_init(p1_ready, DK_PG);
        mbar_init(p2_ready, DK_PG);
        mbar_init(k_scaled, DK_SG);
        mbar_init(v_scaled, DK_OG);
        mbar_init(do_scaled, DK_SG);
        mbar_init(s_ready, DK_SG);
        mbar_init(dv_full, 1);
        mbar_init(dk_full, 1);
        mbar_init(g_done, 1);
        mbar_init(dv_drained, DK_OG);
        mbar_init(dk_drained, DK_OG);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, TCOLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&P.mq);
        prefetch_tmap(&P.mk);
        prefetch_tmap(&P.mv);
        prefetch_tmap(&P.mdo);
        prefetch_tmap(&P.mdk);
        prefetch_tmap(&P.mdv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    // the set-up above touches only shared memory, TMEM and the parameters;
    // global memory only after the stream's previous kernel is done
    grid_dep_wait();
    grid_dep_launch_dependents();

    // work item: the rank-th sequence of the schedule, one head per CTA
    const int rank = blockIdx.x / a.H, h = blockIdx.x % a.H;
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
    const int nc = (int)((len + TC_C - 1) / TC_C);
    const bool rev = a.reverse != 0;
    const bool flip = !rev;   // chunk visiting order and mask direction (against processing)
    auto chunk_t0 = [&](int c) { return (int64_t)(flip ? nc - 1 - c : c) * TC_C; };
    auto chunk_len = [&](int c) {
        const int64_t t0 = chunk_t0(c);
        return (int)(len - t0 < TC_C ? len - t0 : TC_C);
    };
    // tile t = 4c + r of the ring: r = 0 k, 1 q, 2 v, 3 do of chunk c
    auto slot_of = [](int t) { return t % DK_NSLOT; };
    auto use_of = [](int t) { return (uint32_t)((t / DK_NSLOT) & 1); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int hk = h / P.dk_div, hv = h / P.dv_div;
            int issued = 0;
            for (int t = 0; t < 4 * nc; ++t) {
                const int c = t >> 2, r = t & 3, s = slot_of(t);
                if (t >= DK_NSLOT && !bwait(&empty[s], ((t / DK_NSLOT) - 1) & 1, abort_flag))
                    break;
                const CUtensorMap *m = r == 0 ? &P.mk : r == 1 ? &P.mq : r == 2 ? &P.mv : &P.mdo;
                const int hh = r == 0 ? hk : r == 2 ? hv : h;
                const int t0 = (int)(bos + chunk_t0(c));
                if (!LA_OK_AT(t0 >= 0 && t0 < a.T && s >= 0 && s < DK_NSLOT, 114))
                    break;
                if (r == 0) {
                    // the v and do tiles of this chunk wait for slots the
                    // chunk before frees late: have them in L2 by then
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        tma_prefetch_l2_4d(&P.mv, 64 * b, hv, t0, (int)row);
                        tma_prefetch_l2_4d(&P.mdo, 64 * b, h, t0, (int)row);
                    }
                }
                uint8_t *dst = sm + s * DK_TILE;
                mbar_arrive_expect_tx(&full[s], DK_TILE);
                tma_load_4d(dst, m, &full[s], 0, hh, t0, (int)row);
                tma_load_4d(dst + TC_C * 128, m, &full[s], 64, hh, t0, (int)row);
                ++issued;
            }
            // every copy this thread issued has landed before the CTA may exit
            for (int t = issued > DK_NSLOT ? issued - DK_NSLOT : 0; t < issued; ++t)
                drain_wait(&full[slot_of(t)], use_of(t));
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_ss = idesc_bf16_f32(128, 128, 0, 0);    // scores: both K-major
            const uint32_t id_mn = idesc_bf16_f32(128, 128, 0, 1);    // B MN-major, N = 128
            const uint32_t id_g = idesc_bf16_f32(128, 128, 1, 1);     // both MN-major
            const uint32_t sbase = smem_u32(sm), ga = sbase + L::GOFF;
            auto addr = [&](int t) { return sbase + (uint32_t)(slot_of(t) * DK_TILE); };
            bool any = false;
            for (int c = 0; c < nc; ++c) {
                const int tk = 4 * c, tq = tk + 1, tv = tk + 2, to = tk + 3;
                const uint32_t ka = addr(tk), qa = addr(tq), va = addr(tv), oa = addr(to);
                if (!LA_OK_AT(ka + DK_TILE <= ga && qa + DK_TILE <= ga && va + DK_TILE <= ga &&
                                  oa + DK_TILE <= ga && ga + DK_D * DK_D * 2 <= sbase + L::MOFF,
                              107))
                    break;
                // K Q^T goes to [0,128): free once the previous chunk's dK
                // MMAs, the last to read P1 and P2 there, are done
                if (c > 0 && !bwait(dk_full, (c - 1) & 1, abort_flag))
                    break;
                if (!bwait(&full[slot_of(tk)], use_of(tk), abort_flag) ||
                    !bwait(&full[slot_of(tq)], use_of(tq), abort_flag))
                    break;
                tc_fence_after();
                // K Q^T (both K-major, K = d)
#pragma unroll
                for (int kk = 0; kk < DK_D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TS1, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024),
                           id_ss, kk > 0);
                }
                mma_commit(sc1_full);
                any = true;
                // V dO^T to [128,256): after the previous dK has left TMEM
                if (c > 0 && !bwait(dk_drained, (c - 1) & 1, abort_flag))
                    break;
                if (!bwait(&full[slot_of(tv)], use_of(tv), abort_flag) ||
                    !bwait(&full[slot_of(to)], use_of(to), abort_flag))
                    break;
                tc_fence_after();
                // V dO^T (both K-major, K = e)
#pragma unroll
                for (int kk = 0; kk < DK_D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TS2, sdesc_sw128(va + off, 16, 1024), sdesc_sw128(oa + off, 16, 1024),
                           id_ss, kk > 0);
                }
                mma_commit(sc2_full);
                // dV = (lk K) G + P1 dO: K K-major, the G copy MN-major (K = d,
                // N = e); P1 packed in TMEM, do MN-major (K = tokens).  The
                // inter term needs no P, so it goes first.
                if (!bwait(k_scaled, c & 1, abort_flag) || !bwait(s_ready, c & 1, abort_flag))
                    break;
                if (c > 0 && !bwait(dv_drained, (c - 1) & 1, abort_flag))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK_D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    mma_ss(tm + TV, sdesc_sw128(ka + off, 16, 1024),
                           sdesc_sw128(ga + kk * 2048, DK_D * 128, 1024), id_mn, kk > 0);
                }
                if (!bwait(p1_ready, c & 1, abort_flag))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < TC_C / 16; ++kk)
                    mma_ts(tm + TV, tm + TS1 + kk * 8, sdesc_sw128(oa + kk * 2048, TC_C * 128, 1024),
                           id_mn, 1);
                mma_commit(dv_full);
                // dK = (lk V) G^T + P2 Q in the columns of V dO^T, free once
                // P2 is packed: V K-major (K = e), the G copy as K-major rows
                // (N = d, K = e); P2 packed in TMEM, q MN-major (K = tokens)
                if (!bwait(p2_ready, c & 1, abort_flag) || !bwait(v_scaled, c & 1, abort_flag))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK_D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TC_C * 128) + (kk & 3) * 32;
                    const uint32_t goff = (kk >> 2) * (DK_D * 128) + (kk & 3) * 32;
                    mma_ss(tm + TK, sdesc_sw128(va + off, 16, 1024), sdesc_sw128(ga + goff, 16, 1024),
                           id_ss, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < TC_C / 16; ++kk)
                    mma_ts(tm + TK, tm + TP2 + kk * 8, sdesc_sw128(qa + kk * 2048, TC_C * 128, 1024),
                           id_mn, 1);
                mma_commit(dk_full);
                // G += Q^T (lq dO): both MN-major, M = d, K = tokens
                if (!bwait(do_scaled, c & 1, abort_flag))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < TC_C / 16; ++kk)
                    mma_ss(tm + TG, sdesc_sw128(qa + kk * 2048, TC_C * 128, 1024),
                           sdesc_sw128(oa + kk * 2048, TC_C * 128, 1024), id_g, 1);
                mma_commit(g_done);
                mma_commit(&empty[slot_of(to)]);   // q and do have been read for the last time
                mma_commit(&empty[slot_of(tq)]);
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
        for (int m = et; m <= TC_C; m += DK_PG + DK_SG + DK_OG)
            pw[m] = m == 0 ? 1.f : expf(g * (float)m);
        if (et < 32) {   // column factors of the off-diagonal blocks
            const int m = flip ? et : 31 - et;
            cf[et] = m == 0 ? 1.f : expf(g * (float)m);
        } else if (et < 96) {   // diagonal blocks, index jj - lane + 31
            const int u = et - 32;
            const int m = flip ? u - 31 : 31 - u;
            dt[u] = m < 0 || u > 62 ? 0.f : (m == 0 ? scale : scale * expf(g * (float)m));
        }
        consumers_sync();
        const int q = warp & 3;
        const int i = 32 * q + lane;   // TMEM lane = tile row
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;

        if (warp < 10) {
            // ------------------------------------------------------- P group
            const int hh = (warp - 2) >> 2;   // key half: score columns 64 hh ..
            const int j0 = 64 * hh;
            const int b0 = 2 * hh, b1 = b0 + 1;
            // block kinds are warp-uniform: 0 zero, 1 rank one, 2 diagonal
            const int k0 = b0 == q ? 2 : ((flip ? b0 > q : b0 < q) ? 1 : 0);
            const int k1 = b1 == q ? 2 : ((flip ? b1 > q : b1 < q) ? 1 : 0);
            const int ix0 = flip ? 32 * (b0 - q) - lane : 32 * (q - b0) + lane - 31;
            const int ix1 = flip ? 32 * (b1 - q) - lane : 32 * (q - b1) + lane - 31;
            const float rf0 =
                k0 == 1 && LA_OK_AT(ix0 >= 0 && ix0 <= TC_C, 104) ? scale * pw[ix0] : 0.f;
            const float rf1 =
                k1 == 1 && LA_OK_AT(ix1 >= 0 && ix1 <= TC_C, 104) ? scale * pw[ix1] : 0.f;
            bool run = true;
            for (int c = 0; c < nc && run; ++c) {
                const int Lc = chunk_len(c);
                if (!LA_OK_AT(Lc >= 1 && Lc <= TC_C, 105))
                    break;
#pragma unroll 1
                for (int pass = 0; pass < 2; ++pass) {
                    // pass 0: P1 from K Q^T, pass 1: P2 from V dO^T
                    if (!pg_all(bwait(pass ? sc2_full : sc1_full, c & 1, abort_flag))) {
                        run = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = tm + lane_off + (pass ? TS2 : TS1);
                    uint32_t ra[32], rb[32];
                    tmem_ld32_issue(base + j0, ra);
                    tmem_ld32_issue(base + j0 + 32, rb);
                    tmem_wait_ld(ra, rb);
                    p_block_full(ra, k0, rf0, cf, dt, lane);
                    p_block_full(rb, k1, rf1, cf, dt, lane);
                    if (Lc < TC_C) {
                        // the sequence ends inside this chunk: keys past the
                        // end (forward order: query columns) or rows past it
                        // (reverse order) are zero
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
                                ra[2 * m] &=
                                    (ja < Lc ? 0xffffu : 0u) | (ja + 1 < Lc ? 0xffff0000u : 0u);
                                rb[2 * m] &=
                                    (jb < Lc ? 0xffffu : 0u) | (jb + 1 < Lc ? 0xffff0000u : 0u);
                            }
                        }
                    }
                    // keys 64 hh .. of this row go to columns 32 hh .. of P1
                    // (over K Q^T itself: every warp must have read its scores
                    // first) or of P2 (next to P1, in columns K Q^T freed)
                    const uint32_t pbase = tm + lane_off + (pass ? TP2 : TS1) + 32 * hh;
                    if (!pass) {
                        tc_fence_before();
                        pg_sync();
                        tc_fence_after();
                    }
                    tmem_st16_even_issue(pbase, ra);
                    tmem_st16_even_issue(pbase + 16, rb);
                    tmem_wait_st();
                    tc_fence_before();
                    if (!(a.withhold_handoff && c == 0 && pass == 0))   // diagnostic
                        mbar_arrive(pass ? p2_ready : p1_ready);
                }
            }
        } else if (warp < 14) {
            // ------------------------------------------------------- S group
            const int64_t sb = ((int64_t)n * a.H + h) * (int64_t)DK_D * DK_D;
            uint8_t *grow = sm + L::GOFF + i * 128;
            const uint32_t gtm = tm + lane_off + TG;
            // the state tensors' extent: both ends of row i fall inside it
            const int64_t s_total = (int64_t)a.N * a.H * DK_D * DK_D;
            auto s_ok = [&](int64_t rs, int64_t cs) {
                const int64_t lo = sb + i * rs, hi = lo + (int64_t)(DK_D - 1) * cs;
                return lo >= 0 && hi < s_total;
            };
            const bool in_ok = !a.s_in.p || LA_OK_AT(s_ok(a.s_in.rs, a.s_in.cs), 109);
            const bool out_ok = !a.s_out.p || LA_OK_AT(s_ok(a.s_out.rs, a.s_out.cs), 110);
            if (!in_ok || !out_ok) {
                // leave the state alone: the MMA issuer's s_ready wait runs out
            } else if (nc == 0)
                state_copy(a.s_in, a.s_out, sb, i, 0, DK_D);
            else
                state_in(a.s_in, sb, i, 0, DK_D, grow, DK_D * 128, gtm, pw[chunk_len(0)], 1.f);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(s_ready);
            for (int c = 0; c < nc; ++c) {
                const int Lc = chunk_len(c);
                const int tk = 4 * c, to = tk + 3;
                float lk = 0.f, lq = 0.f;
                if (i < Lc) {
                    const int pi = rev ? Lc - 1 - i : i;
                    lk = pw[Lc - 1 - pi];
                    lq = scale * pw[pi + 1];
                }
                // k after K Q^T (rows past the end: zero)
                if (!warp_all(bwait(sc1_full, c & 1, abort_flag)))
                    break;
                scale_tile_row(sm + slot_of(tk) * DK_TILE, i, lk);
                fence_proxy_async_smem();
                mbar_arrive(k_scaled);
                // do after V dO^T and P1 dO (both done with dV)
                if (!warp_all(bwait(dv_full, c & 1, abort_flag)))
                    break;
                scale_tile_row(sm + slot_of(to) * DK_TILE, i, lq);
                fence_proxy_async_smem();
                mbar_arrive(do_scaled);
                // G after its update, the chunk's last MMA (every read of the
                // copy, by dV and dK, came before it)
                if (!warp_all(bwait(g_done, c & 1, abort_flag)))
                    break;
                tc_fence_after();
                const bool last = c + 1 == nc;
                const float gn = last ? 1.f : pw[chunk_len(c + 1)];
#pragma unroll 1
                for (int eb = 0; eb < DK_D / 64; ++eb) {
                    uint32_t ra[32], rb[32];
                    tmem_ld32_issue(gtm + 64 * eb, ra);
                    tmem_ld32_issue(gtm + 64 * eb + 32, rb);
                    tmem_wait_ld(ra, rb);
                    if (last) {
                        if (a.s_out.p && out_ok && !*abort_flag) {
                            float *dst = a.s_out.p + sb + i * a.s_out.rs + 64 * eb * a.s_out.cs;
                            if (a.s_out.cs == 1 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
                                for (int k4 = 0; k4 < 8; ++k4) {
                                    *reinterpret_cast<uint4 *>(dst + 4 * k4) = make_uint4(
                                        ra[4 * k4], ra[4 * k4 + 1], ra[4 * k4 + 2], ra[4 * k4 + 3]);
                                    *reinterpret_cast<uint4 *>(dst + 32 + 4 * k4) = make_uint4(
                                        rb[4 * k4], rb[4 * k4 + 1], rb[4 * k4 + 2], rb[4 * k4 + 3]);
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
                    if (LA_OK_AT(i * 128 + eb * (DK_D * 128) + 128 <= DK_D * DK_D * 2, 103))
                        store_row_sw128(grow + eb * (DK_D * 128), i, ra, rb);
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        ra[k] = __float_as_uint(gn * __uint_as_float(ra[k]));
                        rb[k] = __float_as_uint(gn * __uint_as_float(rb[k]));
                    }
                    tmem_st32_issue(gtm + 64 * eb, ra);
                    tmem_st32_issue(gtm + 64 * eb + 32, rb);
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(s_ready);
            }
        } else {
            // ------------------------------------------------------- O group
            for (int c = 0; c < nc; ++c) {
                const int Lc = chunk_len(c);
                const int64_t t0 = bos + chunk_t0(c);
                // v after V dO^T (rows past the end: zero)
                float lk = 0.f;
                if (i < Lc)
                    lk = pw[Lc - 1 - (rev ? Lc - 1 - i : i)];
                if (!warp_all(bwait(sc2_full, c & 1, abort_flag)))
                    break;
                scale_tile_row(sm + slot_of(4 * c + 2) * DK_TILE, i, lk);
                fence_proxy_async_smem();
                mbar_arrive(v_scaled);
                // a tile store may run past the end of a dense sequence (the
                // copy clips it) but not into the next packed sequence
                const bool tile = Lc == TC_C || !a.cu;
                bool ok = true;
#pragma unroll 1
                for (int which = 0; which < 2; ++which) {
                    // which 0: dV from [256,384) into the k slot; 1: dK from
                    // [128,256) into the v slot; the columns are handed back
                    // as soon as they are read
                    if (!warp_all(bwait(which ? dk_full : dv_full, c & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int s = slot_of(4 * c + (which ? 2 : 0));
                    uint8_t *stage = sm + s * DK_TILE;
#pragma unroll 1
                    for (int part = 0; part < DK_D / 32; ++part) {
                        uint32_t ra[32];
                        tmem_ld32(tm + lane_off + (which ? TK : TV) + 32 * part, ra);
                        if (part == 3) {
                            tc_fence_before();
                            mbar_arrive(which ? dk_drained : dv_drained);
                        }
                        if (LA_OK_AT((part >> 1) * (TC_C * 128) + i * 128 + 128 <= DK_TILE, 102))
                            store_half_row_sw128(stage + (part >> 1) * (TC_C * 128) + i * 128, i,
                                             part & 1, ra);
                    }
                    const TokOut &dst = which ? P.dk : a.out;
                    if (tile) {
                        // each warp sends its own 32 rows once they are
                        // visible to the copy engine
                        fence_proxy_async_smem();
                        __syncwarp();
                        // a store may start past a dense sequence's end (the
                        // copy clips it), never before the tensor's start
                        if (lane == 0 && LA_OK_AT(t0 + 32 * q >= 0 && t0 < a.T, 113)) {
                            const CUtensorMap *m = which ? &P.mdk : &P.mdv;
#pragma unroll
                            for (int b = 0; b < DK_D / 64; ++b)
                                tma_store_4d(m, stage + b * (TC_C * 128) + q * 32 * 128, 64 * b, h,
                                             (int)t0 + 32 * q, (int)row);
                            bulk_commit_group();
                            bulk_wait_read_all();
                        }
                    } else if (i < Lc && LA_OK_AT(t0 + i < a.T, 112)) {
                        // row by row: this thread's own row, back out of the tile
                        __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(dst.p) +
                                              row * dst.sb + (t0 + i) * dst.st + (int64_t)h * dst.sh;
#pragma unroll 1
                        for (int c16 = 0; c16 < DK_D / 8; ++c16)
                            *reinterpret_cast<uint4 *>(orow + 8 * c16) =
                                *reinterpret_cast<const uint4 *>(stage + (c16 >> 3) * (TC_C * 128) +
                                                                 i * 128 +
                                                                 (((c16 & 7) ^ (i & 7)) << 4));
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&empty[s]);   // this warp's rows of the slot may be refilled
                }
                if (!ok)
                    break;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, TCOLS);
    }
}

}  // namespace

bool tc_dkdv_supported(const SweepArgs &a, const Tok &v, const TokOut &dk)
{
    if (!a.bf16 || a.D != DK_D || a.E != DK_D || a.T < 1 || a.B < 1)
        return false;
    if ((int64_t)a.N * a.H > INT_MAX)
        return false;
    return aligned_tok(a.q.p, a.q.sb, a.q.st, a.q.sh) &&
           aligned_tok(a.k.p, a.k.sb, a.k.st, a.k.sh) && aligned_tok(v.p, v.sb, v.st, v.sh) &&
           aligned_tok(a.v.p, a.v.sb, a.v.st, a.v.sh) &&
           aligned_tok(a.out.p, a.out.sb, a.out.st, a.out.sh) &&
           aligned_tok(dk.p, dk.sb, dk.st, dk.sh);
}

cudaError_t tc_dkdv_sweep(const SweepArgs &a, const Tok &v, const TokOut &dk, cudaStream_t s)
{
    if (a.N == 0)
        return cudaSuccess;
    DkParams p;
    if (!make_map(&p.mq, a.q.p, DK_D, a, a.q.sb, a.q.st, a.q.sh, TC_C, a.q.hdiv) ||
        !make_map(&p.mk, a.k.p, DK_D, a, a.k.sb, a.k.st, a.k.sh, TC_C, a.k.hdiv) ||
        !make_map(&p.mv, v.p, DK_D, a, v.sb, v.st, v.sh, TC_C, v.hdiv) ||
        !make_map(&p.mdo, a.v.p, DK_D, a, a.v.sb, a.v.st, a.v.sh, TC_C, a.v.hdiv) ||
        !make_map(&p.mdk, dk.p, DK_D, a, dk.sb, dk.st, dk.sh, 32) ||
        !make_map(&p.mdv, a.out.p, DK_D, a, a.out.sb, a.out.st, a.out.sh, 32))
        return cudaErrorNotSupported;
    p.dk_div = a.k.hdiv;
    p.dv_div = v.hdiv;
    p.a = a;
    p.dk = dk;
    cudaError_t err = cudaFuncSetAttribute(tc_dkdv_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           DkLayout::DYN);
    if (err != cudaSuccess)
        return err;
    // programmatic dependent launch, as the sweep kernels
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)a.N * a.H));
    cfg.blockDim = dim3(DK_THREADS);
    cfg.dynamicSmemBytes = DkLayout::DYN;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, tc_dkdv_kernel, p);
    note_launch();
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

cudaError_t tc_dkdv_read_and_clear_error(cudaStream_t s, int *err)
{
    return read_and_clear_error_word(s, err);
}

}  // namespace la
