// la_tc_common.cuh -- device and host pieces shared by the tensor-core
// (tcgen05 + TMEM + TMA) kernels: bounded mbarrier waits with this
// translation unit's error word, 128-byte-swizzled tile rows, the state's
// entry into TMEM and shared memory, the block-factored decay mask of one
// 32 x 32 block of scores, and the 4-D tensor maps of token tensors.
// Everything sits in an anonymous namespace: each kernel file that includes
// it gets its own copy, including its own error word (read and cleared by
// read_and_clear_error_word on the host side of the same file).
#pragma once

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

// LA_ERR_TIMEOUT once a bounded wait of this file's kernels ran out
__device__ int g_tc_error;

constexpr int TC_C = 128;        // tokens per chunk (MMA M and the P Z K-extent)
constexpr uint64_t TC_WAIT_NS = 2000000000ull;
constexpr int TC_ERR_TIMEOUT = 4;
constexpr int TC_ERR_BOUNDS = 5;   // bounds-checking build: a failed index check

// Index checks of the bounds-checking build (LA_CHECK_BOUNDS defined): LA_OK_AT
// (cond, site) is the condition, and records a failure as TC_ERR_BOUNDS with
// the site number above the low byte of the error word (the first failure
// wins); the caller skips the access it guards.  In the normal build it is
// true without evaluating the condition, and the checks compile away.
#ifdef LA_CHECK_BOUNDS
__device__ __noinline__ bool la_ok_at(bool ok, int site)
{
    if (!ok)
        atomicCAS(&g_tc_error, 0, TC_ERR_BOUNDS | (site << 8));
    return ok;
}
#define LA_OK_AT(cond, site) la_ok_at((cond), (site))
#else
#define LA_OK_AT(cond, site) (true || (cond))
#endif

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

// 16 bytes = 8 bf16 scaled by f, in place.
__device__ __forceinline__ uint4 scale8(uint4 v, float f)
{
    v.x = pack_bf16x2(bf16lo(v.x) * f, bf16hi(v.x) * f);
    v.y = pack_bf16x2(bf16lo(v.y) * f, bf16hi(v.y) * f);
    v.z = pack_bf16x2(bf16lo(v.z) * f, bf16hi(v.z) * f);
    v.w = pack_bf16x2(bf16lo(v.w) * f, bf16hi(v.w) * f);
    return v;
}

// One 128-byte row of a 128B-swizzled bf16 tile, scaled in place.  All eight
// 16-byte chunks are loaded before any is stored, so the loads are not held
// back behind stores the compiler cannot prove to be elsewhere.
__device__ __forceinline__ void scale_row_sw128(uint8_t *row_base, int row, float f)
{
    uint4 v[8];
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16)
        v[c16] = *reinterpret_cast<const uint4 *>(row_base + ((c16 ^ (row & 7)) << 4));
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4 *>(row_base + ((c16 ^ (row & 7)) << 4)) = scale8(v[c16], f);
}

// 64 fp32 (as bits, lo = first 32 columns, hi = next 32) -> one 128-byte
// row of a 128B-swizzled bf16 tile.
__device__ __forceinline__ void store_row_sw128(uint8_t *row_base, int row,
                                                const uint32_t (&lo)[32], const uint32_t (&hi)[32])
{
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
        const uint32_t *x = c16 < 4 ? lo : hi;
        const int o = 8 * (c16 & 3);
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(x[o + 0]), __uint_as_float(x[o + 1]));
        v.y = pack_bf16x2(__uint_as_float(x[o + 2]), __uint_as_float(x[o + 3]));
        v.z = pack_bf16x2(__uint_as_float(x[o + 4]), __uint_as_float(x[o + 5]));
        v.w = pack_bf16x2(__uint_as_float(x[o + 6]), __uint_as_float(x[o + 7]));
        *reinterpret_cast<uint4 *>(row_base + ((c16 ^ (row & 7)) << 4)) = v;
    }
}

// 32 fp32 (as bits) -> 16-byte chunks 4*half .. 4*half+3 of a 128-byte row of
// a 128B-swizzled bf16 tile.
__device__ __forceinline__ void store_half_row_sw128(uint8_t *row_base, int row, int half,
                                                     const uint32_t (&x)[32])
{
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4)
        *reinterpret_cast<uint4 *>(row_base + (((4 * half + k4) ^ (row & 7)) << 4)) = make_uint4(
            pack_bf16x2(__uint_as_float(x[8 * k4 + 0]), __uint_as_float(x[8 * k4 + 1])),
            pack_bf16x2(__uint_as_float(x[8 * k4 + 2]), __uint_as_float(x[8 * k4 + 3])),
            pack_bf16x2(__uint_as_float(x[8 * k4 + 4]), __uint_as_float(x[8 * k4 + 5])),
            pack_bf16x2(__uint_as_float(x[8 * k4 + 6]), __uint_as_float(x[8 * k4 + 7])));
}

// 32 fp32 values as one 128-byte row of a 128B-swizzled tile.
__device__ __forceinline__ void store_row_f32_sw128(uint8_t *row_base, int row,
                                                    const uint32_t (&x)[32])
{
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4 *>(row_base + ((j ^ (row & 7)) << 4)) =
            make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
}

// Initial state row i, 8 columns at a time (once per CTA): fp32 from global
// (any strides; this CTA's value columns start at e0), times colf[column]
// when colf is given, -> times c0 as bf16 into the swizzled S copy (row i at
// sbf, blocks of 64 columns dstride bytes apart), and times g0 into TMEM.
__device__ __forceinline__ void state_in(const StateIn &sin, int64_t base, int i, int e0, int E_,
                                         uint8_t *sbf, int dstride, uint32_t tmem_row, float g0,
                                         float c0, const float *colf = nullptr)
{
#pragma unroll 1
    for (int p8 = 0; p8 < E_ / 8; ++p8) {
        float x[8];
        const float *src =
            sin.p ? sin.p + base + i * sin.rs + (int64_t)(e0 + 8 * p8) * sin.cs : nullptr;
        if (src && sin.cs == 1 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
            // contiguous row: two 16-byte loads
            const float4 lo = *reinterpret_cast<const float4 *>(src);
            const float4 hi = *reinterpret_cast<const float4 *>(src + 4);
            x[0] = lo.x, x[1] = lo.y, x[2] = lo.z, x[3] = lo.w;
            x[4] = hi.x, x[5] = hi.y, x[6] = hi.z, x[7] = hi.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                x[k] = src ? src[k * sin.cs] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            x[k] *= colf ? colf[8 * p8 + k] : 1.f;
        *reinterpret_cast<uint4 *>(sbf + (p8 >> 3) * dstride + (((p8 & 7) ^ (i & 7)) << 4)) =
            make_uint4(pack_bf16x2(c0 * x[0], c0 * x[1]), pack_bf16x2(c0 * x[2], c0 * x[3]),
                       pack_bf16x2(c0 * x[4], c0 * x[5]), pack_bf16x2(c0 * x[6], c0 * x[7]));
        uint32_t r[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            r[k] = __float_as_uint(g0 * x[k]);
        tmem_st8(tmem_row + 8 * p8, r);
    }
}

// Empty sequence: initial state row i (zero when absent) -> final state row i,
// value columns e0 .. e0 + E_ - 1.
__device__ __forceinline__ void state_copy(const StateIn &sin, const StateOut &sout, int64_t base,
                                           int i, int e0, int E_)
{
    if (!sout.p)
        return;
#pragma unroll 1
    for (int k = e0; k < e0 + E_; ++k)
        sout.p[base + i * sout.rs + k * sout.cs] =
            sin.p ? sin.p[base + i * sin.rs + k * sin.cs] : 0.f;
}

// One 32-key block of P for the 32 rows of a warp, on a full chunk.  The
// decay of the chunk's 128 x 128 mask, cut into 32 x 32 blocks, is per block
// either zero (the wrong side of the diagonal), a diagonal block, or the
// product of a row factor and a column factor: gamma^(i-j) =
// gamma^(32(q-b)+lane-31) gamma^(31-jj) below the diagonal (row quarter q, key
// block b, jj = j - 32b), and gamma^(32(b-q)-lane) gamma^jj above it, every
// factor <= 1.  Diagonal blocks take gamma^|lane-jj| (zero on the masked side)
// from a 63-entry table indexed by jj - lane + 31.  scale is folded into the
// row factor and the table.  r holds the block's 32 scores; packed pair m of P
// goes into r[2m].
__device__ __forceinline__ void p_block_full(uint32_t (&r)[32], int kind, float rf, const float *cf,
                                             const float *dt, int lane)
{
    if (kind == 0) {
#pragma unroll
        for (int m = 0; m < 16; ++m)
            r[2 * m] = 0u;
    } else if (kind == 1) {
        const float2 rr = make_float2(rf, rf);
        const uint32_t cfa = smem_u32(cf);
#pragma unroll
        for (int m4 = 0; m4 < 8; ++m4) {
            float4 c;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(c.x), "=f"(c.y), "=f"(c.z), "=f"(c.w)
                         : "r"(cfa + 16 * m4));
            const float2 v0 = mul_f32x2(
                mul_f32x2(make_float2(__uint_as_float(r[4 * m4]), __uint_as_float(r[4 * m4 + 1])),
                          make_float2(c.x, c.y)),
                rr);
            const float2 v1 = mul_f32x2(
                mul_f32x2(make_float2(__uint_as_float(r[4 * m4 + 2]), __uint_as_float(r[4 * m4 + 3])),
                          make_float2(c.z, c.w)),
                rr);
            r[4 * m4] = pack_bf16x2(v0.x, v0.y);
            r[4 * m4 + 2] = pack_bf16x2(v1.x, v1.y);
        }
    } else {
        const float *d = dt + 31 - lane;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float2 v = mul_f32x2(
                make_float2(__uint_as_float(r[2 * m]), __uint_as_float(r[2 * m + 1])),
                make_float2(d[2 * m], d[2 * m + 1]));
            r[2 * m] = pack_bf16x2(v.x, v.y);
        }
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

// 4-D map {channel, head, token, batch} with a {64, 1, rows, 1} box, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *p, int X, const SweepArgs &a, int64_t sb, int64_t st,
              int64_t sh, int rows = TC_C, int hdiv = 1, bool f32 = false)
{
    const int esz = f32 ? 4 : 2;
    auto fn = encode_fn();
    if (!fn)
        return false;
    const int64_t lim = (int64_t)1 << 39;
    // a dimension of extent 1 never moves, any legal stride will do
    const int heads = a.H / hdiv;
    if (heads == 1)
        sh = X;
    if (a.B == 1)
        sb = st * (int64_t)a.T;
    if (sh <= 0 || st <= 0 || sb <= 0 || sh >= lim || st >= lim || sb >= lim)
        return false;
    cuuint64_t dims[4] = {(cuuint64_t)X, (cuuint64_t)heads, (cuuint64_t)a.T, (cuuint64_t)a.B};
    cuuint64_t strides[3] = {(cuuint64_t)(sh * esz), (cuuint64_t)(st * esz),
                             (cuuint64_t)(sb * esz)};
    // the inner box is one 128-byte swizzle row: 64 bf16 or 32 fp32 values
    cuuint32_t box[4] = {(cuuint32_t)(128 / esz), 1, (cuuint32_t)rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void *>(p), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Reads (after synchronizing s) and clears this file's device error word.
cudaError_t read_and_clear_error_word(cudaStream_t s, int *err)
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

}  // namespace
}  // namespace la
