// la_gqa.cu -- gradients of key/value heads shared by a group of query heads.
//
// With grouped key/value heads (the num_kv_heads axis of ejkernel
// `recurrent`'s key and value) a key or value head feeds G query heads, so
// its gradient is the sum of the G per-query-head gradients (each query head
// has its own decay and state).  The backward sweeps write those per-query-
// head contributions, dense [B, T, H, X], and this kernel sums each group in
// fp32 and writes the result in the token dtype.

#include <cstdint>

#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

template <typename T> __device__ __forceinline__ float ld(const T *p);
template <> __device__ __forceinline__ float ld<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st(T *p, float x);
template <> __device__ __forceinline__ void st<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16 *p, float x)
{
    *p = __float2bfloat16_rn(x);
}

template <typename TI, typename T>
__global__ void __launch_bounds__(256) gqa_reduce_kernel(const TI *in, TokOut out, int T_, int Hkv,
                                                         int G, int X, int64_t total)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % X);
        int64_t r = i / X;
        const int j = (int)(r % Hkv);
        r /= Hkv;
        const int64_t t = r % T_, b = r / T_;
        const TI *src = in + (((b * T_ + t) * Hkv + j) * G) * (int64_t)X + c;
        float acc = 0.f;
        for (int g = 0; g < G; ++g)
            acc += ld(src + (int64_t)g * X);
        st(reinterpret_cast<T *>(out.p) + b * out.sb + t * out.st + (int64_t)j * out.sh + c, acc);
    }
}

// Eight channels per thread with 16-byte loads and stores (bf16, X % 8 == 0,
// 16-byte aligned output rows): one row of the input group is G x X
// contiguous elements.
__global__ void __launch_bounds__(256) gqa_reduce_bf16x8(const __nv_bfloat16 *in, TokOut out,
                                                         int T_, int Hkv, int G, int X,
                                                         int64_t total8)
{
    const int X8 = X / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % X8);
        int64_t r = i / X8;
        const int j = (int)(r % Hkv);
        r /= Hkv;
        const int64_t t = r % T_, b = r / T_;
        const __nv_bfloat16 *src = in + (((b * T_ + t) * Hkv + j) * G) * (int64_t)X + 8 * c8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int g = 0; g < G; ++g) {
            const uint4 u = *reinterpret_cast<const uint4 *>(src + (int64_t)g * X);
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(h2[k]);
                acc[2 * k] += f.x;
                acc[2 * k + 1] += f.y;
            }
        }
        uint4 o;
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o2[k] = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out.p) + b * out.sb +
                                   t * out.st + (int64_t)j * out.sh + 8 * c8) = o;
    }
}

}  // namespace

cudaError_t gqa_reduce(const void *in, const TokOut &out, int B, int T, int Hkv, int G, int X,
                       int bf16, cudaStream_t s, bool in_f32)
{
    const int64_t total = (int64_t)B * T * Hkv * X;
    if (total == 0)
        return cudaSuccess;
    const bool vec = bf16 && !in_f32 && X % 8 == 0 && out.sb % 8 == 0 && out.st % 8 == 0 && out.sh % 8 == 0 &&
                     (reinterpret_cast<uintptr_t>(out.p) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(in) & 15) == 0;
    const int64_t work = vec ? total / 8 : total;
    const int64_t want = (work + 255) / 256;
    const unsigned blocks = (unsigned)(want < 16384 ? want : 16384);   // grid-stride loop
    if (vec)
        gqa_reduce_bf16x8<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(in), out, T,
                                                 Hkv, G, X, work);
    else if (bf16 && in_f32)
        gqa_reduce_kernel<float, __nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const float *>(in), out, T, Hkv, G, X, total);
    else if (bf16)
        gqa_reduce_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(in), out, T, Hkv, G, X, total);
    else
        gqa_reduce_kernel<float, float><<<blocks, 256, 0, s>>>(static_cast<const float *>(in),
                                                               out, T, Hkv, G, X, total);
    note_launch();
    return cudaGetLastError();
}

}  // namespace la
