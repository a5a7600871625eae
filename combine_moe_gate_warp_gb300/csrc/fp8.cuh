// fp8.cuh -- pieces of the affine e4m3 transport shared by the dispatch and
// quantiser kernels: order-preserving keys for row extremes, the pinned fp32
// encode of a bf16 pair, and the decode of 16 codes.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// fp32 bit pattern -> int key with numeric order and -0 < +0.
__device__ __forceinline__ int f32_order_key(unsigned b)
{
    return (b & 0x80000000u) ? (int)(b ^ 0x7FFFFFFFu) : (int)b;
}
__device__ __forceinline__ float key_to_f32(int key)
{
    unsigned b = (unsigned)key;
    return __uint_as_float(key < 0 ? (b ^ 0x7FFFFFFFu) : b);
}

// Keys as unsigned words for atomicMax from zero: the max key is stored as
// key ^ 0x80000000 (monotone), the min key as its complement, so a zeroed
// word is the identity of both reductions.
__device__ __forceinline__ unsigned max_word(int key) { return (unsigned)key ^ 0x80000000u; }
__device__ __forceinline__ unsigned min_word(int key) { return ~((unsigned)key ^ 0x80000000u); }
__device__ __forceinline__ int key_of_max_word(unsigned w) { return (int)(w ^ 0x80000000u); }
__device__ __forceinline__ int key_of_min_word(unsigned w) { return (int)(~w ^ 0x80000000u); }

__device__ __forceinline__ unsigned short e4m3x2(float lo, float hi)
{
    return (unsigned short)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Quantise one bf16 pair word into two codes (low code = low element).
__device__ __forceinline__ unsigned quant_pair(unsigned w, float zero, float scale)
{
    const float a = __fdiv_rn(__fsub_rn(bf16lo(w), zero), scale);
    const float b = __fdiv_rn(__fsub_rn(bf16hi(w), zero), scale);
    return (unsigned)e4m3x2(a, b);
}

// 16 bf16 (two 16-byte vectors) -> 16 codes (one 16-byte vector).
__device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float zero, float scale)
{
    uint4 c;
    c.x = quant_pair(a.x, zero, scale) | (quant_pair(a.y, zero, scale) << 16);
    c.y = quant_pair(a.z, zero, scale) | (quant_pair(a.w, zero, scale) << 16);
    c.z = quant_pair(b.x, zero, scale) | (quant_pair(b.y, zero, scale) << 16);
    c.w = quant_pair(b.z, zero, scale) | (quant_pair(b.w, zero, scale) << 16);
    return c;
}

// Max and min keys of the 16 bf16 values of two 16-byte vectors.
__device__ __forceinline__ void minmax16(const uint4 &a, const uint4 &b, int &kmax, int &kmin)
{
    const unsigned w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int klo = f32_order_key(w[q] << 16);
        const int khi = f32_order_key(w[q] & 0xFFFF0000u);
        kmax = max(kmax, max(klo, khi));
        kmin = min(kmin, min(klo, khi));
    }
}
__device__ __forceinline__ void minmax8(const uint4 &a, int &kmax, int &kmin)
{
    const unsigned w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int klo = f32_order_key(w[q] << 16);
        const int khi = f32_order_key(w[q] & 0xFFFF0000u);
        kmax = max(kmax, max(klo, khi));
        kmin = min(kmin, min(klo, khi));
    }
}

// The affine pair of a row or group from its extreme keys: zero = (max +
// min) * 0.5, scale = (max - min) / 896, scale 0 for a constant group.
__device__ __forceinline__ float2 affine_pair(int kmax, int kmin)
{
    const float mx = key_to_f32(kmax), mn = key_to_f32(kmin);
    const float zero = __fmul_rn(__fadd_rn(mx, mn), 0.5f);
    const float scale = (mx == mn) ? 0.0f : __fdiv_rn(__fsub_rn(mx, mn), 896.0f);
    return make_float2(scale, zero);
}

// Two e4m3 codes (low byte = low element) -> their exact fp32 values.
__device__ __forceinline__ float2 e4m3x2_to_float2(unsigned short c)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c, __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

}  // namespace moe
