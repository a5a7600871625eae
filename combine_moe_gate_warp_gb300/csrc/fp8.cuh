// fp8.cuh -- pieces of the affine e4m3 transport shared by the dispatch and
// quantiser kernels: order-preserving keys for row extremes, the pinned fp32
// encode of a bf16 pair, and the decode of 16 codes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "tma.cuh"

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

// The quotient q = RN((v - zero) / scale) decides the code, and the code
// must be the one the correctly rounded quotient gives.  Division is the
// costliest step of the encode, so the quotients are formed as
// q = RN(d * RN(1/scale)), which is within 4 fp32 ulp (relative 2^-21) of
// RN(d / scale): two roundings of at most half an ulp each.  The codes of
// q * (1 - 2^-20) and q * (1 + 2^-20) bracket the code of RN(d / scale),
// because the e4m3 conversion is monotone; where the two agree, that is the
// code, and only where they differ (q next to an e4m3 rounding boundary) is
// the correctly rounded __fdiv_rn taken.  This is Ziv's rounding test
// ("Fast evaluation of elementary mathematical functions with correctly
// rounded last bit", ACM TOMS 17(3), 1991): an approximation plus an exact
// fallback when the rounding is in doubt.  The arithmetic runs on packed
// fp32 pairs (__fadd2_rn / __fmul2_rn), the test over 8 values at once,
// and the fallback recomputes all 8 (a branch too long to be if-converted:
// free when no lane needs it).  rcp = 0 forces the fallback.  The inputs
// are read from shared memory, and the fallback reads them again instead of
// keeping them: held across the conversions for a branch that is rarely
// taken (~1.5 % of 8-value groups of N(0,1) rows, where a quotient lands
// exactly on an e4m3 rounding midpoint), they cost the encode kernel 15
// registers and ~2.7 instructions per element.

// 1 / scale for the fast quotient, or 0 (always fall back) where the
// reciprocal would leave the normal range.
__device__ __forceinline__ float e4m3_rcp(float scale)
{
    return scale >= 1e-30f ? __frcp_rn(scale) : 0.0f;
}

// 8 bf16 (one 16-byte vector in shared memory, unchanged during the call)
// -> 8 codes (two words), code i from element i (low bytes first).
__device__ __forceinline__ uint2 quant8(const unsigned char *src, float zero, float scale, float rcp)
{
    const uint4 a = lds_v4(src);
    const unsigned w[4] = {a.x, a.y, a.z, a.w};
    const float2 nz = make_float2(-zero, -zero), r2 = make_float2(rcp, rcp);
    const float2 dn = make_float2(1.0f - 0x1p-20f, 1.0f - 0x1p-20f), up = make_float2(1.0f + 0x1p-20f, 1.0f + 0x1p-20f);
    unsigned lo[2], hi[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 q0 = __fmul2_rn(__fadd2_rn(make_float2(bf16lo(w[2 * i]), bf16hi(w[2 * i])), nz), r2);
        const float2 q1 = __fmul2_rn(__fadd2_rn(make_float2(bf16lo(w[2 * i + 1]), bf16hi(w[2 * i + 1])), nz), r2);
        const float2 l0 = __fmul2_rn(q0, dn), h0 = __fmul2_rn(q0, up);
        const float2 l1 = __fmul2_rn(q1, dn), h1 = __fmul2_rn(q1, up);
        lo[i] = (unsigned)e4m3x2(l0.x, l0.y) | ((unsigned)e4m3x2(l1.x, l1.y) << 16);
        hi[i] = (unsigned)e4m3x2(h0.x, h0.y) | ((unsigned)e4m3x2(h1.x, h1.y) << 16);
    }
    if (__builtin_expect((lo[0] != hi[0]) | (lo[1] != hi[1]) | (rcp == 0.0f), 0)) {
        const uint4 b = lds_v4(src);  // read again (a volatile load: not forwarded from `a`)
        const unsigned v[4] = {b.x, b.y, b.z, b.w};
        float q[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[2 * i] = __fdiv_rn(__fsub_rn(bf16lo(v[i]), zero), scale);
            q[2 * i + 1] = __fdiv_rn(__fsub_rn(bf16hi(v[i]), zero), scale);
        }
        lo[0] = (unsigned)e4m3x2(q[0], q[1]) | ((unsigned)e4m3x2(q[2], q[3]) << 16);
        lo[1] = (unsigned)e4m3x2(q[4], q[5]) | ((unsigned)e4m3x2(q[6], q[7]) << 16);
    }
    return make_uint2(lo[0], lo[1]);
}

// 16 bf16 (32 bytes in shared memory) -> 16 codes (one 16-byte vector).
__device__ __forceinline__ uint4 quant16(const unsigned char *src, float zero, float scale, float rcp)
{
    const uint2 l = quant8(src, zero, scale, rcp), h = quant8(src + 16, zero, scale, rcp);
    return make_uint4(l.x, l.y, h.x, h.y);
}

// Running max and min of bf16 pairs (packed, two lanes per word).  Signed
// zeros are not ordered here; a caller whose extreme comes out as zero
// recomputes it with the ordered keys below.
__device__ __forceinline__ void hminmax8(const uint4 &a, __nv_bfloat162 &mx, __nv_bfloat162 &mn)
{
    const unsigned w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
        mx = __hmax2(mx, v);
        mn = __hmin2(mn, v);
    }
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
