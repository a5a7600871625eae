// combine.cu -- moe_combine: gather each token's expert outputs through the
// saved routing metadata, gate-weight them, add the shared experts, and
// write the token's output row once.
//
// "MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7
// ("Combine": per token, the weighted sum of its top-k expert outputs, put
// back in original token order using the metadata saved at dispatch, no
// second routing) and sec. 8.2.B (shared experts: every token, no
// all-to-all, outputs added); "DeepSeek MoE sync tax" sec. 2.1 (K_s shared
// experts).
//
// Design (sm_103a): gather form -- y is written exactly once and every
// kept expert-output row is read exactly once (each packed row belongs to
// one assignment), so the traffic is the algorithmic minimum.  One block
// per token; each thread owns U 16-byte column chunks, issues all K*U row
// loads before any arithmetic (K is a template parameter so the slot loop
// unrolls into independent loads), then accumulates in fp32 with explicit
// round-to-nearest FMA/add intrinsics in the pinned order (kept slots
// ascending, then shared experts ascending) and rounds once to bf16.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;

__device__ __forceinline__ void fma8(float (&acc)[8], float g, const uint4 &v)
{
    acc[0] = __fmaf_rn(g, bf16lo(v.x), acc[0]);
    acc[1] = __fmaf_rn(g, bf16hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(g, bf16lo(v.y), acc[2]);
    acc[3] = __fmaf_rn(g, bf16hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(g, bf16lo(v.z), acc[4]);
    acc[5] = __fmaf_rn(g, bf16hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(g, bf16lo(v.w), acc[6]);
    acc[7] = __fmaf_rn(g, bf16hi(v.w), acc[7]);
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v)
{
    acc[0] = __fadd_rn(acc[0], bf16lo(v.x));
    acc[1] = __fadd_rn(acc[1], bf16hi(v.x));
    acc[2] = __fadd_rn(acc[2], bf16lo(v.y));
    acc[3] = __fadd_rn(acc[3], bf16hi(v.y));
    acc[4] = __fadd_rn(acc[4], bf16lo(v.z));
    acc[5] = __fadd_rn(acc[5], bf16hi(v.z));
    acc[6] = __fadd_rn(acc[6], bf16lo(v.w));
    acc[7] = __fadd_rn(acc[7], bf16hi(v.w));
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&h);
}

template <int K, int U>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const uint4 *__restrict__ eo, const float *__restrict__ gates,
               const int32_t *__restrict__ dst_row, int r_max, const int32_t *__restrict__ R_ptr,
               const uint4 *__restrict__ shared, int Ks, long long T, int nvec, uint4 *__restrict__ y,
               void *ws)
{
    // rows at or beyond R (= offsets[E]) are reported and skipped, so an
    // expert-output buffer sized to R is never over-read
    const int rows_valid = min(r_max, __ldg(R_ptr));
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        int rows[K];
        float g[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            rows[j] = __ldg(dst_row + t * K + j);
            g[j] = __ldg(gates + t * K + j);
            if (rows[j] >= rows_valid) {
                if (threadIdx.x == 0) record_status(ws, MOE_ERR_DEVICE_DATA);
                rows[j] = -1;
            }
        }
        for (int c0 = 0; c0 < nvec; c0 += kCombThreads * U) {
            uint4 v[K][U];
#pragma unroll
            for (int j = 0; j < K; ++j) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * kCombThreads + threadIdx.x;
                    if (rows[j] >= 0 && c < nvec) v[j][u] = ld_stream_v4(eo + (long long)rows[j] * nvec + c);
                }
            }
            float acc[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[u][q] = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (rows[j] < 0) continue;
#pragma unroll
                for (int u = 0; u < U; ++u) fma8(acc[u], g[j], v[j][u]);
            }
            for (int sidx = 0; sidx < Ks; ++sidx) {
                const uint4 *sh = shared + ((long long)sidx * T + t) * nvec;
                uint4 sv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * kCombThreads + threadIdx.x;
                    if (c < nvec) sv[u] = ld_stream_v4(sh + c);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) add8(acc[u], sv[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kCombThreads + threadIdx.x;
                if (c < nvec) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                    o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                    o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                    o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                    st_v4(y + t * nvec + c, o);
                }
            }
        }
    }
}

template <int K>
cudaError_t launch_k(const uint4 *eo, const float *gates, const int32_t *dst_row, int r_max,
                     const int32_t *R_ptr, const uint4 *shared, int Ks, int T, int nvec, uint4 *y,
                     void *ws, cudaStream_t s)
{
    const long long cap = 1LL << 30;
    const unsigned grid = (unsigned)(T < cap ? T : cap);
    const int per_thread = (nvec + kCombThreads - 1) / kCombThreads;
    // keep K*U row loads (16 B each) <= 8 per thread: <= 32 data registers
    constexpr int kUMax = (8 / K) < 1 ? 1 : (8 / K);
#define MOE_COMBINE(UU) \
    combine_kernel<K, UU><<<grid, kCombThreads, 0, s>>>(eo, gates, dst_row, r_max, R_ptr, shared, Ks, T, \
                                                        nvec, y, ws)
    if (per_thread <= 1 || kUMax == 1) {
        MOE_COMBINE(1);
    } else if (per_thread <= 2 || kUMax == 2) {
        if constexpr (kUMax >= 2) MOE_COMBINE(2);
    } else if (per_thread <= 4 || kUMax == 4) {
        if constexpr (kUMax >= 4) MOE_COMBINE(4);
    } else {
        if constexpr (kUMax >= 8) MOE_COMBINE(8);
    }
#undef MOE_COMBINE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const void *eo, const moe_layout *L, const float *gates, const void *shared,
                           int Ks, int T, int H, void *y, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const uint4 *ep = static_cast<const uint4 *>(eo);
    const uint4 *sp = static_cast<const uint4 *>(shared);
    uint4 *yp = static_cast<uint4 *>(y);
    const int nvec = H / 8;
    switch (L->k) {
#define MOE_COMBINE_CASE(KK) \
    case KK:                                                                                       \
        return launch_k<KK>(ep, gates, L->dst_row, L->r_max, L->offsets + L->E, sp, Ks, T, nvec, yp, \
                            L->ws, s);
        MOE_COMBINE_CASE(1) MOE_COMBINE_CASE(2) MOE_COMBINE_CASE(3) MOE_COMBINE_CASE(4)
        MOE_COMBINE_CASE(5) MOE_COMBINE_CASE(6) MOE_COMBINE_CASE(7) MOE_COMBINE_CASE(8)
        MOE_COMBINE_CASE(9) MOE_COMBINE_CASE(10) MOE_COMBINE_CASE(11) MOE_COMBINE_CASE(12)
        MOE_COMBINE_CASE(13) MOE_COMBINE_CASE(14) MOE_COMBINE_CASE(15) MOE_COMBINE_CASE(16)
#undef MOE_COMBINE_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
