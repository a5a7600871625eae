// dispatch.cu -- moe_dispatch: permute-and-pack token hidden states into
// the expert-contiguous send buffer, in bf16 or per-token affine FP8.
//
// "MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7
// (dispatch detail: reorder by target expert, pack each destination into
// one contiguous block); "Deepseek-MoE sync-tax ... guide" sec. 3.1 (FP8
// for transport: per token, min/max of its vector, affine map onto FP8).
//
// Design (sm_103a): scatter form -- each token's row is read from HBM
// exactly once and written to each of its (<= k) kept packed rows, so the
// traffic is the algorithmic minimum (x read once, packed written once).
// One block per token; every thread moves a fixed set of 16-byte chunks
// with all loads issued before the stores, giving ~U*16 bytes in flight
// per thread.  The FP8 variant keeps the row in registers, reduces the
// row's max/min (order-independent integer keys, -0 < +0) with warp
// shuffles and a 4-entry shared array, then quantises with the fixed fp32
// operation order (IEEE round-to-nearest intrinsics, no contraction) and
// the hardware e4m3 satfinite conversion, and writes 16 codes per store.
#include <climits>

#include "common.cuh"
#include "fp8.cuh"

namespace moe {
namespace {

constexpr int kDispThreads = 128;

// Kept destination rows of token t, compacted in slot order into s_rows.
// Rows at or beyond R (= offsets[E], the rows the layout produced) are
// reported and skipped, so packed buffers sized to R are never overrun.
__device__ __forceinline__ int load_token_rows(const int32_t *__restrict__ dst_row, long long t, int k,
                                               int rows_valid, int *s_rows, int *s_n, void *ws)
{
    if (threadIdx.x < 32) {
        int r = -1;
        if ((int)threadIdx.x < k) {
            r = dst_row[t * k + threadIdx.x];
            if (r >= rows_valid) {
                record_status(ws, MOE_ERR_DEVICE_DATA);
                r = -1;
            }
        }
        const unsigned kept = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) s_rows[__popc(kept & ((1u << threadIdx.x) - 1u))] = r;
        if (threadIdx.x == 0) *s_n = __popc(kept);
    }
    __syncthreads();
    return *s_n;
}

template <int U>
__global__ void __launch_bounds__(kDispThreads)
dispatch_bf16_kernel(const uint4 *__restrict__ x, long long T, int nvec, int k,
                     const int32_t *__restrict__ dst_row, int r_max, const int32_t *__restrict__ R_ptr,
                     uint4 *__restrict__ packed, void *ws)
{
    __shared__ int s_rows[MOE_MAX_TOPK];
    __shared__ int s_n;
    pdl_wait();
    pdl_launch_dependents();
    const int rows_valid = min(r_max, __ldg(R_ptr));
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const int n = load_token_rows(dst_row, t, k, rows_valid, s_rows, &s_n, ws);
        const uint4 *src = x + t * nvec;
        for (int c0 = 0; c0 < nvec; c0 += kDispThreads * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kDispThreads + threadIdx.x;
                if (c < nvec) v[u] = ld_stream_v4(src + c);
            }
            for (int j = 0; j < n; ++j) {
                uint4 *dst = packed + (long long)s_rows[j] * nvec;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * kDispThreads + threadIdx.x;
                    if (c < nvec) st_v4(dst + c, v[u]);
                }
            }
        }
        __syncthreads();
    }
}

// One block per token.  Thread c handles chunk pairs p = c + i*128 (a pair
// = 16 bf16 = 32 bytes in, 16 codes = 16 bytes out).
template <int CPT>
__global__ void __launch_bounds__(kDispThreads)
dispatch_fp8_kernel(const uint4 *__restrict__ x, long long T, int npairs, int k,
                    const int32_t *__restrict__ dst_row, int r_max, const int32_t *__restrict__ R_ptr,
                    uint4 *__restrict__ packed, float2 *__restrict__ scales, void *ws)
{
    __shared__ int s_rows[MOE_MAX_TOPK];
    __shared__ int s_n;
    __shared__ int s_max[kDispThreads / 32], s_min[kDispThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();
    pdl_launch_dependents();
    const int rows_valid = min(r_max, __ldg(R_ptr));
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const int n = load_token_rows(dst_row, t, k, rows_valid, s_rows, &s_n, ws);
        const uint4 *src = x + t * (2LL * npairs);
        uint4 v[CPT][2];
        int kmax = INT_MIN, kmin = INT_MAX;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int p = i * kDispThreads + threadIdx.x;
            if (p < npairs) {
                v[i][0] = ld_stream_v4(src + 2 * p);
                v[i][1] = ld_stream_v4(src + 2 * p + 1);
            }
        }
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int p = i * kDispThreads + threadIdx.x;
            if (p < npairs) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const unsigned w[4] = {v[i][h].x, v[i][h].y, v[i][h].z, v[i][h].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int klo = f32_order_key(w[q] << 16);
                        const int khi = f32_order_key(w[q] & 0xFFFF0000u);
                        kmax = max(kmax, max(klo, khi));
                        kmin = min(kmin, min(klo, khi));
                    }
                }
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, d));
            kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, d));
        }
        if (lane == 0) {
            s_max[warp] = kmax;
            s_min[warp] = kmin;
        }
        __syncthreads();
        kmax = s_max[0];
        kmin = s_min[0];
#pragma unroll
        for (int w = 1; w < kDispThreads / 32; ++w) {
            kmax = max(kmax, s_max[w]);
            kmin = min(kmin, s_min[w]);
        }
        const float mx = key_to_f32(kmax), mn = key_to_f32(kmin);
        const float zero = __fmul_rn(__fadd_rn(mx, mn), 0.5f);
        const bool flat = (mx == mn);
        const float scale = flat ? 0.0f : __fdiv_rn(__fsub_rn(mx, mn), 896.0f);

#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int p = i * kDispThreads + threadIdx.x;
            if (p < npairs) {
                uint4 codes = make_uint4(0u, 0u, 0u, 0u);
                if (!flat) {
                    const uint4 a = v[i][0], b = v[i][1];
                    codes.x = quant_pair(a.x, zero, scale) | (quant_pair(a.y, zero, scale) << 16);
                    codes.y = quant_pair(a.z, zero, scale) | (quant_pair(a.w, zero, scale) << 16);
                    codes.z = quant_pair(b.x, zero, scale) | (quant_pair(b.y, zero, scale) << 16);
                    codes.w = quant_pair(b.z, zero, scale) | (quant_pair(b.w, zero, scale) << 16);
                }
                for (int j = 0; j < n; ++j) st_v4(packed + (long long)s_rows[j] * npairs + p, codes);
            }
        }
        if (threadIdx.x < n) scales[s_rows[threadIdx.x]] = make_float2(scale, zero);
        __syncthreads();
    }
}

long long grid_for(long long T)
{
    // One block per token; the grid-stride loop covers T beyond 2^31-1.
    const long long cap = 1LL << 30;
    return T < 1 ? 1 : (T < cap ? T : cap);
}

}  // namespace

cudaError_t launch_dispatch_bf16(const void *x, int T, int H, const moe_layout *L, void *packed,
                                 cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const int nvec = H / 8;
    const int per_thread = (nvec + kDispThreads - 1) / kDispThreads;
    const unsigned grid = (unsigned)grid_for(T);
    const uint4 *xp = static_cast<const uint4 *>(x);
    uint4 *pp = static_cast<uint4 *>(packed);
#define MOE_DISPATCH_BF16(UU)                                                                     \
    return launch_pdl(dispatch_bf16_kernel<UU>, dim3(grid), dim3(kDispThreads), 0, s, xp, (long long)T, nvec, \
                      L->k, (const int32_t *)L->dst_row, L->r_max, (const int32_t *)(L->offsets + L->E), pp,  \
                      L->ws)
    if (per_thread <= 1) MOE_DISPATCH_BF16(1);
    else if (per_thread <= 2) MOE_DISPATCH_BF16(2);
    else if (per_thread <= 3) MOE_DISPATCH_BF16(3);
    else if (per_thread <= 4) MOE_DISPATCH_BF16(4);
    else if (per_thread <= 5) MOE_DISPATCH_BF16(5);
    else if (per_thread <= 6) MOE_DISPATCH_BF16(6);
    else MOE_DISPATCH_BF16(8);
#undef MOE_DISPATCH_BF16
    return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const void *x, int T, int H, const moe_layout *L, void *packed,
                                float *scales, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const int npairs = H / 16;
    const int per_thread = (npairs + kDispThreads - 1) / kDispThreads;
    const unsigned grid = (unsigned)grid_for(T);
    const uint4 *xp = static_cast<const uint4 *>(x);
    uint4 *pp = static_cast<uint4 *>(packed);
    float2 *sp = reinterpret_cast<float2 *>(scales);
#define MOE_DISPATCH_FP8(CC)                                                                      \
    return launch_pdl(dispatch_fp8_kernel<CC>, dim3(grid), dim3(kDispThreads), 0, s, xp, (long long)T, npairs, \
                      L->k, (const int32_t *)L->dst_row, L->r_max, (const int32_t *)(L->offsets + L->E), pp,   \
                      sp, L->ws)
    if (per_thread <= 1) MOE_DISPATCH_FP8(1);
    else if (per_thread <= 2) MOE_DISPATCH_FP8(2);
    else if (per_thread <= 4) MOE_DISPATCH_FP8(4);
    else if (per_thread <= 8) MOE_DISPATCH_FP8(8);
    else return cudaErrorInvalidValue;
#undef MOE_DISPATCH_FP8
    return cudaGetLastError();
}

}  // namespace moe
