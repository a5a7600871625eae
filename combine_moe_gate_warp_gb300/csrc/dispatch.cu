// dispatch.cu -- moe_dispatch: permute-and-pack token hidden states into
// the expert-contiguous send buffer (bf16; the FP8 transports are in
// quant.cu).
//
// "MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7
// (dispatch detail: reorder by target expert, pack each destination into
// one contiguous block).
//
// Design (sm_103a): scatter form -- each token's row is read from HBM
// exactly once and written to each of its (<= k) kept packed rows, so the
// traffic is the algorithmic minimum (x read once, packed written once).
// One block per token; every thread moves a fixed set of 32-byte vectors
// (16-byte where x, packed or the row length is not 32-byte aligned) with
// all loads issued before the stores, giving ~U vectors in flight per
// thread.  Rows are read and written with the evict-first L2 policy: they
// are touched once, and what the next calls reuse stays in L2.
#include <climits>

#include "common.cuh"
#include "tma.cuh"

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

// V: the vector moved per load and store -- uint4 (16 bytes) or u32x8 (32
// bytes, when x, packed and the row length are 32-byte aligned).  nvec
// counts vectors of V per row.
template <typename V>
__device__ __forceinline__ V ld_row_vec(const V *p, uint64_t pol);
template <>
__device__ __forceinline__ uint4 ld_row_vec<uint4>(const uint4 *p, uint64_t pol) { return ld_stream_v4(p, pol); }
template <>
__device__ __forceinline__ u32x8 ld_row_vec<u32x8>(const u32x8 *p, uint64_t pol) { return ld_stream_v8(p, pol); }
__device__ __forceinline__ void st_row_vec(uint4 *p, const uint4 &v, uint64_t pol) { st_stream_v4(p, v, pol); }
__device__ __forceinline__ void st_row_vec(u32x8 *p, const u32x8 &v, uint64_t pol) { st_stream_v8(p, v, pol); }

template <int U, typename V>
__global__ void __launch_bounds__(kDispThreads)
dispatch_bf16_kernel(const V *__restrict__ x, long long T, int nvec, int k,
                     const int32_t *__restrict__ dst_row, int r_max, const int32_t *__restrict__ R_ptr,
                     V *__restrict__ packed, void *ws, int first_wave)
{
    __shared__ int s_rows[MOE_MAX_TOPK];
    __shared__ int s_n;
    // the blocks of the first wave (launched while the layout kernel may
    // still run) ask L2 for their token's row: a hint, safe before the
    // wait; later blocks start after the layout and skip it
    if (threadIdx.x == 0 && blockIdx.x < first_wave && blockIdx.x < T)
        bulk_prefetch_l2(x + blockIdx.x * (long long)nvec, (uint32_t)(nvec * sizeof(V)));
    pdl_wait();
    pdl_launch_dependents();
    const uint64_t pol = l2_stream_policy(true);
    const int rows_valid = min(r_max, __ldg(R_ptr));
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const int n = load_token_rows(dst_row, t, k, rows_valid, s_rows, &s_n, ws);
        const V *src = x + t * nvec;
        for (int c0 = 0; c0 < nvec; c0 += kDispThreads * U) {
            V v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kDispThreads + threadIdx.x;
                if (c < nvec) v[u] = ld_row_vec(src + c, pol);
            }
            for (int j = 0; j < n; ++j) {
                V *dst = packed + (long long)s_rows[j] * nvec;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * kDispThreads + threadIdx.x;
                    if (c < nvec) st_row_vec(dst + c, v[u], pol);
                }
            }
        }
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

#ifndef MOE_DISPATCH_V8
#define MOE_DISPATCH_V8 1
#endif

namespace {

template <typename V>
cudaError_t launch_dispatch_vec(const void *x, int T, int nvec, const moe_layout *L, void *packed, cudaStream_t s)
{
    const int per_thread = (nvec + kDispThreads - 1) / kDispThreads;
    const unsigned grid = (unsigned)grid_for(T);
    const V *xp = static_cast<const V *>(x);
    V *pp = static_cast<V *>(packed);
#define MOE_DISPATCH_BF16(UU)                                                                                     \
    return launch_pdl(dispatch_bf16_kernel<UU, V>, dim3(grid), dim3(kDispThreads), 0, s, xp, (long long)T, nvec, \
                      L->k, (const int32_t *)L->dst_row, L->r_max, (const int32_t *)(L->offsets + L->E), pp,     \
                      L->ws,                                                                                     \
                      resident_grid(reinterpret_cast<const void *>(dispatch_bf16_kernel<UU, V>), kDispThreads, 0))
    if (per_thread <= 1) MOE_DISPATCH_BF16(1);
    else if (per_thread <= 2) MOE_DISPATCH_BF16(2);
    else if (per_thread <= 3) MOE_DISPATCH_BF16(3);
    else if (per_thread <= 4) MOE_DISPATCH_BF16(4);
    else if (per_thread <= 5) MOE_DISPATCH_BF16(5);
    else if (per_thread <= 6) MOE_DISPATCH_BF16(6);
    else MOE_DISPATCH_BF16(8);
#undef MOE_DISPATCH_BF16
}

}  // namespace

cudaError_t launch_dispatch_bf16(const void *x, int T, int H, const moe_layout *L, void *packed,
                                 cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    // 32-byte vectors where x, packed and the rows allow them (the C ABI
    // only requires 16-byte alignment)
    const bool v8 = MOE_DISPATCH_V8 && H % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 32 == 0 &&
                    reinterpret_cast<uintptr_t>(packed) % 32 == 0;
    return v8 ? launch_dispatch_vec<u32x8>(x, T, H / 16, L, packed, s)
              : launch_dispatch_vec<uint4>(x, T, H / 8, L, packed, s);
}

}  // namespace moe
