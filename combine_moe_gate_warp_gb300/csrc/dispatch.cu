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
// One block per token; every thread moves a fixed set of 16-byte chunks
// with all loads issued before the stores, giving ~U*16 bytes in flight
// per thread.
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

template <int U>
__global__ void __launch_bounds__(kDispThreads)
dispatch_bf16_kernel(const uint4 *__restrict__ x, long long T, int nvec, int k,
                     const int32_t *__restrict__ dst_row, int r_max, const int32_t *__restrict__ R_ptr,
                     uint4 *__restrict__ packed, void *ws, int first_wave)
{
    __shared__ int s_rows[MOE_MAX_TOPK];
    __shared__ int s_n;
    // the blocks of the first wave (launched while the layout kernel may
    // still run) ask L2 for their token's row: a hint, safe before the
    // wait; later blocks start after the layout and skip it
    if (threadIdx.x == 0 && blockIdx.x < first_wave && blockIdx.x < T)
        bulk_prefetch_l2(x + blockIdx.x * (long long)nvec, (uint32_t)nvec * 16u);
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
#define MOE_DISPATCH_BF16(UU)                                                                                  \
    return launch_pdl(dispatch_bf16_kernel<UU>, dim3(grid), dim3(kDispThreads), 0, s, xp, (long long)T, nvec, \
                      L->k, (const int32_t *)L->dst_row, L->r_max, (const int32_t *)(L->offsets + L->E), pp,  \
                      L->ws, resident_grid(reinterpret_cast<const void *>(dispatch_bf16_kernel<UU>), kDispThreads, 0))
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

}  // namespace moe
