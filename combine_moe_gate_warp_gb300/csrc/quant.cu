// quant.cu -- the grouped FP8 quantiser modes and the FP8 combine.
//
// "Deepseek-MoE sync-tax essence and four-layer optimisation guide" sec. 3.1
// (per token, the min and max of each token's expert-output vector and an
// affine map onto FP8) and sec. 5.2 (the quantiser offers per-token,
// per-expert and global modes).  The affine pair of a group is the per-token
// formula over every element of the group's rows: zero = (max + min) * 0.5,
// scale = (max - min) / 896, code = e4m3 satfinite RNE((v - zero) / scale);
// scale 0 and all-zero codes for a constant group.
//
//   per-token   a packed row is its own group (the dispatch's existing path
//               for x; here for expert-output rows)
//   per-expert  the rows sent to one expert (contiguous in the packed layout)
//   global      every transported row
//
// Design (sm_103a): a group's extremes need every row of the group before
// the first code, so the grouped modes take two passes over the source:
//   1. fp8_group_stats_kernel: persistent warps, one row per warp (16-byte
//      streaming loads, order-preserving integer keys), extremes kept per
//      group in shared memory (shared atomicMax on monotone key words) and
//      merged into the workspace with one global atomicMax per (block,
//      group): the global mode does not serialise on one address.
//   2. fp8_group_encode_kernel: one block per source row; every block turns
//      the workspace keys into the groups' (scale, zero) in shared memory
//      first, then encodes its row with the pinned fp32 operations and the
//      hardware e4m3x2 satfinite conversion; a completion ticket lets the
//      last block reset the keys, so the workspace stays zeroed.
// The dispatch side reads token rows of x and writes each kept copy (a
// token sent to two experts is encoded once per expert in the per-expert
// mode, once in total in the global mode); the expert side reads packed
// expert-output rows and writes the same rows.
//
// FP8 combine: per token y = bf16 RNE of, in fp32 and this order,
//   acc = 0; acc = fmaf(g_j, fmaf(scale_r, e4m3(code), zero_r), acc) over kept
//   slots ascending; acc = acc + shared_s over shared experts ascending.
// One warp per token (persistent warps): a lane owns 16-column groups (one
// 16-byte vector of codes per row, two of bf16 per shared expert), issues
// the loads of all kept rows before any arithmetic, decodes codes pairwise
// through the exact e4m3 -> f16 conversion and writes 32 bytes of y.
#include <climits>

#include <cuda_bf16.h>

#include "common.cuh"
#include "fp8.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 256;
constexpr int kEncThreads = 128;

// Expert of packed row `row` from the layout offsets held in shared memory:
// the largest e with off[e] <= row (experts without rows are skipped).
__device__ __forceinline__ int expert_of_row(const int *s_off, int E, int row)
{
    int lo = 0, hi = E;  // off[lo] <= row < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= row) lo = mid;
        else hi = mid;
    }
    return lo;
}

// TOKENS: source rows are the T token rows of x; a token's groups are those
// of its kept rows.  Otherwise source rows are the packed rows r < R.
template <int MODE, bool TOKENS>
__global__ void __launch_bounds__(kStatThreads)
fp8_group_stats_kernel(const uint4 *__restrict__ src, long long n_src, int nvec, int k,
                       const int32_t *__restrict__ dst_row, const int32_t *__restrict__ offsets, int E, int r_max,
                       void *ws)
{
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ unsigned s_max[MOE_MAX_EXPERTS], s_min[MOE_MAX_EXPERTS];
    constexpr int kWarps = kStatThreads / 32;
    const int ngroups = MODE == MOE_FP8_GLOBAL ? 1 : E;
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i <= E; i += kStatThreads) s_off[i] = __ldg(offsets + i);
    for (int i = threadIdx.x; i < ngroups; i += kStatThreads) s_max[i] = s_min[i] = 0u;
    __syncthreads();
    const int rows_valid = min(r_max, s_off[E]);
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * kWarps;
    for (long long i = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); i < n_src; i += nwarps) {
        if (!TOKENS && i >= rows_valid) break;
        // the row's groups: kept slot rows of a token, or the row itself
        int grow = -1;  // lane j < k: row of slot j (tokens); lane 0: the row
        if (TOKENS) {
            if (lane < k) {
                grow = __ldg(dst_row + i * k + lane);
                if (grow >= rows_valid) grow = -1;  // reported by the encode pass
            }
        } else if (lane == 0) {
            grow = (int)i;
        }
        const unsigned kept = __ballot_sync(0xffffffffu, grow >= 0);
        if (kept == 0u) continue;  // nothing of this token is transported
        const uint4 *row = src + i * nvec;
        int kmax = INT_MIN, kmin = INT_MAX;
        for (int c = lane; c < nvec; c += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c + 32 * u < nvec) v[u] = ld_stream_v4(row + c + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c + 32 * u < nvec) minmax8(v[u], kmax, kmin);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, d));
            kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, d));
        }
        if (grow >= 0) {
            const int g = MODE == MOE_FP8_GLOBAL ? 0 : expert_of_row(s_off, E, grow);
            atomicMax(&s_max[g], max_word(kmax));
            atomicMax(&s_min[g], min_word(kmin));
        }
    }
    __syncthreads();
    WsHeader *h = static_cast<WsHeader *>(ws);
    for (int g = threadIdx.x; g < ngroups; g += kStatThreads) {
        if (s_max[g] != 0u) {
            atomicMax(&h->quant_max[g], s_max[g]);
            atomicMax(&h->quant_min[g], s_min[g]);
        }
    }
}

// One block per source row.  Thread c handles 16-column groups c, c+128, ...
// (CPT of them: 32 bytes of bf16 in, 16 codes out each).
template <int CPT, int MODE, bool TOKENS>
__global__ void __launch_bounds__(kEncThreads)
fp8_group_encode_kernel(const uint4 *__restrict__ src, long long n_src, int npairs, int k,
                        const int32_t *__restrict__ dst_row, const int32_t *__restrict__ offsets, int E, int r_max,
                        uint4 *__restrict__ packed, float2 *__restrict__ scales, void *ws)
{
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ float2 s_par[MOE_MAX_EXPERTS];
    __shared__ int s_rows[MOE_MAX_TOPK];
    __shared__ int s_grp[MOE_MAX_TOPK];
    __shared__ int s_n;
    __shared__ int s_wmax[kEncThreads / 32], s_wmin[kEncThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ngroups = MODE == MOE_FP8_GLOBAL ? 1 : (MODE == MOE_FP8_PER_EXPERT ? E : 0);
    WsHeader *h = static_cast<WsHeader *>(ws);
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i <= E; i += kEncThreads) s_off[i] = __ldg(offsets + i);
    for (int g = threadIdx.x; g < ngroups; g += kEncThreads) {
        const unsigned wmx = *((volatile unsigned *)&h->quant_max[g]);
        const unsigned wmn = *((volatile unsigned *)&h->quant_min[g]);
        s_par[g] = wmx == 0u ? make_float2(0.0f, 0.0f) : affine_pair(key_of_max_word(wmx), key_of_min_word(wmn));
    }
    __syncthreads();
    const int rows_valid = min(r_max, s_off[E]);
    for (long long i = blockIdx.x; i < n_src; i += gridDim.x) {
        // destination rows of this source row, compacted in slot order
        if (threadIdx.x < 32) {
            int r = -1;
            if (TOKENS) {
                if ((int)threadIdx.x < k) {
                    r = __ldg(dst_row + i * k + threadIdx.x);
                    if (r >= rows_valid) {
                        record_status(ws, MOE_ERR_DEVICE_DATA);
                        r = -1;
                    }
                }
            } else if (threadIdx.x == 0 && i < rows_valid) {
                r = (int)i;
            }
            const unsigned kept = __ballot_sync(0xffffffffu, r >= 0);
            if (r >= 0) {
                const int pos = __popc(kept & ((1u << threadIdx.x) - 1u));
                s_rows[pos] = r;
                s_grp[pos] = MODE == MOE_FP8_PER_EXPERT ? expert_of_row(s_off, E, r) : 0;
            }
            if (threadIdx.x == 0) s_n = __popc(kept);
        }
        __syncthreads();
        const int n = s_n;
        if (n > 0) {
            const uint4 *row = src + i * (2LL * npairs);
            uint4 v[CPT][2];
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
                const int p = u * kEncThreads + threadIdx.x;
                if (p < npairs) {
                    v[u][0] = ld_stream_v4(row + 2 * p);
                    v[u][1] = ld_stream_v4(row + 2 * p + 1);
                }
            }
            if (MODE == MOE_FP8_PER_TOKEN) {
                // the row is its own group: block-wide extremes first
                int kmax = INT_MIN, kmin = INT_MAX;
#pragma unroll
                for (int u = 0; u < CPT; ++u)
                    if (u * kEncThreads + (int)threadIdx.x < npairs) minmax16(v[u][0], v[u][1], kmax, kmin);
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, d));
                    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, d));
                }
                if (lane == 0) {
                    s_wmax[warp] = kmax;
                    s_wmin[warp] = kmin;
                }
                __syncthreads();
                if (threadIdx.x == 0) {
                    int a = s_wmax[0], b = s_wmin[0];
                    for (int w = 1; w < kEncThreads / 32; ++w) {
                        a = max(a, s_wmax[w]);
                        b = min(b, s_wmin[w]);
                    }
                    s_par[0] = affine_pair(a, b);
                }
                __syncthreads();
            }
            // rows of one group share their codes: encode once per run of
            // equal groups (slot order), store to every row of the run
            for (int j0 = 0; j0 < n;) {
                const int g = s_grp[j0];
                int j1 = j0 + 1;
                while (j1 < n && s_grp[j1] == g) ++j1;
                const float2 par = s_par[g];
#pragma unroll
                for (int u = 0; u < CPT; ++u) {
                    const int p = u * kEncThreads + threadIdx.x;
                    if (p < npairs) {
                        const uint4 c = par.x == 0.0f ? make_uint4(0u, 0u, 0u, 0u)
                                                      : quant16(v[u][0], v[u][1], par.y, par.x);
                        for (int j = j0; j < j1; ++j) st_v4(packed + (long long)s_rows[j] * npairs + p, c);
                    }
                }
                if ((int)threadIdx.x >= j0 && (int)threadIdx.x < j1) scales[s_rows[threadIdx.x]] = par;
                j0 = j1;
            }
        }
        __syncthreads();  // s_rows / s_par[0] are rewritten for the next row
    }
    if (MODE != MOE_FP8_PER_TOKEN) {
        // the last block to finish resets the group keys (every block read
        // them at its start, before its ticket)
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned done = atomicAdd(&h->quant_ticket, 1u);
            s_n = (done == gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (s_n) {
            for (int g = threadIdx.x; g < ngroups; g += kEncThreads) {
                h->quant_max[g] = 0u;
                h->quant_min[g] = 0u;
            }
            if (threadIdx.x == 0) h->quant_ticket = 0u;
        }
    }
}

// ---- FP8 combine -----------------------------------------------------------
constexpr int kCombFp8Threads = 256;

__device__ __forceinline__ void fma16_fp8(float (&acc)[16], float g, float scale, float zero, const uint4 &c)
{
    const unsigned w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 lo = e4m3x2_to_float2((unsigned short)(w[q] & 0xFFFFu));
        const float2 hi = e4m3x2_to_float2((unsigned short)(w[q] >> 16));
        acc[4 * q + 0] = __fmaf_rn(g, __fmaf_rn(scale, lo.x, zero), acc[4 * q + 0]);
        acc[4 * q + 1] = __fmaf_rn(g, __fmaf_rn(scale, lo.y, zero), acc[4 * q + 1]);
        acc[4 * q + 2] = __fmaf_rn(g, __fmaf_rn(scale, hi.x, zero), acc[4 * q + 2]);
        acc[4 * q + 3] = __fmaf_rn(g, __fmaf_rn(scale, hi.y, zero), acc[4 * q + 3]);
    }
}

__device__ __forceinline__ void add8_bf16(float *acc, const uint4 &v)
{
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __fadd_rn(acc[2 * q], bf16lo(w[q]));
        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf16hi(w[q]));
    }
}

__device__ __forceinline__ unsigned pack2_bf16(float lo, float hi)
{
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&b);
}

template <int K, int V>
__global__ void __launch_bounds__(kCombFp8Threads)
combine_fp8_kernel(const uint4 *__restrict__ codes, const float2 *__restrict__ scales,
                   const float *__restrict__ gates, const int32_t *__restrict__ dst_row, int r_max,
                   const int32_t *__restrict__ R_ptr, const uint4 *__restrict__ shared, int Ks, long long T,
                   int n16, uint4 *__restrict__ y, void *ws)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (kCombFp8Threads / 32);
    const int rows_valid = min(r_max, __ldg(R_ptr));
    for (long long t = (long long)blockIdx.x * (kCombFp8Threads / 32) + (threadIdx.x >> 5); t < T; t += nwarps) {
        int rl = -1;
        float gl = 0.0f;
        float2 pl = make_float2(0.0f, 0.0f);
        if (lane < K) {
            rl = __ldg(dst_row + t * K + lane);
            if (rl >= rows_valid) {
                record_status(ws, MOE_ERR_DEVICE_DATA);
                rl = -1;
            }
            gl = __ldg(gates + t * K + lane);
            if (rl >= 0) pl = __ldg(scales + rl);
        }
        // kept slots, compacted in slot order
        const unsigned kept = __ballot_sync(0xffffffffu, rl >= 0);
        const int n = __popc(kept);
        int row[K];
        float g[K], sc[K], zr[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            // lane holding the j-th kept slot
            unsigned m = kept;
            for (int q = 0; q < j && m; ++q) m &= m - 1u;
            const int src = m ? __ffs(m) - 1 : 0;
            row[j] = __shfl_sync(0xffffffffu, rl, src);
            g[j] = __shfl_sync(0xffffffffu, gl, src);
            sc[j] = __shfl_sync(0xffffffffu, pl.x, src);
            zr[j] = __shfl_sync(0xffffffffu, pl.y, src);
        }
        for (int c0 = lane; c0 < n16; c0 += 32 * V) {
            uint4 cv[K][V];
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (j < n) {
                    const uint4 *src = codes + (long long)row[j] * n16;
#pragma unroll
                    for (int u = 0; u < V; ++u)
                        if (c0 + 32 * u < n16) cv[j][u] = ld_stream_v4(src + c0 + 32 * u);
                }
            }
#pragma unroll
            for (int u = 0; u < V; ++u) {
                const int c = c0 + 32 * u;
                if (c >= n16) break;
                float acc[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (j < n) fma16_fp8(acc, g[j], sc[j], zr[j], cv[j][u]);
                for (int s = 0; s < Ks; ++s) {
                    const uint4 *sh = shared + ((long long)s * T + t) * (2LL * n16) + 2 * c;
                    const uint4 a = ld_stream_v4(sh), b = ld_stream_v4(sh + 1);
                    add8_bf16(acc, a);
                    add8_bf16(acc + 8, b);
                }
                uint4 o0, o1;
                o0.x = pack2_bf16(acc[0], acc[1]);
                o0.y = pack2_bf16(acc[2], acc[3]);
                o0.z = pack2_bf16(acc[4], acc[5]);
                o0.w = pack2_bf16(acc[6], acc[7]);
                o1.x = pack2_bf16(acc[8], acc[9]);
                o1.y = pack2_bf16(acc[10], acc[11]);
                o1.z = pack2_bf16(acc[12], acc[13]);
                o1.w = pack2_bf16(acc[14], acc[15]);
                uint4 *yr = y + t * (2LL * n16) + 2 * c;
                st_v4(yr, o0);
                st_v4(yr + 1, o1);
            }
        }
    }
}

int resident_grid(const void *fn, int threads)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess || n < 1) n = 1;
    return n * device_sm_count();
}

long long rows_grid(long long n)
{
    const long long cap = 1LL << 30;
    return n < 1 ? 1 : (n < cap ? n : cap);
}

template <int MODE, bool TOKENS>
cudaError_t launch_grouped(const void *src, long long n_src, int H, const moe_layout *L, void *out, float *scales,
                           cudaStream_t s)
{
    const int nvec = H / 8, npairs = H / 16;
    cudaError_t err = cudaSuccess;
    if (MODE != MOE_FP8_PER_TOKEN) {
        static int res[64] = {0};
        int dev = 0;
        cudaGetDevice(&dev);
        int &r = res[dev & 63];
        if (r == 0)
            r = resident_grid(reinterpret_cast<const void *>(fp8_group_stats_kernel<MODE, TOKENS>), kStatThreads);
        const long long need = (n_src + kStatThreads / 32 - 1) / (kStatThreads / 32);
        const unsigned grid = (unsigned)(need < r ? (need < 1 ? 1 : need) : r);
        err = launch_pdl(fp8_group_stats_kernel<MODE, TOKENS>, dim3(grid), dim3(kStatThreads), 0, s,
                         static_cast<const uint4 *>(src), n_src, nvec, L->k, (const int32_t *)L->dst_row,
                         (const int32_t *)L->offsets, L->E, L->r_max, L->ws);
        if (err != cudaSuccess) return err;
    }
    const int per_thread = (npairs + kEncThreads - 1) / kEncThreads;
    const unsigned grid = (unsigned)rows_grid(n_src);
#define MOE_ENC(CC)                                                                                            \
    return launch_pdl(fp8_group_encode_kernel<CC, MODE, TOKENS>, dim3(grid), dim3(kEncThreads), 0, s,          \
                      static_cast<const uint4 *>(src), n_src, npairs, L->k, (const int32_t *)L->dst_row,       \
                      (const int32_t *)L->offsets, L->E, L->r_max, static_cast<uint4 *>(out),                  \
                      reinterpret_cast<float2 *>(scales), L->ws)
    if (per_thread <= 1) MOE_ENC(1);
    if (per_thread <= 2) MOE_ENC(2);
    if (per_thread <= 4) MOE_ENC(4);
    if (per_thread <= 8) MOE_ENC(8);
#undef MOE_ENC
    return cudaErrorInvalidValue;
}

template <int K>
cudaError_t launch_cfp8_k(const void *codes, const float *scales, const moe_layout *L, const float *gates,
                          const void *shared, int Ks, int T, int H, void *y, cudaStream_t s)
{
    constexpr int V = K <= 2 ? 2 : 1;
    static int res[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int &r = res[dev & 63];
    if (r == 0) r = resident_grid(reinterpret_cast<const void *>(combine_fp8_kernel<K, V>), kCombFp8Threads);
    const long long need = ((long long)T + kCombFp8Threads / 32 - 1) / (kCombFp8Threads / 32);
    const unsigned grid = (unsigned)(need < r ? need : r);
    return launch_pdl(combine_fp8_kernel<K, V>, dim3(grid), dim3(kCombFp8Threads), 0, s,
                      static_cast<const uint4 *>(codes), reinterpret_cast<const float2 *>(scales), gates,
                      (const int32_t *)L->dst_row, L->r_max, (const int32_t *)(L->offsets + L->E),
                      static_cast<const uint4 *>(shared), Ks, (long long)T, H / 16, static_cast<uint4 *>(y), L->ws);
}

}  // namespace

cudaError_t launch_dispatch_fp8_grouped(const void *x, int T, int H, const moe_layout *L, int mode, void *packed,
                                        float *scales, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    if (mode == MOE_FP8_PER_EXPERT) return launch_grouped<MOE_FP8_PER_EXPERT, true>(x, T, H, L, packed, scales, s);
    if (mode == MOE_FP8_GLOBAL) return launch_grouped<MOE_FP8_GLOBAL, true>(x, T, H, L, packed, scales, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_rows(const void *rows, const moe_layout *L, int H, int mode, void *codes, float *scales,
                                 cudaStream_t s)
{
    const long long n = L->r_max;
    if (n == 0) return cudaSuccess;
    switch (mode) {
    case MOE_FP8_PER_TOKEN: return launch_grouped<MOE_FP8_PER_TOKEN, false>(rows, n, H, L, codes, scales, s);
    case MOE_FP8_PER_EXPERT: return launch_grouped<MOE_FP8_PER_EXPERT, false>(rows, n, H, L, codes, scales, s);
    case MOE_FP8_GLOBAL: return launch_grouped<MOE_FP8_GLOBAL, false>(rows, n, H, L, codes, scales, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine_fp8(const void *codes, const float *scales, const moe_layout *L, const float *gates,
                               const void *shared, int Ks, int T, int H, void *y, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    switch (L->k) {
#define MOE_CFP8_CASE(KK) \
    case KK: return launch_cfp8_k<KK>(codes, scales, L, gates, shared, Ks, T, H, y, s);
        MOE_CFP8_CASE(1) MOE_CFP8_CASE(2) MOE_CFP8_CASE(3) MOE_CFP8_CASE(4)
        MOE_CFP8_CASE(5) MOE_CFP8_CASE(6) MOE_CFP8_CASE(7) MOE_CFP8_CASE(8)
        MOE_CFP8_CASE(9) MOE_CFP8_CASE(10) MOE_CFP8_CASE(11) MOE_CFP8_CASE(12)
        MOE_CFP8_CASE(13) MOE_CFP8_CASE(14) MOE_CFP8_CASE(15) MOE_CFP8_CASE(16)
#undef MOE_CFP8_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
