// gate.cu -- moe_gate: top-k gating over router logits plus routing
// statistics, one fused kernel.
//
// Design (sm_103a).  A block stages a tile of TT tokens' logits in shared
// memory with coalesced loads (row stride E|1 words, so that consecutive
// threads reading "their" row hit distinct banks), then each thread owns one
// token and keeps a sorted register list of its k best (value, expert)
// pairs.  For E <= 256 and k <= 16 that is ~E compares per token, far fewer
// instructions than k rounds of warp-wide shuffle arg-max, which is what the
// A100 warp kernel of "DeepSeek MoE architecture evolution" (sec. 2.2)
// spends per token.  Counts go to a shared-memory histogram, then one
// global atomic per (block, expert) into the workspace; the last block to
// finish (atomic ticket) publishes expert_counts and derives the aux loss
// (fp64, from exact integer sums) and the entropy (exponent + fp32 mantissa
// logarithms, summed exactly in fixed point; ~1e-7 absolute), then clears
// the workspace counters for the next call.
//
// Definitions: "DeepSeek MoE architecture evolution" ch.1 (top2_gating:
// topk, softmax of the selected logits, aux = E * sum f_e^2) and sec. 2.3
// (entropy of the expert counts, base 2, +1e-8 inside the log); "DeepSeek
// MoE sync tax" sec. 4.1 (softmax over all experts, then top-k).
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kGateMaxThreads = 256;
constexpr int kStageLoads = 8;  // loads in flight per thread while staging logits

// Insert (v, e) into the descending list bv/bi of length K if it beats the
// last entry.  Strictly-greater comparisons keep the earlier (lower) expert
// id ahead on ties; -0.0 == +0.0 is a tie.
template <int K>
__device__ __forceinline__ void topk_insert(float (&bv)[K], int (&bi)[K], float v, int e)
{
    if (v > bv[K - 1]) {
        bv[K - 1] = v;
        bi[K - 1] = e;
#pragma unroll
        for (int j = K - 1; j > 0; --j) {
            if (bv[j] > bv[j - 1]) {
                float tv = bv[j]; bv[j] = bv[j - 1]; bv[j - 1] = tv;
                int ti = bi[j]; bi[j] = bi[j - 1]; bi[j - 1] = ti;
            }
        }
    }
}

// log2 of a positive, finite double: exact binary exponent plus log2f of the
// mantissa in [1, 2) (absolute error ~1e-7), avoiding fp64 transcendentals.
__device__ __forceinline__ double log2_via_mantissa(double x)
{
    const long long bits = __double_as_longlong(x);
    const int ex = (int)((bits >> 52) & 0x7FF) - 1023;
    const double m = __longlong_as_double((bits & 0x000FFFFFFFFFFFFFll) | 0x3FF0000000000000ll);
    return (double)ex + (double)log2f((float)m);
}

// 1/x for a positive double: the fp32 reciprocal refined by two
// Newton-Raphson steps (r <- r (2 - x r); each doubles the correct bits:
// 24 -> 48 -> full double), instead of an fp64 divide.
__device__ __forceinline__ double rcp_newton(double x)
{
    double r = (double)__frcp_rn((float)x);
    r = r * (2.0 - x * r);
    r = r * (2.0 - x * r);
    return r;
}

template <int K>
__device__ __forceinline__ void store_row_i32(int32_t *dst, const int (&v)[K])
{
    if constexpr (K % 4 == 0) {
#pragma unroll
        for (int j = 0; j < K; j += 4)
            *reinterpret_cast<int4 *>(dst + j) = make_int4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    } else if constexpr (K % 2 == 0) {
#pragma unroll
        for (int j = 0; j < K; j += 2) *reinterpret_cast<int2 *>(dst + j) = make_int2(v[j], v[j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j) dst[j] = v[j];
    }
}

template <int K>
__device__ __forceinline__ void store_row_f32(float *dst, const float (&v)[K])
{
    if constexpr (K % 4 == 0) {
#pragma unroll
        for (int j = 0; j < K; j += 4)
            *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    } else if constexpr (K % 2 == 0) {
#pragma unroll
        for (int j = 0; j < K; j += 2) *reinterpret_cast<float2 *>(dst + j) = make_float2(v[j], v[j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j) dst[j] = v[j];
    }
}

template <int K, int MODE>
__global__ void __launch_bounds__(kGateMaxThreads)
gate_kernel(const float *__restrict__ logits, int T, int E, int32_t *__restrict__ topk_idx,
            float *__restrict__ gates, int32_t *__restrict__ expert_counts,
            double *__restrict__ aux_out, double *__restrict__ ent_out, void *ws_raw)
{
    extern __shared__ float s_logit[];  // [TT][stride]
    __shared__ unsigned s_hist[MOE_MAX_EXPERTS];
    __shared__ int s_bad;
    __shared__ int s_last;
    WsHeader *ws = static_cast<WsHeader *>(ws_raw);

    const int TT = blockDim.x;
    const int stride = E | 1;
    const long long t0 = (long long)blockIdx.x * TT;
    const int rows = (int)min((long long)TT, (long long)T - t0);

    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0u;
    if (threadIdx.x == 0) s_bad = 0;
    pdl_wait();
    pdl_launch_dependents();

    // Stage the tile.  Its rows are contiguous in global memory, so it is one
    // flat copy: every thread issues kStageLoads independent 16-byte loads
    // before any shared-memory store, so the whole tile is in flight at once.
    {
        const float *src = logits + t0 * (long long)E;
        const int n = rows * E;
        if ((E & 3) == 0) {
            const float4 *src4 = reinterpret_cast<const float4 *>(src);
            const int n4 = n >> 2;
            for (int base = 0; base < n4; base += kStageLoads * blockDim.x) {
                float4 v[kStageLoads];
#pragma unroll
                for (int u = 0; u < kStageLoads; ++u) {
                    const int i = base + u * blockDim.x + threadIdx.x;
                    if (i < n4) v[u] = __ldg(src4 + i);
                }
#pragma unroll
                for (int u = 0; u < kStageLoads; ++u) {
                    const int i = base + u * blockDim.x + threadIdx.x;
                    if (i < n4) {
                        const int r = (4 * i) / E, c = 4 * i - r * E;
                        float *d = s_logit + r * stride + c;
                        d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
                    }
                }
            }
        } else {
            for (int base = 0; base < n; base += kStageLoads * blockDim.x) {
                float v[kStageLoads];
#pragma unroll
                for (int u = 0; u < kStageLoads; ++u) {
                    const int i = base + u * blockDim.x + threadIdx.x;
                    if (i < n) v[u] = __ldg(src + i);
                }
#pragma unroll
                for (int u = 0; u < kStageLoads; ++u) {
                    const int i = base + u * blockDim.x + threadIdx.x;
                    if (i < n) {
                        const int r = i / E;
                        s_logit[r * stride + (i - r * E)] = v[u];
                    }
                }
            }
        }
    }
    __syncthreads();

    float bv[K];
    int bi[K];
    float g[K];
    const bool active = threadIdx.x < rows;
    if (active) {
        const float *row = s_logit + threadIdx.x * stride;
        bool finite = true;
        // First K experts: insertion-sorted in place.
#pragma unroll
        for (int j = 0; j < K; ++j) {
            bv[j] = row[j];
            bi[j] = j;
            finite &= isfinite(bv[j]);
        }
#pragma unroll
        for (int i = 1; i < K; ++i) {
#pragma unroll
            for (int j = i; j > 0; --j) {
                if (bv[j] > bv[j - 1]) {
                    float tv = bv[j]; bv[j] = bv[j - 1]; bv[j - 1] = tv;
                    int ti = bi[j]; bi[j] = bi[j - 1]; bi[j - 1] = ti;
                }
            }
        }
#pragma unroll 8
        for (int e = K; e < E; ++e) {
            float v = row[e];
            finite &= isfinite(v);
            topk_insert<K>(bv, bi, v, e);
        }
        if (!finite) s_bad = 1;

        // Gate weights, fp32, shifted by the largest logit.
        const float m = bv[0];
        if constexpr (MODE == MOE_TOPK_SOFTMAX) {
            float ex[K];
            float sum = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                ex[j] = expf(__fsub_rn(bv[j], m));
                sum = __fadd_rn(sum, ex[j]);
            }
#pragma unroll
            for (int j = 0; j < K; ++j) g[j] = __fdiv_rn(ex[j], sum);
        } else {
            float sum = 0.0f;
            for (int e = 0; e < E; ++e) sum = __fadd_rn(sum, expf(__fsub_rn(row[e], m)));
#pragma unroll
            for (int j = 0; j < K; ++j) g[j] = __fdiv_rn(expf(__fsub_rn(bv[j], m)), sum);
        }

#pragma unroll
        for (int j = 0; j < K; ++j) atomicAdd(&s_hist[bi[j]], 1u);
    }
    __syncthreads();

    // counts first: the fence before the ticket then covers only these few
    // atomics, not the block's output stores, which follow it
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (s_hist[e]) atomicAdd(&ws->gate_counts[e], s_hist[e]);
    if (threadIdx.x == 0 && s_bad) record_status(ws, MOE_ERR_DEVICE_DATA);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&ws->gate_ticket, 1u) == gridDim.x - 1);
    if (active) {
        const long long t = t0 + threadIdx.x;
        store_row_i32<K>(topk_idx + t * K, bi);
        store_row_f32<K>(gates + t * K, g);
    }
    __syncthreads();
    if (!s_last) return;

    // Last block: publish the totals and the statistics.  FP64 units are
    // scarce on this part, so the per-expert work avoids fp64 transcendentals:
    //   entropy = -sum_e p_e log2(p_e + eps),  p_e = c_e / N,  N = T*k
    //           = log2(N) * SUM / N - (1/N) sum_e c_e log2(c_e + eps*N),  SUM = sum_e c_e
    // with each log2 of a double taken as exponent + log2f(mantissa) (error
    // ~1e-7 absolute), the products c_e*log2(.) summed exactly in 2^-32
    // fixed point with integer warp shuffles (deterministic), and
    //   aux = E * (sum_e c_e^2) / T^2  from the exact integer sum of squares.
    __threadfence();
    __shared__ long long s_fix[kGateMaxThreads / 32];
    __shared__ unsigned long long s_sq[kGateMaxThreads / 32], s_sum[kGateMaxThreads / 32];
    const double n_assign = (double)T * (double)K;
    const double eps_n = 1e-8 * n_assign;
    long long fix = 0;
    unsigned long long sq = 0ull, sum = 0ull;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const unsigned c = atomicExch(&ws->gate_counts[e], 0u);
        expert_counts[e] = (int32_t)c;
        sq += (unsigned long long)c * c;
        sum += c;
        if (c) fix += llrint((double)c * log2_via_mantissa((double)c + eps_n) * 4294967296.0);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        fix += __shfl_xor_sync(0xffffffffu, fix, d);
        sq += __shfl_xor_sync(0xffffffffu, sq, d);
        sum += __shfl_xor_sync(0xffffffffu, sum, d);
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) {
        s_fix[wid] = fix;
        s_sq[wid] = sq;
        s_sum[wid] = sum;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        long long F = 0;
        unsigned long long SQ = 0ull, SUM = 0ull;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            F += s_fix[w];
            SQ += s_sq[w];
            SUM += s_sum[w];
        }
        if (T > 0) {
            const double inv_t = rcp_newton((double)T);
            *aux_out = (double)E * ((double)SQ * inv_t * inv_t);
            *ent_out = (log2_via_mantissa(n_assign) * (double)SUM - (double)F * (1.0 / 4294967296.0)) *
                       rcp_newton(n_assign);
        } else {
            *aux_out = 0.0;
            *ent_out = 0.0;
        }
        ws->gate_ticket = 0u;
    }
}

template <int K, int MODE>
cudaError_t launch_k(const float *logits, int T, int E, int32_t *idx, float *gates, int32_t *counts,
                     double *aux, double *ent, void *ws, cudaStream_t s)
{
    const int stride = E | 1;
    // Tile size: keep the staging buffer <= 64 KiB and prefer >= 2 blocks per SM.
    int tt = kGateMaxThreads;
    while (tt > 32 && (size_t)tt * stride * sizeof(float) > 64 * 1024) tt >>= 1;
    const long long want_blocks = 2LL * device_sm_count();
    while (tt > 64 && ((long long)T + tt - 1) / tt < want_blocks) tt >>= 1;
    const size_t smem = (size_t)tt * stride * sizeof(float);
    cudaError_t err = allow_dynamic_smem(reinterpret_cast<const void *>(gate_kernel<K, MODE>), (int)smem);
    if (err != cudaSuccess) return err;
    long long blocks = ((long long)T + tt - 1) / tt;
    if (blocks < 1) blocks = 1;
    return launch_pdl(gate_kernel<K, MODE>, dim3((unsigned)blocks), dim3(tt), smem, s, logits, T, E, idx, gates,
                      counts, aux, ent, ws);
}

template <int MODE>
cudaError_t launch_mode(const float *logits, int T, int E, int k, int32_t *idx, float *gates,
                        int32_t *counts, double *aux, double *ent, void *ws, cudaStream_t s)
{
    switch (k) {
#define MOE_GATE_CASE(KK) \
    case KK: return launch_k<KK, MODE>(logits, T, E, idx, gates, counts, aux, ent, ws, s);
        MOE_GATE_CASE(1) MOE_GATE_CASE(2) MOE_GATE_CASE(3) MOE_GATE_CASE(4)
        MOE_GATE_CASE(5) MOE_GATE_CASE(6) MOE_GATE_CASE(7) MOE_GATE_CASE(8)
        MOE_GATE_CASE(9) MOE_GATE_CASE(10) MOE_GATE_CASE(11) MOE_GATE_CASE(12)
        MOE_GATE_CASE(13) MOE_GATE_CASE(14) MOE_GATE_CASE(15) MOE_GATE_CASE(16)
#undef MOE_GATE_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gate(const float *logits, int T, int E, int k, int mode, int32_t *topk_idx,
                        float *gates, int32_t *expert_counts, double *aux, double *entropy,
                        void *ws, cudaStream_t s)
{
    if (mode == MOE_TOPK_SOFTMAX)
        return launch_mode<MOE_TOPK_SOFTMAX>(logits, T, E, k, topk_idx, gates, expert_counts, aux,
                                             entropy, ws, s);
    return launch_mode<MOE_SOFTMAX_TOPK>(logits, T, E, k, topk_idx, gates, expert_counts, aux,
                                         entropy, ws, s);
}

}  // namespace moe
