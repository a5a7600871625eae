// backward.cu -- the backward of the routing path: moe_combine_backward and
// moe_gate_backward (moe_dispatch_backward reuses the combine kernel with
// unit weights, see combine.cu).
//
// "Deepseek-MoE sync-tax essence and four-layer optimisation guide" sec. 2.4
// (the backward exchange mirrors the forward one, driven by the routing
// indices cached in the forward pass: nothing is re-routed);
// "MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7,
// detail item 3 (the combine stage carries the gradients back in the
// backward pass; gradient sums want fp32 accumulation).
//
// Combine backward, per token t and kept slot j (row r = dst_row[t,j]):
//   d_expert_out[r] = bf16 RNE(fp32(g[t,j] * dy[t]))   -- a dispatch of g*dy
//   d_gates[t,j]    = sum_h dy[t,h] * expert_out[r,h]   -- fp32, 0 if dropped
// Design (sm_103a): scatter form like the forward dispatch.  One warp per
// token; each lane owns 16-byte column vectors of the row.  It loads V dy
// vectors and the matching vectors of all K expert-output rows up front
// (a dropped slot reads the dy row again, an L2 hit, so the loads stay
// unconditional and all in flight together), writes the K scaled rows with
// 16-byte stores, and accumulates the K dot products: the 8 products of a
// vector with FMA from 0 (a bf16 x bf16 product is exact in fp32, so each
// step rounds once), that partial added to the slot's running sum, and the
// 32 lane sums reduced by a warp xor tree.  Fixed order, deterministic;
// summation depth 8 + ceil(H/256) + 5 <= H/256 + 14.
//
// Gate backward, per token (gates recomputed from the logits in fp32):
//   TOPK_SOFTMAX: g = softmax over the k selected logits;
//                 d_logits[sel_j] = g_j (dg_j - s), s = sum_i g_i dg_i, other experts 0
//   SOFTMAX_TOPK: p = softmax over all E, g_j = p[sel_j];
//                 d_logits[e] = (e == sel_j ? g_j dg_j : 0) - p_e s
// A group of lanes per token (a whole warp for E > 16), lanes striding the
// E experts (coalesced row loads and stores), xor trees for max and sums.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kBwdThreads = 256;  // combine backward: 8 token warps per block

__device__ __forceinline__ unsigned pack_bf16x2_rn(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&h);
}

__device__ __forceinline__ uint4 scale_row_vec(float g, const uint4 &d)
{
    uint4 o;
    o.x = pack_bf16x2_rn(__fmul_rn(g, bf16lo(d.x)), __fmul_rn(g, bf16hi(d.x)));
    o.y = pack_bf16x2_rn(__fmul_rn(g, bf16lo(d.y)), __fmul_rn(g, bf16hi(d.y)));
    o.z = pack_bf16x2_rn(__fmul_rn(g, bf16lo(d.z)), __fmul_rn(g, bf16hi(d.z)));
    o.w = pack_bf16x2_rn(__fmul_rn(g, bf16lo(d.w)), __fmul_rn(g, bf16hi(d.w)));
    return o;
}

__device__ __forceinline__ float dot_vec(float acc, const uint4 &d, const uint4 &e)
{
    acc = __fmaf_rn(bf16lo(d.x), bf16lo(e.x), acc);
    acc = __fmaf_rn(bf16hi(d.x), bf16hi(e.x), acc);
    acc = __fmaf_rn(bf16lo(d.y), bf16lo(e.y), acc);
    acc = __fmaf_rn(bf16hi(d.y), bf16hi(e.y), acc);
    acc = __fmaf_rn(bf16lo(d.z), bf16lo(e.z), acc);
    acc = __fmaf_rn(bf16hi(d.z), bf16hi(e.z), acc);
    acc = __fmaf_rn(bf16lo(d.w), bf16lo(e.w), acc);
    acc = __fmaf_rn(bf16hi(d.w), bf16hi(e.w), acc);
    return acc;
}

// One warp per token (persistent warps striding over the tokens): lane l
// owns the 16-byte column vectors l, l+32, ... of the row, V of them per
// pass.  No block-wide barrier, so the warps of an SM drift apart and one
// warp's reduction overlaps the others' loads.
template <int K, int V>
__global__ void __launch_bounds__(kBwdThreads)
combine_bwd_kernel(const uint4 *__restrict__ dy, const uint4 *__restrict__ eo, const float *__restrict__ gates,
                   const int32_t *__restrict__ dst_row, int r_max, const int32_t *__restrict__ R_ptr, long long T,
                   int nvec, uint4 *__restrict__ d_eo, float *__restrict__ d_gates, void *ws)
{
    pdl_wait();
    pdl_launch_dependents();
    const uint64_t pol = l2_stream_policy(false);
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (kBwdThreads / 32);
    const int rows_valid = min(r_max, __ldg(R_ptr));
    for (long long t = (long long)blockIdx.x * (kBwdThreads / 32) + (threadIdx.x >> 5); t < T; t += nwarps) {
        // lane j < K reads slot j; broadcast below
        int rl = -1;
        float gl = 0.0f;
        if (lane < K) {
            rl = __ldg(dst_row + t * K + lane);
            gl = __ldg(gates + t * K + lane);
            if (rl >= rows_valid) {
                record_status(ws, MOE_ERR_DEVICE_DATA);
                rl = -1;
            }
        }
        int row[K];
        float g[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            row[j] = __shfl_sync(0xffffffffu, rl, j);
            g[j] = __shfl_sync(0xffffffffu, gl, j);
        }
        const uint4 *dyrow = dy + t * nvec;
        float dot[K];
#pragma unroll
        for (int j = 0; j < K; ++j) dot[j] = 0.0f;
        for (int c0 = lane; c0 < nvec; c0 += 32 * V) {
            uint4 d[V];
            uint4 e[K][V];
#pragma unroll
            for (int u = 0; u < V; ++u) {
                const int c = c0 + 32 * u;
                d[u] = c < nvec ? ld_stream_v4(dyrow + c, pol) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const uint4 *src = row[j] >= 0 ? eo + (long long)row[j] * nvec : dyrow;
#pragma unroll
                for (int u = 0; u < V; ++u) {
                    const int c = c0 + 32 * u;
                    e[j][u] = c < nvec ? ld_stream_v4(src + c, pol) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (row[j] < 0) continue;
                uint4 *dst = d_eo + (long long)row[j] * nvec;
#pragma unroll
                for (int u = 0; u < V; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < nvec) st_stream_v4(dst + c, scale_row_vec(g[j], d[u]), pol);
                }
            }
            // per vector: its 8 products summed from 0, then added to the slot's sum
#pragma unroll
            for (int j = 0; j < K; ++j)
#pragma unroll
                for (int u = 0; u < V; ++u) dot[j] = __fadd_rn(dot[j], dot_vec(0.0f, d[u], e[j][u]));
        }
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            float v = dot[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == j) mine = row[j] >= 0 ? v : 0.0f;
        }
        if (lane < K) d_gates[t * K + lane] = mine;
    }
}

// Reductions over the G lanes of a group (G a power of two <= 32).
template <int G>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o, G));
    return v;
}
template <int G>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o, G));
    return v;
}

constexpr int kGateBwdThreads = 256;

// Gradient of one token's logits held by a group of G lanes: vals = the
// lane's logits (experts sub, sub+G, ...; -inf past E or for an invalid
// token), sel/dg = slot `sub`'s expert and gate gradient (sel < 0: none).
// Returns the lane's d_logits in out.
template <int MODE, int G, int EPL>
__device__ __forceinline__ void token_logit_grad(float (&vals)[EPL], int sel, float dg, bool valid, int k, int E,
                                                 int sub, float (&out)[EPL])
{
    // the selected expert's logit, from the lane of the group that holds it
    float lsel = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const float v = __shfl_sync(0xffffffffu, vals[i], sel >= 0 ? sel & (G - 1) : 0, G);
        if (sel >= 0 && sel / G == i) lsel = v;
    }
    float m, z;
    if (MODE == MOE_TOPK_SOFTMAX) {
        m = group_max<G>(lsel);
        z = group_sum<G>(sel >= 0 ? expf(__fsub_rn(lsel, m)) : 0.0f);
    } else {
        float lm = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i) lm = fmaxf(lm, vals[i]);
        m = group_max<G>(lm);
        float zs = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            vals[i] = (valid && sub + G * i < E) ? expf(__fsub_rn(vals[i], m)) : 0.0f;
            zs = __fadd_rn(zs, vals[i]);
        }
        z = group_sum<G>(zs);
    }
    const float g = sel >= 0 ? __fdiv_rn(expf(__fsub_rn(lsel, m)), z) : 0.0f;
    const float gdg = __fmul_rn(g, dg);
    const float s = group_sum<G>(gdg);
    // slot j's contribution to its expert's gradient
    const float own = MODE == MOE_TOPK_SOFTMAX ? __fmul_rn(g, __fsub_rn(dg, s)) : gdg;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        out[i] = MODE == MOE_TOPK_SOFTMAX ? 0.0f : -__fmul_rn(__fdiv_rn(vals[i], z), s);
    for (int j = 0; j < k; ++j) {
        const int ej = __shfl_sync(0xffffffffu, sel, j, G);
        const float oj = __shfl_sync(0xffffffffu, own, j, G);
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (ej == sub + G * i) out[i] = __fadd_rn(out[i], oj);
    }
}

// A group of G lanes per token (G = E rounded up to a power of two, at most
// 32), 32/G tokens per warp, so the row loads and stores of a warp stay
// contiguous for small E.  Lane i of a group holds experts i, i+G, ...
// (EPL = ceil(E/G) of them); lane j < k also holds slot j.  Each warp takes
// U token groups per iteration and issues all their loads (logits rows,
// ids, gate gradients) before any arithmetic; the selected logits come
// from the rows through shuffles, not from a dependent second load.
template <int MODE, int G, int EPL, int U>
__global__ void __launch_bounds__(kGateBwdThreads)
gate_bwd_kernel(const float *__restrict__ logits, const int32_t *__restrict__ topk_idx,
                const float *__restrict__ d_gates, long long T, int E, int k, float *__restrict__ d_logits, void *ws)
{
    pdl_wait();
    pdl_launch_dependents();
    constexpr int TPW = 32 / G;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (G - 1), grp = lane / G;
    const long long nwarps = (long long)gridDim.x * (kGateBwdThreads / 32);
    for (long long base = ((long long)blockIdx.x * (kGateBwdThreads / 32) + (threadIdx.x >> 5)) * TPW * U;
         base < T; base += nwarps * TPW * U) {
        float vals[U][EPL];
        int sel[U];
        float dg[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long t = base + u * TPW + grp;
            const bool valid = t < T;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = sub + G * i;
                vals[u][i] = (valid && e < E) ? __ldg(logits + t * E + e) : -INFINITY;
            }
            sel[u] = -1;
            dg[u] = 0.0f;
            if (valid && sub < k) {
                sel[u] = __ldg(topk_idx + t * k + sub);
                dg[u] = __ldg(d_gates + t * k + sub);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long t = base + u * TPW + grp;
            const bool valid = t < T;
            if (sel[u] >= E || (valid && sub < k && sel[u] < 0)) {
                record_status(ws, MOE_ERR_DEVICE_DATA);
                sel[u] = -1;
            }
            float out[EPL];
            token_logit_grad<MODE, G, EPL>(vals[u], sel[u], dg[u], valid, k, E, sub, out);
            if (valid) {
                float *dl = d_logits + t * E;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = sub + G * i;
                    if (e < E) dl[e] = out[i];
                }
            }
        }
    }
}

template <int K>
cudaError_t launch_cbwd_k(const void *dy, const void *eo, const moe_layout *L, const float *gates, int T, int H,
                          void *d_eo, float *d_gates, cudaStream_t s)
{
    const int nvec = H / 8;
    // V vectors per lane and pass, chosen so the (K+1)*V vectors of a pass
    // fit in registers next to each other.
    constexpr int V = K <= 3 ? 4 : (K <= 8 ? 2 : 1);
    const int res = resident_grid(reinterpret_cast<const void *>(combine_bwd_kernel<K, V>), kBwdThreads, 0);
    const long long need = ((long long)T + kBwdThreads / 32 - 1) / (kBwdThreads / 32);
    const unsigned grid = (unsigned)(need < res ? need : res);
    return launch_pdl(combine_bwd_kernel<K, V>, dim3(grid), dim3(kBwdThreads), 0, s, static_cast<const uint4 *>(dy),
                      static_cast<const uint4 *>(eo), gates, (const int32_t *)L->dst_row, (int)L->r_max,
                      (const int32_t *)(L->offsets + L->E), (long long)T, nvec, static_cast<uint4 *>(d_eo), d_gates,
                      L->ws);
}

template <int MODE, int G, int EPL, int U = (EPL <= 2 ? 4 : (EPL <= 4 ? 2 : 1))>
cudaError_t launch_gbwd(const float *logits, const int32_t *topk_idx, const float *d_gates, int T, int E, int k,
                        float *d_logits, void *ws, cudaStream_t s)
{
    const int res = resident_grid(reinterpret_cast<const void *>(gate_bwd_kernel<MODE, G, EPL, U>), kGateBwdThreads, 0);
    const long long per_block = (long long)(kGateBwdThreads / 32) * (32 / G) * U;
    const long long need = ((long long)T + per_block - 1) / per_block;
    const unsigned grid = (unsigned)(need < res ? need : res);
    return launch_pdl(gate_bwd_kernel<MODE, G, EPL, U>, dim3(grid), dim3(kGateBwdThreads), 0, s, logits, topk_idx,
                      d_gates, (long long)T, E, k, d_logits, ws);
}

template <int MODE>
cudaError_t launch_gbwd_m(const float *logits, const int32_t *topk_idx, const float *d_gates, int T, int E, int k,
                          float *d_logits, void *ws, cudaStream_t s)
{
#define MOE_GBWD(G, EPL) return launch_gbwd<MODE, G, EPL>(logits, topk_idx, d_gates, T, E, k, d_logits, ws, s)
    if (E <= 1) MOE_GBWD(1, 1);
    if (E <= 2) MOE_GBWD(2, 1);
    if (E <= 4) MOE_GBWD(4, 1);
    if (E <= 8) MOE_GBWD(8, 1);
    if (E <= 16) MOE_GBWD(16, 1);
    switch ((E + 31) / 32) {
    case 1: MOE_GBWD(32, 1);
    case 2: MOE_GBWD(32, 2);
    case 3: MOE_GBWD(32, 3);
    case 4: MOE_GBWD(32, 4);
    case 5: MOE_GBWD(32, 5);
    case 6: MOE_GBWD(32, 6);
    case 7: MOE_GBWD(32, 7);
    case 8: MOE_GBWD(32, 8);
    default: return cudaErrorInvalidValue;
    }
#undef MOE_GBWD
}

}  // namespace

cudaError_t launch_combine_backward(const void *dy, const void *eo, const moe_layout *L, const float *gates, int T,
                                   int H, void *d_eo, float *d_gates, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    switch (L->k) {
#define MOE_CBWD_CASE(KK) \
    case KK: return launch_cbwd_k<KK>(dy, eo, L, gates, T, H, d_eo, d_gates, s);
        MOE_CBWD_CASE(1) MOE_CBWD_CASE(2) MOE_CBWD_CASE(3) MOE_CBWD_CASE(4)
        MOE_CBWD_CASE(5) MOE_CBWD_CASE(6) MOE_CBWD_CASE(7) MOE_CBWD_CASE(8)
        MOE_CBWD_CASE(9) MOE_CBWD_CASE(10) MOE_CBWD_CASE(11) MOE_CBWD_CASE(12)
        MOE_CBWD_CASE(13) MOE_CBWD_CASE(14) MOE_CBWD_CASE(15) MOE_CBWD_CASE(16)
#undef MOE_CBWD_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gate_backward(const float *logits, const int32_t *topk_idx, const float *d_gates, int T, int E,
                                 int k, int mode, float *d_logits, void *ws, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    return mode == MOE_TOPK_SOFTMAX
               ? launch_gbwd_m<MOE_TOPK_SOFTMAX>(logits, topk_idx, d_gates, T, E, k, d_logits, ws, s)
               : launch_gbwd_m<MOE_SOFTMAX_TOPK>(logits, topk_idx, d_gates, T, E, k, d_logits, ws, s);
}

}  // namespace moe
