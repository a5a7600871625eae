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
//   2. fp8_encode_kernel: blocks walk the rows, every block first turning
//      the workspace keys into the groups' (scale, zero) in shared memory;
//      a completion ticket lets the last block reset the keys, so the
//      workspace stays zeroed.
// The per-token mode is the encode pass alone, with the row's extremes
// reduced inside the block.  The encode does the pinned fp32 operations on
// packed pairs with a rounding test that makes every code the one of the
// correctly rounded division (fp8.cuh), and the hardware e4m3x2 satfinite
// conversion.  The dispatch side reads token rows of x and writes each
// kept copy (a token sent to two experts is encoded once per expert in the
// per-expert mode, once in total in the other modes); the expert side reads
// packed expert-output rows and writes the same rows.
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
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 256;

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
    const uint64_t pol = l2_stream_policy(false);  // measured: evict-first slows the FP8 paths
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
                if (c + 32 * u < nvec) v[u] = ld_stream_v4(row + c + 32 * u, pol);
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

// ---- encode pass ------------------------------------------------------------
// Warp-specialised and TMA-staged, like the combine: a producer warp keeps
// a ring of `stages` source rows in flight in shared memory (one 1-D bulk
// copy per row, completing on the stage's "full" mbarrier), and eight
// consumer warps each take every eighth row of the block (or, for rows of
// expert outputs, pairs of warps every fourth row, each warp half of the
// columns, the halves' extremes exchanged through shared memory and a
// per-stage mbarrier): a warp reads its
// row from shared memory, reduces the extremes with shuffles alone (per-
// token mode; packed bf16 max/min, a zero extreme recomputed with the
// ordered integer keys, which rank -0 below +0), encodes each run of
// destinations with one group once (packed fp32 arithmetic with the
// rounding test of fp8.cuh), stores the codes with 16-byte stores and
// releases the stage on its "empty" mbarrier.  No block-wide barrier sits
// in the loop: the rows in flight per SM are set by shared memory and the
// rows being encoded by the consumer warps.  Every wait is bounded; on
// expiry MOE_ERR_TIMEOUT is recorded, the block stops, and the producer
// waits (bounded) for the copies it issued before the block exits.
constexpr int kEncMaxConsumers = 8;
constexpr int kEncMaxThreads = 32 * (kEncMaxConsumers + 1);
constexpr int kEncRingBytes = 112 * 1024;  // per block at most
constexpr int kEncMaxStages = 16;

struct EncArgs {
    const unsigned char *src;  // [n_src, H] bf16
    long long n_src;           // T (tokens) or r_max (rows; R on the device bounds it)
    int rowbytes;              // 2H
    int npairs;                // H / 16
    int k;
    const int32_t *dst_row;
    const int32_t *offsets;
    int E;
    int r_max;
    uint4 *out;                // [r_max, H / 16] codes
    float2 *scales;            // [r_max]
    void *ws;
    int stages;     // a multiple of the groups: stage st is always read by group st % (consumers / group)
    int consumers;  // consumer warps (block = consumers + 1 warps)
    int group;      // consumer warps sharing a row (1 or 2), each a contiguous half of its columns
};

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kSpinLimitNs) return false;
    return true;
}

template <int MODE, bool TOKENS>
__global__ void __launch_bounds__(kEncMaxThreads)
fp8_encode_kernel(EncArgs a)
{
    extern __shared__ __align__(128) unsigned char s_ring[];
    __shared__ uint64_t s_full[kEncMaxStages], s_empty[kEncMaxStages], s_pair[kEncMaxStages];
    __shared__ float2 s_xch[kEncMaxStages][2];  // per-token extremes of each half of a shared row
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ float2 s_par[MOE_MAX_EXPERTS];
    __shared__ volatile int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ngroups = MODE == MOE_FP8_GLOBAL ? 1 : (MODE == MOE_FP8_PER_EXPERT ? a.E : 0);
    WsHeader *h = static_cast<WsHeader *>(a.ws);
    if (tid == 0) {
        for (int st = 0; st < a.stages; ++st) {
            mbar_init(&s_full[st], 1);
            mbar_init(&s_empty[st], a.group);  // released by every warp of the group
            mbar_init(&s_pair[st], a.group);   // the group's extremes exchange
        }
        mbar_fence_init();
        s_abort = 0;
    }
    pdl_wait();
    pdl_launch_dependents();
    const uint64_t pol = l2_stream_policy(false);  // measured: evict-first slows the FP8 paths
    for (int i = tid; i <= a.E; i += blockDim.x) s_off[i] = __ldg(a.offsets + i);
    for (int g = tid; g < ngroups; g += blockDim.x) {
        const unsigned wmx = *((volatile unsigned *)&h->quant_max[g]);
        const unsigned wmn = *((volatile unsigned *)&h->quant_min[g]);
        s_par[g] = wmx == 0u ? make_float2(0.0f, 0.0f) : affine_pair(key_of_max_word(wmx), key_of_min_word(wmn));
    }
    __syncthreads();
    const int rows_valid = min(a.r_max, s_off[a.E]);
    const long long n_src = TOKENS ? a.n_src : min(a.n_src, (long long)rows_valid);
    const long long stride = gridDim.x;
    const long long n_mine = n_src > blockIdx.x ? (n_src - blockIdx.x + stride - 1) / stride : 0;

    if (warp == 0) {
        // ---- producer: lane 0 keeps the ring full ---------------------------
        if (lane == 0) {
            long long i = 0;
            for (; i < n_mine && !s_abort; ++i) {
                const int st = (int)(i % a.stages);
                if (i >= a.stages && !wait_phase(&s_empty[st], (uint32_t)(((i / a.stages) - 1) & 1))) {
                    record_status(a.ws, MOE_ERR_TIMEOUT);
                    s_abort = 1;
                    break;
                }
                const long long r = blockIdx.x + i * stride;
                mbar_arrive_expect_tx(&s_full[st], (uint32_t)a.rowbytes);
                bulk_load(s_ring + (size_t)st * a.rowbytes, a.src + r * a.rowbytes, (uint32_t)a.rowbytes,
                          &s_full[st], pol);
            }
            // never leave with copies still landing in shared memory: wait for
            // the last copy issued into each stage
            const long long first = i > a.stages ? i - a.stages : 0;
            for (long long q = first; q < i; ++q)
                wait_phase(&s_full[q % a.stages], (uint32_t)((q / a.stages) & 1));
        }
    } else {
        // ---- consumers: groups of G warps (G = a.group); group g takes rows
        // g, g + NG, ... (NG groups), each warp of it a contiguous share of
        // the row's 16-column vectors.  stages is a multiple of NG, so every
        // stage is read by one group only, in order: a warp never waits on a
        // phase two ahead of the last one it consumed there (the parity wait
        // cannot alias).  With G = 2 the per-token extremes of the two halves
        // meet in shared memory through a per-stage mbarrier (bounded wait).
        const int G = a.group;
        const int ng = a.consumers / G;
        const int grp = (warp - 1) / G, part = (warp - 1) - grp * G;
        const int q0 = part * a.npairs / G, q1 = (part + 1) * a.npairs / G;
        for (long long i = grp; i < n_mine; i += ng) {
            if (__any_sync(0xffffffffu, s_abort != 0)) break;  // the warp leaves together
            const int st = (int)(i % a.stages);
            const long long r_src = blockIdx.x + i * stride;
            // destinations: lane j < k holds slot j's row (tokens), lane 0 the row itself
            int r = -1;
            if (TOKENS) {
                if (lane < a.k) {
                    r = __ldg(a.dst_row + r_src * a.k + lane);
                    if (r >= rows_valid) {
                        record_status(a.ws, MOE_ERR_DEVICE_DATA);
                        r = -1;
                    }
                }
            } else if (lane == 0) {
                r = (int)r_src;
            }
            const unsigned kept = __ballot_sync(0xffffffffu, r >= 0);
            const int grp_mine = (r >= 0 && MODE == MOE_FP8_PER_EXPERT) ? expert_of_row(s_off, a.E, r) : 0;
            // every lane waits (the wait makes the copy visible to it); the
            // warp leaves together if any lane's bounded wait expired
            const bool landed = wait_phase(&s_full[st], (uint32_t)((i / a.stages) & 1));
            if (!__all_sync(0xffffffffu, landed)) {
                if (lane == 0) record_status(a.ws, MOE_ERR_TIMEOUT);
                s_abort = 1;
                break;
            }
            const unsigned char *row = s_ring + (size_t)st * a.rowbytes;
            float2 par_tok = make_float2(0.0f, 0.0f);
            if (MODE == MOE_FP8_PER_TOKEN && (kept != 0u || G > 1)) {
                // (a group exchanges for every row, so the exchange barrier's
                // phase counts rows like the others)
                __nv_bfloat162 mx2 = __float2bfloat162_rn(-INFINITY), mn2 = __float2bfloat162_rn(INFINITY);
                for (int q = q0 + lane; q < q1; q += 32) {
                    hminmax8(lds_v4(row + 32 * q), mx2, mn2);
                    hminmax8(lds_v4(row + 32 * q + 16), mx2, mn2);
                }
                float mx = fmaxf(__low2float(mx2), __high2float(mx2));
                float mn = fminf(__low2float(mn2), __high2float(mn2));
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, d));
                }
                if (G > 1) {
                    if (lane == 0) {
                        s_xch[st][part] = make_float2(mx, mn);
                        mbar_arrive(&s_pair[st]);  // release: the pair of values above
                    }
                    const bool met = wait_phase(&s_pair[st], (uint32_t)((i / a.stages) & 1));
                    if (!__all_sync(0xffffffffu, met)) {
                        if (lane == 0) record_status(a.ws, MOE_ERR_TIMEOUT);
                        s_abort = 1;
                        break;
                    }
                    const float2 o = s_xch[st][part ^ 1];
                    mx = fmaxf(mx, o.x);  // the same in both warps: max and min commute
                    mn = fminf(mn, o.y);
                }
                int kmax = f32_order_key(__float_as_uint(mx)), kmin = f32_order_key(__float_as_uint(mn));
                if (mx == 0.0f || mn == 0.0f) {
                    // a zero extreme: its sign needs the ordered keys (-0 < +0);
                    // every warp of a group reads the whole row (rare: no exchange)
                    kmax = INT_MIN;
                    kmin = INT_MAX;
                    for (int q = lane; q < a.npairs; q += 32)
                        minmax16(lds_v4(row + 32 * q), lds_v4(row + 32 * q + 16), kmax, kmin);
#pragma unroll
                    for (int d = 16; d > 0; d >>= 1) {
                        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, d));
                        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, d));
                    }
                }
                par_tok = affine_pair(kmax, kmin);
            }
            // runs of destinations with one group share their codes (slot order)
            unsigned rest = kept;
            while (rest) {
                const int j0 = __ffs(rest) - 1;
                const int g = __shfl_sync(0xffffffffu, grp_mine, j0);
                const unsigned same = __ballot_sync(0xffffffffu, (rest >> lane) & 1u && grp_mine == g);
                rest &= ~same;
                const float2 par = MODE == MOE_FP8_PER_TOKEN ? par_tok : s_par[g];
                const float rcp = e4m3_rcp(par.x);
                // the run's rows, gathered by every lane before the column loop
                // (whose trip count differs between lanes: no warp collective in
                // it).  nr is warp-uniform; both loops stay unrolled so run[]
                // lives in registers, and leave after nr rows instead of
                // predicating all 16 (16 compares and addresses per 16 codes)
                int run[MOE_MAX_TOPK];
                const int nr = __popc(same);
                unsigned m = same;
#pragma unroll
                for (int j = 0; j < MOE_MAX_TOPK; ++j) {
                    if (j >= nr) break;
                    run[j] = __shfl_sync(0xffffffffu, r, __ffs(m) - 1);
                    m &= m - 1u;
                }
                for (int q = q0 + lane; q < q1; q += 32) {
                    const uint4 c = par.x == 0.0f
                                        ? make_uint4(0u, 0u, 0u, 0u)
                                        : quant16(row + 32 * q, par.y, par.x, rcp);
#pragma unroll
                    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
                        if (j >= nr) break;
                        st_stream_v4(a.out + (long long)run[j] * a.npairs + q, c, pol);
                    }
                }
                if (part == 0 && ((same >> lane) & 1u)) a.scales[r] = par;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[st]);
        }
    }
    // After the role split no block-wide barrier is used (the producer's
    // lane 0 leaves its loop long after the other lanes): completion is
    // counted per warp, each warp reconverged first.
    __syncwarp();
    if (MODE != MOE_FP8_PER_TOKEN) {
        // the last warp to finish resets the group keys (every block read
        // them before its role split, so before any of its warps' tickets)
        unsigned last = 0;
        if (lane == 0) {
            __threadfence();
            const unsigned done = atomicAdd(&h->quant_ticket, 1u);
            last = (done == gridDim.x * (blockDim.x / 32) - 1) ? 1u : 0u;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            for (int g = lane; g < ngroups; g += 32) {
                h->quant_max[g] = 0u;
                h->quant_min[g] = 0u;
            }
            if (lane == 0) h->quant_ticket = 0u;
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
    const uint64_t pol = l2_stream_policy(false);
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
                        if (c0 + 32 * u < n16) cv[j][u] = ld_stream_v4(src + c0 + 32 * u, pol);
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
                    const uint4 a = ld_stream_v4(sh, pol), b = ld_stream_v4(sh + 1, pol);
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
                st_stream_v4(yr, o0, pol);
                st_stream_v4(yr + 1, o1, pol);
            }
        }
    }
}

template <int MODE, bool TOKENS>
cudaError_t launch_encode(const void *src, long long n_src, int H, const moe_layout *L, void *out, float *scales,
                          cudaStream_t s)
{
    EncArgs a;
    a.src = static_cast<const unsigned char *>(src);
    a.n_src = n_src;
    a.rowbytes = 2 * H;
    a.npairs = H / 16;
    a.k = L->k;
    a.dst_row = L->dst_row;
    a.offsets = L->offsets;
    a.E = L->E;
    a.r_max = L->r_max;
    a.out = static_cast<uint4 *>(out);
    a.scales = reinterpret_cast<float2 *>(scales);
    a.ws = L->ws;
    // consumer warps: 8 while 8 rows fit the ring, else fewer; stages: the
    // largest multiple of the consumer count that fits (at most 16).  Rows of
    // expert outputs are shared by two consumer warps (each half the
    // columns, two stages per pair); token rows keep one warp per row.
    // Measured on GB300 (65536 x 4096): the expert-side quantise 295.8 ->
    // 286.2 us with pairs, the per-token dispatch 177.6 -> 185.0 us (and
    // the per-expert one 277 -> 296 us), so only the former takes them.
    int c = kEncMaxConsumers;
    while (c > 1 && (long long)c * a.rowbytes > kEncRingBytes) c >>= 1;
    int stages = (int)(kEncRingBytes / a.rowbytes) / c * c;
    if (stages > kEncMaxStages) stages = kEncMaxStages / c * c;
    if (stages < c) stages = c;
    a.consumers = c;
    a.group = (!TOKENS && c >= 2 && a.npairs >= 64) ? 2 : 1;
    a.stages = stages;  // a multiple of c, so of the group count
    const int threads = 32 * (c + 1);
    const void *fn = reinterpret_cast<const void *>(fp8_encode_kernel<MODE, TOKENS>);
    const size_t smem = (size_t)a.stages * a.rowbytes;
    cudaError_t err = allow_dynamic_smem(fn, (int)smem);
    if (err != cudaSuccess) return err;
    const long long resident = resident_grid(fn, threads, smem);
    const unsigned grid = (unsigned)(n_src < resident ? (n_src < 1 ? 1 : n_src) : resident);
    return launch_pdl(fp8_encode_kernel<MODE, TOKENS>, dim3(grid), dim3(threads), smem, s, a);
}

template <int MODE, bool TOKENS>
cudaError_t launch_grouped(const void *src, long long n_src, int H, const moe_layout *L, void *out, float *scales,
                           cudaStream_t s)
{
    const int nvec = H / 8;
    cudaError_t err = cudaSuccess;
    if (MODE != MOE_FP8_PER_TOKEN) {
        const int r = resident_grid(reinterpret_cast<const void *>(fp8_group_stats_kernel<MODE, TOKENS>), kStatThreads, 0);
        const long long need = (n_src + kStatThreads / 32 - 1) / (kStatThreads / 32);
        const unsigned grid = (unsigned)(need < r ? (need < 1 ? 1 : need) : r);
        err = launch_pdl(fp8_group_stats_kernel<MODE, TOKENS>, dim3(grid), dim3(kStatThreads), 0, s,
                         static_cast<const uint4 *>(src), n_src, nvec, L->k, (const int32_t *)L->dst_row,
                         (const int32_t *)L->offsets, L->E, L->r_max, L->ws);
        if (err != cudaSuccess) return err;
    }
    return launch_encode<MODE, TOKENS>(src, n_src, H, L, out, scales, s);
}

template <int K>
cudaError_t launch_cfp8_k(const void *codes, const float *scales, const moe_layout *L, const float *gates,
                          const void *shared, int Ks, int T, int H, void *y, cudaStream_t s)
{
    constexpr int V = K <= 2 ? 2 : 1;
    const int r = resident_grid(reinterpret_cast<const void *>(combine_fp8_kernel<K, V>), kCombFp8Threads, 0);
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
    if (mode == MOE_FP8_PER_TOKEN) return launch_grouped<MOE_FP8_PER_TOKEN, true>(x, T, H, L, packed, scales, s);
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
