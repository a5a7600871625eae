// route.cu -- moe_route: the gate (top-k, gate weights, counts, aux loss,
// entropy) and the dispatch layout (offsets, stable expert-major
// permutation, capacity drops, partitions) in ONE launch.
//
// Definitions are those of moe_gate and moe_dispatch_layout: "DeepSeek MoE
// architecture evolution" ch.1 (top2_gating: top-k, softmax of the selected
// logits, aux = E * sum f_e^2) and sec. 2.3 (entropy of the counts);
// "DeepSeek MoE sync tax" sec. 4.1 (softmax over all experts, then top-k)
// and sec. 4.3 (gate, softmax and top-k fused into one kernel); "MoE data
// traits ... DeepEP and MoE all-to-all data handling" sec. 7 (reorder by
// target expert, contiguous per destination, saved indices) and sec. 8.3.A
// (strict per-expert capacity, in token order).
//
// Why one launch.  The two calls are chains of dependent memory round trips
// with HBM nearly idle (1 MB of logits for 16 K tokens): the gate ends with a
// fence, a completion ticket and a last block that publishes the counts and
// statistics; the layout then starts, draws tiles from a ticket, looks back
// across tiles and ends with another ticket.  Here every tile (block) keeps
// its tokens' expert ids in shared memory, publishes its per-expert
// histogram and adds it to per-expert totals, and then waits ONCE for all
// tiles (a generation-counting barrier word in the workspace, bounded by
// %globaltimer).  After the wait the totals give the offsets, and the
// exclusive prefix of a tile is the sum of the published histograms of the
// tiles before it (all present: no look-back chain).  Tile 0 also writes the
// counts, offsets, partition summary and the statistics.
//
// Co-residency.  The wait needs every block of the grid to be scheduled at
// some point while the others wait.  The host sizes the grid to at most the
// blocks the GPU holds at once (occupancy x SMs), so that holds even when
// other kernels occupy SMs for a while: they finish on their own and free
// their slots.  Should it ever fail, the wait expires after 1 s and records
// MOE_ERR_TIMEOUT; moe_get_status then re-arms the barrier word.
//
// Workspace use: the barrier word and two arrays of per-expert totals
// (selected by the parity of the barrier's generation: a call accumulates
// into one and clears the other for the next call), and one 32-bit count per
// (tile, expert) in a region of its own (the layout kernel's look-back flag
// words are elsewhere, so the two calls may share a workspace).
#include <math.h>

#include "common.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
// Tokens per tile: 512 / k, within [32, 256] (measured on GB300: top-2
// over 16 experts is fastest with 256-token tiles, top-8 over 32 with 32-64:
// the gate's per-token chain grows with k, so smaller tiles spread the
// tokens over more SMs).  A batch that would need more tiles than the GPU
// holds at once does not take the fused kernel (see launch_route).
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kStageLoads = 8;      // logit loads in flight per thread while staging
constexpr int kPrefixUnroll = 32;   // histogram loads in flight per thread in the prefix sums
constexpr int kStageBytes = 68 * 1024;  // staging buffer: one round of 256 tokens up to 64 experts
#ifndef MOE_ROUTE_BALANCE
#define MOE_ROUTE_BALANCE 1  // large batches: tiles sized to the resident slots
#endif
#ifndef MOE_ROUTE_MAX_LANES
#define MOE_ROUTE_MAX_LANES 8   // lanes per token in the gate of a small tile
#endif
#ifndef MOE_ROUTE_INSERT_UNROLL
#define MOE_ROUTE_INSERT_UNROLL 8  // unroll of the one-lane gate's insertion loop
#endif
constexpr int kInsertUnroll = MOE_ROUTE_INSERT_UNROLL;

struct RouteArgs {
    const float *logits;
    int T, E, P;
    unsigned cap;        // 0xFFFFFFFF = none
    int r_max;           // rows the packed buffers hold
    int tile_tokens;     // tokens per tile (block)
    int ntiles;          // = gridDim.x
    int round_tokens;    // tokens staged per gate round (round_tokens * lanes <= kRouteThreads)
    int lanes;           // lanes per token in the gate: 1, 2, 4 or 8
    int32_t *topk_idx;
    float *gates;
    int32_t *expert_counts;
    double *aux, *ent;
    int32_t *counts_out, *offsets, *part_rows, *part_offsets, *part_tokens, *src_pos, *dst_row;
    uint8_t *cmask;
    int64_t *dropped;
    void *ws;
    unsigned *hist;      // [ntiles, E] per-tile histograms (the workspace's route region)
};

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p)
{
    return *reinterpret_cast<const volatile unsigned long long *>(p);
}
__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned *p)
{
    return *reinterpret_cast<const volatile unsigned *>(p);
}

// Insert (v, e) into the descending list bv/bi of length K if it beats the
// last entry.  v goes after every entry >= v, so an equal value keeps the
// lower expert id first (-0.0 == +0.0 is a tie): it enters at the bottom and
// rises while it beats its predecessor strictly, one compare and four
// selects per place.  This chain is K - 1 steps long; the alternative, a
// position counted by independent compares and a shift by independent
// selects, is shorter but takes ~60 % more instructions, and the gate of a
// large batch (256 tokens per round, 8 warps a block) is bound by issue:
// 262144 tokens, 64 experts, top-8: 110 -> 100 us on GB300.
template <int K>
__device__ __forceinline__ void topk_insert(float (&bv)[K], int (&bi)[K], float v, int e)
{
    if (v > bv[K - 1]) {
        bv[K - 1] = v;
        bi[K - 1] = e;
#pragma unroll
        for (int j = K - 1; j > 0; --j) {
            const bool up = bv[j] > bv[j - 1];
            const float hv = up ? bv[j] : bv[j - 1], lv = up ? bv[j - 1] : bv[j];
            const int hx = up ? bi[j] : bi[j - 1], lx = up ? bi[j - 1] : bi[j];
            bv[j - 1] = hv;
            bv[j] = lv;
            bi[j - 1] = hx;
            bi[j] = lx;
        }
    }
}

__host__ __device__ constexpr int pow2_at_least(int k) { return k <= 1 ? 1 : (k <= 2 ? 2 : (k <= 4 ? 4 : (k <= 8 ? 8 : 16))); }

// Strict total order of (logit, expert): the larger logit first, equal
// logits (-0.0 == +0.0) by the lower expert id.
__device__ __forceinline__ bool beats(float v1, int i1, float v2, int i2)
{
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Sort a list of KP (a power of two) candidates by `beats`, best first:
// a bitonic sorting network, every index static.
template <int KP>
__device__ __forceinline__ void sort_list(float (&bv)[KP], int (&bi)[KP])
{
#pragma unroll
    for (int size = 2; size <= KP; size <<= 1) {
#pragma unroll
        for (int st = size >> 1; st > 0; st >>= 1) {
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                const int l = j ^ st;
                if (l > j) {
                    const bool best_first = (j & size) == 0;
                    const bool sw = best_first ? beats(bv[l], bi[l], bv[j], bi[j]) : beats(bv[j], bi[j], bv[l], bi[l]);
                    if (sw) {
                        const float tv = bv[j]; bv[j] = bv[l]; bv[l] = tv;
                        const int ti = bi[j]; bi[j] = bi[l]; bi[l] = ti;
                    }
                }
            }
        }
    }
}

// The G lanes of a token (adjacent lanes, G a power of two) each hold a
// list of KP candidates sorted by `beats`; after log2(G) butterfly rounds
// every lane holds the top KP of the union.  A round takes the partner's
// list, keeps the better of mine[j] and partner[KP-1-j] (the top KP of the
// two, as a bitonic sequence) and sorts it with a bitonic merge.  The order
// is total, so both lanes of a pair end with the same list.
template <int KP>
__device__ __forceinline__ void merge_lanes(float (&bv)[KP], int (&bi)[KP], int G)
{
    for (int m = 1; m < G; m <<= 1) {
        float pv[KP];
        int pi[KP];
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            pv[j] = __shfl_xor_sync(0xffffffffu, bv[j], m);
            pi[j] = __shfl_xor_sync(0xffffffffu, bi[j], m);
        }
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            if (!beats(bv[j], bi[j], pv[KP - 1 - j], pi[KP - 1 - j])) {
                bv[j] = pv[KP - 1 - j];
                bi[j] = pi[KP - 1 - j];
            }
        }
#pragma unroll
        for (int st = KP / 2; st > 0; st >>= 1) {
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                if ((j & st) == 0 && beats(bv[j + st], bi[j + st], bv[j], bi[j])) {
                    const float tv = bv[j]; bv[j] = bv[j + st]; bv[j + st] = tv;
                    const int ti = bi[j]; bi[j] = bi[j + st]; bi[j + st] = ti;
                }
            }
        }
    }
}

// log2 of a positive, finite double: its binary exponent plus log2f of the
// mantissa in [1, 2) (absolute error ~1e-7), with no fp64 transcendental.
__device__ __forceinline__ double log2_via_mantissa(double x)
{
    const long long bits = __double_as_longlong(x);
    const int ex = (int)((bits >> 52) & 0x7FF) - 1023;
    const double m = __longlong_as_double((bits & 0x000FFFFFFFFFFFFFll) | 0x3FF0000000000000ll);
    return (double)ex + (double)log2f((float)m);
}

// 1/x for a positive double: the fp32 reciprocal refined by two
// Newton-Raphson steps (24 -> 48 -> 53 correct bits).
__device__ __forceinline__ double rcp_newton(double x)
{
    double r = (double)__frcp_rn((float)x);
    r = r * (2.0 - x * r);
    r = r * (2.0 - x * r);
    return r;
}

// Add the warp's tokens per partition to s_ptok: one ballot and one shared
// atomic per partition some lane reaches (P <= 64).  Every lane calls it.
__device__ __forceinline__ void count_partition_tokens(unsigned *s_ptok, unsigned long long pmask, int lane)
{
    const unsigned lo = __reduce_or_sync(0xffffffffu, (unsigned)pmask);
    const unsigned hi = __reduce_or_sync(0xffffffffu, (unsigned)(pmask >> 32));
    unsigned long long wm = ((unsigned long long)hi << 32) | lo;
    while (wm) {
        const int p = __ffsll((long long)wm) - 1;
        wm &= wm - 1ull;
        const unsigned b = __ballot_sync(0xffffffffu, (unsigned)(pmask >> p) & 1u);
        if (lane == 0) atomicAdd(&s_ptok[p], (unsigned)__popc(b));
    }
}

template <int K, int MODE>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a)
{
    extern __shared__ int s_dyn[];  // s_idx[tile_tokens*K], then the staging buffer / s_rank
    __shared__ unsigned s_whist[kRouteWarps][MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ unsigned s_excl[MOE_MAX_EXPERTS];
    __shared__ unsigned s_tot[MOE_MAX_EXPERTS];
    __shared__ unsigned s_ptok[MOE_MAX_EXPERTS];
    __shared__ int s_epart[MOE_MAX_EXPERTS];
    __shared__ unsigned s_part_add[kRouteThreads];
    __shared__ unsigned s_warp_tot[kRouteWarps];
    __shared__ long long s_fix[kRouteWarps];
    __shared__ unsigned long long s_sq[kRouteWarps];
    __shared__ unsigned s_gen;
    __shared__ int s_bad, s_abort, s_skip;

    WsHeader *ws = static_cast<WsHeader *>(a.ws);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E;
    const int tile = blockIdx.x;
    const long long tok0 = (long long)tile * a.tile_tokens;
    const long long tok1 = min((long long)a.T, tok0 + a.tile_tokens);
    const int ntok = (int)max(0LL, tok1 - tok0);
    const int A = ntok * K;
    const int stride = E | 1;
    int *s_idx = s_dyn;
    float *s_stage = reinterpret_cast<float *>(s_dyn + a.tile_tokens * K);
    int *s_rank = s_dyn + a.tile_tokens * K;  // reuses the staging buffer after the gate phase

    for (int i = tid; i < kRouteWarps * MOE_MAX_EXPERTS; i += kRouteThreads) (&s_whist[0][0])[i] = 0u;
    for (int p = tid; p < MOE_MAX_EXPERTS; p += kRouteThreads) s_ptok[p] = 0u;
    const int per = E / a.P;
    for (int e = tid; e < E; e += kRouteThreads) s_epart[e] = e / per;
    if (tid == 0) {
        // the tile's logits are contiguous: ask L2 for them while the
        // previous kernel in the stream finishes (a hint, safe before the wait)
        const char *src = reinterpret_cast<const char *>(a.logits + tok0 * (long long)E);
        const long long bytes = ((long long)ntok * E * (long long)sizeof(float)) & ~15LL;
        for (long long o = 0; o < bytes; o += 32768)
            bulk_prefetch_l2(src + o, (uint32_t)min(32768LL, bytes - o));
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) {
        // the previous call on this workspace has completed: the generation
        // is stable until this call's barrier releases
        s_gen = (unsigned)(ld_volatile_u64(&ws->route_bar) >> 32);
        s_bad = 0;
        s_abort = 0;
        s_skip = (ld_volatile_u32(&ws->inject_skip_publish) == (unsigned)tile + 1u);
    }

    // ---- gate: rounds of round_tokens tokens, one thread per token --------
    for (int r0 = 0; r0 < ntok; r0 += a.round_tokens) {
        const int rows = min(a.round_tokens, ntok - r0);
        {   // stage the round's rows (contiguous in memory: one flat copy)
            const float *src = a.logits + (tok0 + r0) * (long long)E;
            const int n = rows * E;
            if ((E & 3) == 0) {
                const float4 *src4 = reinterpret_cast<const float4 *>(src);
                const int n4 = n >> 2;
                for (int base = 0; base < n4; base += kStageLoads * kRouteThreads) {
                    float4 v[kStageLoads];
#pragma unroll
                    for (int u = 0; u < kStageLoads; ++u) {
                        const int i = base + u * kRouteThreads + tid;
                        if (i < n4) v[u] = __ldg(src4 + i);
                    }
#pragma unroll
                    for (int u = 0; u < kStageLoads; ++u) {
                        const int i = base + u * kRouteThreads + tid;
                        if (i < n4) {
                            const int r = (4 * i) / E, c = 4 * i - r * E;
                            float *d = s_stage + r * stride + c;
                            d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
                        }
                    }
                }
            } else {
                for (int base = 0; base < n; base += kStageLoads * kRouteThreads) {
                    float v[kStageLoads];
#pragma unroll
                    for (int u = 0; u < kStageLoads; ++u) {
                        const int i = base + u * kRouteThreads + tid;
                        if (i < n) v[u] = __ldg(src + i);
                    }
#pragma unroll
                    for (int u = 0; u < kStageLoads; ++u) {
                        const int i = base + u * kRouteThreads + tid;
                        if (i < n) {
                            const int r = i / E;
                            s_stage[r * stride + (i - r * E)] = v[u];
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (a.lanes > 1) {
            // G lanes per token: lane `sub` takes a contiguous chunk of the row
            constexpr int KP = pow2_at_least(K);
            const int G = a.lanes;
            const int tk = tid / G, sub = tid - tk * G;
            const bool active = tk < rows;
            const float *row = s_stage + (active ? tk : 0) * stride;
            const int chunk = (E + G - 1) / G;
            const int e0 = sub * chunk, e1 = min(E, e0 + chunk);
            float bv[KP];
            int bi[KP];
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                bv[j] = -INFINITY;
                bi[j] = 0x40000000 + sub * KP + j;  // empty places: lose to every expert
            }
            bool finite = true;
            if (e1 - e0 <= KP) {
                // the chunk fits the list: take it whole and sort it
#pragma unroll
                for (int j = 0; j < KP; ++j) {
                    if (e0 + j < e1) {
                        bv[j] = row[e0 + j];
                        bi[j] = e0 + j;
                        finite &= isfinite(bv[j]);
                    }
                }
                sort_list<KP>(bv, bi);
            } else {
                for (int e = e0; e < e1; ++e) {
                    const float v = row[e];
                    finite &= isfinite(v);
                    topk_insert<KP>(bv, bi, v, e);
                }
            }
            merge_lanes<KP>(bv, bi, G);
            const float m = bv[0];
            // the softmax denominator: SOFTMAX_TOPK over every logit (each lane
            // its chunk), TOPK_SOFTMAX over the selected ones (each lane the
            // slots j = sub, sub + G, ...); then a butterfly over the G lanes
            // (every lane adds the same pairs, so every lane has the same total)
            float part = 0.0f;
            if constexpr (MODE != MOE_TOPK_SOFTMAX) {
                for (int e = e0; e < e1; ++e) part = __fadd_rn(part, expf(__fsub_rn(row[e], m)));
            } else {
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (j % G == sub) part = __fadd_rn(part, expf(__fsub_rn(bv[j], m)));
            }
            for (int mm = 1; mm < G; mm <<= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, mm));
            if (active) {
                if (!finite) s_bad = 1;
                const long long t = tok0 + r0 + tk;
                int *si = s_idx + (r0 + tk) * K;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (j % G != sub) continue;  // lane `sub` writes slots sub, sub + G, ...
                    int id = bi[j];
                    if (id < 0 || id >= E) {  // only with non-finite logits (already reported)
                        id = 0;
                        s_bad = 1;
                    }
                    a.topk_idx[t * K + j] = id;
                    a.gates[t * K + j] = __fdiv_rn(expf(__fsub_rn(bv[j], m)), part);
                    si[j] = id;
                }
            }
        } else if (tid < rows) {
            const float *row = s_stage + tid * stride;
            float bv[K];
            int bi[K];
            bool finite = true;
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
#pragma unroll (kInsertUnroll)
            for (int e = K; e < E; ++e) {
                const float v = row[e];
                finite &= isfinite(v);
                topk_insert<K>(bv, bi, v, e);
            }
            if (!finite) s_bad = 1;
            float g[K];
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
            const long long t = tok0 + r0 + tid;
            int *si = s_idx + (r0 + tid) * K;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                a.topk_idx[t * K + j] = bi[j];
                a.gates[t * K + j] = g[j];
                si[j] = bi[j];
            }
        }
        __syncthreads();  // the next round overwrites the staging buffer
    }

    // ---- tile-local stable ranks (flat assignment order = token order) ----
    const int per_warp = (((A + kRouteWarps - 1) / kRouteWarps) + 31) & ~31;
    {
        const int wb = warp * per_warp;
        const int we = min(A, wb + per_warp);
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = wb; base < we; base += 32) {
            const int i = base + lane;
            const bool valid = i < we;
            const int e = valid ? s_idx[i] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const unsigned rank = __popc(peers & lt_mask);
            const unsigned before = valid ? s_whist[warp][e] : 0u;
            __syncwarp();
            if (valid && rank == 0) s_whist[warp][e] = before + __popc(peers);
            __syncwarp();
            if (valid) s_rank[i] = (int)(((unsigned)warp << 24) | (before + rank));
        }
    }
    __syncthreads();

    // per-expert scan across warps -> warp offsets and the tile's histogram,
    // published and added to this call's totals
    const unsigned gen = s_gen;
    const int parity = (int)(gen & 1u);
    if (tid < E) {
        unsigned agg = 0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) {
            const unsigned v = s_whist[w][tid];
            s_whist[w][tid] = agg;
            agg += v;
        }
        *reinterpret_cast<volatile unsigned *>(a.hist + (size_t)tile * E + tid) = agg;
        if (agg) atomicAdd(&ws->route_counts[parity][tid], agg);
    }
    if (tile == 0) {
        // the other total array is next call's: clear it (the call that last
        // used it has completed); this call's partition tokens start at 0
        for (int e = tid; e < MOE_MAX_EXPERTS; e += kRouteThreads) ws->route_counts[parity ^ 1][e] = 0u;
        for (int p = tid; p < a.P; p += kRouteThreads) a.part_tokens[p] = 0;
    }
    __threadfence();
    __syncthreads();

    // ---- the one grid-wide wait -------------------------------------------
    if (tid == 0) {
        if (s_skip) {
            // test hook (set only from the host): this tile never arrives, so
            // the others' bounded wait expires; the hook is consumed here
            atomicExch(&ws->inject_skip_publish, 0u);
            s_abort = 1;
        } else {
            const unsigned long long old = atomicAdd(&ws->route_bar, 1ull);
            if ((unsigned)old == (unsigned)a.ntiles - 1u) {
                // last to arrive: release the others and re-arm for the next call
                atomicExch(&ws->route_bar, (unsigned long long)(gen + 1u) << 32);
            } else {
                const unsigned long long t_start = global_timer_ns();
                unsigned ns = 32;
                while ((unsigned)(ld_volatile_u64(&ws->route_bar) >> 32) == gen) {
                    if (global_timer_ns() - t_start > kSpinLimitNs ||
                        ld_volatile_u32(&ws->status) == MOE_ERR_TIMEOUT) {
                        record_status(a.ws, MOE_ERR_TIMEOUT);
                        s_abort = 1;
                        break;
                    }
                    __nanosleep(ns);
                    if (ns < 256) ns <<= 1;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    if (s_abort) return;  // outputs of this tile stay unwritten; the status says why

    // ---- totals -> offsets; histograms of earlier tiles -> exclusive prefix -
    if (tid < E) s_tot[tid] = ld_volatile_u32(&ws->route_counts[parity][tid]);
    {
        const int W = kRouteThreads / E;  // threads per expert
        const int my_e = tid % E, my_w = tid / E;
        if (my_w < W) {
            // every tile wrote its histogram before arriving: all are this call's
            unsigned add = 0;
            for (int b0 = my_w; b0 < tile; b0 += W * kPrefixUnroll) {
                unsigned h[kPrefixUnroll];
#pragma unroll
                for (int u = 0; u < kPrefixUnroll; ++u) {
                    const int b = b0 + u * W;
                    h[u] = b < tile ? ld_volatile_u32(a.hist + (size_t)b * E + my_e) : 0u;
                }
#pragma unroll
                for (int u = 0; u < kPrefixUnroll; ++u) add += h[u];
            }
            s_part_add[tid] = add;
        }
    }
    __syncthreads();
    {
        int c = 0;
        if (tid < E) {
            unsigned excl = 0;
            const int W = kRouteThreads / E;
            for (int w = 0; w < W; ++w) excl += s_part_add[w * E + tid];
            s_excl[tid] = excl;
            const unsigned tot = s_tot[tid];
            c = (tot < a.cap) ? (int)tot : (int)a.cap;
        }
        int incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += n;
        }
        if (lane == 31) s_warp_tot[warp] = (unsigned)incl;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += (int)s_warp_tot[w];
        if (tid < E) s_off[tid] = base + incl - c;
        if (tid == E - 1) s_off[E] = base + incl;
    }
    __syncthreads();

    // ---- rows: one thread per assignment (rank -> row, kept or dropped),
    // written out at once; s_rank[i] becomes the row or -1 --------------
    for (int i = tid; i < A; i += kRouteThreads) {
        const int e = s_idx[i];
        const unsigned pr = (unsigned)s_rank[i];
        const unsigned r = s_excl[e] + s_whist[pr >> 24][e] + (pr & 0xFFFFFFu);
        int row = -1;
        if (r < a.cap) {
            const int cand = s_off[e] + (int)r;
            if (cand < s_off[e + 1] && cand < a.r_max) row = cand;
            else s_bad = 1;  // keep writes in bounds
        }
        s_rank[i] = row;
        const long long as = tok0 * K + i;
        a.dst_row[as] = row;
        a.cmask[as] = (uint8_t)(row >= 0 ? 1 : 0);
        if (row >= 0) a.src_pos[row] = (int32_t)as;
        else a.gates[as] = 0.0f;
    }
    __syncthreads();
    // a token counts once for every partition that holds one of its kept slots
    for (int tb = 0; tb < ntok; tb += kRouteThreads) {
        const int tl = tb + tid;
        unsigned long long pmask = 0ull;
        if (tl < ntok) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int i = tl * K + j;
                if (s_rank[i] < 0) continue;
                const int p = s_epart[s_idx[i]];
                if (a.P <= 64) {
                    pmask |= 1ull << p;
                } else {
                    bool first = true;
                    for (int jj = 0; jj < j; ++jj) {
                        const int ii = tl * K + jj;
                        if (s_rank[ii] >= 0 && s_epart[s_idx[ii]] == p) { first = false; break; }
                    }
                    if (first) atomicAdd(&s_ptok[p], 1u);
                }
            }
        }
        count_partition_tokens(s_ptok, pmask, lane);
    }
    __syncthreads();
    for (int p = tid; p < a.P; p += kRouteThreads)
        if (s_ptok[p]) atomicAdd(reinterpret_cast<unsigned *>(a.part_tokens + p), s_ptok[p]);

    if (tile == 0) {
        // the per-expert / per-partition summary and the statistics:
        //   aux = E * (sum_e c_e^2) / T^2 from the exact integer sum of squares;
        //   entropy = -sum_e p_e log2(p_e + eps), p_e = c_e / N, N = T*K
        //           = log2(N) - (1/N) sum_e c_e log2(c_e + eps*N)
        // with each log2 of a double taken as exponent + log2f(mantissa) and
        // the products summed exactly in 2^-32 fixed point (deterministic).
        for (int e = tid; e < E; e += kRouteThreads) {
            a.expert_counts[e] = (int32_t)s_tot[e];
            a.counts_out[e] = s_off[e + 1] - s_off[e];
        }
        for (int e = tid; e <= E; e += kRouteThreads) a.offsets[e] = s_off[e];
        for (int p = tid; p < a.P; p += kRouteThreads) {
            a.part_rows[p] = s_off[(p + 1) * per] - s_off[p * per];
            a.part_offsets[p] = s_off[p * per];
        }
        const double n_assign = (double)a.T * (double)K;
        const double eps_n = 1e-8 * n_assign;
        long long fix = 0;
        unsigned long long sq = 0ull;
        for (int e = tid; e < E; e += kRouteThreads) {
            const unsigned c = s_tot[e];
            sq += (unsigned long long)c * c;
            if (c) fix += llrint((double)c * log2_via_mantissa((double)c + eps_n) * 4294967296.0);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            fix += __shfl_xor_sync(0xffffffffu, fix, d);
            sq += __shfl_xor_sync(0xffffffffu, sq, d);
        }
        if (lane == 0) {
            s_fix[warp] = fix;
            s_sq[warp] = sq;
        }
        __syncthreads();
        if (tid == 0) {
            long long F = 0;
            unsigned long long SQ = 0ull;
            for (int w = 0; w < kRouteWarps; ++w) {
                F += s_fix[w];
                SQ += s_sq[w];
            }
            a.part_offsets[a.P] = s_off[E];
            *a.dropped = (int64_t)a.T * K - s_off[E];
            if (a.T > 0) {
                const double inv_t = rcp_newton((double)a.T);
                *a.aux = (double)E * ((double)SQ * inv_t * inv_t);
                *a.ent = (log2_via_mantissa(n_assign) * n_assign - (double)F * (1.0 / 4294967296.0)) *
                         rcp_newton(n_assign);
            } else {
                *a.aux = 0.0;
                *a.ent = 0.0;
            }
        }
    }
    __syncthreads();
    if (tid == 0 && s_bad) record_status(a.ws, MOE_ERR_DEVICE_DATA);
}

// dynamic shared memory of a block: expert ids of the tile, then the larger
// of the staging buffer and the tile's ranks
size_t route_smem(int tile_tokens, int K, int round_tokens, int E)
{
    const size_t ids = (size_t)tile_tokens * K * sizeof(int);
    const size_t stage = (size_t)round_tokens * (E | 1) * sizeof(float);
    return ids + (stage > ids ? stage : ids);
}

template <int K, int MODE>
cudaError_t launch_k(RouteArgs a, cudaStream_t s, int *too_large, bool dry_run)
{
    const void *fn = reinterpret_cast<const void *>(route_kernel<K, MODE>);
    const int stride = a.E | 1;
    // gate rounds: a staging buffer of at most kStageBytes
    int rt = kRouteThreads;
    while (rt > 32 && (size_t)rt * stride * sizeof(float) > kStageBytes) rt >>= 1;
    // tiles of 512 / K tokens (at most one gate round per thread) while the
    // grid fits the GPU at once (the wait needs every block), else larger
    long long tt = 512 / K;
    if (tt > kRouteThreads) tt = kRouteThreads;
    if (tt > a.T) tt = a.T;
    tt = (tt + kRouteMinTileTokens - 1) / kRouteMinTileTokens * kRouteMinTileTokens;
    if (tt < kRouteMinTileTokens) tt = kRouteMinTileTokens;
    bool grown = false;
    while (true) {
        long long ntiles = ((long long)a.T + tt - 1) / tt;
        if (ntiles < 1) ntiles = 1;
        size_t smem = route_smem((int)tt, K, (int)min((long long)rt, tt), a.E);
        if (smem > 160 * 1024) {
            // the tile's ids and ranks no longer fit beside the staging
            // buffer: the separate gate and layout kernels take the batch
            // (checked before any runtime call, so none fails)
            *too_large = 1;
            return cudaSuccess;
        }
        cudaError_t err = allow_dynamic_smem(fn, (int)smem);
        if (err != cudaSuccess) return err;
        int resident = resident_grid(fn, kRouteThreads, smem);
        if (ntiles <= resident && ntiles <= kRouteMaxTiles) {
            if (MOE_ROUTE_BALANCE && grown && resident <= kRouteMaxTiles) {
                // the doubling overshoots (262144 tokens, top-8: 256 tiles
                // of 1024 on 304 slots, so some SMs hold two tiles and
                // others one, and the wait takes the slowest); tiles of
                // ceil(T / resident) tokens fill every slot evenly.  They
                // are no larger, so they fit as well.
                const long long tb = ((a.T + resident - 1) / resident + kRouteMinTileTokens - 1) /
                                     kRouteMinTileTokens * kRouteMinTileTokens;
                if (tb < tt) {
                    const size_t sb = route_smem((int)tb, K, (int)min((long long)rt, tb), a.E);
                    const int rb = resident_grid(fn, kRouteThreads, sb);
                    const long long nb = ((long long)a.T + tb - 1) / tb;
                    if (nb <= rb) {
                        tt = tb;
                        ntiles = nb;
                        smem = sb;
                        resident = rb;
                    }
                }
            }
            if (dry_run) return cudaSuccess;
            a.tile_tokens = (int)tt;
            a.ntiles = (int)ntiles;
            // a small tile spreads each token over up to 8 lanes, so that
            // every thread of the block works on the gate
            int lanes = 1;
            while (lanes < MOE_ROUTE_MAX_LANES && (long long)lanes * 2 * tt <= kRouteThreads && lanes * 2 <= a.E)
                lanes *= 2;
            a.lanes = lanes;
            a.round_tokens = (int)min((long long)rt, min(tt, (long long)(kRouteThreads / lanes)));
            return launch_pdl(route_kernel<K, MODE>, dim3((unsigned)ntiles), dim3(kRouteThreads), smem, s, a);
        }
        // fewer, larger tiles (several gate rounds per block).  On its own
        // such a batch is routed faster by the separate kernels (262144
        // tokens, 64 experts, top-8: 102 vs 85 us on GB300), but beside the
        // previous batch's copies the fused kernel disturbs them less (per
        // pipelined batch 2836-2845 vs 2898 us), so it keeps the batch.
        tt += tt;
        grown = true;
    }
}

template <int MODE>
cudaError_t launch_mode(const RouteArgs &a, int k, cudaStream_t s, int *too_large, bool dry_run)
{
    switch (k) {
#define MOE_ROUTE_CASE(KK) \
    case KK: return launch_k<KK, MODE>(a, s, too_large, dry_run);
        MOE_ROUTE_CASE(1) MOE_ROUTE_CASE(2) MOE_ROUTE_CASE(3) MOE_ROUTE_CASE(4)
        MOE_ROUTE_CASE(5) MOE_ROUTE_CASE(6) MOE_ROUTE_CASE(7) MOE_ROUTE_CASE(8)
        MOE_ROUTE_CASE(9) MOE_ROUTE_CASE(10) MOE_ROUTE_CASE(11) MOE_ROUTE_CASE(12)
        MOE_ROUTE_CASE(13) MOE_ROUTE_CASE(14) MOE_ROUTE_CASE(15) MOE_ROUTE_CASE(16)
#undef MOE_ROUTE_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_route(const float *logits, int T, int E, int k, int mode, int P, int capacity,
                         int32_t *topk_idx, float *gates, int32_t *expert_counts, double *aux, double *entropy,
                         const moe_layout *L, void *ws, cudaStream_t s, int *too_large, bool dry_run)
{
    *too_large = 0;
    RouteArgs a = {};
    if (dry_run) {  // only the tiling decision (no pointers are read)
        a.T = T;
        a.E = E;
        a.P = P;
        if (mode == MOE_TOPK_SOFTMAX) return launch_mode<MOE_TOPK_SOFTMAX>(a, k, s, too_large, true);
        return launch_mode<MOE_SOFTMAX_TOPK>(a, k, s, too_large, true);
    }
    a.logits = logits;
    a.T = T;
    a.E = E;
    a.P = P;
    a.cap = capacity > 0 ? (unsigned)capacity : 0xFFFFFFFFu;
    a.r_max = L->r_max;
    a.tile_tokens = a.ntiles = a.round_tokens = 0;  // set by the launcher
    a.topk_idx = topk_idx;
    a.gates = gates;
    a.expert_counts = expert_counts;
    a.aux = aux;
    a.ent = entropy;
    a.counts_out = L->counts;
    a.offsets = L->offsets;
    a.part_rows = L->part_rows;
    a.part_offsets = L->part_offsets;
    a.part_tokens = L->part_tokens;
    a.src_pos = L->src_pos;
    a.dst_row = L->dst_row;
    a.cmask = L->capacity_mask;
    a.dropped = L->dropped;
    a.ws = ws;
    a.hist = ws_route_hist(ws, T, k, E);
    if (mode == MOE_TOPK_SOFTMAX) return launch_mode<MOE_TOPK_SOFTMAX>(a, k, s, too_large, false);
    return launch_mode<MOE_SOFTMAX_TOPK>(a, k, s, too_large, false);
}

}  // namespace moe
