// layout.cu -- moe_dispatch_layout: counts, prefix offsets and the stable
// expert-major permutation of all (token, slot) assignments, in ONE pass.
//
// The layout follows "MoE data traits ... DeepEP and MoE all-to-all data
// handling" sec. 7 (reorder by target expert, pack each destination
// contiguously, keep target/source indices for the combine; sec. 7.5.4: no
// padding rows) and sec. 8.3.A (strict per-expert capacity, assignments
// over it taken in order -- here: dropped, token-index order).
//
// Design (sm_103a): one block per tile of consecutive tokens (1024..8192
// assignments, see layout_tile_tokens), tile ids handed out by an atomic
// counter so that every tile a block waits on has already started.
//   1. Per-expert packed offsets from expert_counts (exclusive scan of
//      min(count, capacity); E <= 256, every block recomputes it).
//   2. Tile-local stable ranks: each warp walks its contiguous slice of the
//      tile 32 assignments at a time; __match_any_sync groups equal expert
//      ids, the rank is the popcount of lower peers plus a per-warp running
//      count in shared memory.  Warp slices are then scanned per expert.
//   3. Decoupled look-back across tiles.  A 64-bit flag word per (tile,
//      expert) carries an epoch tag, a state (aggregate / inclusive prefix)
//      and the 30-bit value, so no flag array ever needs clearing.  The
//      whole block looks back at once: 256/E threads per expert each read
//      and reduce 16 consecutive predecessors' words per round, so a round
//      covers 4096/E tiles for every expert with a single memory round
//      trip.  Every wait is
//      bounded by %globaltimer and records MOE_ERR_TIMEOUT instead of
//      hanging.
//   4. Rank r = prefix + warp offset + local rank; kept iff r < capacity;
//      dst_row / src_pos / capacity_mask written, dropped gates zeroed.
//   5. Distinct-partition tokens: a kept assignment counts when no earlier
//      kept slot of its token falls in the same partition; aggregated per
//      warp (ballot per partition), then summed over tiles with integer
//      atomics; the last block to finish publishes them.  Output stores come last, after the completion
//      ticket, so no fence waits behind them.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kLoadBatch = 8;  // expert-id loads in flight per thread
constexpr int kLookPer = 16;   // look-back words read per thread per round
constexpr int kSpecLoads = kLoadBatch;  // ids of the guessed tile fetched before the tile id is known

struct LayoutArgs {
    const int32_t *idx;
    const int32_t *counts_in;
    int T, E, k, P;
    unsigned cap;  // 0xFFFFFFFF = none
    int r_max;     // rows the packed buffers hold
    int tile_tokens;
    int ntiles;
    float *gates;
    int32_t *counts_out, *offsets, *part_rows, *part_offsets, *part_tokens, *src_pos, *dst_row;
    uint8_t *cmask;
    int64_t *dropped;
    void *ws;
    int reassign;  // capacity overflow re-assigned to the least-loaded expert
};

// Water filling of the overflow (re-assign mode).  Experts are ranked by
// (kept load L_e, id); the places left below capacity are the slots
// (level, expert) with level in [L_e, C), taken in (level, expert) order.
// Segment i of the levels, [L_(i), L_(i+1)) (L_(E) = C), has the i+1 lowest
// ranked experts active; G_i = slots below level L_(i).
struct WaterFill {
    int Ls[MOE_MAX_EXPERTS + 1];          // sorted kept loads, Ls[E] = C
    long long G[MOE_MAX_EXPERTS + 1];     // slots below segment i
    unsigned mask[MOE_MAX_EXPERTS][8];    // experts of rank <= i (bit per id)
    int rank[MOE_MAX_EXPERTS];            // rank of each expert
};

// j-th set bit (0-based) of a 256-bit mask.
__device__ __forceinline__ int select_bit(const unsigned (&m)[8], int j)
{
    for (int w = 0; w < 8; ++w) {
        const int c = __popc(m[w]);
        if (j < c) {
            unsigned v = m[w];
            for (int q = 0; q < j; ++q) v &= v - 1u;
            return w * 32 + __ffs(v) - 1;
        }
        j -= c;
    }
    return -1;
}

// Slot m (< G[E]) -> (level, expert).
__device__ __forceinline__ void water_slot(const WaterFill &wf, int E, long long m, int &level, int &expert)
{
    int lo = 0, hi = E - 1;  // largest i with G[i] <= m
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (wf.G[mid] <= m) lo = mid;
        else hi = mid - 1;
    }
    const long long off = m - wf.G[lo];
    level = wf.Ls[lo] + (int)(off / (lo + 1));
    expert = select_bit(wf.mask[lo], (int)(off % (lo + 1)));
}

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p)
{
    return *reinterpret_cast<const volatile unsigned long long *>(p);
}
__device__ __forceinline__ void st_volatile_u64(unsigned long long *p, unsigned long long v)
{
    *reinterpret_cast<volatile unsigned long long *>(p) = v;
}

// Add the warp's tokens per partition to s_ptok: one ballot and one shared
// atomic per partition that some lane of the warp reaches (P <= 64), not
// one atomic per (token, partition) on the same few words.  Every lane of
// the warp calls it.
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

__global__ void __launch_bounds__(kLayoutThreads) layout_kernel(LayoutArgs a)
{
    extern __shared__ int s_dyn[];   // s_idx[tile assignments], s_rank[tile assignments]
    __shared__ unsigned s_whist[kLayoutWarps][MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ unsigned s_excl[MOE_MAX_EXPERTS];
    __shared__ int s_base[MOE_MAX_EXPERTS];
    __shared__ unsigned s_ptok[MOE_MAX_EXPERTS];
    __shared__ int s_epart[MOE_MAX_EXPERTS];  // partition of each expert
    __shared__ unsigned s_part_add[kLayoutThreads];  // look-back segment sums
    __shared__ int s_part_use[kLayoutThreads];       // words used | stop << 8
    __shared__ unsigned s_warp_tot[kLayoutWarps];
    __shared__ unsigned s_tile, s_epoch;
    __shared__ int s_last, s_bad, s_skip, s_abort;
    __shared__ WaterFill s_wf;               // re-assign mode only
    __shared__ long long s_over, s_overbase;  // overflow before this tile / before the chunk
    __shared__ int s_cscan[kLayoutWarps];

    WsHeader *ws = static_cast<WsHeader *>(a.ws);
    unsigned long long *flags = ws_flags(a.ws);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, k = a.k;
    int *s_idx = s_dyn;
    int *s_rank = s_dyn + a.tile_tokens * k;

    pdl_wait();
    pdl_launch_dependents();
    const int raw_count = (tid < E) ? __ldg(a.counts_in + tid) : 0;
    if (tid == 0) {
        const unsigned long long te = atomicAdd(&ws->tile_epoch, 1ull);
        s_tile = (unsigned)te;
        s_epoch = (unsigned)(te >> 32);
        // the block that draws the last tile id retires this call's epoch:
        // every other block of the call has drawn (and knows the epoch)
        if (s_tile == (unsigned)a.ntiles - 1)
            atomicExch(&ws->tile_epoch, (unsigned long long)(s_epoch + 1u) << 32);
        s_bad = 0;
        s_abort = 0;
        s_skip = (*reinterpret_cast<volatile unsigned *>(&ws->inject_skip_publish) == s_tile + 1u);
    }
    for (int i = tid; i < kLayoutWarps * MOE_MAX_EXPERTS; i += kLayoutThreads)
        (&s_whist[0][0])[i] = 0u;
    for (int p = tid; p < a.P; p += kLayoutThreads) s_ptok[p] = 0u;
    const int per = E / a.P;
    for (int e = tid; e < E; e += kLayoutThreads) s_epart[e] = e / per;

    // Tiles are drawn in launch order, so this block almost always gets tile
    // blockIdx.x: fetch that tile's expert ids while the tile-id atomic is in
    // flight, and fetch again only if the guess was wrong.
    int v[kSpecLoads];
    {
        const long long g0 = (long long)blockIdx.x * a.tile_tokens;
        const long long g1 = min((long long)a.T, g0 + a.tile_tokens);
        const int gA = (int)(max(0LL, g1 - g0) * k);
#pragma unroll
        for (int u = 0; u < kSpecLoads; ++u) {
            const int i = u * kLayoutThreads + tid;
            if (i < gA) v[u] = __ldg(a.idx + g0 * k + i);
        }
    }
    __syncthreads();

    const unsigned tile = s_tile, epoch = s_epoch;
    if (tile >= (unsigned)a.ntiles) {  // workspace not clean: refuse to touch outputs
        if (tid == 0) record_status(a.ws, MOE_ERR_DEVICE_DATA);
        return;
    }
    const long long tok0 = (long long)tile * a.tile_tokens;
    const long long tok1 = min((long long)a.T, tok0 + a.tile_tokens);
    const long long a0 = tok0 * k;
    const int A = (int)(max(0LL, tok1 - tok0) * k);

    // the tile's expert ids (kLoadBatch loads in flight per thread); ids
    // outside [0, E) become the sentinel E
    const bool guessed = (tile == blockIdx.x);
    for (int base = 0; base < A; base += kLoadBatch * kLayoutThreads) {
        int w[kLoadBatch];
        const bool spec = guessed && base == 0;
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int i = base + u * kLayoutThreads + tid;
            if (i < A) w[u] = spec ? v[u] : __ldg(a.idx + a0 + i);
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int i = base + u * kLayoutThreads + tid;
            if (i < A) {
                int e = w[u];
                if (e == -1) e = E;  // empty slot
                else if (e < 0 || e >= E) { e = E; s_bad = 1; }
                s_idx[i] = e;
            }
        }
    }

    // 1. packed offsets: exclusive scan of kept counts (block-wide, E <= 256);
    // in re-assign mode of the final loads after the water filling.
    long long total_slots = 0;
    {
        int c = 0;
        if (tid < E) {
            int raw = raw_count;
            if (raw < 0 || (long long)raw > (long long)a.T * k) { raw = 0; s_bad = 1; }
            c = ((unsigned)raw < a.cap) ? raw : (int)a.cap;
        }
        if (a.reassign) {
            const int C = (int)a.cap;
            // overflow total and the expert ranks by (kept load, id)
            const long long over = tid < E ? (long long)(max(raw_count, 0) - c) : 0;
            long long o = over;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) o += __shfl_xor_sync(0xffffffffu, o, d);
            if (tid == 0) s_over = 0;
            if (tid < E) s_wf.Ls[tid] = c;  // kept loads by id, for the ranking
            __syncthreads();
            if (lane == 0 && o) atomicAdd(reinterpret_cast<unsigned long long *>(&s_over), (unsigned long long)o);
            int rk = 0;
            if (tid < E)
                for (int e2 = 0; e2 < E; ++e2) {
                    const int l2 = s_wf.Ls[e2];
                    rk += (l2 < c) || (l2 == c && e2 < tid);
                }
            __syncthreads();
            if (tid < E) {
                s_wf.rank[tid] = rk;
                s_wf.Ls[rk] = c;
                s_wf.G[rk] = tid;  // expert of rank rk (temporarily)
            }
            if (tid == 0) s_wf.Ls[E] = C;
            __syncthreads();
            if (tid < 8) {  // active-set masks, word tid
                unsigned m = 0u;
                for (int i = 0; i < E; ++i) {
                    const int e2 = (int)s_wf.G[i];
                    if ((e2 >> 5) == tid) m |= 1u << (e2 & 31);
                    s_wf.mask[i][tid] = m;
                }
            }
            __syncthreads();
            if (tid == 0) {
                long long g = 0;
                for (int i = 0; i <= E; ++i) {
                    const long long gi = g;
                    if (i < E) g += (long long)(i + 1) * (s_wf.Ls[i + 1] - s_wf.Ls[i]);
                    s_wf.G[i] = gi;
                }
                s_wf.G[E] = g;  // every place left below capacity
            }
            __syncthreads();
            total_slots = s_wf.G[E];
            if (tid < E) {
                // final load: the slots of the first s_over places in (level, expert) order
                const long long O = s_over;
                if (O >= total_slots) {
                    c = C;
                } else {
                    int lvO, eO;
                    water_slot(s_wf, E, O, lvO, eO);
                    (void)eO;
                    // slot O is at (lvO, position pO among the active experts by id)
                    int lo = 0, hi = E - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (s_wf.G[mid] <= O) lo = mid;
                        else hi = mid - 1;
                    }
                    const int pO = (int)((O - s_wf.G[lo]) % (lo + 1));
                    int cc = max(c, lvO);
                    if (s_wf.rank[tid] <= lo) {
                        int idpos = 0;
                        for (int w2 = 0; w2 < 8; ++w2) {
                            const unsigned mw = s_wf.mask[lo][w2];
                            if (w2 < (tid >> 5)) idpos += __popc(mw);
                            else if (w2 == (tid >> 5)) idpos += __popc(mw & ((1u << (tid & 31)) - 1u));
                        }
                        if (idpos < pO) ++cc;
                    }
                    c = min(cc, C);
                }
            }
        }
        int incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += n;
        }
        if (lane == 31) s_warp_tot[warp] = (unsigned)incl;
        __syncthreads();  // also publishes s_idx
        int base = 0;
        for (int w = 0; w < warp; ++w) base += (int)s_warp_tot[w];
        if (tid < E) s_off[tid] = base + incl - c;
        if (tid == E - 1) s_off[E] = base + incl;
    }

    // 2. tile-local stable ranks
    const int per_warp = (((A + kLayoutWarps - 1) / kLayoutWarps) + 31) & ~31;
    {
        const int wb = warp * per_warp;
        const int we = min(A, wb + per_warp);
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = wb; base < we; base += 32) {
            const int i = base + lane;
            const bool valid = i < we;
            const int e = valid ? s_idx[i] : E;
            const bool counted = e < E;
            const unsigned peers = __match_any_sync(0xffffffffu, counted ? e : -1);
            const unsigned rank = __popc(peers & lt_mask);
            const unsigned before = counted ? s_whist[warp][e] : 0u;
            __syncwarp();
            if (counted && rank == 0) s_whist[warp][e] = before + __popc(peers);
            __syncwarp();
            if (valid) s_rank[i] = counted ? (int)(((unsigned)warp << 24) | (before + rank)) : -1;
        }
    }
    __syncthreads();

    // per-expert scan across warps -> warp offsets, tile aggregate; publish
    // the aggregate (tile 0: the inclusive prefix) right away
    unsigned agg = 0;
    const bool publish = !s_skip;
    if (tid < E) {
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            unsigned v = s_whist[w][tid];
            s_whist[w][tid] = agg;
            agg += v;
        }
        unsigned long long *my = flags + (size_t)tile * E + tid;
        if (publish) st_volatile_u64(my, make_flag(epoch, tile == 0 ? kFlagInclusive : kFlagAggregate, agg));
        s_excl[tid] = 0u;
        s_base[tid] = (int)tile - 1;  // next predecessor to read; -1 = prefix complete
    }
    __syncthreads();

    // 3. block-wide decoupled look-back.  Thread (e = tid % E, w = tid / E),
    // w < W = 256/E, reads kLookPer consecutive predecessors of expert e
    // (coalesced across e) and walks them itself: the sum of the aggregates
    // up to its first inclusive prefix or its first word not yet published.
    // One thread per expert then joins the W segments in order, so a round
    // covers W * kLookPer tiles for every expert with one memory round trip.
    {
        const int W = kLayoutThreads / E;  // threads per expert
        const int my_e = tid % E, my_w = tid / E;
        unsigned long long t_start = 0;
        while (true) {
            if (my_w < W) {
                const int b = s_base[my_e];
                if (b >= 0) {
                    unsigned long long f[kLookPer];
#pragma unroll
                    for (int q = 0; q < kLookPer; ++q) {
                        const int p = b - (my_w * kLookPer + q);
                        f[q] = (p >= 0) ? ld_volatile_u64(flags + (size_t)p * E + my_e)
                                        : make_flag(epoch, kFlagInclusive, 0u);
                    }
                    unsigned add = 0;
                    int used = 0, stop = 0;  // stop: 1 = not published yet, 2 = inclusive prefix
#pragma unroll
                    for (int q = 0; q < kLookPer; ++q) {
                        if (stop) continue;
                        const unsigned state = (unsigned)(f[q] >> 30) & 3u;
                        if ((unsigned)(f[q] >> 32) != epoch || state == 0u) {
                            stop = 1;
                        } else {
                            add += (unsigned)(f[q] & 0x3FFFFFFFull);
                            ++used;
                            if (state == (unsigned)kFlagInclusive) stop = 2;
                        }
                    }
                    s_part_add[tid] = add;
                    s_part_use[tid] = used | (stop << 8);
                }
            }
            __syncthreads();
            int open = 0;
            if (tid < E && s_base[tid] >= 0) {
                unsigned add = 0;
                int used = 0;
                bool done = false;
                for (int w = 0; w < W; ++w) {
                    const int u = s_part_use[w * E + tid];
                    add += s_part_add[w * E + tid];
                    used += u & 0xFF;
                    if ((u >> 8) == 2) { done = true; break; }
                    if ((u >> 8) == 1) break;
                }
                s_excl[tid] += add;
                s_base[tid] = done ? -1 : s_base[tid] - used;
                open = !done;
            }
            if (!__syncthreads_or(open)) break;
            if (tid == 0) {
                const unsigned long long now = global_timer_ns();
                if (t_start == 0) t_start = now;
                else if (now - t_start > kSpinLimitNs ||
                         *reinterpret_cast<volatile unsigned *>(&ws->status) == MOE_ERR_TIMEOUT) {
                    record_status(a.ws, MOE_ERR_TIMEOUT);
                    s_abort = 1;
                }
            }
            __syncthreads();
            if (s_abort) break;
        }
    }
    if (tid < E) {
        const unsigned excl = s_excl[tid];
        if (tile > 0 && publish)
            st_volatile_u64(flags + (size_t)tile * E + tid, make_flag(epoch, kFlagInclusive, excl + agg));
        if (tile == (unsigned)a.ntiles - 1 && (int)(excl + agg) != raw_count) s_bad = 1;
    }
    __syncthreads();

    // 4+5. ranks -> rows, one thread per token, kept in shared memory first
    // (the completion step below must not wait behind this block's output
    // stores); s_rank[i] becomes the packed row or -1.  A token counts once
    // for every partition holding at least one of its kept slots (partition
    // bitmask when P <= 64, pairwise check otherwise).
    const int ntok = (int)max(0LL, tok1 - tok0);
    if (a.reassign) {
        // Overflow assignments (global rank >= C) are numbered in flat order
        // across the batch: those of earlier tiles (per expert, its count
        // before this tile beyond C), then this tile's in token order (a
        // block scan per chunk of tokens).  Number m takes water-fill slot m
        // if m < total_slots, else the assignment is dropped.
        if (tid == 0) s_overbase = 0;
        __syncthreads();
        long long ob = (tid < E) ? max(0LL, (long long)s_excl[tid] - (long long)a.cap) : 0;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) ob += __shfl_xor_sync(0xffffffffu, ob, d);
        if (lane == 0 && ob) atomicAdd(reinterpret_cast<unsigned long long *>(&s_overbase), (unsigned long long)ob);
        __syncthreads();
        long long base = s_overbase;
        for (int c0 = 0; c0 < ntok; c0 += kLayoutThreads) {
            const int tl = c0 + tid;
            int nov = 0;
            if (tl < ntok) {
                for (int j = 0; j < k; ++j) {
                    const int i = tl * k + j;
                    const int e = s_idx[i];
                    if (e < E) {
                        const unsigned pr = (unsigned)s_rank[i];
                        const unsigned r = s_excl[e] + s_whist[pr >> 24][e] + (pr & 0xFFFFFFu);
                        nov += r >= a.cap;
                    }
                }
            }
            // exclusive scan of nov over the chunk, in token order
            int incl = nov;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += n;
            }
            if (lane == 31) s_cscan[warp] = incl;
            __syncthreads();
            int wbase = 0, ctot = 0;
            for (int w2 = 0; w2 < kLayoutWarps; ++w2) {
                if (w2 < warp) wbase += s_cscan[w2];
                ctot += s_cscan[w2];
            }
            long long m = base + wbase + incl - nov;
            unsigned long long pmask = 0ull;
            if (tl < ntok) {
                int fe[MOE_MAX_TOPK];
                for (int j = 0; j < k; ++j) {
                    const int i = tl * k + j;
                    const int e = s_idx[i];
                    int row = -1, fin = -1;
                    bool moved = false;
                    if (e < E) {
                        const unsigned pr = (unsigned)s_rank[i];
                        const unsigned r = s_excl[e] + s_whist[pr >> 24][e] + (pr & 0xFFFFFFu);
                        if (r < a.cap) {
                            const int cand = s_off[e] + (int)r;
                            if (cand < s_off[e + 1] && cand < a.r_max) { row = cand; fin = e; }
                            else s_bad = 1;
                        } else {
                            if (m < total_slots) {
                                int lv, e2;
                                water_slot(s_wf, E, m, lv, e2);
                                const int cand = s_off[e2] + lv;
                                if (e2 >= 0 && cand < s_off[e2 + 1] && cand < a.r_max) {
                                    row = cand;
                                    fin = e2;
                                    moved = true;
                                } else {
                                    s_bad = 1;
                                }
                            }
                            ++m;
                        }
                    }
                    fe[j] = fin;
                    s_rank[i] = row < 0 ? -1 : (row | (moved ? 0x40000000 : 0));
                }
                // partitions reached through the final experts
                for (int j = 0; j < k; ++j) {
                    if (fe[j] < 0) continue;
                    const int p = s_epart[fe[j]];
                    if (a.P <= 64) {
                        pmask |= 1ull << p;
                        continue;
                    }
                    bool first = true;
                    for (int jj = 0; jj < j; ++jj)
                        if (fe[jj] >= 0 && s_epart[fe[jj]] == p) { first = false; break; }
                    if (first) atomicAdd(&s_ptok[p], 1u);
                }
            }
            count_partition_tokens(s_ptok, pmask, lane);
            base += ctot;
            __syncthreads();  // s_cscan is rewritten by the next chunk
        }
    } else
    for (int tb = 0; tb < ntok; tb += kLayoutThreads) {
        const int tl = tb + tid;
        unsigned long long pmask = 0ull;
        for (int j = 0; tl < ntok && j < k; ++j) {
            const int i = tl * k + j;
            const int e = s_idx[i];
            int row = -1;
            if (e < E) {
                const unsigned pr = (unsigned)s_rank[i];
                const unsigned r = s_excl[e] + s_whist[pr >> 24][e] + (pr & 0xFFFFFFu);
                if (r < a.cap) {
                    const int cand = s_off[e] + (int)r;
                    if (cand < s_off[e + 1] && cand < a.r_max) row = cand;
                    else s_bad = 1;  // counts do not match the ids: keep writes in bounds
                }
            }
            s_rank[i] = row;
            if (row >= 0) {
                const int p = s_epart[e];
                if (a.P <= 64) {
                    pmask |= 1ull << p;
                } else {
                    bool first = true;
                    for (int jj = 0; jj < j; ++jj) {
                        const int ii = tl * k + jj;
                        if (s_rank[ii] >= 0 && s_epart[s_idx[ii]] == p) { first = false; break; }
                    }
                    if (first) atomicAdd(&s_ptok[p], 1u);
                }
            }
        }
        count_partition_tokens(s_ptok, pmask, lane);
    }
    __syncthreads();
    for (int p = tid; p < a.P; p += kLayoutThreads)
        if (s_ptok[p]) atomicAdd(&ws->part_tok[p], s_ptok[p]);

    // completion: the last tile to get here publishes partition tokens and
    // returns the done counter and the test hook to zero (the tile/epoch word
    // was advanced when the last tile id was drawn)
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&ws->done_ctr, 1u) == (unsigned)a.ntiles - 1);
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int p = tid; p < a.P; p += kLayoutThreads)
            a.part_tokens[p] = (int32_t)atomicExch(&ws->part_tok[p], 0u);
        if (tid == 0) {
            ws->done_ctr = 0u;
            ws->inject_skip_publish = 0u;
        }
    }

    // outputs of this tile (no block reads the workspace after this point)
    for (int i = tid; i < A; i += kLayoutThreads) {
        const long long as = a0 + i;
        const int v = s_rank[i];
        const int row = v < 0 ? -1 : (v & 0x3FFFFFFF);
        a.dst_row[as] = row;
        a.cmask[as] = (uint8_t)(v < 0 ? 0 : ((v >> 30) ? 2 : 1));  // kept / re-assigned / dropped
        if (row >= 0) a.src_pos[row] = (int32_t)as;
        else if (a.gates) a.gates[as] = 0.0f;
    }
    if (tile == 0) {  // the per-expert / per-partition summary
        for (int e = tid; e < E; e += kLayoutThreads) a.counts_out[e] = s_off[e + 1] - s_off[e];
        for (int e = tid; e <= E; e += kLayoutThreads) a.offsets[e] = s_off[e];
        for (int p = tid; p < a.P; p += kLayoutThreads) {
            a.part_rows[p] = s_off[(p + 1) * per] - s_off[p * per];
            a.part_offsets[p] = s_off[p * per];
        }
        if (tid == 0) {
            a.part_offsets[a.P] = s_off[E];
            *a.dropped = (int64_t)a.T * k - s_off[E];
        }
    }
    __syncthreads();
    if (tid == 0 && s_bad) record_status(a.ws, MOE_ERR_DEVICE_DATA);
}

}  // namespace

cudaError_t launch_layout(const int32_t *topk_idx, const int32_t *counts_in, int T, int E, int k,
                          int P, int capacity, float *gates, const moe_layout *L, void *ws,
                          cudaStream_t s, int reassign)
{
    LayoutArgs a;
    a.reassign = (reassign && capacity > 0) ? 1 : 0;
    a.idx = topk_idx;
    a.counts_in = counts_in;
    a.T = T;
    a.E = E;
    a.k = k;
    a.P = P;
    a.cap = capacity > 0 ? (unsigned)capacity : 0xFFFFFFFFu;
    a.r_max = L->r_max;
    a.tile_tokens = layout_tile_tokens(T, k);
    a.ntiles = layout_tiles(T, k);
    a.gates = gates;
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
    const size_t smem = 2 * sizeof(int) * (size_t)a.tile_tokens * k;
    cudaError_t err = allow_dynamic_smem(reinterpret_cast<const void *>(layout_kernel), (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(layout_kernel, dim3(a.ntiles), dim3(kLayoutThreads), smem, s, a);
}

}  // namespace moe
