// layout.cu -- moe_dispatch_layout: counts, prefix offsets and the stable
// expert-major permutation of all (token, slot) assignments, in ONE pass.
//
// The layout follows "MoE data traits ... DeepEP and MoE all-to-all data
// handling" sec. 7 (reorder by target expert, pack each destination
// contiguously, keep target/source indices for the combine; sec. 7.5.4: no
// padding rows) and sec. 8.3.A (strict per-expert capacity, assignments
// over it taken in order -- here: dropped, token-index order).
//
// Design (sm_103a): one block per tile of ~1024 consecutive assignments,
// tile ids handed out by an atomic counter so that every tile a block waits
// on has already started.
//   1. Per-expert packed offsets from expert_counts (exclusive scan of
//      min(count, capacity); E <= 256, every block recomputes it).
//   2. Tile-local stable ranks: each warp walks its contiguous slice of the
//      tile 32 assignments at a time; __match_any_sync groups equal expert
//      ids, the rank is the popcount of lower peers plus a per-warp running
//      count in shared memory.  Warp slices are then scanned per expert.
//   3. Decoupled look-back across tiles, one thread per expert column: a
//      64-bit flag word per (tile, expert) carries an epoch tag, a state
//      (aggregate / inclusive prefix) and the 30-bit value, so no flag array
//      ever needs clearing; every wait is bounded by %globaltimer and
//      records MOE_ERR_TIMEOUT instead of hanging.
//   4. Rank r = prefix + warp offset + local rank; kept iff r < capacity;
//      dst_row / src_pos / capacity_mask written, dropped gates zeroed.
//   5. Distinct-partition tokens per tile, summed with integer atomics; the
//      last block to finish publishes them and resets the counters.
#include "common.cuh"

namespace moe {
namespace {

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
};

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p)
{
    return *reinterpret_cast<const volatile unsigned long long *>(p);
}
__device__ __forceinline__ void st_volatile_u64(unsigned long long *p, unsigned long long v)
{
    *reinterpret_cast<volatile unsigned long long *>(p) = v;
}

__global__ void __launch_bounds__(kLayoutThreads) layout_kernel(LayoutArgs a)
{
    __shared__ int s_idx[kLayoutTileAssign];
    __shared__ int s_rank[kLayoutTileAssign];
    __shared__ unsigned s_whist[kLayoutWarps][MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ unsigned s_excl[MOE_MAX_EXPERTS];
    __shared__ unsigned s_ptok[MOE_MAX_EXPERTS];
    __shared__ unsigned s_warp_tot[kLayoutWarps];
    __shared__ unsigned s_tile, s_epoch;
    __shared__ int s_last, s_bad, s_skip;

    WsHeader *ws = static_cast<WsHeader *>(a.ws);
    unsigned long long *flags = ws_flags(a.ws);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, k = a.k;

    if (tid == 0) {
        unsigned ep = *reinterpret_cast<volatile unsigned *>(&ws->epoch);
        __threadfence();
        s_tile = atomicAdd(&ws->tile_ctr, 1u);
        s_epoch = ep;
        s_bad = 0;
        s_skip = (*reinterpret_cast<volatile unsigned *>(&ws->inject_skip_publish) == s_tile + 1u);
    }
    for (int i = tid; i < kLayoutWarps * MOE_MAX_EXPERTS; i += kLayoutThreads)
        (&s_whist[0][0])[i] = 0u;
    for (int p = tid; p < a.P; p += kLayoutThreads) s_ptok[p] = 0u;
    __syncthreads();

    // 1. packed offsets: exclusive scan of kept counts (block-wide, E <= 256).
    {
        int c = 0;
        if (tid < E) {
            int raw = a.counts_in[tid];
            if (raw < 0 || (long long)raw > (long long)a.T * k) { raw = 0; s_bad = 1; }
            c = ((unsigned)raw < a.cap) ? raw : (int)a.cap;
        }
        int incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, incl, d);
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

    const unsigned tile = s_tile, epoch = s_epoch;
    if (tile >= (unsigned)a.ntiles) {  // workspace not clean: refuse to touch outputs
        if (tid == 0) record_status(a.ws, MOE_ERR_DEVICE_DATA);
        return;
    }
    const long long tok0 = (long long)tile * a.tile_tokens;
    const long long tok1 = min((long long)a.T, tok0 + a.tile_tokens);
    const long long a0 = tok0 * k;
    const int A = (int)(max(0LL, tok1 - tok0) * k);

    // load the tile's expert ids; out-of-range ids become the sentinel E
    for (int i = tid; i < A; i += kLayoutThreads) {
        int e = a.idx[a0 + i];
        if (e < 0 || e >= E) { e = E; s_bad = 1; }
        s_idx[i] = e;
    }
    __syncthreads();

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
            if (valid) s_rank[i] = counted ? (int)(before + rank) : -1;
        }
    }
    __syncthreads();

    // per-expert scan across warps -> warp offsets, tile aggregate
    unsigned agg = 0;
    if (tid < E) {
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            unsigned v = s_whist[w][tid];
            s_whist[w][tid] = agg;
            agg += v;
        }
    }

    // 3. decoupled look-back, one thread per expert column
    if (tid < E) {
        unsigned excl = 0;
        unsigned long long *my = flags + (size_t)tile * E + tid;
        const bool publish = !s_skip;
        if (tile == 0) {
            if (publish) st_volatile_u64(my, make_flag(epoch, kFlagInclusive, agg));
        } else {
            if (publish) st_volatile_u64(my, make_flag(epoch, kFlagAggregate, agg));
            long long p = (long long)tile - 1;
            unsigned long long t_start = 0;
            unsigned spins = 0;
            while (p >= 0) {
                const unsigned long long w = ld_volatile_u64(flags + (size_t)p * E + tid);
                const unsigned state = (unsigned)(w >> 30) & 3u;
                if ((unsigned)(w >> 32) == epoch && state != 0u) {
                    excl += (unsigned)(w & 0x3FFFFFFFull);
                    if (state == (unsigned)kFlagInclusive) break;
                    --p;
                    continue;
                }
                if ((++spins & 63u) == 0u) {
                    const unsigned long long now = global_timer_ns();
                    if (t_start == 0) t_start = now;
                    else if (now - t_start > kSpinLimitNs ||
                             *reinterpret_cast<volatile unsigned *>(&ws->status) == MOE_ERR_TIMEOUT) {
                        record_status(a.ws, MOE_ERR_TIMEOUT);
                        break;
                    }
                }
            }
            if (publish) st_volatile_u64(my, make_flag(epoch, kFlagInclusive, excl + agg));
        }
        s_excl[tid] = excl;
        if (tile == (unsigned)a.ntiles - 1 && (int)(excl + agg) != a.counts_in[tid]) s_bad = 1;
    }
    __syncthreads();

    // 4. ranks -> rows
    for (int i = tid; i < A; i += kLayoutThreads) {
        const long long as = a0 + i;
        const int e = s_idx[i];
        int kept = 0;
        if (e < E) {
            const unsigned r = s_excl[e] + s_whist[i / per_warp][e] + (unsigned)s_rank[i];
            if (r < a.cap) {
                const int row = s_off[e] + (int)r;
                if (row < s_off[e + 1] && row < a.r_max) {
                    a.dst_row[as] = row;
                    a.src_pos[row] = (int32_t)as;
                    kept = 1;
                } else {
                    s_bad = 1;  // counts do not match the ids: keep writes in bounds
                }
            }
        }
        if (!kept) {
            a.dst_row[as] = -1;
            if (a.gates) a.gates[as] = 0.0f;
        }
        a.cmask[as] = (uint8_t)kept;
        s_rank[i] = kept;
    }
    __syncthreads();

    // 5. tokens with >= 1 kept assignment per partition (distinct partitions)
    const int per = E / a.P;
    const int ntok = (int)max(0LL, tok1 - tok0);
    for (int tl = tid; tl < ntok; tl += kLayoutThreads) {
        for (int j = 0; j < k; ++j) {
            const int i = tl * k + j;
            if (!s_rank[i]) continue;
            const int p = s_idx[i] / per;
            bool first = true;
            for (int jj = 0; jj < j; ++jj) {
                const int ii = tl * k + jj;
                if (s_rank[ii] && s_idx[ii] / per == p) { first = false; break; }
            }
            if (first) atomicAdd(&s_ptok[p], 1u);
        }
    }
    __syncthreads();
    for (int p = tid; p < a.P; p += kLayoutThreads)
        if (s_ptok[p]) atomicAdd(&ws->part_tok[p], s_ptok[p]);

    // tile 0 publishes the per-expert / per-partition summary
    if (tile == 0) {
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
    if (tid == 0 && s_bad) record_status(a.ws, MOE_ERR_DEVICE_DATA);

    // completion: the last tile to finish publishes partition tokens and
    // returns every counter to zero; the epoch bump retires this call's flags
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&ws->done_ctr, 1u) == (unsigned)a.ntiles - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int p = tid; p < a.P; p += kLayoutThreads)
        a.part_tokens[p] = (int32_t)atomicExch(&ws->part_tok[p], 0u);
    if (tid == 0) {
        ws->done_ctr = 0u;
        ws->tile_ctr = 0u;
        ws->inject_skip_publish = 0u;
        __threadfence();
        ws->epoch = epoch + 1u;
    }
}

}  // namespace

cudaError_t launch_layout(const int32_t *topk_idx, const int32_t *counts_in, int T, int E, int k,
                          int P, int capacity, float *gates, const moe_layout *L, void *ws,
                          cudaStream_t s)
{
    LayoutArgs a;
    a.idx = topk_idx;
    a.counts_in = counts_in;
    a.T = T;
    a.E = E;
    a.k = k;
    a.P = P;
    a.cap = capacity > 0 ? (unsigned)capacity : 0xFFFFFFFFu;
    a.r_max = L->r_max;
    a.tile_tokens = layout_tile_tokens(k);
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
    layout_kernel<<<a.ntiles, kLayoutThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
