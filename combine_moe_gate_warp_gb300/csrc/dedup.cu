// dedup.cu -- moe_dedup_layout: per-partition token de-duplication.
//
// "MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7
// (dispatch detail: the rows bound for one destination are packed into one
// contiguous block).  A token that keeps several slots in one partition is
// sent there once, with its local expert ids and gates in slot order; the
// partition expands it to its experts, combines them, and returns one row.
// From a layout (the final expert of a kept slot is the expert whose rows
// contain its dst_row) and the gates it writes, for P <= 64 partitions:
//   send_offsets[P+1]  exclusive scan of the tokens sent to each partition
//   send_row[t*P + p]  send row of (t, p) or -1; rows are partition-major,
//                      tokens ascending within a partition
//   send_token[s], slot_local[s*k + q], slot_gate[s*k + q]
//
// Design (sm_103a): three short launches over tiles of tokens (every token
// is read by one thread: k dst_row words, a binary search of the layout
// offsets held in shared memory):
//   1. dedup_count_kernel: per tile, tokens per partition (a ballot and a
//      shared atomic per warp and partition);
//   2. dedup_scan_kernel: one block scans the tile counts per partition and
//      the partition totals;
//   3. dedup_write_kernel: per tile, rounds of 256 tokens; the rank of a
//      token among the tile's tokens of partition p comes from warp ballots
//      per partition and a per-round prefix over the warps.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kDedupThreads = 256;
constexpr int kDedupTile = 2048;  // tokens per tile
constexpr int kDedupWarps = kDedupThreads / 32;

struct DedupArgs {
    const int32_t *dst_row;
    const int32_t *offsets;  // [E+1] of the source layout
    const float *gates;      // [T, k]
    long long T;
    int E, k, P, r_max;
    int ntiles;
    int32_t *tile_counts;    // scratch [ntiles, P]
    int32_t *send_offsets, *send_row, *send_token, *slot_local;
    float *slot_gate;
    void *ws;
};

// Expert whose rows contain `row` (offsets in shared memory, E entries + 1).
__device__ __forceinline__ int expert_of(const int *s_off, int E, int row)
{
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= row) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Partition mask of token t (bit p: a kept slot in partition p).
__device__ __forceinline__ unsigned long long token_mask(const DedupArgs &a, const int *s_off, int rows_valid,
                                                         long long t)
{
    const int per = a.E / a.P;
    unsigned long long m = 0ull;
    for (int j = 0; j < a.k; ++j) {
        const int r = __ldg(a.dst_row + t * a.k + j);
        if (r < 0) continue;
        if (r >= rows_valid) {
            record_status(a.ws, MOE_ERR_DEVICE_DATA);
            continue;
        }
        m |= 1ull << (expert_of(s_off, a.E, r) / per);
    }
    return m;
}

__device__ __forceinline__ int load_offsets(const DedupArgs &a, int *s_off)
{
    for (int i = threadIdx.x; i <= a.E; i += kDedupThreads) s_off[i] = __ldg(a.offsets + i);
    __syncthreads();
    return min(a.r_max, s_off[a.E]);
}

__global__ void __launch_bounds__(kDedupThreads) dedup_count_kernel(DedupArgs a)
{
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ int s_cnt[64];
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x < 64) s_cnt[threadIdx.x] = 0;
    const int rows_valid = load_offsets(a, s_off);
    const long long t0 = (long long)blockIdx.x * kDedupTile;
    const long long t1 = min(a.T, t0 + kDedupTile);
    const int lane = threadIdx.x & 31;
    for (long long tb = t0; tb < t1; tb += kDedupThreads) {
        const long long t = tb + threadIdx.x;
        const unsigned long long m = t < t1 ? token_mask(a, s_off, rows_valid, t) : 0ull;
        // one ballot and one shared atomic per partition the warp reaches
        const unsigned lo = __reduce_or_sync(0xffffffffu, (unsigned)m);
        const unsigned hi = __reduce_or_sync(0xffffffffu, (unsigned)(m >> 32));
        unsigned long long wm = ((unsigned long long)hi << 32) | lo;
        while (wm) {
            const int p = __ffsll((long long)wm) - 1;
            wm &= wm - 1ull;
            const unsigned b = __ballot_sync(0xffffffffu, (unsigned)(m >> p) & 1u);
            if (lane == 0) atomicAdd(&s_cnt[p], __popc(b));
        }
    }
    __syncthreads();
    for (int p = threadIdx.x; p < a.P; p += kDedupThreads) a.tile_counts[(size_t)blockIdx.x * a.P + p] = s_cnt[p];
}

// One block: tile_counts becomes the first send row of each (tile, p).
__global__ void __launch_bounds__(kDedupThreads) dedup_scan_kernel(DedupArgs a)
{
    __shared__ int s_tot[64];
    pdl_wait();
    pdl_launch_dependents();
    const int p = threadIdx.x;
    if (p < a.P) {
        int run = 0;
        for (int tile = 0; tile < a.ntiles; ++tile) {
            const int c = a.tile_counts[(size_t)tile * a.P + p];
            a.tile_counts[(size_t)tile * a.P + p] = run;
            run += c;
        }
        s_tot[p] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int q = 0; q < a.P; ++q) {
            a.send_offsets[q] = s;
            s += s_tot[q];
        }
        a.send_offsets[a.P] = s;
    }
    __syncthreads();
    if (p < a.P) {
        int base = 0;
        for (int q = 0; q < p; ++q) base += s_tot[q];
        for (int tile = 0; tile < a.ntiles; ++tile) a.tile_counts[(size_t)tile * a.P + p] += base;
    }
}

__global__ void __launch_bounds__(kDedupThreads) dedup_write_kernel(DedupArgs a)
{
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ int s_wcnt[kDedupWarps][64];
    __shared__ int s_base[64];
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = a.E / a.P;
    const int rows_valid = load_offsets(a, s_off);
    if (threadIdx.x < a.P) s_base[threadIdx.x] = a.tile_counts[(size_t)blockIdx.x * a.P + threadIdx.x];
    const long long t0 = (long long)blockIdx.x * kDedupTile;
    const long long t1 = min(a.T, t0 + kDedupTile);
    for (long long r0 = t0; r0 < t1; r0 += kDedupThreads) {
        const long long t = r0 + threadIdx.x;
        const unsigned long long m = t < t1 ? token_mask(a, s_off, rows_valid, t) : 0ull;
        // rank of this token among the round's tokens of each partition
        int rank_in_warp[64];
        for (int p = 0; p < a.P; ++p) {
            const unsigned b = __ballot_sync(0xffffffffu, (m >> p) & 1ull);
            rank_in_warp[p] = __popc(b & ((1u << lane) - 1u));
            if (lane == 0) s_wcnt[warp][p] = __popc(b);
        }
        __syncthreads();
        if (t < t1) {
            for (int p = 0; p < a.P; ++p) {
                const long long key = t * a.P + p;
                if (!((m >> p) & 1ull)) {
                    a.send_row[key] = -1;
                    continue;
                }
                int before = 0;
                for (int w = 0; w < warp; ++w) before += s_wcnt[w][p];
                const int s = s_base[p] + before + rank_in_warp[p];
                a.send_row[key] = s;
                a.send_token[s] = (int32_t)t;
                int q = 0;
                for (int j = 0; j < a.k; ++j) {
                    const int r = __ldg(a.dst_row + t * a.k + j);
                    if (r < 0 || r >= rows_valid) continue;
                    const int e = expert_of(s_off, a.E, r);
                    if (e / per != p) continue;
                    a.slot_local[(size_t)s * a.k + q] = e - p * per;
                    a.slot_gate[(size_t)s * a.k + q] = __ldg(a.gates + t * a.k + j);
                    ++q;
                }
                for (; q < a.k; ++q) {
                    a.slot_local[(size_t)s * a.k + q] = -1;
                    a.slot_gate[(size_t)s * a.k + q] = 0.0f;
                }
            }
        }
        __syncthreads();
        if (threadIdx.x < a.P) {
            int tot = 0;
            for (int w = 0; w < kDedupWarps; ++w) tot += s_wcnt[w][threadIdx.x];
            s_base[threadIdx.x] += tot;
        }
        __syncthreads();
    }
}

}  // namespace

size_t dedup_scratch_bytes(long long T, int P)
{
    const long long ntiles = (T + kDedupTile - 1) / kDedupTile;
    return (size_t)(ntiles < 1 ? 1 : ntiles) * (size_t)P * sizeof(int32_t);
}

cudaError_t launch_dedup_layout(const moe_layout *L, const float *gates, moe_dedup *D, void *scratch,
                                cudaStream_t s)
{
    if (L->T == 0) return cudaMemsetAsync(D->send_offsets, 0, sizeof(int32_t) * (size_t)(L->P + 1), s);
    DedupArgs a;
    a.dst_row = L->dst_row;
    a.offsets = L->offsets;
    a.gates = gates;
    a.T = L->T;
    a.E = L->E;
    a.k = L->k;
    a.P = L->P;
    a.r_max = L->r_max;
    a.ntiles = (int)((a.T + kDedupTile - 1) / kDedupTile);
    a.tile_counts = static_cast<int32_t *>(scratch);
    a.send_offsets = D->send_offsets;
    a.send_row = D->send_row;
    a.send_token = D->send_token;
    a.slot_local = D->slot_local;
    a.slot_gate = D->slot_gate;
    a.ws = L->ws;
    cudaError_t err = launch_pdl(dedup_count_kernel, dim3(a.ntiles), dim3(kDedupThreads), 0, s, a);
    if (err != cudaSuccess) return err;
    err = launch_pdl(dedup_scan_kernel, dim3(1), dim3(kDedupThreads), 0, s, a);
    if (err != cudaSuccess) return err;
    return launch_pdl(dedup_write_kernel, dim3(a.ntiles), dim3(kDedupThreads), 0, s, a);
}

}  // namespace moe
