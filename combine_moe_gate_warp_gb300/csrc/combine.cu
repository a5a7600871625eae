// combine.cu -- moe_combine: gather each token's expert outputs through the
// saved routing metadata, gate-weight them, add the shared experts, and
// write the token's output row once.
//
// "MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7
// ("Combine": per token, the weighted sum of its top-k expert outputs, put
// back in original token order using the metadata saved at dispatch, no
// second routing) and sec. 8.2.B (shared experts: every token, no
// all-to-all, outputs added); "DeepSeek MoE sync tax" sec. 2.1 (K_s shared
// experts).
//
// Design (sm_103a): gather form -- y is written exactly once and every kept
// expert-output row is read exactly once, so the traffic is the algorithmic
// minimum.  A persistent grid (as many blocks as fit on the SMs) works
// through units = (token, column chunk of the row).  Each block owns a byte
// ring in shared memory and is warp-specialised: a producer warp reads the
// routing metadata of 32 upcoming units in one round trip, allocates
// exactly (kept rows + shared experts) x chunk bytes per unit in the ring
// (dropped slots take no space, so skewed or capacity-limited routing keeps
// as many bytes in flight as dense routing), and fills them with 1-D bulk
// copies (cp.async.bulk, the TMA engine) completing on the unit's "full"
// mbarrier; four consumer warps (one unit per warp for small units, all
// four on one unit for large ones) wait on "full", accumulate
// in fp32 with explicit round-to-nearest FMA/add in the pinned order (kept
// slots ascending, then shared experts ascending), round once to bf16,
// store y with 16-byte coalesced stores, and release the unit on its
// "empty" mbarrier; the producer reclaims ring space in unit order.  No block-wide barrier sits in the loop, and the bytes
// in flight per SM are bounded by shared memory, not registers.  Every
// mbarrier wait is bounded; on expiry the waiter records MOE_ERR_TIMEOUT,
// and the producer always waits (bounded) for its copies still in flight
// before it returns.
//
// With no gates (weight 1 for every kept slot, no shared experts) the same
// kernel is the dispatch backward: dx[t] = bf16 RNE of the fp32 sum, in slot
// order, of the gradient rows of t's kept copies (an FMA with weight 1
// rounds exactly like the plain fp32 add).
#include <cuda_bf16.h>

#include "common.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;
// Ring policy (compile-time): ring size per block, the share of the ring a
// fully kept unit may take before rows are split into column chunks (in
// percent), and the unit size from which all four consumer warps share a
// unit.
#ifndef MOE_COMBINE_RING_KB
#define MOE_COMBINE_RING_KB 108
#endif
#ifndef MOE_COMBINE_UNIT_PCT
#define MOE_COMBINE_UNIT_PCT 60
#endif
#ifndef MOE_COMBINE_GROUP_KB
#define MOE_COMBINE_GROUP_KB 32
#endif
constexpr int kDesc = 16;                                  // units in flight per block at most
constexpr int kRingBytes = MOE_COMBINE_RING_KB * 1024;     // byte ring per block (108 KiB: two blocks per SM)

struct CombineArgs {
    const char *eo;        // [rows, H] bf16
    const float *gates;    // [T, K], or null: every weight 1 (dispatch backward)
    const int32_t *dst_row;
    const int32_t *R_ptr;  // offsets + E: rows the layout produced
    const char *shared;    // [Ks, T, H] bf16 or null
    char *y;               // [T, H] bf16
    void *ws;
    long long T;
    long long units;       // T * nch
    int r_max;
    int Ks;
    int rowbytes;          // H * 2
    int nch;               // column chunks per row
    int cb;                // chunk bytes (multiple of 16)
    int ring_bytes;        // shared-memory byte ring per block
    int group;             // consumer warps per unit (1, 2 or 4)
    int interleave;        // units from both ends of a block's share (layouts with a capacity)
};

__device__ __forceinline__ void fma8(float (&acc)[8], float g, const uint4 &v)
{
    acc[0] = __fmaf_rn(g, bf16lo(v.x), acc[0]);
    acc[1] = __fmaf_rn(g, bf16hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(g, bf16lo(v.y), acc[2]);
    acc[3] = __fmaf_rn(g, bf16hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(g, bf16lo(v.z), acc[4]);
    acc[5] = __fmaf_rn(g, bf16hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(g, bf16lo(v.w), acc[6]);
    acc[7] = __fmaf_rn(g, bf16hi(v.w), acc[7]);
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v)
{
    acc[0] = __fadd_rn(acc[0], bf16lo(v.x));
    acc[1] = __fadd_rn(acc[1], bf16hi(v.x));
    acc[2] = __fadd_rn(acc[2], bf16lo(v.y));
    acc[3] = __fadd_rn(acc[3], bf16hi(v.y));
    acc[4] = __fadd_rn(acc[4], bf16lo(v.z));
    acc[5] = __fadd_rn(acc[5], bf16hi(v.z));
    acc[6] = __fadd_rn(acc[6], bf16lo(v.w));
    acc[7] = __fadd_rn(acc[7], bf16hi(v.w));
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&h);
}

// The order in which a block takes its units.  With capacity drops the kept
// rows per token fall along the batch (the first tokens fill the experts:
// all 8 of 8 kept in the first eighth of a 262144-token top-8 prefill batch
// with capacity 1.25, ~1.3 in its last eighth), and in token order every
// block would meet only 64 KB units at once, of which its ring holds one.
// So a layout with a capacity takes a block's units alternately from the
// front and the back of its share (0, n-1, 1, n-2, ...: a bijection on
// [0, n)), and large and small units share the ring: that combine 1468 ->
// 1377 us on GB300.  Without a capacity every token keeps k rows, and token
// order (better locality: 0.5-1 % faster there) is kept.
__device__ __forceinline__ long long unit_order(long long i, long long n, int interleave)
{
    return !interleave ? i : ((i & 1) ? n - 1 - (i >> 1) : (i >> 1));
}

// Token of unit u.  The producer pays this per unit on its serial path,
// where a 64-bit division costs more than the rest of the unit's
// bookkeeping: in the four-warp mode rows of up to ~8 KiB are one unit each
// (nch == 1: no division) and otherwise a 32-bit division serves where u
// allows it (262144 x 4096, top-8 with capacity: 1387 -> 1363 us on GB300).
// The one-warp mode keeps the plain division: there the faster producer
// measured slower (65536 x 4096, top-2: 230 -> 242 us).
template <bool FAST>
__device__ __forceinline__ long long unit_token(long long u, int nch)
{
    if constexpr (FAST) {
        if (nch == 1) return u;
        if (u < (1LL << 32)) return (long long)((unsigned)u / (unsigned)nch);
    }
    return u / nch;
}

// Bounded wait on a stage barrier.  Returns false if the bound expired.
__device__ __forceinline__ bool wait_stage(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kSpinLimitNs) return false;
    return true;
}

// WIDE: all four consumer warps share each (large) unit, chosen per launch
// from the unit size.  Two choices follow it, both measured on GB300:
//  * the producer sleeps (suspend hint) instead of polling while it waits
//    for ring space.  With four warps on one large unit (many slots per
//    token) a polling producer competes with them for issue slots (262144
//    tokens x 4096, top-8 with capacity drops: 1520 -> 1463 us); with one
//    warp per small unit the producer must react at once (65536 x 4096,
//    top-2: 231 -> 243 us when it sleeps).  A runtime switch inside the
//    wait loop cost more than either, so it is a template parameter;
//  * the rows are read and y is written with the evict-first L2 policy
//    (8192 x 2048, top-8 + 2 shared experts: the batch 118 -> 111 us;
//    the top-8 prefill batch 2886 -> 2861 us), which slows the one-warp
//    mode (65536 x 4096, top-2: 230 -> 238 us), so that mode keeps the
//    normal policy.
template <int K, bool WIDE>
__global__ void __launch_bounds__(kCombThreads + 32) combine_tma_kernel(CombineArgs a)
{
    extern __shared__ __align__(128) unsigned char s_ring[];  // byte ring of a.ring_bytes
    __shared__ uint64_t s_full[kDesc];   // producer -> consumers: unit loaded
    __shared__ uint64_t s_empty[kDesc];  // consumers -> producer: unit consumed
    __shared__ float s_g[kDesc][K];
    __shared__ int s_n[kDesc];
    __shared__ int s_off[kDesc];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const long long stride = gridDim.x;
    const long long n_units = (a.units - blockIdx.x + stride - 1) / stride;  // units of this block
    if (n_units <= 0) return;

    if (tid == 0) {
        for (int d = 0; d < kDesc; ++d) {
            mbar_init(&s_full[d], 1);
            mbar_init(&s_empty[d], 32 * a.group);  // released by the warps that consumed the unit
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const uint64_t pol = l2_stream_policy(WIDE);

    if (warp == 0) {
        // ---- producer warp ----------------------------------------------
        // Lane l fetches the routing metadata of the l-th unit of the current
        // batch of 32 (one round trip per 32 units); lane 0 allocates each
        // unit's bytes in the ring and issues its bulk copies.
        const int rows_valid = min(a.r_max, __ldg(a.R_ptr));
        long long oldest = 0;  // first unit whose bytes are not yet known to be free
        int head = 0;          // next free byte of the ring
        bool stop = false;
        long long i = 0;
        // wait (bounded) until unit `oldest` has been consumed, then retire it
        auto retire_oldest = [&]() -> bool {
            const int d = (int)(oldest % kDesc);
            const uint32_t par = (uint32_t)((oldest / kDesc) & 1);
            auto probe = [&]() {
                if constexpr (WIDE) return mbar_try_wait_sleep(&s_empty[d], par);
                else return mbar_try_wait(&s_empty[d], par);
            };
            bool ok = probe();
            if (!ok) {
                const unsigned long long t0 = global_timer_ns();
                while (!(ok = probe()) && global_timer_ns() - t0 < kSpinLimitNs) {
                }
            }
            ++oldest;
            return ok;
        };
        for (long long batch = 0; !stop && batch < n_units; batch += 32) {
            int rows[K];
            float g[K];
            if (batch + lane < n_units) {
                const long long t = unit_token<WIDE>(blockIdx.x + unit_order(batch + lane, n_units, a.interleave) * stride, a.nch);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    rows[j] = __ldg(a.dst_row + t * K + j);
                    g[j] = a.gates ? __ldg(a.gates + t * K + j) : 1.0f;
                }
            }
            for (int b = 0; b < 32 && i < n_units; ++b, ++i) {
                int rb[K];
                float gb[K];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    rb[j] = __shfl_sync(0xffffffffu, rows[j], b);
                    gb[j] = __shfl_sync(0xffffffffu, g[j], b);
                }
                int ok = 1;
                if (lane == 0) {
                    const long long u = blockIdx.x + unit_order(i, n_units, a.interleave) * stride;
                    const long long t = unit_token<WIDE>(u, a.nch);
                    const int col0 = (int)(u - t * a.nch) * a.cb;
                    const int bytes = min(a.cb, a.rowbytes - col0);
                    int n = 0;
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        if (rb[j] >= rows_valid) {
                            record_status(a.ws, MOE_ERR_DEVICE_DATA);
                            rb[j] = -1;
                        }
                        n += rb[j] >= 0;
                    }
                    const int need = (n + a.Ks) * bytes;
                    // a free descriptor, then `need` contiguous ring bytes
                    while (ok && oldest <= i - kDesc) ok = retire_oldest();
                    int pos = 0;
                    while (ok) {
                        if (oldest == i) { pos = 0; break; }  // nothing in flight
                        const int tail = s_off[oldest % kDesc];
                        if (head > tail) {
                            if (a.ring_bytes - head >= need) { pos = head; break; }
                            if (tail >= need) { pos = 0; break; }
                        } else if (tail - head >= need) {
                            pos = head;
                            break;
                        }
                        ok = retire_oldest();
                    }
                    if (ok) {
                        const int d = (int)(i % kDesc);
                        int k2 = 0;
#pragma unroll
                        for (int j = 0; j < K; ++j)
                            if (rb[j] >= 0) s_g[d][k2++] = gb[j];  // kept slots, in slot order
                        s_n[d] = n;
                        s_off[d] = pos;
                        head = pos + need;
                        // expected bytes first (release: s_g / s_n / s_off visible to the waiters)
                        mbar_arrive_expect_tx(&s_full[d], (uint32_t)need);
                        unsigned char *dst = s_ring + pos;
#pragma unroll
                        for (int j = 0; j < K; ++j) {
                            if (rb[j] >= 0) {
                                bulk_load(dst, a.eo + (long long)rb[j] * a.rowbytes + col0, bytes, &s_full[d], pol);
                                dst += bytes;
                            }
                        }
                        for (int q = 0; q < a.Ks; ++q) {
                            bulk_load(dst, a.shared + ((long long)q * a.T + t) * a.rowbytes + col0, bytes, &s_full[d], pol);
                            dst += bytes;
                        }
                    } else {
                        record_status(a.ws, MOE_ERR_TIMEOUT);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) { stop = true; break; }
            }
        }
        // drain: never leave with copies still landing in this block's shared memory
        if (lane == 0) {
            for (long long q = oldest; q < i; ++q) {
                const int d = (int)(q % kDesc);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&s_full[d], (uint32_t)((q / kDesc) & 1)) &&
                       global_timer_ns() - t0 < kSpinLimitNs) {
                }
            }
        }
        return;
    }

    // ---- consumer warps ---------------------------------------------------
    // Groups of a.group warps consume units round-robin: with one-warp groups
    // four units are combined concurrently (small units do not serialise);
    // with one four-warp group a large unit is spread over 128 threads.
    const int cw = warp - 1;
    constexpr int kConsumerWarps = kCombThreads / 32;
    const int ngroups = kConsumerWarps / a.group;
    const int grp = cw / a.group;
    const int gt = (cw - grp * a.group) * 32 + lane;  // thread index within the group
    const int gthreads = 32 * a.group;
    for (long long i = grp; i < n_units; i += ngroups) {
        const int d = (int)(i % kDesc);
        if (!wait_stage(&s_full[d], (uint32_t)((i / kDesc) & 1))) {
            if (gt == 0) record_status(a.ws, MOE_ERR_TIMEOUT);
            return;
        }
        const long long u = blockIdx.x + unit_order(i, n_units, a.interleave) * stride;
        const long long t = unit_token<WIDE>(u, a.nch);
        const int col0 = (int)(u - t * a.nch) * a.cb;
        const int bytes = min(a.cb, a.rowbytes - col0);
        const int nv = bytes >> 4;
        const int n = s_n[d];
        const unsigned char *st = s_ring + s_off[d];
        uint4 *yrow = reinterpret_cast<uint4 *>(a.y + t * a.rowbytes + col0);
        for (int v = gt; v < nv; v += gthreads) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
            // pinned order: kept slots ascending, then shared experts ascending
            for (int r = 0; r < n; ++r) fma8(acc, s_g[d][r], lds_v4(st + (size_t)r * bytes + v * 16));
            for (int q = 0; q < a.Ks; ++q) add8(acc, lds_v4(st + (size_t)(n + q) * bytes + v * 16));
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            st_stream_v4(yrow + v, o, pol);
        }
        mbar_arrive(&s_empty[d]);
    }
}

template <int K, bool WIDE>
cudaError_t launch_kp(const CombineArgs &a, cudaStream_t s)
{
    const void *fn = reinterpret_cast<const void *>(combine_tma_kernel<K, WIDE>);
    const size_t smem = (size_t)a.ring_bytes;
    cudaError_t err = allow_dynamic_smem(fn, (int)smem);
    if (err != cudaSuccess) return err;
    const long long resident = resident_grid(fn, kCombThreads + 32, smem);
    const unsigned grid = (unsigned)(a.units < resident ? a.units : resident);
    return launch_pdl(combine_tma_kernel<K, WIDE>, dim3(grid), dim3(kCombThreads + 32), smem, s, a);
}

template <int K>
cudaError_t launch_k(const CombineArgs &a, cudaStream_t s)
{
    return a.group == 4 ? launch_kp<K, true>(a, s) : launch_kp<K, false>(a, s);
}

}  // namespace

cudaError_t launch_combine(const void *eo, const moe_layout *L, const float *gates, const void *shared,
                           int Ks, int T, int H, void *y, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    CombineArgs a;
    a.eo = static_cast<const char *>(eo);
    a.gates = gates;
    a.dst_row = L->dst_row;
    a.R_ptr = L->offsets + L->E;
    a.shared = static_cast<const char *>(shared);
    a.y = static_cast<char *>(y);
    a.ws = L->ws;
    a.T = T;
    a.r_max = L->r_max;
    a.Ks = Ks;
    a.rowbytes = H * 2;
    // Whole rows per unit unless a unit with every slot kept would take more
    // than MOE_COMBINE_UNIT_PCT% of the ring; then equal 16-byte-aligned
    // column chunks.
    const int slots = L->k + Ks;
    const int cb_max = (kRingBytes / 100 * MOE_COMBINE_UNIT_PCT / slots) & ~15;
    a.nch = (a.rowbytes + cb_max - 1) / cb_max;
    a.cb = (((a.rowbytes + a.nch - 1) / a.nch) + 15) & ~15;
    a.ring_bytes = kRingBytes;
    // a unit of >= MOE_COMBINE_GROUP_KB KiB (all slots kept) is shared by all
    // four consumer warps; smaller units go one per warp
    a.group = (slots * a.cb >= MOE_COMBINE_GROUP_KB * 1024) ? 4 : 1;
    a.units = (long long)T * a.nch;
    a.interleave = L->capacity > 0 ? 1 : 0;
    switch (L->k) {
#define MOE_COMBINE_CASE(KK) \
    case KK: return launch_k<KK>(a, s);
        MOE_COMBINE_CASE(1) MOE_COMBINE_CASE(2) MOE_COMBINE_CASE(3) MOE_COMBINE_CASE(4)
        MOE_COMBINE_CASE(5) MOE_COMBINE_CASE(6) MOE_COMBINE_CASE(7) MOE_COMBINE_CASE(8)
        MOE_COMBINE_CASE(9) MOE_COMBINE_CASE(10) MOE_COMBINE_CASE(11) MOE_COMBINE_CASE(12)
        MOE_COMBINE_CASE(13) MOE_COMBINE_CASE(14) MOE_COMBINE_CASE(15) MOE_COMBINE_CASE(16)
#undef MOE_COMBINE_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
