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
// through units = (token, column chunk of the row).  Each block owns a ring
// of S shared-memory stages and is warp-specialised: a producer warp reads
// the routing metadata of 32 upcoming units in one round trip and fills
// stages with 1-D bulk copies (cp.async.bulk, the TMA engine) of the kept
// expert-output chunks and the shared-expert chunks, completing on the
// stage's "full" mbarrier; four consumer warps wait on "full", accumulate
// in fp32 with explicit round-to-nearest FMA/add in the pinned order (kept
// slots ascending, then shared experts ascending), round once to bf16,
// store y with 16-byte coalesced stores, and release the stage on its
// "empty" mbarrier.  No block-wide barrier sits in the loop, and the bytes
// in flight per SM are bounded by shared memory, not registers.  Every
// mbarrier wait is bounded; on expiry the waiter records MOE_ERR_TIMEOUT,
// and the producer always waits (bounded) for its copies still in flight
// before it returns.
#include <cuda_bf16.h>

#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 108 * 1024;  // dynamic shared memory per block (two blocks per SM)

struct CombineArgs {
    const char *eo;        // [rows, H] bf16
    const float *gates;    // [T, K]
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
    int stages;
    int slots;             // K + Ks
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

// Bounded wait on a stage barrier.  Returns false if the bound expired.
__device__ __forceinline__ bool wait_stage(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kSpinLimitNs) return false;
    return true;
}

template <int K>
__global__ void __launch_bounds__(kCombThreads + 32) combine_tma_kernel(CombineArgs a)
{
    extern __shared__ __align__(128) unsigned char s_stage[];  // [stages][slots][cb]
    __shared__ uint64_t s_full[kMaxStages];   // producer -> consumers: stage loaded
    __shared__ uint64_t s_empty[kMaxStages];  // consumers -> producer: stage free
    __shared__ float s_g[kMaxStages][K];
    __shared__ int s_n[kMaxStages];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const long long stride = gridDim.x;
    const size_t stage_bytes = (size_t)a.slots * a.cb;

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], kCombThreads);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    if (warp == 0) {
        // ---- producer warp ----------------------------------------------
        // Lane l fetches the routing metadata (kept rows, gates) of the l-th
        // unit of the current batch of 32, so one memory round trip serves
        // 32 stage fills; lane 0 issues the bulk copies.
        const int rows_valid = min(a.r_max, __ldg(a.R_ptr));
        unsigned issued = 0;  // parity of each stage's last fill (bit) once filled
        long long i = 0;
        bool stop = false;
        for (long long batch = 0; !stop; batch += 32) {
            const long long ul = blockIdx.x + (batch + lane) * stride;
            int rows[K];
            float g[K];
            if (ul < a.units) {
                const long long t = ul / a.nch;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    rows[j] = __ldg(a.dst_row + t * K + j);
                    g[j] = __ldg(a.gates + t * K + j);
                }
            }
            for (int b = 0; b < 32; ++b, ++i) {
                const long long u = blockIdx.x + i * stride;
                if (u >= a.units) { stop = true; break; }
                const int s = (int)(i % a.stages);
                const long long use = i / a.stages;  // how many times stage s was filled before
                if (use > 0) {
                    bool ok = mbar_try_wait(&s_empty[s], (uint32_t)((use - 1) & 1));
                    if (!ok) {
                        const unsigned long long t0 = global_timer_ns();
                        while (!(ok = mbar_try_wait(&s_empty[s], (uint32_t)((use - 1) & 1))) &&
                               global_timer_ns() - t0 < kSpinLimitNs) {
                        }
                    }
                    if (!ok) {
                        if (lane == 0) record_status(a.ws, MOE_ERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                }
                int rb[K];
                float gb[K];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    rb[j] = __shfl_sync(0xffffffffu, rows[j], b);
                    gb[j] = __shfl_sync(0xffffffffu, g[j], b);
                }
                if (lane == 0) {
                    const long long t = u / a.nch;
                    const int col0 = (int)(u - t * a.nch) * a.cb;
                    const int bytes = min(a.cb, a.rowbytes - col0);
                    int n = 0;
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        if (rb[j] >= rows_valid) {
                            record_status(a.ws, MOE_ERR_DEVICE_DATA);
                            rb[j] = -1;
                        }
                        if (rb[j] >= 0) s_g[s][n++] = gb[j];  // gates of the kept slots, in slot order
                    }
                    s_n[s] = n;
                    // expected bytes first (release: s_g / s_n become visible to the waiters)
                    mbar_arrive_expect_tx(&s_full[s], (uint32_t)((n + a.Ks) * bytes));
                    unsigned char *st = s_stage + (size_t)s * stage_bytes;
                    int slot = 0;
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        if (rb[j] >= 0) {
                            bulk_load(st + (size_t)slot * a.cb, a.eo + (long long)rb[j] * a.rowbytes + col0,
                                      bytes, &s_full[s]);
                            ++slot;
                        }
                    }
                    for (int q = 0; q < a.Ks; ++q)
                        bulk_load(st + (size_t)(K + q) * a.cb,
                                  a.shared + ((long long)q * a.T + t) * a.rowbytes + col0, bytes, &s_full[s]);
                }
                issued = (issued & ~(1u << s)) | ((unsigned)(use & 1) << s) | (1u << (s + 16));
            }
        }
        // drain: never leave with copies still landing in this block's shared memory
        if (lane == 0) {
            for (int s = 0; s < a.stages; ++s) {
                if (!(issued & (1u << (s + 16)))) continue;
                const uint32_t par = (issued >> s) & 1u;
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&s_full[s], par) && global_timer_ns() - t0 < kSpinLimitNs) {
                }
            }
        }
        return;
    }

    // ---- consumer warps ---------------------------------------------------
    const int ct = tid - 32;
    long long i = 0;
    for (long long u = blockIdx.x; u < a.units; u += stride, ++i) {
        const int s = (int)(i % a.stages);
        const uint32_t par = (uint32_t)((i / a.stages) & 1);
        if (!wait_stage(&s_full[s], par)) {
            if (ct == 0) record_status(a.ws, MOE_ERR_TIMEOUT);
            return;
        }
        const long long t = u / a.nch;
        const int col0 = (int)(u - t * a.nch) * a.cb;
        const int nv = min(a.cb, a.rowbytes - col0) >> 4;
        const int n = s_n[s];
        const unsigned char *st = s_stage + (size_t)s * stage_bytes;
        uint4 *yrow = reinterpret_cast<uint4 *>(a.y + t * a.rowbytes + col0);
        for (int v = ct; v < nv; v += kCombThreads) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
            // pinned order: kept slots ascending, then shared experts ascending
            for (int r = 0; r < n; ++r) fma8(acc, s_g[s][r], lds_v4(st + (size_t)r * a.cb + v * 16));
            for (int q = 0; q < a.Ks; ++q) add8(acc, lds_v4(st + (size_t)(K + q) * a.cb + v * 16));
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            st_v4(yrow + v, o);
        }
        mbar_arrive(&s_empty[s]);
    }
}

int blocks_per_sm(const void *fn, size_t smem)
{
    static std::mutex mu;
    static std::unordered_map<unsigned long long, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long key = (reinterpret_cast<unsigned long long>(fn) * 1315423911ull) ^
                                   ((unsigned long long)smem << 8) ^ (unsigned long long)dev;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kCombThreads + 32, smem) != cudaSuccess || n < 1) n = 1;
    cache[key] = n;
    return n;
}

template <int K>
cudaError_t launch_k(const CombineArgs &a, cudaStream_t s)
{
    const void *fn = reinterpret_cast<const void *>(combine_tma_kernel<K>);
    const size_t smem = (size_t)a.stages * a.slots * a.cb;
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBudget);
        if (err != cudaSuccess) return err;
    }
    const long long resident = (long long)device_sm_count() * blocks_per_sm(fn, smem);
    const unsigned grid = (unsigned)(a.units < resident ? a.units : resident);
    return launch_pdl(combine_tma_kernel<K>, dim3(grid), dim3(kCombThreads + 32), smem, s, a);
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
    a.slots = L->k + Ks;
    // Chunk the row so that at least three stages fit the budget, then use as
    // many stages (<= kMaxStages) as the budget holds.
    const int cb_max = (kStageBudget / 3 / a.slots) & ~15;
    a.nch = (a.rowbytes + cb_max - 1) / cb_max;
    a.cb = (((a.rowbytes + a.nch - 1) / a.nch) + 15) & ~15;
    a.stages = kStageBudget / (a.slots * a.cb);
    if (a.stages > kMaxStages) a.stages = kMaxStages;
    if (a.stages < 1) return cudaErrorInvalidValue;
    a.units = (long long)T * a.nch;
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
