// common.cuh -- pieces shared by the libmoeroute kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_route.h"

namespace moe {

// ---------------------------------------------------------------------------
// Workspace.  A fixed 8 KiB header of counters followed by the decoupled
// look-back flag words of the layout scan (one 64-bit word per tile and
// expert).  Every counter is returned to zero by the kernel that used it, so
// a zeroed workspace stays valid from call to call.
// ---------------------------------------------------------------------------
struct WsHeader {
    unsigned status;               // first device error wins (atomicCAS from 0)
    unsigned done_ctr;             // layout: completed tiles
    unsigned gate_ticket;          // gate: finished blocks
    // Failure-injection hook for tests, written only from the host: when it
    // holds tile+1, that layout tile does not publish its look-back flags,
    // so its successor's bounded wait expires (MOE_ERR_TIMEOUT).  Zero in
    // normal use; the layout call that sees it clears it.
    unsigned inject_skip_publish;
    // layout: {tile id (low 32 bits), epoch (high 32 bits)} in one word, so a
    // block learns both with a single atomic; the epoch tags flag words and
    // is bumped by the block that draws the last tile id of a call
    unsigned long long tile_epoch;
    unsigned quant_ticket;         // grouped FP8 encode: finished blocks
    unsigned pad0[25];
    unsigned gate_counts[MOE_MAX_EXPERTS];  // gate: per-expert totals
    unsigned part_tok[MOE_MAX_EXPERTS];     // layout: per-partition token totals
    // grouped FP8 quantiser: per group (expert, or group 0 for global) the
    // max key (max_word) and min key (min_word) of its rows, zero = empty
    unsigned quant_max[MOE_MAX_EXPERTS];
    unsigned quant_min[MOE_MAX_EXPERTS];
    // fused route kernel: grid barrier word {generation (high 32 bits),
    // blocks arrived (low 32)}; the generation's parity selects which of the
    // two per-expert total arrays a call accumulates into (the other one is
    // cleared for the next call)
    unsigned long long route_bar;
    unsigned route_counts[2][MOE_MAX_EXPERTS];
};
static_assert(sizeof(WsHeader) <= 8192, "workspace header must fit 8 KiB");
constexpr size_t kWsHeaderBytes = 8192;

__host__ __device__ inline unsigned long long *ws_flags(void *ws)
{
    return reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kWsHeaderBytes);
}

// Layout tiling.  A tile holds layout_tile_tokens(T, k) consecutive tokens,
// i.e. up to kLayoutMaxTileAssign assignments: about A/256 assignments
// rounded up to a multiple of 1024, within [1024, 8192], so that large
// problems use ~256 tiles (short look-back chains) and small ones still
// spread over many blocks.  The rule depends only on (T, k): the
// workspace size is known on the host without a device.  T*k < 2^30 keeps
// every count inside the 30-bit value field of a flag word.
constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kLayoutMinTileAssign = 1024;
constexpr int kLayoutMaxTileAssign = 8192;
__host__ __device__ inline int layout_tile_tokens(long long T, int k)
{
    const long long A = T * k;
    long long t = (A + 255) / 256;
    t = (t + kLayoutMinTileAssign - 1) / kLayoutMinTileAssign * kLayoutMinTileAssign;
    if (t < kLayoutMinTileAssign) t = kLayoutMinTileAssign;
    if (t > kLayoutMaxTileAssign) t = kLayoutMaxTileAssign;
    const int tt = (int)(t / k);
    return tt < 1 ? 1 : tt;
}
__host__ __device__ inline int layout_tiles(long long T, int k)
{
    const long long tt = layout_tile_tokens(T, k);
    const long long n = (T + tt - 1) / tt;
    return n < 1 ? 1 : (int)n;
}

// The route kernel's histogram region: after the layout's flag words.
__host__ __device__ inline unsigned *ws_route_hist(void *ws, long long T, int k, int E)
{
    return reinterpret_cast<unsigned *>(static_cast<char *>(ws) + kWsHeaderBytes +
                                        (size_t)layout_tiles(T, k) * (size_t)E * sizeof(unsigned long long));
}

// Fused route kernel tiling (gate and layout in one launch, one bounded
// grid-wide wait): at most kRouteMaxTiles tiles of at least
// kRouteMinTileTokens tokens.  Its per-tile histograms (one 32-bit count per
// (tile, expert)) live in their own region after the layout's flag words,
// so neither kernel can mistake the other's words for its own.
constexpr int kRouteMinTileTokens = 32;
constexpr int kRouteMaxTiles = 1024;
__host__ __device__ inline int route_tiles_bound(long long T)
{
    long long n = (T + kRouteMinTileTokens - 1) / kRouteMinTileTokens;
    if (n < 1) n = 1;
    return n > kRouteMaxTiles ? kRouteMaxTiles : (int)n;
}

// Flag word: [63:32] epoch, [31:30] state, [29:0] value.
constexpr unsigned long long kFlagAggregate = 1ull;
constexpr unsigned long long kFlagInclusive = 2ull;
__device__ __forceinline__ unsigned long long make_flag(unsigned epoch, unsigned long long state, unsigned value)
{
    return (static_cast<unsigned long long>(epoch) << 32) | (state << 30) | (value & 0x3FFFFFFFu);
}

// Bound on any spin-wait, in nanoseconds of %globaltimer.
constexpr unsigned long long kSpinLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_status(void *ws, unsigned code)
{
    if (ws) atomicCAS(&static_cast<WsHeader *>(ws)->status, 0u, code);
}

// Rows that a call reads or writes once (token rows, packed rows, expert
// outputs, y, FP8 codes) may go through L2 with an evict-first policy, so
// that what the next calls reuse -- their code, the router logits, the
// routing metadata and the workspace, a few MB -- stays in L2 while hundreds
// of MB of rows stream through it.  Each kernel picks evict-first or the
// normal policy by what was measured for it, and creates the policy once
// per thread.
#ifndef MOE_L2_STREAM_HINT
#define MOE_L2_STREAM_HINT 1
#endif
__device__ __forceinline__ uint64_t l2_stream_policy(bool evict_first)
{
    uint64_t pol = 0;
#if MOE_L2_STREAM_HINT
    if (evict_first) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
#endif
    return pol;
}

// Streaming 16-byte load (read once: not kept in L1, evicted first from L2).
__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p, uint64_t pol)
{
    uint4 v;
#if MOE_L2_STREAM_HINT
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
#else
    (void)pol;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#endif
    return v;
}

// Streaming 16-byte store (written once: evicted first from L2).
__device__ __forceinline__ void st_stream_v4(uint4 *p, const uint4 &v, uint64_t pol)
{
#if MOE_L2_STREAM_HINT
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
#else
    (void)pol;
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
#endif
}

// 32-byte vectors (sm_100 and later move 256 bits per load or store
// instruction: half the load/store instructions of 16-byte vectors).  The
// address must be 32-byte aligned.
struct __align__(32) u32x8 {
    uint4 lo, hi;
};

__device__ __forceinline__ u32x8 ld_stream_v8(const u32x8 *p, uint64_t pol)
{
    u32x8 v;
#if MOE_L2_STREAM_HINT
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                 : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x), "=r"(v.hi.y), "=r"(v.hi.z),
                   "=r"(v.hi.w)
                 : "l"(p), "l"(pol));
#else
    (void)pol;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x), "=r"(v.hi.y), "=r"(v.hi.z),
                   "=r"(v.hi.w)
                 : "l"(p));
#endif
    return v;
}

__device__ __forceinline__ void st_stream_v8(u32x8 *p, const u32x8 &v, uint64_t pol)
{
#if MOE_L2_STREAM_HINT
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p),
                 "r"(v.lo.x), "r"(v.lo.y), "r"(v.lo.z), "r"(v.lo.w), "r"(v.hi.x), "r"(v.hi.y), "r"(v.hi.z),
                 "r"(v.hi.w), "l"(pol)
                 : "memory");
#else
    (void)pol;
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.lo.x), "r"(v.lo.y),
                 "r"(v.lo.z), "r"(v.lo.w), "r"(v.hi.x), "r"(v.hi.y), "r"(v.hi.z), "r"(v.hi.w)
                 : "memory");
#endif
}

// Programmatic dependent launch.  Every kernel of the path is launched so
// that it may start while the previous kernel in the stream finishes.  It
// first waits for that kernel to complete (all its memory visible), and only
// then allows the next kernel to launch, so "kernel N+1 running" implies
// "kernel N-1 complete".  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// bf16 pair (one 32-bit word) -> two fp32
__device__ __forceinline__ float bf16lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(unsigned w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace moe

namespace moe {
int device_sm_count();

// Blocks of `fn` that fit on the device at once (per SM, for `threads` per
// block and `smem` bytes of dynamic shared memory, times the SM count):
// the grid of a persistent kernel.  Cached per kernel, shape and device.
int resident_grid(const void *fn, int threads, size_t smem);

// Allow `fn` up to `bytes` of dynamic shared memory on the current device
// (once per kernel, device and size; static + dynamic above 48 KiB needs it).
cudaError_t allow_dynamic_smem(const void *fn, int bytes);

// Launch `kernel` on `s` with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
}  // namespace moe
