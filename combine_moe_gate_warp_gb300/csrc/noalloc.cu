// noalloc.cu -- moe_dispatch_layout_noalloc: the dispatch layout for callers
// that may not allocate device memory.  Its scratch (the workspace that
// moe_dispatch_layout otherwise takes from the caller) is a fixed array
// compiled into the library; see include/moe_route.h for the contract.
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "launchers.h"

namespace {

// The scratch itself.  Zero-initialised when the module loads on a device;
// every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) unsigned char g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// In host code `g_layout_scratch` names a host-side stand-in, not device
// memory: the device address must be looked up per device, with that device
// current, and that address is what the kernels receive.
moe_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_dispatch_layout_noalloc(const int32_t *topk_idx, const int32_t *expert_counts,
                                                  int T, int E, int k, int P, int capacity,
                                                  float *gates_or_null, moe_layout *L,
                                                  moe_stream_t stream)
{
    const size_t need = moe_workspace_size(T, E, k, P);
    if (need == 0) {
        // unsupported sizes: let the regular entry point report the exact code
        return moe_dispatch_layout(topk_idx, expert_counts, T, E, k, P, capacity, gates_or_null, L,
                                   nullptr, 0, stream);
    }
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
    // the argument checks of moe_dispatch_layout, done before anything is enqueued
    if (!L || !expert_counts || (T > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
    if (!L->counts || !L->offsets || !L->part_rows || !L->part_offsets || !L->part_tokens ||
        !L->dropped || (T > 0 && (!L->src_pos || !L->dst_row || !L->capacity_mask)))
        return MOE_ERR_INVALID_ARG;
    void *scratch = nullptr;
    moe_status st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    // Counters that each layout call expects at zero (they are reset by a
    // completed call; an aborted one could leave them dirty): the done and
    // gate tickets, the test hook, the tile-id half of the tile/epoch word,
    // and the partition-token totals.  The status word and the flag epoch
    // are kept: the epoch tags old flag words so they are never mistaken for
    // this call's.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(scratch);
    const size_t c0 = offsetof(moe::WsHeader, done_ctr);
    const size_t c1 = offsetof(moe::WsHeader, tile_epoch) + sizeof(unsigned);  // low (tile) half, little-endian
    if (cudaMemsetAsync(base + c0, 0, c1 - c0, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(base + offsetof(moe::WsHeader, part_tok), 0,
                        sizeof(((moe::WsHeader *)nullptr)->part_tok), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_dispatch_layout(topk_idx, expert_counts, T, E, k, P, capacity, gates_or_null, L, scratch,
                               MOE_NOALLOC_SCRATCH_BYTES, stream);
}
