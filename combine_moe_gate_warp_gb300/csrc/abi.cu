// abi.cu -- the extern "C" entry points declared in include/moe_route.h.
// Each call validates its arguments on the host (nothing is enqueued when
// they are bad) and then launches the kernels of one step on `stream`.
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "launchers.h"

namespace moe {

int device_sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int resident_grid(const void *fn, int threads, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, size_t, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(fn, threads, smem, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1) n = 1;
    const int grid = n * device_sm_count();
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = grid;
    return grid;
}

cudaError_t allow_dynamic_smem(const void *fn, int bytes)
{
    // The attribute is a per-kernel maximum: only ever raise it, so a later
    // smaller request never lowers the limit a larger launch relies on.
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> limit;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    int &cur = limit[std::make_pair(fn, dev)];
    if (bytes <= cur) return cudaSuccess;
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess) cur = bytes;
    return err;
}

}  // namespace moe

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sizes of the layout, dispatch and combine calls.  k may exceed E there: a
// row of a de-duplicated receive buffer has up to k slots over the
// partition's experts, the unused ones empty (-1).
inline moe_status check_sizes(int T, int E, int k)
{
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
    if (k < 1 || k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// The gate selects k distinct experts: k <= E as well.
inline moe_status check_gate_sizes(int T, int E, int k)
{
    const moe_status st = check_sizes(T, E, k);
    if (st != MOE_OK) return st;
    return k > E ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

inline moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

size_t moe_workspace_size(int T, int E, int k, int P)
{
    if (check_sizes(T, E, k) != MOE_OK) return 0;
    if (P < 1 || P > E || E % P != 0) return 0;
    // header, the layout's look-back flag words, moe_route's tile histograms
    return moe::kWsHeaderBytes + (size_t)moe::layout_tiles(T, k) * (size_t)E * sizeof(unsigned long long) +
           (size_t)moe::route_tiles_bound(T) * (size_t)E * sizeof(unsigned);
}

moe_status moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!ws || ws_bytes < moe::kWsHeaderBytes) return MOE_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t moe_rows_max(int T, int E, int k, int capacity)
{
    if (check_sizes(T, E, k) != MOE_OK) return -1;
    const int64_t A = (int64_t)T * k;
    if (capacity <= 0) return A;
    const int64_t c = (int64_t)E * capacity;
    return c < A ? c : A;
}

moe_status moe_gate(const float *logits, int T, int E, int k, int mode, int32_t *topk_idx,
                    float *gates, int32_t *expert_counts, double *aux_loss, double *entropy,
                    void *ws, size_t ws_bytes, moe_stream_t stream)
{
    moe_status st = check_gate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (mode != MOE_TOPK_SOFTMAX && mode != MOE_SOFTMAX_TOPK) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !aux_loss || !entropy || !ws) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !gates)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(gates) || !aligned16(ws))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe::kWsHeaderBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return from_cuda(moe::launch_gate(logits, T, E, k, mode, topk_idx, gates, expert_counts, aux_loss,
                                      entropy, ws, reinterpret_cast<cudaStream_t>(stream)));
}

static moe_status dispatch_layout_impl(const int32_t *topk_idx, const int32_t *expert_counts, int T, int E,
                                       int k, int P, int capacity, float *gates_or_null, moe_layout *L,
                                       void *ws, size_t ws_bytes, moe_stream_t stream, int reassign)
{
    moe_status st = check_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (P < 1 || P > E || E % P != 0) return MOE_ERR_UNSUPPORTED;
    if (!L || !expert_counts || !ws) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !topk_idx) return MOE_ERR_INVALID_ARG;
    if (!L->counts || !L->offsets || !L->part_rows || !L->part_offsets || !L->part_tokens ||
        !L->dropped || (T > 0 && (!L->src_pos || !L->dst_row || !L->capacity_mask)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_workspace_size(T, E, k, P)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    L->T = T;
    L->E = E;
    L->k = k;
    L->P = P;
    L->capacity = capacity > 0 ? capacity : 0;
    L->r_max = (int32_t)moe_rows_max(T, E, k, capacity);
    L->ws = ws;
    return from_cuda(moe::launch_layout(topk_idx, expert_counts, T, E, k, P, capacity, gates_or_null, L,
                                        ws, reinterpret_cast<cudaStream_t>(stream), reassign));
}

moe_status moe_dispatch_layout(const int32_t *topk_idx, const int32_t *expert_counts, int T, int E,
                               int k, int P, int capacity, float *gates_or_null, moe_layout *L,
                               void *ws, size_t ws_bytes, moe_stream_t stream)
{
    return dispatch_layout_impl(topk_idx, expert_counts, T, E, k, P, capacity, gates_or_null, L, ws, ws_bytes,
                                stream, 0);
}

moe_status moe_dispatch_layout_reassign(const int32_t *topk_idx, const int32_t *expert_counts, int T, int E,
                                        int k, int P, int capacity, float *gates_or_null, moe_layout *L,
                                        void *ws, size_t ws_bytes, moe_stream_t stream)
{
    return dispatch_layout_impl(topk_idx, expert_counts, T, E, k, P, capacity, gates_or_null, L, ws, ws_bytes,
                                stream, 1);
}

moe_status moe_route(const float *logits, int T, int E, int k, int mode, int P, int capacity, int32_t *topk_idx,
                     float *gates, int32_t *expert_counts, double *aux_loss, double *entropy, moe_layout *L,
                     void *ws, size_t ws_bytes, moe_stream_t stream)
{
    // the argument checks of moe_gate and moe_dispatch_layout
    moe_status st = check_gate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (mode != MOE_TOPK_SOFTMAX && mode != MOE_SOFTMAX_TOPK) return MOE_ERR_INVALID_ARG;
    if (P < 1 || P > E || E % P != 0) return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !aux_loss || !entropy || !ws || !L) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !gates)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(gates) || !aligned16(ws))
        return MOE_ERR_INVALID_ARG;
    if (!L->counts || !L->offsets || !L->part_rows || !L->part_offsets || !L->part_tokens || !L->dropped ||
        (T > 0 && (!L->src_pos || !L->dst_row || !L->capacity_mask)))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_workspace_size(T, E, k, P)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    L->T = T;
    L->E = E;
    L->k = k;
    L->P = P;
    L->capacity = capacity > 0 ? capacity : 0;
    L->r_max = (int32_t)moe_rows_max(T, E, k, capacity);
    L->ws = ws;
    int too_large = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = moe::launch_route(logits, T, E, k, mode, P, capacity, topk_idx, gates, expert_counts,
                                        aux_loss, entropy, L, ws, s, &too_large);
    if (too_large) {
        // nothing enqueued: the batch does not fit the fused kernel's grid;
        // the gate and layout kernels give the same outputs in two launches
        err = moe::launch_gate(logits, T, E, k, mode, topk_idx, gates, expert_counts, aux_loss, entropy, ws, s);
        if (err == cudaSuccess)
            err = moe::launch_layout(topk_idx, expert_counts, T, E, k, P, capacity, gates, L, ws, s, 0);
    }
    return from_cuda(err);
}

int moe_route_launches(int T, int E, int k, int mode, int P)
{
    if (check_gate_sizes(T, E, k) != MOE_OK) return 0;
    if (mode != MOE_TOPK_SOFTMAX && mode != MOE_SOFTMAX_TOPK) return 0;
    if (P < 1 || P > E || E % P != 0) return 0;
    int too_large = 0;
    if (moe::launch_route(nullptr, T, E, k, mode, P, 0, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                          nullptr, nullptr, &too_large, true) != cudaSuccess)
        return 0;
    return too_large ? 2 : 1;
}

static moe_status check_layout(const moe_layout *L, int T)
{
    if (!L || !L->ws || !L->offsets || (T > 0 && !L->dst_row)) return MOE_ERR_INVALID_ARG;
    if (L->T != T) return MOE_ERR_INVALID_ARG;
    return check_sizes(L->T, L->E, L->k);
}

moe_status moe_dispatch(const void *x, int T, int H, const moe_layout *L, int fp8, void *packed,
                        float *scales, moe_stream_t stream)
{
    moe_status st = check_layout(L, T);
    if (st != MOE_OK) return st;
    if (fp8 < 0 || fp8 > MOE_FP8_GLOBAL) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (fp8 && (H % 16 != 0 || H > MOE_MAX_H_FP8)) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !packed || (fp8 && !scales))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fp8 != 0) return from_cuda(moe::launch_dispatch_fp8_grouped(x, T, H, L, fp8, packed, scales, s));
    return from_cuda(moe::launch_dispatch_bf16(x, T, H, L, packed, s));
}

moe_status moe_combine(const void *expert_out, const moe_layout *L, const float *gates,
                       const void *shared_out, int Ks, int T, int H, void *y, moe_stream_t stream)
{
    moe_status st = check_layout(L, T);
    if (st != MOE_OK) return st;
    if (H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (Ks < 0 || Ks > MOE_MAX_SHARED) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!expert_out || !gates || !y || (Ks > 0 && !shared_out))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(expert_out) || !aligned16(y) || !aligned16(shared_out)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine(expert_out, L, gates, Ks > 0 ? shared_out : nullptr, Ks, T, H, y,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_rows(const void *rows, const moe_layout *L, int H, int mode, void *codes, float *scales,
                             moe_stream_t stream)
{
    if (!L) return MOE_ERR_INVALID_ARG;
    moe_status st = check_layout(L, L->T);
    if (st != MOE_OK) return st;
    if (mode < MOE_FP8_PER_TOKEN || mode > MOE_FP8_GLOBAL) return MOE_ERR_INVALID_ARG;
    if (H < 16 || H % 16 != 0 || H > MOE_MAX_H_FP8) return MOE_ERR_UNSUPPORTED;
    if (L->r_max > 0 && (!rows || !codes || !scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(rows) || !aligned16(codes) || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_quantize_rows(rows, L, H, mode, codes, scales, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_fp8(const void *codes, const float *scales, const moe_layout *L, const float *gates,
                           const void *shared_out, int Ks, int T, int H, void *y, moe_stream_t stream)
{
    moe_status st = check_layout(L, T);
    if (st != MOE_OK) return st;
    if (H < 16 || H % 16 != 0) return MOE_ERR_UNSUPPORTED;
    if (Ks < 0 || Ks > MOE_MAX_SHARED) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!codes || !scales || !gates || !y || (Ks > 0 && !shared_out))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(y) || !aligned16(shared_out)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine_fp8(codes, scales, L, gates, Ks > 0 ? shared_out : nullptr, Ks, T, H, y,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_backward(const void *dy, const void *expert_out, const moe_layout *L, const float *gates,
                                int T, int H, void *d_expert_out, float *d_gates, moe_stream_t stream)
{
    moe_status st = check_layout(L, T);
    if (st != MOE_OK) return st;
    if (H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!dy || !expert_out || !gates || !d_expert_out || !d_gates)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(expert_out) || !aligned16(d_expert_out)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine_backward(dy, expert_out, L, gates, T, H, d_expert_out, d_gates,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_backward(const void *d_packed, const moe_layout *L, int T, int H, void *dx,
                                 moe_stream_t stream)
{
    moe_status st = check_layout(L, T);
    if (st != MOE_OK) return st;
    if (H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!d_packed || !dx)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(d_packed) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine(d_packed, L, nullptr, nullptr, 0, T, H, dx,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_gate_backward(const float *logits, const int32_t *topk_idx, const float *d_gates, int T, int E,
                             int k, int mode, float *d_logits, void *ws, size_t ws_bytes, moe_stream_t stream)
{
    moe_status st = check_gate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (mode != MOE_TOPK_SOFTMAX && mode != MOE_SOFTMAX_TOPK) return MOE_ERR_INVALID_ARG;
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !d_gates || !d_logits)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe::kWsHeaderBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return from_cuda(moe::launch_gate_backward(logits, topk_idx, d_gates, T, E, k, mode, d_logits, ws,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_dedup_scratch_size(int T, int P)
{
    if (T < 0 || P < 1 || P > 16) return 0;
    return moe::dedup_scratch_bytes(T, P);
}

// A layout view of the send rows: P slots per token, rows = send rows.
static moe_layout dedup_view(const moe_dedup *D)
{
    moe_layout v = {};
    v.T = D->T;
    v.E = D->P;
    v.k = D->P;
    v.P = 1;
    v.r_max = D->s_max;
    v.ws = D->ws;
    v.offsets = D->send_offsets;
    v.dst_row = D->send_row;
    return v;
}

moe_status moe_dedup_layout(const moe_layout *L, const float *gates, moe_dedup *D, void *scratch,
                            size_t scratch_bytes, moe_stream_t stream)
{
    if (!L || !D) return MOE_ERR_INVALID_ARG;
    moe_status st = check_layout(L, L->T);
    if (st != MOE_OK) return st;
    if (L->P < 1 || L->P > 16) return MOE_ERR_UNSUPPORTED;
    if (!D->send_offsets || (L->T > 0 && (!gates || !scratch || !D->send_row || !D->send_token || !D->slot_local ||
                                          !D->slot_gate)))
        return MOE_ERR_INVALID_ARG;
    if (L->T > 0 && scratch_bytes < moe::dedup_scratch_bytes(L->T, L->P)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    D->T = L->T;
    D->k = L->k;
    D->P = L->P;
    D->s_max = L->T * (L->k < L->P ? L->k : L->P);
    D->ws = L->ws;
    return from_cuda(moe::launch_dedup_layout(L, gates, D, scratch, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_dedup(const void *x, int T, int H, const moe_dedup *D, int fp8, void *send_buf,
                              float *scales, moe_stream_t stream)
{
    if (!D || !D->send_offsets || D->T != T || D->P < 1 || D->P > 16) return MOE_ERR_INVALID_ARG;
    if (fp8 != 0 && fp8 != MOE_FP8_PER_TOKEN) return MOE_ERR_UNSUPPORTED;
    if (H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (fp8 && (H % 16 != 0 || H > MOE_MAX_H_FP8)) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !send_buf || !D->send_row || (fp8 && !scales))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(send_buf) || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
    const moe_layout v = dedup_view(D);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(fp8 ? moe::launch_dispatch_fp8_grouped(x, T, H, &v, MOE_FP8_PER_TOKEN, send_buf, scales, s)
                         : moe::launch_dispatch_bf16(x, T, H, &v, send_buf, s));
}

moe_status moe_combine_partials(const void *partials, const moe_dedup *D, const void *shared_out, int Ks, int T,
                                int H, void *y, moe_stream_t stream)
{
    if (!D || !D->send_offsets || D->T != T || D->P < 1 || D->P > 16) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (Ks < 0 || Ks > MOE_MAX_SHARED) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!partials || !y || !D->send_row || (Ks > 0 && !shared_out))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(partials) || !aligned16(y) || !aligned16(shared_out)) return MOE_ERR_INVALID_ARG;
    const moe_layout v = dedup_view(D);
    return from_cuda(moe::launch_combine(partials, &v, nullptr, Ks > 0 ? shared_out : nullptr, Ks, T, H, y,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_get_status(void *ws, moe_stream_t stream)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    unsigned status = 0;
    if (cudaMemcpy(&status, ws, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (status != 0) {
        if (cudaMemsetAsync(ws, 0, sizeof(status), s) != cudaSuccess) return MOE_ERR_CUDA;
        if (status == MOE_ERR_TIMEOUT) {
            // a wait of moe_route expired: its grid barrier may hold arrivals
            // and totals of the unfinished call; the stream is idle, so
            // re-arm it (arrivals and both total arrays to zero, generation kept)
            char *base = static_cast<char *>(ws);
            if (cudaMemsetAsync(base + offsetof(moe::WsHeader, route_bar), 0, sizeof(unsigned), s) != cudaSuccess ||
                cudaMemsetAsync(base + offsetof(moe::WsHeader, route_counts), 0,
                                sizeof(((moe::WsHeader *)nullptr)->route_counts), s) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return (moe_status)status;
}

const char *moe_status_string(moe_status status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or option";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_DATA: return "invalid data found on the device";
    default: return "unknown status";
    }
}

}  // extern "C"
