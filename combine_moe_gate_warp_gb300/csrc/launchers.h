// launchers.h -- host-side launchers (one per kernel family), called by the
// C ABI layer after argument validation.  They enqueue on `s` and return the
// CUDA launch status.  Kept apart from common.cuh (the device-side pieces
// every kernel shares), so that adding a call here leaves the kernels'
// sources unchanged.
#pragma once

#include "common.cuh"

namespace moe {
cudaError_t launch_gate(const float *logits, int T, int E, int k, int mode, int32_t *topk_idx,
                        float *gates, int32_t *expert_counts, double *aux, double *entropy,
                        void *ws, cudaStream_t s);
// gate + dropping layout in one launch; *too_large = 1 (nothing enqueued)
// when the batch does not fit the fused kernel's grid; with dry_run only
// that decision is made (nothing is read or launched)
cudaError_t launch_route(const float *logits, int T, int E, int k, int mode, int P, int capacity,
                         int32_t *topk_idx, float *gates, int32_t *expert_counts, double *aux, double *entropy,
                         const moe_layout *L, void *ws, cudaStream_t s, int *too_large, bool dry_run = false);
cudaError_t launch_layout(const int32_t *topk_idx, const int32_t *counts_in, int T, int E, int k,
                          int P, int capacity, float *gates, const moe_layout *L, void *ws,
                          cudaStream_t s, int reassign = 0);
cudaError_t launch_dispatch_bf16(const void *x, int T, int H, const moe_layout *L, void *packed,
                                 cudaStream_t s);
cudaError_t launch_combine(const void *eo, const moe_layout *L, const float *gates,
                           const void *shared, int Ks, int T, int H, void *y, cudaStream_t s);
cudaError_t launch_dispatch_fp8_grouped(const void *x, int T, int H, const moe_layout *L, int mode, void *packed,
                                        float *scales, cudaStream_t s);
cudaError_t launch_quantize_rows(const void *rows, const moe_layout *L, int H, int mode, void *codes, float *scales,
                                 cudaStream_t s);
cudaError_t launch_combine_fp8(const void *codes, const float *scales, const moe_layout *L, const float *gates,
                               const void *shared, int Ks, int T, int H, void *y, cudaStream_t s);
cudaError_t launch_combine_backward(const void *dy, const void *eo, const moe_layout *L, const float *gates, int T,
                                   int H, void *d_eo, float *d_gates, cudaStream_t s);
cudaError_t launch_gate_backward(const float *logits, const int32_t *topk_idx, const float *d_gates, int T, int E,
                                 int k, int mode, float *d_logits, void *ws, cudaStream_t s);
size_t dedup_scratch_bytes(long long T, int P);
cudaError_t launch_dedup_layout(const moe_layout *L, const float *gates, moe_dedup *D, void *scratch,
                                cudaStream_t s);
}  // namespace moe
