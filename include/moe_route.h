/*
 * moe_route.h -- C ABI of libmoeroute, the GB300 (sm_103a) CUDA library for
 * the token-routing hot path of a Mixture-of-Experts layer:
 *
 *     moe_gate -> moe_dispatch_layout -> moe_dispatch -> (expert FFN) -> moe_combine
 *
 * and its backward through the same layout:
 *
 *     moe_combine_backward -> (expert FFN backward) -> moe_dispatch_backward
 *     moe_gate_backward (gate gradients -> router-logit gradients)
 *
 * Source pages cited below:
 *   [P1] "Deepseek-MoE sync-tax essence and four-layer optimisation guide"
 *        (gsyq.cn news 1572160)
 *   [P2] "DeepSeek MoE sync tax" (wmrh.cn news 47329)
 *   [P3] "DeepSeek MoE architecture evolution" (lpnh.cn news 699721)
 *   [P4] "MoE data traits ... DeepEP and MoE all-to-all data handling"
 *        (zzszmyf.github.io notes, mirror of a Zhihu article)
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array argument is a DEVICE pointer owned by the caller.  The
 *   library never allocates, frees or synchronises inside the four hot
 *   calls; they only enqueue kernels on `stream` and return.
 * - Array base pointers must be 16-byte aligned (128-bit vector access);
 *   a misaligned pointer is MOE_ERR_INVALID_ARG.
 * - Argument errors are detected on the host before anything is enqueued:
 *   such a call has no effect.  Problems found on the device (out-of-range
 *   expert ids, non-finite logits, inconsistent counts, an expired wait)
 *   are recorded in a status word inside the workspace and read back with
 *   moe_get_status().  Kernels never trap; they skip the bad element.
 * - A "workspace" is a caller-owned device buffer of moe_workspace_size()
 *   bytes, zeroed once by moe_workspace_init().  The gate and layout calls
 *   use it for counters and cross-block flags and leave it clean for the
 *   next call.  One workspace serves calls issued in order on ONE stream;
 *   calls that may run concurrently need separate workspaces.
 * - Assignment a = t*k + j is slot j (descending logit order) of token t.
 * - bf16 tensors are raw 16-bit bfloat16 patterns; e4m3 codes are bytes in
 *   the OCP "E4M3FN" encoding.
 *
 * Supported range: 1 <= E <= 256, 1 <= k <= 16 (k <= E for the gate; the
 * layout, dispatch and combine also take k > E, for rows with empty slots),
 * 1 <= P <= E with E % P == 0, 0 <= T and T*k < 2^30, H % 8 == 0 (H % 16 == 0
 * and H <= 16384 for FP8), 0 <= Ks <= 8.  Anything else is
 * MOE_ERR_UNSUPPORTED; there is no fallback path.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef int moe_status;
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1          /* null/misaligned pointer, bad enum, T < 0 */
#define MOE_ERR_UNSUPPORTED 2          /* outside the supported range above */
#define MOE_ERR_WORKSPACE_TOO_SMALL 3  /* ws_bytes < moe_workspace_size(...) */
#define MOE_ERR_CUDA 4                 /* a CUDA runtime call or launch failed */
#define MOE_ERR_TIMEOUT 5              /* device: a cross-block wait expired */
#define MOE_ERR_DEVICE_DATA 6          /* device: bad expert id / non-finite logit / counts mismatch */

/* Gate modes. */
#define MOE_TOPK_SOFTMAX 0  /* softmax over the k selected logits ([P3] ch.1 top2_gating) */
#define MOE_SOFTMAX_TOPK 1  /* softmax over all E logits, keep the k selected, no renormalisation
                               (DeepSeekMoE fine-grained routing, [P2] sec. 2.1 and 4.1) */

/* FP8 quantiser modes ([P1] sec. 5.2: per-token, per-expert and global),
 * for moe_dispatch's `fp8` argument and moe_quantize_rows.  One affine
 * (scale, zero) pair per group, from the max and min over every element of
 * the group's rows ([P1] sec. 3.1's per-token formula). */
#define MOE_FP8_PER_TOKEN 1   /* each packed row is its own group */
#define MOE_FP8_PER_EXPERT 2  /* the rows sent to one expert */
#define MOE_FP8_GLOBAL 3      /* every transported row */

#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 16
#define MOE_MAX_SHARED 8
#define MOE_MAX_H_FP8 16384

/*
 * Routing metadata written by moe_dispatch_layout and read by moe_dispatch
 * and moe_combine: the target/source index maps the dispatch saves so that
 * the combine needs no second routing ([P4] sec. 7.5.2, "indices" and
 * "locations").  The struct itself lives in host memory; its array members
 * are caller-allocated DEVICE buffers of the sizes shown.  The scalar
 * members and `ws` are filled in by moe_dispatch_layout.
 */
typedef struct moe_layout {
    int32_t T, E, k, P;      /* filled by moe_dispatch_layout */
    int32_t capacity;        /* per-expert row limit, 0 = none (filled) */
    int32_t r_max;           /* rows that packed buffers must hold (filled) */
    void *ws;                /* workspace used for device status (filled) */
    int32_t *counts;         /* [E]   kept rows per expert = min(count_e, capacity) */
    int32_t *offsets;        /* [E+1] exclusive prefix of counts; offsets[E] = R */
    int32_t *part_rows;      /* [P]   rows of logical partition p (experts p*E/P ..) */
    int32_t *part_offsets;   /* [P+1] first packed row of partition p; [P] = R */
    int32_t *part_tokens;    /* [P]   tokens with >= 1 kept assignment in partition p */
    int32_t *src_pos;        /* [r_max] packed row -> assignment a (rows >= R untouched) */
    int32_t *dst_row;        /* [T*k] assignment -> packed row, -1 if dropped */
    uint8_t *capacity_mask;  /* [T*k] 1 kept, 0 dropped */
    int64_t *dropped;        /* [1]   T*k - R */
} moe_layout;

/* Bytes of workspace needed by moe_gate, moe_dispatch_layout and
 * moe_route for these sizes (0 if the sizes are unsupported). */
size_t moe_workspace_size(int T, int E, int k, int P);

/* Zero a workspace (cudaMemsetAsync on `stream`).  Needed once after
 * allocation, and again only if a kernel using it was aborted. */
moe_status moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* Packed rows the layout can produce: T*k, or min(T*k, E*capacity). */
int64_t moe_rows_max(int T, int E, int k, int capacity);

/*
 * moe_gate -- top-k gating over router logits, with routing statistics.
 * [P3] ch.1 (top2_gating: torch.topk, softmax of the selected logits, aux
 * loss = E * sum_e f_e^2); [P3] sec. 2.3 (entropy of the expert counts);
 * [P2] sec. 4.1 (softmax over all experts then top-k).
 *
 *   logits        [T, E] fp32, row-major.  Must be finite (else
 *                 MOE_ERR_DEVICE_DATA is recorded).
 *   topk_idx  out [T, k] int32: the k largest logits per token, value
 *                 descending, equal values to the lower expert id
 *                 (-0.0 equals +0.0).
 *   gates     out [T, k] fp32 gate weights (mode above), fp32 arithmetic.
 *   expert_counts out [E] int32: assignments per expert (sums to T*k).
 *   aux_loss  out [1] fp64: E * sum_e (count_e / T)^2.
 *   entropy   out [1] fp64: -sum_e p_e log2(p_e + 1e-8), p_e = count_e / (T*k).
 *                 Both are 0 when T == 0.
 *   ws, ws_bytes  workspace (>= moe_workspace_size(T, E, k, 1)).
 */
moe_status moe_gate(const float *logits, int T, int E, int k, int mode,
                    int32_t *topk_idx, float *gates, int32_t *expert_counts,
                    double *aux_loss, double *entropy,
                    void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_dispatch_layout -- per-expert and per-partition counts, prefix
 * offsets and the stable permutation.  [P4] sec. 7 "Dispatch" detail
 * (reorder by target expert id, pack same-destination tokens
 * contiguously); sec. 7.5.4 (sparse-aware packing: valid tokens only, no
 * padding); sec. 8.3.A (strict per-expert capacity; assignments over it
 * are taken in order and here dropped).
 *
 *   topk_idx       [T, k] int32 from moe_gate (ids outside [0, E) are
 *                  recorded as MOE_ERR_DEVICE_DATA and treated as dropped;
 *                  -1 marks an empty slot, e.g. of a de-duplicated receive
 *                  row with fewer than k experts: no row, no error, and
 *                  expert_counts must not count it).
 *   expert_counts  [E] int32 from moe_gate (must match topk_idx; a
 *                  mismatch is recorded as MOE_ERR_DEVICE_DATA).
 *   P              logical partitions; partition p = experts
 *                  [p*E/P, (p+1)*E/P), a contiguous slice of the packed rows.
 *   capacity       per-expert row limit; <= 0 means none.  Within an expert
 *                  the first `capacity` assignments in token order are kept.
 *   gates_or_null  [T, k] fp32; if given, dropped slots are set to 0.
 *   L              host struct with caller-allocated device arrays
 *                  (see moe_layout); scalar members are filled in here.
 *   ws, ws_bytes   workspace (>= moe_workspace_size(T, E, k, P)), the same
 *                  one moe_gate used is fine.
 * Packed row of a kept assignment: offsets[e] + (its rank within expert e).
 * R = offsets[E] stays on the device; size packed buffers with L->r_max.
 */
moe_status moe_dispatch_layout(const int32_t *topk_idx, const int32_t *expert_counts,
                               int T, int E, int k, int P, int capacity,
                               float *gates_or_null, moe_layout *L,
                               void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_route -- moe_gate followed by moe_dispatch_layout (dropping capacity
 * or none), with exactly their outputs: topk_idx, gates (dropped slots set
 * to 0), expert_counts, aux_loss, entropy and every moe_layout array, in
 * one kernel launch where the batch allows.  [P2] sec. 4.3 fuses the
 * routing kernels (gate, softmax, top-k) into one launch to cut their
 * latency; here the layout joins them.  Definitions: those of moe_gate
 * ([P3] ch.1, sec. 2.3; [P2] sec. 4.1) and moe_dispatch_layout ([P4] sec.
 * 7, 7.5.4, 8.3.A).
 *
 *   Arguments: those of moe_gate and of moe_dispatch_layout (gates is the
 *   layout's gates_or_null), one workspace of moe_workspace_size(T, E, k, P)
 *   bytes.  In the fused kernel every block waits once for all the others
 *   (to learn the per-expert totals before it places rows), so its grid is
 *   sized to the blocks the GPU holds at once (larger tiles for larger
 *   batches); a batch whose tiles would not fit in shared memory runs the
 *   kernels of moe_gate and moe_dispatch_layout instead (two launches, the
 *   same outputs; moe_route_launches tells which).  The wait is bounded (1 s); if it
 *   expires, MOE_ERR_TIMEOUT is recorded in the workspace and the outputs
 *   are incomplete; moe_get_status then also re-arms the workspace, so the
 *   next call is exact.  Capacity re-assignment is not offered here
 *   (moe_dispatch_layout_reassign).
 */
moe_status moe_route(const float *logits, int T, int E, int k, int mode, int P, int capacity,
                     int32_t *topk_idx, float *gates, int32_t *expert_counts, double *aux_loss,
                     double *entropy, moe_layout *L, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Kernel launches moe_route takes for these sizes on the current device: 1
 * (the fused kernel) or 2 (gate and layout kernels); 0 if unsupported.
 * Queries the device's occupancy; enqueues nothing. */
int moe_route_launches(int T, int E, int k, int mode, int P);

/*
 * moe_dispatch_layout_noalloc -- the same layout as moe_dispatch_layout,
 * for callers that cannot allocate device memory.  The source pages have no
 * counterpart to this entry point; it exists for integration only.
 *
 * Some callers are not allowed to allocate: a plug-in running inside a
 * host framework that owns every byte of device memory through its own
 * pool, or a latency-critical loop that must not enter the CUDA allocator
 * (cudaMalloc can synchronise the device and take unbounded time) after
 * start-up.  This variant takes no workspace: it uses a scratch array
 * compiled into the library (a file-scope static __device__ buffer of
 * MOE_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that loads the library
 * until the process exits).  The caller still provides all inputs and the
 * moe_layout output arrays.
 *
 *   Arguments and outputs: as moe_dispatch_layout, minus ws / ws_bytes.
 *   L->ws is set to the scratch's device address, so moe_dispatch,
 *   moe_combine and moe_get_status(L->ws, stream) work as usual.
 *   Sizes whose moe_workspace_size(T, E, k, P) exceeds
 *   MOE_NOALLOC_SCRATCH_BYTES are rejected with MOE_ERR_WORKSPACE_TOO_SMALL
 *   before anything is enqueued.
 *   The first call on each device looks up the scratch's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  Every call clears the scratch counters that
 *   must start at zero.  All calls in the process share the one array, so
 *   calls that may overlap on the GPU (different streams, or several host
 *   threads) race with each other: serialise them.
 *   No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (2u << 20)
moe_status moe_dispatch_layout_noalloc(const int32_t *topk_idx, const int32_t *expert_counts,
                                       int T, int E, int k, int P, int capacity,
                                       float *gates_or_null, moe_layout *L, moe_stream_t stream);

/*
 * moe_dispatch_layout_reassign -- moe_dispatch_layout with the capacity
 * overflow re-assigned instead of dropped ([P4] sec. 8.3.A: greedy top-k
 * under a hard per-expert capacity, then a rolling fallback to the
 * lowest-loaded expert of the batch).  Arguments and outputs as
 * moe_dispatch_layout, in two passes:
 *   1. each expert keeps its first `capacity` assignments in token order;
 *   2. the remaining assignments, in flat order a = t*k + j, each go to the
 *      expert with the lowest current load (ties to the lower id) that is
 *      below capacity, raising its load by one; with none left the
 *      assignment is dropped.
 * counts[e] is the final load (<= capacity); an expert's rows hold its kept
 * assignments in token order, then those it received in the order received.
 * capacity_mask: 1 kept where routed, 2 re-assigned, 0 dropped.  Gates are
 * zeroed for dropped slots only (a re-assigned slot keeps its weight).
 * Partitions and part_tokens follow the final experts.  capacity <= 0: no
 * overflow, identical to moe_dispatch_layout.  Pass 2 runs inside the same
 * kernel: overflow assignment number m (numbered across the batch) takes
 * place m of the water filling in (level, expert) order.
 */
moe_status moe_dispatch_layout_reassign(const int32_t *topk_idx, const int32_t *expert_counts,
                                        int T, int E, int k, int P, int capacity,
                                        float *gates_or_null, moe_layout *L,
                                        void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_dispatch -- permute and pack token hidden states into the
 * expert-contiguous send buffer ([P4] sec. 7 Dispatch detail), optionally
 * as affine FP8 ([P1] sec. 3.1: per-token min/max, affine map; sec. 5.2:
 * per-token, per-expert or global groups).
 *
 *   x       [T, H] bf16.
 *   fp8 = 0: packed [r_max, H] bf16; row r = x[src_pos[r] / k] bit-exactly.
 *   fp8 = MOE_FP8_PER_TOKEN (1): packed [r_max, H] uint8 e4m3 codes, scales
 *            [r_max, 2] fp32 (scale, zero) of the row's token, with (fp32, in
 *            this order) mx, mn = max and min of the row (-0 < +0),
 *            zero = (mx + mn) * 0.5, scale = (mx - mn) / 896,
 *            code = e4m3 satfinite RNE((x - zero) / scale);
 *            a constant row has scale 0 and all-zero codes.
 *            Dequantise as zero + scale * e4m3_value(code).  x must be finite.
 *   fp8 = MOE_FP8_PER_EXPERT (2) / MOE_FP8_GLOBAL (3): the same, with mx, mn
 *            taken over every element of the rows sent to the row's expert /
 *            of every transported row; scales still holds the pair per row.
 *            Two kernels (extremes, then codes), which use the workspace L->ws
 *            and leave it clean.
 *   Rows >= R are not written.
 *   x and packed must be 16-byte aligned; for fp8 = 0 with both 32-byte
 *   aligned and H a multiple of 16, the copy moves 32-byte vectors (fewer
 *   load/store instructions: faster for large k).
 */
moe_status moe_dispatch(const void *x, int T, int H, const moe_layout *L, int fp8,
                        void *packed, float *scales, moe_stream_t stream);

/*
 * moe_combine -- gather the expert outputs back into token order and
 * gate-weight them ([P4] sec. 7 "Combine": weighted sum of each token's
 * top-k expert outputs, placed by the saved routing metadata), adding the
 * shared experts' outputs with weight 1 ([P4] sec. 8.2.B; [P2] sec. 2.1).
 *
 *   expert_out  [r_max, H] bf16, packed-row layout (row r = output of the
 *               expert for assignment src_pos[r]).
 *   gates       [T, k] fp32 (as left by the layout: dropped slots are 0).
 *   shared_out  [Ks, T, H] bf16 or NULL when Ks == 0.
 *   y       out [T, H] bf16:
 *     acc = 0; for kept j ascending: acc = fmaf(g[t,j], eo[dst_row[t,j]], acc);
 *     for s ascending: acc = acc + shared[s,t]; y = bf16 round-to-nearest-even(acc).
 */
moe_status moe_combine(const void *expert_out, const moe_layout *L, const float *gates,
                       const void *shared_out, int Ks, int T, int H, void *y,
                       moe_stream_t stream);

/*
 * moe_quantize_rows -- affine FP8 encode of packed bf16 rows, e.g. the
 * expert outputs before they travel back to the combine ([P1] sec. 3.1: the
 * per-token map applies to each token's expert output vector; sec. 5.2:
 * per-token, per-expert or global groups).
 *
 *   rows      [r_max, H] bf16 in the packed-row layout of L (rows >= R are
 *             neither read nor written).
 *   mode      MOE_FP8_PER_TOKEN (each row its own group), MOE_FP8_PER_EXPERT
 *             (rows offsets[e] .. offsets[e+1]-1), MOE_FP8_GLOBAL (rows 0..R-1).
 *   codes out [r_max, H] uint8 e4m3, scales out [r_max, 2] fp32 (scale, zero),
 *             with the formulas of moe_dispatch.  H % 16 == 0, H <= 16384.
 *   The grouped modes use the workspace L->ws and leave it clean.
 */
moe_status moe_quantize_rows(const void *rows, const moe_layout *L, int H, int mode,
                             void *codes, float *scales, moe_stream_t stream);

/*
 * moe_combine_fp8 -- moe_combine over FP8 expert outputs (codes and
 * (scale, zero) per packed row, as written by moe_quantize_rows):
 *     acc = 0; for kept j ascending:
 *         acc = fmaf(g[t,j], fmaf(scale_r, e4m3_value(code_r), zero_r), acc);
 *     for s ascending: acc = acc + shared[s,t]; y = bf16 RNE(acc)
 * (r = dst_row[t,j]; every operation fp32 round-to-nearest).  Arguments as
 * moe_combine; H % 16 == 0.
 */
moe_status moe_combine_fp8(const void *codes, const float *scales, const moe_layout *L,
                           const float *gates, const void *shared_out, int Ks, int T, int H,
                           void *y, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Per-partition token de-duplication ([P4] sec. 7 dispatch detail: the rows
 * bound for one destination are packed into one block).  A token that keeps
 * several slots in one partition is sent there once, with its local expert
 * ids and gates; the partition expands it to its experts with
 * moe_dispatch_layout (empty slots: id -1), moe_dispatch and the experts,
 * combines them with moe_combine (one partial row per received token) and
 * returns that row; the source adds the partial rows with
 * moe_combine_partials.  Supported: P <= 16.
 * ------------------------------------------------------------------------ */
typedef struct moe_dedup {
    int32_t T, k, P;         /* filled by moe_dedup_layout */
    int32_t s_max;           /* send rows the buffers hold: T * min(k, P) (filled) */
    void *ws;                /* the layout's workspace, for device status (filled) */
    int32_t *send_offsets;   /* [P+1] first send row of partition p; [P] = S */
    int32_t *send_row;       /* [T*P] send row of (t, p), -1 if t keeps no slot in p */
    int32_t *send_token;     /* [s_max] token of each send row (rows >= S untouched) */
    int32_t *slot_local;     /* [s_max*k] local expert ids of the row's slots, -1 past the last */
    float *slot_gate;        /* [s_max*k] their gates, 0 past the last */
} moe_dedup;

/* Bytes of scratch moe_dedup_layout needs (0 if unsupported). */
size_t moe_dedup_scratch_size(int T, int P);

/*
 * moe_dedup_layout -- the send rows of a layout (L from moe_dispatch_layout
 * or moe_dispatch_layout_reassign; the final expert of a kept slot is the
 * expert whose rows hold its dst_row).  Send rows are partition-major and,
 * within a partition, in token order; a row's slots keep the token's slot
 * order, with local ids (expert - p*E/P) and the gates from `gates` [T, k]
 * (as left by the layout).  `scratch` is caller-owned device memory of
 * moe_dedup_scratch_size(T, P) bytes.  Only L's T, E, k, P, r_max, ws,
 * offsets and dst_row are read, so a caller may pass a copy of *L with P
 * set to any divisor of E up to 16 to group the experts differently from
 * the layout's partitions: one group per rank of an expert-parallel
 * exchange whose ranks own several partitions sends a token to a rank once.
 */
moe_status moe_dedup_layout(const moe_layout *L, const float *gates, moe_dedup *D,
                            void *scratch, size_t scratch_bytes, moe_stream_t stream);

/*
 * moe_dispatch_dedup -- copy x[send_token[s]] to send row s of `send_buf`
 * ([s_max, H] bf16, or uint8 e4m3 with per-row (scale, zero) in `scales` for
 * fp8 = MOE_FP8_PER_TOKEN: the token's own pair, as moe_dispatch).
 */
moe_status moe_dispatch_dedup(const void *x, int T, int H, const moe_dedup *D, int fp8,
                              void *send_buf, float *scales, moe_stream_t stream);

/*
 * moe_combine_partials -- y[t] = bf16 RNE of, in fp32 and this order,
 *   acc = 0; acc = acc + partial[send_row[t,p]] for p ascending (p with a
 *   send row); acc = acc + shared[s,t] for s ascending.
 * partials [s_max, H] bf16: the row each partition returned for each send
 * row (rows >= S are not read).
 */
moe_status moe_combine_partials(const void *partials, const moe_dedup *D, const void *shared_out,
                                int Ks, int T, int H, void *y, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward of the path.  The gradients retrace the forward routing through
 * the same layout; nothing is re-routed ([P1] sec. 2.4: the backward
 * exchange mirrors the forward one using the routing indices cached in the
 * forward pass; [P4] sec. 7, detail item 3: the combine stage carries the
 * gradients back, with fp32 accumulation of the gradient sums).  The shared
 * experts' output gradient is dy itself (weight 1) and needs no call.
 * ------------------------------------------------------------------------ */

/*
 * moe_combine_backward -- gradients of moe_combine with respect to the
 * expert outputs and the gates.
 *
 *   dy            [T, H] bf16, gradient of y.
 *   expert_out    [r_max, H] bf16, the combine's input.
 *   gates         [T, k] fp32, the combine's gates.
 *   d_expert_out out [r_max, H] bf16: for every kept slot (t, j) with
 *                 r = dst_row[t,j]: row r = bf16 RNE(fp32(gates[t,j] * dy[t]))
 *                 (one fp32 rounding per element); rows >= R are not written.
 *   d_gates   out [T, k] fp32: sum_h dy[t,h] * expert_out[r,h] accumulated in
 *                 fp32 (each bf16 x bf16 product is exact) in a fixed order of
 *                 summation depth <= H/256 + 14, so |error| <= (H/256 + 14) *
 *                 2^-24 * sum_h |dy[t,h] * expert_out[r,h]|; 0 for dropped
 *                 slots.  Deterministic for fixed (H, k).
 * dst_row entries >= R are recorded as MOE_ERR_DEVICE_DATA and treated as dropped.
 */
moe_status moe_combine_backward(const void *dy, const void *expert_out, const moe_layout *L,
                                const float *gates, int T, int H, void *d_expert_out,
                                float *d_gates, moe_stream_t stream);

/*
 * moe_dispatch_backward -- gradient of moe_dispatch (bf16 transport; for
 * the FP8 transport the quantiser is passed straight through) with respect
 * to x: each token's gradient is the sum of the gradients of its packed
 * copies.
 *
 *   d_packed  [r_max, H] bf16, gradient of the packed rows.
 *   dx    out [T, H] bf16:
 *     acc = 0; for kept j ascending: acc = acc + d_packed[dst_row[t,j]] (fp32);
 *     dx = bf16 RNE(acc).  A token with no kept slot gets 0.
 */
moe_status moe_dispatch_backward(const void *d_packed, const moe_layout *L, int T, int H,
                                 void *dx, moe_stream_t stream);

/*
 * moe_gate_backward -- gradient of the gates with respect to the router
 * logits, the gates recomputed from (logits, topk_idx) in fp32 ([P3] ch.1:
 * softmax of the selected logits; [P2] sec. 4.1: softmax over all experts
 * then top-k).  The selection itself and the aux loss (a function of the
 * counts only) carry no gradient.
 *
 *   logits        [T, E] fp32, the gate's input.
 *   topk_idx      [T, k] int32 from moe_gate (ids outside [0, E) are recorded
 *                 as MOE_ERR_DEVICE_DATA and ignored).
 *   d_gates       [T, k] fp32, gradient of the gates.
 *   d_logits  out [T, E] fp32, with s = sum_j g_j d_gates[t,j]:
 *     MOE_TOPK_SOFTMAX: g = softmax of the selected logits;
 *                       d_logits[sel_j] = g_j (d_gates[t,j] - s), others 0.
 *     MOE_SOFTMAX_TOPK: p = softmax of all E logits, g_j = p[sel_j];
 *                       d_logits[e] = (e == sel_j ? g_j d_gates[t,j] : 0) - p_e s.
 *   ws, ws_bytes  any workspace of >= 8192 bytes (only its status word is used).
 */
moe_status moe_gate_backward(const float *logits, const int32_t *topk_idx, const float *d_gates,
                             int T, int E, int k, int mode, float *d_logits,
                             void *ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream`, return the device status recorded in `ws` since the
 * last call (MOE_OK if none) and clear it. */
moe_status moe_get_status(void *ws, moe_stream_t stream);

/* Static description of a status code. */
const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
