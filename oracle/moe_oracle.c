/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for MoE token
 * routing (gate -> dispatch layout -> dispatch -> combine).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load it.  It shares no source, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared -o liboracle.so
 *        moe_oracle.c -lm
 * (-ffp-contract=off: every fp32 expression below rounds once per operator,
 *  exactly as written; no fused multiply-add is formed behind our back.  The
 *  one fused multiply-add the combine definition asks for is spelled fmaf.)
 *
 * Each function cites the passage of the source pages it follows:
 *   [P1] "Deepseek-MoE sync-tax essence and four-layer optimisation guide"
 *        (gsyq.cn news 1572160)
 *   [P2] "DeepSeek MoE sync tax" (wmrh.cn news 47329)
 *   [P3] "DeepSeek MoE architecture evolution" (lpnh.cn news 699721)
 *   [P4] "MoE data traits ... DeepEP and MoE all-to-all data handling"
 *        (zzszmyf.github.io notes, mirror of a Zhihu article)
 *
 * Pins: every function here is checked by the `-m "not gpu"` tests against
 * brute force, closed forms, hand-worked fixtures, library routines (numpy,
 * torch) and the published OCP FP8 format definition.  No function is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32 (bf16 is the upper half of an IEEE binary32)          */
/* ------------------------------------------------------------------ */

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even of a binary32 to bfloat16: add half an ulp of the
 * kept part, plus one if the kept part is odd, then truncate.  NaN stays
 * NaN (quiet bit forced). */
static uint16_t float_to_bf16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint16_t oracle_bf16_from_float(float f) { return float_to_bf16_bits_rne(f); }
float oracle_float_from_bf16(uint16_t h) { return bf16_bits_to_float(h); }

/* ------------------------------------------------------------------ */
/* a1: top-k over router logits                                        */
/* [P3] ch.1 top2_gating (torch.topk over the expert axis); [P4] sec. 7 */
/* "Dispatch", step 1 (route: score every expert, keep the top-k).      */
/* Order: value descending; equal values (including -0 vs +0) go to the */
/* lower expert index.  Implemented as a full sort of all E experts by  */
/* the key (-logit, e) and keeping the first k.                         */
/* ------------------------------------------------------------------ */

typedef struct {
    float v;
    int32_t e;
} scored_expert;

static int by_value_desc_then_index(const void *pa, const void *pb)
{
    const scored_expert *a = (const scored_expert *)pa;
    const scored_expert *b = (const scored_expert *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->e < b->e) ? -1 : (a->e > b->e);
}

/* Returns 0, or -1 if a logit is not finite (the order is then undefined). */
int oracle_topk(const float *logits, int64_t T, int E, int k, int32_t *topk_idx)
{
    scored_expert *row = (scored_expert *)malloc(sizeof(scored_expert) * (size_t)E);
    if (!row) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float v = logits[t * E + e];
            if (!isfinite(v)) { free(row); return -1; }
            row[e].v = v;
            row[e].e = e;
        }
        qsort(row, (size_t)E, sizeof(scored_expert), by_value_desc_then_index);
        for (int j = 0; j < k; ++j) topk_idx[t * k + j] = row[j].e;
    }
    free(row);
    return 0;
}

/* ------------------------------------------------------------------ */
/* a2: gate weights, in fp64                                            */
/* mode 0 (TOPK_SOFTMAX): softmax over the k selected logits             */
/*   [P3] ch.1 top2_gating: gates = softmax(top-k logits).               */
/* mode 1 (SOFTMAX_TOPK): softmax over all E logits, keep the k selected */
/*   probabilities, no renormalisation (DeepSeekMoE fine-grained routing */
/*   as [P2] sec. 2.1 describes it; [P2] sec. 4.1 shows softmax over all */
/*   experts followed by top-k).                                         */
/* Both are shifted by the largest logit before exp (same value, no     */
/* overflow).                                                            */
/* ------------------------------------------------------------------ */

int oracle_gates(const float *logits, const int32_t *topk_idx, int64_t T, int E,
                 int k, int mode, double *gates)
{
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        const int32_t *ix = topk_idx + t * k;
        double m = (double)l[ix[0]];
        double denom = 0.0;
        if (mode == 0) {
            for (int i = 0; i < k; ++i) denom += exp((double)l[ix[i]] - m);
        } else if (mode == 1) {
            for (int e = 0; e < E; ++e) denom += exp((double)l[e] - m);
        } else {
            return -1;
        }
        for (int j = 0; j < k; ++j) gates[t * k + j] = exp((double)l[ix[j]] - m) / denom;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* a3: routing statistics                                               */
/* counts: number of (token, slot) assignments per expert, before any   */
/*   capacity limit ([P3] sec. 2.3, bincount of the routed indices).     */
/* aux:   E * sum_e f_e^2 with f_e = mean over tokens of the per-token   */
/*   one-hot expert mask = count_e / T ([P3] ch.1 top2_gating).          */
/* entropy: -sum_e p_e log2(p_e + 1e-8), p_e = count_e / sum(count)     */
/*   ([P3] sec. 2.3; [P1] sec. 5.1 TaxMeter, "ideal 4.0" for 16 experts). */
/* An empty batch (T == 0) has aux = entropy = 0 by convention.          */
/* ------------------------------------------------------------------ */

int oracle_stats(const int32_t *topk_idx, int64_t T, int E, int k,
                 int32_t *counts, double *aux, double *entropy)
{
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t a = 0; a < T * k; ++a) {
        int32_t e = topk_idx[a];
        if (e < 0 || e >= E) return -1;
        counts[e] += 1;
    }
    if (T == 0) {
        *aux = 0.0;
        *entropy = 0.0;
        return 0;
    }
    double sum_f2 = 0.0;
    for (int e = 0; e < E; ++e) {
        double f = (double)counts[e] / (double)T;
        sum_f2 += f * f;
    }
    *aux = sum_f2 * (double)E;

    double total = (double)T * (double)k;
    double h = 0.0;
    for (int e = 0; e < E; ++e) {
        double p = (double)counts[e] / total;
        h -= p * log2(p + 1e-8);
    }
    *entropy = h;
    return 0;
}

/* ------------------------------------------------------------------ */
/* a4: dispatch layout                                                   */
/* [P4] sec. 7 "Dispatch" detail: reorder tokens by target expert id and */
/* pack everything bound for one destination contiguously; sec. 7.5.2:   */
/* keep "indices" (target positions) and "locations" (source positions)  */
/* for the combine; sec. 7.5.4: pack only valid tokens, no padding;      */
/* sec. 8.3.A: strict per-expert token capacity, assignments over it are */
/* handled in order (dropped here).                                      */
/*                                                                       */
/* Assignment a = t*k + j.  All assignments are sorted by (expert, a):   */
/* a stable sort by expert, so within one expert the order is token      */
/* order.  rank(a) = position within its expert; kept iff rank < C      */
/* (capacity <= 0: no limit).  Packed rows: experts in order, kept       */
/* assignments of one expert in token order.                             */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t e;
    int64_t a;
} routed_assignment;

static int by_expert_then_assignment(const void *pa, const void *pb)
{
    const routed_assignment *x = (const routed_assignment *)pa;
    const routed_assignment *y = (const routed_assignment *)pb;
    if (x->e != y->e) return (x->e < y->e) ? -1 : 1;
    return (x->a < y->a) ? -1 : (x->a > y->a);
}

int oracle_layout(const int32_t *topk_idx, int64_t T, int E, int k, int P, int64_t capacity,
                  float *gates_or_null, int32_t *kept_counts, int32_t *offsets,
                  int32_t *dst_row, int32_t *src_pos, uint8_t *capacity_mask,
                  int32_t *part_rows, int32_t *part_offsets, int32_t *part_tokens,
                  int64_t *dropped)
{
    if (P <= 0 || E % P != 0) return -1;
    const int64_t A = T * k;
    routed_assignment *list = (routed_assignment *)malloc(sizeof(routed_assignment) * (size_t)(A > 0 ? A : 1));
    int64_t *raw_start = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    if (!list || !raw_start) { free(list); free(raw_start); return -2; }

    /* id -1 marks an empty slot (a row with fewer than k assignments, as in
     * the de-duplicated receive rows): no row, not counted, not an error */
    int64_t n = 0;
    for (int64_t a = 0; a < A; ++a) {
        int32_t e = topk_idx[a];
        if (e == -1) {
            dst_row[a] = -1;
            capacity_mask[a] = 0;
            continue;
        }
        if (e < 0 || e >= E) { free(list); free(raw_start); return -1; }
        list[n].e = e;
        list[n].a = a;
        ++n;
        raw_start[e + 1] += 1;
    }
    qsort(list, (size_t)n, sizeof(routed_assignment), by_expert_then_assignment);
    for (int e = 0; e < E; ++e) raw_start[e + 1] += raw_start[e];

    /* kept counts and packed-row offsets */
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t c = raw_start[e + 1] - raw_start[e];
        if (capacity > 0 && c > capacity) c = capacity;
        kept_counts[e] = (int32_t)c;
        offsets[e + 1] = offsets[e] + (int32_t)c;
    }
    const int32_t R = offsets[E];

    /* ranks, drops, the two index maps */
    for (int64_t s = 0; s < n; ++s) {
        int32_t e = list[s].e;
        int64_t a = list[s].a;
        int64_t rank = s - raw_start[e];
        int kept = (capacity <= 0) || (rank < capacity);
        if (kept) {
            int32_t row = offsets[e] + (int32_t)rank;
            dst_row[a] = row;
            src_pos[row] = (int32_t)a;
            capacity_mask[a] = 1;
        } else {
            dst_row[a] = -1;
            capacity_mask[a] = 0;
            if (gates_or_null) gates_or_null[a] = 0.0f;
        }
    }

    /* logical partitions: partition p holds experts [p*E/P, (p+1)*E/P) */
    const int per = E / P;
    for (int p = 0; p < P; ++p) {
        int32_t rows = 0;
        for (int e = p * per; e < (p + 1) * per; ++e) rows += kept_counts[e];
        part_rows[p] = rows;
        part_offsets[p] = offsets[p * per];
        part_tokens[p] = 0;
    }
    part_offsets[P] = R;
    for (int64_t t = 0; t < T; ++t) {
        for (int p = 0; p < P; ++p) {
            int hit = 0;
            for (int j = 0; j < k; ++j) {
                int64_t a = t * k + j;
                if (capacity_mask[a] && topk_idx[a] >= 0 && topk_idx[a] / per == p) hit = 1;
            }
            part_tokens[p] += hit;
        }
    }
    *dropped = A - (int64_t)R;
    free(list);
    free(raw_start);
    return 0;
}

/* Capacity overflow re-assigned instead of dropped ([P4] sec. 8.3.A:
 * greedy top-k selection under a hard per-expert capacity, then a rolling
 * fallback that sends the assignments an expert cannot take to the expert
 * with the lowest load in the batch).  Read as two passes:
 *   1. every expert keeps its first `capacity` assignments in token order
 *      (exactly as oracle_layout);
 *   2. the remaining ("overflow") assignments, in flat order a = t*k + j,
 *      each go to the expert with the lowest current load (ties: lower id)
 *      among experts below capacity, raising its load by one; with no such
 *      expert the assignment is dropped.
 * Rows: an expert's kept assignments in token order, then the ones it
 * received in pass 2 in the order received.  capacity_mask: 1 kept where
 * routed, 2 re-assigned, 0 dropped.  final_expert[a]: the expert that
 * processes assignment a (-1 if dropped).  A re-assigned slot keeps its gate
 * weight; only dropped slots get gate 0.  Partitions follow the final
 * experts. */
int oracle_layout_reassign(const int32_t *topk_idx, int64_t T, int E, int k, int P, int64_t capacity,
                           float *gates_or_null, int32_t *counts, int32_t *offsets, int32_t *dst_row,
                           int32_t *src_pos, uint8_t *capacity_mask, int32_t *final_expert,
                           int32_t *part_rows, int32_t *part_offsets, int32_t *part_tokens, int64_t *dropped)
{
    if (P <= 0 || E % P != 0 || capacity <= 0) return -1;
    const int64_t A = T * k;
    routed_assignment *list = (routed_assignment *)malloc(sizeof(routed_assignment) * (size_t)(A > 0 ? A : 1));
    int64_t *raw_start = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t *load = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *level = (int64_t *)malloc(sizeof(int64_t) * (size_t)(A > 0 ? A : 1));
    if (!list || !raw_start || !load || !level) { free(list); free(raw_start); free(load); free(level); return -2; }
    for (int64_t a = 0; a < A; ++a) {
        int32_t e = topk_idx[a];
        if (e < 0 || e >= E) { free(list); free(raw_start); free(load); free(level); return -1; }
        list[a].e = e;
        list[a].a = a;
        raw_start[e + 1] += 1;
    }
    qsort(list, (size_t)A, sizeof(routed_assignment), by_expert_then_assignment);
    for (int e = 0; e < E; ++e) raw_start[e + 1] += raw_start[e];

    /* pass 1: the first `capacity` assignments of each expert, in token order */
    for (int64_t a = 0; a < A; ++a) final_expert[a] = -1;
    for (int64_t s = 0; s < A; ++s) {
        int32_t e = list[s].e;
        int64_t rank = s - raw_start[e];
        if (rank < capacity) {
            final_expert[list[s].a] = e;
            level[list[s].a] = rank;
            capacity_mask[list[s].a] = 1;
            load[e] += 1;
        }
    }
    /* pass 2: overflow assignments in flat order to the least-loaded expert */
    for (int64_t a = 0; a < A; ++a) {
        if (final_expert[a] >= 0) continue;
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (load[e] < capacity && (best < 0 || load[e] < load[best])) best = e;
        if (best < 0) {
            capacity_mask[a] = 0;
            continue;
        }
        final_expert[a] = best;
        level[a] = load[best];
        load[best] += 1;
        capacity_mask[a] = 2;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        counts[e] = (int32_t)load[e];
        offsets[e + 1] = offsets[e] + counts[e];
    }
    const int32_t R = offsets[E];
    for (int64_t a = 0; a < A; ++a) {
        int32_t e = final_expert[a];
        if (e < 0) {
            dst_row[a] = -1;
            if (gates_or_null) gates_or_null[a] = 0.0f;
            continue;
        }
        int32_t row = offsets[e] + (int32_t)level[a];
        dst_row[a] = row;
        src_pos[row] = (int32_t)a;
    }
    const int per = E / P;
    for (int p = 0; p < P; ++p) {
        int32_t rows = 0;
        for (int e = p * per; e < (p + 1) * per; ++e) rows += counts[e];
        part_rows[p] = rows;
        part_offsets[p] = offsets[p * per];
        part_tokens[p] = 0;
    }
    part_offsets[P] = R;
    for (int64_t t = 0; t < T; ++t) {
        for (int p = 0; p < P; ++p) {
            int hit = 0;
            for (int j = 0; j < k; ++j) {
                int32_t e = final_expert[t * k + j];
                if (e >= 0 && e / per == p) hit = 1;
            }
            part_tokens[p] += hit;
        }
    }
    *dropped = A - (int64_t)R;
    free(list);
    free(raw_start);
    free(load);
    free(level);
    return 0;
}

/* Per-partition token de-duplication ([P4] sec. 7 dispatch detail: the
 * rows bound for one destination are packed together; a token that picks
 * several experts of one partition is sent there once, with the list of
 * its experts and gates, and the partition returns one row for it).
 * From a layout (dst_row, offsets: the final expert of every kept slot is
 * the expert whose rows contain dst_row) and the gates:
 *   send_offsets[P+1]  exclusive scan of the tokens sent to each partition
 *   send_row[t*P + p]  the send row of (t, p), or -1 if t keeps no slot in p
 *   send_token[s]      the token of send row s (rows: partition-major,
 *                      tokens ascending)
 *   slot_local[s*k+q], slot_gate[s*k+q]  the q-th kept slot (slot order)
 *                      of the token in that partition: local expert id
 *                      (expert - p*E/P) and gate; -1 / 0 past the last.
 * Returns the number of send rows, or -1 on bad input. */
int64_t oracle_dedup_layout(const int32_t *dst_row, const int32_t *offsets, const float *gates, int64_t T,
                            int E, int k, int P, int32_t *send_offsets, int32_t *send_row, int32_t *send_token,
                            int32_t *slot_local, float *slot_gate)
{
    if (P <= 0 || E % P != 0) return -1;
    const int per = E / P;
    const int32_t R = offsets[E];
    send_offsets[0] = 0;
    for (int p = 0; p < P; ++p) {
        int32_t cnt = 0;
        for (int64_t t = 0; t < T; ++t) {
            int hit = 0;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0 || r >= R) continue;
                int e = 0;
                while (offsets[e + 1] <= r) ++e;
                if (e / per == p) hit = 1;
            }
            cnt += hit;
        }
        send_offsets[p + 1] = send_offsets[p] + cnt;
    }
    for (int p = 0; p < P; ++p) {
        int32_t s = send_offsets[p];
        for (int64_t t = 0; t < T; ++t) {
            int q = 0;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0 || r >= R) continue;
                int e = 0;
                while (offsets[e + 1] <= r) ++e;
                if (e / per != p) continue;
                slot_local[(int64_t)s * k + q] = e - p * per;
                slot_gate[(int64_t)s * k + q] = gates[t * k + j];
                ++q;
            }
            if (q == 0) {
                send_row[t * P + p] = -1;
                continue;
            }
            for (int qq = q; qq < k; ++qq) {
                slot_local[(int64_t)s * k + qq] = -1;
                slot_gate[(int64_t)s * k + qq] = 0.0f;
            }
            send_row[t * P + p] = s;
            send_token[s] = (int32_t)t;
            ++s;
        }
    }
    return send_offsets[P];
}

/* ------------------------------------------------------------------ */
/* a5: dispatch (bf16 transport): packed row r is a bit copy of the     */
/* hidden state of token src_pos[r] / k ([P4] sec. 7 Dispatch detail,   */
/* "reorder and pack").  Evaluated for an explicit list of packed rows. */
/* ------------------------------------------------------------------ */

void oracle_dispatch_bf16_rows(const uint16_t *x, int64_t H, int k, const int32_t *src_pos,
                               const int64_t *rows, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = (int64_t)src_pos[rows[i]] / k;
        memcpy(out + i * H, x + t * H, sizeof(uint16_t) * (size_t)H);
    }
}

/* ------------------------------------------------------------------ */
/* a6: per-token affine FP8 (e4m3) transport                            */
/* [P1] sec. 3.1: per token, take the min and max of its vector and map */
/* it affinely onto FP8.  The constants: zero = (max + min) / 2,         */
/* scale = (max - min) / 896 (so [min, max] maps onto [-448, 448], the  */
/* e4m3 finite range), code = e4m3(round-to-nearest-even((x - zero) /   */
/* scale)) with saturation to +-448.  A constant row (max == min) has   */
/* scale 0 and all-zero codes.                                           */
/* ------------------------------------------------------------------ */

/* e4m3 ("E4M3FN" of the OCP 8-bit floating point specification): sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
 * subnormals m * 2^-9; the largest finite value is 1.75 * 2^8 = 448; there
 * is no infinity.  Conversion: round to nearest, ties to even mantissa;
 * magnitudes above 448 (and infinities) saturate to 448; the sign is kept,
 * so -0 and negative values that round to zero encode as 0x80.  NaN maps to
 * 0x7F (sign kept: 0xFF). */
uint8_t oracle_e4m3_satfinite(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return (uint8_t)(sign | 0x7Fu); /* NaN */
    float a = fabsf(v);
    if (a > 448.0f) return (uint8_t)(sign | 0x7Eu); /* satfinite */
    if (a < 0.015625f) {
        /* below the smallest normal 2^-6: multiples of 2^-9.  a * 512 is
         * exact in double; rint rounds half to even (default mode). */
        double q = rint((double)a * 512.0);
        return (uint8_t)(sign | (uint8_t)q); /* q == 8 is 2^-6, code 0x08 */
    }
    int exp2 = (int)((mag >> 23) & 0xFFu) - 127; /* -6 .. 8 */
    uint32_t m23 = mag & 0x7FFFFFu;
    uint32_t m3 = m23 >> 20;
    uint32_t rest = m23 & 0xFFFFFu;
    if (rest > 0x80000u || (rest == 0x80000u && (m3 & 1u))) {
        m3 += 1u;
        if (m3 == 8u) { m3 = 0u; exp2 += 1; }
    }
    return (uint8_t)(sign | (uint8_t)(((exp2 + 7) << 3) | (int)m3));
}

/* Decode of an e4m3 code (for dequantisation checks). */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int ex = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (ex == 0xF && m == 7) return NAN;
    if (ex == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, ex - 7);
    return s ? -v : v;
}

/* Total order used for the row extremes: numeric order, with -0 below +0,
 * so the max and min of a row do not depend on the scan order. */
static int total_less(float a, float b)
{
    if (a < b) return 1;
    if (a > b) return 0;
    return signbit(a) && !signbit(b);
}

void oracle_fp8_token_params(const uint16_t *xrow, int64_t H, float *scale, float *zero)
{
    float mx = bf16_bits_to_float(xrow[0]);
    float mn = mx;
    for (int64_t h = 1; h < H; ++h) {
        float v = bf16_bits_to_float(xrow[h]);
        if (total_less(mx, v)) mx = v;
        if (total_less(v, mn)) mn = v;
    }
    float z = (mx + mn) * 0.5f;
    float s = (mx == mn) ? 0.0f : (mx - mn) / 896.0f;
    *zero = z;
    *scale = s;
}

void oracle_quantize_row_fp8(const uint16_t *xrow, int64_t H, uint8_t *codes,
                             float *scale_out, float *zero_out)
{
    float scale, zero;
    oracle_fp8_token_params(xrow, H, &scale, &zero);
    for (int64_t h = 0; h < H; ++h) {
        if (scale == 0.0f) {
            codes[h] = 0x00u;
        } else {
            float d = bf16_bits_to_float(xrow[h]) - zero;
            float q = d / scale;
            codes[h] = oracle_e4m3_satfinite(q);
        }
    }
    *scale_out = scale;
    *zero_out = zero;
}

/* Packed FP8 rows for an explicit list of rows: codes [n, H] and
 * scales [n, 2] = (scale, zero) of the row's token. */
void oracle_dispatch_fp8_rows(const uint16_t *x, int64_t H, int k, const int32_t *src_pos,
                              const int64_t *rows, int64_t n, uint8_t *codes, float *scales)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = (int64_t)src_pos[rows[i]] / k;
        oracle_quantize_row_fp8(x + t * H, H, codes + i * H, &scales[2 * i], &scales[2 * i + 1]);
    }
}

/* Grouped variants of the same affine map ([P1] sec. 5.2: the FP8
 * quantiser offers per-token, per-expert and global modes).  One (scale,
 * zero) pair per group, from the max and min over every element of the
 * group's rows, with the per-token formula above; each row is encoded with
 * its group's pair.  Per-token: a row is its own group; per-expert: the
 * rows sent to one expert; global: every transported row.
 *
 * Rows are given as src [*, H] bf16 with row i = src row src_row[i] in
 * group group[i] (0 <= group < ngroups). */

/* params [ngroups, 2] = (scale, zero) per group; a group without rows gets
 * (0, 0).  Returns 0, or -1 on a bad group id / allocation failure. */
int oracle_fp8_group_params(const uint16_t *src, int64_t H, const int64_t *src_row,
                            const int32_t *group, int64_t n, int64_t ngroups, float *params)
{
    float *gmx = (float *)malloc(sizeof(float) * (size_t)(ngroups > 0 ? ngroups : 1));
    float *gmn = (float *)malloc(sizeof(float) * (size_t)(ngroups > 0 ? ngroups : 1));
    unsigned char *seen = (unsigned char *)calloc((size_t)(ngroups > 0 ? ngroups : 1), 1);
    int rc = 0;
    if (!gmx || !gmn || !seen) { rc = -1; goto done; }
    for (int64_t i = 0; i < n; ++i) {
        if (group[i] < 0 || group[i] >= ngroups) { rc = -1; goto done; }
        const uint16_t *row = src + src_row[i] * H;
        int32_t g = group[i];
        for (int64_t h = 0; h < H; ++h) {
            float v = bf16_bits_to_float(row[h]);
            if (!seen[g]) { gmx[g] = v; gmn[g] = v; seen[g] = 1; continue; }
            if (total_less(gmx[g], v)) gmx[g] = v;
            if (total_less(v, gmn[g])) gmn[g] = v;
        }
    }
    for (int64_t g = 0; g < ngroups; ++g) {
        if (!seen[g]) { params[2 * g] = 0.0f; params[2 * g + 1] = 0.0f; continue; }
        params[2 * g] = (gmx[g] == gmn[g]) ? 0.0f : (gmx[g] - gmn[g]) / 896.0f;
        params[2 * g + 1] = (gmx[g] + gmn[g]) * 0.5f;
    }
done:
    free(gmx);
    free(gmn);
    free(seen);
    return rc;
}

/* codes [n, H] and scales [n, 2] of the listed rows, encoded with their
 * group's (scale, zero) from params. */
void oracle_quantize_rows_with_params(const uint16_t *src, int64_t H, const int64_t *src_row,
                                      const int32_t *group, int64_t n, const float *params,
                                      uint8_t *codes, float *scales)
{
    for (int64_t i = 0; i < n; ++i) {
        float scale = params[2 * (int64_t)group[i]];
        float zero = params[2 * (int64_t)group[i] + 1];
        const uint16_t *row = src + src_row[i] * H;
        for (int64_t h = 0; h < H; ++h) {
            if (scale == 0.0f) {
                codes[i * H + h] = 0x00u;
            } else {
                float q = (bf16_bits_to_float(row[h]) - zero) / scale;
                codes[i * H + h] = oracle_e4m3_satfinite(q);
            }
        }
        scales[2 * i] = scale;
        scales[2 * i + 1] = zero;
    }
}

/* ------------------------------------------------------------------ */
/* a7: combine                                                          */
/* [P4] sec. 7 "Combine": per token, the weighted sum of its top-k      */
/* expert outputs, put back in original token order using the routing  */
/* metadata saved at dispatch; [P4] sec. 8.2.B: shared experts are seen */
/* by every token, bypass the all-to-all, and their outputs are added.  */
/*                                                                       */
/* y[t] = sum over kept slots j (ascending) of g[t,j] * eo[dst_row[t,j]] */
/*        + sum over shared experts s (ascending) of shared[s, t]         */
/* Dropped slots (dst_row == -1) contribute nothing.                     */
/* ------------------------------------------------------------------ */

/* Pinned fp32 order: acc = 0; acc = fmaf(g, eo, acc) over kept slots in
 * ascending j; acc = acc + shared over s ascending; y = bf16 RNE(acc). */
void oracle_combine_f32order_tokens(const uint16_t *eo, int64_t H, int k, const float *gates,
                                    const int32_t *dst_row, const uint16_t *shared, int Ks,
                                    int64_t T, const int64_t *tokens, int64_t n, uint16_t *y)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0) continue;
                acc = fmaf(gates[t * k + j], bf16_bits_to_float(eo[(int64_t)r * H + h]), acc);
            }
            for (int s = 0; s < Ks; ++s)
                acc = acc + bf16_bits_to_float(shared[((int64_t)s * T + t) * H + h]);
            y[i * H + h] = float_to_bf16_bits_rne(acc);
        }
    }
}

/* fp64 reference of the same sum, plus sum |term| (for the error bound). */
void oracle_combine_ref64_tokens(const uint16_t *eo, int64_t H, int k, const float *gates,
                                 const int32_t *dst_row, const uint16_t *shared, int Ks,
                                 int64_t T, const int64_t *tokens, int64_t n,
                                 double *ref, double *abs_terms)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0, mag = 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0) continue;
                double term = (double)gates[t * k + j] * (double)bf16_bits_to_float(eo[(int64_t)r * H + h]);
                acc += term;
                mag += fabs(term);
            }
            for (int s = 0; s < Ks; ++s) {
                double term = (double)bf16_bits_to_float(shared[((int64_t)s * T + t) * H + h]);
                acc += term;
                mag += fabs(term);
            }
            ref[i * H + h] = acc;
            abs_terms[i * H + h] = mag;
        }
    }
}

/* Combine of FP8 expert outputs ([P1] sec. 3.1: the per-token affine
 * FP8 map is applied to each token's expert output vector, i.e. on the
 * combine side of the exchange too).  Each packed row r carries codes and
 * (scale, zero); its value is dequantised in fp32 with one rounding,
 *   v = fmaf(scale, e4m3_value(code), zero),
 * and then combined in the pinned order of the bf16 combine:
 *   acc = 0; acc = fmaf(g, v, acc) over kept slots ascending;
 *   acc = acc + shared (bf16) over s ascending; y = bf16 RNE(acc).
 * (e4m3 values are exact in fp32.) */
void oracle_combine_fp8_f32order_tokens(const uint8_t *codes, const float *scales, int64_t H, int k,
                                        const float *gates, const int32_t *dst_row,
                                        const uint16_t *shared, int Ks, int64_t T,
                                        const int64_t *tokens, int64_t n, uint16_t *y)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0) continue;
                float val = (float)oracle_e4m3_decode(codes[(int64_t)r * H + h]);
                float v = fmaf(scales[2 * (int64_t)r], val, scales[2 * (int64_t)r + 1]);
                acc = fmaf(gates[t * k + j], v, acc);
            }
            for (int s = 0; s < Ks; ++s)
                acc = acc + bf16_bits_to_float(shared[((int64_t)s * T + t) * H + h]);
            y[i * H + h] = float_to_bf16_bits_rne(acc);
        }
    }
}

/* fp64 reference of the FP8 combine: sum g * (zero + scale * value) (+
 * shared), and sum |term|. */
void oracle_combine_fp8_ref64_tokens(const uint8_t *codes, const float *scales, int64_t H, int k,
                                     const float *gates, const int32_t *dst_row,
                                     const uint16_t *shared, int Ks, int64_t T,
                                     const int64_t *tokens, int64_t n, double *ref, double *abs_terms)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0, mag = 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0) continue;
                double v = (double)scales[2 * (int64_t)r + 1] +
                           (double)scales[2 * (int64_t)r] * oracle_e4m3_decode(codes[(int64_t)r * H + h]);
                double term = (double)gates[t * k + j] * v;
                acc += term;
                mag += fabs(term);
            }
            for (int s = 0; s < Ks; ++s) {
                double term = (double)bf16_bits_to_float(shared[((int64_t)s * T + t) * H + h]);
                acc += term;
                mag += fabs(term);
            }
            ref[i * H + h] = acc;
            abs_terms[i * H + h] = mag;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Backward of the path: the gradient retraces the forward routing     */
/* with the saved indices ([P1] sec. 2.4: the backward all-to-all      */
/* mirrors the forward one using cached routing indices; [P4] sec. 7,  */
/* detail item 3: the combine stage is also the backward gradient     */
/* dispatch).                                                          */
/* ------------------------------------------------------------------ */

/* Combine backward, for the listed tokens:
 *   d_eo[dst_row[t,j]] = bf16 RNE(fp32(g[t,j] * dy[t]))  for kept j
 *   d_gates[t,j]       = sum_h dy[t,h] * eo[dst_row[t,j],h]  (fp64), 0 if dropped
 * d_eo rows are written to d_eo_rows[i*k + j] (row-major [n*k, H]); rows of
 * dropped slots are left as they are. */
void oracle_combine_backward_tokens(const uint16_t *dy, const uint16_t *eo, int64_t H, int k,
                                    const float *gates, const int32_t *dst_row,
                                    const int64_t *tokens, int64_t n, uint16_t *d_eo_rows,
                                    double *d_gates)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        for (int j = 0; j < k; ++j) {
            int32_t r = dst_row[t * k + j];
            double dot = 0.0;
            if (r >= 0) {
                float g = gates[t * k + j];
                for (int64_t h = 0; h < H; ++h) {
                    float d = bf16_bits_to_float(dy[t * H + h]);
                    float prod = g * d; /* one fp32 rounding */
                    d_eo_rows[(i * k + j) * H + h] = float_to_bf16_bits_rne(prod);
                    dot += (double)d * (double)bf16_bits_to_float(eo[(int64_t)r * H + h]);
                }
            }
            d_gates[i * k + j] = dot;
        }
    }
}

/* Dispatch backward (bf16 gradients), for the listed tokens, pinned fp32
 * order: acc = 0; acc = acc + d_packed[dst_row[t,j]] over kept j ascending;
 * dx[t] = bf16 RNE(acc).  Also the fp64 sum. */
void oracle_dispatch_backward_tokens(const uint16_t *d_packed, int64_t H, int k,
                                     const int32_t *dst_row, const int64_t *tokens, int64_t n,
                                     uint16_t *dx, double *dx64)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            double acc64 = 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t r = dst_row[t * k + j];
                if (r < 0) continue;
                float v = bf16_bits_to_float(d_packed[(int64_t)r * H + h]);
                acc = acc + v;
                acc64 += (double)v;
            }
            dx[i * H + h] = float_to_bf16_bits_rne(acc);
            dx64[i * H + h] = acc64;
        }
    }
}

/* Gate backward in fp64: gradient of L = sum_j d_gates[t,j] * g[t,j] with
 * respect to the logits, the gates g recomputed from logits and topk_idx as
 * oracle_gates does.
 *   TOPK_SOFTMAX: g = softmax(l_sel):  dl_sel[j] = g_j (dg_j - sum_i g_i dg_i),
 *                 other experts 0.
 *   SOFTMAX_TOPK: g_j = p[sel_j], p = softmax(l):  dl_e = p_e (dp_e - sum_j g_j dg_j)
 *                 with dp_e = dg_j at e = sel_j, else 0.
 * (The aux loss depends on the indices only and has no gradient.) */
int oracle_gate_backward(const float *logits, const int32_t *topk_idx, const double *d_gates,
                         int64_t T, int E, int k, int mode, double *d_logits)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)k);
    if (!g) return -2;
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        const int32_t *ix = topk_idx + t * k;
        const double *dg = d_gates + t * k;
        double *dl = d_logits + t * E;
        if (oracle_gates(l, ix, 1, E, k, mode, g) != 0) { free(g); return -1; }
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += g[j] * dg[j];
        for (int e = 0; e < E; ++e) dl[e] = 0.0;
        if (mode == 0) {
            for (int j = 0; j < k; ++j) dl[ix[j]] = g[j] * (dg[j] - s);
        } else {
            double m = (double)l[ix[0]];
            double denom = 0.0;
            for (int e = 0; e < E; ++e) denom += exp((double)l[e] - m);
            for (int e = 0; e < E; ++e) dl[e] = -exp((double)l[e] - m) / denom * s;
            for (int j = 0; j < k; ++j) dl[ix[j]] += g[j] * dg[j];
        }
    }
    free(g);
    return 0;
}
