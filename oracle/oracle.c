/*
 * Oracle: a plain, slow, single-threaded CPU statement of what the MoE token
 * permute / unpermute path computes.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the library
 * never does.  It shares no code, header or constant with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [d9d]   "d9d 0.1.0 -- d9d/kernel/moe/permute_with_probs.py" (a copy of
 *           TransformerEngine permutation.py): make_row_id_map and its worked
 *           example, _permute_kernel, _unpermute_kernel,
 *           _unpermute_bwd_with_merging_probs_kernel, and the autograd
 *           backward of _moe_permute_mask_map / _moe_unpermute_mask_map.
 *   [MBI]   "core.transformer.moe.batch_invariant" (Megatron-Core API docs):
 *           _rank_tree_unpermute_kernel (FP32 FMA of prob and row in slot
 *           order, from zero, quantized once to BF16), _unpermute_loop (the
 *           slot loop as the reference form), _rank_tree_unpermute_bwd_kernel.
 *   [xt]    "permute different with torch version" (xtuner issue 1323): the
 *           forward map (k,i) -> row vs. the argsort inverse.
 *   [mops]  "moe-ops 0.1.0" README, sections "Layout conventions" and
 *           "Operators": counting sort, offsets[E+1].
 *   [TE-PR] "[PyTorch] Fuse MoE chunk sorting and padding" (TransformerEngine
 *           PR 3509), sections Description, Changes and Diagram.
 *
 * Conventions fixed here (the pages leave them open; the readings are listed
 * in the design notes):
 *   - row order: expert, then token, then slot (sort key (e, t, k));
 *   - idx[t,k] == -1 is an empty slot: no row, row_id_map[t,k] = -1;
 *     any other value outside [0,E) is counted as bad and treated as empty;
 *   - probs are [T,K] fp32, aligned with idx;
 *   - bf16 values are carried as their 16-bit patterns (uint16_t).
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (-ffp-contract=off so that only the explicit fmaf() calls fuse.)
 *
 * Parity pins for every function live in the CPU test-suite; nothing here is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 keeps the top 16 bits of an IEEE-754 binary32 value, so widening is
 * exact: place the 16 bits in the high half. */
float orc_f32_from_bf16(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Narrowing with IEEE round-to-nearest, ties to even, taken on the 16
 * discarded bits.  A carry out of the mantissa bumps the exponent, which is
 * the correct result (and gives +-inf past the largest finite bf16).
 * NaN stays NaN (sign kept, quiet bit set); the workloads never make one.
 * "quantized to BF16" [MBI, _rank_tree_unpermute_kernel]. */
uint16_t orc_bf16_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u) != 0u))
        hi += 1u;
    return (uint16_t)hi;
}

/* ------------------------------------------------------------------------ */
/* Routing map                                                               */
/* ------------------------------------------------------------------------ */

static int orc_expert_of(const int32_t *idx, int64_t i, int32_t E)
{
    int32_t e = idx[i];
    return (e >= 0 && e < E) ? e : -1;
}

/*
 * Counting sort of the T*K routes by expert, stable in the flat (t,k) order.
 *   counts[e]        = #{(t,k) : idx[t,k] == e}                 (histogram)
 *   offsets[0] = 0,  offsets[e+1] = offsets[e] + counts[e]      (exclusive scan;
 *                    offsets[E] = number of routed slots)  [mops, Layout conventions]
 *   row_id_map[t,k]  = offsets[e] + #{(t',k') before (t,k) in flat order with
 *                      the same expert}, or -1 for an empty slot.
 * Rows therefore run expert-major, tokens ascending inside each expert, and
 * slots ascending for a token that names one expert twice.  This is the order
 * of the worked example after "pass 2" in [d9d, make_row_id_map], and the
 * forward map "row_id_map[k][i]" of [xt] stored [T,K] instead of [K,T].
 *   sorted_to_flat[row] = t*K + k for routed rows (the argsort inverse of
 *   [xt]); entries from offsets[E] up to T*K are -1.  May be NULL.
 * Returns the number of idx entries outside [-1, E).
 */
int64_t orc_build_map(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                      int32_t *row_id_map, int32_t *sorted_to_flat,
                      int32_t *counts, int32_t *offsets)
{
    const int64_t n = T * (int64_t)K;
    int64_t bad = 0;
    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        int e = orc_expert_of(idx, i, E);
        if (e >= 0)
            counts[e] += 1;
        else if (idx[i] != -1)
            bad += 1;
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];

    for (int64_t i = 0; i < n; ++i)
        row_id_map[i] = -1;
    if (sorted_to_flat)
        for (int64_t i = 0; i < n; ++i)
            sorted_to_flat[i] = -1;

    /* Plainest form of the stable counting sort: visit experts in order and,
     * for each, every (t,k) in flat order. */
    int32_t next = 0;
    for (int32_t e = 0; e < E; ++e) {
        for (int64_t t = 0; t < T; ++t) {
            for (int32_t k = 0; k < K; ++k) {
                int64_t i = t * K + k;
                if (orc_expert_of(idx, i, E) == e) {
                    row_id_map[i] = next;
                    if (sorted_to_flat)
                        sorted_to_flat[next] = (int32_t)i;
                    next += 1;
                }
            }
        }
    }
    return bad;
}

/*
 * Counting sort with an expert capacity: expert e keeps at most `capacity`
 * routes, the first ones in flat (t,k) order; the others are dropped like
 * empty slots (row_id_map = -1).  counts[e] is the number kept, offsets its
 * exclusive scan, so offsets[E] is the number of rows the permuted tensor
 * holds -- the "effective output token count, ... tokens not dropped" of
 * num_out_tokens [d9d, moe_permute_with_probs].  capacity < 0: no limit.
 * sorted_to_flat: t*K+k for kept rows, -1 from offsets[E] on.
 * Returns the number of idx entries outside [-1, E).
 */
int64_t orc_build_map_capacity(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                               int32_t capacity, int32_t *row_id_map,
                               int32_t *sorted_to_flat, int32_t *counts, int32_t *offsets)
{
    const int64_t n = T * (int64_t)K;
    int64_t bad = 0;
    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        int e = orc_expert_of(idx, i, E);
        if (e >= 0) {
            if (capacity < 0 || counts[e] < capacity)
                counts[e] += 1;
        } else if (idx[i] != -1) {
            bad += 1;
        }
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    for (int64_t i = 0; i < n; ++i)
        row_id_map[i] = -1;
    if (sorted_to_flat)
        for (int64_t i = 0; i < n; ++i)
            sorted_to_flat[i] = -1;
    for (int32_t e = 0; e < E; ++e) {
        int32_t taken = 0;
        for (int64_t t = 0; t < T; ++t) {
            for (int32_t k = 0; k < K; ++k) {
                int64_t i = t * K + k;
                if (orc_expert_of(idx, i, E) != e)
                    continue;
                if (capacity < 0 || taken < capacity) {
                    int32_t row = offsets[e] + taken;
                    row_id_map[i] = row;
                    if (sorted_to_flat)
                        sorted_to_flat[row] = (int32_t)i;
                }
                taken += 1;
            }
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Permute / unpermute                                                       */
/* ------------------------------------------------------------------------ */

/* out[row_id_map[t,k], :] = x[t, :]; out_probs[row_id_map[t,k]] = probs[t,k].
 * The row is copied whatever its probability ([d9d, _permute_kernel] writes a
 * zero row for prob == 0 as a mask-padding device; with [T,K] index routing
 * there is no such padding).  probs / out_probs may be NULL together. */
void orc_permute(const uint16_t *x, const float *probs, const int32_t *row_id_map,
                 int64_t T, int32_t K, int32_t H, uint16_t *out, float *out_probs)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t k = 0; k < K; ++k) {
            int32_t row = row_id_map[t * K + k];
            if (row < 0)
                continue;
            for (int32_t h = 0; h < H; ++h)
                out[(int64_t)row * H + h] = x[t * H + h];
            if (probs && out_probs)
                out_probs[row] = probs[t * K + k];
        }
    }
}

/* Batch-invariant combine [MBI, _rank_tree_unpermute_kernel and
 * _unpermute_loop]: each token owns its sum.  Per element h:
 *   acc = +0.0f;  for k = 0..K-1 in slot order, skipping empty slots:
 *       acc = fmaf(probs[t,k], float(rows[row_id_map[t,k], h]), acc)
 *   out[t,h] = bf16_rne(acc)
 * With probs == NULL the tokens are "directly merged by accumulation"
 * [d9d, moe_unpermute_mask]: acc = acc + float(row), which equals
 * fmaf(1, row, acc). */
void orc_unpermute(const uint16_t *rows, const float *probs, const int32_t *row_id_map,
                   int64_t T, int32_t K, int32_t H, uint16_t *out)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                int32_t row = row_id_map[t * K + k];
                if (row < 0)
                    continue;
                float r = orc_f32_from_bf16(rows[(int64_t)row * H + h]);
                if (probs)
                    acc = fmaf(probs[t * K + k], r, acc);
                else
                    acc = acc + r;
            }
            out[t * H + h] = orc_bf16_from_f32(acc);
        }
    }
}

/* fp64 -> bf16, round to nearest even, in one rounding (no detour through
 * fp32): scale by the bf16 quantum at the value's binade (2^(e-7) for normal
 * bf16, 2^-133 below 2^-126), round to an integer with rint() (ties to even in
 * the default rounding mode), scale back -- all exact in double -- then read
 * the result's bits through float, where it is exactly representable.
 * Magnitudes that round past the largest finite bf16 become +-inf. */
uint16_t orc_bf16_from_f64(double d)
{
    if (isnan(d))
        return 0x7fc0u;
    if (isinf(d) || d == 0.0) {
        float f = (float)d;
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    double a = fabs(d);
    int e2;
    frexp(a, &e2);               /* a = m * 2^e2, m in [0.5, 1): binade exponent e2-1 */
    int binade = e2 - 1;
    if (binade < -126)
        binade = -126;           /* bf16 subnormals share the quantum 2^-133 */
    double q = ldexp(1.0, binade - 7);
    double r = rint(a / q) * q;
    const double max_bf16 = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
    uint16_t sign = d < 0 ? 0x8000u : 0;
    if (r > max_bf16)
        return (uint16_t)(sign | 0x7f80u);
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7fffu));
}

/* The rank-ordered combine of a token over EP ranks [MBI,
 * _rank_tree_unpermute_kernel, unpermute_with_bf16_rank_partials, unpermute]:
 * experts are split into ep_size ranks of E/ep_size consecutive experts.  Per
 * element, for each rank r in order, the rank's partial is the slot-order
 * chain of FP32 fused multiply-adds of prob and row over the token's routed
 * slots whose expert lies on r, from +0 (plain adds without probs); with
 * bf16_partials it is then quantized to BF16.  The partials are added in rank
 * order from zero, in fp32, or in fp64 when fp64_cross_rank is set, and the
 * sum is rounded once to BF16.  With ep_size = 1 and neither flag this is
 * orc_unpermute.  idx[T,K] holds each slot's expert. */
void orc_unpermute_ep(const uint16_t *rows, const float *probs, const int32_t *row_id_map,
                      const int32_t *idx, int64_t T, int32_t K, int32_t H, int32_t E,
                      int32_t ep_size, int32_t bf16_partials, int32_t fp64_cross_rank,
                      uint16_t *out)
{
    const int32_t per_rank = E / ep_size;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            float acc32 = 0.0f;
            double acc64 = 0.0;
            for (int32_t r = 0; r < ep_size; ++r) {
                float partial = 0.0f;
                for (int32_t k = 0; k < K; ++k) {
                    int32_t row = row_id_map[t * K + k];
                    if (row < 0 || idx[t * K + k] / per_rank != r)
                        continue;
                    float x = orc_f32_from_bf16(rows[(int64_t)row * H + h]);
                    if (probs)
                        partial = fmaf(probs[t * K + k], x, partial);
                    else
                        partial = partial + x;
                }
                if (bf16_partials)
                    partial = orc_f32_from_bf16(orc_bf16_from_f32(partial));
                if (fp64_cross_rank)
                    acc64 = acc64 + (double)partial;
                else
                    acc32 = acc32 + partial;
            }
            out[t * H + h] = fp64_cross_rank ? orc_bf16_from_f64(acc64) : orc_bf16_from_f32(acc32);
        }
    }
}

/* Backward of permute [d9d, _moe_permute_mask_map.backward]: the permuted
 * gradient is unpermuted without merging probs (a sum over the token's rows,
 * fp32 from +0 in slot order, one bf16 rounding), and the permuted-probs
 * gradient is gathered back to [T,K], 0 for empty slots. */
void orc_permute_bwd(const uint16_t *g_out, const float *g_out_probs,
                     const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                     uint16_t *g_x, float *g_probs)
{
    orc_unpermute(g_out, NULL, row_id_map, T, K, H, g_x);
    if (g_out_probs && g_probs) {
        for (int64_t t = 0; t < T; ++t)
            for (int32_t k = 0; k < K; ++k) {
                int32_t row = row_id_map[t * K + k];
                g_probs[t * K + k] = row >= 0 ? g_out_probs[row] : 0.0f;
            }
    }
}

/* Backward of unpermute.
 * With probs [d9d, _unpermute_bwd_with_merging_probs_kernel]:
 *   g_rows[row, h] = bf16_rne(probs[t,k] * float(g_y[t,h]))    (one fp32 product)
 *   g_probs[t,k]   = sum_h float(rows[row,h]) * float(g_y[t,h])
 * The oracle sums g_probs in fp64 (each bf16*bf16 product is exact there) so
 * that the GPU's fp32 reduction can be held to a stated error bound; empty
 * slots get 0.
 * Without probs [MBI, _rank_tree_unpermute_bwd_kernel]: the token's gradient
 * is scattered unchanged to each of its rows; g_probs is not touched. */
void orc_unpermute_bwd(const uint16_t *g_y, const uint16_t *rows, const float *probs,
                       const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                       uint16_t *g_rows, double *g_probs)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t k = 0; k < K; ++k) {
            int32_t row = row_id_map[t * K + k];
            if (row < 0) {
                if (probs && g_probs)
                    g_probs[t * K + k] = 0.0;
                continue;
            }
            if (!probs) {
                for (int32_t h = 0; h < H; ++h)
                    g_rows[(int64_t)row * H + h] = g_y[t * H + h];
                continue;
            }
            float p = probs[t * K + k];
            double dot = 0.0;
            for (int32_t h = 0; h < H; ++h) {
                float g = orc_f32_from_bf16(g_y[t * H + h]);
                float prod = p * g;
                g_rows[(int64_t)row * H + h] = orc_bf16_from_f32(prod);
                double r = (double)orc_f32_from_bf16(rows[(int64_t)row * H + h]);
                dot += r * (double)g;
            }
            if (g_probs)
                g_probs[t * K + k] = dot;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Router: fused top-k softmax  [mops "Operators: fused_topk_softmax"]       */
/* ------------------------------------------------------------------------ */

/*
 * Per token: optionally keep only the topk_groups best of n_groups equal
 * groups of consecutive experts (a group's score is its largest logit; equal
 * scores favour the lower group), then pick the K largest logits among the
 * kept experts one at a time (equal logits favour the lower expert), so slot
 * 0 holds the largest.  probs are the fp32 softmax over the K picked logits:
 * z_k = l_k - l_0, e_k = expf(z_k), s = e_0 + ... + e_{K-1} in slot order,
 * p_k = e_k / s.  n_groups = topk_groups = 1 is plain top-K.
 */
void orc_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t K,
                      int32_t n_groups, int32_t topk_groups, int32_t *idx, float *probs)
{
    const int32_t per_group = E / n_groups;
    char *kept = (char *)malloc((size_t)E);
    char *taken = (char *)malloc((size_t)E);
    char *gtaken = (char *)malloc((size_t)n_groups);
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        for (int32_t g = 0; g < n_groups; ++g)
            gtaken[g] = 0;
        for (int32_t e = 0; e < E; ++e)
            kept[e] = (n_groups == 1);
        if (n_groups > 1) {
            for (int32_t j = 0; j < topk_groups; ++j) {
                int32_t best = -1;
                float best_score = 0.0f;
                for (int32_t g = 0; g < n_groups; ++g) {
                    if (gtaken[g])
                        continue;
                    float score = l[g * per_group];
                    for (int32_t e = g * per_group + 1; e < (g + 1) * per_group; ++e)
                        if (l[e] > score)
                            score = l[e];
                    if (best < 0 || score > best_score) {
                        best = g;
                        best_score = score;
                    }
                }
                gtaken[best] = 1;
                for (int32_t e = best * per_group; e < (best + 1) * per_group; ++e)
                    kept[e] = 1;
            }
        }
        for (int32_t e = 0; e < E; ++e)
            taken[e] = 0;
        for (int32_t k = 0; k < K; ++k) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (kept[e] && !taken[e] && (best < 0 || l[e] > l[best]))
                    best = e;
            taken[best] = 1;
            idx[t * K + k] = best;
        }
        float s = 0.0f;
        const float m = l[idx[t * K]];
        for (int32_t k = 0; k < K; ++k) {
            float z = l[idx[t * K + k]] - m;
            probs[t * K + k] = expf(z);
            s = s + probs[t * K + k];
        }
        for (int32_t k = 0; k < K; ++k)
            probs[t * K + k] = probs[t * K + k] / s;
    }
    free(kept);
    free(taken);
    free(gtaken);
}

/* Gradient of the router w.r.t. the logits: the picked logits get the softmax
 * gradient g_l_k = p_k * (g_k - d) with d = sum_j p_j * g_j (fused
 * multiply-adds in slot order from +0); every other logit gets 0 (the choice
 * itself is piecewise constant). */
void orc_topk_softmax_bwd(const float *g_probs, const float *probs, const int32_t *idx,
                          int64_t T, int32_t E, int32_t K, float *g_logits)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e)
            g_logits[t * E + e] = 0.0f;
        float d = 0.0f;
        for (int32_t k = 0; k < K; ++k)
            d = fmaf(probs[t * K + k], g_probs[t * K + k], d);
        for (int32_t k = 0; k < K; ++k)
            g_logits[t * E + idx[t * K + k]] = probs[t * K + k] * (g_probs[t * K + k] - d);
    }
}

/* ------------------------------------------------------------------------ */
/* Chunk sort + pad, unpad + restore  [TE-PR]                                */
/* ------------------------------------------------------------------------ */

/* Flags the oracle reports for data it had to repair (the GPU reports the
 * same conditions in its own status word). */
typedef struct {
    int32_t bad_split;      /* some split_sizes[c] < 0 (taken as 0)           */
    int32_t bad_order;      /* some chunk_order entry outside [0,C) (skipped)  */
    int32_t split_overflow; /* sum of split sizes > N (rows >= N not read)     */
    int32_t rows_overflow;  /* sum of padded group sizes > out_rows (dropped)  */
    int32_t bad_padded;     /* a given padded size below its group's rows      */
} orc_chunk_flags;

/*
 * Rows here are W 16-bit units wide: H for bf16 / fp16 tokens, 2H for fp32
 * (the copies only move bits, so the element type does not matter).
 *
 * Fused sort + pad: input rows arrive as C consecutive chunks whose sizes are
 * split_sizes (input order).  The output holds G groups; group g is made of
 * the chunks chunk_order[g*C/G .. (g+1)*C/G) in that order, each chunk's rows
 * consecutive and in their input order, and the group is then zero-padded up
 * to a multiple of `align` rows ("zero-fills each expert group up to an
 * alignment").  group_off[g] is the first output row of group g and
 * group_off[G] the padded total.  row_map[d] is the input row placed at output
 * row d, or -1 for a padding row; output rows from group_off[G] to out_rows
 * are padding too.  Padding rows are zero and their probabilities 0.
 * probs / out_probs may be NULL together.  With padded_sizes given ("padded
 * sizes are explicit", [TE-PR, Description]), group g takes exactly
 * padded_sizes[g] rows instead (negative counts as 0); a group with more rows
 * than that keeps its first padded_sizes[g] rows and is flagged.
 */
void orc_sort_chunks_pad(const uint16_t *x, const float *probs,
                         const int32_t *split_sizes, const int32_t *chunk_order,
                         const int32_t *padded_sizes, int32_t C, int32_t G, int32_t align,
                         int64_t N, int64_t out_rows, int32_t H, uint16_t *out,
                         float *out_probs, int32_t *row_map, int64_t *group_off,
                         orc_chunk_flags *flags)
{
    orc_chunk_flags f = {0, 0, 0, 0, 0};
    int64_t *in_start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
    int64_t total = 0;
    for (int32_t c = 0; c < C; ++c) {
        int64_t s = split_sizes[c];
        if (s < 0) {
            f.bad_split = 1;
            s = 0;
        }
        in_start[c] = total;
        total += s;
    }
    if (total > N)
        f.split_overflow = 1;

    /* Every output row starts as padding. */
    for (int64_t d = 0; d < out_rows; ++d) {
        row_map[d] = -1;
        for (int32_t h = 0; h < H; ++h)
            out[d * H + h] = 0;
        if (probs && out_probs)
            out_probs[d] = 0.0f;
    }

    const int32_t per_group = C / G;
    int64_t d = 0;
    for (int32_t g = 0; g < G; ++g) {
        group_off[g] = d;
        /* rows the group holds before padding */
        int64_t rows_in_group = 0;
        for (int32_t j = 0; j < per_group; ++j) {
            int32_t c = chunk_order[g * per_group + j];
            if (c >= 0 && c < C && split_sizes[c] > 0)
                rows_in_group += split_sizes[c];
        }
        int64_t padded = ((rows_in_group + align - 1) / align) * align;
        if (padded_sizes) {
            padded = padded_sizes[g] < 0 ? 0 : padded_sizes[g];
            if (padded < rows_in_group)
                f.bad_padded = 1;
        }
        /* place the rows in order, as many as the padded size holds */
        int64_t placed = 0;
        for (int32_t j = 0; j < per_group; ++j) {
            int32_t c = chunk_order[g * per_group + j];
            if (c < 0 || c >= C) {
                f.bad_order = 1;
                continue;
            }
            int64_t s = split_sizes[c] < 0 ? 0 : split_sizes[c];
            for (int64_t i = 0; i < s && placed < padded; ++i) {
                int64_t src = in_start[c] + i;
                int64_t dd = d + placed;
                if (dd < out_rows && src < N) {
                    row_map[dd] = (int32_t)src;
                    for (int32_t h = 0; h < H; ++h)
                        out[dd * H + h] = x[src * H + h];
                    if (probs && out_probs)
                        out_probs[dd] = probs[src];
                }
                placed += 1;
            }
        }
        d += padded;
    }
    group_off[G] = d;
    if (d > out_rows)
        f.rows_overflow = 1;
    free(in_start);
    if (flags)
        *flags = f;
}

/* Unpad + restore [TE-PR, Diagram "Unpad and restore using row map"]: every
 * output row d that holds an input row goes back to it, y[row_map[d]] =
 * padded[d] (and the probability likewise); padding rows are dropped.  Rows of
 * y that no d names are left as they are. */
void orc_unpad_restore(const uint16_t *padded, const float *padded_probs,
                       const int32_t *row_map, int64_t out_rows, int64_t N, int32_t H,
                       uint16_t *y, float *y_probs)
{
    for (int64_t d = 0; d < out_rows; ++d) {
        int32_t s = row_map[d];
        if (s < 0 || s >= N)
            continue;
        for (int32_t h = 0; h < H; ++h)
            y[(int64_t)s * H + h] = padded[d * H + h];
        if (padded_probs && y_probs)
            y_probs[s] = padded_probs[d];
    }
}

/* Backward of sort + pad: the gradient of each input row is the gradient of
 * the output row it was copied to; padding gradients are discarded.  This is
 * unpad + restore applied to the gradients. */
void orc_sort_chunks_pad_bwd(const uint16_t *g_out, const float *g_out_probs,
                             const int32_t *row_map, int64_t out_rows, int64_t N,
                             int32_t H, uint16_t *g_x, float *g_probs)
{
    orc_unpad_restore(g_out, g_out_probs, row_map, out_rows, N, H, g_x, g_probs);
}

/* Backward of unpad + restore: output row d receives the gradient of the row
 * it restored; padding rows get a zero gradient ("Padding is zero-filled and
 * contributes zero gradient", [TE-PR, Changes]). */
void orc_unpad_restore_bwd(const uint16_t *g_y, const float *g_y_probs,
                           const int32_t *row_map, int64_t out_rows, int64_t N,
                           int32_t H, uint16_t *g_padded, float *g_padded_probs)
{
    for (int64_t d = 0; d < out_rows; ++d) {
        int32_t s = row_map[d];
        int ok = (s >= 0 && s < N);
        for (int32_t h = 0; h < H; ++h)
            g_padded[d * H + h] = ok ? g_y[(int64_t)s * H + h] : (uint16_t)0;
        if (g_y_probs && g_padded_probs)
            g_padded_probs[d] = ok ? g_y_probs[s] : 0.0f;
    }
}
