/*
 * mp.h -- C ABI of libmp: Mixture-of-Experts token permute / unpermute on one
 * GB300 GPU (sm_103a).
 *
 * The operations and their sources (web pages, cited by title and section):
 *   [d9d]   "d9d 0.1.0 -- d9d/kernel/moe/permute_with_probs.py", a copy of
 *           TransformerEngine permutation.py: make_row_id_map (and its worked
 *           example), _permute_kernel, _unpermute_kernel,
 *           _unpermute_bwd_with_merging_probs_kernel, and the autograd classes
 *           _moe_permute_mask_map / _moe_unpermute_mask_map.
 *   [MBI]   "core.transformer.moe.batch_invariant" (Megatron-Core API docs):
 *           _rank_tree_unpermute_kernel, _rank_tree_unpermute_bwd_kernel,
 *           _unpermute_loop, unpermute.
 *   [xt]    "permute different with torch version" (xtuner issue 1323).
 *   [mops]  "moe-ops 0.1.0" README: "Why this library", "Layout conventions",
 *           "Operators" (permute / unpermute / permute_backward).
 *   [TE-PR] "[PyTorch] Fuse MoE chunk sorting and padding"
 *           (TransformerEngine PR 3509): Description, Changes, Diagram.
 *
 * Common rules for every entry point
 * ----------------------------------
 *  - Pointers marked "device" are CUDA device (or managed) pointers; the
 *    caller owns every buffer.  The library never allocates, never frees and
 *    never synchronises: each call enqueues kernels on `stream` (a
 *    cudaStream_t passed as void*; NULL is the legacy default stream) and
 *    returns.  Grids depend on the shape arguments only, so a call can be
 *    captured in a CUDA graph and replayed with new routing in the same
 *    buffers.
 *  - Kernels are launched as programmatic dependents of the work before them
 *    in the stream: a kernel may be scheduled while the previous kernel
 *    drains, but it waits for that kernel to finish before it touches
 *    memory.  Stream order holds as for ordinary launches, and a caller needs
 *    no extra synchronisation.
 *  - Tensors are dense and row-major.  bf16 tensors are passed as their
 *    16-bit patterns (mp_bf16_t).  A row of H bf16 values is 2*H bytes.
 *    Rows move as 16-byte vectors when H % 8 == 0 and every row pointer is
 *    16-byte aligned, else element by element.  The permute on rows of more
 *    than 4 KiB and the sort+pad on outputs of more than 16,384 rows of at
 *    least 1 KiB move 32-byte vectors when the row size is a multiple of 32
 *    bytes and the tensors are 32-byte aligned.  Results are identical on
 *    every path.
 *  - Routes: T tokens, K slots per token, R = T*K <= 2^31 - 1.
 *    E <= MP_MAX_EXPERTS.
 *  - Errors found on the host (a NULL required pointer, a negative or
 *    out-of-range size, a too-small workspace) return a negative mp_status_t
 *    and launch nothing.  A failing launch returns MP_ERR_CUDA;
 *    mp_last_cuda_error() then gives the cudaError_t of the calling thread.
 *  - Errors in the data (an expert index outside [-1,E), bad chunk sizes) are
 *    never fatal: the offending entry is treated as empty, and, if
 *    `dev_status` is not NULL, the kernel ORs an MP_STATUS_* bit into the
 *    device word *dev_status (which the caller zeroes beforehand and reads
 *    when it likes).
 *  - Empty inputs (T == 0 or N == 0) are valid: nothing is copied.
 */
#ifndef MP_H
#define MP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mp_status_t;
typedef uint16_t mp_bf16_t;   /* bit pattern of a bfloat16 value            */
typedef void *mp_stream_t;    /* a cudaStream_t                             */

#define MP_OK 0
#define MP_ERR_INVALID_ARG (-1) /* bad pointer or size: nothing launched     */
#define MP_ERR_WORKSPACE (-2)   /* workspace NULL, misaligned or too small   */
#define MP_ERR_UNSUPPORTED (-3) /* size beyond a documented limit            */
#define MP_ERR_CUDA (-4)        /* a launch failed (see mp_last_cuda_error)  */

/* Bits ORed into *dev_status by the kernels. */
#define MP_STATUS_BAD_EXPERT 0x1     /* idx value outside [-1,E): taken as -1   */
#define MP_STATUS_BAD_SPLIT 0x2      /* split_sizes[c] < 0: taken as 0          */
#define MP_STATUS_BAD_ORDER 0x4      /* chunk_order entry outside [0,C): skipped */
#define MP_STATUS_SPLIT_OVERFLOW 0x8 /* sum of split sizes > N: rows >= N unread */
#define MP_STATUS_ROWS_OVERFLOW 0x10 /* padded total > out_rows: excess dropped  */
#define MP_STATUS_BAD_ROW 0x20       /* row_map entry outside [-1,N): skipped    */
#define MP_STATUS_BAD_PADDED 0x40    /* a padded size below its group's rows     */

/* Token types of the chunk entry points with a dtype argument. */
#define MP_DTYPE_BF16 0
#define MP_DTYPE_FP16 1
#define MP_DTYPE_FP32 2

#define MP_MAX_EXPERTS 1024
#define MP_MAX_CHUNKS 1024

/* Text for a status code (static storage). */
const char *mp_status_string(mp_status_t status);

/* cudaError_t of the last MP_ERR_CUDA returned on the calling thread. */
int32_t mp_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Routing map  [d9d make_row_id_map; mops "Operators: permute"; xt]         */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace mp_build_map (and mp_build_map_capacity) needs
 * for these sizes: a multiple of 256, at least 256.  Returns 0 only for
 * invalid sizes (those mp_build_map rejects). */
size_t mp_build_map_workspace_size(int64_t T, int32_t K, int32_t E);

/*
 * Counting sort of the routes by expert: histogram, exclusive scan, stable
 * rank.  Rows are ordered by expert, then token, then slot.
 *   idx            device int32 [T,K]  expert of slot k of token t; -1 = empty
 *                                      slot (no row).
 *   row_id_map     device int32 [T,K]  out: row of (t,k) in the permuted
 *                                      tensor, -1 for an empty slot.
 *   sorted_to_flat device int32 [T*K]  out, may be NULL: t*K+k for each row
 *                                      below offsets[E], -1 after it.
 *   counts         device int32 [E]    out: routes per expert.
 *   offsets        device int32 [E+1]  out: offsets[0] = 0, offsets[e+1] =
 *                                      offsets[e] + counts[e]; expert e owns
 *                                      rows [offsets[e], offsets[e+1]).
 *   workspace      device, >= mp_build_map_workspace_size(T,K,E) bytes,
 *                  4-byte aligned; scratch, contents undefined after the call.
 *   dev_status     device int32 or NULL: MP_STATUS_BAD_EXPERT.
 * Deterministic: the result does not depend on scheduling.
 */
mp_status_t mp_build_map(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                         int32_t *row_id_map, int32_t *sorted_to_flat, int32_t *counts,
                         int32_t *offsets, void *workspace, size_t workspace_bytes,
                         int32_t *dev_status, mp_stream_t stream);

/*
 * mp_build_map with an expert capacity (token dropping).  Expert e keeps at
 * most `capacity` routes -- the first ones in (token, slot) order -- and the
 * others are dropped like empty slots (row_id_map = -1).  counts[e] is the
 * number kept and offsets its exclusive scan, so offsets[E] is the effective
 * output row count, the "num_out_tokens" of [d9d moe_permute_with_probs]
 * ("the number of tokens not dropped"); sorted_to_flat is -1 from offsets[E]
 * on.  capacity < 0 means no limit (the same result as mp_build_map).  Other
 * arguments, workspace and errors as mp_build_map.
 */
mp_status_t mp_build_map_capacity(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                                  int32_t capacity, int32_t *row_id_map,
                                  int32_t *sorted_to_flat, int32_t *counts, int32_t *offsets,
                                  void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                  mp_stream_t stream);

/*
 * Allocation-free mp_build_map.  The pages have no counterpart: this entry
 * point exists for callers that cannot call cudaMalloc -- an inference
 * runtime or plugin that plans all device memory at start-up and forbids
 * allocation afterwards, a framework whose allocator owns the device memory,
 * or a latency-critical path that must not risk the implicit device
 * synchronisation of cudaMalloc.  It computes exactly what mp_build_map
 * computes, but its scratch (the per-tile expert counts) lives in a static
 * device array inside the library, MP_NOALLOC_SCRATCH_BYTES per GPU, which
 * every GPU that loads the library holds until the process exits.  The
 * caller still passes every input and output.
 *   - Limit: (E+1) * tiles * 4 <= MP_NOALLOC_SCRATCH_BYTES, where tiles =
 *     ceil(T*K / (2048*f)) and f is the smallest of 1, 2, 4, 8 that gives at
 *     most 64 tiles (so every E is accepted up to 1,048,576 routes; E=128 up
 *     to 33,292,288 routes, E=1024 up to 4,177,920).  Larger sizes return
 *     MP_ERR_UNSUPPORTED and launch nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and caches it for the
 *     life of the process; make that first call before any stream capture.
 *     Resetting a device (cudaDeviceReset) after that first call is not
 *     supported: the array may then move and the cached address would be
 *     stale.
 *   - All calls share the one array.  Calls that overlap on the GPU (other
 *     streams, other threads) race on it and give wrong maps: serialise them.
 *     Nothing needs clearing between calls: every entry a call reads was
 *     written earlier in the same call.
 *   - Never calls cudaMalloc, cudaFree or any allocating routine.
 * Arguments, outputs and errors are those of mp_build_map without the
 * workspace.
 */
#define MP_NOALLOC_SCRATCH_BYTES (1u << 20)

mp_status_t mp_build_map_noalloc(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                                 int32_t *row_id_map, int32_t *sorted_to_flat,
                                 int32_t *counts, int32_t *offsets, int32_t *dev_status,
                                 mp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Router  [mops "Operators: fused_topk_softmax"]                            */
/* ------------------------------------------------------------------------ */

/*
 * Fused top-k softmax: the routing input of mp_build_map from router logits.
 * Per token: if n_groups > 1, keep only the topk_groups best of n_groups equal
 * groups of consecutive experts (score = the group's largest logit; equal
 * scores favour the lower group); then pick the K largest logits among the
 * kept experts (equal logits favour the lower expert), slot 0 the largest.
 * probs = fp32 softmax over the K picked logits: z_k = l_k - l_0, expf
 * (CUDA's full-accuracy expf), sum in slot order, IEEE division.  Logits
 * compare as floats (+0 and -0 are equal); with a NaN logit the picks are
 * unspecified.
 *   logits  device fp32 [T,E];  idx device int32 [T,K];  probs device fp32 [T,K]
 * Limits: E <= MP_MAX_EXPERTS, K <= 32, n_groups <= 32, E % n_groups == 0,
 * topk_groups * E / n_groups >= K.
 */
mp_status_t mp_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t K,
                            int32_t n_groups, int32_t topk_groups, int32_t *idx, float *probs,
                            mp_stream_t stream);

/*
 * Backward of mp_topk_softmax: g_logits[t,e] = p_k * (g_probs[t,k] - d) at
 * the picked expert e = idx[t,k], with d = sum_k p_k * g_probs[t,k] (fused
 * multiply-adds in slot order from +0), and 0 for every other expert.
 *   g_probs, probs device fp32 [T,K];  idx device int32 [T,K];
 *   g_logits device fp32 [T,E] (every element written).
 */
mp_status_t mp_topk_softmax_bwd(const float *g_probs, const float *probs, const int32_t *idx,
                                int64_t T, int32_t E, int32_t K, float *g_logits,
                                mp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Permute / unpermute  [d9d _permute_kernel, _unpermute_kernel; MBI]        */
/* ------------------------------------------------------------------------ */

/*
 * out[row_id_map[t,k], :] = x[t, :]  and  out_probs[row_id_map[t,k]] =
 * probs[t,k], for every non-empty slot.  The row is copied whatever its
 * probability.
 *   x          device bf16 [T,H]
 *   probs      device fp32 [T,K] or NULL
 *   row_id_map device int32 [T,K] from mp_build_map
 *   out        device bf16 [R_out,H], R_out > every row id (T*K suffices);
 *              rows no slot maps to are not written.
 *   out_probs  device fp32 [R_out] or NULL; given exactly when probs is
 *              (otherwise MP_ERR_INVALID_ARG)
 */
mp_status_t mp_permute(const mp_bf16_t *x, const float *probs, const int32_t *row_id_map,
                       int64_t T, int32_t K, int32_t H, mp_bf16_t *out, float *out_probs,
                       mp_stream_t stream);

/*
 * Batch-invariant combine: for each token t and element h,
 *   acc = +0.0f; for k = 0..K-1 (slot order, empty slots skipped):
 *       acc = fmaf(probs[t,k], float(rows[row_id_map[t,k], h]), acc)
 *   out[t,h] = bf16 round-to-nearest-even(acc)
 * With probs == NULL: acc = acc + float(row) (a plain sum).  FP32 fused
 * multiply-adds in slot order from zero, one BF16 rounding
 * [MBI _rank_tree_unpermute_kernel; unpermute].  A token with no routed
 * slot gets +0.
 *   rows  device bf16 [>= max row id + 1, H];  out device bf16 [T,H].
 */
mp_status_t mp_unpermute(const mp_bf16_t *rows, const float *probs,
                         const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                         mp_bf16_t *out, mp_stream_t stream);

/* Flags of mp_unpermute_ep. */
#define MP_EP_BF16_PARTIALS 0x1   /* quantize each rank's partial to BF16     */
#define MP_EP_FP64_CROSS_RANK 0x2 /* add the rank partials in FP64 (else FP32) */

/*
 * Rank-ordered combine over expert-parallel ranks, simulated on one GPU
 * [MBI _rank_tree_unpermute_kernel, unpermute_with_bf16_rank_partials,
 * unpermute]: rank r owns experts [r*E/ep_size, (r+1)*E/ep_size).  For each
 * token and element: for every rank r in increasing order, the rank's partial
 * is the slot-order chain fmaf(probs[t,k], row, partial) from +0 over the
 * token's routed slots whose expert idx[t,k] lies on r (plain adds when probs
 * is NULL), rounded to BF16 if MP_EP_BF16_PARTIALS; the partials are added in
 * rank order from zero in FP32, or FP64 with MP_EP_FP64_CROSS_RANK; the sum
 * is rounded once (RNE, from FP64 directly) to BF16.  ep_size = 1 without
 * flags gives exactly mp_unpermute.
 *   idx        device int32 [T,K]: the expert of each slot (the routing input
 *              of mp_build_map); other arguments as mp_unpermute.
 * Limits: K <= 16, E % ep_size == 0.
 */
mp_status_t mp_unpermute_ep(const mp_bf16_t *rows, const float *probs,
                            const int32_t *row_id_map, const int32_t *idx, int64_t T, int32_t K,
                            int32_t H, int32_t E, int32_t ep_size, int32_t flags, mp_bf16_t *out,
                            mp_stream_t stream);

/*
 * Backward of mp_permute [d9d _moe_permute_mask_map.backward; mops
 * permute_backward]:
 *   g_x[t,h]     = bf16_rne(sum over k in slot order, fp32 from +0, of
 *                  float(g_out[row_id_map[t,k], h]))      (= mp_unpermute, no probs)
 *   g_probs[t,k] = g_out_probs[row_id_map[t,k]], 0 for an empty slot.
 *   g_out_probs / g_probs: both NULL or both given.
 */
mp_status_t mp_permute_bwd(const mp_bf16_t *g_out, const float *g_out_probs,
                           const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                           mp_bf16_t *g_x, float *g_probs, mp_stream_t stream);

/*
 * Backward of mp_unpermute.
 * With probs [d9d _unpermute_bwd_with_merging_probs_kernel]:
 *   g_rows[row_id_map[t,k], h] = bf16_rne(probs[t,k] * float(g_y[t,h]))
 *   g_probs[t,k] = sum_h float(rows[row_id_map[t,k], h]) * float(g_y[t,h])
 *                  in fp32 (fixed reduction tree, so deterministic; 0 for an
 *                  empty slot).  `rows` is the forward input.
 * Without probs [MBI _rank_tree_unpermute_bwd_kernel]: g_rows[row] = g_y[t]
 * for each routed slot; rows and g_probs may be NULL.
 */
mp_status_t mp_unpermute_bwd(const mp_bf16_t *g_y, const mp_bf16_t *rows,
                             const float *probs, const int32_t *row_id_map, int64_t T,
                             int32_t K, int32_t H, mp_bf16_t *g_rows, float *g_probs,
                             mp_stream_t stream);

/*
 * Zeroes rows [*first_row, rows) of a row-major device buffer.  The start row
 * is read from device memory -- typically offsets + E of mp_build_map or
 * mp_build_map_capacity, the routed row count, so that the rows of a
 * permuted buffer (or of its gradient) that no slot maps to, left unwritten
 * by mp_permute and mp_unpermute_bwd, become zero without a host round trip
 * ["d9d 0.1.0 -- permute_with_probs.py", num_out_tokens: rows past the
 * tokens kept].  *first_row is clamped to [0, rows]; at or past rows
 * nothing is written.
 *   buf        device, rows * row_bytes bytes (any alignment; 16-byte
 *              aligned with row_bytes % 16 == 0 takes vector stores)
 *   rows       >= 0;  row_bytes >= 0 (e.g. 2*H for bf16 rows, 4 for probs)
 *   first_row  device int32 [1]
 * rows == 0 or row_bytes == 0 is a no-op (NULL pointers allowed);
 * otherwise NULL pointers or a negative size give MP_ERR_INVALID_ARG.
 */
mp_status_t mp_zero_rows_from(void *buf, int64_t rows, int64_t row_bytes,
                              const int32_t *first_row, mp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Chunk sort + pad, unpad + restore  [TE-PR]                                */
/* ------------------------------------------------------------------------ */

/*
 * Fused sort + pad.  The N-row input holds C consecutive chunks, chunk c
 * having split_sizes[c] rows (input order).  Output group g (G groups, C % G
 * == 0) is made of chunks chunk_order[g*C/G .. (g+1)*C/G) in that order, each
 * chunk's rows consecutive and in input order, then zero rows up to a
 * multiple of `align`.  Output rows past the padded total, up to out_rows,
 * are zero too.
 *   x, probs            device bf16 [N,H], fp32 [N] or NULL (probs and
 *                       out_probs are both given or both NULL)
 *   split_sizes         device int32 [C]   (runtime data: a graph replays with
 *   chunk_order         device int32 [C]    new sizes in the same buffers)
 *   out, out_probs      device bf16 [out_rows,H], fp32 [out_rows] or NULL
 *   row_map             device int32 [out_rows] out: input row at each output
 *                       row, -1 for padding (the map the restore uses)
 *   group_off           device int64 [G+1] out: first row of each group, and
 *                       the padded total at [G]
 *   dev_status          MP_STATUS_BAD_SPLIT / BAD_ORDER / SPLIT_OVERFLOW /
 *                       ROWS_OVERFLOW
 * Limits: 1 <= C <= MP_MAX_CHUNKS, align >= 1, N < 2^31, out_rows < 2^31.
 */
mp_status_t mp_sort_chunks_pad(const mp_bf16_t *x, const float *probs,
                               const int32_t *split_sizes, const int32_t *chunk_order,
                               int32_t C, int32_t G, int32_t align, int64_t N,
                               int64_t out_rows, int32_t H, mp_bf16_t *out,
                               float *out_probs, int32_t *row_map, int64_t *group_off,
                               int32_t *dev_status, mp_stream_t stream);

/*
 * Unpad + restore: y[row_map[d]] = padded[d] (and y_probs likewise) for every
 * d with row_map[d] >= 0; padding rows are dropped.  Rows of y that no d
 * names are not written.  row_map must not name a row twice.
 * dev_status: MP_STATUS_BAD_ROW for an entry outside [-1,N).
 */
mp_status_t mp_unpad_restore(const mp_bf16_t *padded, const float *padded_probs,
                             const int32_t *row_map, int64_t out_rows, int64_t N,
                             int32_t H, mp_bf16_t *y, float *y_probs, int32_t *dev_status,
                             mp_stream_t stream);

/* Backward of mp_sort_chunks_pad: g_x[row_map[d]] = g_out[d] (padding
 * gradients discarded) -- mp_unpad_restore applied to the gradients. */
mp_status_t mp_sort_chunks_pad_bwd(const mp_bf16_t *g_out, const float *g_out_probs,
                                   const int32_t *row_map, int64_t out_rows, int64_t N,
                                   int32_t H, mp_bf16_t *g_x, float *g_probs,
                                   int32_t *dev_status, mp_stream_t stream);

/* Backward of mp_unpad_restore: g_padded[d] = g_y[row_map[d]], and zero for
 * padding rows ("contributes zero gradient"). */
mp_status_t mp_unpad_restore_bwd(const mp_bf16_t *g_y, const float *g_y_probs,
                                 const int32_t *row_map, int64_t out_rows, int64_t N,
                                 int32_t H, mp_bf16_t *g_padded, float *g_padded_probs,
                                 int32_t *dev_status, mp_stream_t stream);

/*
 * The chunk entry points for FP32, FP16 and BF16 tokens ([TE-PR Changes]):
 * `dtype` is an MP_DTYPE_*, rows are H elements of that type, and the other
 * arguments are those of the bf16 entry points above.  mp_sort_chunks_pad_ex
 * also takes padded_sizes, device int32 [G] or NULL ("Chunk order and padded
 * sizes are explicit", [TE-PR Description]): when given, group g occupies
 * exactly padded_sizes[g] output rows (a negative size counts as 0; `align`
 * is then unused), and a group with more rows keeps its first
 * padded_sizes[g] rows and sets MP_STATUS_BAD_PADDED.
 */
mp_status_t mp_sort_chunks_pad_ex(const void *x, int32_t dtype, const float *probs,
                                  const int32_t *split_sizes, const int32_t *chunk_order,
                                  const int32_t *padded_sizes, int32_t C, int32_t G,
                                  int32_t align, int64_t N, int64_t out_rows, int32_t H,
                                  void *out, float *out_probs, int32_t *row_map,
                                  int64_t *group_off, int32_t *dev_status, mp_stream_t stream);
mp_status_t mp_unpad_restore_ex(const void *padded, int32_t dtype, const float *padded_probs,
                                const int32_t *row_map, int64_t out_rows, int64_t N, int32_t H,
                                void *y, float *y_probs, int32_t *dev_status,
                                mp_stream_t stream);
mp_status_t mp_sort_chunks_pad_bwd_ex(const void *g_out, int32_t dtype,
                                      const float *g_out_probs, const int32_t *row_map,
                                      int64_t out_rows, int64_t N, int32_t H, void *g_x,
                                      float *g_probs, int32_t *dev_status, mp_stream_t stream);
mp_status_t mp_unpad_restore_bwd_ex(const void *g_y, int32_t dtype, const float *g_y_probs,
                                    const int32_t *row_map, int64_t out_rows, int64_t N,
                                    int32_t H, void *g_padded, float *g_padded_probs,
                                    int32_t *dev_status, mp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MP_H */
