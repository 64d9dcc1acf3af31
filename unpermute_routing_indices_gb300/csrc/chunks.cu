// Fused chunk sort + pad and its unpad + restore ("[PyTorch] Fuse MoE chunk
// sorting and padding", TransformerEngine PR 3509: one pass that copies the
// tokens and probabilities into expert order with zero padding, and one copy
// back through the saved row map).
//
//   k_sort_pad     one launch for map + copy.  Every CTA rebuilds the small
//                  chunk metadata in shared memory (C <= MP_MAX_CHUNKS sizes:
//                  input starts, output-order starts, group rows, padded group
//                  offsets), then resolves the source row of each of its
//                  CH_ROWS output rows by two binary searches and copies the
//                  rows (zero for padding).  CTA 0 also writes group_off and
//                  the status bits.  Nothing is carried between CTAs, so the
//                  grid depends on out_rows only and sizes are runtime data.
//   k_rows_gather  out[d] = in[map[d]] or zero     (unpad+restore backward)
//   k_rows_scatter out[map[d]] = in[d] if map[d] >= 0  (unpad+restore, and the
//                  sort+pad backward)
#include "common.cuh"

namespace mp {
namespace {

constexpr int CH_THREADS = 256;
constexpr int CH_WARPS = CH_THREADS / 32;
constexpr int CH_ROWS = 16;   // output rows per CTA
constexpr int CH_UNROLL = 8;  // vectors in flight per thread

// In-place exclusive scan of a[0..n), n <= 4 * CH_THREADS, in shared memory.
// Returns the total.  Every thread of the CTA must call it.
__device__ int64_t cta_exclusive_scan(int64_t *a, int n, int64_t *s_warp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = tid * 4;
    int64_t v[4], sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[j] = (lo + j < n) ? a[lo + j] : 0;
        sum += v[j];
    }
    int64_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int64_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < CH_WARPS; ++w) {
        if (w < warp) before += s_warp[w];
        total += s_warp[w];
    }
    int64_t run = before + incl - sum;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (lo + j < n) a[lo + j] = run;
        run += v[j];
    }
    __syncthreads();
    return total;
}

// Largest i in [lo, hi) with a[i] <= key (a non-decreasing, a[lo] <= key).
__device__ __forceinline__ int last_le(const int64_t *a, int lo, int hi, int64_t key)
{
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= key) lo = mid; else hi = mid;
    }
    return lo;
}

// Copies the CTA's rows: out[row0 + r] = src[r] >= 0 ? in[src[r]] : 0 (gather)
// or out[dst[r]] = in[row0 + r] (scatter, rows with dst < 0 skipped).
template <typename V, bool SCATTER>
__device__ __forceinline__ void copy_rows(const V *__restrict__ in, V *__restrict__ out,
                                          const int32_t *s_map, int64_t row0, int nrows, int nvec)
{
    const int total = nrows * nvec;
    for (int w0 = 0; w0 < total; w0 += CH_THREADS * CH_UNROLL) {
        V v[CH_UNROLL];
        int64_t dst_off[CH_UNROLL];
#pragma unroll
        for (int u = 0; u < CH_UNROLL; ++u) {
            const int w = w0 + u * CH_THREADS + threadIdx.x;
            dst_off[u] = -1;
            v[u] = zero_vec<V>();
            if (w < total) {
                const int r = w / nvec, c = w - r * nvec;
                const int32_t m = s_map[r];
                if (SCATTER) {
                    if (m >= 0) {
                        v[u] = ld_stream(in + (row0 + r) * nvec + c);
                        dst_off[u] = (int64_t)m * nvec + c;
                    }
                } else {
                    if (m >= 0) v[u] = ld_stream(in + (int64_t)m * nvec + c);
                    dst_off[u] = (row0 + r) * nvec + c;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < CH_UNROLL; ++u)
            if (dst_off[u] >= 0) st_row(out + dst_off[u], v[u]);
    }
}

template <typename V>
__global__ void __launch_bounds__(CH_THREADS)
    k_sort_pad(const V *__restrict__ x, const float *__restrict__ probs,
               const int32_t *__restrict__ split, const int32_t *__restrict__ order,
               const int32_t *__restrict__ padded_sizes, int C, int G,
               int align, int64_t N, int64_t out_rows, int nvec, V *__restrict__ out,
               float *__restrict__ out_probs, int32_t *__restrict__ row_map,
               int64_t *__restrict__ group_off, int32_t *status)
{
    extern __shared__ int64_t sm[];
    int64_t *s_start = sm;               // [C]   first input row of chunk c
    int64_t *s_cum = s_start + C;        // [C+1] rows before position p in output order
    int64_t *s_goff = s_cum + C + 1;     // [G+1] padded group offsets
    int64_t *s_grows = s_goff + G + 1;   // [G]   unpadded rows of group g
    int64_t *s_warp = s_grows + G;       // [CH_WARPS]
    int32_t *s_chunk = reinterpret_cast<int32_t *>(s_warp + CH_WARPS);  // [C]
    int32_t *s_src = s_chunk + C;        // [CH_ROWS]
    __shared__ int s_flags;

    const int tid = threadIdx.x;
    if (tid == 0) s_flags = 0;
    __syncthreads();
    int flags = 0;
    for (int c = tid; c < C; c += CH_THREADS) {
        int64_t v = split[c];
        if (v < 0) { flags |= MP_STATUS_BAD_SPLIT; v = 0; }
        s_start[c] = v;
    }
    __syncthreads();
    const int64_t total_in = cta_exclusive_scan(s_start, C, s_warp);

    for (int p = tid; p < C; p += CH_THREADS) {
        const int32_t c = order[p];
        const bool ok = c >= 0 && c < C;
        if (!ok) flags |= MP_STATUS_BAD_ORDER;
        s_chunk[p] = ok ? c : -1;
        s_cum[p] = ok ? ((c + 1 < C ? s_start[c + 1] : total_in) - s_start[c]) : 0;
    }
    if (flags) atomicOr(&s_flags, flags);
    __syncthreads();
    const int64_t total_ord = cta_exclusive_scan(s_cum, C, s_warp);
    if (tid == 0) s_cum[C] = total_ord;
    __syncthreads();

    const int per_group = C / G;
    for (int g = tid; g < G; g += CH_THREADS) {
        const int64_t rows = s_cum[(g + 1) * per_group] - s_cum[g * per_group];
        s_grows[g] = rows;
        int64_t padded = (rows + align - 1) / align * align;
        if (padded_sizes != nullptr) {   // explicit padded sizes
            const int32_t ps = padded_sizes[g];
            padded = ps < 0 ? 0 : ps;
            if (padded < rows) atomicOr(&s_flags, MP_STATUS_BAD_PADDED);
        }
        s_goff[g] = padded;
    }
    __syncthreads();
    const int64_t total_pad = cta_exclusive_scan(s_goff, G, s_warp);
    if (tid == 0) s_goff[G] = total_pad;
    __syncthreads();

    if (blockIdx.x == 0) {
        for (int g = tid; g <= G; g += CH_THREADS) group_off[g] = s_goff[g];
        if (tid == 0) {
            int bits = s_flags;
            if (total_in > N) bits |= MP_STATUS_SPLIT_OVERFLOW;
            if (total_pad > out_rows) bits |= MP_STATUS_ROWS_OVERFLOW;
            or_status(status, bits);
        }
    }

    const int64_t row0 = (int64_t)blockIdx.x * CH_ROWS;
    const int64_t left = out_rows - row0;
    const int nrows = left < CH_ROWS ? (int)left : CH_ROWS;
    if (tid < nrows) {
        const int64_t d = row0 + tid;
        int32_t src = -1;
        if (d < total_pad) {
            const int g = last_le(s_goff, 0, G, d);
            const int64_t j = d - s_goff[g];
            if (j < s_grows[g]) {
                const int64_t target = s_cum[g * per_group] + j;
                const int p = last_le(s_cum, g * per_group, (g + 1) * per_group, target);
                const int64_t s = s_start[s_chunk[p]] + (target - s_cum[p]);
                src = s < N ? (int32_t)s : -1;
            }
        }
        s_src[tid] = src;
        row_map[d] = src;
        if (out_probs != nullptr) out_probs[d] = src >= 0 ? __ldg(probs + src) : 0.0f;
    }
    __syncthreads();
    if (nrows > 0) copy_rows<V, false>(x, out, s_src, row0, nrows, nvec);
}

template <typename V, bool SCATTER>
__global__ void __launch_bounds__(CH_THREADS)
    k_rows_remap(const V *__restrict__ in, const float *__restrict__ in_probs,
                 const int32_t *__restrict__ map, int64_t out_rows, int64_t N, int nvec,
                 V *__restrict__ out, float *__restrict__ out_probs, int32_t *status)
{
    __shared__ int32_t s_map[CH_ROWS];
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * CH_ROWS;
    const int64_t left = out_rows - row0;
    const int nrows = left < CH_ROWS ? (int)left : CH_ROWS;
    if (tid < nrows) {
        const int64_t d = row0 + tid;
        int32_t m = __ldg(map + d);
        if (m < -1 || m >= N) {
            or_status(status, MP_STATUS_BAD_ROW);
            m = -1;
        }
        s_map[tid] = m;
        if (in_probs != nullptr) {
            if (SCATTER) {
                if (m >= 0) out_probs[m] = __ldg(in_probs + d);
            } else {
                out_probs[d] = m >= 0 ? __ldg(in_probs + m) : 0.0f;
            }
        }
    }
    __syncthreads();
    copy_rows<V, SCATTER>(in, out, s_map, row0, nrows, nvec);
}

inline bool chunk_vec_ok(int32_t H, std::initializer_list<const void *> ptrs)
{
    if (H % 8 != 0) return false;
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p)) return false;
    return true;
}

inline size_t sort_pad_smem(int C, int G)
{
    return sizeof(int64_t) * (size_t)(C + (C + 1) + (G + 1) + G + CH_WARPS) +
           sizeof(int32_t) * (size_t)(C + CH_ROWS);
}

// Rows are H 16-bit units wide.
mp_status_t remap(const void *in, const float *in_probs, const int32_t *map, int64_t out_rows,
                  int64_t N, int32_t H, void *out, float *out_probs, int32_t *status,
                  cudaStream_t s, bool scatter)
{
    if (out_rows < 0 || N < 0 || H < 1 || out_rows > INT32_MAX || N > INT32_MAX)
        return MP_ERR_INVALID_ARG;
    if ((in_probs == nullptr) != (out_probs == nullptr)) return MP_ERR_INVALID_ARG;
    if (out_rows == 0) return MP_OK;
    // scatter: in is [out_rows,H], out is [N,H]; gather: the other way round.
    const void *rows_side = scatter ? in : out;
    const void *n_side = scatter ? out : in;
    if (map == nullptr || rows_side == nullptr || (N > 0 && n_side == nullptr))
        return MP_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((out_rows + CH_ROWS - 1) / CH_ROWS);
    if (chunk_vec_ok(H, {in, out})) {
        if (scatter)
            k_rows_remap<uint4, true><<<blocks, CH_THREADS, 0, s>>>(
                (const uint4 *)in, in_probs, map, out_rows, N, H / 8, (uint4 *)out, out_probs, status);
        else
            k_rows_remap<uint4, false><<<blocks, CH_THREADS, 0, s>>>(
                (const uint4 *)in, in_probs, map, out_rows, N, H / 8, (uint4 *)out, out_probs, status);
    } else {
        if (scatter)
            k_rows_remap<uint16_t, true><<<blocks, CH_THREADS, 0, s>>>(
                (const uint16_t *)in, in_probs, map, out_rows, N, H, (uint16_t *)out, out_probs,
                status);
        else
            k_rows_remap<uint16_t, false><<<blocks, CH_THREADS, 0, s>>>(
                (const uint16_t *)in, in_probs, map, out_rows, N, H, (uint16_t *)out, out_probs,
                status);
    }
    return check_launch();
}

inline int elem_units(int32_t dtype)
{
    switch (dtype) {
    case MP_DTYPE_BF16:
    case MP_DTYPE_FP16: return 1;
    case MP_DTYPE_FP32: return 2;
    default: return 0;
    }
}

// Rows are W 16-bit units wide (H for 2-byte types, 2H for fp32).
mp_status_t sort_pad_impl(const void *x, const float *probs, const int32_t *split_sizes,
                          const int32_t *chunk_order, const int32_t *padded_sizes, int32_t C,
                          int32_t G, int32_t align, int64_t N, int64_t out_rows, int64_t W,
                          void *out, float *out_probs, int32_t *row_map, int64_t *group_off,
                          int32_t *dev_status, cudaStream_t s)
{
    if (C < 1 || G < 1 || align < 1 || N < 0 || out_rows < 0 || W < 1) return MP_ERR_INVALID_ARG;
    if (C % G != 0) return MP_ERR_INVALID_ARG;
    if (C > MP_MAX_CHUNKS || N > INT32_MAX || out_rows > INT32_MAX || W > INT32_MAX)
        return MP_ERR_UNSUPPORTED;
    if (split_sizes == nullptr || chunk_order == nullptr || group_off == nullptr)
        return MP_ERR_INVALID_ARG;
    if ((probs == nullptr) != (out_probs == nullptr)) return MP_ERR_INVALID_ARG;
    if (out_rows > 0 && (out == nullptr || row_map == nullptr)) return MP_ERR_INVALID_ARG;
    if (N > 0 && x == nullptr) return MP_ERR_INVALID_ARG;
    const unsigned blocks = out_rows > 0 ? (unsigned)((out_rows + CH_ROWS - 1) / CH_ROWS) : 1u;
    const size_t smem = sort_pad_smem(C, G);
    const int32_t w = (int32_t)W;
    if (chunk_vec_ok(w, {x, out}))
        k_sort_pad<uint4><<<blocks, CH_THREADS, smem, s>>>(
            (const uint4 *)x, probs, split_sizes, chunk_order, padded_sizes, C, G, align, N,
            out_rows, w / 8, (uint4 *)out, out_probs, row_map, group_off, dev_status);
    else
        k_sort_pad<uint16_t><<<blocks, CH_THREADS, smem, s>>>(
            (const uint16_t *)x, probs, split_sizes, chunk_order, padded_sizes, C, G, align, N,
            out_rows, w, (uint16_t *)out, out_probs, row_map, group_off, dev_status);
    return check_launch();
}

mp_status_t remap_ex(const void *in, int32_t dtype, const float *in_probs, const int32_t *map,
                     int64_t out_rows, int64_t N, int32_t H, void *out, float *out_probs,
                     int32_t *status, cudaStream_t s, bool scatter)
{
    const int u = elem_units(dtype);
    if (u == 0 || H < 1) return MP_ERR_INVALID_ARG;
    if ((int64_t)H * u > INT32_MAX) return MP_ERR_UNSUPPORTED;
    return remap(in, in_probs, map, out_rows, N, H * u, out, out_probs, status, s, scatter);
}

}  // namespace
}  // namespace mp

using namespace mp;

extern "C" mp_status_t mp_sort_chunks_pad(const mp_bf16_t *x, const float *probs,
                                          const int32_t *split_sizes, const int32_t *chunk_order,
                                          int32_t C, int32_t G, int32_t align, int64_t N,
                                          int64_t out_rows, int32_t H, mp_bf16_t *out,
                                          float *out_probs, int32_t *row_map, int64_t *group_off,
                                          int32_t *dev_status, mp_stream_t stream)
{
    if (H < 1) return MP_ERR_INVALID_ARG;
    return sort_pad_impl(x, probs, split_sizes, chunk_order, nullptr, C, G, align, N, out_rows, H,
                         out, out_probs, row_map, group_off, dev_status, as_stream(stream));
}

extern "C" mp_status_t mp_sort_chunks_pad_ex(const void *x, int32_t dtype, const float *probs,
                                             const int32_t *split_sizes,
                                             const int32_t *chunk_order,
                                             const int32_t *padded_sizes, int32_t C, int32_t G,
                                             int32_t align, int64_t N, int64_t out_rows, int32_t H,
                                             void *out, float *out_probs, int32_t *row_map,
                                             int64_t *group_off, int32_t *dev_status,
                                             mp_stream_t stream)
{
    const int u = elem_units(dtype);
    if (u == 0 || H < 1) return MP_ERR_INVALID_ARG;
    return sort_pad_impl(x, probs, split_sizes, chunk_order, padded_sizes, C, G, align, N,
                         out_rows, (int64_t)H * u, out, out_probs, row_map, group_off, dev_status,
                         as_stream(stream));
}

extern "C" mp_status_t mp_unpad_restore(const mp_bf16_t *padded, const float *padded_probs,
                                        const int32_t *row_map, int64_t out_rows, int64_t N,
                                        int32_t H, mp_bf16_t *y, float *y_probs,
                                        int32_t *dev_status, mp_stream_t stream)
{
    return remap(padded, padded_probs, row_map, out_rows, N, H, y, y_probs, dev_status,
                 as_stream(stream), true);
}

extern "C" mp_status_t mp_unpad_restore_ex(const void *padded, int32_t dtype,
                                           const float *padded_probs, const int32_t *row_map,
                                           int64_t out_rows, int64_t N, int32_t H, void *y,
                                           float *y_probs, int32_t *dev_status, mp_stream_t stream)
{
    return remap_ex(padded, dtype, padded_probs, row_map, out_rows, N, H, y, y_probs, dev_status,
                    as_stream(stream), true);
}

extern "C" mp_status_t mp_sort_chunks_pad_bwd(const mp_bf16_t *g_out, const float *g_out_probs,
                                              const int32_t *row_map, int64_t out_rows, int64_t N,
                                              int32_t H, mp_bf16_t *g_x, float *g_probs,
                                              int32_t *dev_status, mp_stream_t stream)
{
    return remap(g_out, g_out_probs, row_map, out_rows, N, H, g_x, g_probs, dev_status,
                 as_stream(stream), true);
}

extern "C" mp_status_t mp_sort_chunks_pad_bwd_ex(const void *g_out, int32_t dtype,
                                                 const float *g_out_probs, const int32_t *row_map,
                                                 int64_t out_rows, int64_t N, int32_t H, void *g_x,
                                                 float *g_probs, int32_t *dev_status,
                                                 mp_stream_t stream)
{
    return remap_ex(g_out, dtype, g_out_probs, row_map, out_rows, N, H, g_x, g_probs, dev_status,
                    as_stream(stream), true);
}

extern "C" mp_status_t mp_unpad_restore_bwd(const mp_bf16_t *g_y, const float *g_y_probs,
                                            const int32_t *row_map, int64_t out_rows, int64_t N,
                                            int32_t H, mp_bf16_t *g_padded, float *g_padded_probs,
                                            int32_t *dev_status, mp_stream_t stream)
{
    return remap(g_y, g_y_probs, row_map, out_rows, N, H, g_padded, g_padded_probs, dev_status,
                 as_stream(stream), false);
}

extern "C" mp_status_t mp_unpad_restore_bwd_ex(const void *g_y, int32_t dtype,
                                               const float *g_y_probs, const int32_t *row_map,
                                               int64_t out_rows, int64_t N, int32_t H,
                                               void *g_padded, float *g_padded_probs,
                                               int32_t *dev_status, mp_stream_t stream)
{
    return remap_ex(g_y, dtype, g_y_probs, row_map, out_rows, N, H, g_padded, g_padded_probs,
                    dev_status, as_stream(stream), false);
}
