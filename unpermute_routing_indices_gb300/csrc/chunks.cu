// Fused chunk sort + pad and its unpad + restore ("[PyTorch] Fuse MoE chunk
// sorting and padding", TransformerEngine PR 3509: one pass that copies the
// tokens and probabilities into expert order with zero padding, and one copy
// back through the saved row map).
//
//   k_sort_pad     one launch for map + copy.  Every CTA rebuilds the small
//                  chunk metadata in shared memory (C <= MP_MAX_CHUNKS sizes:
//                  input starts, output-order starts, group rows, padded group
//                  offsets) -- one warp with register-segment shuffle scans
//                  for up to 256 chunks in up to 32 groups, the whole CTA
//                  beyond -- then resolves the source row of each of its
//                  output rows (SP_ROWS per CTA; SP_SMALL_ROWS per smaller CTA
//                  for outputs of up to MP_SP_RP2_MAX_ROWS rows with one-warp
//                  metadata) by two binary searches and copies the rows (zero
//                  for padding).  CTA 0 also writes group_off and the status
//                  bits.  Nothing is carried between CTAs, so the grid depends
//                  on out_rows only and sizes are runtime data.
//   k_rows_remap   through a saved row map: out[d] = in[map[d]] or zero
//                  (gather: unpad+restore backward) or out[map[d]] = in[d]
//                  (scatter: unpad+restore and the sort+pad backward).
//   Rows of >= 32 vectors are copied one warp per row, lanes across the row.
#include "common.cuh"

namespace mp {
namespace {

#ifndef MP_CH_ROWS
#define MP_CH_ROWS 16
#endif
#ifndef MP_CH_UNROLL
#define MP_CH_UNROLL 8
#endif

#ifndef MP_CH_MIN_BLOCKS
#define MP_CH_MIN_BLOCKS 1
#endif
#ifndef MP_SP_RP2_MAX_ROWS
#define MP_SP_RP2_MAX_ROWS 16384
#endif
#ifndef MP_SP_ROWS
#define MP_SP_ROWS 32
#endif

constexpr int CH_THREADS = 256;
constexpr int CH_WARPS = CH_THREADS / 32;
constexpr int CH_ROWS = MP_CH_ROWS;      // output rows per CTA (restore kernels)
constexpr int SP_ROWS = MP_SP_ROWS;      // output rows per CTA (sort+pad)
#ifndef MP_SP_SMALL_THREADS
#define MP_SP_SMALL_THREADS 128
#endif
#ifndef MP_SP_SMALL_ROWS
#define MP_SP_SMALL_ROWS 16
#endif
constexpr int SP_SMALL_THREADS = MP_SP_SMALL_THREADS;  // sort+pad CTA, small outputs
constexpr int SP_SMALL_ROWS = MP_SP_SMALL_ROWS;
constexpr int CH_UNROLL = MP_CH_UNROLL;  // vectors in flight per thread

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
// Rows of at least 32 vectors go one warp per row, the lanes across the row
// (CH_UNROLL 16-byte vectors, or half as many 32-byte ones, in flight per
// lane, addresses by immediate offsets from the row base); narrower rows are
// spread over the CTA as one flat range.
template <typename V, bool SCATTER, int RP = 1, int THREADS = CH_THREADS>
__device__ __forceinline__ void copy_rows(const V *__restrict__ in, V *__restrict__ out,
                                          const int32_t *s_map, int64_t row0, int nrows, int nvec)
{
    // the same bytes in flight per lane for 16- and 32-byte vectors
    constexpr int UNR = sizeof(V) == 32 ? CH_UNROLL / 2 : CH_UNROLL;
    if (nvec >= 32) {
        // One warp per RP rows at a time: RP * UNR vectors in flight per lane.
        const int lane = threadIdx.x & 31;
        for (int r0 = (threadIdx.x >> 5) * RP; r0 < nrows; r0 += (THREADS / 32) * RP) {
            const V *src[RP];
            V *dst[RP];
            bool live[RP], zero[RP];
#pragma unroll
            for (int q = 0; q < RP; ++q) {
                const int r = r0 + q;
                const int32_t m = r < nrows ? s_map[r] : -1;
                live[q] = r < nrows && (!SCATTER || m >= 0);
                zero[q] = !SCATTER && m < 0;
                src[q] = in + (SCATTER ? row0 + r : (int64_t)(m < 0 ? 0 : m)) * nvec;
                dst[q] = out + (SCATTER ? (int64_t)(m < 0 ? 0 : m) : row0 + r) * nvec;
            }
            for (int c0 = lane; c0 < nvec; c0 += 32 * UNR) {
                V v[RP][UNR];
#pragma unroll
                for (int q = 0; q < RP; ++q)
#pragma unroll
                    for (int u = 0; u < UNR; ++u) {
                        const int c = c0 + 32 * u;
                        v[q][u] = (live[q] && !zero[q] && c < nvec) ? ld_stream(src[q] + c)
                                                                     : zero_vec<V>();
                    }
#pragma unroll
                for (int q = 0; q < RP; ++q)
#pragma unroll
                    for (int u = 0; u < UNR; ++u) {
                        const int c = c0 + 32 * u;
                        if (live[q] && c < nvec) st_row(dst[q] + c, v[q][u]);
                    }
            }
        }
        return;
    }
    const int total = nrows * nvec;
    for (int w0 = 0; w0 < total; w0 += THREADS * UNR) {
        V v[UNR];
        int64_t dst_off[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int w = w0 + u * THREADS + threadIdx.x;
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
        for (int u = 0; u < UNR; ++u)
            if (dst_off[u] >= 0) st_row(out + dst_off[u], v[u]);
    }
}

// The chunk metadata of sort+pad, in shared memory:
//   s_start[c]  first input row of chunk c (exclusive scan of the sizes)
//   s_chunk[p]  the chunk at output position p (-1 if out of range)
//   s_cum[p]    rows before position p in output order; s_cum[C] = all
//   s_grows[g]  unpadded rows of group g;  s_goff[g] its padded offset,
//               s_goff[G] = the padded total
// CTA 0 also writes group_off and the status bits.  Built by one warp (WARP,
// few chunks: no CTA barrier inside) or by the whole CTA.
struct SortPadMeta {
    int64_t *s_start, *s_cum, *s_goff, *s_grows, *s_warp;
    int32_t *s_chunk;
};

__device__ __forceinline__ int sort_pad_group_rows(const SortPadMeta &m, int g, int per_group,
                                                   int align, const int32_t *padded_sizes)
{
    const int64_t rows = m.s_cum[(g + 1) * per_group] - m.s_cum[g * per_group];
    m.s_grows[g] = rows;
    int64_t padded = (rows + align - 1) / align * align;
    int flags = 0;
    if (padded_sizes != nullptr) {   // explicit padded sizes (loaded into s_goff first)
        const int64_t ps = m.s_goff[g];
        padded = ps < 0 ? 0 : ps;
        if (padded < rows) flags = MP_STATUS_BAD_PADDED;
    }
    m.s_goff[g] = padded;
    return flags;
}

// Inclusive warp scan of a 64-bit value (5 shuffle steps of two words each).
__device__ __forceinline__ int64_t warp_inclusive_scan64(int64_t v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(FULL_MASK, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// The metadata built by one warp, for C <= 256 and G <= 32, with a short
// dependency chain: lane l owns the q = ceil(C/32) consecutive chunk
// positions [l*q, l*q + q), sums them in registers, and the input-order and
// output-order scans are two independent 5-step warp scans (interleaved by
// the compiler) instead of rounds of 32.  The group offsets are one more
// warp scan (lane g holds group g).
constexpr int SP_FAST_META_MAX_Q = 8;   // C <= 256
__device__ void sort_pad_meta_fast(const SortPadMeta &m, const int32_t *split,
                                   const int32_t *order, const int32_t *padded_sizes, int C,
                                   int G, int align, int64_t N, int64_t out_rows,
                                   int64_t *group_off, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int q = (C + 31) >> 5;
    const int lo = lane * q;
    int flags = 0;
    int32_t sz[SP_FAST_META_MAX_Q], od[SP_FAST_META_MAX_Q];
#pragma unroll
    for (int j = 0; j < SP_FAST_META_MAX_Q; ++j) {   // every metadata load issued together
        const int c = lo + j;
        const bool in = j < q && c < C;
        sz[j] = in ? split[c] : 0;
        od[j] = in ? order[c] : -1;
    }
    const int32_t ps = (padded_sizes != nullptr && lane < G) ? padded_sizes[lane] : 0;
    int64_t sum_in = 0;
#pragma unroll
    for (int j = 0; j < SP_FAST_META_MAX_Q; ++j) {
        const int c = lo + j;
        if (j < q && c < C) {
            if (sz[j] < 0) { flags |= MP_STATUS_BAD_SPLIT; sz[j] = 0; }
            m.s_start[c] = sz[j];                    // sizes by chunk id, for the gather
            const bool ok = od[j] >= 0 && od[j] < C;
            if (!ok) { flags |= MP_STATUS_BAD_ORDER; od[j] = -1; }
            m.s_chunk[c] = od[j];
            sum_in += sz[j];
        }
    }
    __syncwarp();
    int64_t so[SP_FAST_META_MAX_Q];
    int64_t sum_out = 0;
#pragma unroll
    for (int j = 0; j < SP_FAST_META_MAX_Q; ++j) {   // size of the chunk at position lo + j
        so[j] = (j < q && lo + j < C && od[j] >= 0) ? m.s_start[od[j]] : 0;
        sum_out += so[j];
    }
    __syncwarp();                                    // every gather done before the overwrite
    const int64_t inc_in = warp_inclusive_scan64(sum_in);
    const int64_t inc_out = warp_inclusive_scan64(sum_out);
    int64_t run_in = inc_in - sum_in, run_out = inc_out - sum_out;
#pragma unroll
    for (int j = 0; j < SP_FAST_META_MAX_Q; ++j) {
        const int c = lo + j;
        if (j < q && c < C) {
            m.s_start[c] = run_in;
            m.s_cum[c] = run_out;
            run_in += sz[j];
            run_out += so[j];
        }
    }
    const int64_t total_in = __shfl_sync(FULL_MASK, inc_in, 31);
    const int64_t total_ord = __shfl_sync(FULL_MASK, inc_out, 31);
    if (lane == 0) m.s_cum[C] = total_ord;
    __syncwarp();
    const int per_group = C / G;
    int64_t padded = 0;
    if (lane < G) {
        const int64_t rows = m.s_cum[(lane + 1) * per_group] - m.s_cum[lane * per_group];
        m.s_grows[lane] = rows;
        padded = (rows + align - 1) / align * align;
        if (padded_sizes != nullptr) {
            padded = ps < 0 ? 0 : ps;
            if (padded < rows) flags |= MP_STATUS_BAD_PADDED;
        }
    }
    const int64_t inc_pad = warp_inclusive_scan64(padded);
    if (lane < G) m.s_goff[lane] = inc_pad - padded;
    const int64_t total_pad = __shfl_sync(FULL_MASK, inc_pad, 31);
    if (lane == 0) m.s_goff[G] = total_pad;
    flags = __reduce_or_sync(FULL_MASK, flags);
    __syncwarp();
    if (blockIdx.x == 0) {
        for (int g = lane; g <= G; g += 32) group_off[g] = m.s_goff[g];
        if (lane == 0) {
            if (total_in > N) flags |= MP_STATUS_SPLIT_OVERFLOW;
            if (total_pad > out_rows) flags |= MP_STATUS_ROWS_OVERFLOW;
            or_status(status, flags);
        }
    }
}

__device__ void sort_pad_meta_cta(const SortPadMeta &m, const int32_t *split,
                                  const int32_t *order, const int32_t *padded_sizes, int C,
                                  int G, int align, int64_t N, int64_t out_rows,
                                  int64_t *group_off, int32_t *status, int *s_flags)
{
    const int tid = threadIdx.x;
    if (tid == 0) *s_flags = 0;
    int flags = 0;
    for (int c = tid; c < C; c += CH_THREADS) {   // every metadata load issued together
        int64_t v = split[c];
        m.s_chunk[c] = order[c];
        if (v < 0) { flags |= MP_STATUS_BAD_SPLIT; v = 0; }
        m.s_start[c] = v;
    }
    if (padded_sizes != nullptr)
        for (int g = tid; g < G; g += CH_THREADS) m.s_goff[g] = padded_sizes[g];
    __syncthreads();
    const int64_t total_in = cta_exclusive_scan(m.s_start, C, m.s_warp);
    for (int p = tid; p < C; p += CH_THREADS) {
        const int32_t c = m.s_chunk[p];
        const bool ok = c >= 0 && c < C;
        if (!ok) flags |= MP_STATUS_BAD_ORDER;
        m.s_chunk[p] = ok ? c : -1;
        m.s_cum[p] = ok ? ((c + 1 < C ? m.s_start[c + 1] : total_in) - m.s_start[c]) : 0;
    }
    __syncthreads();
    const int64_t total_ord = cta_exclusive_scan(m.s_cum, C, m.s_warp);
    if (tid == 0) m.s_cum[C] = total_ord;
    __syncthreads();
    const int per_group = C / G;
    for (int g = tid; g < G; g += CH_THREADS)
        flags |= sort_pad_group_rows(m, g, per_group, align, padded_sizes);
    if (flags) atomicOr(s_flags, flags);
    __syncthreads();
    const int64_t total_pad = cta_exclusive_scan(m.s_goff, G, m.s_warp);
    if (tid == 0) m.s_goff[G] = total_pad;
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int g = tid; g <= G; g += CH_THREADS) group_off[g] = m.s_goff[g];
        if (tid == 0) {
            int bits = *s_flags;
            if (total_in > N) bits |= MP_STATUS_SPLIT_OVERFLOW;
            if (total_pad > out_rows) bits |= MP_STATUS_ROWS_OVERFLOW;
            or_status(status, bits);
        }
    }
}

template <typename V, bool FAST_META, int RP, int THREADS, int ROWS>
__global__ void __launch_bounds__(THREADS, MP_CH_MIN_BLOCKS)
    k_sort_pad(const V *__restrict__ x, const float *__restrict__ probs,
               const int32_t *__restrict__ split, const int32_t *__restrict__ order,
               const int32_t *__restrict__ padded_sizes, int C, int G,
               int align, int64_t N, int64_t out_rows, int nvec, V *__restrict__ out,
               float *__restrict__ out_probs, int32_t *__restrict__ row_map,
               int64_t *__restrict__ group_off, int32_t *status)
{
    pdl_trigger();
    pdl_wait();
    extern __shared__ int64_t sm[];
    SortPadMeta m;
    m.s_start = sm;                      // [C]
    m.s_cum = m.s_start + C;             // [C+1]
    m.s_goff = m.s_cum + C + 1;          // [G+1]
    m.s_grows = m.s_goff + G + 1;        // [G]
    m.s_warp = m.s_grows + G;            // [CH_WARPS]
    m.s_chunk = reinterpret_cast<int32_t *>(m.s_warp + CH_WARPS);  // [C]
    int32_t *s_src = m.s_chunk + C;      // [ROWS]
    __shared__ int s_flags;
    // The whole-CTA metadata and the row resolve assume these shapes.
    static_assert(FAST_META || THREADS == CH_THREADS, "CTA metadata needs CH_THREADS threads");
    static_assert(ROWS <= THREADS && THREADS % 32 == 0, "one thread resolves each row");

    const int tid = threadIdx.x;
    if (FAST_META) {
        if (tid < 32)
            sort_pad_meta_fast(m, split, order, padded_sizes, C, G, align, N, out_rows,
                               group_off, status);
        __syncthreads();
    } else {
        sort_pad_meta_cta(m, split, order, padded_sizes, C, G, align, N, out_rows, group_off,
                          status, &s_flags);
    }
    const int64_t total_pad = m.s_goff[G];
    const int per_group = C / G;

    const int64_t row0 = (int64_t)blockIdx.x * ROWS;
    const int64_t left = out_rows - row0;
    const int nrows = left < ROWS ? (int)left : ROWS;
    float pv = 0.0f;   // this row's prob: loaded now, stored after the copy
    if (tid < nrows) {
        const int64_t d = row0 + tid;
        int32_t src = -1;
        if (d < total_pad) {
            const int g = last_le(m.s_goff, 0, G, d);
            const int64_t j = d - m.s_goff[g];
            if (j < m.s_grows[g]) {
                const int64_t target = m.s_cum[g * per_group] + j;
                const int p = last_le(m.s_cum, g * per_group, (g + 1) * per_group, target);
                const int64_t s = m.s_start[m.s_chunk[p]] + (target - m.s_cum[p]);
                src = s < N ? (int32_t)s : -1;
            }
        }
        s_src[tid] = src;
        row_map[d] = src;
        if (out_probs != nullptr && src >= 0) pv = __ldg(probs + src);
    }
    __syncthreads();
    if (nrows > 0) copy_rows<V, false, RP, THREADS>(x, out, s_src, row0, nrows, nvec);
    if (out_probs != nullptr && tid < nrows) out_probs[row0 + tid] = pv;
}

template <typename V, bool SCATTER>
__global__ void __launch_bounds__(CH_THREADS, MP_CH_MIN_BLOCKS)
    k_rows_remap(const V *__restrict__ in, const float *__restrict__ in_probs,
                 const int32_t *__restrict__ map, int64_t out_rows, int64_t N, int nvec,
                 V *__restrict__ out, float *__restrict__ out_probs, int32_t *status)
{
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t s_map[CH_ROWS];
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * CH_ROWS;
    const int64_t left = out_rows - row0;
    const int nrows = left < CH_ROWS ? (int)left : CH_ROWS;
    // The row's prob is loaded before the copy and stored after it, so its
    // latency does not hold the CTA at the barrier.
    float pv = 0.0f;
    int32_t m = -1;
    if (tid < nrows) {
        const int64_t d = row0 + tid;
        if (SCATTER && in_probs != nullptr) pv = __ldg(in_probs + d);
        m = __ldg(map + d);
        if (m < -1 || m >= N) {
            or_status(status, MP_STATUS_BAD_ROW);
            m = -1;
        }
        s_map[tid] = m;
        if (!SCATTER && in_probs != nullptr && m >= 0) pv = __ldg(in_probs + m);
    }
    __syncthreads();
    copy_rows<V, SCATTER>(in, out, s_map, row0, nrows, nvec);
    if (in_probs != nullptr && tid < nrows) {
        if (SCATTER) {
            if (m >= 0) out_probs[m] = pv;
        } else {
            out_probs[row0 + tid] = pv;
        }
    }
}

inline bool chunk_vec_ok(int32_t H, std::initializer_list<const void *> ptrs)
{
    if (H % 8 != 0) return false;
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p)) return false;
    return true;
}

inline size_t sort_pad_smem(int C, int G, int rows)
{
    return sizeof(int64_t) * (size_t)(C + (C + 1) + (G + 1) + G + CH_WARPS) +
           sizeof(int32_t) * (size_t)(C + rows);
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
            (void)launch_pdl(k_rows_remap<uint4, true>, blocks, CH_THREADS, 0, s,
                             (const uint4 *)in, in_probs, map, out_rows, N, H / 8, (uint4 *)out,
                             out_probs, status);
        else
            (void)launch_pdl(k_rows_remap<uint4, false>, blocks, CH_THREADS, 0, s,
                             (const uint4 *)in, in_probs, map, out_rows, N, H / 8, (uint4 *)out,
                             out_probs, status);
    } else {
        if (scatter)
            (void)launch_pdl(k_rows_remap<uint16_t, true>, blocks, CH_THREADS, 0, s,
                             (const uint16_t *)in, in_probs, map, out_rows, N, H, (uint16_t *)out,
                             out_probs, status);
        else
            (void)launch_pdl(k_rows_remap<uint16_t, false>, blocks, CH_THREADS, 0, s,
                             (const uint16_t *)in, in_probs, map, out_rows, N, H, (uint16_t *)out,
                             out_probs, status);
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
    const int32_t w = (int32_t)W;
    const bool fast_meta = C <= 32 * SP_FAST_META_MAX_Q && G <= 32;
    const bool vec = chunk_vec_ok(w, {x, out});
    // Small outputs (about one wave of CTAs) keep two rows per warp in
    // flight; larger ones keep one, for more resident CTAs.  Small outputs
    // whose metadata one warp builds run in CTAs of SP_SMALL_THREADS threads
    // and SP_SMALL_ROWS rows, so that the grid is one wave.
    const bool two = out_rows <= MP_SP_RP2_MAX_ROWS;
#define MP_SORT_PAD_LAUNCH(VT, FM, RPV, TH, RW, NV)                                           \
    (void)launch_pdl(k_sort_pad<VT, FM, RPV, TH, RW>,                                        \
                     out_rows > 0 ? (unsigned)((out_rows + RW - 1) / RW) : 1u, TH,           \
                     sort_pad_smem(C, G, RW), s, (const VT *)x, probs, split_sizes,          \
                     chunk_order, padded_sizes, C, G, align, N, out_rows, NV, (VT *)out,     \
                     out_probs, row_map, group_off, dev_status)
    // Outputs past the two-rows-in-flight size, 32-byte aligned with rows of
    // at least 32 32-byte vectors, copy 32-byte vectors: half the load and
    // store instructions (32,768 rows of 2,048 bf16: 43.5 -> 42.65 us; at
    // 8,192 rows no change, and unpad+restore was slower with them).
    const bool vec32 = vec && !two && w % 16 == 0 && w / 16 >= 32 && aligned32(x) &&
                       aligned32(out);
    if (vec32) {
        if (fast_meta) MP_SORT_PAD_LAUNCH(u32x8, true, 1, CH_THREADS, SP_ROWS, w / 16);
        else MP_SORT_PAD_LAUNCH(u32x8, false, 1, CH_THREADS, SP_ROWS, w / 16);
    } else if (vec) {
        if (fast_meta && two)
            MP_SORT_PAD_LAUNCH(uint4, true, 2, SP_SMALL_THREADS, SP_SMALL_ROWS, w / 8);
        else if (fast_meta) MP_SORT_PAD_LAUNCH(uint4, true, 1, CH_THREADS, SP_ROWS, w / 8);
        else if (two) MP_SORT_PAD_LAUNCH(uint4, false, 2, CH_THREADS, SP_ROWS, w / 8);
        else MP_SORT_PAD_LAUNCH(uint4, false, 1, CH_THREADS, SP_ROWS, w / 8);
    } else {
        if (fast_meta) MP_SORT_PAD_LAUNCH(uint16_t, true, 1, CH_THREADS, SP_ROWS, w);
        else MP_SORT_PAD_LAUNCH(uint16_t, false, 1, CH_THREADS, SP_ROWS, w);
    }
#undef MP_SORT_PAD_LAUNCH
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
