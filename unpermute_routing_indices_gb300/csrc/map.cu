// Routing map: histogram -> exclusive scan -> stable rank.
//
// A counting sort of the T*K routes by expert, the "counting sort ... block
// histogram + exclusive prefix sums, O(N)" of the moe-ops README ("Why this
// library"), producing the forward map (t,k) -> row of the xtuner issue
// "permute different with torch version" and the row order of the worked
// example in make_row_id_map (d9d / TransformerEngine permutation.py):
// expert-major, tokens ascending, slots ascending.
//
// Three launches, no atomics whose order reaches the result:
//   k_map_count  one CTA per tile of MAP_TILE routes: per-tile histogram over
//                E+1 buckets (bucket E collects empty and bad slots), stored
//                expert-major as tile_counts[b][tile].
//   k_map_scan   one CTA: exclusive scan of tile_counts in expert-major order.
//                Entry [b][tile] becomes the first row of bucket b's routes in
//                that tile; [b][0] is offsets[b], and [E][0] the routed total.
//   k_map_rank   one CTA per tile: each warp walks 8 chunks of 32 consecutive
//                routes; __match_any_sync groups the lanes of one expert and
//                popc(peers & lanemask_lt) is the stable rank inside the chunk.
//                Per-warp counters, seeded by a scan across the CTA's warps
//                from the tile base, carry the rank from chunk to chunk.
#include <mutex>

#include "common.cuh"

namespace mp {

namespace {
thread_local int32_t g_last_cuda_error = 0;
}

void set_last_cuda_error(cudaError_t err) { g_last_cuda_error = static_cast<int32_t>(err); }

namespace {

constexpr int MAP_THREADS = 256;
constexpr int MAP_WARPS = MAP_THREADS / 32;
constexpr int MAP_CHUNKS = 8;                          // 32-route chunks per warp
constexpr int MAP_TILE = MAP_WARPS * MAP_CHUNKS * 32;  // 2048 routes per tile
constexpr int SCAN_THREADS = 1024;
constexpr int SCAN_ITEMS = 8;                          // per thread and pass
constexpr int SCAN_PASS = SCAN_THREADS * SCAN_ITEMS;

__device__ __forceinline__ int bucket_of(int32_t v, int E) { return (v >= 0 && v < E) ? v : E; }

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Buckets of this lane's 8 routes; -1 past the end.
__device__ __forceinline__ void load_buckets(const int32_t *__restrict__ idx, int64_t n, int E,
                                             int64_t base, int lane, int (&bk)[MAP_CHUNKS],
                                             bool &bad)
{
#pragma unroll
    for (int c = 0; c < MAP_CHUNKS; ++c) {
        const int64_t i = base + c * 32 + lane;
        int32_t v = -1;
        if (i < n) v = __ldg(idx + i);
        bk[c] = (i < n) ? bucket_of(v, E) : -1;
        bad |= (i < n) && v != -1 && bk[c] == E;
    }
}

__global__ void __launch_bounds__(MAP_THREADS)
    k_map_count(const int32_t *__restrict__ idx, int64_t n, int E, int ntiles,
                int32_t *__restrict__ tile_counts, int32_t *status)
{
    extern __shared__ int32_t s_hist[];  // [E+1]
    for (int b = threadIdx.x; b <= E; b += MAP_THREADS) s_hist[b] = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = (int64_t)blockIdx.x * MAP_TILE + warp * (MAP_CHUNKS * 32);
    int bk[MAP_CHUNKS];
    bool bad = false;
    load_buckets(idx, n, E, base, lane, bk, bad);
#pragma unroll
    for (int c = 0; c < MAP_CHUNKS; ++c) {
        const unsigned peers = __match_any_sync(FULL_MASK, bk[c]);
        if (bk[c] >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bk[c]], __popc(peers));
    }
    if (__any_sync(FULL_MASK, bad) && lane == 0) or_status(status, MP_STATUS_BAD_EXPERT);
    __syncthreads();
    for (int b = threadIdx.x; b <= E; b += MAP_THREADS)
        tile_counts[(int64_t)b * ntiles + blockIdx.x] = s_hist[b];
}

// Padded shared-memory index: one spare word per 32 keeps both the coalesced
// (stride 1) and the per-thread segment (stride SCAN_ITEMS) accesses free of
// bank conflicts.
__device__ __forceinline__ int spad(int i) { return i + (i >> 5); }

__global__ void __launch_bounds__(SCAN_THREADS)
    k_map_scan(int32_t *__restrict__ tile_counts, int E, int ntiles, int32_t *__restrict__ counts,
               int32_t *__restrict__ offsets)
{
    __shared__ int32_t s_val[SCAN_PASS + SCAN_PASS / 32];
    __shared__ int32_t s_warp[SCAN_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t M = (int64_t)(E + 1) * ntiles;
    int32_t carry = 0;

    for (int64_t base = 0; base < M; base += SCAN_PASS) {
#pragma unroll
        for (int j = 0; j < SCAN_ITEMS; ++j) {
            const int i = j * SCAN_THREADS + tid;
            s_val[spad(i)] = (base + i < M) ? tile_counts[base + i] : 0;
        }
        __syncthreads();

        int32_t v[SCAN_ITEMS];
        int32_t sum = 0;
#pragma unroll
        for (int j = 0; j < SCAN_ITEMS; ++j) {
            v[j] = s_val[spad(tid * SCAN_ITEMS + j)];
            sum += v[j];
        }
        int32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int32_t w = s_warp[lane];
            int32_t wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(FULL_MASK, wi, o);
                if (lane >= o) wi += y;
            }
            s_warp[lane] = wi - w;  // exclusive prefix of warp totals
        }
        __syncthreads();
        int32_t run = carry + s_warp[warp] + incl - sum;
#pragma unroll
        for (int j = 0; j < SCAN_ITEMS; ++j) {
            s_val[spad(tid * SCAN_ITEMS + j)] = run;
            run += v[j];
        }
        // every thread learns the pass total from the last thread's prefix
        __syncthreads();
        const int32_t last = s_val[spad(SCAN_PASS - 1)];
#pragma unroll
        for (int j = 0; j < SCAN_ITEMS; ++j) {
            const int i = j * SCAN_THREADS + tid;
            if (base + i < M) tile_counts[base + i] = s_val[spad(i)];
        }
        // the last element's own count is still in the owning thread's v[]
        if (tid == SCAN_THREADS - 1) s_warp[0] = last + v[SCAN_ITEMS - 1];
        __syncthreads();
        carry = s_warp[0];
        __syncthreads();
    }

    for (int e = tid; e <= E; e += SCAN_THREADS) {
        const int32_t start = ntiles > 0 ? tile_counts[(int64_t)e * ntiles] : 0;
        offsets[e] = start;
        if (e < E) {
            const int32_t next = ntiles > 0 ? tile_counts[(int64_t)(e + 1) * ntiles] : 0;
            counts[e] = next - start;
        }
    }
}

__global__ void __launch_bounds__(MAP_THREADS)
    k_map_rank(const int32_t *__restrict__ idx, int64_t n, int E, int ntiles,
               const int32_t *__restrict__ bases, int32_t *__restrict__ row_id_map,
               int32_t *__restrict__ sorted_to_flat)
{
    extern __shared__ int32_t s_cnt[];  // [MAP_WARPS][E+1]
    const int stride = E + 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t *mine = s_cnt + warp * stride;
    for (int b = threadIdx.x; b < MAP_WARPS * stride; b += MAP_THREADS) s_cnt[b] = 0;
    __syncthreads();

    const int64_t base = (int64_t)blockIdx.x * MAP_TILE + warp * (MAP_CHUNKS * 32);
    int bk[MAP_CHUNKS];
    bool bad = false;
    load_buckets(idx, n, E, base, lane, bk, bad);
    unsigned peers[MAP_CHUNKS];
#pragma unroll
    for (int c = 0; c < MAP_CHUNKS; ++c) {
        peers[c] = __match_any_sync(FULL_MASK, bk[c]);
        if (bk[c] >= 0 && lane == __ffs(peers[c]) - 1) mine[bk[c]] += __popc(peers[c]);
        __syncwarp();
    }
    __syncthreads();

    // Per bucket: exclusive scan over the warps, seeded with the tile's base row.
    for (int b = threadIdx.x; b <= E; b += MAP_THREADS) {
        int32_t run = bases[(int64_t)b * ntiles + blockIdx.x];
#pragma unroll
        for (int w = 0; w < MAP_WARPS; ++w) {
            const int32_t c = s_cnt[w * stride + b];
            s_cnt[w * stride + b] = run;
            run += c;
        }
    }
    __syncthreads();

    const unsigned lt = lanemask_lt();
#pragma unroll
    for (int c = 0; c < MAP_CHUNKS; ++c) {
        const int b = bk[c];
        int32_t row = 0;
        if (b >= 0) row = mine[b] + __popc(peers[c] & lt);
        __syncwarp();
        if (b >= 0 && lane == __ffs(peers[c]) - 1) mine[b] += __popc(peers[c]);
        __syncwarp();
        if (b >= 0) {
            const int64_t i = base + c * 32 + lane;
            const bool routed = b < E;
            row_id_map[i] = routed ? row : -1;
            if (sorted_to_flat != nullptr) sorted_to_flat[row] = routed ? (int32_t)i : -1;
        }
    }
}

inline int64_t map_tiles(int64_t n) { return (n + MAP_TILE - 1) / MAP_TILE; }

inline bool map_sizes_ok(int64_t T, int32_t K, int32_t E)
{
    return T >= 0 && K >= 1 && E >= 1 && E <= MP_MAX_EXPERTS && T * (int64_t)K <= INT32_MAX;
}

}  // namespace
}  // namespace mp

using namespace mp;

extern "C" const char *mp_status_string(mp_status_t s)
{
    switch (s) {
    case MP_OK: return "ok";
    case MP_ERR_INVALID_ARG: return "invalid argument";
    case MP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MP_ERR_UNSUPPORTED: return "size beyond a documented limit";
    case MP_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
    }
}

extern "C" int32_t mp_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" size_t mp_build_map_workspace_size(int64_t T, int32_t K, int32_t E)
{
    if (!map_sizes_ok(T, K, E)) return 0;
    const int64_t ntiles = map_tiles(T * (int64_t)K);
    const size_t bytes = (size_t)(E + 1) * (size_t)ntiles * sizeof(int32_t);
    return bytes == 0 ? 256 : (bytes + 255) / 256 * 256;
}

extern "C" mp_status_t mp_build_map(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                                    int32_t *row_id_map, int32_t *sorted_to_flat,
                                    int32_t *counts, int32_t *offsets, void *workspace,
                                    size_t workspace_bytes, int32_t *dev_status,
                                    mp_stream_t stream)
{
    if (T < 0 || K < 1 || E < 1) return MP_ERR_INVALID_ARG;
    if (!map_sizes_ok(T, K, E)) return MP_ERR_UNSUPPORTED;
    if (counts == nullptr || offsets == nullptr) return MP_ERR_INVALID_ARG;
    const int64_t n = T * (int64_t)K;
    if (n > 0 && (idx == nullptr || row_id_map == nullptr)) return MP_ERR_INVALID_ARG;
    const int64_t ntiles = map_tiles(n);
    int32_t *tile_counts = static_cast<int32_t *>(workspace);
    if (ntiles > 0) {
        const size_t need = mp_build_map_workspace_size(T, K, E);
        if (workspace == nullptr || workspace_bytes < need ||
            (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
            return MP_ERR_WORKSPACE;
    }
    cudaStream_t s = as_stream(stream);
    if (ntiles > 0)
        k_map_count<<<(unsigned)ntiles, MAP_THREADS, (E + 1) * sizeof(int32_t), s>>>(
            idx, n, E, (int)ntiles, tile_counts, dev_status);
    k_map_scan<<<1, SCAN_THREADS, 0, s>>>(tile_counts, E, (int)ntiles, counts, offsets);
    if (ntiles > 0)
        k_map_rank<<<(unsigned)ntiles, MAP_THREADS, MAP_WARPS * (E + 1) * sizeof(int32_t), s>>>(
            idx, n, E, (int)ntiles, tile_counts, row_id_map, sorted_to_flat);
    return check_launch();
}

// ---------------------------------------------------------------------------
// Allocation-free routing map: the same three launches as mp_build_map, with
// the tile counts in a static device array owned by the library, for callers
// that cannot allocate device memory.
// ---------------------------------------------------------------------------

namespace mp {

constexpr int NOALLOC_SCRATCH_INTS = MP_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);

// One copy per GPU that loads the library, held until the process exits.
static __device__ __align__(256) int32_t g_map_scratch[NOALLOC_SCRATCH_INTS];

namespace {
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_scratch_mutex;
int32_t *g_scratch_addr[NOALLOC_MAX_DEVICES] = {};

// Device address of g_map_scratch on the current device.  The host-side name
// is only a stand-in, so the address is looked up once per device (with that
// device current) and cached.
mp_status_t scratch_on_current_device(int32_t **addr)
{
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        set_last_cuda_error(err);
        return MP_ERR_CUDA;
    }
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return MP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_map_scratch);
        if (err != cudaSuccess || p == nullptr) {
            set_last_cuda_error(err);
            return MP_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<int32_t *>(p);
    }
    *addr = g_scratch_addr[dev];
    return MP_OK;
}
}  // namespace
}  // namespace mp

extern "C" mp_status_t mp_build_map_noalloc(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                                            int32_t *row_id_map, int32_t *sorted_to_flat,
                                            int32_t *counts, int32_t *offsets,
                                            int32_t *dev_status, mp_stream_t stream)
{
    if (T < 0 || K < 1 || E < 1) return MP_ERR_INVALID_ARG;
    if (!map_sizes_ok(T, K, E)) return MP_ERR_UNSUPPORTED;
    if (counts == nullptr || offsets == nullptr) return MP_ERR_INVALID_ARG;
    const int64_t n = T * (int64_t)K;
    if (n > 0 && (idx == nullptr || row_id_map == nullptr)) return MP_ERR_INVALID_ARG;
    const int64_t ntiles = map_tiles(n);
    if ((int64_t)(E + 1) * ntiles > NOALLOC_SCRATCH_INTS) return MP_ERR_UNSUPPORTED;
    int32_t *tile_counts = nullptr;
    const mp_status_t st = scratch_on_current_device(&tile_counts);
    if (st != MP_OK) return st;
    // Every tile count the scan and rank kernels read is first written by
    // k_map_count in this call, so the array needs no clearing.
    cudaStream_t s = as_stream(stream);
    if (ntiles > 0)
        k_map_count<<<(unsigned)ntiles, MAP_THREADS, (E + 1) * sizeof(int32_t), s>>>(
            idx, n, E, (int)ntiles, tile_counts, dev_status);
    k_map_scan<<<1, SCAN_THREADS, 0, s>>>(tile_counts, E, (int)ntiles, counts, offsets);
    if (ntiles > 0)
        k_map_rank<<<(unsigned)ntiles, MAP_THREADS, MAP_WARPS * (E + 1) * sizeof(int32_t), s>>>(
            idx, n, E, (int)ntiles, tile_counts, row_id_map, sorted_to_flat);
    return check_launch();
}
