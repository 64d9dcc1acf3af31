// Routing map: histogram -> exclusive scan -> stable rank.
//
// A counting sort of the T*K routes by expert, the "counting sort ... block
// histogram + exclusive prefix sums, O(N)" of the moe-ops README ("Why this
// library"), producing the forward map (t,k) -> row of the xtuner issue
// "permute different with torch version" and the row order of the worked
// example in make_row_id_map (d9d / TransformerEngine permutation.py):
// expert-major, tokens ascending, slots ascending.
//
// The routes are cut into tiles of 2048*f consecutive routes (f, a power of
// two up to 8, keeps the tile count near 64).  Inside a tile (16 warps), warp
// w owns the contiguous range [w*128f, (w+1)*128f) and walks it in chunks of
// 32 routes (more warps with shorter walks: the map is latency-bound):
// __match_any_sync groups the lanes that name one expert, and
// popc(peers & lanemask_lt) is a lane's stable rank inside the chunk.
//
//   k_map_count  one CTA per tile: per-tile histogram over E+1 buckets
//                (bucket E collects empty and bad slots, so sorted_to_flat is
//                written in full), stored expert-major as tile_counts[b][tile].
//   k_map_rank   one CTA per tile.  Before it needs the counts it builds its
//                per-warp histograms from idx alone; launched as a
//                programmatic dependent of k_map_count, that part overlaps
//                the count kernel.  It then waits for the tile counts, derives
//                for every bucket the routes in earlier tiles and the total
//                (the exclusive scan, done redundantly by every CTA with warp
//                reductions over the count matrix in L2), seeds per-warp
//                counters with a scan across its warps, and ranks its routes:
//                a route's rank within its expert, below the expert's
//                capacity, gives row = offsets[e] + rank, else the route is
//                dropped (-1).  For tiles of up to two warp groups the first
//                pass keeps each route's bucket and in-warp rank in
//                registers; larger tiles walk their routes again.  CTA 0
//                writes counts and offsets.
// When the count matrix is large (every rank CTA would read too much), a single-CTA
// k_map_scan turns it into bases first and k_map_rank reads them (3 launches).
// Maps of at most 4,096 routes take one launch: a single k_map_rank CTA whose
// per-warp histograms are the whole count (no count kernel, no dependency).
// Maps of up to 32,768 routes take one launch of one thread-block cluster of
// k_map_rank CTAs (a 2,048-route tile each) that exchange their tile
// histograms through distributed shared memory.
// No atomics whose order reaches the result: the map is deterministic.
#include <mutex>

#include "common.cuh"

namespace mp {

namespace {
thread_local int32_t g_last_cuda_error = 0;
}

void set_last_cuda_error(cudaError_t err) { g_last_cuda_error = static_cast<int32_t>(err); }

namespace {

#ifndef MP_MAP_THREADS
#define MP_MAP_THREADS 512
#endif
#ifndef MP_MAP_CHUNKS
#define MP_MAP_CHUNKS 4
#endif

constexpr int MAP_THREADS = MP_MAP_THREADS;
constexpr int MAP_WARPS = MAP_THREADS / 32;
constexpr int MAP_CHUNKS = MP_MAP_CHUNKS;              // 32-route chunks per warp group
constexpr int MAP_GROUP = MAP_CHUNKS * 32;             // 128 routes per warp group
constexpr int MAP_SUB = MAP_WARPS * MAP_GROUP;         // 2048 routes: a tile with f = 1
#ifndef MP_MAP_TARGET_TILES
#define MP_MAP_TARGET_TILES 64
#endif
constexpr int MAP_TARGET_TILES = MP_MAP_TARGET_TILES;
constexpr int MAP_MAX_F = 8;
constexpr int64_t MAP_FUSED_MAX_COUNTS = 32768;        // count matrix each rank CTA reads
constexpr int SCAN_THREADS = 1024;
constexpr int SCAN_ITEMS = 8;                          // per thread and pass
constexpr int SCAN_PASS = SCAN_THREADS * SCAN_ITEMS;

struct MapPlan {
    int f;           // tile = 2048 * f routes
    int64_t ntiles;
    bool fused;      // scan inside k_map_rank
};

inline MapPlan map_plan(int64_t n, int E)
{
    int f = 1;
    while (f < MAP_MAX_F && (n + (int64_t)MAP_SUB * f - 1) / ((int64_t)MAP_SUB * f) > MAP_TARGET_TILES)
        f *= 2;
    const int64_t ntiles = (n + (int64_t)MAP_SUB * f - 1) / ((int64_t)MAP_SUB * f);
    return MapPlan{f, ntiles, (int64_t)(E + 1) * ntiles <= MAP_FUSED_MAX_COUNTS};
}

__device__ __forceinline__ int bucket_of(int32_t v, int E) { return (v >= 0 && v < E) ? v : E; }

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Thread-block cluster helpers (one cluster holds every CTA of a map).
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// The int32 at `p` in the shared memory of the cluster's CTA `rank`.
__device__ __forceinline__ int32_t ld_cluster(const int32_t *p, unsigned rank)
{
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
    unsigned ra;
    int32_t v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

// Buckets of this lane's 8 routes of one warp group; -1 past the end.
__device__ __forceinline__ void load_buckets(const int32_t *__restrict__ idx, int64_t n, int E,
                                             int64_t base, int lane, int (&bk)[MAP_CHUNKS],
                                             bool &bad)
{
    int32_t v[MAP_CHUNKS];
#pragma unroll
    for (int c = 0; c < MAP_CHUNKS; ++c) {
        const int64_t i = base + c * 32 + lane;
        v[c] = (i < n) ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int c = 0; c < MAP_CHUNKS; ++c) {
        const int64_t i = base + c * 32 + lane;
        bk[c] = (i < n) ? bucket_of(v[c], E) : -1;
        bad |= (i < n) && v[c] != -1 && bk[c] == E;
    }
}

// First route of warp `warp`'s range in tile `tile`.
__device__ __forceinline__ int64_t warp_base(int tile, int warp, int f)
{
    return (int64_t)tile * MAP_SUB * f + (int64_t)warp * MAP_GROUP * f;
}

__global__ void __launch_bounds__(MAP_THREADS)
    k_map_count(const int32_t *__restrict__ idx, int64_t n, int E, int f, int ntiles,
                int32_t *__restrict__ tile_counts, int32_t *status)
{
    // Wait before the trigger: the rank kernel reads idx before its own wait,
    // so it may start only once whatever wrote idx has finished.
    pdl_wait();
    pdl_trigger();   // the rank kernel's idx-only pass may start now
    extern __shared__ int32_t s_hist[];  // [E+1]
    for (int b = threadIdx.x; b <= E; b += MAP_THREADS) s_hist[b] = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = warp_base(blockIdx.x, warp, f);
    bool bad = false;
    for (int g = 0; g < f; ++g) {
        int bk[MAP_CHUNKS];
        load_buckets(idx, n, E, base + g * MAP_GROUP, lane, bk, bad);
#pragma unroll
        for (int c = 0; c < MAP_CHUNKS; ++c) {
            const unsigned peers = __match_any_sync(FULL_MASK, bk[c]);
            if (bk[c] >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bk[c]], __popc(peers));
        }
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

// Single-CTA exclusive scan of the expert-major count matrix (3-launch path,
// and the T == 0 case where it only writes zero counts and offsets).  Entry
// [b][tile] becomes the routes of buckets before b plus the bucket-b routes of
// earlier tiles; counts / offsets get the capacity-capped expert totals and
// their exclusive scan.
__global__ void __launch_bounds__(SCAN_THREADS)
    k_map_scan(int32_t *__restrict__ tile_counts, int E, int ntiles, int cap,
               int32_t *__restrict__ counts, int32_t *__restrict__ offsets)
{
    __shared__ int32_t s_val[SCAN_PASS + SCAN_PASS / 32];
    __shared__ int32_t s_warp[SCAN_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t M = (int64_t)(E + 1) * ntiles;
    int32_t carry = 0;
    pdl_wait();      // the count kernel has finished, and so has idx's writer
    pdl_trigger();   // the rank kernel reads idx before its wait: only after this one's

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

    // Capped expert totals (one expert per thread, E <= 1024) and their scan.
    int32_t c = 0;
    if (tid < E && ntiles > 0) {
        const int32_t start = tile_counts[(int64_t)tid * ntiles];
        const int32_t next = tile_counts[(int64_t)(tid + 1) * ntiles];
        c = min(next - start, cap);
    }
    if (tid < E) counts[tid] = c;
    int32_t incl = c;
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
        s_warp[lane] = wi - w;
    }
    __syncthreads();
    const int32_t excl = s_warp[warp] + incl - c;
    if (tid < E) offsets[tid] = excl;
    if (tid == SCAN_THREADS - 1) offsets[E] = excl + c;
}

// In-place exclusive scan of a[0..n), n <= 5 * MAP_THREADS, in shared memory;
// returns the total.  Every thread of the CTA calls it.
__device__ int32_t cta_exclusive_scan(int32_t *a, int n, int32_t *s_warp)
{
    constexpr int PER = 5;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = tid * PER;
    int32_t v[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        v[j] = (lo + j < n) ? a[lo + j] : 0;
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
    int32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < MAP_WARPS; ++w) {
        if (w < warp) before += s_warp[w];
        total += s_warp[w];
    }
    int32_t run = before + incl - sum;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        if (lo + j < n) a[lo + j] = run;
        run += v[j];
    }
    __syncthreads();
    return total;
}

inline size_t rank_smem(int E) { return ((size_t)(MAP_WARPS + 3) * (E + 1) + MAP_WARPS) * sizeof(int32_t); }

constexpr int MAP_CACHE_F = 2;   // tiles of up to 2 warp groups keep their ranks in registers
// Buckets each warp reads at once for the totals: 16 warps x 9 cover E + 1 =
// 129 in one round trip to L2 (build_map alone on the skewed T=16,384 map:
// 12.2 us with 8 per warp, 11.1 with 9, 12.4 with 17).
#ifndef MP_MAP_TOTALS_BU
#define MP_MAP_TOTALS_BU 9
#endif

// How k_map_rank gets each bucket's totals and earlier-tile counts:
//   MAP_MODE_PDL     from the tile counts of k_map_count, reduced in every
//                    CTA (a programmatic dependent launch of the count kernel);
//   MAP_MODE_SCANNED from the bases k_map_scan computed;
//   MAP_MODE_SINGLE  one CTA holds all routes (one tile): its own per-warp
//                    histograms are the counts, and no other kernel runs;
//   MAP_MODE_CLUSTER one thread-block cluster holds all routes, a tile per
//                    CTA: each CTA publishes its tile's histogram in shared
//                    memory, and every CTA reads all of them across the
//                    cluster (distributed shared memory) after a cluster
//                    barrier.  One launch, no count kernel, no global round
//                    trip.
constexpr int MAP_MODE_PDL = 0, MAP_MODE_SCANNED = 1, MAP_MODE_SINGLE = 2, MAP_MODE_CLUSTER = 3;
// Maps of up to this many routes are built by one CTA in one launch.  Measured
// (build_map alone, event-timed after an L2 flush): one CTA 8.2 us up to 2,048
// routes and 10.3 us at 4,096, against 10.2-12.3 us for the two kernels; from
// 8,192 routes on the two kernels are as fast or faster (12.3 vs 12.8 / 18.5).
#ifndef MP_MAP_SINGLE_MAX
#define MP_MAP_SINGLE_MAX 4096
#endif
constexpr int64_t MAP_SINGLE_MAX = MP_MAP_SINGLE_MAX;
static_assert(MAP_SINGLE_MAX <= (int64_t)MAP_SUB * MAP_MAX_F, "one tile must hold the routes");

#ifndef MP_MAP_CLUSTER_MAX
#define MP_MAP_CLUSTER_MAX 16
#endif
template <int MODE, bool CACHE>
__global__ void __launch_bounds__(MAP_THREADS)
    k_map_rank(const int32_t *__restrict__ idx, int64_t n, int E, int f, int ntiles, int cap,
               const int32_t *__restrict__ tile_counts, int32_t *__restrict__ row_id_map,
               int32_t *__restrict__ sorted_to_flat, int32_t *__restrict__ counts,
               int32_t *__restrict__ offsets, int32_t *status)
{
    pdl_trigger();
    // A single launch reads nothing from another map kernel: it waits here.
    // The two-kernel forms read idx first and wait below for the counts; the
    // kernel before them waited for idx's writer before it let them start.
    constexpr bool ONE_LAUNCH = MODE == MAP_MODE_SINGLE || MODE == MAP_MODE_CLUSTER;
    if (ONE_LAUNCH) pdl_wait();
    extern __shared__ int32_t sm[];
    const int stride = E + 1;
    int32_t *s_cnt = sm;                              // [MAP_WARPS][E+1] per-warp counters
    int32_t *s_base = s_cnt + MAP_WARPS * stride;     // [E+1] bucket routes in earlier tiles
    int32_t *s_warp = s_base + stride;                // [MAP_WARPS]
    int32_t *s_off = s_warp + MAP_WARPS;              // [E+1] first row of each expert
    int32_t *s_tot = s_off + stride;                  // [E+1] this tile's histogram (cluster)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x;
    int32_t *mine = s_cnt + warp * stride;
    for (int b = tid; b < MAP_WARPS * stride; b += MAP_THREADS) s_cnt[b] = 0;
    if (MODE == MAP_MODE_CLUSTER)
        for (int b = tid; b < stride; b += MAP_THREADS) s_tot[b] = 0;
    __syncthreads();

    // Per-warp histograms of this tile: reads idx only.  With CACHE (f <= CF)
    // each lane also keeps its routes' buckets and their ranks within the
    // warp's range, so the final pass needs no second walk; all of a warp's
    // loads are issued before the first is used.
    const int64_t base = warp_base(tile, warp, f);
    const unsigned lt = lanemask_lt();
    bool bad = false;
    constexpr int CF = ONE_LAUNCH ? MAP_MAX_F : MAP_CACHE_F;
    int cb[CACHE ? CF : 1][MAP_CHUNKS];   // bucket of each route (CACHE)
    int cr[CACHE ? CF : 1][MAP_CHUNKS];   // its rank within the warp's range
    if (CACHE) {
#pragma unroll
        for (int g = 0; g < CF; ++g)
#pragma unroll
            for (int c = 0; c < MAP_CHUNKS; ++c) {
                const int64_t i = base + g * MAP_GROUP + c * 32 + lane;
                cb[g][c] = (g < f && i < n) ? __ldg(idx + i) : -1;   // raw value first
            }
#pragma unroll
        for (int g = 0; g < CF; ++g) {
            if (g >= f) break;
#pragma unroll
            for (int c = 0; c < MAP_CHUNKS; ++c) {
                const int64_t i = base + g * MAP_GROUP + c * 32 + lane;
                const int32_t v = cb[g][c];
                cb[g][c] = (i < n) ? bucket_of(v, E) : -1;
                bad |= (i < n) && v != -1 && cb[g][c] == E;
            }
#pragma unroll
            for (int c = 0; c < MAP_CHUNKS; ++c) {
                const int b = cb[g][c];
                const unsigned peers = __match_any_sync(FULL_MASK, b);
                cr[g][c] = (b >= 0) ? mine[b] + __popc(peers & lt) : 0;
                __syncwarp();
                if (b >= 0 && lane == __ffs(peers) - 1) {
                    mine[b] += __popc(peers);
                    if (MODE == MAP_MODE_CLUSTER) atomicAdd(&s_tot[b], __popc(peers));
                }
                __syncwarp();
            }
        }
    } else {
        for (int g = 0; g < f; ++g) {
            int bk[MAP_CHUNKS];
            load_buckets(idx, n, E, base + g * MAP_GROUP, lane, bk, bad);
#pragma unroll
            for (int c = 0; c < MAP_CHUNKS; ++c) {
                const unsigned peers = __match_any_sync(FULL_MASK, bk[c]);
                if (bk[c] >= 0 && lane == __ffs(peers) - 1) mine[bk[c]] += __popc(peers);
                __syncwarp();
            }
        }
    }

    if (!ONE_LAUNCH)
        pdl_wait();   // the tile counts of every tile are complete from here on

    int32_t kept;     // rows of the permuted tensor (routes kept), offsets[E]
    if constexpr (MODE == MAP_MODE_SINGLE) {
        __syncthreads();   // every warp's histogram is complete
        for (int b = tid; b <= E; b += MAP_THREADS) {
            int32_t tot = 0;
#pragma unroll
            for (int w = 0; w < MAP_WARPS; ++w) tot += s_cnt[w * stride + b];
            s_off[b] = (b < E) ? min(tot, cap) : 0;   // rows the expert keeps
            s_base[b] = 0;
            if (b < E) counts[b] = min(tot, cap);
        }
        if (__syncthreads_or(bad) && tid == 0) or_status(status, MP_STATUS_BAD_EXPERT);
        kept = cta_exclusive_scan(s_off, stride, s_warp);  // s_off: first row of each expert
        for (int b = tid; b <= E; b += MAP_THREADS) offsets[b] = s_off[b];
    } else if constexpr (MODE == MAP_MODE_CLUSTER) {
        // The CTA's cluster rank is its tile (the grid is one cluster).  The
        // tile histogram s_tot was summed by the warps' leaders as they went
        // (integer adds: the order does not reach the result), and the
        // cluster barrier also orders this CTA's own shared memory, so no
        // CTA barrier and no pass over the per-warp counts come first; each
        // bucket's scan over the warps runs in the same pass as its
        // cross-tile totals.  Mid map (12 tiles) 11.65 -> 11.05 us, 4,096
        // to 16,384 routes 0.3-0.4 us faster.
        if (__any_sync(FULL_MASK, bad) && lane == 0) or_status(status, MP_STATUS_BAD_EXPERT);
        cluster_arrive();
        cluster_wait();    // every tile's histogram is visible across the cluster
        for (int b = tid; b <= E; b += MAP_THREADS) {
            // every tile's count of b requested before any is added (one
            // distributed-shared-memory round trip instead of one per tile:
            // mid map, 12 tiles, 11.8 -> 11.0 us)
            int32_t v[MP_MAP_CLUSTER_MAX];
#pragma unroll
            for (int c = 0; c < MP_MAP_CLUSTER_MAX; ++c)
                v[c] = c < ntiles ? ld_cluster(s_tot + b, (unsigned)c) : 0;
            int32_t tot = 0, pre = 0;
#pragma unroll
            for (int c = 0; c < MP_MAP_CLUSTER_MAX; ++c) {
                tot += v[c];
                pre += (c < tile) ? v[c] : 0;
            }
            s_off[b] = (b < E) ? min(tot, cap) : 0;   // rows the expert keeps
            if (tile == 0 && b < E) counts[b] = min(tot, cap);
            // bucket b's exclusive scan over the warps, seeded with its routes
            // in earlier tiles
            int32_t run = pre;
#pragma unroll
            for (int w = 0; w < MAP_WARPS; ++w) {
                const int32_t c = s_cnt[w * stride + b];
                s_cnt[w * stride + b] = run;
                run += c;
            }
        }
        cluster_arrive();  // done reading the others' shared memory (waited on at exit)
        __syncthreads();
        kept = cta_exclusive_scan(s_off, stride, s_warp);  // ends with a CTA barrier
        if (tile == 0)
            for (int b = tid; b <= E; b += MAP_THREADS) offsets[b] = s_off[b];
    } else if constexpr (MODE == MAP_MODE_PDL) {
        // Warp w sums buckets w, w+16, ...: its lanes read the bucket's row of
        // the expert-major count matrix (consecutive tiles, coalesced) and
        // two warp reductions give the bucket's total and the routes of
        // earlier tiles.  BU buckets are read before any is reduced.
        constexpr int BU = MP_MAP_TOTALS_BU;
        for (int b0 = warp; b0 <= E; b0 += MAP_WARPS * BU) {
            int32_t v0[BU], v1[BU];
#pragma unroll
            for (int u = 0; u < BU; ++u) {
                const int b = b0 + u * MAP_WARPS;
                const int32_t *row = tile_counts + (int64_t)b * ntiles;
                v0[u] = (b <= E && lane < ntiles) ? row[lane] : 0;
                v1[u] = (b <= E && lane + 32 < ntiles) ? row[lane + 32] : 0;
            }
#pragma unroll
            for (int u = 0; u < BU; ++u) {
                const int b = b0 + u * MAP_WARPS;
                if (b > E) break;   // warp-uniform: no reductions for absent buckets
                int32_t tot = v0[u] + v1[u];
                int32_t pre = (lane < tile ? v0[u] : 0) + (lane + 32 < tile ? v1[u] : 0);
                if (b <= E)
                    for (int t = lane + 64; t < ntiles; t += 32) {   // more than 64 tiles
                        const int32_t v = tile_counts[(int64_t)b * ntiles + t];
                        tot += v;
                        pre += (t < tile) ? v : 0;
                    }
                const int32_t T_ = __reduce_add_sync(FULL_MASK, tot);
                const int32_t P_ = __reduce_add_sync(FULL_MASK, pre);
                if (lane == 0 && b <= E) {
                    s_off[b] = (b < E) ? min(T_, cap) : 0;   // rows the expert keeps
                    s_base[b] = P_;
                    if (tile == 0 && b < E) counts[b] = min(T_, cap);
                }
            }
        }
        __syncthreads();
        kept = cta_exclusive_scan(s_off, stride, s_warp);  // s_off: first row of each expert
        if (tile == 0)
            for (int b = tid; b <= E; b += MAP_THREADS) offsets[b] = s_off[b];
    } else {
        for (int b = tid; b <= E; b += MAP_THREADS) {
            s_base[b] = tile_counts[(int64_t)b * ntiles + tile] - tile_counts[(int64_t)b * ntiles];
            s_off[b] = offsets[b];
        }
        kept = offsets[E];
    }
    if constexpr (MODE != MAP_MODE_CLUSTER) {   // the cluster form did this above
        __syncthreads();
        // Per bucket: exclusive scan over the warps, seeded with the routes of
        // the bucket in earlier tiles, so the counters hold ranks within the
        // expert.
        for (int b = tid; b <= E; b += MAP_THREADS) {
            int32_t run = s_base[b];
#pragma unroll
            for (int w = 0; w < MAP_WARPS; ++w) {
                const int32_t c = s_cnt[w * stride + b];
                s_cnt[w * stride + b] = run;
                run += c;
            }
        }
        __syncthreads();
    }

    if (CACHE) {
        // mine[b] is now the warp's first rank in bucket b within the expert.
#pragma unroll
        for (int g = 0; g < CF; ++g) {
            if (g >= f) break;
            const int64_t gbase = base + g * MAP_GROUP;
#pragma unroll
            for (int c = 0; c < MAP_CHUNKS; ++c) {
                const int b = cb[g][c];
                if (b >= 0) {
                    const int32_t rank = mine[b] + cr[g][c];
                    const int64_t i = gbase + c * 32 + lane;
                    const bool keep = b < E && rank < cap;
                    const int32_t row = keep ? s_off[b] + rank : -1;
                    row_id_map[i] = row;
                    if (keep && sorted_to_flat != nullptr) sorted_to_flat[row] = (int32_t)i;
                }
            }
        }
    } else {
        for (int g = 0; g < f; ++g) {
            int bk[MAP_CHUNKS];
            const int64_t gbase = base + g * MAP_GROUP;
            load_buckets(idx, n, E, gbase, lane, bk, bad);
#pragma unroll
            for (int c = 0; c < MAP_CHUNKS; ++c) {
                const int b = bk[c];
                const unsigned peers = __match_any_sync(FULL_MASK, b);
                int32_t rank = 0;
                if (b >= 0) rank = mine[b] + __popc(peers & lt);
                __syncwarp();
                if (b >= 0 && lane == __ffs(peers) - 1) mine[b] += __popc(peers);
                __syncwarp();
                if (b >= 0) {
                    const int64_t i = gbase + c * 32 + lane;
                    const bool keep = b < E && rank < cap;
                    const int32_t row = keep ? s_off[b] + rank : -1;
                    row_id_map[i] = row;
                    if (keep && sorted_to_flat != nullptr) sorted_to_flat[row] = (int32_t)i;
                }
            }
        }
    }

    // Rows past the kept ones hold no route: each CTA clears a share.
    if (sorted_to_flat != nullptr) {
        const int64_t tail = n - kept;
        const int64_t per = (tail + ntiles - 1) / ntiles;
        const int64_t lo = kept + (int64_t)tile * per;
        const int64_t hi = min(n, lo + per);
        for (int64_t i = lo + tid; i < hi; i += MAP_THREADS) sorted_to_flat[i] = -1;
    }
    // A CTA's shared memory must outlive every other CTA's reads of it.
    if constexpr (MODE == MAP_MODE_CLUSTER) cluster_wait();
}

inline bool map_sizes_ok(int64_t T, int32_t K, int32_t E)
{
    return T >= 0 && K >= 1 && E >= 1 && E <= MP_MAX_EXPERTS && T * (int64_t)K <= INT32_MAX;
}

inline size_t map_workspace_bytes(int64_t n, int E)
{
    const MapPlan p = map_plan(n, E);
    const size_t bytes = (size_t)(E + 1) * (size_t)p.ntiles * sizeof(int32_t);
    return bytes == 0 ? 256 : (bytes + 255) / 256 * 256;
}

// The cluster form: tiles of 2048 * f routes, f from MP_MAP_CLUSTER_F0 up to
// MAP_MAX_F, one CTA each, at most MP_MAP_CLUSTER_MAX CTAs in the cluster.
#ifndef MP_MAP_CLUSTER_F0
#define MP_MAP_CLUSTER_F0 1
#endif
#ifndef MP_MAP_CLUSTER_ROUTES
#define MP_MAP_CLUSTER_ROUTES (MP_MAP_CLUSTER_MAX * 2048)
#endif
constexpr int MAP_CLUSTER_MAX = MP_MAP_CLUSTER_MAX;
constexpr int64_t MAP_CLUSTER_ROUTES = MP_MAP_CLUSTER_ROUTES;
static_assert(MAP_CLUSTER_ROUTES <= (int64_t)MAP_CLUSTER_MAX * MAP_SUB * MAP_MAX_F,
              "the cluster must hold the routes");

// Launches the cluster form when the GPU can hold such a cluster; returns
// false (nothing launched) otherwise, or when the launch is refused.  Whether
// it fits is asked once per (cluster size, shared memory) and remembered for
// the process (which drives one GPU).
bool launch_map_cluster(const int32_t *idx, int64_t n, int E, int cap, int32_t *row_id_map,
                        int32_t *sorted_to_flat, int32_t *counts, int32_t *offsets,
                        int32_t *dev_status, cudaStream_t s, size_t smem, cudaError_t &err)
{
    int f = MP_MAP_CLUSTER_F0;
    int64_t nc = (n + (int64_t)MAP_SUB * f - 1) / ((int64_t)MAP_SUB * f);
    while (nc > MAP_CLUSTER_MAX && f < MAP_MAX_F) {
        f *= 2;
        nc = (n + (int64_t)MAP_SUB * f - 1) / ((int64_t)MAP_SUB * f);
    }
    if (nc > MAP_CLUSTER_MAX) return false;
    auto fn = k_map_rank<MAP_MODE_CLUSTER, true>;
    static std::mutex mu;
    static bool attrs_set = false;
    static int fits[MAP_CLUSTER_MAX + 1][2] = {};   // per size: smem tried, 1 + (fits ? 1 : 0)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nc);
    cfg.blockDim = dim3(MAP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attrs_set) {
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)rank_smem(MP_MAX_EXPERTS));
            if (err != cudaSuccess) {
                cudaGetLastError();
                err = cudaSuccess;
                return false;
            }
            attrs_set = true;
        }
        int *slot = fits[nc];
        if (slot[0] != (int)smem || slot[1] == 0) {
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
                cudaGetLastError();
                clusters = 0;
            }
            slot[0] = (int)smem;
            slot[1] = 1 + (clusters >= 1 ? 1 : 0);
        }
        if (slot[1] != 2) return false;
    }
    err = cudaLaunchKernelEx(&cfg, fn, idx, n, E, f, (int)nc, cap, (const int32_t *)nullptr,
                             row_id_map, sorted_to_flat, counts, offsets, dev_status);
    if (err != cudaSuccess) {
        // The launch was refused (nothing ran): remember, and take the two kernels.
        cudaGetLastError();
        err = cudaSuccess;
        std::lock_guard<std::mutex> lock(mu);
        fits[nc][1] = 1;
        return false;
    }
    return true;
}

// Enqueues the map kernels; tile_counts holds (E+1) * plan.ntiles words.
mp_status_t launch_map(const int32_t *idx, int64_t n, int E, int cap, int32_t *row_id_map,
                       int32_t *sorted_to_flat, int32_t *counts, int32_t *offsets,
                       int32_t *tile_counts, int32_t *dev_status, cudaStream_t s)
{
    const MapPlan p = map_plan(n, E);
    if (p.ntiles == 0) {
        (void)launch_pdl(k_map_scan, 1, SCAN_THREADS, 0, s, tile_counts, E, 0, cap, counts,
                         offsets);
        return check_launch();
    }
    const size_t smem = rank_smem(E);
    cudaError_t err = cudaSuccess;
    if (n <= MAP_SINGLE_MAX) {
        // One CTA, one launch: for small maps the two-kernel form is all
        // latency (launches, the dependency, L2 round trips).
        int f = 1;
        while ((int64_t)MAP_SUB * f < n) f *= 2;
        auto fn = k_map_rank<MAP_MODE_SINGLE, true>;   // every group cached (f <= MAP_MAX_F)
        if (smem > 48 * 1024)
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err == cudaSuccess)
            (void)launch_pdl(fn, 1, MAP_THREADS, smem, s, idx, n, E, f, 1, cap, nullptr,
                             row_id_map, sorted_to_flat, counts, offsets, dev_status);
        if (err != cudaSuccess) {
            cudaGetLastError();
            set_last_cuda_error(err);
            return MP_ERR_CUDA;
        }
        return check_launch();
    }
    if (n <= MAP_CLUSTER_ROUTES &&
        launch_map_cluster(idx, n, E, cap, row_id_map, sorted_to_flat, counts, offsets,
                           dev_status, s, smem, err))
        return check_launch();
    const unsigned grid = (unsigned)p.ntiles;
    (void)launch_pdl(k_map_count, grid, MAP_THREADS, (E + 1) * sizeof(int32_t), s, idx, n, E,
                     p.f, (int)p.ntiles, tile_counts, dev_status);
    const bool cache = p.f <= MAP_CACHE_F;
    if (p.fused) {
        auto fn = cache ? k_map_rank<MAP_MODE_PDL, true> : k_map_rank<MAP_MODE_PDL, false>;
        if (smem > 48 * 1024)
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err == cudaSuccess)
            err = launch_pdl(fn, grid, MAP_THREADS, smem, s, idx, n, E, p.f, (int)p.ntiles, cap,
                             (const int32_t *)tile_counts, row_id_map, sorted_to_flat, counts,
                             offsets, (int32_t *)nullptr);
    } else {
        auto fn = cache ? k_map_rank<MAP_MODE_SCANNED, true> : k_map_rank<MAP_MODE_SCANNED, false>;
        if (smem > 48 * 1024)
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err == cudaSuccess) {
            (void)launch_pdl(k_map_scan, 1, SCAN_THREADS, 0, s, tile_counts, E, (int)p.ntiles,
                             cap, counts, offsets);
            (void)launch_pdl(fn, grid, MAP_THREADS, smem, s, idx, n, E, p.f, (int)p.ntiles, cap,
                             (const int32_t *)tile_counts, row_id_map, sorted_to_flat, counts,
                             offsets, (int32_t *)nullptr);
        }
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        set_last_cuda_error(err);
        return MP_ERR_CUDA;
    }
    return check_launch();
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
    return map_workspace_bytes(T * (int64_t)K, E);
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
    if (n > 0) {
        if (workspace == nullptr || workspace_bytes < map_workspace_bytes(n, E) ||
            (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
            return MP_ERR_WORKSPACE;
    }
    return launch_map(idx, n, E, INT32_MAX, row_id_map, sorted_to_flat, counts, offsets,
                      static_cast<int32_t *>(workspace), dev_status, as_stream(stream));
}

extern "C" mp_status_t mp_build_map_capacity(const int32_t *idx, int64_t T, int32_t K, int32_t E,
                                             int32_t capacity, int32_t *row_id_map,
                                             int32_t *sorted_to_flat, int32_t *counts,
                                             int32_t *offsets, void *workspace,
                                             size_t workspace_bytes, int32_t *dev_status,
                                             mp_stream_t stream)
{
    if (T < 0 || K < 1 || E < 1) return MP_ERR_INVALID_ARG;
    if (!map_sizes_ok(T, K, E)) return MP_ERR_UNSUPPORTED;
    if (counts == nullptr || offsets == nullptr) return MP_ERR_INVALID_ARG;
    const int64_t n = T * (int64_t)K;
    if (n > 0 && (idx == nullptr || row_id_map == nullptr)) return MP_ERR_INVALID_ARG;
    if (n > 0) {
        if (workspace == nullptr || workspace_bytes < map_workspace_bytes(n, E) ||
            (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
            return MP_ERR_WORKSPACE;
    }
    return launch_map(idx, n, E, capacity < 0 ? INT32_MAX : capacity, row_id_map, sorted_to_flat,
                      counts, offsets, static_cast<int32_t *>(workspace), dev_status,
                      as_stream(stream));
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
    if ((int64_t)(E + 1) * map_plan(n, E).ntiles > NOALLOC_SCRATCH_INTS) return MP_ERR_UNSUPPORTED;
    int32_t *tile_counts = nullptr;
    const mp_status_t st = scratch_on_current_device(&tile_counts);
    if (st != MP_OK) return st;
    // Every tile count the rank (and scan) kernels read is first written by
    // k_map_count in this call, so the array needs no clearing.
    return launch_map(idx, n, E, INT32_MAX, row_id_map, sorted_to_flat, counts, offsets,
                      tile_counts, dev_status, as_stream(stream));
}
