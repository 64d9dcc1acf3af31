// Row movement of the permute / unpermute path and its backward.
//
//   k_permute        out[row_id_map[t,k]] = x[t]            (d9d _permute_kernel)
//   k_unpermute      out[t] = bf16(fma chain over slots)     (Megatron
//                    batch_invariant _rank_tree_unpermute_kernel); also the
//                    permute backward (plain sum + probs gather)
//   k_unpermute_bwd  g_rows[row] = bf16(p * g_y[t]), g_probs = <rows[row], g_y[t]>
//                    (d9d _unpermute_bwd_with_merging_probs_kernel)
//
// One group of `tpt` threads (a power of two, at most a CTA) owns a token;
// a CTA of ROW_THREADS threads holds ROW_THREADS / tpt tokens.  Each thread
// moves VPT 16-byte vectors of the row per pass (uint4 = 8 bf16), or single
// bf16 elements when rows are not 16-byte aligned.  The token's row is read
// once into registers and stored once per slot (permute), or its K source
// rows are all requested before the first FMA so that K * VPT loads are in
// flight per thread (unpermute).  Every token writes only its own rows, so no
// store ever collides and no atomics are needed.
#include "common.cuh"

namespace mp {

namespace {

// Launch shape (overridable at build time for tuning sweeps).
#ifndef MP_ROW_THREADS
#define MP_ROW_THREADS 128
#endif
#ifndef MP_SLOT_BATCH
#define MP_SLOT_BATCH 8
#endif
#ifndef MP_PERMUTE_VPT
#define MP_PERMUTE_VPT 4
#endif
#ifndef MP_UNPERMUTE_VPT
#define MP_UNPERMUTE_VPT 1
#endif
#ifndef MP_BWD_VPT
#define MP_BWD_VPT 1
#endif

constexpr int ROW_THREADS = MP_ROW_THREADS;
constexpr int KB = MP_SLOT_BATCH;  // slots whose rows are in flight together
// Slot batches.  The gathers and the backward, register and staged forms,
// are compiled for batches of 2, 4, KB_SMALL and KB slots, and a token of K
// slots takes the smallest batch that holds it (K > KB: batches of KB, in the
// register forms only).  The registers, and in the staged forms the shared
// memory, of a batch's unused slots would cost resident CTAs.  Fwd+bwd
// steps, K = 2: 8,192 tokens of 4,096 (register forms) 165.7 -> 148.7 us;
// 4,096 tokens of 2,048: 52.3 -> 44.0; 16,384 / 32,768 tokens of 4,096
// (staged) 328.2 / 632.0 -> 283.3 / 547.7.  K = 4: 253.7 -> 250.8, 64.2 ->
// 60.8; 32,768 tokens of 2,048 (staged) 519.1 -> 479.1.
//
// The register-form backward on 16-byte vectors is compiled for 8 CTAs per
// SM with batches of up to KB_SMALL slots (64 registers, no spills) and for
// 5 with KB (92 to 94 registers).  On the T=4,096, H=2,048, K=6 fwd+bwd step:
// 95.2 -> 86.6 us with 6 CTAs per SM (unpermute_bwd 41.0 -> 36.8 us,
// unpermute 23.1 -> 22.2), 84.8 us with 8 (unpermute_bwd 34.7 us; 7 CTAs:
// 84.7 / 34.9); the 6-slot batch alone 98.4 (its backward then took more
// registers), the cap of 6 alone 92.9.  A cap of 6 on the KB form (K = 8)
// made the skewed T=2,048 step slower (115.7 -> 117.9 us).
constexpr int KB_SMALL = 6;
// CTAs per SM the register-form backward is compiled for, by vector type
// (16-byte vectors or single elements) and slot batch.
__host__ __device__ constexpr int bwd_min_blocks(bool vec, int sb)
{
    return vec ? (sb <= KB_SMALL ? 8 : 5) : 3;
}

struct RowGrid {
    int tpt_log2;
    unsigned blocks;
};

inline RowGrid row_grid(int64_t T, int nvec, int vpt)
{
    const int want = (nvec + vpt - 1) / vpt;
    int l = ceil_log2(want < 1 ? 1 : want);
    const int lmax = ceil_log2(ROW_THREADS);
    if (l > lmax) l = lmax;
    const int64_t tokens_per_block = ROW_THREADS >> l;
    return RowGrid{l, (unsigned)((T + tokens_per_block - 1) / tokens_per_block)};
}

template <typename V, int VPT, bool PROBS>
__global__ void __launch_bounds__(ROW_THREADS)
    k_permute(const V *__restrict__ x, const float *__restrict__ probs,
              const int32_t *__restrict__ map, int64_t T, int K, int nvec, int tpt_log2,
              V *__restrict__ out, float *__restrict__ out_probs)
{
    pdl_trigger();
    pdl_wait();
    const int tpt = 1 << tpt_log2;
    const int lane = threadIdx.x & (tpt - 1);
    const int64_t t = (int64_t)blockIdx.x * (ROW_THREADS >> tpt_log2) + (threadIdx.x >> tpt_log2);
    if (t >= T) return;
    const int32_t *m = map + t * K;
    const V *src = x + t * nvec;
    for (int c0 = 0; c0 < nvec; c0 += tpt * VPT) {
        V v[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = c0 + j * tpt + lane;
            v[j] = (c < nvec) ? ld_stream(src + c) : zero_vec<V>();
        }
        for (int k = 0; k < K; ++k) {
            const int32_t row = __ldg(m + k);
            if (row < 0) continue;
            V *dst = out + (int64_t)row * nvec;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int c = c0 + j * tpt + lane;
                if (c < nvec) st_row(dst + c, v[j]);
            }
        }
    }
    if (PROBS && lane == 0) {
        for (int k = 0; k < K; ++k) {
            const int32_t row = __ldg(m + k);
            if (row >= 0) out_probs[row] = __ldg(probs + t * K + k);
        }
    }
}

// acc = fmaf(p, r, acc) per slot in slot order (PROBS), or acc = acc + r.
template <typename V, int VPT, bool PROBS, bool GATHER_PROBS, int SB>
__global__ void __launch_bounds__(ROW_THREADS)
    k_unpermute(const V *__restrict__ rows, const float *__restrict__ probs,
                const int32_t *__restrict__ map, int64_t T, int K, int nvec, int tpt_log2,
                V *__restrict__ out, const float *__restrict__ g_out_probs,
                float *__restrict__ g_probs)
{
    pdl_trigger();
    pdl_wait();
    constexpr int L = Lanes<V>::N;
    const int tpt = 1 << tpt_log2;
    const int lane = threadIdx.x & (tpt - 1);
    const int64_t t = (int64_t)blockIdx.x * (ROW_THREADS >> tpt_log2) + (threadIdx.x >> tpt_log2);
    if (t >= T) return;
    const int32_t *m = map + t * K;
    for (int c0 = 0; c0 < nvec; c0 += tpt * VPT) {
        float acc[VPT][L];
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < L; ++e) acc[j][e] = 0.0f;
        for (int kb = 0; kb < K; kb += SB) {
            int32_t rk[SB];
            float pk[SB];
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                const int k = kb + i;
                rk[i] = (k < K) ? __ldg(m + k) : -1;
                pk[i] = (PROBS && k < K) ? __ldg(probs + t * K + k) : 1.0f;
            }
            V r[SB][VPT];
#pragma unroll
            for (int i = 0; i < SB; ++i)
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int c = c0 + j * tpt + lane;
                    r[i][j] = (rk[i] >= 0 && c < nvec) ? ld_stream(rows + (int64_t)rk[i] * nvec + c)
                                                       : zero_vec<V>();
                }
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                if (rk[i] < 0) continue;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    float f[L];
                    unpack(r[i][j], f);
#pragma unroll
                    for (int e = 0; e < L; ++e)
                        acc[j][e] = PROBS ? __fmaf_rn(pk[i], f[e], acc[j][e]) : __fadd_rn(acc[j][e], f[e]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int c = c0 + j * tpt + lane;
            if (c < nvec) st_row(out + t * nvec + c, pack(acc[j]));
        }
    }
    if (GATHER_PROBS && lane == 0) {
        for (int k = 0; k < K; ++k) {
            const int32_t row = __ldg(m + k);
            g_probs[t * K + k] = row >= 0 ? __ldg(g_out_probs + row) : 0.0f;
        }
    }
}

// Backward of the weighted combine.  All threads stay to the end (the probs
// gradient is a CTA reduction), so tokens past T run with no routed slot.
template <typename V, int VPT, int SB>
__global__ void __launch_bounds__(ROW_THREADS, bwd_min_blocks(Lanes<V>::N == 8, SB))
    k_unpermute_bwd(const V *__restrict__ gy, const V *__restrict__ rows,
                    const float *__restrict__ probs, const int32_t *__restrict__ map, int64_t T,
                    int K, int nvec, int tpt_log2, V *__restrict__ g_rows,
                    float *__restrict__ g_probs)
{
    pdl_trigger();
    pdl_wait();
    constexpr int L = Lanes<V>::N;
    __shared__ float s_red[ROW_THREADS / 32][SB];
    const int tpt = 1 << tpt_log2;
    const int lane = threadIdx.x & (tpt - 1);
    const int64_t t = (int64_t)blockIdx.x * (ROW_THREADS >> tpt_log2) + (threadIdx.x >> tpt_log2);
    const bool active = t < T;
    const int32_t *m = map + t * K;

    for (int kb = 0; kb < K; kb += SB) {
        int32_t rk[SB];
        float pk[SB], dot[SB];
#pragma unroll
        for (int i = 0; i < SB; ++i) {
            const int k = kb + i;
            rk[i] = (active && k < K) ? __ldg(m + k) : -1;
            pk[i] = (active && k < K) ? __ldg(probs + t * K + k) : 0.0f;
            dot[i] = 0.0f;
        }
        for (int c0 = 0; c0 < nvec; c0 += tpt * VPT) {
            V g[VPT];
            V r[SB][VPT];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int c = c0 + j * tpt + lane;
                g[j] = (active && c < nvec) ? ld_stream(gy + t * nvec + c) : zero_vec<V>();
            }
#pragma unroll
            for (int i = 0; i < SB; ++i)
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int c = c0 + j * tpt + lane;
                    r[i][j] = (rk[i] >= 0 && c < nvec) ? ld_stream(rows + (int64_t)rk[i] * nvec + c)
                                                       : zero_vec<V>();
                }
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                if (rk[i] < 0) continue;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int c = c0 + j * tpt + lane;
                    if (c >= nvec) continue;
                    float gf[L], rf[L], o[L];
                    unpack(g[j], gf);
                    unpack(r[i][j], rf);
#pragma unroll
                    for (int e = 0; e < L; ++e) {
                        o[e] = __fmul_rn(pk[i], gf[e]);
                        dot[i] = __fmaf_rn(rf[e], gf[e], dot[i]);
                    }
                    st_row(g_rows + (int64_t)rk[i] * nvec + c, pack(o));
                }
            }
        }
        // Reduce each slot's partial over the token's threads: a butterfly
        // inside the warp, then the token's warps in order.
        const int width = tpt < 32 ? tpt : 32;
#pragma unroll
        for (int i = 0; i < SB; ++i)
            for (int o = width >> 1; o > 0; o >>= 1) dot[i] += __shfl_xor_sync(FULL_MASK, dot[i], o);
        if (tpt > 32) {
            const int warp = threadIdx.x >> 5;
            if ((threadIdx.x & 31) == 0)
#pragma unroll
                for (int i = 0; i < SB; ++i) s_red[warp][i] = dot[i];
            __syncthreads();
            if (active && lane == 0) {
                const int w0 = warp, nw = tpt >> 5;
                for (int i = 0; i < SB && kb + i < K; ++i) {
                    float s = 0.0f;
                    for (int w = 0; w < nw; ++w) s += s_red[w0 + w][i];
                    g_probs[t * K + kb + i] = rk[i] >= 0 ? s : 0.0f;
                }
            }
            __syncthreads();
        } else if (active && lane == 0) {
            for (int i = 0; i < SB && kb + i < K; ++i)
                g_probs[t * K + kb + i] = rk[i] >= 0 ? dot[i] : 0.0f;
        }
    }
}

// Staged forms (16-byte vectors, one vector per thread per pass, K <= SB, a
// slot batch; the shared memory holds SB slots per buffer, plus g_y's
// backward).  Each thread copies its own slots' row vectors (and g_y's) into
// shared memory with cp.async and reads back only those, so no barrier is
// needed.  Two buffers keep a pass ahead: the copies for pass p + 1 are issued
// before pass p is computed, so the rows hold no registers while in flight
// and twice as many bytes are requested per thread.  Same arithmetic, in the
// same order, as k_unpermute / k_unpermute_bwd.
constexpr int STAGE_BUFS = 2;
// The staged forms run only on grids of at least this many CTAs, for the
// gathers and the backward alike.  With 8-slot batches their shared memory
// caps an SM at 6 CTAs where the register forms run 7 (gathers) or 5
// (backward).  On the skewed
// fwd+bwd step (H=4096, one token per CTA) the staged kernels make the step
// faster from 16,384 tokens (0.880 -> 0.870 ms; 32,768: 1.731 -> 1.695;
// 65,536: 3.433 -> 3.350) and slower below (4,096: 0.231 -> 0.241 ms).  A
// step that mixed register gathers with the staged backward was slower
// than either, 0.899 ms at 16,384 tokens.  Switching between the two forms
// costs: an SM changes its L1 / shared-memory split only when idle, and the
// staged forms want most of it as shared memory.  On the T=4,096, H=2,048,
// K=6 step the staged backward alone is faster (41.0 -> 36.9 us) but the
// register-form kernel after it slows by 3 us even with an event between
// them, and the step gets slower (0.097 -> 0.100 ms).  Preferring the
// largest shared split for every kernel instead makes the register forms
// slower still (T=8,192, H=4,096: unpermute 95 -> 112 us; the smaller L1
// holds fewer loads in flight).  The overrides are for tuning sweeps.
#ifndef MP_STAGE_MIN_BLOCKS
#define MP_STAGE_MIN_BLOCKS 16384
#endif
#ifndef MP_STAGE_MIN_BLOCKS_BWD
#define MP_STAGE_MIN_BLOCKS_BWD MP_STAGE_MIN_BLOCKS
#endif
constexpr unsigned STAGE_MIN_BLOCKS = MP_STAGE_MIN_BLOCKS;
constexpr unsigned STAGE_MIN_BLOCKS_BWD = MP_STAGE_MIN_BLOCKS_BWD;
// The staged kernels are launched without raising their dynamic shared memory
// limit, so both stage sizes must fit the default 48 KB (an MP_ROW_THREADS or
// MP_SLOT_BATCH override that breaks this fails to compile, not to launch).
static_assert((size_t)STAGE_BUFS * KB * ROW_THREADS * sizeof(uint4) <= 48 * 1024,
              "forward stage buffers exceed the default dynamic shared memory limit");
static_assert((size_t)STAGE_BUFS * (KB + 1) * ROW_THREADS * sizeof(uint4) <= 48 * 1024,
              "backward stage buffers exceed the default dynamic shared memory limit");

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool PROBS, bool GATHER_PROBS, int SB>
__global__ void __launch_bounds__(ROW_THREADS)
    k_unpermute_staged(const uint4 *__restrict__ rows, const float *__restrict__ probs,
                       const int32_t *__restrict__ map, int64_t T, int K, int nvec,
                       int tpt_log2, uint4 *__restrict__ out,
                       const float *__restrict__ g_out_probs, float *__restrict__ g_probs)
{
    pdl_trigger();
    pdl_wait();
    extern __shared__ uint4 row_stage[];   // [STAGE_BUFS][SB][ROW_THREADS]
    const int tpt = 1 << tpt_log2;
    const int lane = threadIdx.x & (tpt - 1);
    const int64_t t = (int64_t)blockIdx.x * (ROW_THREADS >> tpt_log2) + (threadIdx.x >> tpt_log2);
    if (t >= T) return;
    const int32_t *m = map + t * K;
    int32_t rk[SB];
    float pk[SB];
#pragma unroll
    for (int i = 0; i < SB; ++i) {
        rk[i] = (i < K) ? __ldg(m + i) : -1;
        pk[i] = (PROBS && i < K) ? __ldg(probs + t * K + i) : 1.0f;
    }
    const auto issue = [&](int c, int buf) {
        uint4 *const dst = row_stage + buf * SB * ROW_THREADS + threadIdx.x;
#pragma unroll
        for (int i = 0; i < SB; ++i)
            if (rk[i] >= 0) cp_async16(dst + i * ROW_THREADS, rows + (int64_t)rk[i] * nvec + c);
        cp_async_commit();
    };
    if (lane < nvec) issue(lane, 0);
    int pass = 0;
    for (int c = lane; c < nvec; c += tpt, ++pass) {
        if (c + tpt < nvec) {
            issue(c + tpt, (pass + 1) & 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        const uint4 *const mine = row_stage + (pass & 1) * SB * ROW_THREADS + threadIdx.x;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
        for (int i = 0; i < SB; ++i) {
            if (rk[i] < 0) continue;
            float f[8];
            unpack(mine[i * ROW_THREADS], f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] = PROBS ? __fmaf_rn(pk[i], f[e], acc[e]) : __fadd_rn(acc[e], f[e]);
        }
        st_row(out + t * nvec + c, pack(acc));
    }
    if (GATHER_PROBS && lane == 0) {
        for (int k = 0; k < K; ++k) {
            const int32_t row = __ldg(m + k);
            g_probs[t * K + k] = row >= 0 ? __ldg(g_out_probs + row) : 0.0f;
        }
    }
}

template <int SB>
__global__ void __launch_bounds__(ROW_THREADS)
    k_unpermute_bwd_staged(const uint4 *__restrict__ gy, const uint4 *__restrict__ rows,
                           const float *__restrict__ probs, const int32_t *__restrict__ map,
                           int64_t T, int K, int nvec, int tpt_log2,
                           uint4 *__restrict__ g_rows, float *__restrict__ g_probs)
{
    pdl_trigger();
    pdl_wait();
    extern __shared__ uint4 row_stage[];   // [STAGE_BUFS][SB + 1][ROW_THREADS]; slot SB: g_y
    __shared__ float s_red[ROW_THREADS / 32][SB];
    const int tpt = 1 << tpt_log2;
    const int lane = threadIdx.x & (tpt - 1);
    const int64_t t = (int64_t)blockIdx.x * (ROW_THREADS >> tpt_log2) + (threadIdx.x >> tpt_log2);
    const bool active = t < T;
    const int32_t *m = map + t * K;
    int32_t rk[SB];
    float pk[SB], dot[SB];
#pragma unroll
    for (int i = 0; i < SB; ++i) {
        rk[i] = (active && i < K) ? __ldg(m + i) : -1;
        pk[i] = (active && i < K) ? __ldg(probs + t * K + i) : 0.0f;
        dot[i] = 0.0f;
    }
    const auto issue = [&](int c, int buf) {
        uint4 *const dst = row_stage + buf * (SB + 1) * ROW_THREADS + threadIdx.x;
        cp_async16(dst + SB * ROW_THREADS, gy + t * nvec + c);
#pragma unroll
        for (int i = 0; i < SB; ++i)
            if (rk[i] >= 0) cp_async16(dst + i * ROW_THREADS, rows + (int64_t)rk[i] * nvec + c);
        cp_async_commit();
    };
    if (active) {
        if (lane < nvec) issue(lane, 0);
        int pass = 0;
        for (int c = lane; c < nvec; c += tpt, ++pass) {
            if (c + tpt < nvec) {
                issue(c + tpt, (pass + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            const uint4 *const mine = row_stage + (pass & 1) * (SB + 1) * ROW_THREADS + threadIdx.x;
            float gf[8];
            unpack(mine[SB * ROW_THREADS], gf);
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                if (rk[i] < 0) continue;
                float rf[8], o[8];
                unpack(mine[i * ROW_THREADS], rf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    o[e] = __fmul_rn(pk[i], gf[e]);
                    dot[i] = __fmaf_rn(rf[e], gf[e], dot[i]);
                }
                st_row(g_rows + (int64_t)rk[i] * nvec + c, pack(o));
            }
        }
    }
    // Each slot's partial reduced over the token's threads, as in k_unpermute_bwd.
    const int width = tpt < 32 ? tpt : 32;
#pragma unroll
    for (int i = 0; i < SB; ++i)
        for (int o = width >> 1; o > 0; o >>= 1) dot[i] += __shfl_xor_sync(FULL_MASK, dot[i], o);
    if (tpt > 32) {
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0)
#pragma unroll
            for (int i = 0; i < SB; ++i) s_red[warp][i] = dot[i];
        __syncthreads();
        if (active && lane == 0) {
            const int w0 = warp, nw = tpt >> 5;
            for (int i = 0; i < SB && i < K; ++i) {
                float s = 0.0f;
                for (int w = 0; w < nw; ++w) s += s_red[w0 + w][i];
                g_probs[t * K + i] = rk[i] >= 0 ? s : 0.0f;
            }
        }
    } else if (active && lane == 0) {
        for (int i = 0; i < SB && i < K; ++i) g_probs[t * K + i] = rk[i] >= 0 ? dot[i] : 0.0f;
    }
}

inline bool rows_ok(int64_t T, int32_t K, int32_t H)
{
    return T >= 0 && K >= 1 && H >= 1 && T * (int64_t)K <= INT32_MAX;
}

inline bool vec_ok(int32_t H, std::initializer_list<const void *> ptrs)
{
    if (H % 8 != 0) return false;
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p)) return false;
    return true;
}

constexpr int PERMUTE_VPT = MP_PERMUTE_VPT;
#ifndef MP_PERMUTE_VPT_MID
#define MP_PERMUTE_VPT_MID 2
#endif
// Rows of 129 to 256 vectors (1,032 to 2,048 bf16) take MP_PERMUTE_VPT_MID
// vectors per thread, so that a token is one pass of a whole 128-thread CTA
// rather than half a CTA: the T=4,096, H=2,048, K=6 fwd+bwd step 97.5 ->
// 95.2 us.  With H=4,096 or 7,168 four per thread stay faster (two per
// thread: T=16,384 step 868 -> 872 us).  Wider rows (more than 256
// vectors), 32-byte aligned with an even vector count, move as 32-byte
// vectors, four per thread: half the load and store instructions
// (permute on the skewed T=16,384 batch 180.3 -> 179.2 us, the large
// T=8,192 step 790.4 -> 783.7 us; on 2,048-element rows they were slower,
// 84.3 -> 86.1 us for the mid step).
constexpr int UNPERMUTE_VPT = MP_UNPERMUTE_VPT;
constexpr int BWD_VPT = MP_BWD_VPT;
constexpr int ELEM_VPT = 8;

template <typename V, int VPT>
void launch_permute(const void *x, const float *probs, const int32_t *map, int64_t T, int K,
                    int nvec, void *out, float *out_probs, cudaStream_t s)
{
    const RowGrid g = row_grid(T, nvec, VPT);
    if (probs != nullptr && out_probs != nullptr)
        (void)launch_pdl(k_permute<V, VPT, true>, g.blocks, ROW_THREADS, 0, s,
            (const V *)x, probs, map, T, K, nvec, g.tpt_log2, (V *)out, out_probs);
    else
        (void)launch_pdl(k_permute<V, VPT, false>, g.blocks, ROW_THREADS, 0, s,
            (const V *)x, nullptr, map, T, K, nvec, g.tpt_log2, (V *)out, nullptr);
}

// The permute's row copy on 16-byte vectors (see PERMUTE_VPT above).
inline void launch_permute_vec(const void *x, const float *probs, const int32_t *map,
                               int64_t T, int K, int nvec, void *out, float *out_probs,
                               cudaStream_t s)
{
    if (nvec > 2 * ROW_THREADS && nvec % 2 == 0 && aligned32(x) && aligned32(out)) {
        launch_permute<u32x8, PERMUTE_VPT>(x, probs, map, T, K, nvec / 2, out, out_probs, s);
        return;
    }
    if (nvec > ROW_THREADS && nvec <= 2 * ROW_THREADS)
        launch_permute<uint4, MP_PERMUTE_VPT_MID>(x, probs, map, T, K, nvec, out, out_probs, s);
    else
        launch_permute<uint4, PERMUTE_VPT>(x, probs, map, T, K, nvec, out, out_probs, s);
}

template <int SB>
void launch_unpermute_st(const RowGrid &g, const void *rows, const float *probs,
                         const int32_t *map, int64_t T, int K, int nvec, void *out,
                         const float *g_out_probs, float *g_probs, cudaStream_t s)
{
    const size_t smem = (size_t)STAGE_BUFS * SB * ROW_THREADS * sizeof(uint4);
    if (probs != nullptr)
        (void)launch_pdl(k_unpermute_staged<true, false, SB>, g.blocks, ROW_THREADS, smem, s,
            (const uint4 *)rows, probs, map, T, K, nvec, g.tpt_log2, (uint4 *)out,
            nullptr, nullptr);
    else if (g_probs != nullptr)
        (void)launch_pdl(k_unpermute_staged<false, true, SB>, g.blocks, ROW_THREADS, smem, s,
            (const uint4 *)rows, nullptr, map, T, K, nvec, g.tpt_log2, (uint4 *)out,
            g_out_probs, g_probs);
    else
        (void)launch_pdl(k_unpermute_staged<false, false, SB>, g.blocks, ROW_THREADS, smem,
            s, (const uint4 *)rows, nullptr, map, T, K, nvec, g.tpt_log2, (uint4 *)out,
            nullptr, nullptr);
}

template <int SB>
void launch_unpermute_bwd_st(const RowGrid &g, const void *gy, const void *rows,
                             const float *probs, const int32_t *map, int64_t T, int K,
                             int nvec, void *g_rows, float *g_probs, cudaStream_t s)
{
    const size_t smem = (size_t)STAGE_BUFS * (SB + 1) * ROW_THREADS * sizeof(uint4);
    (void)launch_pdl(k_unpermute_bwd_staged<SB>, g.blocks, ROW_THREADS, smem, s,
        (const uint4 *)gy, (const uint4 *)rows, probs, map, T, K, nvec, g.tpt_log2,
        (uint4 *)g_rows, g_probs);
}

template <typename V, int VPT, int SB>
void launch_unpermute_reg(const RowGrid &g, const void *rows, const float *probs,
                          const int32_t *map, int64_t T, int K, int nvec, void *out,
                          const float *g_out_probs, float *g_probs, cudaStream_t s)
{
    if (probs != nullptr)
        (void)launch_pdl(k_unpermute<V, VPT, true, false, SB>, g.blocks, ROW_THREADS, 0, s,
            (const V *)rows, probs, map, T, K, nvec, g.tpt_log2, (V *)out, nullptr, nullptr);
    else if (g_probs != nullptr)
        (void)launch_pdl(k_unpermute<V, VPT, false, true, SB>, g.blocks, ROW_THREADS, 0, s,
            (const V *)rows, nullptr, map, T, K, nvec, g.tpt_log2, (V *)out, g_out_probs,
            g_probs);
    else
        (void)launch_pdl(k_unpermute<V, VPT, false, false, SB>, g.blocks, ROW_THREADS, 0, s,
            (const V *)rows, nullptr, map, T, K, nvec, g.tpt_log2, (V *)out, nullptr, nullptr);
}

template <typename V, int VPT>
void launch_unpermute(const void *rows, const float *probs, const int32_t *map, int64_t T, int K,
                      int nvec, void *out, const float *g_out_probs, float *g_probs,
                      cudaStream_t s)
{
    const RowGrid g = row_grid(T, nvec, VPT);
    if constexpr (Lanes<V>::N == 8 && VPT == 1) {
        if (K <= KB && g.blocks >= STAGE_MIN_BLOCKS) {
            if (K <= 2)
                launch_unpermute_st<2>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                       g_probs, s);
            else if (K <= 4)
                launch_unpermute_st<4>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                       g_probs, s);
            else if (K <= KB_SMALL)
                launch_unpermute_st<KB_SMALL>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                              g_probs, s);
            else
                launch_unpermute_st<KB>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                        g_probs, s);
            return;
        }
    }
    if (K <= 2)
        launch_unpermute_reg<V, VPT, 2>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                        g_probs, s);
    else if (K <= 4)
        launch_unpermute_reg<V, VPT, 4>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                        g_probs, s);
    else if (K <= KB_SMALL)
        launch_unpermute_reg<V, VPT, KB_SMALL>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                               g_probs, s);
    else
        launch_unpermute_reg<V, VPT, KB>(g, rows, probs, map, T, K, nvec, out, g_out_probs,
                                         g_probs, s);
}

template <typename V, int VPT>
void launch_unpermute_bwd(const void *gy, const void *rows, const float *probs,
                          const int32_t *map, int64_t T, int K, int nvec, void *g_rows,
                          float *g_probs, cudaStream_t s)
{
    const RowGrid g = row_grid(T, nvec, VPT);
    if constexpr (Lanes<V>::N == 8 && VPT == 1) {
        if (K <= KB && g.blocks >= STAGE_MIN_BLOCKS_BWD) {
            if (K <= 2)
                launch_unpermute_bwd_st<2>(g, gy, rows, probs, map, T, K, nvec, g_rows, g_probs,
                                           s);
            else if (K <= 4)
                launch_unpermute_bwd_st<4>(g, gy, rows, probs, map, T, K, nvec, g_rows, g_probs,
                                           s);
            else if (K <= KB_SMALL)
                launch_unpermute_bwd_st<KB_SMALL>(g, gy, rows, probs, map, T, K, nvec, g_rows,
                                                  g_probs, s);
            else
                launch_unpermute_bwd_st<KB>(g, gy, rows, probs, map, T, K, nvec, g_rows, g_probs,
                                            s);
            return;
        }
    }
    if (K <= 2)
        (void)launch_pdl(k_unpermute_bwd<V, VPT, 2>, g.blocks, ROW_THREADS, 0, s,
            (const V *)gy, (const V *)rows, probs, map, T, K, nvec, g.tpt_log2, (V *)g_rows,
            g_probs);
    else if (K <= 4)
        (void)launch_pdl(k_unpermute_bwd<V, VPT, 4>, g.blocks, ROW_THREADS, 0, s,
            (const V *)gy, (const V *)rows, probs, map, T, K, nvec, g.tpt_log2, (V *)g_rows,
            g_probs);
    else if (K <= KB_SMALL)
        (void)launch_pdl(k_unpermute_bwd<V, VPT, KB_SMALL>, g.blocks, ROW_THREADS, 0, s,
            (const V *)gy, (const V *)rows, probs, map, T, K, nvec, g.tpt_log2, (V *)g_rows,
            g_probs);
    else
        (void)launch_pdl(k_unpermute_bwd<V, VPT, KB>, g.blocks, ROW_THREADS, 0, s,
            (const V *)gy, (const V *)rows, probs, map, T, K, nvec, g.tpt_log2, (V *)g_rows,
            g_probs);
}

}  // namespace
}  // namespace mp

using namespace mp;

extern "C" mp_status_t mp_permute(const mp_bf16_t *x, const float *probs,
                                  const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                                  mp_bf16_t *out, float *out_probs, mp_stream_t stream)
{
    if (!rows_ok(T, K, H)) return MP_ERR_INVALID_ARG;
    if (T == 0) return MP_OK;
    if (x == nullptr || row_id_map == nullptr || out == nullptr) return MP_ERR_INVALID_ARG;
    if ((probs == nullptr) != (out_probs == nullptr)) return MP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (vec_ok(H, {x, out}))
        launch_permute_vec(x, probs, row_id_map, T, K, H / 8, out, out_probs, s);
    else
        launch_permute<uint16_t, ELEM_VPT>(x, probs, row_id_map, T, K, H, out, out_probs, s);
    return check_launch();
}

extern "C" mp_status_t mp_unpermute(const mp_bf16_t *rows, const float *probs,
                                    const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                                    mp_bf16_t *out, mp_stream_t stream)
{
    if (!rows_ok(T, K, H)) return MP_ERR_INVALID_ARG;
    if (T == 0) return MP_OK;
    if (rows == nullptr || row_id_map == nullptr || out == nullptr) return MP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (vec_ok(H, {rows, out}))
        launch_unpermute<uint4, UNPERMUTE_VPT>(rows, probs, row_id_map, T, K, H / 8, out, nullptr,
                                               nullptr, s);
    else
        launch_unpermute<uint16_t, ELEM_VPT>(rows, probs, row_id_map, T, K, H, out, nullptr,
                                             nullptr, s);
    return check_launch();
}

extern "C" mp_status_t mp_permute_bwd(const mp_bf16_t *g_out, const float *g_out_probs,
                                      const int32_t *row_id_map, int64_t T, int32_t K, int32_t H,
                                      mp_bf16_t *g_x, float *g_probs, mp_stream_t stream)
{
    if (!rows_ok(T, K, H)) return MP_ERR_INVALID_ARG;
    if (T == 0) return MP_OK;
    if (g_out == nullptr || row_id_map == nullptr || g_x == nullptr) return MP_ERR_INVALID_ARG;
    if ((g_out_probs == nullptr) != (g_probs == nullptr)) return MP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (vec_ok(H, {g_out, g_x}))
        launch_unpermute<uint4, UNPERMUTE_VPT>(g_out, nullptr, row_id_map, T, K, H / 8, g_x,
                                               g_out_probs, g_probs, s);
    else
        launch_unpermute<uint16_t, ELEM_VPT>(g_out, nullptr, row_id_map, T, K, H, g_x,
                                             g_out_probs, g_probs, s);
    return check_launch();
}

extern "C" mp_status_t mp_unpermute_bwd(const mp_bf16_t *g_y, const mp_bf16_t *rows,
                                        const float *probs, const int32_t *row_id_map, int64_t T,
                                        int32_t K, int32_t H, mp_bf16_t *g_rows, float *g_probs,
                                        mp_stream_t stream)
{
    if (!rows_ok(T, K, H)) return MP_ERR_INVALID_ARG;
    if (T == 0) return MP_OK;
    if (g_y == nullptr || row_id_map == nullptr || g_rows == nullptr) return MP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (probs == nullptr) {
        // No merging probs: the token's gradient goes unchanged to each row.
        if (vec_ok(H, {g_y, g_rows}))
            launch_permute_vec(g_y, nullptr, row_id_map, T, K, H / 8, g_rows, nullptr, s);
        else
            launch_permute<uint16_t, ELEM_VPT>(g_y, nullptr, row_id_map, T, K, H, g_rows, nullptr,
                                               s);
        return check_launch();
    }
    if (rows == nullptr || g_probs == nullptr) return MP_ERR_INVALID_ARG;
    if (vec_ok(H, {g_y, rows, g_rows}))
        launch_unpermute_bwd<uint4, BWD_VPT>(g_y, rows, probs, row_id_map, T, K, H / 8, g_rows,
                                             g_probs, s);
    else
        launch_unpermute_bwd<uint16_t, ELEM_VPT>(g_y, rows, probs, row_id_map, T, K, H, g_rows,
                                                 g_probs, s);
    return check_launch();
}
