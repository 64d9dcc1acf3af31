// Fused top-k softmax router: the routing input of the map, from logits.
//
// "moe-ops 0.1.0" README, "Operators": fused_topk_softmax fuses the top-K
// selection and the softmax normalisation in registers, and its backward
// computes the exact softmax gradient scattered back to the logits.  The
// group-limited choice (keep the best groups of experts first) follows the
// large routed workload of the pages' configurations.
//
// k_topk_softmax: one warp per token; lane l holds logits l, l+32, ... (so
// every load instruction reads 32 consecutive floats).  Logits are compared
// through an order-preserving 32-bit key (-0 folded into +0), so a warp's
// arg-max on (logit desc, expert asc) is two single-instruction warp
// reductions: the largest key, then the smallest expert holding it.  Group
// scores are warp max-reductions of the same keys; when every group is a
// whole number of 32-expert columns (each lane's slot j then lies in group
// j / s for every lane), a group's score is one reduction of the column
// maxima, and no lane computes a group index.  For the K picks (up to
// 256 experts) each lane first sorts its own experts with a fixed sorting
// network, so a round is the two reductions on the lanes' heads and the
// winner drops its head; when at most half of the columns hold a live expert
// (groups not kept, or few experts), the live ones are gathered and only
// they are sorted.  Wider rows rescan each lane's experts per round.
// Lane k keeps pick k.  The softmax runs in fp32: z_k = l_k - l_0, expf
// (full accuracy), the sum in slot order, IEEE division.
// k_topk_softmax_bwd: one warp per token: zero the token's E gradients, then
// p_k * (g_k - sum_j p_j g_j) at the picked experts.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace mp {
namespace {

constexpr int RT_THREADS = 256;
constexpr int RT_WARPS = RT_THREADS / 32;

// A 32-bit key with the order of the floats: key(a) < key(b) iff a < b (for
// non-NaN values; -0 and +0 get the same key).  Every float's key is > 0, so 0
// stands for "no candidate".
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Arg-max across the warp on (key desc, index asc); every lane gets the
// winning index (the key is returned through `key`).
__device__ __forceinline__ uint32_t warp_argmax_key(uint32_t &key, uint32_t idx)
{
    const uint32_t m = __reduce_max_sync(FULL_MASK, key);
    const uint32_t i = __reduce_min_sync(FULL_MASK, key == m ? idx : 0xffffffffu);
    key = m;
    return i;
}

// Compare-exchange for a descending order on (key desc, index asc).
__device__ __forceinline__ void cx_desc(uint32_t &ka, uint32_t &ia, uint32_t &kb, uint32_t &ib)
{
    const bool keep = ka > kb || (ka == kb && ia < ib);
    const uint32_t k0 = keep ? ka : kb, k1 = keep ? kb : ka;
    const uint32_t i0 = keep ? ia : ib, i1 = keep ? ib : ia;
    ka = k0; kb = k1; ia = i0; ib = i1;
}

// Batcher's odd-even merge sort of N (a power of two) (key, index) pairs,
// descending; every index is a compile-time constant once unrolled.
template <int N>
__device__ __forceinline__ void sort_desc(uint32_t (&k)[N], uint32_t (&ix)[N])
{
#pragma unroll
    for (int p = 1; p < N; p <<= 1)
#pragma unroll
        for (int q = p; q >= 1; q >>= 1)
#pragma unroll
            for (int j = q % p; j + q < N; j += 2 * q)
#pragma unroll
                for (int i = 0; i < q; ++i)
                    if (i + j + q < N && (i + j) / (2 * p) == (i + j + q) / (2 * p))
                        cx_desc(k[i + j], ix[i + j], k[i + j + q], ix[i + j + q]);
}

// Sorts a lane's N (key, expert) slots, then runs the K pick rounds: each
// round is two warp reductions on the lanes' heads, and the lane whose head
// is the picked expert (a live head's expert is unique) drops it.  Lane k
// keeps pick k.
// KT > 0: K is the compile-time KT (the rounds unrolled).
template <int N, int KT = 0>
__device__ __forceinline__ void pick_rounds(uint32_t (&key)[N], uint32_t (&ex)[N], int K,
                                            int lane, uint32_t &my_key, int &my_i)
{
    sort_desc<N>(key, ex);
    if (KT > 0) K = KT;
#pragma unroll
    for (int k = 0; k < (KT > 0 ? KT : K); ++k) {
        uint32_t bk = key[0];
        const uint32_t pick = warp_argmax_key(bk, ex[0]);
        if (ex[0] == pick) {
#pragma unroll
            for (int j = 0; j + 1 < N; ++j) {
                key[j] = key[j + 1];
                ex[j] = ex[j + 1];
            }
            key[N - 1] = 0u;
        }
        if (lane == k) {
            my_key = bk;
            my_i = (int)pick;
        }
    }
}

// KT > 0: a form for K = KT, with the pick rounds and the softmax sum
// unrolled (K = 8 on the skewed T=16,384, E=128 batch: 12.0 -> 10.2 us; the
// grouped T=32,768, E=256 one: 31.5 -> 30.8 us).
template <int PER, int KT = 0>
__global__ void __launch_bounds__(RT_THREADS)
    k_topk_softmax(const float *__restrict__ logits, int64_t T, int E, int K, int n_groups,
                   int topk_groups, int32_t *__restrict__ idx, float *__restrict__ probs)
{
    pdl_trigger();
    pdl_wait();
    if (KT > 0) K = KT;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * RT_WARPS + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warps exit together
    const float *l = logits + t * E;
    float v[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? __ldg(l + e) : -FLT_MAX;
    }
    // Experts still eligible: bit j of `live` stands for expert lane + 32*j.
    unsigned live = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
        if (lane + 32 * j < E) live |= 1u << j;

    if (n_groups > 1 && (E / n_groups) % 32 == 0) {
        // Groups of whole 32-expert columns: slot j of every lane is in group
        // j / s (s = columns per group), so a group's score is a warp max
        // over its s slots; slots are walked with a counter, not a division.
        const int s = (E / n_groups) / 32;
        const int ncols = E / 32;
        unsigned group_kept = 0;
        uint32_t score_g = 0;      // lane g holds group g's score key
        uint32_t colmax = 0;
        int cnt = 0, gcur = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            if (j < ncols) {
                colmax = max(colmax, (live >> j & 1u) ? order_key(v[j]) : 0u);
                if (++cnt == s) {
                    const uint32_t m = __reduce_max_sync(FULL_MASK, colmax);
                    if (lane == gcur) score_g = m;
                    colmax = 0;
                    cnt = 0;
                    ++gcur;
                }
            }
        }
        for (int j = 0; j < topk_groups; ++j) {
            uint32_t sk = (lane < n_groups && !(group_kept >> lane & 1u)) ? score_g : 0u;
            const uint32_t gi = warp_argmax_key(sk, (uint32_t)lane);
            group_kept |= 1u << gi;
        }
        cnt = 0;
        gcur = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            if (j < ncols && !(group_kept >> gcur & 1u)) live &= ~(1u << j);
            if (++cnt == s) {
                cnt = 0;
                ++gcur;
            }
        }
    } else if (n_groups > 1) {
        const int per_group = E / n_groups;
        int grp[PER];              // group of each of this lane's experts (one division each)
        uint32_t kj[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            grp[j] = (lane + 32 * j) / per_group;
            kj[j] = (live >> j & 1u) ? order_key(v[j]) : 0u;
        }
        unsigned group_kept = 0;   // bit g: group g kept (same in every lane)
        uint32_t score_g = 0;      // lane g holds group g's score key
        for (int g = 0; g < n_groups; ++g) {
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < PER; ++j)
                if (grp[j] == g) m = max(m, kj[j]);
            m = __reduce_max_sync(FULL_MASK, m);
            if (lane == g) score_g = m;
        }
        for (int j = 0; j < topk_groups; ++j) {
            uint32_t sk = (lane < n_groups && !(group_kept >> lane & 1u)) ? score_g : 0u;
            const uint32_t gi = warp_argmax_key(sk, (uint32_t)lane);
            group_kept |= 1u << gi;
        }
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if ((live >> j & 1u) && !(group_kept >> grp[j] & 1u)) live &= ~(1u << j);
    }

    float my_v = 0.0f;
    int my_i = -1;
    if constexpr (PER <= 8) {
        // Each lane sorts its live experts once (dead ones get key 0, last);
        // a round's winner then drops its head, so every lane's head stays
        // its best remaining expert (pick_rounds).
        uint32_t key[PER], ex[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            key[j] = (live >> j & 1u) ? order_key(v[j]) : 0u;
            ex[j] = (uint32_t)(lane + 32 * j);
        }
        uint32_t my_key = 0u;
        // Columns with a live expert in any lane (the same in every lane).
        const unsigned cols = __reduce_or_sync(FULL_MASK, live);
        if (PER >= 4 && __popc(cols) <= PER / 2) {
            // At most half the columns live (unkept groups, or E <= 16*PER):
            // gather them into half as many slots, in any order, and sort
            // those.
            constexpr int HALF = PER >= 4 ? PER / 2 : 1;
            uint32_t kc[HALF], xc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
                kc[i] = 0u;
                xc[i] = 0xffffffffu;
            }
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                if (cols >> j & 1u) {
#pragma unroll
                    for (int i = HALF - 1; i > 0; --i) {
                        kc[i] = kc[i - 1];
                        xc[i] = xc[i - 1];
                    }
                    kc[0] = key[j];
                    xc[0] = ex[j];
                }
            }
            pick_rounds<HALF, KT>(kc, xc, K, lane, my_key, my_i);
        } else {
            pick_rounds<PER, KT>(key, ex, K, lane, my_key, my_i);
        }
        my_v = key_value(my_key);
    } else {
        // Wide rows (more than 256 experts): each round rescans the lane's
        // live experts (a sort network that large would not stay in registers).
        uint32_t key[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) key[j] = order_key(v[j]);
        for (int k = 0; k < K; ++k) {
            uint32_t bk = 0u, bi = 0xffffffffu;   // this lane's best live expert
#pragma unroll
            for (int j = 0; j < PER; ++j)
                if ((live >> j & 1u) && key[j] > bk) {
                    bk = key[j];
                    bi = (uint32_t)(lane + 32 * j);
                }
            const uint32_t pick = warp_argmax_key(bk, bi);
            if ((int)(pick & 31u) == lane) live &= ~(1u << (pick >> 5));
            if (lane == k) {
                my_v = key_value(bk);
                my_i = (int)pick;
            }
        }
    }
    const float m = __shfl_sync(FULL_MASK, my_v, 0);
    const float ez = lane < K ? expf(my_v - m) : 0.0f;
    float s = 0.0f;
    for (int k = 0; k < K; ++k) s = __fadd_rn(s, __shfl_sync(FULL_MASK, ez, k));
    if (lane < K) {
        idx[t * K + lane] = my_i;
        probs[t * K + lane] = __fdiv_rn(ez, s);
    }
}

__global__ void __launch_bounds__(RT_THREADS)
    k_topk_softmax_bwd(const float *__restrict__ g_probs, const float *__restrict__ probs,
                       const int32_t *__restrict__ idx, int64_t T, int E, int K,
                       float *__restrict__ g_logits)
{
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * RT_WARPS + (threadIdx.x >> 5);
    if (t >= T) return;
    float *gl = g_logits + t * E;
    for (int e = lane; e < E; e += 32) gl[e] = 0.0f;
    const float p = lane < K ? __ldg(probs + t * K + lane) : 0.0f;
    const float g = lane < K ? __ldg(g_probs + t * K + lane) : 0.0f;
    const int32_t ex = lane < K ? __ldg(idx + t * K + lane) : -1;
    float dsum = 0.0f;
    for (int k = 0; k < K; ++k)
        dsum = __fmaf_rn(__shfl_sync(FULL_MASK, p, k), __shfl_sync(FULL_MASK, g, k), dsum);
    __syncwarp();  // the zeros above land before the picked gradients
    if (lane < K && ex >= 0 && ex < E) gl[ex] = __fmul_rn(p, __fsub_rn(g, dsum));
}

}  // namespace
}  // namespace mp

using namespace mp;

extern "C" mp_status_t mp_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t K,
                                       int32_t n_groups, int32_t topk_groups, int32_t *idx,
                                       float *probs, mp_stream_t stream)
{
    if (T < 0 || E < 1 || K < 1 || n_groups < 1 || topk_groups < 1) return MP_ERR_INVALID_ARG;
    if (E > MP_MAX_EXPERTS || K > 32 || n_groups > 32) return MP_ERR_UNSUPPORTED;
    if (E % n_groups != 0 || topk_groups > n_groups ||
        (int64_t)topk_groups * (E / n_groups) < K || K > E)
        return MP_ERR_INVALID_ARG;
    if (T == 0) return MP_OK;
    if (logits == nullptr || idx == nullptr || probs == nullptr) return MP_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((T + RT_WARPS - 1) / RT_WARPS);
    cudaStream_t s = as_stream(stream);
    const int per = (E + 31) / 32;   // logits per lane
    if (per <= 4 && K == 8)
        (void)launch_pdl(k_topk_softmax<4, 8>, blocks, RT_THREADS, 0, s, logits, T, E, K,
                         n_groups, topk_groups, idx, probs);
    else if (per <= 8 && K == 8)
        (void)launch_pdl(k_topk_softmax<8, 8>, blocks, RT_THREADS, 0, s, logits, T, E, K,
                         n_groups, topk_groups, idx, probs);
    else if (per <= 4)
        (void)launch_pdl(k_topk_softmax<4>, blocks, RT_THREADS, 0, s, logits, T, E, K,
                         n_groups, topk_groups, idx, probs);
    else if (per <= 8)
        (void)launch_pdl(k_topk_softmax<8>, blocks, RT_THREADS, 0, s, logits, T, E, K,
                         n_groups, topk_groups, idx, probs);
    else if (per <= 16)
        (void)launch_pdl(k_topk_softmax<16>, blocks, RT_THREADS, 0, s, logits, T, E, K,
                         n_groups, topk_groups, idx, probs);
    else
        (void)launch_pdl(k_topk_softmax<32>, blocks, RT_THREADS, 0, s, logits, T, E, K,
                         n_groups, topk_groups, idx, probs);
    return check_launch();
}

extern "C" mp_status_t mp_topk_softmax_bwd(const float *g_probs, const float *probs,
                                           const int32_t *idx, int64_t T, int32_t E, int32_t K,
                                           float *g_logits, mp_stream_t stream)
{
    if (T < 0 || E < 1 || K < 1) return MP_ERR_INVALID_ARG;
    if (K > 32 || E > MP_MAX_EXPERTS) return MP_ERR_UNSUPPORTED;
    if (T == 0) return MP_OK;
    if (g_probs == nullptr || probs == nullptr || idx == nullptr || g_logits == nullptr)
        return MP_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((T + RT_WARPS - 1) / RT_WARPS);
    (void)launch_pdl(k_topk_softmax_bwd, blocks, RT_THREADS, 0, as_stream(stream), g_probs, probs,
                     idx, T, E, K, g_logits);
    return check_launch();
}
