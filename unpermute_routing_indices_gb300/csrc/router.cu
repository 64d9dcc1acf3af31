// Fused top-k softmax router: the routing input of the map, from logits.
//
// "moe-ops 0.1.0" README, "Operators": fused_topk_softmax fuses the top-K
// selection and the softmax normalisation in registers, and its backward
// computes the exact softmax gradient scattered back to the logits.  The
// group-limited choice (keep the best groups of experts first) follows the
// large routed workload of the pages' configurations.
//
// k_topk_softmax: one warp per token; lane l holds logits l, l+32, ... (so
// every load instruction reads 32 consecutive floats).  Group scores are warp
// max-reductions; the K picks are K warp arg-max reductions on (logit desc,
// expert asc), lane k keeping pick k.  The softmax runs in fp32: z_k = l_k -
// l_0, expf (full accuracy), the sum in slot order, IEEE division.
// k_topk_softmax_bwd: one warp per token: zero the token's E gradients, then
// p_k * (g_k - sum_j p_j g_j) at the picked experts.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace mp {
namespace {

constexpr int RT_THREADS = 256;
constexpr int RT_WARPS = RT_THREADS / 32;

// (value, index) arg-max across the warp: larger value, then smaller index.
__device__ __forceinline__ void warp_argmax(float &v, int &i)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL_MASK, v, o);
        const int oi = __shfl_xor_sync(FULL_MASK, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, o));
    return v;
}

template <int PER>
__global__ void __launch_bounds__(RT_THREADS)
    k_topk_softmax(const float *__restrict__ logits, int64_t T, int E, int K, int n_groups,
                   int topk_groups, int32_t *__restrict__ idx, float *__restrict__ probs)
{
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

    if (n_groups > 1) {
        const int per_group = E / n_groups;
        unsigned group_kept = 0;   // bit g: group g kept (same in every lane)
        float score_g = -FLT_MAX;  // lane g holds group g's score
        for (int g = 0; g < n_groups; ++g) {
            float m = -FLT_MAX;
            bool any = false;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int e = lane + 32 * j;
                if ((live >> j & 1u) && e / per_group == g) {
                    m = any ? fmaxf(m, v[j]) : v[j];
                    any = true;
                }
            }
            m = warp_max(m);
            if (lane == g) score_g = m;
        }
        for (int j = 0; j < topk_groups; ++j) {
            float sv = (lane < n_groups && !(group_kept >> lane & 1u)) ? score_g : -FLT_MAX;
            int si = (lane < n_groups && !(group_kept >> lane & 1u)) ? lane : INT_MAX;
            warp_argmax(sv, si);
            group_kept |= 1u << si;
        }
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane + 32 * j;
            if ((live >> j & 1u) && !(group_kept >> (e / per_group) & 1u)) live &= ~(1u << j);
        }
    }

    float my_v = 0.0f;
    int my_i = -1;
    for (int k = 0; k < K; ++k) {
        float bv = -FLT_MAX;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane + 32 * j;
            if ((live >> j & 1u) && (bi == INT_MAX || v[j] > bv)) {
                bv = v[j];
                bi = e;
            }
        }
        warp_argmax(bv, bi);
        if (bi != INT_MAX && (bi & 31) == lane) live &= ~(1u << (bi >> 5));
        if (lane == (k & 31) && k < 32) {
            my_v = bv;
            my_i = bi;
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
    if (per <= 4)
        k_topk_softmax<4><<<blocks, RT_THREADS, 0, s>>>(logits, T, E, K, n_groups, topk_groups,
                                                        idx, probs);
    else if (per <= 8)
        k_topk_softmax<8><<<blocks, RT_THREADS, 0, s>>>(logits, T, E, K, n_groups, topk_groups,
                                                        idx, probs);
    else if (per <= 16)
        k_topk_softmax<16><<<blocks, RT_THREADS, 0, s>>>(logits, T, E, K, n_groups, topk_groups,
                                                         idx, probs);
    else
        k_topk_softmax<32><<<blocks, RT_THREADS, 0, s>>>(logits, T, E, K, n_groups, topk_groups,
                                                         idx, probs);
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
    k_topk_softmax_bwd<<<blocks, RT_THREADS, 0, as_stream(stream)>>>(g_probs, probs, idx, T, E, K,
                                                                     g_logits);
    return check_launch();
}
