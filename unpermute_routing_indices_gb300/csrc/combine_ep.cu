// Rank-ordered combine over expert-parallel ranks, on one GPU.
//
// "core.transformer.moe.batch_invariant" (Megatron-Core API docs) defines the
// batch-invariant unpermute over EP ranks: accumulation is token-owned and
// adds contributions by EP rank, then top-k slot (unpermute); each rank's
// partial is the slot-order chain of FP32 fused multiply-adds of probability
// and row from zero, optionally quantized to BF16 (BF16_RANK_PARTIALS,
// unpermute_with_bf16_rank_partials), and the ranks are added in rank order,
// optionally in FP64 (CROSS_RANK_FP64, _rank_tree_unpermute_kernel).  Here the
// EP ranks are simulated: rank r owns experts [r*E/ep, (r+1)*E/ep).
//
// k_unpermute_ep_token (rows of 1,024 elements or more, K <= 8): one token
// per CTA of 128 threads.  k_unpermute_ep (shorter rows, odd H, or K <= 16):
// one group of tpt threads per token.  Both: one 16-byte vector (8 elements)
// per thread per pass.  Each thread sorts the token's K slots by (rank, slot)
// once, with a fixed sorting network on registers.  Per pass it copies its slots' row vectors into
// shared memory (cp.async; the element path for odd H keeps them in
// registers), reads them back in
// sorted order and runs one fused multiply-add chain that hands the rank's
// partial to the cross-rank sum at each rank's last slot: K FMAs per element
// whatever the number of ranks.  A rank with no
// routed slot would add +0 to an accumulator that is never -0, so skipping it
// changes no bit.  GB300 runs FP64 at a small fraction of its FP32 rate, so
// the fp64 cross-rank forms bracket the fp64 sum between two fp32 sums
// rounded toward -inf and +inf; where both round to the same bf16 value that
// is the result, and only the rare elements whose bracket holds a bf16
// midpoint take fp64 additions.  Those forms run the FMA chains and the
// bracket on packed fp32 pairs (f32x2: two elements per instruction, each
// rounded as the scalar operation would be).  Without the fp64 sum, bf16
// partials are added to their fp32 sum by a mixed-precision add
// (add.rn.f32.bf16: the bf16 operand widened exactly, one fp32 rounding),
// with no separate widening step.
#include <climits>

#include "common.cuh"

namespace mp {
namespace {

constexpr int EP_THREADS = 128;
constexpr int EP_THREADS_LOG2 = 7;
static_assert((1 << EP_THREADS_LOG2) == EP_THREADS, "EP_THREADS is a power of two");
constexpr int EP_KMAX = 16;   // slots per token: kernels for K <= 8 and for K <= 16


// fp64 -> bf16, round to nearest even, in a single rounding, from the binary64
// fields: keep the top 8 significant bits (1 + 7) for normal bf16 results, or
// the bits at or above the 2^-133 quantum for subnormal ones; a carry out of
// the kept bits moves to the next binade (and to +-inf past 2^128).
__device__ __forceinline__ uint16_t bf16_from_f64(double d)
{
    const uint64_t u = static_cast<uint64_t>(__double_as_longlong(d));
    const uint16_t sign = static_cast<uint16_t>((u >> 48) & 0x8000u);
    const int ex = static_cast<int>((u >> 52) & 0x7ff);
    const uint64_t mant = u & 0xFFFFFFFFFFFFFull;
    if (ex == 0x7ff) return mant ? 0x7fc0 : static_cast<uint16_t>(sign | 0x7f80u);
    if (ex == 0) return sign;  // zero, or far below half the smallest bf16 subnormal
    const int e = ex - 1023;   // value = 1.mant * 2^e
    if (e > 127) return static_cast<uint16_t>(sign | 0x7f80u);
    const uint64_t full = (1ull << 52) | mant;
    if (e >= -126) {
        uint64_t keep = full >> 45;
        const uint64_t rest = full & ((1ull << 45) - 1), half = 1ull << 44;
        if (rest > half || (rest == half && (keep & 1u))) keep += 1;
        return static_cast<uint16_t>(sign | (((uint32_t)(e + 127) << 7) + (uint32_t)(keep - 128)));
    }
    const int s = -81 - e;  // shift to the 2^-133 quantum (>= 46 here)
    if (s >= 54) return sign;
    uint64_t keep = full >> s;
    const uint64_t rest = full & ((1ull << s) - 1), half = 1ull << (s - 1);
    if (rest > half || (rest == half && (keep & 1u))) keep += 1;
    return static_cast<uint16_t>(sign | keep);
}

__device__ __forceinline__ uint4 pack_bits(const uint16_t (&b)[8])
{
    return make_uint4((uint32_t)b[0] | ((uint32_t)b[1] << 16),
                      (uint32_t)b[2] | ((uint32_t)b[3] << 16),
                      (uint32_t)b[4] | ((uint32_t)b[5] << 16),
                      (uint32_t)b[6] | ((uint32_t)b[7] << 16));
}

__device__ __forceinline__ uint16_t pack_bits(const uint16_t (&b)[1]) { return b[0]; }

// Packed pairs of fp32 (the f32x2 arithmetic of sm_100 and later): one
// instruction rounds each half exactly as the scalar operation would.
__device__ __forceinline__ uint64_t f2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// The same add rounded toward -inf (rm) and toward +inf (rp).
__device__ __forceinline__ uint64_t add2_rm(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rm.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add2_rp(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rp.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// a0 += bf16 lo half of w, a1 += bf16 hi half (each one fp32 rounding, the
// bf16 operand widened exactly, as in a plain fp32 add of the widened value).
__device__ __forceinline__ void add_bf16x2(uint32_t w, float &a0, float &a1)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(w));
}
// The two bf16 of a 32-bit word as a pair of fp32 (exact).
__device__ __forceinline__ uint64_t bf16x2_wide(uint32_t w) { return f2(bf16_lo(w), bf16_hi(w)); }

// Compare-exchange on (key, row, prob) triples, smaller key first.
__device__ __forceinline__ void cx(int32_t &ka, int32_t &ra, float &pa, int32_t &kb, int32_t &rb,
                                   float &pb)
{
    const bool sw = kb < ka;
    const int32_t k0 = sw ? kb : ka, k1 = sw ? ka : kb;
    const int32_t r0 = sw ? rb : ra, r1 = sw ? ra : rb;
    const float p0 = sw ? pb : pa, p1 = sw ? pa : pb;
    ka = k0; kb = k1; ra = r0; rb = r1; pa = p0; pb = p1;
}

// Batcher's odd-even merge sort of 8 keys (19 comparators, fixed indices).
__device__ __forceinline__ void sort8(int32_t (&k)[8], int32_t (&r)[8], float (&p)[8])
{
#define MP_CX(a, b) cx(k[a], r[a], p[a], k[b], r[b], p[b])
    MP_CX(0, 1); MP_CX(2, 3); MP_CX(4, 5); MP_CX(6, 7);
    MP_CX(0, 2); MP_CX(1, 3); MP_CX(4, 6); MP_CX(5, 7);
    MP_CX(1, 2); MP_CX(5, 6);
    MP_CX(0, 4); MP_CX(1, 5); MP_CX(2, 6); MP_CX(3, 7);
    MP_CX(2, 4); MP_CX(3, 5);
    MP_CX(1, 2); MP_CX(3, 4); MP_CX(5, 6);
#undef MP_CX
}

// The same merge sort for any power-of-two N (63 comparators for 16; every
// index a compile-time constant once unrolled).  N = 8 uses the hand-ordered
// network above, which the compiler schedules into fewer registers.
template <int N>
__device__ __forceinline__ void sort_slots(int32_t (&k)[N], int32_t (&r)[N], float (&p)[N])
{
    if constexpr (N == 8) {
        sort8(k, r, p);
    } else {
#pragma unroll
        for (int w = 1; w < N; w <<= 1)
#pragma unroll
            for (int q = w; q >= 1; q >>= 1)
#pragma unroll
                for (int j = q % w; j + q < N; j += 2 * q)
#pragma unroll
                    for (int i = 0; i < q; ++i)
                        if (i + j + q < N && (i + j) / (2 * w) == (i + j + q) / (2 * w))
                            cx(k[i + j], r[i + j], p[i + j], k[i + j + q], r[i + j + q],
                               p[i + j + q]);
    }
}

// Walks the token's slots sorted by (rank, slot): a slot-order chain of fused
// multiply-adds (plain adds without probs) from +0 per rank, and add(e, p) at
// each rank's last slot with the rank's partial p for element e (rounded to
// bf16 if BF16P).  `valid` / `last` are bit masks over the sorted positions.
template <bool PROBS, bool BF16P, int L, int KM, typename Get, typename Add>
__device__ __forceinline__ void walk_ranks(Get row, const float (&p)[KM], unsigned valid,
                                           unsigned last, Add add)
{
    float part[L];
#pragma unroll
    for (int e = 0; e < L; ++e) part[e] = 0.0f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (!(valid >> j & 1u)) continue;
        float f[L];
        unpack(row(j), f);
#pragma unroll
        for (int e = 0; e < L; ++e)
            part[e] = PROBS ? __fmaf_rn(p[j], f[e], part[e]) : __fadd_rn(part[e], f[e]);
        if (last >> j & 1u) {
#pragma unroll
            for (int e = 0; e < L; ++e) {
                add(e, BF16P ? __bfloat162float(__float2bfloat16_rn(part[e])) : part[e]);
                part[e] = 0.0f;
            }
        }
    }
}

// walk_ranks on packed pairs: the four element pairs of a 16-byte vector;
// row(j) gives the vector of sorted slot j.
template <bool PROBS, int KM, typename Get, typename Add>
__device__ __forceinline__ void walk_ranks2(Get row, const float (&p)[KM], unsigned valid,
                                            unsigned last, Add add)
{
    uint64_t part[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) part[i] = 0;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (!(valid >> j & 1u)) continue;
        const uint4 v = row(j);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const uint64_t pp = f2(p[j], p[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            part[i] = PROBS ? fma2(pp, bf16x2_wide(w[i]), part[i])
                            : add2(part[i], bf16x2_wide(w[i]));
        if (last >> j & 1u) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                add(i, part[i]);
                part[i] = 0;
            }
        }
    }
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Element e of a vector as fp32 (exact).
__device__ __forceinline__ float elem(const uint4 &v, int e)
{
    const uint32_t w = e < 2 ? v.x : (e < 4 ? v.y : (e < 6 ? v.z : v.w));
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}
__device__ __forceinline__ float elem(uint16_t v, int)
{
    return __uint_as_float((uint32_t)v << 16);
}

__device__ __forceinline__ uint32_t bf16_bits(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// The fp64 cross-rank combine of element e by its definition: per rank the
// slot-order fp32 chain from +0 (rounded to bf16 if BF16P), the partials added
// in rank order to an fp64 sum from +0, rounded once to bf16.
template <bool PROBS, bool BF16P, int KM, typename Get>
__device__ __forceinline__ uint16_t rank_sum_f64(Get row, const float (&p)[KM], unsigned valid,
                                                 unsigned last, int e)
{
    double acc = 0.0;
    float part = 0.0f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (!(valid >> j & 1u)) continue;
        const float f = elem(row(j), e);
        part = PROBS ? __fmaf_rn(p[j], f, part) : __fadd_rn(part, f);
        if (last >> j & 1u) {
            const float q = BF16P ? __bfloat162float(__float2bfloat16_rn(part)) : part;
            acc = __dadd_rn(acc, (double)q);
            part = 0.0f;
        }
    }
    return bf16_from_f64(acc);
}

// Shared memory a CTA stages its rows in: on 16-byte vectors, KM slots x
// EP_THREADS vectors per buffer, two buffers for K <= 8 and one for K <= 16.
__host__ __device__ constexpr int ep_stage_bufs(int km) { return km > 8 ? 1 : 2; }
template <typename V, int KM>
constexpr size_t ep_stage_bytes()
{
    return Lanes<V>::N == 8 ? (size_t)ep_stage_bufs(KM) * KM * EP_THREADS * 16 : 0;
}

// CTAs per SM each form of the general kernel is compiled for (registers are
// capped to fit; the two 16 KB stage buffers allow 6).  On the skewed
// T=16384, ep=8 combine (before the one-token kernel took those rows), 6 CTAs
// gave fp32 174 us, bf16 partials 183, fp64 sum 194 (fp32 partials) / 197
// (bf16 partials); 5 CTAs the same within 1%.  With up to 16 slots: 2 CTAs
// per SM (rare shapes; correctness first).
constexpr int ep_min_blocks(int km) { return km > 8 ? 2 : 6; }

// A token's K map entries, expert ids and probabilities as loaded.
template <int KM>
struct EpRaw {
    int32_t row[KM], expert[KM];
    float p[KM];
};

// The token's routed slots sorted by (rank, slot), unrouted slots last: the
// row and probability of each sorted position, and bit masks over the sorted
// positions of the routed slots (valid) and of each rank's last slot (last).
template <int KM>
struct EpSlots {
    int32_t rk[KM];
    float pk[KM];
    unsigned valid, last;
};

template <bool PROBS, int KM>
__device__ __forceinline__ void ep_load(EpRaw<KM> &r, const int32_t *__restrict__ map,
                                        const int32_t *__restrict__ idx,
                                        const float *__restrict__ probs, int64_t t, int K)
{
#pragma unroll
    for (int i = 0; i < KM; ++i) {
        const bool in = i < K;
        r.row[i] = in ? __ldg(map + t * K + i) : -1;
        r.expert[i] = in ? __ldg(idx + t * K + i) : 0;
        r.p[i] = (PROBS && in) ? __ldg(probs + t * K + i) : 1.0f;
    }
}

template <int KM>
__device__ __forceinline__ void ep_prepare(const EpRaw<KM> &r, int per_rank, EpSlots<KM> &s)
{
    int32_t key[KM];
#pragma unroll
    for (int i = 0; i < KM; ++i) {
        int32_t rank = r.expert[i] / per_rank;
        rank = rank < -(1 << 20) ? -(1 << 20) : (rank > (1 << 20) ? (1 << 20) : rank);
        key[i] = r.row[i] >= 0 ? rank * KM + i : INT_MAX;
        s.rk[i] = r.row[i];
        s.pk[i] = r.p[i];
    }
    sort_slots<KM>(key, s.rk, s.pk);
    s.valid = 0;
    s.last = 0;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (key[j] == INT_MAX) continue;
        s.valid |= 1u << j;
        const bool next_same = j + 1 < KM && key[j + 1] != INT_MAX &&
                               (key[j + 1] - (key[j + 1] & (KM - 1))) ==
                                   (key[j] - (key[j] & (KM - 1)));
        if (!next_same) s.last |= 1u << j;
    }
}

// One output vector of the rank-ordered combine; row(j) gives the vector of
// sorted slot j.
template <typename V, bool PROBS, bool BF16P, bool FP64, int KM, typename Get>
__device__ __forceinline__ V ep_vec(Get row, const EpSlots<KM> &s)
{
    constexpr int L = Lanes<V>::N;
    if constexpr (FP64) {
        // The fp64 cross-rank sum, rounded once to bf16, without fp64
        // arithmetic on the common path.  The partials are summed in rank
        // order twice in fp32, every add rounded toward -inf (lo) and toward
        // +inf (hi).  Then lo <= s <= hi for the fp64 sum s, by induction
        // over the adds: a float rounded down (up) from x is an fp64 value
        // <= x (>= x), so rounding x to the nearest fp64 value cannot pass
        // it.  Rounding to bf16 is monotone, so where lo and hi round to the
        // same bf16 value, and it is not NaN, that is the bf16 of s.  An
        // element whose bracket holds a bf16 midpoint (about 1 in 10^4 on
        // N(0,1) rows), or that cancels exactly (lo = -0 where s is +0), or
        // meets inf or NaN, takes the definition itself: fp64 adds in rank
        // order, per element.  On 16-byte vectors the walk runs on packed
        // fp32 pairs.
        uint16_t bits[L];
        unsigned open = 0;   // elements whose bracket does not decide
        if constexpr (L == 8) {
            uint64_t lo2[4], hi2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) lo2[i] = hi2[i] = 0;
            walk_ranks2<PROBS, KM>(row, s.pk, s.valid, s.last, [&](int i, uint64_t p) {
                if constexpr (BF16P) {
                    float lo, hi;
                    f2_split(p, lo, hi);
                    p = bf16x2_wide(pack_bf16x2(lo, hi));
                }
                lo2[i] = add2_rm(lo2[i], p);
                hi2[i] = add2_rp(hi2[i], p);
            });
            bool any = false;
            uint32_t wl[4], wh[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float l0, l1, h0, h1;
                f2_split(lo2[i], l0, l1);
                f2_split(hi2[i], h0, h1);
                wl[i] = pack_bf16x2(l0, l1);
                wh[i] = pack_bf16x2(h0, h1);
                bits[2 * i] = static_cast<uint16_t>(wl[i] & 0xffffu);
                bits[2 * i + 1] = static_cast<uint16_t>(wl[i] >> 16);
                any |= wl[i] != wh[i] ||
                       max_u16x2(wl[i] & 0x7fff7fffu, 0x7f807f80u) != 0x7f807f80u;
            }
            if (any) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t a = (e & 1) ? wl[e / 2] >> 16 : wl[e / 2] & 0xffffu;
                    const uint32_t b = (e & 1) ? wh[e / 2] >> 16 : wh[e / 2] & 0xffffu;
                    if (a != b || (a & 0x7fffu) > 0x7f80u) open |= 1u << e;
                }
            }
        } else {
            float lo[L], hi[L];
#pragma unroll
            for (int e = 0; e < L; ++e) lo[e] = hi[e] = 0.0f;
            walk_ranks<PROBS, BF16P, L, KM>(row, s.pk, s.valid, s.last, [&](int e, float p) {
                lo[e] = __fadd_rd(lo[e], p);
                hi[e] = __fadd_ru(hi[e], p);
            });
#pragma unroll
            for (int e = 0; e < L; ++e) {
                const uint32_t a = bf16_bits(lo[e]), b = bf16_bits(hi[e]);
                bits[e] = static_cast<uint16_t>(a);
                if (a != b || (a & 0x7fffu) > 0x7f80u) open |= 1u << e;
            }
        }
        if (open) {
#pragma unroll
            for (int e = 0; e < L; ++e)
                if (open >> e & 1u)
                    bits[e] = rank_sum_f64<PROBS, BF16P, KM>(row, s.pk, s.valid, s.last, e);
        }
        return pack_bits(bits);
    } else {
        float acc[L];
#pragma unroll
        for (int e = 0; e < L; ++e) acc[e] = 0.0f;
        if constexpr (BF16P && L == 8) {
            walk_ranks2<PROBS, KM>(row, s.pk, s.valid, s.last, [&](int i, uint64_t p) {
                float lo, hi;
                f2_split(p, lo, hi);
                add_bf16x2(pack_bf16x2(lo, hi), acc[2 * i], acc[2 * i + 1]);
            });
        } else {
            walk_ranks<PROBS, BF16P, L, KM>(row, s.pk, s.valid, s.last,
                                            [&](int e, float p) { acc[e] = __fadd_rn(acc[e], p); });
        }
        return pack(acc);
    }
}

// Copies this thread's vector cc of every routed sorted slot into its column
// of a stage buffer (cp.async, 16 bytes each), as one commit group.
template <int KM>
__device__ __forceinline__ void ep_issue(uint4 *buf, const uint4 *__restrict__ rows,
                                         const EpSlots<KM> &s, int nvec, int cc)
{
    uint4 *const dst = buf + threadIdx.x;
#pragma unroll
    for (int i = 0; i < KM; ++i)
        if (s.valid >> i & 1u)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                         ::"r"(smem_u32(dst + i * EP_THREADS)),
                           "l"(rows + (int64_t)s.rk[i] * nvec + cc)
                         : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <typename V, bool PROBS, bool BF16P, bool FP64, int KM>
__global__ void __launch_bounds__(EP_THREADS, ep_min_blocks(KM))
    k_unpermute_ep(const V *__restrict__ rows, const float *__restrict__ probs,
                   const int32_t *__restrict__ map, const int32_t *__restrict__ idx, int64_t T,
                   int K, int nvec, int tpt_log2, int per_rank, V *__restrict__ out)
{
    pdl_trigger();
    pdl_wait();
    constexpr int L = Lanes<V>::N;
    const int tpt = 1 << tpt_log2;
    const int lane = threadIdx.x & (tpt - 1);
    const int64_t t = (int64_t)blockIdx.x * (EP_THREADS >> tpt_log2) + (threadIdx.x >> tpt_log2);
    if (t >= T) return;

    EpSlots<KM> sl;
    {
        EpRaw<KM> raw;
        ep_load<PROBS, KM>(raw, map, idx, probs, t, K);
        ep_prepare<KM>(raw, per_rank, sl);
    }
    // On 16-byte vectors each pass's rows are staged in shared memory
    // (cp.async, 16 bytes per copy) instead of registers, two passes deep:
    // the copies of pass p + 1 are issued before pass p is computed.  Each
    // thread copies and reads back only its own slots, so no barrier is
    // needed; the registers the rows would hold go to more resident warps.
    constexpr bool STAGE = L == 8;
    constexpr int NBUF = STAGE ? ep_stage_bufs(KM) : 1;
    extern __shared__ uint4 ep_stage[];   // [NBUF][KM][EP_THREADS] when STAGE
    const auto *const vrows = reinterpret_cast<const uint4 *>(rows);
    if constexpr (STAGE && NBUF == 2)
        if (lane < nvec) ep_issue<KM>(ep_stage, vrows, sl, nvec, lane);
    int pass = 0;
    for (int c0 = 0; c0 < nvec; c0 += tpt, ++pass) {
        const int c = c0 + lane;
        V r[KM];
        if constexpr (STAGE) {
            if (c >= nvec) break;
            if constexpr (NBUF == 2) {
                if (c + tpt < nvec) {
                    ep_issue<KM>(ep_stage + ((pass + 1) & 1) * KM * EP_THREADS, vrows, sl, nvec,
                                 c + tpt);
                    asm volatile("cp.async.wait_group 1;" ::: "memory");
                } else {
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                }
            } else {
                ep_issue<KM>(ep_stage, vrows, sl, nvec, c);
            }
        } else {
#pragma unroll
            for (int i = 0; i < KM; ++i)
                r[i] = ((sl.valid >> i & 1u) && c < nvec)
                           ? ld_stream(rows + (int64_t)sl.rk[i] * nvec + c) : zero_vec<V>();
        }
        uint4 *const mine = ep_stage + (pass & (NBUF - 1)) * KM * EP_THREADS + threadIdx.x;
        const auto row = [&](int j) -> V {
            if constexpr (STAGE) return mine[j * EP_THREADS];
            else return r[j];
        };
        if constexpr (FP64 && NBUF == 1) {
            // the fp64 forms without a second stage buffer compute long
            // enough per pass to hide an L2 fill of the next pass's rows
            const int cn = c + tpt;
#pragma unroll
            for (int i = 0; i < KM; ++i)
                if ((sl.valid >> i & 1u) && cn < nvec)
                    asm volatile("prefetch.global.L2 [%0];"
                                 ::"l"(rows + (int64_t)sl.rk[i] * nvec + cn));
        }
        if constexpr (STAGE && NBUF == 1) asm volatile("cp.async.wait_group 0;" ::: "memory");
        const V v = ep_vec<V, PROBS, BF16P, FP64, KM>(row, sl);
        if (c < nvec) st_row(out + t * nvec + c, v);
    }
}

// One token per CTA, for rows of EP_THREADS 16-byte vectors or more with
// K <= 8: the CTA's threads cover the row in passes of EP_THREADS vectors,
// and the token index is the block index.  The token's slot data is then the
// same in every thread of the CTA, and the kernel has no token-group
// arithmetic.  The fp32-sum forms keep two stage buffers (the next pass's
// copies in flight while this one computes) at 6 CTAs per SM.  The fp64
// forms need fewer registers here (60 against 76-78), and run one stage
// buffer at 8 CTAs per SM: each pass's copies are waited for at once, while
// the next pass's rows are prefetched into L2, so that its copies hit in L2.
// One thread issues that prefetch as one bulk prefetch per slot (the pass's
// vectors of a row are contiguous), which costs the other warps no issue
// slots; a prefetch.global.L2 per thread and slot cost 8 instructions per
// warp and pass.  Measured on the skewed T=16384, H=4096, ep=8 combine,
// against the general kernel: fp32 174.5 -> 171.5 us, bf16 partials
// 183.5 -> 174.7, fp64 sum with fp32 / bf16 partials 192.9 / 200.0 -> 178.7
// / 181.6 (per-thread prefetches: 179.3 / 187.0; two buffers at 6 CTAs:
// 186.4 / 197.4; one buffer at 7, 9 or 10 CTAs: 181.8-190.1 / 187.0-202.9).
template <bool FP64>
__host__ __device__ constexpr int ep_token_bufs() { return FP64 ? 1 : 2; }
template <bool FP64>
constexpr size_t ep_token_stage_bytes() { return (size_t)ep_token_bufs<FP64>() * 8 * EP_THREADS * 16; }

template <bool PROBS, bool BF16P, bool FP64>
__global__ void __launch_bounds__(EP_THREADS, FP64 ? 8 : 6)
    k_unpermute_ep_token(const uint4 *__restrict__ rows, const float *__restrict__ probs,
                         const int32_t *__restrict__ map, const int32_t *__restrict__ idx,
                         int64_t T, int K, int nvec, int per_rank, uint4 *__restrict__ out)
{
    constexpr int KM = 8;
    pdl_trigger();
    pdl_wait();
    const int64_t t = blockIdx.x;
    if (t >= T) return;
    const int lane = threadIdx.x;
    extern __shared__ uint4 ep_stage[];   // [ep_token_bufs][KM][EP_THREADS]

    EpSlots<KM> sl;
    {
        EpRaw<KM> raw;
        ep_load<PROBS, KM>(raw, map, idx, probs, t, K);
        ep_prepare<KM>(raw, per_rank, sl);
    }
    const uint4 *const mine0 = ep_stage + threadIdx.x;
    if constexpr (ep_token_bufs<FP64>() == 1) {
        for (int c = lane; c < nvec; c += EP_THREADS) {
            ep_issue<KM>(ep_stage, rows, sl, nvec, c);
            // the next pass's rows, one contiguous run of up to EP_THREADS
            // vectors per slot, prefetched into L2 by one thread (bulk
            // prefetches: 16-byte aligned, whole vectors)
            const int cn0 = c - lane + EP_THREADS;
            if (threadIdx.x == 0 && cn0 < nvec) {
                const int nbytes = (nvec - cn0 < EP_THREADS ? nvec - cn0 : EP_THREADS) * 16;
#pragma unroll
                for (int i = 0; i < KM; ++i)
                    if (sl.valid >> i & 1u)
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                                     ::"l"(rows + (int64_t)sl.rk[i] * nvec + cn0), "r"(nbytes)
                                     : "memory");
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            const uint4 v = ep_vec<uint4, PROBS, BF16P, FP64, KM>(
                [&](int j) -> uint4 { return mine0[j * EP_THREADS]; }, sl);
            st_row(out + t * nvec + c, v);
        }
    } else {
        ep_issue<KM>(ep_stage, rows, sl, nvec, lane);   // lane < EP_THREADS <= nvec
        int pass = 0;   // stage buffer pass & 1
        for (int c = lane; c - lane < nvec; c += EP_THREADS, ++pass) {
            if (c - lane + EP_THREADS < nvec) {
                // the next pass's copies (an empty group for a thread past the row)
                if (c + EP_THREADS < nvec)
                    ep_issue<KM>(ep_stage + ((pass + 1) & 1) * KM * EP_THREADS, rows, sl, nvec,
                                 c + EP_THREADS);
                else
                    asm volatile("cp.async.commit_group;" ::: "memory");
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            if (c < nvec) {
                const uint4 *const mine = mine0 + (pass & 1) * KM * EP_THREADS;
                const uint4 v = ep_vec<uint4, PROBS, BF16P, FP64, KM>(
                    [&](int j) -> uint4 { return mine[j * EP_THREADS]; }, sl);
                st_row(out + t * nvec + c, v);
            }
        }
    }
}

template <typename V, bool PROBS, bool BF16P, bool FP64, int KM>
void launch_ep(const void *rows, const float *probs, const int32_t *map, const int32_t *idx,
               int64_t T, int K, int nvec, int per_rank, void *out, cudaStream_t s)
{
    int l = ceil_log2(nvec < 1 ? 1 : nvec);
    const int lmax = ceil_log2(EP_THREADS);
    if (l > lmax) l = lmax;
    const int64_t per_block = EP_THREADS >> l;
    const unsigned blocks = (unsigned)((T + per_block - 1) / per_block);
    const size_t smem = ep_stage_bytes<V, KM>();
    if constexpr (Lanes<V>::N == 8 && KM == 8) {
        if (nvec >= EP_THREADS) {
            (void)launch_pdl(k_unpermute_ep_token<PROBS, BF16P, FP64>, (unsigned)T, EP_THREADS,
                             ep_token_stage_bytes<FP64>(), s, (const uint4 *)rows, probs, map,
                             idx, T, K, nvec, per_rank, (uint4 *)out);
            return;
        }
    }
    (void)launch_pdl(k_unpermute_ep<V, PROBS, BF16P, FP64, KM>, blocks, EP_THREADS, smem, s,
        (const V *)rows, probs, map, idx, T, K, nvec, l, per_rank, (V *)out);
}

template <typename V, bool PROBS, int KM>
void launch_ep_km(int flags, const void *rows, const float *probs, const int32_t *map,
                  const int32_t *idx, int64_t T, int K, int nvec, int per_rank, void *out,
                  cudaStream_t s)
{
    const bool b = flags & MP_EP_BF16_PARTIALS, d = flags & MP_EP_FP64_CROSS_RANK;
    if (b && d)
        launch_ep<V, PROBS, true, true, KM>(rows, probs, map, idx, T, K, nvec, per_rank, out, s);
    else if (b)
        launch_ep<V, PROBS, true, false, KM>(rows, probs, map, idx, T, K, nvec, per_rank, out, s);
    else if (d)
        launch_ep<V, PROBS, false, true, KM>(rows, probs, map, idx, T, K, nvec, per_rank, out, s);
    else
        launch_ep<V, PROBS, false, false, KM>(rows, probs, map, idx, T, K, nvec, per_rank, out,
                                              s);
}

template <typename V, bool PROBS>
void launch_ep_flags(int flags, const void *rows, const float *probs, const int32_t *map,
                     const int32_t *idx, int64_t T, int K, int nvec, int per_rank, void *out,
                     cudaStream_t s)
{
    if (K <= 8)
        launch_ep_km<V, PROBS, 8>(flags, rows, probs, map, idx, T, K, nvec, per_rank, out, s);
    else
        launch_ep_km<V, PROBS, 16>(flags, rows, probs, map, idx, T, K, nvec, per_rank, out, s);
}

}  // namespace
}  // namespace mp

using namespace mp;

extern "C" mp_status_t mp_unpermute_ep(const mp_bf16_t *rows, const float *probs,
                                       const int32_t *row_id_map, const int32_t *idx, int64_t T,
                                       int32_t K, int32_t H, int32_t E, int32_t ep_size,
                                       int32_t flags, mp_bf16_t *out, mp_stream_t stream)
{
    if (T < 0 || K < 1 || H < 1 || E < 1 || ep_size < 1 || T * (int64_t)K > INT32_MAX)
        return MP_ERR_INVALID_ARG;
    if (E % ep_size != 0 || (flags & ~(MP_EP_BF16_PARTIALS | MP_EP_FP64_CROSS_RANK)) != 0)
        return MP_ERR_INVALID_ARG;
    if (K > EP_KMAX) return MP_ERR_UNSUPPORTED;
    if (T == 0) return MP_OK;
    if (rows == nullptr || row_id_map == nullptr || idx == nullptr || out == nullptr)
        return MP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    const int per_rank = E / ep_size;
    const bool vec = H % 8 == 0 && aligned16(rows) && aligned16(out);
    if (vec) {
        if (probs)
            launch_ep_flags<uint4, true>(flags, rows, probs, row_id_map, idx, T, K, H / 8, per_rank,
                                         out, s);
        else
            launch_ep_flags<uint4, false>(flags, rows, nullptr, row_id_map, idx, T, K, H / 8,
                                          per_rank, out, s);
    } else {
        if (probs)
            launch_ep_flags<uint16_t, true>(flags, rows, probs, row_id_map, idx, T, K, H, per_rank,
                                            out, s);
        else
            launch_ep_flags<uint16_t, false>(flags, rows, nullptr, row_id_map, idx, T, K, H,
                                             per_rank, out, s);
    }
    return check_launch();
}
