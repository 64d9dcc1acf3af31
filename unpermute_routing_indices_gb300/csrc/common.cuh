// Shared device helpers for the libmp kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>

#include "mp.h"

namespace mp {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Records the CUDA error of the last failed launch for mp_last_cuda_error().
void set_last_cuda_error(cudaError_t err);

// Returns MP_ERR_CUDA if the launches just made on this thread failed.
inline mp_status_t check_launch()
{
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) {
        set_last_cuda_error(err);
        return MP_ERR_CUDA;
    }
    return MP_OK;
}

inline cudaStream_t as_stream(mp_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel is launched with programmatic
// stream serialisation and calls pdl_trigger() and pdl_wait() before it
// touches global memory: its launch and CTA scheduling overlap the tail of
// the kernel before it in the stream, while pdl_wait() holds every thread
// until that kernel has finished and its memory is visible.  (The map's count
// and scan kernels wait before they trigger; the map's rank kernel reads idx
// before its wait.)  After a copy, a memset or a kernel launched the usual way
// the attribute has no effect.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int ceil_log2(int v)
{
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

// ---------------------------------------------------------------------------
// Global memory access.  Rows are streamed: read once through the
// non-coherent path without L1 allocation; written with plain stores.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_stream(const uint16_t *p)
{
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_row(uint4 *p, const uint4 &v) { *p = v; }
__device__ __forceinline__ void st_row(uint16_t *p, uint16_t v) { *p = v; }

template <typename V> __device__ __forceinline__ V zero_vec();
template <> __device__ __forceinline__ uint4 zero_vec<uint4>() { return make_uint4(0, 0, 0, 0); }
template <> __device__ __forceinline__ uint16_t zero_vec<uint16_t>() { return 0; }

// 32-byte vectors (256-bit loads and stores, sm_100 and later), for the row
// copies of wide rows that start on 32-byte boundaries.
struct alignas(32) u32x8 {
    uint4 a, b;
};
__device__ __forceinline__ u32x8 ld_stream(const u32x8 *p)
{
    u32x8 v;
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(v.a.x), "=r"(v.a.y), "=r"(v.a.z), "=r"(v.a.w), "=r"(v.b.x), "=r"(v.b.y),
          "=r"(v.b.z), "=r"(v.b.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ void st_row(u32x8 *p, const u32x8 &v)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"l"(p), "r"(v.a.x), "r"(v.a.y), "r"(v.a.z), "r"(v.a.w), "r"(v.b.x),
                   "r"(v.b.y), "r"(v.b.z), "r"(v.b.w)
                 : "memory");
}
template <> __device__ __forceinline__ u32x8 zero_vec<u32x8>()
{
    return u32x8{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
}
inline bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// ---------------------------------------------------------------------------
// bf16 <-> fp32.  Widening is exact (the 16 bits become the high half of the
// binary32 pattern); narrowing is the hardware round-to-nearest-even.
// ---------------------------------------------------------------------------

template <typename V> struct Lanes;
template <> struct Lanes<uint4> { static constexpr int N = 8; };
template <> struct Lanes<uint16_t> { static constexpr int N = 1; };

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void unpack(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ void unpack(uint16_t v, float (&f)[1])
{
    f[0] = __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ uint4 pack(const float (&f)[8])
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint16_t pack(const float (&f)[1])
{
    __nv_bfloat16 h = __float2bfloat16_rn(f[0]);
    return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ void or_status(int32_t *status, int32_t bits)
{
    if (status != nullptr && bits != 0) atomicOr(status, bits);
}

}  // namespace mp
