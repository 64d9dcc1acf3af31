// Zero fill of the rows of a permuted buffer that no slot maps to.
//
// Token dropping leaves the permuted tensor with fewer routed rows than it
// has rows ("d9d 0.1.0 — d9d/kernel/moe/permute_with_probs.py", num_out_tokens,
// "the number of tokens not dropped"), and so do empty slots.  Those rows are
// never written by the row kernels.  A training step that runs an expert
// computation over the whole buffer needs them at zero (a NaN there would
// reach the weight gradients through 0 * NaN).  The routed row count lives on
// the device (offsets[E] of the map), so the start row is read there: no host
// round trip, and a CUDA graph replays it with new routing.
//
// k_zero_rows_from: a grid-stride store loop over [first_row * row, rows * row)
// in units of V (16, 4 or 1 bytes, the widest the pointer and row size allow),
// four stores per thread per step (a CTA owns 4 * 256 consecutive units).
// Every CTA reads the start once; with everything routed no store is issued.
#include "common.cuh"

namespace mp {
namespace {

#ifndef MP_FILL_MAX_BLOCKS
#define MP_FILL_MAX_BLOCKS (152 * 8)
#endif

constexpr int FILL_THREADS = 256;
constexpr int FILL_UNROLL = 4;   // stores in flight per thread per step
constexpr int FILL_MAX_BLOCKS = MP_FILL_MAX_BLOCKS;

template <typename V>
__global__ void __launch_bounds__(FILL_THREADS)
    k_zero_rows_from(V *__restrict__ buf, int64_t rows, int64_t units_per_row,
                     const int32_t *__restrict__ first_row)
{
    pdl_trigger();
    pdl_wait();
    int64_t s = __ldg(first_row);
    s = s < 0 ? 0 : (s > rows ? rows : s);
    const int64_t end = rows * units_per_row;
    const int64_t step = (int64_t)gridDim.x * FILL_THREADS;
    V z;
    if constexpr (sizeof(V) == 16)
        z = make_uint4(0, 0, 0, 0);
    else
        z = 0;
    constexpr int U = FILL_UNROLL;
    int64_t i = s * units_per_row + (int64_t)blockIdx.x * FILL_THREADS * U + threadIdx.x;
    for (; i + (U - 1) * FILL_THREADS < end; i += step * U) {
#pragma unroll
        for (int u = 0; u < U; ++u) buf[i + u * FILL_THREADS] = z;
    }
    for (; i < end; i += FILL_THREADS) buf[i] = z;
}

template <typename V>
void launch_fill(void *buf, int64_t rows, int64_t units_per_row, const int32_t *first_row,
                 cudaStream_t s)
{
    const int64_t total = rows * units_per_row;
    int64_t blocks = (total + FILL_THREADS * FILL_UNROLL - 1) / (FILL_THREADS * FILL_UNROLL);
    blocks = blocks < 1 ? 1 : (blocks > FILL_MAX_BLOCKS ? FILL_MAX_BLOCKS : blocks);
    (void)launch_pdl(k_zero_rows_from<V>, (unsigned)blocks, FILL_THREADS, 0, s,
                     static_cast<V *>(buf), rows, units_per_row, first_row);
}

}  // namespace
}  // namespace mp

using namespace mp;

extern "C" mp_status_t mp_zero_rows_from(void *buf, int64_t rows, int64_t row_bytes,
                                         const int32_t *first_row, mp_stream_t stream)
{
    if (rows < 0 || row_bytes < 0) return MP_ERR_INVALID_ARG;
    if (rows > 0 && row_bytes > INT64_MAX / rows) return MP_ERR_INVALID_ARG;
    if (rows == 0 || row_bytes == 0) return MP_OK;
    if (buf == nullptr || first_row == nullptr) return MP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    const uintptr_t a = reinterpret_cast<uintptr_t>(buf);
    if ((a & 15u) == 0 && row_bytes % 16 == 0)
        launch_fill<uint4>(buf, rows, row_bytes / 16, first_row, s);
    else if ((a & 3u) == 0 && row_bytes % 4 == 0)
        launch_fill<uint32_t>(buf, rows, row_bytes / 4, first_row, s);
    else
        launch_fill<uint8_t>(buf, rows, row_bytes, first_row, s);
    return check_launch();
}
