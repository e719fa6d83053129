// MXFP8 codec kernels: quantize (2-D, strided, covers staged slices) and materialize.
//
// Format from "feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary (E4M3 values,
// one E8M0 scale per 32 values) and the review comment on mxfp8_scale_byte (zero
// group -> 127, else E8M0 of amax/448 rounded toward +inf, saturating). Slices follow
// "[II] Support staged MXFP8 linear inputs", Behavior and Compatibility: a slice of
// 128-column-aligned width written at a 128-column-aligned offset of a wider buffer.
//
// A "block" here is 128 consecutive columns of one row (four MX groups), so the
// warp decomposition of bq_device.cuh applies unchanged: a half-warp holds a block,
// a quad of lanes holds a group, and the block's four scale bytes form one 32-bit
// word written by a single lane.
#include "bq_device.cuh"
#include "bq_launch.h"

namespace bqk {
namespace {

__device__ __forceinline__ int64_t first_chunk() { return (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); }
__device__ __forceinline__ int64_t chunk_stride() { return (int64_t)gridDim.x * (kThreads / 32); }

// Row and 128-column block of linear block index row0 * bpr + cb0 + k.
__device__ __forceinline__ void advance(int64_t row0, int64_t cb0, int k, int64_t bpr, int64_t &row, int64_t &cb)
{
    row = row0;
    cb = cb0 + k;
    while (cb >= bpr) {
        cb -= bpr;
        ++row;
    }
}

__global__ void __launch_bounds__(kThreads)
quant_mx_kernel(const uint16_t *__restrict__ x, int64_t ld_x, int64_t bpr, int64_t nblk, uint8_t *__restrict__ q,
                int64_t ld_q, uint8_t *__restrict__ s, int64_t ld_s)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    for (int64_t c = first_chunk(); c < nchunk; c += chunk_stride()) {
        const int64_t b0 = c * kChunkBlocks;
        const int64_t row0 = b0 / bpr, cb0 = b0 - row0 * bpr;
        uint4 raw[kSegs];
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            int64_t row, cb;
            advance(row0, cb0, 2 * j + half, bpr, row, cb);
            raw[j] = (b0 + 2 * j + half < nblk) ? ld_stream_v4(x + row * ld_x + cb * 128 + hl * 8)
                                                : make_uint4(0, 0, 0, 0);
        }
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            int64_t row, cb;
            advance(row0, cb0, 2 * j + half, bpr, row, cb);
            float v[8];
            bf16x8_to_f32(raw[j], v);
            float m = amax8(v);
            m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));  // the 4 lanes of a 32-value group
            m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
            const uint32_t e = mx_scale_byte(m);
            const float p = exp2i(127 - static_cast<int>(e));
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; i++) y[i] = __fmul_rn(v[i], p);  // exact: a power-of-two scaling
            if (b0 + 2 * j + half < nblk) st_v2(q + row * ld_q + cb * 128 + hl * 8, f32x8_to_e4m3x8(y));
            // the block's four scale bytes, group g in byte g
            uint32_t word = e << (8 * (hl >> 2));
            word |= __shfl_xor_sync(kFull, word, 4);
            word |= __shfl_xor_sync(kFull, word, 8);
            const uint32_t lo = __shfl_sync(kFull, word, 0);
            const uint32_t hi = __shfl_sync(kFull, word, 16);
            if (lane == 2 * j) mine = lo;
            if (lane == 2 * j + 1) mine = hi;
        }
        if (lane < kChunkBlocks && b0 + lane < nblk) {
            int64_t row, cb;
            advance(row0, cb0, lane, bpr, row, cb);
            st_u32(s + row * ld_s + cb * 4, mine);
        }
    }
}

__global__ void __launch_bounds__(kThreads)
dequant_mx_kernel(const uint8_t *__restrict__ q, int64_t ld_q, const uint8_t *__restrict__ s, int64_t ld_s,
                  int64_t bpr, int64_t nblk, uint16_t *__restrict__ out, int64_t ld_out)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    for (int64_t c = first_chunk(); c < nchunk; c += chunk_stride()) {
        const int64_t b0 = c * kChunkBlocks;
        const int64_t row0 = b0 / bpr, cb0 = b0 - row0 * bpr;
        uint2 raw[kSegs];
        uint32_t sw[kSegs];
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            int64_t row, cb;
            advance(row0, cb0, 2 * j + half, bpr, row, cb);
            const bool ok = b0 + 2 * j + half < nblk;
            raw[j] = ok ? ld_stream_v2(q + row * ld_q + cb * 128 + hl * 8) : make_uint2(0, 0);
            sw[j] = ok ? ld_stream_u32(s + row * ld_s + cb * 4) : 0u;
        }
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            int64_t row, cb;
            advance(row0, cb0, 2 * j + half, bpr, row, cb);
            const uint32_t e = (sw[j] >> (8 * (hl >> 2))) & 0xffu;
            const float p = e == 255u ? __uint_as_float(0x7fc00000u) : exp2i(static_cast<int>(e) - 127);
            float v[8];
            e4m3x8_to_f32(raw[j], p, v);
            if (b0 + 2 * j + half < nblk) st_v4(out + row * ld_out + cb * 128 + hl * 8, f32x8_to_bf16x8(v));
        }
    }
}

#define BQK_GRID(kernel, nchunk)                                          \
    int grid = 0;                                                         \
    if (cudaError_t e_ = grid_for((const void *)(kernel), (nchunk), &grid)) \
        return e_;

}  // namespace

cudaError_t launch_quant_mx(const uint16_t *x, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q, int64_t ld_q,
                            uint8_t *s, int64_t ld_s, cudaStream_t st)
{
    const int64_t bpr = cols / 128, nblk = rows * bpr;
    BQK_GRID(quant_mx_kernel, (nblk + kChunkBlocks - 1) / kChunkBlocks);
    quant_mx_kernel<<<grid, kThreads, 0, st>>>(x, ld_x, bpr, nblk, q, ld_q, s, ld_s);
    return cudaGetLastError();
}

cudaError_t launch_dequant_mx(const uint8_t *q, int64_t ld_q, const uint8_t *s, int64_t ld_s, int64_t rows,
                              int64_t cols, uint16_t *out, int64_t ld_out, cudaStream_t st)
{
    const int64_t bpr = cols / 128, nblk = rows * bpr;
    BQK_GRID(dequant_mx_kernel, (nblk + kChunkBlocks - 1) / kChunkBlocks);
    dequant_mx_kernel<<<grid, kThreads, 0, st>>>(q, ld_q, s, ld_s, bpr, nblk, out, ld_out);
    return cudaGetLastError();
}

}  // namespace bqk
