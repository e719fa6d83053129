// Block-INT8 codec kernels: quantize, materialize, multi-source accumulate, ring hop.
//
// Operations from "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A",
// Implementation (the four kernels) and Summary (128 values per block, one FP32
// scale = amax/127, owners materialize the forwarded payload). The decomposition into
// warp chunks and segments is described in bq_device.cuh.
#include "bq_device.cuh"
#include "bq_launch.h"

namespace bqk {
namespace {

__device__ __forceinline__ int64_t first_chunk() { return (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); }
__device__ __forceinline__ int64_t chunk_stride() { return (int64_t)gridDim.x * (kThreads / 32); }

// Hand the scale of segment j (held by every lane of each half-warp) to lane 2j+h, so
// that after the chunk lanes 0..kChunkBlocks-1 hold the chunk's scales in block order.
__device__ __forceinline__ void collect_scale(float s_seg, int j, int lane, float &mine)
{
    const float lo = __shfl_sync(kFull, s_seg, 0);
    const float hi = __shfl_sync(kFull, s_seg, 16);
    if (lane == 2 * j) mine = lo;
    if (lane == 2 * j + 1) mine = hi;
}

// Requantize one segment (8 FP32 values per lane), store its payload and, when kOut,
// its BF16 materialization; returns the block scale.
template <bool kOut>
__device__ __forceinline__ float requant_segment(const float (&v)[8], int64_t elem, bool valid,
                                                 int8_t *__restrict__ q, uint16_t *__restrict__ out)
{
    const I8Scale sc = i8_scale(halfwarp_max(amax8(v)));
    float qf[8];
    const uint2 packed = i8_quant8(v, sc, qf);
    if (valid) {
        st_v2(q + elem, packed);
        if (kOut) st_v4(out + elem, i8_materialize8(qf, sc.s));
    }
    return sc.s;
}

__global__ void __launch_bounds__(kThreads)
quant_i8_kernel(const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    for (int64_t c = first_chunk(); c < nchunk; c += chunk_stride()) {
        const int64_t b0 = c * kChunkBlocks;
        uint4 raw[kSegs];
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            raw[j] = blk < nblk ? ld_stream_v4(x + blk * 128 + hl * 8) : make_uint4(0, 0, 0, 0);
        }
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            float v[8];
            bf16x8_to_f32(raw[j], v);
            const float sj = requant_segment<false>(v, blk * 128 + hl * 8, blk < nblk, q, nullptr);
            collect_scale(sj, j, lane, mine);
        }
        if (lane < kChunkBlocks && b0 + lane < nblk) s[b0 + lane] = mine;
    }
}

__global__ void __launch_bounds__(kThreads)
dequant_i8_kernel(const int8_t *__restrict__ q, const float *__restrict__ s, int64_t nblk,
                  uint16_t *__restrict__ out)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    for (int64_t c = first_chunk(); c < nchunk; c += chunk_stride()) {
        const int64_t b0 = c * kChunkBlocks;
        uint2 raw[kSegs];
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            raw[j] = blk < nblk ? ld_stream_v2(q + blk * 128 + hl * 8) : make_uint2(0, 0);
        }
        const float sc =
            (lane < kChunkBlocks && b0 + lane < nblk) ? __uint_as_float(ld_stream_u32(s + b0 + lane)) : 0.0f;
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            const float sj = __shfl_sync(kFull, sc, 2 * j + half);
            float v[8];
            i8x8_to_f32(raw[j], v);
            if (blk < nblk) st_v4(out + blk * 128 + hl * 8, i8_materialize8(v, sj));
        }
    }
}

// Sources are consumed in groups of four so that each group's loads are in flight
// together; the running sum is carried across groups in source order.
template <bool kOut>
__global__ void __launch_bounds__(kThreads)
accum_i8_kernel(const SourceList src, int W, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s,
                uint16_t *__restrict__ out)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    for (int64_t c = first_chunk(); c < nchunk; c += chunk_stride()) {
        const int64_t b0 = c * kChunkBlocks;
        const bool lane_blk_ok = lane < kChunkBlocks && b0 + lane < nblk;
        float acc[kSegs][8];
        for (int w0 = 0; w0 < W; w0 += 4) {
            uint2 raw[4][kSegs];
            float sc[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                if (w0 + i < W) {
                    const int8_t *qw = src.q[w0 + i];
#pragma unroll
                    for (int j = 0; j < kSegs; j++) {
                        const int64_t blk = b0 + 2 * j + half;
                        raw[i][j] = blk < nblk ? ld_stream_v2(qw + blk * 128 + hl * 8) : make_uint2(0, 0);
                    }
                    sc[i] = lane_blk_ok ? __uint_as_float(ld_stream_u32(src.s[w0 + i] + b0 + lane)) : 0.0f;
                }
            }
#pragma unroll
            for (int i = 0; i < 4; i++) {
                if (w0 + i < W) {
#pragma unroll
                    for (int j = 0; j < kSegs; j++) {
                        const float sj = __shfl_sync(kFull, sc[i], 2 * j + half);
                        float v[8];
                        i8x8_to_f32(raw[i][j], v);
                        if (w0 + i == 0) {
#pragma unroll
                            for (int e = 0; e < 8; e++) acc[j][e] = __fmul_rn(v[e], sj);
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; e++) acc[j][e] = __fadd_rn(acc[j][e], __fmul_rn(v[e], sj));
                        }
                    }
                }
            }
        }
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            const float sj = requant_segment<kOut>(acc[j], blk * 128 + hl * 8, blk < nblk, q, out);
            collect_scale(sj, j, lane, mine);
        }
        if (lane_blk_ok) s[b0 + lane] = mine;
    }
}

template <bool kOut>
__global__ void __launch_bounds__(kThreads)
ring_hop_i8_kernel(const int8_t *__restrict__ q_in, const float *__restrict__ s_in,
                   const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q,
                   float *__restrict__ s, uint16_t *__restrict__ out)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t nchunk = (nblk + kChunkBlocks - 1) / kChunkBlocks;
    for (int64_t c = first_chunk(); c < nchunk; c += chunk_stride()) {
        const int64_t b0 = c * kChunkBlocks;
        const bool lane_blk_ok = lane < kChunkBlocks && b0 + lane < nblk;
        uint2 rq[kSegs];
        uint4 rx[kSegs];
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            const bool ok = blk < nblk;
            rq[j] = ok ? ld_stream_v2(q_in + blk * 128 + hl * 8) : make_uint2(0, 0);
            rx[j] = ok ? ld_stream_v4(x + blk * 128 + hl * 8) : make_uint4(0, 0, 0, 0);
        }
        const float sc = lane_blk_ok ? __uint_as_float(ld_stream_u32(s_in + b0 + lane)) : 0.0f;
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < kSegs; j++) {
            const int64_t blk = b0 + 2 * j + half;
            const float sj = __shfl_sync(kFull, sc, 2 * j + half);
            float d[8], xl[8], v[8];
            i8x8_to_f32(rq[j], d);
            bf16x8_to_f32(rx[j], xl);
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = __fadd_rn(__fmul_rn(d[e], sj), xl[e]);
            const float so = requant_segment<kOut>(v, blk * 128 + hl * 8, blk < nblk, q, out);
            collect_scale(so, j, lane, mine);
        }
        if (lane_blk_ok) s[b0 + lane] = mine;
    }
}

int64_t chunks_of(int64_t nblk) { return (nblk + kChunkBlocks - 1) / kChunkBlocks; }

}  // namespace

#define BQK_GRID(kernel, nchunk)                                          \
    int grid = 0;                                                         \
    if (cudaError_t e_ = grid_for((const void *)(kernel), (nchunk), &grid)) \
        return e_;

cudaError_t launch_quant_i8(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st)
{
    BQK_GRID(quant_i8_kernel, chunks_of(nblk));
    quant_i8_kernel<<<grid, kThreads, 0, st>>>(x, nblk, q, s);
    return cudaGetLastError();
}

cudaError_t launch_dequant_i8(const int8_t *q, const float *s, int64_t nblk, uint16_t *out, cudaStream_t st)
{
    BQK_GRID(dequant_i8_kernel, chunks_of(nblk));
    dequant_i8_kernel<<<grid, kThreads, 0, st>>>(q, s, nblk, out);
    return cudaGetLastError();
}

cudaError_t launch_accum_i8(const SourceList &src, int W, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                            cudaStream_t st)
{
    if (out) {
        BQK_GRID(accum_i8_kernel<true>, chunks_of(nblk));
        accum_i8_kernel<true><<<grid, kThreads, 0, st>>>(src, W, nblk, q, s, out);
    } else {
        BQK_GRID(accum_i8_kernel<false>, chunks_of(nblk));
        accum_i8_kernel<false><<<grid, kThreads, 0, st>>>(src, W, nblk, q, s, nullptr);
    }
    return cudaGetLastError();
}

cudaError_t launch_ring_hop_i8(const int8_t *q_in, const float *s_in, const uint16_t *x, int64_t nblk, int8_t *q,
                               float *s, uint16_t *out, cudaStream_t st)
{
    if (out) {
        BQK_GRID(ring_hop_i8_kernel<true>, chunks_of(nblk));
        ring_hop_i8_kernel<true><<<grid, kThreads, 0, st>>>(q_in, s_in, x, nblk, q, s, out);
    } else {
        BQK_GRID(ring_hop_i8_kernel<false>, chunks_of(nblk));
        ring_hop_i8_kernel<false><<<grid, kThreads, 0, st>>>(q_in, s_in, x, nblk, q, s, nullptr);
    }
    return cudaGetLastError();
}

}  // namespace bqk
