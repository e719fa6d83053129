// Legacy E4M3 codec kernels: quantize, materialize, and the E4M3 all-gather mode's
// BF16 reduce fused with quantization.
//
// The block-INT8 page ("feat(pcie_dma): add block-INT8 wire modes for AG, ring, and
// A2A", Summary and Why) describes the codec it replaces: one E4M3 byte per value and
// one FP32 scale per 128-value block, the same 132-byte block and wire geometry as
// block INT8. The pages print no scale rule; the one taken here is block INT8's with
// the largest finite E4M3 value in place of 127: s = fl(amax / 448) and
// code = E4M3 (nearest even, saturating, sign of zero kept) of fl(x / s); an all-zero
// block has s = 0 and codes 0x00. Materialization is BF16(fl(decode(code) * s)).
#include "bq_chunks.cuh"

namespace bqk {
namespace {

// Requantize SEGS segments of binary32 values as E4M3 blocks: the block amaxes are
// gathered into lanes 0..2*SEGS-1, which compute each block's scale, reciprocal and
// correction term once; they are broadcast back per segment.
template <int SEGS, bool kTail, bool kOut, class Vals>
__device__ __forceinline__ void requant_e4m3_chunk(const Vals &vals, int64_t e0, int64_t b0, int64_t nblk, int lane,
                                                   uint8_t *__restrict__ q, float *__restrict__ s,
                                                   uint16_t *__restrict__ out)
{
    const int half = lane >> 4;
    float m[SEGS];
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        float2 v[4];
        vals.seg(j, v);
        m[j] = halfwarp_max(amax8(v));
    }
    const I8Scale mine = e4m3_block_scale(gather_amax<SEGS>(m, lane));
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        I8Scale bj;
        bj.s = __shfl_sync(kFull, mine.s, 2 * j + half);
        bj.r = __shfl_sync(kFull, mine.r, 2 * j + half);
        bj.rl = __shfl_sync(kFull, mine.rl, 2 * j + half);
        float2 v[4];
        vals.seg(j, v);
        const uint2 codes = e4m3_quant8(v, bj);
        if (!kTail || b0 + 2 * j + half < nblk) {
            st_v2(q + e0 + 256 * j, codes);
            if (kOut) st_v4(out + e0 + 256 * j, e4m3_materialize8(codes, bj.s));
        }
    }
    if (lane < 2 * SEGS && (!kTail || b0 + lane < nblk) && dbg_ok(s + b0 + lane, 4, true)) s[b0 + lane] = mine.s;
}

struct E4m3Codec {
    using Q = uint8_t;
    using S = float;
    template <int SEGS, bool kTail, bool kOut, class Vals>
    static __device__ __forceinline__ void requant(const Vals &vals, int64_t e0, int64_t b0, int64_t nblk, int lane,
                                                   uint8_t *q, float *s, uint16_t *out)
    {
        requant_e4m3_chunk<SEGS, kTail, kOut>(vals, e0, b0, nblk, lane, q, s, out);
    }
    static __device__ __forceinline__ uint4 dequant8(uint2 q, uint32_t word, int)
    {
        return e4m3_materialize8(q, __uint_as_float(word));
    }
};

#ifndef BQ_QUANT_E4M3_MIN_CTAS
#define BQ_QUANT_E4M3_MIN_CTAS 4
#endif
// Threads per CTA of the E4M3 quantize and materialize (registers per thread at the
// 4-CTA budget of 256-thread CTAs whatever the size). Per 469.8M-value launch on GB300:
// quantize 231.6 us in one 1024-thread CTA per SM against 241.9 us in 256-thread CTAs;
// the materialize 247.7 against 241.7 us, so it keeps 256.
#ifndef BQ_QUANT_E4M3_THREADS
#define BQ_QUANT_E4M3_THREADS 1024
#endif
#ifndef BQ_DEQUANT_E4M3_THREADS
#define BQ_DEQUANT_E4M3_THREADS 256
#endif
constexpr int kQuantE4m3Threads = BQ_QUANT_E4M3_THREADS;
constexpr int kDequantE4m3Threads = BQ_DEQUANT_E4M3_THREADS;

template <int SEGS>
__global__ void __launch_bounds__(kQuantE4m3Threads, BQ_QUANT_E4M3_MIN_CTAS * kThreads / kQuantE4m3Threads)
quant_e4m3_kernel(const uint16_t *__restrict__ x, int64_t nblk, uint8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_begin();
    dbg_begin();
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_ready();
    const QuantOp<E4m3Codec, SEGS, true> op{x, q, s, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false, kQuantE4m3Threads>(op, nblk, 2 * SEGS);
}

template <int SEGS>
__global__ void __launch_bounds__(kDequantE4m3Threads, 4 * kThreads / kDequantE4m3Threads)
dequant_e4m3_kernel(const uint8_t *__restrict__ q, const float *__restrict__ s, int64_t nblk,
                    uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q, s, nblk, false);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const DequantOp<E4m3Codec, SEGS> op{q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<true, kDequantE4m3Threads>(op, nblk, 2 * SEGS);
}

template <int SEGS, int W, bool kOut>
__global__ void __launch_bounds__(kThreads)
reduce_quant_e4m3_kernel(const __grid_constant__ Bf16List src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                         float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const ReduceQuantOp<E4m3Codec, SEGS, W, kOut> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

#ifndef BQ_SEGS_REDUCE_E4M3_ASYNC
#define BQ_SEGS_REDUCE_E4M3_ASYNC 2
#endif

template <int W, bool kOut>
__global__ void __launch_bounds__(kReduceAsyncThreads, kReduceAsyncMinCtas)
reduce_quant_e4m3_async_kernel(const __grid_constant__ Bf16List src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                               float *__restrict__ s, uint16_t *__restrict__ out)
{
    extern __shared__ __align__(16) unsigned char stages[];
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    reduce_quant_async_body<E4m3Codec, BQ_SEGS_REDUCE_E4M3_ASYNC, W, kOut>(src, nsrc, nblk, q, s, out, stages);
}

// E4M3 quantize, 469.8M values on GB300 (graph-timed): 264 us with 4 segments per chunk
// and the values widened once (spilling at 64 registers), 245 us widened per read (62
// registers), 224 us widened per read with 8 segments (64 registers, no spills).
#ifndef BQ_SEGS_QUANT_E4M3
#define BQ_SEGS_QUANT_E4M3 8
#endif
#ifndef BQ_SEGS_DEQUANT_E4M3
#define BQ_SEGS_DEQUANT_E4M3 8
#endif
#ifndef BQ_SEGS_REDUCE_E4M3
#define BQ_SEGS_REDUCE_E4M3 2
#endif
constexpr int kSegsQuant = BQ_SEGS_QUANT_E4M3;
constexpr int kSegsDequant = BQ_SEGS_DEQUANT_E4M3;
constexpr int kSegsReduce = BQ_SEGS_REDUCE_E4M3;

template <int W, bool kOut>
cudaError_t launch_reduce_w(const Bf16List &src, int nsrc, int64_t nblk, uint8_t *q, float *s, uint16_t *out,
                            cudaStream_t st)
{
    if (BQ_REDUCE_ASYNC && nsrc == W)
        return launch_reduce_async<E4m3Codec, BQ_SEGS_REDUCE_E4M3_ASYNC, W, kOut>(
            reduce_quant_e4m3_async_kernel<W, kOut>, nblk, st, src, nsrc, nblk, q, s, out);
    auto kernel = reduce_quant_e4m3_kernel<kSegsReduce, W, kOut>;
    BQK_GRID(kernel, chunks(nblk, kSegsReduce));
    return launch_kernel(kernel, grid, st, src, nsrc, nblk, q, s, out);
}

}  // namespace

cudaError_t launch_quant_e4m3(const uint16_t *x, int64_t nblk, uint8_t *q, float *s, cudaStream_t st)
{
    auto kernel = quant_e4m3_kernel<kSegsQuant>;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, kSegsQuant), &grid, 0, kQuantE4m3Threads)) return e;
    return launch_kernel_block(kernel, grid, kQuantE4m3Threads, 0, st, x, nblk, q, s);
}

cudaError_t launch_dequant_e4m3(const uint8_t *q, const float *s, int64_t nblk, uint16_t *out, cudaStream_t st)
{
    auto kernel = dequant_e4m3_kernel<kSegsDequant>;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, kSegsDequant), &grid, 0, kDequantE4m3Threads))
        return e;
    return launch_kernel_block(kernel, grid, kDequantE4m3Threads, 0, st, q, s, nblk, out);
}

// One source width per common case (1..4 at once); more sources in groups of four.
cudaError_t launch_reduce_quant_e4m3(const Bf16List &src, int W, int64_t nblk, uint8_t *q, float *s, uint16_t *out,
                                     cudaStream_t st)
{
    const bool o = out != nullptr;
    switch (W) {
    case 1: return o ? launch_reduce_w<1, true>(src, W, nblk, q, s, out, st) : launch_reduce_w<1, false>(src, W, nblk, q, s, out, st);
    case 2: return o ? launch_reduce_w<2, true>(src, W, nblk, q, s, out, st) : launch_reduce_w<2, false>(src, W, nblk, q, s, out, st);
    case 3: return o ? launch_reduce_w<3, true>(src, W, nblk, q, s, out, st) : launch_reduce_w<3, false>(src, W, nblk, q, s, out, st);
    default: return o ? launch_reduce_w<4, true>(src, W, nblk, q, s, out, st) : launch_reduce_w<4, false>(src, W, nblk, q, s, out, st);
    }
}

cudaError_t read_wait_counters_e4m3(unsigned long long (&v)[3]) { return read_wait_counters(v); }

}  // namespace bqk
