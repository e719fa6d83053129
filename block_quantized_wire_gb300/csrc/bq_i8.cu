// Block-INT8 codec kernels: quantize, materialize, multi-source accumulate, ring hop.
//
// Operations from "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A",
// Implementation (the four kernels) and Summary (128 values per block, one FP32
// scale = amax/127, owners materialize the forwarded payload).
//
// Decomposition (see bq_device.cuh): a warp processes a chunk of SEGS segments of 256
// values; in segment j lane l holds values [256j + 8l, 256j + 8l + 8) of the chunk, so
// half-warp h holds block 2j + h. Per chunk, the block amaxes are gathered into lanes
// 0..2*SEGS-1, which compute the chunk's scales once; the scales are then broadcast
// back per segment and stored by those lanes in one coalesced store. Full chunks run
// without bounds checks; the one partial chunk at the end (n not a multiple of the
// chunk) runs the same code with checks.
#include "bq_device.cuh"
#include "bq_launch.h"

namespace bqk {
namespace {

__device__ __forceinline__ int64_t warp_id() { return ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; }
__device__ __forceinline__ int64_t warp_count() { return ((int64_t)gridDim.x * kThreads) >> 5; }

// Lane-held amax of each segment -> lane 2j+h holds block (2j+h)'s amax.
template <int SEGS>
__device__ __forceinline__ float gather_amax(const float (&m)[SEGS], int lane)
{
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        const float g = __shfl_sync(kFull, m[j], (lane & 1) << 4);
        if ((lane >> 1) == j) mine = g;
    }
    return mine;
}

// Requantize SEGS segments of FP32 values (v[j] = lane's 8 values of segment j):
// writes the payload, the chunk's scales and, when kOut, the BF16 materialization.
template <int SEGS, bool kTail, bool kOut>
__device__ __forceinline__ void requant_chunk(const float2 (&v)[SEGS][4], int64_t e0, int64_t b0, int64_t nblk,
                                              int lane, int8_t *__restrict__ q, float *__restrict__ s,
                                              uint16_t *__restrict__ out)
{
    const int half = lane >> 4;
    float m[SEGS];
#pragma unroll
    for (int j = 0; j < SEGS; j++) m[j] = halfwarp_max(amax8(v[j]));
    const I8Scale mine = i8_block_scale(gather_amax<SEGS>(m, lane));
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        I8Scale bj;
        bj.s = __shfl_sync(kFull, mine.s, 2 * j + half);
        bj.r = __shfl_sync(kFull, mine.r, 2 * j + half);
        bj.rl = __shfl_sync(kFull, mine.rl, 2 * j + half);
        uint32_t w[8];
        i8_quant8(v[j], bj, w);
        if (!kTail || b0 + 2 * j + half < nblk) {
            st_v2(q + e0 + 256 * j, pack_payload8(w));
            if (kOut) st_v4(out + e0 + 256 * j, i8_materialize_words(w, bj.s));
        }
    }
    if (lane < 2 * SEGS && (!kTail || b0 + lane < nblk)) s[b0 + lane] = mine.s;
}

// Grid-stride driver over warp chunks. With kPrefetch, the loads of a warp's next
// chunk (c + number of warps) are issued before chunk c is computed (a register
// pipeline; it pays only where registers are cheap, as in materialize). Op provides
//   In                                 registers holding one chunk's inputs
//   load<kTail>(In&, c) / compute<kTail>(const In&, c)
// Full chunks use kTail = false (no bounds checks); the one partial chunk, if any,
// is loaded and computed by the warp whose stride lands on it.
template <bool kPrefetch, class Op>
__device__ __forceinline__ void run_chunks(const Op &op, int64_t nblk, int chunk_blocks)
{
    const int64_t nfull = nblk / chunk_blocks;
    const int64_t stride = warp_count();
    int64_t c = warp_id();
    if (!kPrefetch) {
        for (; c < nfull; c += stride) {
            typename Op::In cur;
            op.template load<false>(cur, c);
            op.template compute<false>(cur, c);
        }
    } else if (c < nfull) {
        typename Op::In cur;
        op.template load<false>(cur, c);
        while (true) {
            const int64_t nc = c + stride;
            const bool more = nc < nfull;
            typename Op::In nxt;
            if (more) op.template load<false>(nxt, nc);
            op.template compute<false>(cur, c);
            c = nc;
            if (!more) break;
            cur = nxt;
        }
    }
    if (c == nfull && nblk % chunk_blocks) {
        typename Op::In t;
        op.template load<true>(t, c);
        op.template compute<true>(t, c);
    }
}

// ---------------------------------------------------------------- quantize
template <int SEGS>
struct QuantOp {
    const uint16_t *__restrict__ x;
    int8_t *__restrict__ q;
    float *__restrict__ s;
    int64_t nblk;
    int lane;
    struct In {
        uint4 x[SEGS];
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
#pragma unroll
        for (int j = 0; j < SEGS; j++)
            in.x[j] = (!kTail || b0 + 2 * j + (lane >> 4) < nblk) ? ld_stream_v4(x + e0 + 256 * j)
                                                                  : make_uint4(0, 0, 0, 0);
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 v[SEGS][4];
#pragma unroll
        for (int j = 0; j < SEGS; j++) bf16x8_to_f32(in.x[j], v[j]);
        requant_chunk<SEGS, kTail, false>(v, c * (256 * SEGS) + lane * 8, c * (2 * SEGS), nblk, lane, q, s, nullptr);
    }
};

template <int SEGS>
__global__ void __launch_bounds__(kThreads)
quant_i8_kernel(const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_begin();
    const QuantOp<SEGS> op{x, q, s, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

// ---------------------------------------------------------------- materialize
template <int SEGS>
struct DequantOp {
    const int8_t *__restrict__ q;
    const float *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint2 q[SEGS];
        float sc;
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
#pragma unroll
        for (int j = 0; j < SEGS; j++)
            in.q[j] = (!kTail || b0 + 2 * j + (lane >> 4) < nblk) ? ld_stream_v2(q + e0 + 256 * j) : make_uint2(0, 0);
        in.sc = (lane < 2 * SEGS && (!kTail || b0 + lane < nblk)) ? __uint_as_float(ld_stream_u32(s + b0 + lane))
                                                                   : 0.0f;
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
        const int half = lane >> 4;
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            const float sj = __shfl_sync(kFull, in.sc, 2 * j + half);
            float2 v[4];
            i8x8_to_f32(in.q[j], v);
            if (!kTail || b0 + 2 * j + half < nblk) st_v4(out + e0 + 256 * j, i8_materialize8(v, sj));
        }
    }
};

template <int SEGS>
__global__ void __launch_bounds__(kThreads)
dequant_i8_kernel(const int8_t *__restrict__ q, const float *__restrict__ s, int64_t nblk, uint16_t *__restrict__ out)
{
    pdl_begin();
    const DequantOp<SEGS> op{q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<true>(op, nblk, 2 * SEGS);
}

// ---------------------------------------------------------------- accumulate
// Sources are summed in source order 0..nsrc-1. The first W sources of a chunk are
// loaded together (and prefetched by the pipeline); any further sources are loaded
// in groups of W with the running sum carried in registers.
template <int SEGS, int W>
struct SourceRegs {
    uint2 q[W][SEGS];
    float sc[W];
};

template <int SEGS, int W, bool kTail>
__device__ __forceinline__ void load_sources(SourceRegs<SEGS, W> &r, const SourceList &src, int g, int nsrc,
                                             int64_t c, int64_t nblk, int lane)
{
    const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
    const bool lane_ok = lane < 2 * SEGS && (!kTail || b0 + lane < nblk);
#pragma unroll
    for (int i = 0; i < W; i++) {
        const bool src_ok = g + i < nsrc;
        const int8_t *qw = src.q[src_ok ? g + i : g];
        const float *sw = src.s[src_ok ? g + i : g];
#pragma unroll
        for (int j = 0; j < SEGS; j++)
            r.q[i][j] = (src_ok && (!kTail || b0 + 2 * j + (lane >> 4) < nblk)) ? ld_stream_v2(qw + e0 + 256 * j)
                                                                                 : make_uint2(0, 0);
        r.sc[i] = (src_ok && lane_ok) ? __uint_as_float(ld_stream_u32(sw + b0 + lane)) : 0.0f;
    }
}

template <int SEGS, int W, bool kFirst>
__device__ __forceinline__ void add_sources(const SourceRegs<SEGS, W> &r, int g, int nsrc, float2 (&acc)[SEGS][4],
                                            int lane)
{
    const int half = lane >> 4;
#pragma unroll
    for (int i = 0; i < W; i++) {
        if (g + i >= nsrc) break;
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            const float2 sj = splat(__shfl_sync(kFull, r.sc[i], 2 * j + half));
            float2 v[4];
            i8x8_to_f32(r.q[i][j], v);
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float2 d = mul2_unfused(v[e], sj);
                acc[j][e] = (kFirst && i == 0) ? d : add2(acc[j][e], d);
            }
        }
    }
}

template <int SEGS, int W, bool kOut>
struct AccumOp {
    const SourceList &src;  // the kernel's __grid_constant__ parameter, read in place
    int nsrc;
    int8_t *__restrict__ q;
    float *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    using In = SourceRegs<SEGS, W>;
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        load_sources<SEGS, W, kTail>(in, src, 0, nsrc, c, nblk, lane);
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 acc[SEGS][4];
        add_sources<SEGS, W, true>(in, 0, nsrc, acc, lane);
        for (int g = W; g < nsrc; g += W) {
            In more;
            load_sources<SEGS, W, kTail>(more, src, g, nsrc, c, nblk, lane);
            add_sources<SEGS, W, false>(more, g, nsrc, acc, lane);
        }
        requant_chunk<SEGS, kTail, kOut>(acc, c * (256 * SEGS) + lane * 8, c * (2 * SEGS), nblk, lane, q, s, out);
    }
};

template <int SEGS, int W, bool kOut>
__global__ void __launch_bounds__(kThreads)
accum_i8_kernel(const __grid_constant__ SourceList src, int nsrc, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s,
                uint16_t *__restrict__ out)
{
    pdl_begin();
    const AccumOp<SEGS, W, kOut> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

// ---------------------------------------------------------------- ring hop
template <int SEGS, bool kOut>
struct HopOp {
    const int8_t *__restrict__ q_in;
    const float *__restrict__ s_in;
    const uint16_t *__restrict__ x;
    int8_t *__restrict__ q;
    float *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint2 q[SEGS];
        uint4 x[SEGS];
        float sc;
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            const bool ok = !kTail || b0 + 2 * j + (lane >> 4) < nblk;
            in.q[j] = ok ? ld_stream_v2(q_in + e0 + 256 * j) : make_uint2(0, 0);
            in.x[j] = ok ? ld_stream_v4(x + e0 + 256 * j) : make_uint4(0, 0, 0, 0);
        }
        in.sc = (lane < 2 * SEGS && (!kTail || b0 + lane < nblk)) ? __uint_as_float(ld_stream_u32(s_in + b0 + lane))
                                                                   : 0.0f;
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        const int half = lane >> 4;
        float2 v[SEGS][4];
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            const float2 sj = splat(__shfl_sync(kFull, in.sc, 2 * j + half));
            float2 d[4], xl[4];
            i8x8_to_f32(in.q[j], d);
            bf16x8_to_f32(in.x[j], xl);
#pragma unroll
            for (int e = 0; e < 4; e++) v[j][e] = add2(mul2_unfused(d[e], sj), xl[e]);
        }
        requant_chunk<SEGS, kTail, kOut>(v, c * (256 * SEGS) + lane * 8, c * (2 * SEGS), nblk, lane, q, s, out);
    }
};

template <int SEGS, bool kOut>
__global__ void __launch_bounds__(kThreads)
ring_hop_i8_kernel(const int8_t *__restrict__ q_in, const float *__restrict__ s_in, const uint16_t *__restrict__ x,
                   int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    const HopOp<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

// Segments per warp chunk for each kernel (tuned on GB300; overridable at build time).
#ifndef BQ_SEGS_QUANT
#define BQ_SEGS_QUANT 4
#endif
#ifndef BQ_SEGS_DEQUANT
#define BQ_SEGS_DEQUANT 8
#endif
#ifndef BQ_SEGS_ACCUM
#define BQ_SEGS_ACCUM 4
#endif
#ifndef BQ_SEGS_HOP
#define BQ_SEGS_HOP 4
#endif
constexpr int kSegsQuant = BQ_SEGS_QUANT;
constexpr int kSegsDequant = BQ_SEGS_DEQUANT;
constexpr int kSegsAccum = BQ_SEGS_ACCUM;
constexpr int kSegsHop = BQ_SEGS_HOP;

int64_t chunks(int64_t nblk, int segs) { return (nblk + 2 * segs - 1) / (2 * segs); }

#define BQK_GRID(kernel, nchunk)                                          \
    int grid = 0;                                                         \
    if (cudaError_t e_ = grid_for((const void *)(kernel), (nchunk), &grid)) \
        return e_;

template <int W, bool kOut>
cudaError_t launch_accum_w(const SourceList &src, int nsrc, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                           cudaStream_t st)
{
    auto kernel = accum_i8_kernel<kSegsAccum, W, kOut>;
    BQK_GRID(kernel, chunks(nblk, kSegsAccum));
    return launch_kernel(kernel, grid, st, src, nsrc, nblk, q, s, out);
}

}  // namespace

cudaError_t launch_quant_i8(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st)
{
    BQK_GRID(quant_i8_kernel<kSegsQuant>, chunks(nblk, kSegsQuant));
    return launch_kernel(quant_i8_kernel<kSegsQuant>, grid, st, x, nblk, q, s);
}

cudaError_t launch_dequant_i8(const int8_t *q, const float *s, int64_t nblk, uint16_t *out, cudaStream_t st)
{
    BQK_GRID(dequant_i8_kernel<kSegsDequant>, chunks(nblk, kSegsDequant));
    return launch_kernel(dequant_i8_kernel<kSegsDequant>, grid, st, q, s, nblk, out);
}

// One source width is compiled per common case (1, 2, 3, 4 sources at once); more
// sources run in groups of four.
cudaError_t launch_accum_i8(const SourceList &src, int W, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                            cudaStream_t st)
{
    const bool o = out != nullptr;
    switch (W) {
    case 1: return o ? launch_accum_w<1, true>(src, W, nblk, q, s, out, st) : launch_accum_w<1, false>(src, W, nblk, q, s, out, st);
    case 2: return o ? launch_accum_w<2, true>(src, W, nblk, q, s, out, st) : launch_accum_w<2, false>(src, W, nblk, q, s, out, st);
    case 3: return o ? launch_accum_w<3, true>(src, W, nblk, q, s, out, st) : launch_accum_w<3, false>(src, W, nblk, q, s, out, st);
    default: return o ? launch_accum_w<4, true>(src, W, nblk, q, s, out, st) : launch_accum_w<4, false>(src, W, nblk, q, s, out, st);
    }
}

cudaError_t launch_ring_hop_i8(const int8_t *q_in, const float *s_in, const uint16_t *x, int64_t nblk, int8_t *q,
                               float *s, uint16_t *out, cudaStream_t st)
{
    if (out) {
        BQK_GRID((ring_hop_i8_kernel<kSegsHop, true>), chunks(nblk, kSegsHop));
        return launch_kernel(ring_hop_i8_kernel<kSegsHop, true>, grid, st, q_in, s_in, x, nblk, q, s, out);
    }
    BQK_GRID((ring_hop_i8_kernel<kSegsHop, false>), chunks(nblk, kSegsHop));
    return launch_kernel(ring_hop_i8_kernel<kSegsHop, false>, grid, st, q_in, s_in, x, nblk, q, s,
                         static_cast<uint16_t *>(nullptr));
}

}  // namespace bqk
