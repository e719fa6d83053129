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

// Staged driver: each warp keeps the inputs of its next STAGES full chunks in flight
// as bulk copies into its own slice of shared memory (issued by lane 0, completed on
// one mbarrier per stage), reads a chunk's inputs from shared memory into the same
// registers the global-memory path fills, computes it exactly as that path does, and
// then reuses the stage for the chunk STAGES ahead. Op additionally provides
//   kStageBytes                      bytes of one chunk's staged inputs
//   issue(c, stage, bar)             lane 0: expect_tx + bulk copies of chunk c
//   load_staged(In&, stage pointer)  fill In from the staged copy
// The ragged last chunk, if any, takes the global-memory path.
template <class Op, int STAGES>
__host__ __device__ constexpr uint32_t staged_warp_bytes()
{
    return 128u + STAGES * ((Op::kStageBytes + 127u) / 128u * 128u);
}

template <int STAGES, class Op>
__device__ __forceinline__ void run_staged(const Op &op, int64_t nblk, int chunk_blocks, unsigned char *warp_smem)
{
    constexpr uint32_t kStride = (Op::kStageBytes + 127u) / 128u * 128u;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(warp_smem);
    unsigned char *buf = warp_smem + 128;
    const uint32_t buf0 = smem_u32(buf);
    const int64_t nfull = nblk / chunk_blocks;
    const int64_t stride = warp_count();
    const int64_t c0 = warp_id();
    const int64_t K = c0 < nfull ? (nfull - c0 + stride - 1) / stride : 0;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < STAGES; st++) mbar_init(bar0 + 8 * st, 1);
        mbar_init_fence();
#pragma unroll
        for (int st = 0; st < STAGES; st++)
            if (st < K) op.issue(c0 + st * stride, buf0 + st * kStride, bar0 + 8 * st);
    }
    __syncwarp();
    for (int64_t k = 0; k < K; k++) {
        const int st = static_cast<int>(k % STAGES);
        const uint32_t parity = static_cast<uint32_t>((k / STAGES) & 1);
        if (!mbar_wait(bar0 + 8 * st, parity, kWaitLimitNs)) {
            // a copy did not complete in time: record it, let the copies still in
            // flight land (bounded) so no write reaches freed shared memory, and stop
            if (lane == 0) atomicAdd(&g_wait_timeouts, 1ull);
            for (int64_t j = k + 1; j < K && j < k + STAGES; j++)
                mbar_wait(bar0 + 8 * static_cast<int>(j % STAGES), static_cast<uint32_t>((j / STAGES) & 1),
                          kWaitLimitNs);
            return;
        }
        typename Op::In in;
        op.load_staged(in, buf + st * kStride);
        __syncwarp();
        if (lane == 0 && k + STAGES < K) {
            fence_proxy_async();
            op.issue(c0 + (k + STAGES) * stride, buf0 + st * kStride, bar0 + 8 * st);
        }
        op.template compute<false>(in, c0 + k * stride);
    }
    const int64_t c = c0 + K * stride;
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
    static constexpr uint32_t kStageBytes = 512u * SEGS;  // the chunk's BF16 values
    static_assert(kStageBytes % 16 == 0, "bulk copies move whole 16-byte units");
    __device__ __forceinline__ void issue(int64_t c, uint32_t stage, uint32_t bar) const
    {
        mbar_expect_tx(bar, kStageBytes);
        bulk_load(stage, x + c * (256 * SEGS), kStageBytes, bar);
    }
    __device__ __forceinline__ void load_staged(In &in, const unsigned char *stage) const
    {
#pragma unroll
        for (int j = 0; j < SEGS; j++) in.x[j] = *reinterpret_cast<const uint4 *>(stage + 512 * j + 16 * lane);
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

template <int SEGS, int STAGES>
__global__ void __launch_bounds__(kThreads)
quant_i8_staged_kernel(const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_begin();
    extern __shared__ __align__(128) unsigned char smem[];
    const QuantOp<SEGS> op{x, q, s, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS, smem + (threadIdx.x >> 5) * staged_warp_bytes<QuantOp<SEGS>, STAGES>());
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
    // staged inputs: the first W sources' payload runs, then their scale runs
    static constexpr uint32_t kPayloadBytes = 256u * SEGS, kScaleBytes = 8u * SEGS;
    static constexpr uint32_t kStageBytes = W * (kPayloadBytes + kScaleBytes);
    static_assert(kPayloadBytes % 16 == 0 && kScaleBytes % 16 == 0 && kStageBytes % 16 == 0,
                  "bulk copies move whole 16-byte units");
    __device__ __forceinline__ void issue(int64_t c, uint32_t stage, uint32_t bar) const
    {
        mbar_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int i = 0; i < W; i++) {
            bulk_load(stage + i * kPayloadBytes, src.q[i] + c * (256 * SEGS), kPayloadBytes, bar);
            bulk_load(stage + W * kPayloadBytes + i * kScaleBytes, src.s[i] + c * (2 * SEGS), kScaleBytes, bar);
        }
    }
    __device__ __forceinline__ void load_staged(In &in, const unsigned char *stage) const
    {
#pragma unroll
        for (int i = 0; i < W; i++) {
#pragma unroll
            for (int j = 0; j < SEGS; j++)
                in.q[i][j] = *reinterpret_cast<const uint2 *>(stage + i * kPayloadBytes + 256 * j + 8 * lane);
            in.sc[i] = lane < 2 * SEGS
                           ? *reinterpret_cast<const float *>(stage + W * kPayloadBytes + i * kScaleBytes + 4 * lane)
                           : 0.0f;
        }
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

#ifndef BQ_ACCUM_MIN_CTAS
#define BQ_ACCUM_MIN_CTAS 3
#endif

template <int SEGS, int W, bool kOut, int STAGES>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MIN_CTAS)
accum_i8_staged_kernel(const __grid_constant__ SourceList src, int nsrc, int64_t nblk, int8_t *__restrict__ q,
                       float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    extern __shared__ __align__(128) unsigned char smem[];
    const AccumOp<SEGS, W, kOut> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS,
                       smem + (threadIdx.x >> 5) * staged_warp_bytes<AccumOp<SEGS, W, kOut>, STAGES>());
}

template <int SEGS, int W, bool kOut>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MIN_CTAS)
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
    static constexpr uint32_t kQBytes = 256u * SEGS, kXBytes = 512u * SEGS, kSBytes = 8u * SEGS;
    static constexpr uint32_t kStageBytes = kQBytes + kXBytes + kSBytes;
    static_assert(kQBytes % 16 == 0 && kXBytes % 16 == 0 && kSBytes % 16 == 0 && kStageBytes % 16 == 0,
                  "bulk copies move whole 16-byte units");
    __device__ __forceinline__ void issue(int64_t c, uint32_t stage, uint32_t bar) const
    {
        mbar_expect_tx(bar, kStageBytes);
        bulk_load(stage, x + c * (256 * SEGS), kXBytes, bar);
        bulk_load(stage + kXBytes, q_in + c * (256 * SEGS), kQBytes, bar);
        bulk_load(stage + kXBytes + kQBytes, s_in + c * (2 * SEGS), kSBytes, bar);
    }
    __device__ __forceinline__ void load_staged(In &in, const unsigned char *stage) const
    {
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            in.x[j] = *reinterpret_cast<const uint4 *>(stage + 512 * j + 16 * lane);
            in.q[j] = *reinterpret_cast<const uint2 *>(stage + kXBytes + 256 * j + 8 * lane);
        }
        in.sc = lane < 2 * SEGS ? *reinterpret_cast<const float *>(stage + kXBytes + kQBytes + 4 * lane) : 0.0f;
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

template <int SEGS, bool kOut, int STAGES>
__global__ void __launch_bounds__(kThreads)
ring_hop_i8_staged_kernel(const int8_t *__restrict__ q_in, const float *__restrict__ s_in,
                          const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q,
                          float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    extern __shared__ __align__(128) unsigned char smem[];
    const HopOp<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS, smem + (threadIdx.x >> 5) * staged_warp_bytes<HopOp<SEGS, kOut>, STAGES>());
}

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

// Bulk-copy stages per warp (0: the kernel reads global memory directly). Measured on
// GB300: staging pays for the four-stream accumulate and costs for quantize.
#ifndef BQ_STAGES_QUANT
#define BQ_STAGES_QUANT 0
#endif
#ifndef BQ_STAGES_ACCUM
#define BQ_STAGES_ACCUM 0
#endif
#ifndef BQ_STAGES_HOP
#define BQ_STAGES_HOP 3
#endif
constexpr int kStagesQuant = BQ_STAGES_QUANT;
constexpr int kStagesHop = BQ_STAGES_HOP;
constexpr int kStagesAccum = BQ_STAGES_ACCUM;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Staged kernels keep STAGES bulk-copy slots per warp in dynamic shared memory.
template <class Op, int STAGES, class Kernel, class... Args>
cudaError_t launch_staged(Kernel kernel, int64_t nchunk, cudaStream_t st, Args... args)
{
    const size_t smem = (kThreads / 32) * staged_warp_bytes<Op, STAGES>();
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, nchunk, &grid, smem)) return e;
    return launch_kernel_smem(kernel, grid, smem, st, args...);
}

template <int W, bool kOut>
cudaError_t launch_accum_w(const SourceList &src, int nsrc, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                           cudaStream_t st)
{
    if constexpr (kStagesAccum > 0) {
        // Bulk copies need 16-byte aligned scale runs; scale pointers are only required
        // to be 4-byte aligned, so other alignments take the global-memory path.
        bool staged = true;
        for (int i = 0; i < W && i < nsrc; i++) staged = staged && aligned16(src.s[i]);
        if (staged)
            return launch_staged<AccumOp<kSegsAccum, W, kOut>, kStagesAccum>(
                accum_i8_staged_kernel<kSegsAccum, W, kOut, kStagesAccum>, chunks(nblk, kSegsAccum), st, src, nsrc,
                nblk, q, s, out);
    }
    auto kernel = accum_i8_kernel<kSegsAccum, W, kOut>;
    BQK_GRID(kernel, chunks(nblk, kSegsAccum));
    return launch_kernel(kernel, grid, st, src, nsrc, nblk, q, s, out);
}

}  // namespace

namespace {
template <int STAGES>
cudaError_t launch_quant_stages(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st)
{
    if constexpr (STAGES > 0)  // x is 16-byte aligned by contract
        return launch_staged<QuantOp<kSegsQuant>, STAGES>(quant_i8_staged_kernel<kSegsQuant, STAGES>,
                                                           chunks(nblk, kSegsQuant), st, x, nblk, q, s);
    BQK_GRID(quant_i8_kernel<kSegsQuant>, chunks(nblk, kSegsQuant));
    return launch_kernel(quant_i8_kernel<kSegsQuant>, grid, st, x, nblk, q, s);
}
}  // namespace

cudaError_t launch_quant_i8(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st)
{
    return launch_quant_stages<kStagesQuant>(x, nblk, q, s, st);
}

namespace {
// One warp waits, with a short limit, on a barrier that no thread arrives at and no
// copy completes: the bounded wait must give up and count the timeout.
__global__ void wait_selftest_kernel()
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_init_fence();
    }
    __syncwarp();
    const bool done = mbar_wait(b, 0, 20000000ull);  // 20 ms
    if (!done && threadIdx.x == 0) atomicAdd(&g_wait_timeouts, 1ull);
}
}  // namespace

cudaError_t launch_wait_selftest(cudaStream_t st)
{
    wait_selftest_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

cudaError_t take_wait_timeouts_i8(unsigned long long *count)
{
    unsigned long long zero = 0;
    if (cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof zero)) return e;
    return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof zero);
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

namespace {
template <int STAGES, bool kOut>
cudaError_t launch_hop_stages(const int8_t *q_in, const float *s_in, const uint16_t *x, int64_t nblk, int8_t *q,
                              float *s, uint16_t *out, cudaStream_t st)
{
    if constexpr (STAGES > 0) {
        // the incoming scales are only required to be 4-byte aligned
        if (aligned16(s_in))
            return launch_staged<HopOp<kSegsHop, kOut>, STAGES>(ring_hop_i8_staged_kernel<kSegsHop, kOut, STAGES>,
                                                                 chunks(nblk, kSegsHop), st, q_in, s_in, x, nblk, q, s,
                                                                 out);
    }
    BQK_GRID((ring_hop_i8_kernel<kSegsHop, kOut>), chunks(nblk, kSegsHop));
    return launch_kernel(ring_hop_i8_kernel<kSegsHop, kOut>, grid, st, q_in, s_in, x, nblk, q, s, out);
}
}  // namespace

cudaError_t launch_ring_hop_i8(const int8_t *q_in, const float *s_in, const uint16_t *x, int64_t nblk, int8_t *q,
                               float *s, uint16_t *out, cudaStream_t st)
{
    if (out) return launch_hop_stages<kStagesHop, true>(q_in, s_in, x, nblk, q, s, out, st);
    return launch_hop_stages<kStagesHop, false>(q_in, s_in, x, nblk, q, s, nullptr, st);
}

}  // namespace bqk
