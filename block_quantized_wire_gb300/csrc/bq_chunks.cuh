// Warp-chunk drivers and the codec operations shared by the wire formats: quantize,
// materialize, the all-to-all accumulate, the ring hop, and the all-gather modes'
// reduce + quantize.
//
// Every wire carries, per 128-value block, 128 payload bytes and 4 scale bytes: one
// FP32 scale for block INT8 ("feat(pcie_dma): add block-INT8 wire modes for AG,
// ring, and A2A", Summary) and for the legacy E4M3 codec it compares against, and four
// E8M0 bytes, one per 32 values, for MXFP8 ("feat(pcie_dma): add INT8 and MXFP8 wire
// modes", Summary). A flat wire of n values is the payload [n] followed by the scale
// words [n/128], so the same loads serve all three; a codec policy supplies what
// differs:
//
//   struct Codec {
//     using Q = payload element type;  using S = 4-byte scale word type;
//     // exact binary32 values of a lane's 8 payload elements, given the scale word
//     // of the lane's block
//     static void decode8(uint2 payload, uint32_t word, int lane, float2 (&d)[4]);
//     // quantize a chunk of binary32 values: payload, scale words and, when kOut,
//     // the BF16 materialization of the new payload
//     template <int SEGS, bool kTail, bool kOut>
//     static void requant(const float2 (&v)[SEGS][4], int64_t e0, int64_t b0,
//                         int64_t nblk, int lane, Q *q, S *s, uint16_t *out);
//     // BF16 materialization of a lane's 8 payload elements
//     static uint4 dequant8(uint2 payload, uint32_t word, int lane);
//   };
// (a policy defines only what the ops it is used with call).
//
// The reductions are the all-to-all accumulate (sources decoded and added left to
// right in source order in binary32, then requantized) and the ring hop (incoming
// wire decoded, plus the local BF16 shard, then requantized), the Implementation
// section of the block-INT8 page; the MXFP8 page's Summary runs the same topologies
// (mx_a2a, mx_ring) with its codec.
//
// Decomposition: a warp processes a chunk of SEGS segments of 256 values; in segment
// j lane l holds values [256j + 8l, 256j + 8l + 8) of the chunk, so half-warp h holds
// block 2j + h and lanes 0..2*SEGS-1 hold the chunk's scale words.
#pragma once

#include "bq_device.cuh"
#include "bq_launch.h"

namespace bqk {
namespace {

// Warp index in the grid and number of warps, for a kernel launched with kBlock threads
// per CTA (kThreads unless the kernel and its launch both say otherwise).
template <int kBlock = kThreads>
__device__ __forceinline__ int64_t warp_id()
{
    return ((int64_t)blockIdx.x * kBlock + threadIdx.x) >> 5;
}
template <int kBlock = kThreads>
__device__ __forceinline__ int64_t warp_count()
{
    return ((int64_t)gridDim.x * kBlock) >> 5;
}

// Grid-stride driver over warp chunks. With kPrefetch, the loads of a warp's next
// chunk (c + number of warps) are issued before chunk c is computed (a register
// pipeline; it pays only where registers are cheap, as in materialize). Op provides
//   In                                 registers holding one chunk's inputs
//   load<kTail>(In&, c) / compute<kTail>(const In&, c)
// Full chunks use kTail = false (no bounds checks); the one partial chunk, if any,
// is loaded and computed by the warp whose stride lands on it. kBlock: threads per CTA
// of the launch.
template <bool kPrefetch, int kBlock = kThreads, class Op>
__device__ __forceinline__ void run_chunks(const Op &op, int64_t nblk, int chunk_blocks)
{
    const int64_t nfull = nblk / chunk_blocks;
    const int64_t stride = warp_count<kBlock>();
    int64_t c = warp_id<kBlock>();
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

// A warp's shared-memory stage for one chunk's inputs copied lane by lane: NV4 slots
// of 16 bytes and NU32 slots of 4 bytes per lane. Slot k of lane l sits at
// (32k + l) * 16 (then (32k + l) * 4 after the 16-byte slots), so a warp reading one
// slot reads 512 (or 128) contiguous bytes, free of bank conflicts.
template <int NV4, int NU32>
struct LaneSlots {
    static constexpr uint32_t kBytes = NV4 * 512u + NU32 * 128u;
    const unsigned char *p;  // the stage, generic address
    uint32_t a;              // the stage, shared-window address
    int lane;
    __device__ __forceinline__ void copy_v4(int k, const void *src) const
    {
        lane_copy16(a + (32u * k + lane) * 16u, src);
    }
    __device__ __forceinline__ void copy_u32(int k, const void *src) const
    {
        lane_copy4(a + NV4 * 512u + (32u * k + lane) * 4u, src);
    }
    __device__ __forceinline__ uint4 v4(int k) const
    {
        return *reinterpret_cast<const uint4 *>(p + (32u * k + lane) * 16u);
    }
    __device__ __forceinline__ uint32_t u32(int k) const
    {
        return *reinterpret_cast<const uint32_t *>(p + NV4 * 512u + (32u * k + lane) * 4u);
    }
};

// The wide accumulates' inputs for one full chunk c of exactly W sources, as per-lane
// copies: each source's 16 payload bytes in both 512-value segments (slots 2i, 2i + 1)
// and, in lanes 0..7, the scale word of the chunk's block `lane` (slot i). take fills
// the accumulates' In {q[W][2], sc[W]} exactly as their global-memory load does.
template <int W, class List>
__device__ __forceinline__ void issue_wide_sources(const LaneSlots<2 * W, W> &sl, const List &src, int64_t c,
                                                   int lane)
{
    const int64_t e0 = c * 1024 + lane * 16, b0 = c * 8;
#pragma unroll
    for (int i = 0; i < W; i++)
#pragma unroll
        for (int j = 0; j < 2; j++) sl.copy_v4(2 * i + j, src.q[i] + e0 + 512 * j);
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < W; i++) sl.copy_u32(i, src.s[i] + b0 + lane);
    }
}

template <int W, class In>
__device__ __forceinline__ void take_wide_sources(In &in, const LaneSlots<2 * W, W> &sl, int lane)
{
#pragma unroll
    for (int i = 0; i < W; i++) {
#pragma unroll
        for (int j = 0; j < 2; j++) in.q[i][j] = sl.v4(2 * i + j);
        in.sc[i] = lane < 8 ? sl.u32(i) : 0u;  // lanes 8..31 copied no scale word
    }
}

// Grid-stride driver whose loads run STAGES - 1 chunks ahead through per-lane async
// copies into the warp's STAGES stages (warp_smem, STAGES * Op::Slots::kBytes bytes):
// before chunk c is computed, the copies of chunk c + (STAGES - 1) * stride are issued,
// so the warp's next inputs are in flight while it computes and hold no registers.
// Op additionally provides
//   Slots                               a LaneSlots type
//   issue(const Slots&, c)              the lane's copies of full chunk c
//   take(In&, const Slots&)             fill In from the stage, as load<false> would
// The stage refilled in an iteration is the one the previous iteration read; those reads
// fed that chunk's results, which were stored before the new copies are issued, so no
// copy lands in bytes still to be read. The ragged last chunk, if any, takes the
// global-memory path. kBlock: threads per CTA of the launch.
template <int STAGES, int kBlock = kThreads, class Op>
__device__ __forceinline__ void run_chunks_lane_async(const Op &op, int64_t nblk, int chunk_blocks,
                                                      unsigned char *warp_smem)
{
    using Slots = typename Op::Slots;
    const int lane = threadIdx.x & 31;
    const uint32_t a0 = smem_u32(warp_smem);
    const int64_t nfull = nblk / chunk_blocks;
    const int64_t stride = warp_count<kBlock>();
    int64_t c = warp_id<kBlock>();
    if (c < nfull) {
#pragma unroll
        for (int k = 0; k < STAGES - 1; k++) {
            if (c + k * stride < nfull)
                op.issue(Slots{warp_smem + k * Slots::kBytes, a0 + k * Slots::kBytes, lane}, c + k * stride);
            lane_copy_commit();  // empty groups keep the count of groups in flight fixed
        }
        int st = 0;
        while (true) {
            const int64_t ahead = c + (STAGES - 1) * stride;
            const int fst = (st + STAGES - 1) % STAGES;
            if (ahead < nfull)
                op.issue(Slots{warp_smem + fst * Slots::kBytes, a0 + fst * Slots::kBytes, lane}, ahead);
            lane_copy_commit();
            lane_copy_wait<STAGES - 1>();  // chunk c's group has completed
            typename Op::In in;
            op.take(in, Slots{warp_smem + st * Slots::kBytes, a0 + st * Slots::kBytes, lane});
            op.template compute<false>(in, c);
            c += stride;
            st = (st + 1) % STAGES;
            if (c >= nfull) break;
        }
    }
    lane_copy_wait<0>();
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
        // lanes poll on their own clocks; the warp gives up only together
        if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * st, parity, kWaitLimitNs))) {
            // a copy did not complete in time: record it, give the copies still in
            // flight (this one included) time to land, each wait bounded, and stop. No
            // write reaches shared memory after the block exits only if every one of
            // them lands within its limit; one that does not is counted separately.
            if (lane == 0) atomicAdd(&g_wait_timeouts, 1ull);
            for (int64_t j = k; j < K && j < k + STAGES; j++) {
                const bool landed = mbar_wait(bar0 + 8 * static_cast<int>(j % STAGES),
                                              static_cast<uint32_t>((j / STAGES) & 1), kWaitLimitNs);
                if (!__all_sync(0xffffffffu, landed)) {
                    if (lane == 0) atomicAdd(&g_wait_unlanded, 1ull);
                    break;
                }
            }
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

// ---------------------------------------------------------------- quantize
// kRewiden: the chunk goes to the codec's requantization as its raw BF16 words, widened
// again for each read (Bf16Vals), instead of as FP32 values widened once (RegVals);
// fewer registers for one more widening.
template <class Codec, int SEGS, bool kRewiden = false>
struct QuantOp {
    const uint16_t *__restrict__ x;
    typename Codec::Q *__restrict__ q;
    typename Codec::S *__restrict__ s;
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
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
        if constexpr (kRewiden) {
            Codec::template requant<SEGS, kTail, false>(Bf16Vals<SEGS>{in.x}, e0, b0, nblk, lane, q, s, nullptr);
        } else {
            float2 v[SEGS][4];
#pragma unroll
            for (int j = 0; j < SEGS; j++) bf16x8_to_f32(in.x[j], v[j]);
            Codec::template requant<SEGS, kTail, false>(RegVals<SEGS>{v}, e0, b0, nblk, lane, q, s, nullptr);
        }
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

// ---------------------------------------------------------------- materialize
template <class Codec, int SEGS>
struct DequantOp {
    const typename Codec::Q *__restrict__ q;
    const typename Codec::S *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint2 q[SEGS];
        uint32_t sc;
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
#pragma unroll
        for (int j = 0; j < SEGS; j++)
            in.q[j] = (!kTail || b0 + 2 * j + (lane >> 4) < nblk) ? ld_stream_v2(q + e0 + 256 * j) : make_uint2(0, 0);
        in.sc = (lane < 2 * SEGS && (!kTail || b0 + lane < nblk)) ? ld_stream_u32(s + b0 + lane) : 0u;
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
        const int half = lane >> 4;
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            const uint32_t wj = __shfl_sync(kFull, in.sc, 2 * j + half);
            if (!kTail || b0 + 2 * j + half < nblk) st_v4(out + e0 + 256 * j, Codec::dequant8(in.q[j], wj, lane));
        }
    }
};

// ---------------------------------------------------------------- reduce + quantize
// The all-gather modes' BF16 reduce-scatter fused with quantization of its result: the
// W ranks' BF16 shards are added left to right in rank order in binary32, the sum is
// rounded once to BF16 (the reduce-scatter's result) and widened back exactly, and the
// codec quantizes it. The first W sources are loaded together; further sources in
// groups of W.
template <int SEGS, int W>
struct Bf16Regs {
    uint4 x[W][SEGS];
};

// kMore: further source groups may follow, so a source slot may be past the last source
// (without it the launch has exactly W sources and carries no source-count checks).
template <int SEGS, int W, bool kTail, bool kMore = true>
__device__ __forceinline__ void load_bf16_sources(Bf16Regs<SEGS, W> &r, const Bf16List &src, int g, int nsrc,
                                                  int64_t c, int64_t nblk, int lane)
{
    const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
#pragma unroll
    for (int i = 0; i < W; i++) {
        const bool src_ok = !kMore || g + i < nsrc;
        const uint16_t *xw = src.x[src_ok ? g + i : g];
#pragma unroll
        for (int j = 0; j < SEGS; j++)
            r.x[i][j] = (src_ok && (!kTail || b0 + 2 * j + (lane >> 4) < nblk)) ? ld_stream_v4(xw + e0 + 256 * j)
                                                                                 : make_uint4(0, 0, 0, 0);
    }
}

template <int SEGS, int W, bool kFirst, bool kMore = true>
__device__ __forceinline__ void add_bf16_sources(const Bf16Regs<SEGS, W> &r, int g, int nsrc, float2 (&acc)[SEGS][4])
{
#pragma unroll
    for (int i = 0; i < W; i++) {
        if (kMore && g + i >= nsrc) break;
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            float2 v[4];
            bf16x8_to_f32(r.x[i][j], v);
#pragma unroll
            for (int e = 0; e < 4; e++) acc[j][e] = (kFirst && i == 0) ? v[e] : add2(acc[j][e], v[e]);
        }
    }
}

template <class Codec, int SEGS, int W, bool kOut, bool kMore = true>
struct ReduceQuantOp {
    const Bf16List &src;  // the kernel's __grid_constant__ parameter, read in place
    int nsrc;
    typename Codec::Q *__restrict__ q;
    typename Codec::S *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    using In = Bf16Regs<SEGS, W>;
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        load_bf16_sources<SEGS, W, kTail, kMore>(in, src, 0, nsrc, c, nblk, lane);
    }
    // per-lane async copies (run_chunks_lane_async), for exactly W sources: source i's
    // 16 bytes of segment j in slot SEGS * i + j
    using Slots = LaneSlots<W * SEGS, 0>;
    __device__ __forceinline__ void issue(const Slots &sl, int64_t c) const
    {
        static_assert(!kMore, "the async driver serves launches of exactly W sources");
        const int64_t e0 = c * (256 * SEGS) + lane * 8;
#pragma unroll
        for (int i = 0; i < W; i++)
#pragma unroll
            for (int j = 0; j < SEGS; j++) sl.copy_v4(SEGS * i + j, src.x[i] + e0 + 256 * j);
    }
    __device__ __forceinline__ void take(In &in, const Slots &sl) const
    {
#pragma unroll
        for (int i = 0; i < W; i++)
#pragma unroll
            for (int j = 0; j < SEGS; j++) in.x[i][j] = sl.v4(SEGS * i + j);
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 acc[SEGS][4];
        add_bf16_sources<SEGS, W, true, kMore>(in, 0, nsrc, acc);
        if constexpr (kMore) {
            for (int g = W; g < nsrc; g += W) {
                In more;
                load_bf16_sources<SEGS, W, kTail>(more, src, g, nsrc, c, nblk, lane);
                add_bf16_sources<SEGS, W, false>(more, g, nsrc, acc);
            }
        }
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            const uint4 rounded = f32x8_to_bf16x8(acc[j]);  // the reduce-scatter's BF16 result
            bf16x8_to_f32(rounded, acc[j]);
        }
        Codec::template requant<SEGS, kTail, kOut>(RegVals<SEGS>{acc}, c * (256 * SEGS) + lane * 8, c * (2 * SEGS),
                                                   nblk, lane, q, s, out);
    }
};

// The reduce + quantize of exactly W (<= 4) sources with each warp's next chunk in
// flight through per-lane async copies, one CTA of kReduceAsyncThreads per SM (all of
// an SM's warps at the same age): 649 against 682 us for four 469.8M-value BF16 sources
// on GB300, for either codec. Each codec's translation unit wraps the body in its
// own kernel; launch_reduce_async (with the host-side helpers below) sizes the stages
// and the grid.
#ifndef BQ_REDUCE_ASYNC
#define BQ_REDUCE_ASYNC 1
#endif
#ifndef BQ_REDUCE_ASYNC_THREADS
#define BQ_REDUCE_ASYNC_THREADS 512
#endif
constexpr int kReduceAsyncThreads = BQ_REDUCE_ASYNC_THREADS;
constexpr int kReduceAsyncStages = 2;
constexpr int kReduceAsyncMinCtas = kReduceAsyncThreads >= 512 ? 1 : 512 / kReduceAsyncThreads;

template <class Codec, int SEGS, int W, bool kOut>
__device__ __forceinline__ void reduce_quant_async_body(const Bf16List &src, int nsrc, int64_t nblk,
                                                        typename Codec::Q *q, typename Codec::S *s, uint16_t *out,
                                                        unsigned char *stages)
{
    using Op = ReduceQuantOp<Codec, SEGS, W, kOut, false>;
    const Op op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks_lane_async<kReduceAsyncStages, kReduceAsyncThreads>(
        op, nblk, 2 * SEGS, stages + (threadIdx.x >> 5) * kReduceAsyncStages * Op::Slots::kBytes);
}

// ---------------------------------------------------------------- accumulate
// Sources are summed in source order 0..nsrc-1. The first W sources of a chunk are
// loaded together; any further sources are loaded in groups of W with the running
// sum carried in registers.
template <int SEGS, int W>
struct SourceRegs {
    uint2 q[W][SEGS];
    uint32_t sc[W];  // lane < 2*SEGS: scale word of the chunk's block `lane`
};

template <int SEGS, int W, bool kTail, class List>
__device__ __forceinline__ void load_sources(SourceRegs<SEGS, W> &r, const List &src, int g, int nsrc, int64_t c,
                                             int64_t nblk, int lane)
{
    const int64_t e0 = c * (256 * SEGS) + lane * 8, b0 = c * (2 * SEGS);
    const bool lane_ok = lane < 2 * SEGS && (!kTail || b0 + lane < nblk);
#pragma unroll
    for (int i = 0; i < W; i++) {
        const bool src_ok = g + i < nsrc;
        const auto *qw = src.q[src_ok ? g + i : g];
        const auto *sw = src.s[src_ok ? g + i : g];
#pragma unroll
        for (int j = 0; j < SEGS; j++)
            r.q[i][j] = (src_ok && (!kTail || b0 + 2 * j + (lane >> 4) < nblk)) ? ld_stream_v2(qw + e0 + 256 * j)
                                                                                 : make_uint2(0, 0);
        r.sc[i] = (src_ok && lane_ok) ? ld_stream_u32(sw + b0 + lane) : 0u;
    }
}

template <class Codec, int SEGS, int W, bool kFirst>
__device__ __forceinline__ void add_sources(const SourceRegs<SEGS, W> &r, int g, int nsrc, float2 (&acc)[SEGS][4],
                                            int lane)
{
    const int half = lane >> 4;
#pragma unroll
    for (int i = 0; i < W; i++) {
        if (g + i >= nsrc) break;
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            float2 d[4];
            Codec::decode8(r.q[i][j], __shfl_sync(kFull, r.sc[i], 2 * j + half), lane, d);
#pragma unroll
            for (int e = 0; e < 4; e++) acc[j][e] = (kFirst && i == 0) ? d[e] : add2(acc[j][e], d[e]);
        }
    }
}

// kMore: the call may have more than W sources, added W at a time after the first
// group; without it the operation serves nsrc <= W and keeps no registers for a
// second group (the four-source kernel spilled with them).
template <class Codec, int SEGS, int W, bool kOut, bool kMore = true>
struct AccumOp {
    using Q = typename Codec::Q;
    using S = typename Codec::S;
    const WireList<Q, S> &src;  // the kernel's __grid_constant__ parameter, read in place
    int nsrc;
    Q *__restrict__ q;
    S *__restrict__ s;
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
                           ? *reinterpret_cast<const uint32_t *>(stage + W * kPayloadBytes + i * kScaleBytes + 4 * lane)
                           : 0u;
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 acc[SEGS][4];
        add_sources<Codec, SEGS, W, true>(in, 0, nsrc, acc, lane);
        if constexpr (kMore) {
            for (int g = W; g < nsrc; g += W) {
                In more;
                load_sources<SEGS, W, kTail>(more, src, g, nsrc, c, nblk, lane);
                add_sources<Codec, SEGS, W, false>(more, g, nsrc, acc, lane);
            }
        }
        Codec::template requant<SEGS, kTail, kOut>(RegVals<SEGS>{acc}, c * (256 * SEGS) + lane * 8, c * (2 * SEGS),
                                                   nblk, lane, q, s, out);
    }
};

// ---------------------------------------------------------------- ring hop
template <class Codec, int SEGS, bool kOut>
struct HopOp {
    using Q = typename Codec::Q;
    using S = typename Codec::S;
    const Q *__restrict__ q_in;
    const S *__restrict__ s_in;
    const uint16_t *__restrict__ x;
    Q *__restrict__ q;
    S *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint2 q[SEGS];
        uint4 x[SEGS];
        uint32_t sc;
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
        in.sc = (lane < 2 * SEGS && (!kTail || b0 + lane < nblk)) ? ld_stream_u32(s_in + b0 + lane) : 0u;
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
        in.sc = lane < 2 * SEGS ? *reinterpret_cast<const uint32_t *>(stage + kXBytes + kQBytes + 4 * lane) : 0u;
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        const int half = lane >> 4;
        float2 v[SEGS][4];
#pragma unroll
        for (int j = 0; j < SEGS; j++) {
            float2 d[4], xl[4];
            Codec::decode8(in.q[j], __shfl_sync(kFull, in.sc, 2 * j + half), lane, d);
            bf16x8_to_f32(in.x[j], xl);
#pragma unroll
            for (int e = 0; e < 4; e++) v[j][e] = add2(d[e], xl[e]);
        }
        Codec::template requant<SEGS, kTail, kOut>(RegVals<SEGS>{v}, c * (256 * SEGS) + lane * 8, c * (2 * SEGS),
                                                   nblk, lane, q, s, out);
    }
};

// ---------------------------------------------------------------- host-side launch helpers
int64_t chunks(int64_t nblk, int segs) { return (nblk + 2 * segs - 1) / (2 * segs); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Staged kernels keep STAGES bulk-copy slots per warp in dynamic shared memory.
template <class Op, int STAGES, class Kernel, class... Args>
cudaError_t launch_staged(Kernel kernel, int64_t nchunk, cudaStream_t st, Args... args)
{
    const size_t smem = (kThreads / 32) * staged_warp_bytes<Op, STAGES>();
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, nchunk, &grid, smem)) return e;
    return launch_kernel_smem(kernel, grid, smem, st, args...);
}

// The async reduce + quantize (reduce_quant_async_body) of exactly W sources.
template <class Codec, int SEGS, int W, bool kOut, typename... KArgs, typename... Args>
cudaError_t launch_reduce_async(void (*kernel)(KArgs...), int64_t nblk, cudaStream_t st, Args... args)
{
    const size_t smem =
        (kReduceAsyncThreads / 32) * kReduceAsyncStages * ReduceQuantOp<Codec, SEGS, W, kOut, false>::Slots::kBytes;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, SEGS), &grid, smem, kReduceAsyncThreads)) return e;
    return launch_kernel_block(kernel, grid, kReduceAsyncThreads, smem, st, args...);
}

}  // namespace
}  // namespace bqk

#define BQK_GRID(kernel, nchunk)                                          \
    int grid = 0;                                                         \
    if (cudaError_t e_ = bqk::grid_for((const void *)(kernel), (nchunk), &grid)) \
        return e_;
