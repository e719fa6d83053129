// Block-INT8 codec kernels: quantize, materialize, multi-source accumulate, ring hop.
//
// Operations from "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A",
// Implementation (the four kernels) and Summary (128 values per block, one FP32
// scale = amax/127, owners materialize the forwarded payload).
//
// Decomposition (bq_chunks.cuh): per chunk, the block amaxes are gathered into lanes
// 0..2*SEGS-1, which compute the chunk's scales once; the scales are then broadcast
// back per segment and stored by those lanes in one coalesced store. Full chunks run
// without bounds checks; the one partial chunk at the end (n not a multiple of the
// chunk) runs the same code with checks.
#include "bq_chunks.cuh"

namespace bqk {
namespace {

// Requantize SEGS segments of FP32 values (v[j] = lane's 8 values of segment j):
// writes the payload, the chunk's scales and, when kOut, the BF16 materialization.
template <int SEGS, bool kTail, bool kOut, class Vals>
__device__ __forceinline__ void requant_chunk(const Vals &vals, int64_t e0, int64_t b0, int64_t nblk, int lane,
                                              int8_t *__restrict__ q, float *__restrict__ s,
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
    const I8Scale mine = i8_block_scale(gather_amax<SEGS>(m, lane));
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        I8Scale bj;
        bj.s = __shfl_sync(kFull, mine.s, 2 * j + half);
        bj.r = __shfl_sync(kFull, mine.r, 2 * j + half);
        bj.rl = __shfl_sync(kFull, mine.rl, 2 * j + half);
        float2 v[4];
        vals.seg(j, v);
        uint32_t w[8];
        i8_quant8(v, bj, w);
        if (!kTail || b0 + 2 * j + half < nblk) {
            st_v2(q + e0 + 256 * j, pack_payload8(w));
            if (kOut) st_v4(out + e0 + 256 * j, i8_materialize_words(w, bj.s));
        }
    }
    if (lane < 2 * SEGS && (!kTail || b0 + lane < nblk) && dbg_ok(s + b0 + lane, 4, true)) s[b0 + lane] = mine.s;
}

// Block-INT8 codec policy for the shared reductions: d = fl(q * s) per element
// (the product is kept unfused from the sum that consumes it), requantization as
// in quantize.
struct I8Codec {
    using Q = int8_t;
    using S = float;
    static __device__ __forceinline__ void decode8(uint2 q, uint32_t word, int, float2 (&d)[4])
    {
        const float2 s = splat(__uint_as_float(word));
        float2 v[4];
        i8x8_to_f32(q, v);
#pragma unroll
        for (int e = 0; e < 4; e++) d[e] = mul2_unfused(v[e], s);
    }
    template <int SEGS, bool kTail, bool kOut, class Vals>
    static __device__ __forceinline__ void requant(const Vals &vals, int64_t e0, int64_t b0, int64_t nblk, int lane,
                                                   int8_t *q, float *s, uint16_t *out)
    {
        requant_chunk<SEGS, kTail, kOut>(vals, e0, b0, nblk, lane, q, s, out);
    }
    static __device__ __forceinline__ uint4 dequant8(uint2 q, uint32_t word, int)
    {
        float2 v[4];
        i8x8_to_f32(q, v);
        return i8_materialize8(v, __uint_as_float(word));
    }
};

// ---------------------------------------------------------------- quantize
template <int SEGS>
using QuantI8 = QuantOp<I8Codec, SEGS>;

// Quantize at 4 resident CTAs per SM (64 registers): 226.7 us per 469.8M-value launch
// on GB300. Left to the compiler it takes 72 registers and 3 CTAs per SM (245 us); 8
// segments per chunk took 241 us at 3 CTAs per SM and 449 us (spilling) at 4.
#ifndef BQ_QUANT_MIN_CTAS
#define BQ_QUANT_MIN_CTAS 4
#endif

template <int SEGS>
__global__ void __launch_bounds__(kThreads, BQ_QUANT_MIN_CTAS)
quant_i8_kernel(const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_begin();
    dbg_begin();
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_ready();
    const QuantI8<SEGS> op{x, q, s, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

template <int SEGS, int STAGES>
__global__ void __launch_bounds__(kThreads)
quant_i8_staged_kernel(const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_begin();
    dbg_begin();
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_ready();
    extern __shared__ __align__(128) unsigned char smem[];
    const QuantI8<SEGS> op{x, q, s, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS, smem + (threadIdx.x >> 5) * staged_warp_bytes<QuantI8<SEGS>, STAGES>());
}

// ---------------------------------------------------------------- materialize
template <int SEGS>
using DequantI8 = DequantOp<I8Codec, SEGS>;

// Threads per CTA of the INT8 materialization: 256, 512 and 768 measured the same in the
// prefill step (225.3 us per launch); 1024 was slower in an A/B (243.9 against 241.5 us).
#ifndef BQ_DEQUANT_I8_THREADS
#define BQ_DEQUANT_I8_THREADS 256
#endif
constexpr int kDequantI8Threads = BQ_DEQUANT_I8_THREADS;

template <int SEGS>
__global__ void __launch_bounds__(kDequantI8Threads)
dequant_i8_kernel(const int8_t *__restrict__ q, const float *__restrict__ s, int64_t nblk, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q, s, nblk, false);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const DequantI8<SEGS> op{q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<true, kDequantI8Threads>(op, nblk, 2 * SEGS);
}

// ---------------------------------------------------------------- accumulate
template <int SEGS, int W, bool kOut, bool kMore>
using AccumI8 = AccumOp<I8Codec, SEGS, W, kOut, kMore>;

#ifndef BQ_ACCUM_MIN_CTAS
#define BQ_ACCUM_MIN_CTAS 3
#endif

template <int SEGS, int W, bool kOut, bool kMore, int STAGES>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MIN_CTAS)
accum_i8_staged_kernel(const __grid_constant__ SourceList src, int nsrc, int64_t nblk, int8_t *__restrict__ q,
                       float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    extern __shared__ __align__(128) unsigned char smem[];
    const AccumI8<SEGS, W, kOut, kMore> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS,
                       smem + (threadIdx.x >> 5) * staged_warp_bytes<AccumI8<SEGS, W, kOut, kMore>, STAGES>());
}

template <int SEGS, int W, bool kOut, bool kMore>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MIN_CTAS)
accum_i8_kernel(const __grid_constant__ SourceList src, int nsrc, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s,
                uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const AccumI8<SEGS, W, kOut, kMore> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

// ---------------------------------------------------------------- wide lanes
// Quantize and accumulate laid out for fewer instructions per value. A lane takes 16
// consecutive values (one 16-byte payload word, two 16-byte BF16 words) instead of 8,
// so a 128-value block spans 8 lanes; a warp chunk is two such 512-value segments, the
// same 8 blocks as the 4-segment layout. The block amax then takes a 3-step butterfly
// over twice the values per lane, and the scale shuffles, the loads and the payload
// stores halve per value. The arithmetic and its order are those of the 8-value layout.
__device__ __forceinline__ float octet_max(float m)
{
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
    return m;
}

// Requantize one wide chunk: v[j][h] are the lane's values 8h..8h+7 of segment j
// (elements e0 + 512 j + 8 h ...), whose block is b0 + 4 j + (lane >> 3). Writes the
// payload, the chunk's 8 scales and, when kOut, the BF16 materialization.
// kV8: out is 32-byte aligned and the lane's 16 BF16 values go out in one 256-bit store.
template <bool kTail, bool kOut, bool kV8>
__device__ __forceinline__ void requant_wide(const float2 (&v)[2][2][4], int64_t e0, int64_t b0, int64_t nblk,
                                             int lane, int8_t *__restrict__ q, float *__restrict__ s,
                                             uint16_t *__restrict__ out)
{
    const int g = lane >> 3;
    float m[2];
#pragma unroll
    for (int j = 0; j < 2; j++) m[j] = octet_max(amax16(v[j][0], v[j][1]));
    // lane b < 8 computes the scale of the chunk's block b: segment b / 4, lane group b % 4
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const float gm = __shfl_sync(kFull, m[j], (lane & 3) << 3);
        if ((lane >> 2) == j) mine = gm;
    }
    const I8Scale sb = i8_block_scale(mine);
    // one warp-uniform choice per chunk: the reciprocal path for all 8 blocks (every
    // scale >= 2^-100, the rule for real data) or the per-block choice
    const bool fast = __all_sync(kFull, sb.r >= 0.0f);
#pragma unroll
    for (int j = 0; j < 2; j++) {
        I8Scale bj;
        bj.s = __shfl_sync(kFull, sb.s, 4 * j + g);
        bj.r = __shfl_sync(kFull, sb.r, 4 * j + g);
        bj.rl = __shfl_sync(kFull, sb.rl, 4 * j + g);
        uint32_t w0[8], w1[8];
        if (fast) {
            i8_quant8_fast(v[j][0], bj, w0);
            i8_quant8_fast(v[j][1], bj, w1);
        } else {
            i8_quant8(v[j][0], bj, w0);
            i8_quant8(v[j][1], bj, w1);
        }
        if (!kTail || b0 + 4 * j + g < nblk) {
            const uint2 p0 = pack_payload8(w0), p1 = pack_payload8(w1);
            st_v4(q + e0 + 512 * j, make_uint4(p0.x, p0.y, p1.x, p1.y));
            if (kOut) {
                const uint4 o0 = i8_materialize_words(w0, bj.s), o1 = i8_materialize_words(w1, bj.s);
                if (kV8) {
                    st_v8(out + e0 + 512 * j, o0, o1);
                } else {
                    st_v4(out + e0 + 512 * j, o0);
                    st_v4(out + e0 + 512 * j + 8, o1);
                }
            }
        }
    }
    if (lane < 8 && (!kTail || b0 + lane < nblk) && dbg_ok(s + b0 + lane, 4, true)) s[b0 + lane] = sb.s;
}

template <bool kV8>
__device__ __forceinline__ void load_bf16x16(const uint16_t *p, bool ok, uint4 (&w)[2])
{
    if (!ok) {
        w[0] = w[1] = make_uint4(0, 0, 0, 0);
    } else if (kV8) {
        ld_stream_v8(p, w[0], w[1]);
    } else {
        w[0] = ld_stream_v4(p);
        w[1] = ld_stream_v4(p + 8);
    }
}

// Quantize: the lane's 16 BF16 values are two 16-byte words per segment, read in one
// 256-bit access when kV8 (x 32-byte aligned).
template <bool kV8>
struct QuantWideI8 {
    const uint16_t *__restrict__ x;
    int8_t *__restrict__ q;
    float *__restrict__ s;
    int64_t nblk;
    int lane;
    struct In {
        uint4 x[2][2];
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * 1024 + lane * 16, b0 = c * 8;
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const bool ok = !kTail || b0 + 4 * j + (lane >> 3) < nblk;
            load_bf16x16<kV8>(x + e0 + 512 * j, ok, in.x[j]);
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 v[2][2][4];
#pragma unroll
        for (int j = 0; j < 2; j++)
#pragma unroll
            for (int h = 0; h < 2; h++) bf16x8_to_f32(in.x[j][h], v[j][h]);
        requant_wide<kTail, false, false>(v, c * 1024 + lane * 16, c * 8, nblk, lane, q, s, nullptr);
    }
};

// Accumulate of W sources at a time (kMore: further groups of W follow the first).
// Without kMore the launch has exactly W sources, so the source loop carries no
// source-count checks (on GB300 the checks and pointer selects cost 2.5 instructions
// per value and 6% of the four-source launch's time).
template <int W, bool kOut, bool kMore, bool kV8>
struct AccumWideI8 {
    const SourceList &src;  // the kernel's __grid_constant__ parameter, read in place
    int nsrc;
    int8_t *__restrict__ q;
    float *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint4 q[W][2];
        uint32_t sc[W];  // lanes 0..7: the scales of the chunk's blocks 0..7
    };
    template <bool kTail>
    __device__ __forceinline__ void load_group(In &in, int gsrc, int64_t c) const
    {
        const int64_t e0 = c * 1024 + lane * 16, b0 = c * 8;
        const int g = lane >> 3;
        const bool lane_ok = lane < 8 && (!kTail || b0 + lane < nblk);
#pragma unroll
        for (int i = 0; i < W; i++) {
            const bool src_ok = !kMore || gsrc + i < nsrc;
            const int8_t *qw = src.q[src_ok ? gsrc + i : gsrc];
            const float *sw = src.s[src_ok ? gsrc + i : gsrc];
#pragma unroll
            for (int j = 0; j < 2; j++)
                in.q[i][j] = (src_ok && (!kTail || b0 + 4 * j + g < nblk)) ? ld_stream_v4(qw + e0 + 512 * j)
                                                                           : make_uint4(0, 0, 0, 0);
            in.sc[i] = (src_ok && lane_ok) ? ld_stream_u32(sw + b0 + lane) : 0u;
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        load_group<kTail>(in, 0, c);
    }
    // per-lane async copies (run_chunks_lane_async), for exactly W sources
    using Slots = LaneSlots<2 * W, W>;
    __device__ __forceinline__ void issue(const Slots &sl, int64_t c) const
    {
        static_assert(!kMore, "the async driver serves launches of exactly W sources");
        issue_wide_sources<W>(sl, src, c, lane);
    }
    __device__ __forceinline__ void take(In &in, const Slots &sl) const { take_wide_sources<W>(in, sl, lane); }
    template <bool kFirst>
    __device__ __forceinline__ void add_group(const In &in, int gsrc, float2 (&acc)[2][2][4]) const
    {
        const int g = lane >> 3;
#pragma unroll
        for (int i = 0; i < W; i++) {
            if (kMore && gsrc + i >= nsrc) break;
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const float2 sc = splat(__uint_as_float(__shfl_sync(kFull, in.sc[i], 4 * j + g)));
                float2 v[2][4];
                i8x8_to_f32(make_uint2(in.q[i][j].x, in.q[i][j].y), v[0]);
                i8x8_to_f32(make_uint2(in.q[i][j].z, in.q[i][j].w), v[1]);
#pragma unroll
                for (int h = 0; h < 2; h++)
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float2 d = mul2_unfused(v[h][e], sc);
                        acc[j][h][e] = (kFirst && i == 0) ? d : add2(acc[j][h][e], d);
                    }
            }
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 acc[2][2][4];  // [segment][half of the lane's 16 values][pair]
        add_group<true>(in, 0, acc);
        if constexpr (kMore) {
            for (int gsrc = W; gsrc < nsrc; gsrc += W) {
                In more;
                load_group<kTail>(more, gsrc, c);
                add_group<false>(more, gsrc, acc);
            }
        }
        requant_wide<kTail, kOut, kV8>(acc, c * 1024 + lane * 16, c * 8, nblk, lane, q, s, out);
    }
};

// Ring hop: v = fl(fl(q_in * s_in) + x_local) for the lane's 16 values, requantized.
template <bool kOut, bool kV8>
struct HopWideI8 {
    const int8_t *__restrict__ q_in;
    const float *__restrict__ s_in;
    const uint16_t *__restrict__ x;
    int8_t *__restrict__ q;
    float *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint4 q[2];
        uint4 x[2][2];
        float sc[2];
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * 1024 + lane * 16, b0 = c * 8 + (lane >> 3);
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const bool ok = !kTail || b0 + 4 * j < nblk;
            in.q[j] = ok ? ld_stream_v4(q_in + e0 + 512 * j) : make_uint4(0, 0, 0, 0);
            load_bf16x16<kV8>(x + e0 + 512 * j, ok, in.x[j]);
            in.sc[j] = ok ? __uint_as_float(ld_stream_u32(s_in + b0 + 4 * j)) : 0.0f;
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 v[2][2][4];
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const float2 sc = splat(in.sc[j]);
            float2 d[2][4], xl[2][4];
            i8x8_to_f32(make_uint2(in.q[j].x, in.q[j].y), d[0]);
            i8x8_to_f32(make_uint2(in.q[j].z, in.q[j].w), d[1]);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                bf16x8_to_f32(in.x[j][h], xl[h]);
#pragma unroll
                for (int e = 0; e < 4; e++) v[j][h][e] = add2(mul2_unfused(d[h][e], sc), xl[h][e]);
            }
        }
        requant_wide<kTail, kOut, kV8>(v, c * 1024 + lane * 16, c * 8, nblk, lane, q, s, out);
    }
};

// 256-bit accesses for the BF16 side when its pointer is 32-byte aligned.
#ifndef BQ_WIDE_V8
#define BQ_WIDE_V8 1
#endif
#ifndef BQ_HOP_WIDE
#define BQ_HOP_WIDE 1
#endif
// Wide ring hop: 284.9 us per 469.8M-value launch at 4 CTAs per SM (64 registers)
// against 300 us at 3 (76 registers), and 298.9 us for the staged 8-value kernel.
#ifndef BQ_HOP_MIN_CTAS
#define BQ_HOP_MIN_CTAS 4
#endif
// Threads per CTA of the wide hop (registers per thread at the BQ_HOP_MIN_CTAS budget).
// One CTA per SM, all warps of the same age: 287.8 against 291.4 us with 256 threads.
#ifndef BQ_HOP_WIDE_THREADS
#define BQ_HOP_WIDE_THREADS 1024
#endif
constexpr int kHopWideThreads = BQ_HOP_WIDE_THREADS;

template <bool kOut, bool kV8>
__global__ void __launch_bounds__(kHopWideThreads, BQ_HOP_MIN_CTAS * kThreads / kHopWideThreads)
ring_hop_i8_wide_kernel(const int8_t *__restrict__ q_in, const float *__restrict__ s_in,
                        const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s,
                        uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q_in, s_in, nblk, false);
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const HopWideI8<kOut, kV8> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false, kHopWideThreads>(op, nblk, 8);
}

#ifndef BQ_ACCUM_WIDE
#define BQ_ACCUM_WIDE 1
#endif
#ifndef BQ_QUANT_WIDE
#define BQ_QUANT_WIDE 1
#endif

// The accumulate of exactly W sources without the owner output, with each warp's next
// chunk in flight through per-lane async copies while it computes the current one.
// On GB300, per 469.8M-value launch: 387 against 414 us with four sources, 288 against
// 298 with two, 231 against 243 with one; at 2 CTAs per SM (121 registers for four
// sources, two 36 KB stages per CTA). Four sources at 3 CTAs per SM took 394 us, with
// 3 stages 395 us, one CTA of 4 stages 500 us. With the owner output the same loads
// were 5% slower than direct ones (604 against 574 us, in 256- and in 512-thread CTAs),
// so that form keeps the direct path.
#ifndef BQ_ACCUM_ASYNC
#define BQ_ACCUM_ASYNC 1
#endif
// Threads per CTA, one CTA per SM at 512: the warp schedulers favour a CTA's warps by
// the CTA's age, so of two 256-thread CTAs on an SM the older finishes about 14% of the
// launch earlier and the other runs alone until the end. With all of the SM's warps in
// one CTA they keep pace: 379 against 385 us for the four-source launch.
#ifndef BQ_ACCUM_ASYNC_THREADS
#define BQ_ACCUM_ASYNC_THREADS 512
#endif
constexpr int kAccumAsyncThreads = BQ_ACCUM_ASYNC_THREADS;
constexpr int kAccumAsyncStages = 2;

template <int W>
__global__ void __launch_bounds__(kAccumAsyncThreads, kAccumAsyncThreads >= 512 ? 1 : 512 / kAccumAsyncThreads)
accum_i8_async_kernel(const __grid_constant__ SourceList src, int nsrc, int64_t nblk, int8_t *__restrict__ q,
                      float *__restrict__ s)
{
    extern __shared__ __align__(16) unsigned char stages[];
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_ready();
    using Op = AccumWideI8<W, false, false, false>;
    const Op op{src, nsrc, q, s, nullptr, nblk, (int)(threadIdx.x & 31)};
    run_chunks_lane_async<kAccumAsyncStages, kAccumAsyncThreads>(
        op, nblk, 8, stages + (threadIdx.x >> 5) * kAccumAsyncStages * Op::Slots::kBytes);
}

// Threads per CTA of the wide accumulate with direct loads (the owner-output form and
// launches of more than four sources); registers per thread at the BQ_ACCUM_MIN_CTAS
// budget of 256-thread CTAs whatever the size. One 768-thread CTA per SM measured within
// noise of three 256-thread CTAs for the four-source owner-output launch (576.2 against
// 579.9 us, medians; the minima the other way round).
#ifndef BQ_ACCUM_WIDE_THREADS
#define BQ_ACCUM_WIDE_THREADS 256
#endif
constexpr int kAccumWideThreads = BQ_ACCUM_WIDE_THREADS;

template <int W, bool kOut, bool kMore, bool kV8>
__global__ void __launch_bounds__(kAccumWideThreads, BQ_ACCUM_MIN_CTAS * kThreads / kAccumWideThreads)
accum_i8_wide_kernel(const __grid_constant__ SourceList src, int nsrc, int64_t nblk, int8_t *__restrict__ q,
                     float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const AccumWideI8<W, kOut, kMore, kV8> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false, kAccumWideThreads>(op, nblk, 8);
}

// Threads per CTA of the wide quantize; its registers per thread stay at the 4-CTA
// budget (64) whatever the CTA size. One CTA per SM (1024 threads) keeps all of an SM's
// warps at the same age for the warp schedulers: 219.2 against 222.9 us per 469.8M-value
// launch with 256-thread CTAs (221.3 with 512).
#ifndef BQ_QUANT_WIDE_THREADS
#define BQ_QUANT_WIDE_THREADS 1024
#endif
constexpr int kQuantWideThreads = BQ_QUANT_WIDE_THREADS;

template <bool kV8>
__global__ void __launch_bounds__(kQuantWideThreads, BQ_QUANT_MIN_CTAS * kThreads / kQuantWideThreads)
quant_i8_wide_kernel(const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_begin();
    dbg_begin();
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_ready();
    const QuantWideI8<kV8> op{x, q, s, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false, kQuantWideThreads>(op, nblk, 8);
}

// ---------------------------------------------------------------- ring hop
template <int SEGS, bool kOut>
using HopI8 = HopOp<I8Codec, SEGS, kOut>;

template <int SEGS, bool kOut, int STAGES>
__global__ void __launch_bounds__(kThreads)
ring_hop_i8_staged_kernel(const int8_t *__restrict__ q_in, const float *__restrict__ s_in,
                          const uint16_t *__restrict__ x, int64_t nblk, int8_t *__restrict__ q,
                          float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q_in, s_in, nblk, false);
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    extern __shared__ __align__(128) unsigned char smem[];
    const HopI8<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS, smem + (threadIdx.x >> 5) * staged_warp_bytes<HopI8<SEGS, kOut>, STAGES>());
}

template <int SEGS, bool kOut>
__global__ void __launch_bounds__(kThreads)
ring_hop_i8_kernel(const int8_t *__restrict__ q_in, const float *__restrict__ s_in, const uint16_t *__restrict__ x,
                   int64_t nblk, int8_t *__restrict__ q, float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q_in, s_in, nblk, false);
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const HopI8<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

// ---------------------------------------------------------------- reduce + quantize
#ifndef BQ_SEGS_REDUCE_I8_ASYNC
#define BQ_SEGS_REDUCE_I8_ASYNC 2
#endif

template <int SEGS, int W, bool kOut>
__global__ void __launch_bounds__(kThreads)
reduce_quant_i8_kernel(const __grid_constant__ Bf16List src, int nsrc, int64_t nblk, int8_t *__restrict__ q,
                       float *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const ReduceQuantOp<I8Codec, SEGS, W, kOut> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

template <int W, bool kOut>
__global__ void __launch_bounds__(kReduceAsyncThreads, kReduceAsyncMinCtas)
reduce_quant_i8_async_kernel(const __grid_constant__ Bf16List src, int nsrc, int64_t nblk, int8_t *__restrict__ q,
                             float *__restrict__ s, uint16_t *__restrict__ out)
{
    extern __shared__ __align__(16) unsigned char stages[];
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    reduce_quant_async_body<I8Codec, BQ_SEGS_REDUCE_I8_ASYNC, W, kOut>(src, nsrc, nblk, q, s, out, stages);
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
#ifndef BQ_SEGS_REDUCE
#define BQ_SEGS_REDUCE 2
#endif
constexpr int kSegsQuant = BQ_SEGS_QUANT;
constexpr int kSegsDequant = BQ_SEGS_DEQUANT;
constexpr int kSegsAccum = BQ_SEGS_ACCUM;
constexpr int kSegsHop = BQ_SEGS_HOP;
constexpr int kSegsReduce = BQ_SEGS_REDUCE;

// Bulk-copy stages per warp (0: the kernel reads global memory directly). Measured on
// GB300: staging pays for the ring hop (payload, BF16 and scale streams) and costs for
// quantize and the W = 4 accumulate, whose shared memory would lower occupancy.
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

template <int W, bool kOut, bool kMore>
cudaError_t launch_accum_wide(const SourceList &src, int nsrc, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                              cudaStream_t st)
{
    if constexpr (!kOut && !kMore) {
        if (BQ_ACCUM_ASYNC) {
            auto kernel = accum_i8_async_kernel<W>;
            const size_t smem =
                (kAccumAsyncThreads / 32) * kAccumAsyncStages * AccumWideI8<W, false, false, false>::Slots::kBytes;
            int grid = 0;
            if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, 4), &grid, smem, kAccumAsyncThreads))
                return e;
            return launch_kernel_block(kernel, grid, kAccumAsyncThreads, smem, st, src, nsrc, nblk, q, s);
        }
    }
    auto kernel = accum_i8_wide_kernel<W, kOut, kMore, false>;
    if constexpr (kOut)
        if (BQ_WIDE_V8 && aligned32(out)) kernel = accum_i8_wide_kernel<W, kOut, kMore, true>;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, 4), &grid, 0, kAccumWideThreads)) return e;
    return launch_kernel_block(kernel, grid, kAccumWideThreads, 0, st, src, nsrc, nblk, q, s, out);
}

template <int W, bool kOut, bool kMore>
cudaError_t launch_accum_w(const SourceList &src, int nsrc, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                           cudaStream_t st)
{
    if constexpr (kStagesAccum > 0) {
        // Bulk copies need 16-byte aligned scale runs; scale pointers are only required
        // to be 4-byte aligned, so other alignments take the global-memory path.
        bool staged = true;
        for (int i = 0; i < W && i < nsrc; i++) staged = staged && aligned16(src.s[i]);
        if (staged)
            return launch_staged<AccumI8<kSegsAccum, W, kOut, kMore>, kStagesAccum>(
                accum_i8_staged_kernel<kSegsAccum, W, kOut, kMore, kStagesAccum>, chunks(nblk, kSegsAccum), st, src,
                nsrc, nblk, q, s, out);
    }
    auto kernel = accum_i8_kernel<kSegsAccum, W, kOut, kMore>;
    BQK_GRID(kernel, chunks(nblk, kSegsAccum));
    return launch_kernel(kernel, grid, st, src, nsrc, nblk, q, s, out);
}

}  // namespace

namespace {
template <int STAGES>
cudaError_t launch_quant_stages(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st)
{
    if constexpr (STAGES > 0)  // x is 16-byte aligned by contract
        return launch_staged<QuantI8<kSegsQuant>, STAGES>(quant_i8_staged_kernel<kSegsQuant, STAGES>,
                                                           chunks(nblk, kSegsQuant), st, x, nblk, q, s);
    BQK_GRID(quant_i8_kernel<kSegsQuant>, chunks(nblk, kSegsQuant));
    return launch_kernel(quant_i8_kernel<kSegsQuant>, grid, st, x, nblk, q, s);
}
}  // namespace

cudaError_t launch_quant_i8(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st)
{
    if (BQ_QUANT_WIDE) {
        auto kernel = BQ_WIDE_V8 && aligned32(x) ? quant_i8_wide_kernel<true> : quant_i8_wide_kernel<false>;
        int grid = 0;
        if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, 4), &grid, 0, kQuantWideThreads)) return e;
        return launch_kernel_block(kernel, grid, kQuantWideThreads, 0, st, x, nblk, q, s);
    }
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

// Debug build: the kernel lists only the first 256 bytes of a 1 KB caller buffer and
// then loads 16 bytes at byte 512, which the check declines (and counts) instead of
// performing. The load would stay inside the caller's buffer in any case.
__global__ void index_selftest_kernel(unsigned char *buf)
{
    dbg_begin();
    dbg_allow(buf, 256, true);
    dbg_ready();
    if (threadIdx.x == 0) {
        const uint4 v = ld_stream_v4(buf + 512);
        st_v4(buf, v);  // inside the listed range: performed (zeros from the declined load)
    }
}

cudaError_t launch_index_selftest(void *buf, cudaStream_t st)
{
    index_selftest_kernel<<<1, 32, 0, st>>>(static_cast<unsigned char *>(buf));
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(cudaStream_t st)
{
    wait_selftest_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

cudaError_t read_wait_counters_i8(unsigned long long (&v)[3]) { return read_wait_counters(v); }

cudaError_t launch_dequant_i8(const int8_t *q, const float *s, int64_t nblk, uint16_t *out, cudaStream_t st)
{
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)dequant_i8_kernel<kSegsDequant>, chunks(nblk, kSegsDequant), &grid, 0,
                                 kDequantI8Threads))
        return e;
    return launch_kernel_block(dequant_i8_kernel<kSegsDequant>, grid, kDequantI8Threads, 0, st, q, s, nblk, out);
}

// One source width is compiled per common case (1, 2, 3, 4 sources at once); more
// sources run in groups of four.
cudaError_t launch_accum_i8(const SourceList &src, int W, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                            cudaStream_t st)
{
    const bool o = out != nullptr;
    if (BQ_ACCUM_WIDE) {
        switch (W) {
        case 1: return o ? launch_accum_wide<1, true, false>(src, W, nblk, q, s, out, st)
                       : launch_accum_wide<1, false, false>(src, W, nblk, q, s, out, st);
        case 2: return o ? launch_accum_wide<2, true, false>(src, W, nblk, q, s, out, st)
                       : launch_accum_wide<2, false, false>(src, W, nblk, q, s, out, st);
        case 3: return o ? launch_accum_wide<3, true, false>(src, W, nblk, q, s, out, st)
                       : launch_accum_wide<3, false, false>(src, W, nblk, q, s, out, st);
        case 4: return o ? launch_accum_wide<4, true, false>(src, W, nblk, q, s, out, st)
                       : launch_accum_wide<4, false, false>(src, W, nblk, q, s, out, st);
        default: return o ? launch_accum_wide<4, true, true>(src, W, nblk, q, s, out, st)
                          : launch_accum_wide<4, false, true>(src, W, nblk, q, s, out, st);
        }
    }
    switch (W) {
    case 1: return o ? launch_accum_w<1, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_w<1, false, true>(src, W, nblk, q, s, out, st);
    case 2: return o ? launch_accum_w<2, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_w<2, false, true>(src, W, nblk, q, s, out, st);
    case 3: return o ? launch_accum_w<3, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_w<3, false, true>(src, W, nblk, q, s, out, st);
    case 4: return o ? launch_accum_w<4, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_w<4, false, false>(src, W, nblk, q, s, out, st);
    default: return o ? launch_accum_w<4, true, true>(src, W, nblk, q, s, out, st)
                      : launch_accum_w<4, false, true>(src, W, nblk, q, s, out, st);
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
            return launch_staged<HopI8<kSegsHop, kOut>, STAGES>(ring_hop_i8_staged_kernel<kSegsHop, kOut, STAGES>,
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
    if (BQ_HOP_WIDE) {
        const bool v8 = BQ_WIDE_V8 && aligned32(x) && (!out || aligned32(out));
        auto kernel = out ? (v8 ? ring_hop_i8_wide_kernel<true, true> : ring_hop_i8_wide_kernel<true, false>)
                          : (v8 ? ring_hop_i8_wide_kernel<false, true> : ring_hop_i8_wide_kernel<false, false>);
        int grid = 0;
        if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, 4), &grid, 0, kHopWideThreads)) return e;
        return launch_kernel_block(kernel, grid, kHopWideThreads, 0, st, q_in, s_in, x, nblk, q, s, out);
    }
    if (out) return launch_hop_stages<kStagesHop, true>(q_in, s_in, x, nblk, q, s, out, st);
    return launch_hop_stages<kStagesHop, false>(q_in, s_in, x, nblk, q, s, nullptr, st);
}

namespace {
template <int W, bool kOut>
cudaError_t launch_reduce_i8_w(const Bf16List &src, int nsrc, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                               cudaStream_t st)
{
    if (BQ_REDUCE_ASYNC && nsrc == W)
        return launch_reduce_async<I8Codec, BQ_SEGS_REDUCE_I8_ASYNC, W, kOut>(
            reduce_quant_i8_async_kernel<W, kOut>, nblk, st, src, nsrc, nblk, q, s, out);
    auto kernel = reduce_quant_i8_kernel<kSegsReduce, W, kOut>;
    BQK_GRID(kernel, chunks(nblk, kSegsReduce));
    return launch_kernel(kernel, grid, st, src, nsrc, nblk, q, s, out);
}
}  // namespace

// One source width per common case (1..4 at once); more sources in groups of four.
cudaError_t launch_reduce_quant_i8(const Bf16List &src, int W, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                                   cudaStream_t st)
{
    const bool o = out != nullptr;
    switch (W) {
    case 1: return o ? launch_reduce_i8_w<1, true>(src, W, nblk, q, s, out, st) : launch_reduce_i8_w<1, false>(src, W, nblk, q, s, out, st);
    case 2: return o ? launch_reduce_i8_w<2, true>(src, W, nblk, q, s, out, st) : launch_reduce_i8_w<2, false>(src, W, nblk, q, s, out, st);
    case 3: return o ? launch_reduce_i8_w<3, true>(src, W, nblk, q, s, out, st) : launch_reduce_i8_w<3, false>(src, W, nblk, q, s, out, st);
    default: return o ? launch_reduce_i8_w<4, true>(src, W, nblk, q, s, out, st) : launch_reduce_i8_w<4, false>(src, W, nblk, q, s, out, st);
    }
}

}  // namespace bqk
