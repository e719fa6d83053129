// MXFP8 wire reductions: the all-to-all accumulate and the ring hop of the mx_a2a and
// mx_ring modes ("feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary: the MXFP8
// codec runs on the same all-gather, ring and all-to-all topologies as block INT8, and
// every mode materializes the owner shard from the payload it forwards).
//
// A flat MX wire of n values is E4M3 codes [n] followed by E8M0 bytes [n/32]; the four
// bytes of a 128-value block form one 32-bit scale word, so the chunk drivers and the
// reductions of bq_chunks.cuh serve it unchanged. Arithmetic (same rules as the MX
// quantizer): a wire element is decode(code) * 2^(e - 127), exact in binary32; sums
// are binary32 in source order; requantization takes the E8M0 byte of each group's
// binary32 amax and scales each value by 2^(127 - e) before the E4M3 conversion.
#include "bq_chunks.cuh"

namespace bqk {
namespace {

// Requantize SEGS segments of binary32 values (v[j] = lane's 8 values of segment j)
// as MX groups. After the group amaxes are reduced (a quad of lanes per group), lane
// L holds the amax of the chunk's group L (block L/4, group L%4 of that block) and
// computes its E8M0 byte and multipliers once; each lane then fetches its own group's
// multiplier per segment, and lanes 4b store block b's four scale bytes as one word.
template <int SEGS, bool kTail, bool kOut, class Vals>
__device__ __forceinline__ void requant_mx_chunk(const Vals &vals, int64_t e0, int64_t b0, int64_t nblk, int lane,
                                                 uint8_t *__restrict__ q, uint32_t *__restrict__ s,
                                                 uint16_t *__restrict__ out)
{
    static_assert(8 * SEGS <= 32, "a chunk's groups fit one per lane");
    const int half = lane >> 4;
    float gmax = 0.0f;
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        float2 v[4];
        vals.seg(j, v);
        float m = amax8(v);
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
        const float g = __shfl_sync(kFull, m, (lane & 7) << 2);
        if ((lane >> 3) == j) gmax = g;
    }
    const uint32_t e = mx_scale_byte(gmax);
    const float p = exp2i(127 - static_cast<int>(e));
    const float pinv = exp2i(static_cast<int>(e) - 127);
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        const int src = 8 * j + (lane >> 2);
        const float2 pj = splat(__shfl_sync(kFull, p, src));
        const float pinv_j = kOut ? __shfl_sync(kFull, pinv, src) : 0.0f;
        float2 v[4], y[4];
        vals.seg(j, v);
#pragma unroll
        for (int i = 0; i < 4; i++) y[i] = mul2(v[i], pj);  // exact: a power-of-two scaling
        const uint2 codes = f32x8_to_e4m3x8(y);
        if (!kTail || b0 + 2 * j + half < nblk) {
            st_v2(q + e0 + 256 * j, codes);
            if (kOut) {
                float2 d[4];
                e4m3x8_to_f32(codes, pinv_j, d);
                st_v4(out + e0 + 256 * j, f32x8_to_bf16x8(d));
            }
        }
    }
    uint32_t word = e << (8 * (lane & 3));
    word |= __shfl_xor_sync(kFull, word, 1);
    word |= __shfl_xor_sync(kFull, word, 2);
    if ((lane & 3) == 0 && (lane >> 2) < 2 * SEGS && (!kTail || b0 + (lane >> 2) < nblk) &&
        dbg_ok(s + b0 + (lane >> 2), 4, true))
        s[b0 + (lane >> 2)] = word;
}

// MXFP8 codec policy for the shared reductions.
struct MxCodec {
    using Q = uint8_t;
    using S = uint32_t;
    // A lane's 8 values lie in group (lane % 16) / 4 of its block: byte of the word.
    static __device__ __forceinline__ void decode8(uint2 q, uint32_t word, int lane, float2 (&d)[4])
    {
        const uint32_t e = (word >> (8 * ((lane & 15) >> 2))) & 0xffu;
        const float p = e == 255u ? __uint_as_float(0x7fc00000u) : exp2i(static_cast<int>(e) - 127);
        e4m3x8_to_f32(q, p, d);
    }
    template <int SEGS, bool kTail, bool kOut, class Vals>
    static __device__ __forceinline__ void requant(const Vals &vals, int64_t e0, int64_t b0, int64_t nblk,
                                                   int lane, uint8_t *q, uint32_t *s, uint16_t *out)
    {
        requant_mx_chunk<SEGS, kTail, kOut>(vals, e0, b0, nblk, lane, q, s, out);
    }
};

// ---------------------------------------------------------------- wide lanes
// The layout of the block-INT8 wide kernels: a lane takes 16 consecutive values, so an
// MX group spans 2 lanes and a 128-value block 8; a warp chunk is two 512-value
// segments, 8 blocks, 32 groups: one per lane for the E8M0 computation. Same
// arithmetic, same order.

// Decode multiplier 2^(e-127) of the lane's group, from its block's scale word.
__device__ __forceinline__ float mx_wide_mult(uint32_t word, int lane)
{
    const uint32_t e = (word >> (8 * ((lane & 7) >> 1))) & 0xffu;
    return e == 255u ? __uint_as_float(0x7fc00000u) : exp2i(static_cast<int>(e) - 127);
}

// v[j][h]: the lane's values 8h..8h+7 of segment j (elements e0 + 512 j + 8 h ...), in
// block b0 + 4 j + (lane >> 3), group ((lane & 7) >> 1) of that block. kV8: out is
// 32-byte aligned and takes one 256-bit store per lane.
template <bool kTail, bool kOut, bool kV8>
__device__ __forceinline__ void requant_mx_wide(const float2 (&v)[2][2][4], int64_t e0, int64_t b0, int64_t nblk,
                                                int lane, uint8_t *__restrict__ q, uint32_t *__restrict__ s,
                                                uint16_t *__restrict__ out)
{
    const int g = lane >> 3;
    float gmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        float m = amax16(v[j][0], v[j][1]);
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));  // the group's two lanes
        // lane L takes chunk group L: segment L / 16, block (L / 4) % 4 of it, group L % 4
        const float gm = __shfl_sync(kFull, m, 8 * ((lane >> 2) & 3) + 2 * (lane & 3));
        if ((lane >> 4) == j) gmax = gm;
    }
    const uint32_t e = mx_scale_byte(gmax);
    const float p = exp2i(127 - static_cast<int>(e));
    const float pinv = exp2i(static_cast<int>(e) - 127);
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int src = 16 * j + 4 * g + ((lane & 7) >> 1);
        const float2 pj = splat(__shfl_sync(kFull, p, src));
        const float pinv_j = kOut ? __shfl_sync(kFull, pinv, src) : 0.0f;
        float2 y0[4], y1[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {  // exact: a power-of-two scaling
            y0[i] = mul2(v[j][0][i], pj);
            y1[i] = mul2(v[j][1][i], pj);
        }
        const uint2 c0 = f32x8_to_e4m3x8(y0), c1 = f32x8_to_e4m3x8(y1);
        if (!kTail || b0 + 4 * j + g < nblk) {
            st_v4(q + e0 + 512 * j, make_uint4(c0.x, c0.y, c1.x, c1.y));
            if (kOut) {
                float2 d0[4], d1[4];
                e4m3x8_to_f32(c0, pinv_j, d0);
                e4m3x8_to_f32(c1, pinv_j, d1);
                const uint4 o0 = f32x8_to_bf16x8(d0), o1 = f32x8_to_bf16x8(d1);
                if (kV8) {
                    st_v8(out + e0 + 512 * j, o0, o1);
                } else {
                    st_v4(out + e0 + 512 * j, o0);
                    st_v4(out + e0 + 512 * j + 8, o1);
                }
            }
        }
    }
    uint32_t word = e << (8 * (lane & 3));
    word |= __shfl_xor_sync(kFull, word, 1);
    word |= __shfl_xor_sync(kFull, word, 2);
    if ((lane & 3) == 0 && (!kTail || b0 + (lane >> 2) < nblk) && dbg_ok(s + b0 + (lane >> 2), 4, true))
        s[b0 + (lane >> 2)] = word;
}

// Accumulate of W sources at a time (kMore: further groups of W follow the first).
// Without kMore the launch has exactly W sources, so the source loop carries no
// source-count checks (2% of the four-source launch's time on GB300).
template <int W, bool kOut, bool kMore, bool kV8>
struct AccumWideMx {
    const MxSourceList &src;  // the kernel's __grid_constant__ parameter, read in place
    int nsrc;
    uint8_t *__restrict__ q;
    uint32_t *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint4 q[W][2];
        uint32_t sc[W];  // lanes 0..7: the scale words of the chunk's blocks 0..7
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
            const uint8_t *qw = src.q[src_ok ? gsrc + i : gsrc];
            const uint32_t *sw = src.s[src_ok ? gsrc + i : gsrc];
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
        // segment by segment, each segment's sources in source order: the same sums, and
        // a segment's payload registers are free once it is summed (75 registers instead
        // of 80 with 8 B of spills)
#pragma unroll
        for (int j = 0; j < 2; j++) {
#pragma unroll
            for (int i = 0; i < W; i++) {
                if (kMore && gsrc + i >= nsrc) break;
                const float mult = mx_wide_mult(__shfl_sync(kFull, in.sc[i], 4 * j + g), lane);
                float2 d[2][4];
                e4m3x8_to_f32(make_uint2(in.q[i][j].x, in.q[i][j].y), mult, d[0]);
                e4m3x8_to_f32(make_uint2(in.q[i][j].z, in.q[i][j].w), mult, d[1]);
#pragma unroll
                for (int h = 0; h < 2; h++)
#pragma unroll
                    for (int e = 0; e < 4; e++) acc[j][h][e] = (kFirst && i == 0) ? d[h][e] : add2(acc[j][h][e], d[h][e]);
            }
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 acc[2][2][4];
        add_group<true>(in, 0, acc);
        if constexpr (kMore) {
            for (int gsrc = W; gsrc < nsrc; gsrc += W) {
                In more;
                load_group<kTail>(more, gsrc, c);
                add_group<false>(more, gsrc, acc);
            }
        }
        requant_mx_wide<kTail, kOut, kV8>(acc, c * 1024 + lane * 16, c * 8, nblk, lane, q, s, out);
    }
};

template <bool kOut, bool kV8>
struct HopWideMx {
    const uint8_t *__restrict__ q_in;
    const uint32_t *__restrict__ s_in;
    const uint16_t *__restrict__ x;
    uint8_t *__restrict__ q;
    uint32_t *__restrict__ s;
    uint16_t *__restrict__ out;
    int64_t nblk;
    int lane;
    struct In {
        uint4 q[2];
        uint4 x[2][2];
        uint32_t sc[2];  // the scale word of the lane's block, per segment
    };
    template <bool kTail>
    __device__ __forceinline__ void load(In &in, int64_t c) const
    {
        const int64_t e0 = c * 1024 + lane * 16, b0 = c * 8 + (lane >> 3);
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const bool ok = !kTail || b0 + 4 * j < nblk;
            in.q[j] = ok ? ld_stream_v4(q_in + e0 + 512 * j) : make_uint4(0, 0, 0, 0);
            if (!ok) {
                in.x[j][0] = in.x[j][1] = make_uint4(0, 0, 0, 0);
            } else if (kV8) {
                ld_stream_v8(x + e0 + 512 * j, in.x[j][0], in.x[j][1]);
            } else {
                in.x[j][0] = ld_stream_v4(x + e0 + 512 * j);
                in.x[j][1] = ld_stream_v4(x + e0 + 512 * j + 8);
            }
            in.sc[j] = ok ? ld_stream_u32(s_in + b0 + 4 * j) : 0u;
        }
    }
    template <bool kTail>
    __device__ __forceinline__ void compute(const In &in, int64_t c) const
    {
        float2 v[2][2][4];
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const float mult = mx_wide_mult(in.sc[j], lane);
            float2 d[2][4], xl[2][4];
            e4m3x8_to_f32(make_uint2(in.q[j].x, in.q[j].y), mult, d[0]);
            e4m3x8_to_f32(make_uint2(in.q[j].z, in.q[j].w), mult, d[1]);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                bf16x8_to_f32(in.x[j][h], xl[h]);
#pragma unroll
                for (int e = 0; e < 4; e++) v[j][h][e] = add2(d[h][e], xl[h][e]);
            }
        }
        requant_mx_wide<kTail, kOut, kV8>(v, c * 1024 + lane * 16, c * 8, nblk, lane, q, s, out);
    }
};

#ifndef BQ_MX_WIDE
#define BQ_MX_WIDE 1
#endif
#ifndef BQ_HOP_MX_MIN_CTAS
#define BQ_HOP_MX_MIN_CTAS 4
#endif

template <int SEGS, int W, bool kOut, bool kMore>
using AccumMx = AccumOp<MxCodec, SEGS, W, kOut, kMore>;
template <int SEGS, bool kOut>
using HopMx = HopOp<MxCodec, SEGS, kOut>;

#ifndef BQ_ACCUM_MX_MIN_CTAS
#define BQ_ACCUM_MX_MIN_CTAS 3
#endif

template <int SEGS, int W, bool kOut, bool kMore>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MX_MIN_CTAS)
accum_mx_kernel(const __grid_constant__ MxSourceList src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const AccumMx<SEGS, W, kOut, kMore> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

template <int SEGS, int W, bool kOut, bool kMore, int STAGES>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MX_MIN_CTAS)
accum_mx_staged_kernel(const __grid_constant__ MxSourceList src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                       uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    extern __shared__ __align__(128) unsigned char smem[];
    const AccumMx<SEGS, W, kOut, kMore> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS,
                       smem + (threadIdx.x >> 5) * staged_warp_bytes<AccumMx<SEGS, W, kOut, kMore>, STAGES>());
}

template <int SEGS, bool kOut>
__global__ void __launch_bounds__(kThreads)
ring_hop_mx_kernel(const uint8_t *__restrict__ q_in, const uint32_t *__restrict__ s_in, const uint16_t *__restrict__ x,
                   int64_t nblk, uint8_t *__restrict__ q, uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q_in, s_in, nblk, false);
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const HopMx<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

template <int SEGS, bool kOut, int STAGES>
__global__ void __launch_bounds__(kThreads)
ring_hop_mx_staged_kernel(const uint8_t *__restrict__ q_in, const uint32_t *__restrict__ s_in,
                          const uint16_t *__restrict__ x, int64_t nblk, uint8_t *__restrict__ q,
                          uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q_in, s_in, nblk, false);
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    extern __shared__ __align__(128) unsigned char smem[];
    const HopMx<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS, smem + (threadIdx.x >> 5) * staged_warp_bytes<HopMx<SEGS, kOut>, STAGES>());
}

// Threads per CTA of the wide MX accumulate with direct loads (the owner-output form and
// launches of more than four sources); registers at the 256-thread budget. One 768-thread
// CTA per SM measured within noise of three 256-thread CTAs (576.3 against 582.2 us).
#ifndef BQ_ACCUM_MX_WIDE_THREADS
#define BQ_ACCUM_MX_WIDE_THREADS 256
#endif
constexpr int kAccumMxWideThreads = BQ_ACCUM_MX_WIDE_THREADS;

template <int W, bool kOut, bool kMore, bool kV8>
__global__ void __launch_bounds__(kAccumMxWideThreads, BQ_ACCUM_MX_MIN_CTAS * kThreads / kAccumMxWideThreads)
accum_mx_wide_kernel(const __grid_constant__ MxSourceList src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                     uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const AccumWideMx<W, kOut, kMore, kV8> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false, kAccumMxWideThreads>(op, nblk, 8);
}

// The accumulate of exactly W sources without the owner output, with each warp's next
// chunk in flight through per-lane async copies while it computes the current one.
// On GB300, per 469.8M-value launch at 2 CTAs per SM: 369 against 396 us with four
// sources, 233 against 265 with two.
#ifndef BQ_ACCUM_MX_ASYNC
#define BQ_ACCUM_MX_ASYNC 1
#endif
// Threads per CTA (one CTA per SM at 512, so that all of an SM's warps have the same
// age for the warp schedulers): 363 against 368 us for the four-source launch.
#ifndef BQ_ACCUM_MX_ASYNC_THREADS
#define BQ_ACCUM_MX_ASYNC_THREADS 512
#endif
constexpr int kAccumMxAsyncThreads = BQ_ACCUM_MX_ASYNC_THREADS;
constexpr int kAccumMxAsyncStages = 2;

template <int W>
__global__ void __launch_bounds__(kAccumMxAsyncThreads, kAccumMxAsyncThreads >= 512 ? 1 : 512 / kAccumMxAsyncThreads)
accum_mx_async_kernel(const __grid_constant__ MxSourceList src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                      uint32_t *__restrict__ s)
{
    extern __shared__ __align__(16) unsigned char stages[];
    pdl_begin();
    dbg_begin();
    dbg_sources(src, nsrc, nblk);
    dbg_wire(q, s, nblk, true);
    dbg_ready();
    using Op = AccumWideMx<W, false, false, false>;
    const Op op{src, nsrc, q, s, nullptr, nblk, (int)(threadIdx.x & 31)};
    run_chunks_lane_async<kAccumMxAsyncStages, kAccumMxAsyncThreads>(
        op, nblk, 8, stages + (threadIdx.x >> 5) * kAccumMxAsyncStages * Op::Slots::kBytes);
}

template <bool kOut, bool kV8>
__global__ void __launch_bounds__(kThreads, BQ_HOP_MX_MIN_CTAS)
ring_hop_mx_wide_kernel(const uint8_t *__restrict__ q_in, const uint32_t *__restrict__ s_in,
                        const uint16_t *__restrict__ x, int64_t nblk, uint8_t *__restrict__ q,
                        uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
    dbg_begin();
    dbg_wire(q_in, s_in, nblk, false);
    dbg_bf16(x, nblk, false);
    dbg_wire(q, s, nblk, true);
    dbg_bf16(out, nblk, true);
    dbg_ready();
    const HopWideMx<kOut, kV8> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 8);
}


// Segments per warp chunk and bulk-copy stages per warp (0: direct global loads).
#ifndef BQ_SEGS_ACCUM_MX
#define BQ_SEGS_ACCUM_MX 4
#endif
#ifndef BQ_SEGS_HOP_MX
#define BQ_SEGS_HOP_MX 4
#endif
#ifndef BQ_STAGES_ACCUM_MX
#define BQ_STAGES_ACCUM_MX 0
#endif
#ifndef BQ_STAGES_HOP_MX
#define BQ_STAGES_HOP_MX 3
#endif
constexpr int kSegsAccumMx = BQ_SEGS_ACCUM_MX;
constexpr int kSegsHopMx = BQ_SEGS_HOP_MX;
constexpr int kStagesAccumMx = BQ_STAGES_ACCUM_MX;
constexpr int kStagesHopMx = BQ_STAGES_HOP_MX;

template <int W, bool kMore>
cudaError_t launch_accum_mx_wide(const MxSourceList &src, int nsrc, int64_t nblk, uint8_t *q, uint32_t *s,
                                 uint16_t *out, bool o, bool v8, cudaStream_t st)
{
    if constexpr (!kMore) {
        if (BQ_ACCUM_MX_ASYNC && !o) {
            auto kernel = accum_mx_async_kernel<W>;
            const size_t smem =
                (kAccumMxAsyncThreads / 32) * kAccumMxAsyncStages * AccumWideMx<W, false, false, false>::Slots::kBytes;
            int grid = 0;
            if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, 4), &grid, smem, kAccumMxAsyncThreads))
                return e;
            return launch_kernel_block(kernel, grid, kAccumMxAsyncThreads, smem, st, src, nsrc, nblk, q, s);
        }
    }
    auto kernel = o ? (v8 ? accum_mx_wide_kernel<W, true, kMore, true> : accum_mx_wide_kernel<W, true, kMore, false>)
                    : accum_mx_wide_kernel<W, false, kMore, false>;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, chunks(nblk, 4), &grid, 0, kAccumMxWideThreads)) return e;
    return launch_kernel_block(kernel, grid, kAccumMxWideThreads, 0, st, src, nsrc, nblk, q, s, out);
}

template <int W, bool kOut, bool kMore>
cudaError_t launch_accum_mx_w(const MxSourceList &src, int nsrc, int64_t nblk, uint8_t *q, uint32_t *s,
                              uint16_t *out, cudaStream_t st)
{
    if constexpr (kStagesAccumMx > 0) {
        // bulk copies need 16-byte aligned scale runs; scale pointers need only 4
        bool staged = true;
        for (int i = 0; i < W && i < nsrc; i++) staged = staged && aligned16(src.s[i]);
        if (staged)
            return launch_staged<AccumMx<kSegsAccumMx, W, kOut, kMore>, kStagesAccumMx>(
                accum_mx_staged_kernel<kSegsAccumMx, W, kOut, kMore, kStagesAccumMx>, chunks(nblk, kSegsAccumMx), st,
                src, nsrc, nblk, q, s, out);
    }
    auto kernel = accum_mx_kernel<kSegsAccumMx, W, kOut, kMore>;
    BQK_GRID(kernel, chunks(nblk, kSegsAccumMx));
    return launch_kernel(kernel, grid, st, src, nsrc, nblk, q, s, out);
}

template <int STAGES, bool kOut>
cudaError_t launch_hop_mx_stages(const uint8_t *q_in, const uint32_t *s_in, const uint16_t *x, int64_t nblk,
                                 uint8_t *q, uint32_t *s, uint16_t *out, cudaStream_t st)
{
    if constexpr (STAGES > 0) {
        if (aligned16(s_in))
            return launch_staged<HopMx<kSegsHopMx, kOut>, STAGES>(ring_hop_mx_staged_kernel<kSegsHopMx, kOut, STAGES>,
                                                                  chunks(nblk, kSegsHopMx), st, q_in, s_in, x, nblk, q,
                                                                  s, out);
    }
    BQK_GRID((ring_hop_mx_kernel<kSegsHopMx, kOut>), chunks(nblk, kSegsHopMx));
    return launch_kernel(ring_hop_mx_kernel<kSegsHopMx, kOut>, grid, st, q_in, s_in, x, nblk, q, s, out);
}

}  // namespace

// One source width is compiled per common case (1, 2, 3, 4 sources at once); more
// sources run in groups of four.
cudaError_t launch_accum_mx(const MxSourceList &src, int W, int64_t nblk, uint8_t *q, uint32_t *s, uint16_t *out,
                            cudaStream_t st)
{
    if (BQ_MX_WIDE) {
        const bool o = out != nullptr, v8 = o && aligned32(out);
        switch (W) {
        case 1: return launch_accum_mx_wide<1, false>(src, W, nblk, q, s, out, o, v8, st);
        case 2: return launch_accum_mx_wide<2, false>(src, W, nblk, q, s, out, o, v8, st);
        case 3: return launch_accum_mx_wide<3, false>(src, W, nblk, q, s, out, o, v8, st);
        case 4: return launch_accum_mx_wide<4, false>(src, W, nblk, q, s, out, o, v8, st);
        default: return launch_accum_mx_wide<4, true>(src, W, nblk, q, s, out, o, v8, st);
        }
    }
    const bool o = out != nullptr;
    switch (W) {
    case 1: return o ? launch_accum_mx_w<1, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_mx_w<1, false, true>(src, W, nblk, q, s, out, st);
    case 2: return o ? launch_accum_mx_w<2, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_mx_w<2, false, true>(src, W, nblk, q, s, out, st);
    case 3: return o ? launch_accum_mx_w<3, true, true>(src, W, nblk, q, s, out, st)
                   : launch_accum_mx_w<3, false, true>(src, W, nblk, q, s, out, st);
    default: return o ? launch_accum_mx_w<4, true, true>(src, W, nblk, q, s, out, st)
                      : launch_accum_mx_w<4, false, true>(src, W, nblk, q, s, out, st);
    }
}

cudaError_t launch_ring_hop_mx(const uint8_t *q_in, const uint32_t *s_in, const uint16_t *x, int64_t nblk, uint8_t *q,
                               uint32_t *s, uint16_t *out, cudaStream_t st)
{
    if (BQ_MX_WIDE) {
        const bool v8 = aligned32(x) && (!out || aligned32(out));
        auto kernel = out ? (v8 ? ring_hop_mx_wide_kernel<true, true> : ring_hop_mx_wide_kernel<true, false>)
                          : (v8 ? ring_hop_mx_wide_kernel<false, true> : ring_hop_mx_wide_kernel<false, false>);
        BQK_GRID(kernel, chunks(nblk, 4));
        return launch_kernel(kernel, grid, st, q_in, s_in, x, nblk, q, s, out);
    }
    if (out) return launch_hop_mx_stages<kStagesHopMx, true>(q_in, s_in, x, nblk, q, s, out, st);
    return launch_hop_mx_stages<kStagesHopMx, false>(q_in, s_in, x, nblk, q, s, nullptr, st);
}

cudaError_t read_wait_counters_mx_wire(unsigned long long (&v)[3]) { return read_wait_counters(v); }

}  // namespace bqk
