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
    if ((lane & 3) == 0 && (lane >> 2) < 2 * SEGS && (!kTail || b0 + (lane >> 2) < nblk)) s[b0 + (lane >> 2)] = word;
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
    const AccumMx<SEGS, W, kOut, kMore> op{src, nsrc, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_chunks<false>(op, nblk, 2 * SEGS);
}

template <int SEGS, int W, bool kOut, bool kMore, int STAGES>
__global__ void __launch_bounds__(kThreads, BQ_ACCUM_MX_MIN_CTAS)
accum_mx_staged_kernel(const __grid_constant__ MxSourceList src, int nsrc, int64_t nblk, uint8_t *__restrict__ q,
                       uint32_t *__restrict__ s, uint16_t *__restrict__ out)
{
    pdl_begin();
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
    extern __shared__ __align__(128) unsigned char smem[];
    const HopMx<SEGS, kOut> op{q_in, s_in, x, q, s, out, nblk, (int)(threadIdx.x & 31)};
    run_staged<STAGES>(op, nblk, 2 * SEGS, smem + (threadIdx.x >> 5) * staged_warp_bytes<HopMx<SEGS, kOut>, STAGES>());
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
    if (out) return launch_hop_mx_stages<kStagesHopMx, true>(q_in, s_in, x, nblk, q, s, out, st);
    return launch_hop_mx_stages<kStagesHopMx, false>(q_in, s_in, x, nblk, q, s, nullptr, st);
}

cudaError_t take_wait_timeouts_mx(unsigned long long *count)
{
    unsigned long long zero = 0;
    if (cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof zero)) return e;
    return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof zero);
}

}  // namespace bqk
