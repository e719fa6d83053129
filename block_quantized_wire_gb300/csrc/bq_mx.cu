// MXFP8 codec kernels: quantize (2-D, strided, covers staged slices) and materialize.
//
// Format from "feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary (E4M3 values,
// one E8M0 scale per 32 values) and the review comment on mxfp8_scale_byte (zero
// group -> 127, else E8M0 of amax/448 rounded toward +inf, saturating). Slices follow
// "[II] Support staged MXFP8 linear inputs", Behavior and Compatibility: a slice of
// 128-column-aligned width written at a 128-column-aligned offset of a wider buffer;
// the same page's Behavior accepts BF16 or FP16 slices (FP16 widens exactly to binary32
// and the rules are unchanged).
//
// A "block" here is 128 consecutive columns of one row (four MX groups), so the
// warp decomposition of bq_device.cuh applies unchanged: a half-warp holds a block,
// a quad of lanes holds a group, and the block's four scale bytes form one 32-bit
// word written by a single lane.
#include "bq_device.cuh"
#include "bq_launch.h"

namespace bqk {
namespace {

// Position (row, 128-column block) of linear block index row0 * bpr + cb0 + k, k >= 0.
__device__ __forceinline__ void advance(int64_t row0, int64_t cb0, int k, int64_t bpr, int64_t &row, int64_t &cb)
{
    row = row0;
    cb = cb0 + k;
    while (cb >= bpr) {
        cb -= bpr;
        ++row;
    }
}

// Element offsets of the blocks a lane touches in one chunk of kChunkBlocks blocks that
// starts at (row0, cb0): off[j] for segment j (block 2j + half), for each of up to three
// row-major arrays with leading dimensions ld[a] (in elements, or bytes for byte
// arrays) and per-block widths wid[a] (128 values or 4 scale bytes). A chunk that lies
// in one row (the common case: 8 of the row's cols/128 blocks) takes one multiply per
// array; a chunk that crosses rows walks the block positions.
struct ChunkPos {
    int64_t row0, cb0;
};

// Offset of block k of the chunk in a row-major array with leading dimension ld and
// per-block width wid. kOneRow (the chunk lies in one row, decided per chunk and
// warp-uniform) makes it base + k * wid with the base shared by all blocks.
template <bool kOneRow>
__device__ __forceinline__ int64_t block_offset(const ChunkPos &p, int k, int64_t bpr, int64_t ld, int64_t wid)
{
    if (kOneRow) return p.row0 * ld + p.cb0 * wid + k * wid;
    int64_t r, c;
    advance(p.row0, p.cb0, k, bpr, r, c);
    return r * ld + c * wid;
}

// Byte offset of the four scale bytes of block k of the chunk. Row-major: row * ld_s +
// 4 * (block column). kTiled: the tiled layout of block-scaled GEMM operands, where a
// 128-value block's four E8M0 bytes are one row of a 128-row x 4-column tile; ld_s is
// then the number of tiles per tile row (scale columns of the whole tensor / 4) and c0
// the slice's first tile column. Inside a tile, row r sits at (r % 32) * 16 + (r / 32) * 4.
template <bool kOneRow, bool kTiled>
__device__ __forceinline__ int64_t scale_offset(const ChunkPos &p, int k, int64_t bpr, int64_t ld_s, int64_t c0)
{
    if (!kTiled) return block_offset<kOneRow>(p, k, bpr, ld_s, 4);
    int64_t r, cb;
    if (kOneRow) {
        r = p.row0;
        cb = p.cb0 + k;
    } else {
        advance(p.row0, p.cb0, k, bpr, r, cb);
    }
    return ((r >> 7) * ld_s + c0 + cb) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

// One warp chunk = 4 segments = 8 blocks = 32 groups of 32 values. A lane loads 16
// bytes (8 values) of block 2j + half for each segment j.
template <bool kTail, bool kOneRow>
__device__ __forceinline__ void quant_mx_load(const uint16_t *__restrict__ x, int64_t ld_x, int64_t bpr, int64_t nblk,
                                              int64_t b0, ChunkPos pos, int lane, uint4 (&raw)[kSegs])
{
    const int half = lane >> 4, hl = lane & 15;
#pragma unroll
    for (int j = 0; j < kSegs; j++) {
        const int64_t ox = block_offset<kOneRow>(pos, 2 * j + half, bpr, ld_x, 128);
        raw[j] = (!kTail || b0 + 2 * j + half < nblk) ? ld_stream_v4(x + ox + hl * 8) : make_uint4(0, 0, 0, 0);
    }
}

template <bool kTail>
__device__ __forceinline__ void quant_mx_load_any(const uint16_t *__restrict__ x, int64_t ld_x, int64_t bpr,
                                                  int64_t nblk, int64_t b0, ChunkPos pos, int lane,
                                                  uint4 (&raw)[kSegs])
{
    if (pos.cb0 + kChunkBlocks <= bpr)
        quant_mx_load<kTail, true>(x, ld_x, bpr, nblk, b0, pos, lane, raw);
    else
        quant_mx_load<kTail, false>(x, ld_x, bpr, nblk, b0, pos, lane, raw);
}

template <bool kF16>
__device__ __forceinline__ void widen8(const uint4 &raw, float2 (&v)[4])
{
    if (kF16)
        f16x8_to_f32(raw, v);
    else
        bf16x8_to_f32(raw, v);
}

// Quantize a loaded chunk. After the group amaxes are reduced (4 lanes per group), lane
// L gathers the amax of the chunk's group L (group order = scale-byte order within the
// chunk: block-major, 4 groups per block) and computes that group's E8M0 byte and
// multiplier 2^(127-e) once; each lane then fetches its own group's multiplier per
// segment, and lanes 4b (b = 0..7) store block b's four scale bytes as one 32-bit word.
// The values are widened from the raw registers twice (for the amax, then for the
// codes) rather than kept as 32 floats: 64 registers instead of 80.
template <bool kF16, bool kTiled, bool kTail, bool kOneRow>
__device__ __forceinline__ void quant_mx_compute(const uint4 (&raw)[kSegs], int64_t bpr, int64_t nblk,
                                                 uint8_t *__restrict__ q, int64_t ld_q, uint8_t *__restrict__ s,
                                                 int64_t ld_s, int64_t c0, int64_t b0, ChunkPos pos, int lane)
{
    const int half = lane >> 4, hl = lane & 15;
    float gmax = 0.0f;
#pragma unroll
    for (int j = 0; j < kSegs; j++) {
        float2 v[4];
        widen8<kF16>(raw[j], v);
        float m = amax8(v);
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
        const float g = __shfl_sync(kFull, m, (lane & 7) << 2);
        if ((lane >> 3) == j) gmax = g;
    }
    const uint32_t e = mx_scale_byte(gmax);
    const float p = exp2i(127 - static_cast<int>(e));
#pragma unroll
    for (int j = 0; j < kSegs; j++) {
        const float2 pj = splat(__shfl_sync(kFull, p, 8 * j + (lane >> 2)));
        float2 v[4], y[4];
        widen8<kF16>(raw[j], v);
#pragma unroll
        for (int i = 0; i < 4; i++) y[i] = mul2(v[i], pj);  // exact: a power-of-two scaling
        if (!kTail || b0 + 2 * j + half < nblk) {
            const int64_t oq = block_offset<kOneRow>(pos, 2 * j + half, bpr, ld_q, 128);
            st_v2(q + oq + hl * 8, f32x8_to_e4m3x8(y));
        }
    }
    uint32_t word = e << (8 * (lane & 3));
    word |= __shfl_xor_sync(kFull, word, 1);
    word |= __shfl_xor_sync(kFull, word, 2);
    if ((lane & 3) == 0 && (!kTail || b0 + (lane >> 2) < nblk))
        st_u32(s + scale_offset<kOneRow, kTiled>(pos, lane >> 2, bpr, ld_s, c0), word);
}

template <bool kF16, bool kTiled, bool kTail>
__device__ __forceinline__ void quant_mx_compute_any(const uint4 (&raw)[kSegs], int64_t bpr, int64_t nblk,
                                                     uint8_t *__restrict__ q, int64_t ld_q, uint8_t *__restrict__ s,
                                                     int64_t ld_s, int64_t c0, int64_t b0, ChunkPos pos, int lane)
{
    if (pos.cb0 + kChunkBlocks <= bpr)
        quant_mx_compute<kF16, kTiled, kTail, true>(raw, bpr, nblk, q, ld_q, s, ld_s, c0, b0, pos, lane);
    else
        quant_mx_compute<kF16, kTiled, kTail, false>(raw, bpr, nblk, q, ld_q, s, ld_s, c0, b0, pos, lane);
}

// Grid-stride walk over chunks with the chunk's (row, column block) advanced
// incrementally: one division per warp at the start instead of one per chunk.
template <int CB, int kBlock = kThreads>
struct ChunkWalkT {
    int64_t c, stride, b0, step;
    ChunkPos pos;
    int64_t drow, dcb, bpr;
    // cta, ncta: this CTA's index among the ncta CTAs that share the walk
    __device__ __forceinline__ ChunkWalkT(int64_t bpr_, int64_t cta, int64_t ncta)
    {
        bpr = bpr_;
        stride = (ncta * kBlock) >> 5;
        c = (cta * kBlock + threadIdx.x) >> 5;
        b0 = c * CB;
        pos.row0 = b0 / bpr;
        pos.cb0 = b0 - pos.row0 * bpr;
        step = stride * CB;
        drow = step / bpr;
        dcb = step - drow * bpr;
    }
    __device__ __forceinline__ void next()
    {
        c += stride;
        b0 += step;
        pos.row0 += drow;
        pos.cb0 += dcb;
        if (pos.cb0 >= bpr) {
            pos.cb0 -= bpr;
            ++pos.row0;
        }
    }
};

// 4 resident CTAs per SM (64 registers, no spills): 16.4 us per 4096x7168 slice on
// GB300 against 16.8 us at 3 CTAs per SM. Issuing the next chunk's loads before
// quantizing the current one (80 registers, 3 CTAs per SM) measured the same, 16.5 us.
#ifndef BQ_QUANT_MX_MIN_CTAS
#define BQ_QUANT_MX_MIN_CTAS 4
#endif

// Quantize one [rows, bpr * 128] matrix with ncta CTAs, this one being number cta.
// kF16: the input is FP16 instead of BF16. kTiled: scales go to the tiled GEMM layout
// (see scale_offset), c0 the slice's first tile column.
template <bool kF16, bool kTiled, int kBlock = kThreads>
__device__ __forceinline__ void quant_mx_matrix(const uint16_t *__restrict__ x, int64_t ld_x, int64_t bpr, int64_t nblk,
                                                uint8_t *__restrict__ q, int64_t ld_q, uint8_t *__restrict__ s,
                                                int64_t ld_s, int64_t c0, int64_t cta, int64_t ncta)
{
    const int lane = threadIdx.x & 31;
    const int64_t nfull = nblk / kChunkBlocks;
    ChunkWalkT<kChunkBlocks, kBlock> w(bpr, cta, ncta);
    for (; w.c < nfull; w.next()) {
        uint4 raw[kSegs];
        quant_mx_load_any<false>(x, ld_x, bpr, nblk, w.b0, w.pos, lane, raw);
        quant_mx_compute_any<kF16, kTiled, false>(raw, bpr, nblk, q, ld_q, s, ld_s, c0, w.b0, w.pos, lane);
    }
    if (w.c == nfull && nblk % kChunkBlocks) {
        uint4 raw[kSegs];
        quant_mx_load_any<true>(x, ld_x, bpr, nblk, w.b0, w.pos, lane, raw);
        quant_mx_compute_any<kF16, kTiled, true>(raw, bpr, nblk, q, ld_q, s, ld_s, c0, w.b0, w.pos, lane);
    }
}

// Threads per CTA of the MX quantize (registers per thread at the BQ_QUANT_MX_MIN_CTAS
// budget of 256-thread CTAs whatever the size). For the 89 MB slices of the prefill step
// 256, 512 and 1024 threads measured the same inside the step: 20.5 us per launch with an
// event after every launch, and the same step time, so the launch's fixed cost is not
// the distribution of its CTAs.
#ifndef BQ_QUANT_MX_THREADS
#define BQ_QUANT_MX_THREADS 256
#endif
constexpr int kQuantMxThreads = BQ_QUANT_MX_THREADS;

template <bool kF16, bool kTiled>
__global__ void __launch_bounds__(kQuantMxThreads, BQ_QUANT_MX_MIN_CTAS * kThreads / kQuantMxThreads)
quant_mx_kernel(const uint16_t *__restrict__ x, int64_t ld_x, int64_t bpr, int64_t nblk, uint8_t *__restrict__ q,
                int64_t ld_q, uint8_t *__restrict__ s, int64_t ld_s, int64_t c0)
{
    pdl_begin();
    dbg_begin();
    if (bpr > 0) {
        const int64_t rows = nblk / bpr;
        dbg_allow_2d(x, rows, 256 * bpr, 2 * ld_x, false);
        dbg_allow_2d(q, rows, 128 * bpr, ld_q, true);
        if (kTiled)
            dbg_allow(s, (rows + 127) / 128 * ld_s * 512, true);  // ld_s: tiles per tile row
        else
            dbg_allow_2d(s, rows, 4 * bpr, ld_s, true);
    }
    dbg_ready();
    quant_mx_matrix<kF16, kTiled, kQuantMxThreads>(x, ld_x, bpr, nblk, q, ld_q, s, ld_s, c0, blockIdx.x, gridDim.x);
}

// Several staged slices in one launch (bq_quant_mx_slices): the CTAs are split between
// the slices in proportion to their work, CTAs [cta0[i], cta0[i + 1]) taking slice i;
// each CTA finds its slice once and then walks that slice's chunks exactly as a launch
// of the slice alone would, with its slice-local index and the slice's CTA count.
template <bool kF16>
__global__ void __launch_bounds__(kThreads, BQ_QUANT_MX_MIN_CTAS)
quant_mx_slices_kernel(const __grid_constant__ MxSliceList sl, int64_t rows, uint8_t *__restrict__ q, int64_t ld_q,
                       uint8_t *__restrict__ s, int64_t ld_s)
{
    pdl_begin();
    dbg_begin();
    for (int i = 0; i < sl.n; i++) dbg_allow_2d(sl.x[i], rows, 256 * sl.bpr[i], 2 * sl.ld_x[i], false);
    if (sl.n > 0) {
        const int64_t blocks = sl.cb0[sl.n - 1] + sl.bpr[sl.n - 1];
        dbg_allow_2d(q, rows, 128 * blocks, ld_q, true);
        dbg_allow_2d(s, rows, 4 * blocks, ld_s, true);
    }
    dbg_ready();
    int i = 0;
    while (i + 1 < sl.n && static_cast<int>(blockIdx.x) >= sl.cta0[i + 1]) ++i;
    const int64_t bpr = sl.bpr[i];
    quant_mx_matrix<kF16, false>(sl.x[i], sl.ld_x[i], bpr, rows * bpr, q + 128 * sl.cb0[i], ld_q, s + 4 * sl.cb0[i],
                                 ld_s, 0, static_cast<int64_t>(blockIdx.x) - sl.cta0[i], sl.cta0[i + 1] - sl.cta0[i]);
}

// Materialize one chunk of SEGS segments (2 * SEGS blocks); all loads of the chunk are
// issued before any conversion.
template <int SEGS, bool kTail, bool kOneRow>
__device__ __forceinline__ void dequant_mx_chunk(const uint8_t *__restrict__ q, int64_t ld_q,
                                                 const uint8_t *__restrict__ s, int64_t ld_s, int64_t bpr,
                                                 int64_t nblk, uint16_t *__restrict__ out, int64_t ld_out,
                                                 int64_t b0, ChunkPos pos, int lane)
{
    const int half = lane >> 4, hl = lane & 15;
    uint2 raw[SEGS];
    uint32_t sw[SEGS];
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        const bool ok = !kTail || b0 + 2 * j + half < nblk;
        const int64_t oq = block_offset<kOneRow>(pos, 2 * j + half, bpr, ld_q, 128);
        const int64_t os = block_offset<kOneRow>(pos, 2 * j + half, bpr, ld_s, 4);
        raw[j] = ok ? ld_stream_v2(q + oq + hl * 8) : make_uint2(0, 0);
        sw[j] = ok ? ld_stream_u32(s + os) : 0u;
    }
#pragma unroll
    for (int j = 0; j < SEGS; j++) {
        const uint32_t e = (sw[j] >> (8 * (hl >> 2))) & 0xffu;
        const float p = e == 255u ? __uint_as_float(0x7fc00000u) : exp2i(static_cast<int>(e) - 127);
        float2 v[4];
        e4m3x8_to_f32(raw[j], p, v);
        if (!kTail || b0 + 2 * j + half < nblk) {
            const int64_t oo = block_offset<kOneRow>(pos, 2 * j + half, bpr, ld_out, 128);
            st_v4(out + oo + hl * 8, f32x8_to_bf16x8(v));
        }
    }
}

template <int SEGS, bool kTail>
__device__ __forceinline__ void dequant_mx_chunk_any(const uint8_t *__restrict__ q, int64_t ld_q,
                                                     const uint8_t *__restrict__ s, int64_t ld_s, int64_t bpr,
                                                     int64_t nblk, uint16_t *__restrict__ out, int64_t ld_out,
                                                     int64_t b0, ChunkPos pos, int lane)
{
    if (pos.cb0 + 2 * SEGS <= bpr)
        dequant_mx_chunk<SEGS, kTail, true>(q, ld_q, s, ld_s, bpr, nblk, out, ld_out, b0, pos, lane);
    else
        dequant_mx_chunk<SEGS, kTail, false>(q, ld_q, s, ld_s, bpr, nblk, out, ld_out, b0, pos, lane);
}

// Threads per CTA of the MX materialization: one CTA of 768 threads per SM (24 warps,
// the register file would hold 32) measured 88.0 against 90.2 us per 534 MB launch in
// the prefill step; 512 and 1024 threads measured 90.1. The 1:2 read:write mix runs
// faster with fewer warps storing at once (a zero-compute probe: 6.44 TB/s at 24 warps
// per SM, 6.26 at 32).
#ifndef BQ_DEQUANT_MX_THREADS
#define BQ_DEQUANT_MX_THREADS 768
#endif
constexpr int kDequantMxThreads = BQ_DEQUANT_MX_THREADS;

template <int SEGS>
__global__ void __launch_bounds__(kDequantMxThreads)
dequant_mx_kernel(const uint8_t *__restrict__ q, int64_t ld_q, const uint8_t *__restrict__ s, int64_t ld_s,
                  int64_t bpr, int64_t nblk, uint16_t *__restrict__ out, int64_t ld_out)
{
    pdl_begin();
    dbg_begin();
    if (bpr > 0) {
        const int64_t rows = nblk / bpr;
        dbg_allow_2d(q, rows, 128 * bpr, ld_q, false);
        dbg_allow_2d(s, rows, 4 * bpr, ld_s, false);
        dbg_allow_2d(out, rows, 256 * bpr, 2 * ld_out, true);
    }
    dbg_ready();
    const int lane = threadIdx.x & 31;
    constexpr int CB = 2 * SEGS;
    const int64_t nfull = nblk / CB;
    ChunkWalkT<CB, kDequantMxThreads> w(bpr, blockIdx.x, gridDim.x);
    for (; w.c < nfull; w.next())
        dequant_mx_chunk_any<SEGS, false>(q, ld_q, s, ld_s, bpr, nblk, out, ld_out, w.b0, w.pos, lane);
    if (w.c == nfull && nblk % CB)
        dequant_mx_chunk_any<SEGS, true>(q, ld_q, s, ld_s, bpr, nblk, out, ld_out, w.b0, w.pos, lane);
}

// Segments per warp chunk of the materialization; 2, 4 and 8 measured within 2% of
// each other on GB300 (87-89 us for the 534 MB launch).
#ifndef BQ_SEGS_DEQUANT_MX
#define BQ_SEGS_DEQUANT_MX 4
#endif
constexpr int kSegsDequantMx = BQ_SEGS_DEQUANT_MX;

#define BQK_GRID(kernel, nchunk)                                          \
    int grid = 0;                                                         \
    if (cudaError_t e_ = grid_for((const void *)(kernel), (nchunk), &grid)) \
        return e_;

}  // namespace

namespace {
template <bool kF16, bool kTiled>
cudaError_t launch_quant_mx_any(const uint16_t *x, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q, int64_t ld_q,
                                uint8_t *s, int64_t ld_s, int64_t c0, cudaStream_t st)
{
    const int64_t bpr = cols / 128, nblk = rows * bpr;
    auto kernel = quant_mx_kernel<kF16, kTiled>;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)kernel, (nblk + kChunkBlocks - 1) / kChunkBlocks, &grid, 0,
                                 kQuantMxThreads))
        return e;
    return launch_kernel_block(kernel, grid, kQuantMxThreads, 0, st, x, ld_x, bpr, nblk, q, ld_q, s, ld_s, c0);
}
}  // namespace

cudaError_t launch_quant_mx(const uint16_t *x, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q, int64_t ld_q,
                            uint8_t *s, int64_t ld_s, cudaStream_t st)
{
    return launch_quant_mx_any<false, false>(x, ld_x, rows, cols, q, ld_q, s, ld_s, 0, st);
}

cudaError_t launch_quant_mx_f16(const uint16_t *x, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q, int64_t ld_q,
                                uint8_t *s, int64_t ld_s, cudaStream_t st)
{
    return launch_quant_mx_any<true, false>(x, ld_x, rows, cols, q, ld_q, s, ld_s, 0, st);
}

// Work split of a slice batch: grid CTAs (at least one per slice) in proportion to
// each slice's chunks, no slice given more CTAs than its warps have chunks for.
cudaError_t launch_quant_mx_slices(MxSliceList sl, bool f16, int64_t rows, uint8_t *q, int64_t ld_q, uint8_t *s,
                                   int64_t ld_s, cudaStream_t st)
{
    auto kernel = f16 ? quant_mx_slices_kernel<true> : quant_mx_slices_kernel<false>;
    int64_t chunks[kMaxSlices], total = 0;
    for (int i = 0; i < sl.n; i++) {
        chunks[i] = (rows * sl.bpr[i] + kChunkBlocks - 1) / kChunkBlocks;
        total += chunks[i];
    }
    BQK_GRID(kernel, total);
    constexpr int64_t kWarps = kThreads / 32;
    int64_t ctas[kMaxSlices], used = 0;
    for (int i = 0; i < sl.n; i++) {
        const int64_t most = (chunks[i] + kWarps - 1) / kWarps;
        int64_t c = static_cast<int64_t>(grid) * chunks[i] / total;
        c = c < 1 ? 1 : (c > most ? most : c);
        ctas[i] = c;
        used += c;
    }
    // CTAs left over by the rounding go, one at a time, to the slice with the most
    // chunks per CTA that can still take one
    for (; used < grid; used++) {
        int best = -1;
        for (int i = 0; i < sl.n; i++)
            if (ctas[i] < (chunks[i] + kWarps - 1) / kWarps &&
                (best < 0 || chunks[i] * ctas[best] > chunks[best] * ctas[i]))
                best = i;
        if (best < 0) break;
        ctas[best]++;
    }
    sl.cta0[0] = 0;
    for (int i = 0; i < sl.n; i++) sl.cta0[i + 1] = sl.cta0[i] + static_cast<int>(ctas[i]);
    return launch_kernel(kernel, sl.cta0[sl.n], st, sl, rows, q, ld_q, s, ld_s);
}

cudaError_t launch_quant_mx_tiled(const uint16_t *x, bool f16, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q,
                                  int64_t ld_q, uint8_t *s_tiled, int64_t tiles_per_row, int64_t c0, cudaStream_t st)
{
    if (f16) return launch_quant_mx_any<true, true>(x, ld_x, rows, cols, q, ld_q, s_tiled, tiles_per_row, c0, st);
    return launch_quant_mx_any<false, true>(x, ld_x, rows, cols, q, ld_q, s_tiled, tiles_per_row, c0, st);
}

cudaError_t launch_dequant_mx(const uint8_t *q, int64_t ld_q, const uint8_t *s, int64_t ld_s, int64_t rows,
                              int64_t cols, uint16_t *out, int64_t ld_out, cudaStream_t st)
{
    const int64_t bpr = cols / 128, nblk = rows * bpr;
    constexpr int CB = 2 * kSegsDequantMx;
    int grid = 0;
    if (cudaError_t e = grid_for((const void *)dequant_mx_kernel<kSegsDequantMx>, (nblk + CB - 1) / CB, &grid, 0,
                                 kDequantMxThreads))
        return e;
    return launch_kernel_block(dequant_mx_kernel<kSegsDequantMx>, grid, kDequantMxThreads, 0, st, q, ld_q, s, ld_s,
                               bpr, nblk, out, ld_out);
}

cudaError_t read_wait_counters_mx(unsigned long long (&v)[3]) { return read_wait_counters(v); }

}  // namespace bqk
