// C ABI of libbq.so: argument checks (all before any CUDA call) and kernel dispatch.
// The operations and conventions are specified in include/bq.h.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "bq.h"
#include "bq_launch.h"

#ifndef BQ_DEBUG
#define BQ_DEBUG 0
#endif

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range span(const void *p, int64_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

// Bounding interval of a row-major strided region: rows of `row_bytes`, `ld_bytes` apart.
Range span2d(const void *p, int64_t rows, int64_t row_bytes, int64_t ld_bytes)
{
    return span(p, (rows - 1) * ld_bytes + row_bytes);
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Outputs must be disjoint from each other and from every input.
bool any_alias(const Range *outs, int n_out, const Range *ins, int n_in)
{
    for (int i = 0; i < n_out; i++) {
        for (int j = i + 1; j < n_out; j++)
            if (overlap(outs[i], outs[j])) return true;
        for (int j = 0; j < n_in; j++)
            if (overlap(outs[i], ins[j])) return true;
    }
    return false;
}

bq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BQ_OK : BQ_ERR_CUDA; }

}  // namespace

// ------------------------------------------------------------------ launch sizing
namespace bqk {

namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxKernels = 1024;  // (kernel, dynamic smem, block, device) entries
std::atomic<int> g_sms[kMaxDevices];
struct OccEntry {
    const void *kernel;
    size_t smem;
    int block;
    int device;
    int ctas_per_sm;
};
OccEntry g_occ[kMaxKernels];
int g_occ_n = 0;
std::mutex g_occ_mu;
}  // namespace

cudaError_t grid_for(const void *kernel, int64_t nchunk, int *grid, size_t smem, int block)
{
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    int sms = (dev >= 0 && dev < kMaxDevices) ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    if (sms == 0) {
        if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) return e;
        if (dev >= 0 && dev < kMaxDevices) g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    int occ = 0;
    {
        std::lock_guard<std::mutex> lock(g_occ_mu);
        for (int i = 0; i < g_occ_n; i++)
            if (g_occ[i].kernel == kernel && g_occ[i].smem == smem && g_occ[i].block == block && g_occ[i].device == dev)
                occ = g_occ[i].ctas_per_sm;
    }
    if (occ == 0) {
        if (smem > 48 * 1024) {
            if (cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(smem)))
                return e;
        }
        if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, block, smem)) return e;
        if (occ < 1) occ = 1;
        std::lock_guard<std::mutex> lock(g_occ_mu);
        if (g_occ_n < kMaxKernels) g_occ[g_occ_n++] = OccEntry{kernel, smem, block, dev, occ};
    }
    const int64_t warps_per_cta = block / 32;
    const int64_t need = (nchunk + warps_per_cta - 1) / warps_per_cta;
    const int64_t full = static_cast<int64_t>(sms) * occ;
    *grid = static_cast<int>(need < full ? (need > 0 ? need : 1) : full);
    return cudaSuccess;
}

}  // namespace bqk

// ------------------------------------------------------------------ C ABI
extern "C" {

int bq_abi_version(void) { return BQ_ABI_VERSION; }

const char *bq_status_string(int status)
{
    switch (status) {
    case BQ_OK: return "ok";
    case BQ_ERR_NULL: return "a required pointer is NULL";
    case BQ_ERR_SHAPE: return "size not a multiple of 128, negative, W out of range, or leading dimension too small";
    case BQ_ERR_ALIGN: return "pointer or leading dimension breaks the alignment rules";
    case BQ_ERR_ALIAS: return "an output overlaps an input or another output";
    case BQ_ERR_CUDA: return "the CUDA runtime reported an error for the launch";
    case BQ_ERR_UNSUPPORTED: return "the call needs the debug build (BQ_DEBUG=1)";
    default: return "unknown status";
    }
}

int64_t bq_wire_bytes(int64_t n)
{
    if (n < 0 || n % BQ_BLOCK_I8) return -1;
    return n + 4 * (n / BQ_BLOCK_I8);
}

bq_status bq_quant_i8(const void *x_bf16, int64_t n, int8_t *q, float *scales, cudaStream_t stream)
{
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!x_bf16 || !q || !scales) return BQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(q, 16) || !aligned(scales, 4)) return BQ_ERR_ALIGN;
    const int64_t nblk = n / BQ_BLOCK_I8;
    const Range ins[] = {span(x_bf16, 2 * n)};
    const Range outs[] = {span(q, n), span(scales, 4 * nblk)};
    if (any_alias(outs, 2, ins, 1)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_quant_i8(static_cast<const uint16_t *>(x_bf16), nblk, q, scales, stream));
}

bq_status bq_dequant_i8(const int8_t *q, const float *scales, int64_t n, void *out_bf16, cudaStream_t stream)
{
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!q || !scales || !out_bf16) return BQ_ERR_NULL;
    if (!aligned(q, 16) || !aligned(scales, 4) || !aligned(out_bf16, 16)) return BQ_ERR_ALIGN;
    const int64_t nblk = n / BQ_BLOCK_I8;
    const Range ins[] = {span(q, n), span(scales, 4 * nblk)};
    const Range outs[] = {span(out_bf16, 2 * n)};
    if (any_alias(outs, 1, ins, 2)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_dequant_i8(q, scales, nblk, static_cast<uint16_t *>(out_bf16), stream));
}

bq_status bq_dequant_accum_i8(const int8_t *const *q_srcs, const float *const *scale_srcs, int W, int64_t n,
                              int8_t *q_out, float *scales_out, void *out_bf16, cudaStream_t stream)
{
    if (W < 1 || W > BQ_MAX_W) return BQ_ERR_SHAPE;
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!q_srcs || !scale_srcs || !q_out || !scales_out) return BQ_ERR_NULL;
    const int64_t nblk = n / BQ_BLOCK_I8;
    bqk::SourceList src = {};
    Range ins[2 * BQ_MAX_W];
    for (int w = 0; w < W; w++) {
        if (!q_srcs[w] || !scale_srcs[w]) return BQ_ERR_NULL;
        if (!aligned(q_srcs[w], 16) || !aligned(scale_srcs[w], 4)) return BQ_ERR_ALIGN;
        src.q[w] = q_srcs[w];
        src.s[w] = scale_srcs[w];
        ins[2 * w] = span(q_srcs[w], n);
        ins[2 * w + 1] = span(scale_srcs[w], 4 * nblk);
    }
    if (!aligned(q_out, 16) || !aligned(scales_out, 4) || (out_bf16 && !aligned(out_bf16, 16))) return BQ_ERR_ALIGN;
    Range outs[3] = {span(q_out, n), span(scales_out, 4 * nblk), {}};
    int n_out = 2;
    if (out_bf16) outs[n_out++] = span(out_bf16, 2 * n);
    if (any_alias(outs, n_out, ins, 2 * W)) return BQ_ERR_ALIAS;
    return from_cuda(
        bqk::launch_accum_i8(src, W, nblk, q_out, scales_out, static_cast<uint16_t *>(out_bf16), stream));
}

bq_status bq_ring_hop_i8(const int8_t *q_in, const float *s_in, const void *x_local_bf16, int64_t n, int8_t *q_out,
                         float *s_out, void *out_bf16, cudaStream_t stream)
{
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!q_in || !s_in || !x_local_bf16 || !q_out || !s_out) return BQ_ERR_NULL;
    if (!aligned(q_in, 16) || !aligned(s_in, 4) || !aligned(x_local_bf16, 16) || !aligned(q_out, 16) ||
        !aligned(s_out, 4) || (out_bf16 && !aligned(out_bf16, 16)))
        return BQ_ERR_ALIGN;
    const int64_t nblk = n / BQ_BLOCK_I8;
    const Range ins[] = {span(q_in, n), span(s_in, 4 * nblk), span(x_local_bf16, 2 * n)};
    Range outs[3] = {span(q_out, n), span(s_out, 4 * nblk), {}};
    int n_out = 2;
    if (out_bf16) outs[n_out++] = span(out_bf16, 2 * n);
    if (any_alias(outs, n_out, ins, 3)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_ring_hop_i8(q_in, s_in, static_cast<const uint16_t *>(x_local_bf16), nblk, q_out,
                                             s_out, static_cast<uint16_t *>(out_bf16), stream));
}

bq_status bq_quant_mx(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q_e4m3, int64_t ld_q,
                      uint8_t *s_e8m0, int64_t ld_s, cudaStream_t stream)
{
    if (rows < 0 || cols < 0 || cols % 128) return BQ_ERR_SHAPE;
    if (rows == 0 || cols == 0) return BQ_OK;
    if (ld_x < cols || ld_q < cols || ld_s < cols / BQ_GROUP_MX) return BQ_ERR_SHAPE;
    if (!x_bf16 || !q_e4m3 || !s_e8m0) return BQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || ld_x % 8 || !aligned(q_e4m3, 16) || ld_q % 16 || !aligned(s_e8m0, 4) || ld_s % 4)
        return BQ_ERR_ALIGN;
    const Range ins[] = {span2d(x_bf16, rows, 2 * cols, 2 * ld_x)};
    const Range outs[] = {span2d(q_e4m3, rows, cols, ld_q), span2d(s_e8m0, rows, cols / BQ_GROUP_MX, ld_s)};
    if (any_alias(outs, 2, ins, 1)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_quant_mx(static_cast<const uint16_t *>(x_bf16), ld_x, rows, cols, q_e4m3, ld_q,
                                          s_e8m0, ld_s, stream));
}

bq_status bq_dequant_mx(const uint8_t *q_e4m3, int64_t ld_q, const uint8_t *s_e8m0, int64_t ld_s, int64_t rows,
                        int64_t cols, void *out_bf16, int64_t ld_out, cudaStream_t stream)
{
    if (rows < 0 || cols < 0 || cols % 128) return BQ_ERR_SHAPE;
    if (rows == 0 || cols == 0) return BQ_OK;
    if (ld_q < cols || ld_s < cols / BQ_GROUP_MX || ld_out < cols) return BQ_ERR_SHAPE;
    if (!q_e4m3 || !s_e8m0 || !out_bf16) return BQ_ERR_NULL;
    if (!aligned(q_e4m3, 16) || ld_q % 16 || !aligned(s_e8m0, 4) || ld_s % 4 || !aligned(out_bf16, 16) || ld_out % 8)
        return BQ_ERR_ALIGN;
    const Range ins[] = {span2d(q_e4m3, rows, cols, ld_q), span2d(s_e8m0, rows, cols / BQ_GROUP_MX, ld_s)};
    const Range outs[] = {span2d(out_bf16, rows, 2 * cols, 2 * ld_out)};
    if (any_alias(outs, 1, ins, 2)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_dequant_mx(q_e4m3, ld_q, s_e8m0, ld_s, rows, cols, static_cast<uint16_t *>(out_bf16),
                                            ld_out, stream));
}

bq_status bq_dequant_accum_mx(const uint8_t *const *q_srcs, const uint8_t *const *s_srcs, int W, int64_t n,
                              uint8_t *q_out, uint8_t *s_out, void *out_bf16, cudaStream_t stream)
{
    if (W < 1 || W > BQ_MAX_W) return BQ_ERR_SHAPE;
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!q_srcs || !s_srcs || !q_out || !s_out) return BQ_ERR_NULL;
    const int64_t nblk = n / BQ_BLOCK_I8;
    bqk::MxSourceList src = {};
    Range ins[2 * BQ_MAX_W];
    for (int w = 0; w < W; w++) {
        if (!q_srcs[w] || !s_srcs[w]) return BQ_ERR_NULL;
        if (!aligned(q_srcs[w], 16) || !aligned(s_srcs[w], 4)) return BQ_ERR_ALIGN;
        src.q[w] = q_srcs[w];
        src.s[w] = reinterpret_cast<const uint32_t *>(s_srcs[w]);
        ins[2 * w] = span(q_srcs[w], n);
        ins[2 * w + 1] = span(s_srcs[w], 4 * nblk);
    }
    if (!aligned(q_out, 16) || !aligned(s_out, 4) || (out_bf16 && !aligned(out_bf16, 16))) return BQ_ERR_ALIGN;
    Range outs[3] = {span(q_out, n), span(s_out, 4 * nblk), {}};
    int n_out = 2;
    if (out_bf16) outs[n_out++] = span(out_bf16, 2 * n);
    if (any_alias(outs, n_out, ins, 2 * W)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_accum_mx(src, W, nblk, q_out, reinterpret_cast<uint32_t *>(s_out),
                                          static_cast<uint16_t *>(out_bf16), stream));
}

bq_status bq_ring_hop_mx(const uint8_t *q_in, const uint8_t *s_in, const void *x_local_bf16, int64_t n,
                         uint8_t *q_out, uint8_t *s_out, void *out_bf16, cudaStream_t stream)
{
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!q_in || !s_in || !x_local_bf16 || !q_out || !s_out) return BQ_ERR_NULL;
    if (!aligned(q_in, 16) || !aligned(s_in, 4) || !aligned(x_local_bf16, 16) || !aligned(q_out, 16) ||
        !aligned(s_out, 4) || (out_bf16 && !aligned(out_bf16, 16)))
        return BQ_ERR_ALIGN;
    const int64_t nblk = n / BQ_BLOCK_I8;
    const Range ins[] = {span(q_in, n), span(s_in, 4 * nblk), span(x_local_bf16, 2 * n)};
    Range outs[3] = {span(q_out, n), span(s_out, 4 * nblk), {}};
    int n_out = 2;
    if (out_bf16) outs[n_out++] = span(out_bf16, 2 * n);
    if (any_alias(outs, n_out, ins, 3)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_ring_hop_mx(q_in, reinterpret_cast<const uint32_t *>(s_in),
                                             static_cast<const uint16_t *>(x_local_bf16), nblk, q_out,
                                             reinterpret_cast<uint32_t *>(s_out), static_cast<uint16_t *>(out_bf16),
                                             stream));
}

bq_status bq_quant_mx_f16(const void *x_f16, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q_e4m3, int64_t ld_q,
                          uint8_t *s_e8m0, int64_t ld_s, cudaStream_t stream)
{
    if (rows < 0 || cols < 0 || cols % 128) return BQ_ERR_SHAPE;
    if (rows == 0 || cols == 0) return BQ_OK;
    if (ld_x < cols || ld_q < cols || ld_s < cols / BQ_GROUP_MX) return BQ_ERR_SHAPE;
    if (!x_f16 || !q_e4m3 || !s_e8m0) return BQ_ERR_NULL;
    if (!aligned(x_f16, 16) || ld_x % 8 || !aligned(q_e4m3, 16) || ld_q % 16 || !aligned(s_e8m0, 4) || ld_s % 4)
        return BQ_ERR_ALIGN;
    const Range ins[] = {span2d(x_f16, rows, 2 * cols, 2 * ld_x)};
    const Range outs[] = {span2d(q_e4m3, rows, cols, ld_q), span2d(s_e8m0, rows, cols / BQ_GROUP_MX, ld_s)};
    if (any_alias(outs, 2, ins, 1)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_quant_mx_f16(static_cast<const uint16_t *>(x_f16), ld_x, rows, cols, q_e4m3, ld_q,
                                              s_e8m0, ld_s, stream));
}

bq_status bq_quant_mx_tiled(const void *x, int x_is_f16, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q_e4m3,
                            int64_t ld_q, uint8_t *s_tiled, int64_t g_total, int64_t g0, cudaStream_t stream)
{
    if (rows < 0 || cols < 0 || cols % 128) return BQ_ERR_SHAPE;
    if (g_total < 0 || g_total % 4 || g0 < 0 || g0 % 4 || g0 + cols / BQ_GROUP_MX > g_total) return BQ_ERR_SHAPE;
    if (rows == 0 || cols == 0) return BQ_OK;
    if (ld_x < cols || ld_q < cols) return BQ_ERR_SHAPE;
    if (!x || !q_e4m3 || !s_tiled) return BQ_ERR_NULL;
    if (!aligned(x, 16) || ld_x % 8 || !aligned(q_e4m3, 16) || ld_q % 16 || !aligned(s_tiled, 4)) return BQ_ERR_ALIGN;
    const int64_t tiled_bytes = ((rows + 127) / 128) * (g_total / 4) * 512;
    const Range ins[] = {span2d(x, rows, 2 * cols, 2 * ld_x)};
    const Range outs[] = {span2d(q_e4m3, rows, cols, ld_q), span(s_tiled, tiled_bytes)};
    if (any_alias(outs, 2, ins, 1)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_quant_mx_tiled(static_cast<const uint16_t *>(x), x_is_f16 != 0, ld_x, rows, cols,
                                                q_e4m3, ld_q, s_tiled, g_total / 4, g0 / 4, stream));
}

bq_status bq_quant_mx_slices(const bq_mx_slice *slices, int nslices, int x_is_f16, int64_t rows, uint8_t *q_e4m3,
                             int64_t ld_q, uint8_t *s_e8m0, int64_t ld_s, cudaStream_t stream)
{
    if (nslices < 1 || nslices > BQ_MAX_SLICES || rows < 0) return BQ_ERR_SHAPE;
    if (!slices) return BQ_ERR_NULL;
    int64_t total = 0;
    for (int i = 0; i < nslices; i++) {
        const int64_t c = slices[i].cols;
        if (c < 0 || c % 128 || slices[i].ld_x < c) return BQ_ERR_SHAPE;
        total += c;
    }
    if (rows == 0 || total == 0) return BQ_OK;
    if (ld_q < total || ld_s < total / BQ_GROUP_MX) return BQ_ERR_SHAPE;
    if (!q_e4m3 || !s_e8m0) return BQ_ERR_NULL;
    if (!aligned(q_e4m3, 16) || ld_q % 16 || !aligned(s_e8m0, 4) || ld_s % 4) return BQ_ERR_ALIGN;
    Range ins[BQ_MAX_SLICES];
    bqk::MxSliceList sl = {};
    int64_t col = 0;
    for (int i = 0; i < nslices; i++) {
        const int64_t c = slices[i].cols;
        if (c == 0) continue;
        if (!slices[i].x) return BQ_ERR_NULL;
        if (!aligned(slices[i].x, 16) || slices[i].ld_x % 8) return BQ_ERR_ALIGN;
        ins[sl.n] = span2d(slices[i].x, rows, 2 * c, 2 * slices[i].ld_x);
        sl.x[sl.n] = static_cast<const uint16_t *>(slices[i].x);
        sl.ld_x[sl.n] = slices[i].ld_x;
        sl.bpr[sl.n] = c / 128;
        sl.cb0[sl.n] = col / 128;
        sl.n++;
        col += c;
    }
    const Range outs[] = {span2d(q_e4m3, rows, total, ld_q), span2d(s_e8m0, rows, total / BQ_GROUP_MX, ld_s)};
    if (any_alias(outs, 2, ins, sl.n)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_quant_mx_slices(sl, x_is_f16 != 0, rows, q_e4m3, ld_q, s_e8m0, ld_s, stream));
}

int64_t bq_mx_tiled_scale_bytes(int64_t rows, int64_t g_total)
{
    if (rows < 0 || g_total < 0 || g_total % 4) return -1;
    return ((rows + 127) / 128) * (g_total / 4) * 512;
}

namespace {
// Shared checks of the reduce + quantize calls: W BF16 sources -> payload [n] (1 byte
// per value, 16-byte aligned), FP32 scales [n/128] (4-byte aligned), optional BF16.
bq_status check_reduce(const void *const *x_srcs, int W, int64_t n, const void *q, const void *scales,
                       const void *out_bf16, bqk::Bf16List *src)
{
    if (W < 1 || W > BQ_MAX_W) return BQ_ERR_SHAPE;
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!x_srcs || !q || !scales) return BQ_ERR_NULL;
    Range ins[BQ_MAX_W];
    for (int w = 0; w < W; w++) {
        if (!x_srcs[w]) return BQ_ERR_NULL;
        if (!aligned(x_srcs[w], 16)) return BQ_ERR_ALIGN;
        src->x[w] = static_cast<const uint16_t *>(x_srcs[w]);
        ins[w] = span(x_srcs[w], 2 * n);
    }
    if (!aligned(q, 16) || !aligned(scales, 4) || (out_bf16 && !aligned(out_bf16, 16))) return BQ_ERR_ALIGN;
    Range outs[3] = {span(q, n), span(scales, 4 * (n / BQ_BLOCK_I8)), {}};
    int n_out = 2;
    if (out_bf16) outs[n_out++] = span(out_bf16, 2 * n);
    if (any_alias(outs, n_out, ins, W)) return BQ_ERR_ALIAS;
    return BQ_OK;
}
}  // namespace

bq_status bq_reduce_quant_i8(const void *const *x_srcs, int W, int64_t n, int8_t *q, float *scales, void *out_bf16,
                             cudaStream_t stream)
{
    bqk::Bf16List src = {};
    if (bq_status e = check_reduce(x_srcs, W, n, q, scales, out_bf16, &src)) return e;
    if (n == 0) return BQ_OK;
    return from_cuda(bqk::launch_reduce_quant_i8(src, W, n / BQ_BLOCK_I8, q, scales,
                                                 static_cast<uint16_t *>(out_bf16), stream));
}

bq_status bq_quant_e4m3(const void *x_bf16, int64_t n, uint8_t *q, float *scales, cudaStream_t stream)
{
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!x_bf16 || !q || !scales) return BQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(q, 16) || !aligned(scales, 4)) return BQ_ERR_ALIGN;
    const int64_t nblk = n / BQ_BLOCK_I8;
    const Range ins[] = {span(x_bf16, 2 * n)};
    const Range outs[] = {span(q, n), span(scales, 4 * nblk)};
    if (any_alias(outs, 2, ins, 1)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_quant_e4m3(static_cast<const uint16_t *>(x_bf16), nblk, q, scales, stream));
}

bq_status bq_dequant_e4m3(const uint8_t *q, const float *scales, int64_t n, void *out_bf16, cudaStream_t stream)
{
    if (n < 0 || n % BQ_BLOCK_I8) return BQ_ERR_SHAPE;
    if (n == 0) return BQ_OK;
    if (!q || !scales || !out_bf16) return BQ_ERR_NULL;
    if (!aligned(q, 16) || !aligned(scales, 4) || !aligned(out_bf16, 16)) return BQ_ERR_ALIGN;
    const int64_t nblk = n / BQ_BLOCK_I8;
    const Range ins[] = {span(q, n), span(scales, 4 * nblk)};
    const Range outs[] = {span(out_bf16, 2 * n)};
    if (any_alias(outs, 1, ins, 2)) return BQ_ERR_ALIAS;
    return from_cuda(bqk::launch_dequant_e4m3(q, scales, nblk, static_cast<uint16_t *>(out_bf16), stream));
}

bq_status bq_reduce_quant_e4m3(const void *const *x_srcs, int W, int64_t n, uint8_t *q, float *scales,
                               void *out_bf16, cudaStream_t stream)
{
    bqk::Bf16List src = {};
    if (bq_status e = check_reduce(x_srcs, W, n, q, scales, out_bf16, &src)) return e;
    if (n == 0) return BQ_OK;
    return from_cuda(bqk::launch_reduce_quant_e4m3(src, W, n / BQ_BLOCK_I8, q, scales,
                                                   static_cast<uint16_t *>(out_bf16), stream));
}

}  // extern "C"

namespace {
// Growth of the current device's counter `which` (0: abandoned waits, 1: copies that
// did not land after one, 2: accesses a debug build declined) since the previous call
// for it. The device counters only grow; the last totals seen are kept per device here,
// and they are advanced only after every translation unit's counters were read.
constexpr int kMaxDevices = 64;
std::mutex g_seen_mu;
unsigned long long g_seen[kMaxDevices][3];

bq_status take_wait_counter(int which, int64_t *count)
{
    if (!count) return BQ_ERR_NULL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BQ_ERR_CUDA;
    unsigned long long total = 0;
    for (auto read : {bqk::read_wait_counters_i8, bqk::read_wait_counters_mx_wire, bqk::read_wait_counters_mx,
                      bqk::read_wait_counters_e4m3}) {
        unsigned long long v[3] = {0, 0, 0};
        if (read(v) != cudaSuccess) return BQ_ERR_CUDA;
        total += v[which];
    }
    std::lock_guard<std::mutex> lock(g_seen_mu);
    *count = static_cast<int64_t>(total - g_seen[dev][which]);
    g_seen[dev][which] = total;
    return BQ_OK;
}
}  // namespace

extern "C" {

bq_status bq_take_wait_timeouts(int64_t *count) { return take_wait_counter(0, count); }

bq_status bq_take_wait_unlanded(int64_t *count) { return take_wait_counter(1, count); }

bq_status bq_take_index_errors(int64_t *count) { return take_wait_counter(2, count); }

int bq_debug_build(void) { return BQ_DEBUG; }

bq_status bq_selftest_index_check(void *buf, int64_t bytes, cudaStream_t stream)
{
    if (!BQ_DEBUG) return BQ_ERR_UNSUPPORTED;
    if (!buf) return BQ_ERR_NULL;
    if (bytes < 1024) return BQ_ERR_SHAPE;
    if (!aligned(buf, 16)) return BQ_ERR_ALIGN;
    return from_cuda(bqk::launch_index_selftest(buf, stream));
}

bq_status bq_selftest_wait_timeout(cudaStream_t stream) { return from_cuda(bqk::launch_wait_selftest(stream)); }

}  // extern "C"
