/*
 * bq.h — C ABI of libbq.so, the block-quantized wire codec for GB300 (sm_103a).
 *
 * The codec compresses BF16 all-reduce payloads into wire formats of 132 bytes per
 * 128 values: the two of the pages' compressed modes below, and the legacy E4M3 codec
 * (one E4M3 byte per value and one FP32 scale per 128 values) they replace:
 *
 *   block INT8   128 signed payload bytes + one FP32 scale = amax/127 per block of
 *                128 consecutive values ("feat(pcie_dma): add block-INT8 wire modes
 *                for AG, ring, and A2A", Summary);
 *   MXFP8        E4M3 values + one E8M0 scale byte per 32 consecutive values of a
 *                row ("feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary).
 *
 * Wire layout of an n-value tensor (n % 128 == 0). The pages fix the size of a block
 * (132 bytes) but not how payload and scales interleave; this library keeps them in
 * two regions so that both can be moved with 16-byte vector accesses:
 *   INT8   payload  int8_t  q[n]          value i in block i/128
 *          scales   float   s[n/128]      little-endian IEEE binary32
 *   MXFP8  values   uint8_t q[rows][ld_q] E4M3 codes (OCP: bias 7, max 448)
 *          scales   uint8_t s[rows][ld_s] E8M0 byte e stands for 2^(e-127);
 *                                         s[r][g] covers columns [32g, 32g+32)
 * A caller that wants one contiguous wire buffer places the scale region directly
 * after the payload region (byte offset n, which keeps 16-byte alignment).
 * A flat MX wire (the all-reduce shard of the mx_a2a and mx_ring modes) is the
 * one-row case: codes q[n], then E8M0 bytes s[n/32]; the four scale bytes of a
 * 128-value block form one 4-byte word, as the INT8 scale of that block does.
 *
 * Arithmetic (bit-exact; no fused multiply-add anywhere):
 *   quantize   amax = max |x| over the block; s = fl(amax / 127) (IEEE binary32
 *              division, round to nearest even); q = nearest integer to fl(x / s),
 *              ties to even, clamped to [-127, 127]; a block with s == 0 (all-zero
 *              block) has q == 0.
 *   materialize  out = BF16_rne(fl((float)q * s)) — a binary32 product, then BF16.
 *   accumulate   d_w = fl(q_w * s_w); acc = (((d_0 + d_1) + d_2) + ...) in binary32
 *              in source order; acc is requantized as above.
 *   ring hop   v = fl(fl(q_in * s_in) + x_local), requantized as above.
 *   MX scale   all-zero group -> 127; else the smallest e in [0, 254] with
 *              2^(e-127) >= fl(amax / 448) ("feat(pcie_dma): add INT8 and MXFP8 wire
 *              modes", review comment on mxfp8_scale_byte: round toward +inf,
 *              saturating).
 *   MX values  code = E4M3_rne_satfinite(x * 2^(127-e)); the sign of zero is kept.
 *   MX materialize  out = BF16_rne(decode(code) * 2^(e-127)) (the product is exact).
 *   MX accumulate   d_w = decode(code_w) * 2^(e_w-127) (exact in binary32);
 *              acc = (((d_0 + d_1) + d_2) + ...) in binary32 in source order; acc is
 *              requantized per 32-value group with the MX scale and value rules,
 *              the amax taken over the binary32 sums.
 *   reduce + quantize  (the all-gather modes' BF16 reduce-scatter fused with the
 *              payload) y = BF16_rne(((x_0 + x_1) + ...) in binary32 in rank
 *              order), then y is quantized by the codec.
 *   legacy E4M3  s = fl(amax / 448) per 128-value block; code =
 *              E4M3_rne_satfinite(fl(x / s)), sign of zero kept; a block with s == 0
 *              has every code 0x00; materialize out = BF16_rne(fl(decode(code) * s)).
 *   MX ring hop  v = fl(decode(code_in) * 2^(e_in-127) + x_local), requantized as
 *              MX. (The MXFP8 page's Summary runs its codec on the same ring and
 *              all-to-all topologies, mx_ring and mx_a2a; these two rules are the
 *              INT8 ones with the MX codec.)
 * Inputs must be finite; results for NaN or infinity inputs are not specified.
 *
 * Conventions shared by every call:
 *   - All data pointers are DEVICE pointers owned by the caller (host arrays of
 *     device pointers where stated). The library allocates nothing, keeps no state
 *     between calls beyond a per-device cache of launch parameters, and never
 *     synchronizes: work is enqueued on `stream` (0 = the legacy default stream)
 *     and the call returns.
 *   - Every check happens before any launch; a call that returns an error has not
 *     touched device memory. n == 0 (or rows == 0 / cols == 0) is a valid no-op and
 *     returns BQ_OK without launching.
 *   - Shape: n % 128 == 0 and, for MX, cols % 128 == 0 — otherwise BQ_ERR_SHAPE and
 *     the caller keeps its BF16 path ("feat(pcie_dma): add INT8 and MXFP8 wire
 *     modes", Configuration: compressed transport needs a shard divisible by 128).
 *   - Alignment: BF16 and payload/value pointers 16-byte aligned; INT8 scale pointers
 *     4-byte aligned; MX scale pointers 4-byte aligned with ld_s % 4 == 0; MX strides
 *     keep every row 16-byte aligned (ld_x % 8 == 0 elements, ld_q % 16 == 0 bytes,
 *     ld_out % 8 == 0 elements). Otherwise BQ_ERR_ALIGN.
 *   - Outputs may not overlap inputs or each other (checked on the address ranges
 *     the call touches; strided MX ranges are taken as their bounding intervals).
 *     Otherwise BQ_ERR_ALIAS.
 *   - A failed kernel launch returns BQ_ERR_CUDA (the CUDA error is left readable
 *     through cudaGetLastError's usual rules only as far as this call consumed it).
 *   - Errors in earlier asynchronous work on the stream are not detected here.
 */
#ifndef BQ_H
#define BQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BQ_API __attribute__((visibility("default")))
#else
#define BQ_API
#endif

#define BQ_ABI_VERSION 5
#define BQ_BLOCK_I8 128 /* values per INT8 block */
#define BQ_GROUP_MX 32  /* values per E8M0 scale */
#define BQ_MAX_W 16     /* most sources one accumulate call takes */

typedef enum {
    BQ_OK = 0,
    BQ_ERR_NULL = 1,  /* a required pointer is NULL */
    BQ_ERR_SHAPE = 2, /* n or cols not a multiple of 128, negative size, W out of
                         [1, BQ_MAX_W], or a leading dimension too small */
    BQ_ERR_ALIGN = 3, /* a pointer or leading dimension breaks the alignment rules */
    BQ_ERR_ALIAS = 4, /* an output overlaps an input or another output */
    BQ_ERR_CUDA = 5,  /* the CUDA runtime reported an error for this call's launch */
    BQ_ERR_UNSUPPORTED = 6 /* the call exists only in the debug build (bq_selftest_index_check) */
} bq_status;

/* BQ_ABI_VERSION of the loaded library. */
BQ_API int bq_abi_version(void);

/* Static English description of a status code (never NULL). */
BQ_API const char *bq_status_string(int status);

/* Bytes on the wire for n values in either codec: 132 * n / 128 ("feat(pcie_dma):
 * add block-INT8 wire modes for AG, ring, and A2A", Summary). Returns -1 when
 * n < 0 or n % 128 != 0. */
BQ_API int64_t bq_wire_bytes(int64_t n);

/* BF16 -> block INT8 ("feat(pcie_dma): add block-INT8 wire modes for AG, ring, and
 * A2A", Implementation: BF16 -> signed INT8 quantization, one scale per 128 values).
 *   x_bf16   [n] BF16, 16-byte aligned (read)
 *   q        [n] int8 payload, 16-byte aligned (written)
 *   scales   [n/128] FP32, 4-byte aligned (written) */
BQ_API bq_status bq_quant_i8(const void *x_bf16, int64_t n, int8_t *q, float *scales,
                      cudaStream_t stream);

/* Block INT8 -> BF16 materialization (same page, Implementation: signed INT8 -> BF16
 * materialization; Summary: owners materialize from the forwarded payload).
 *   q [n] int8 (read), scales [n/128] FP32 (read), out_bf16 [n] BF16 (written). */
BQ_API bq_status bq_dequant_i8(const int8_t *q, const float *scales, int64_t n, void *out_bf16,
                        cudaStream_t stream);

/* Multi-source dequantize with FP32 accumulation, then requantize (same page,
 * Implementation: multi-source INT8 dequantization with FP32 accumulation for A2A).
 *   q_srcs, scale_srcs  HOST arrays of W DEVICE pointers ([n] int8 and [n/128] FP32
 *                       each); their order is the summation order
 *   W                   1 <= W <= BQ_MAX_W
 *   q_out, scales_out   the requantized payload (written)
 *   out_bf16            NULL, or [n] BF16 receiving the materialization of the new
 *                       payload, bit-identical to bq_dequant_i8(q_out, scales_out)
 *                       (the owner materializes the payload it forwards).
 * Sources may repeat or overlap one another. */
BQ_API bq_status bq_dequant_accum_i8(const int8_t *const *q_srcs, const float *const *scale_srcs,
                              int W, int64_t n, int8_t *q_out, float *scales_out,
                              void *out_bf16, cudaStream_t stream);

/* Fused ring reduce-scatter hop: dequantize the incoming payload, add the local BF16
 * shard in FP32, requantize (same page, Implementation: fused INT8
 * dequantize-add-requantize for each ring reduce-scatter hop).
 *   q_in [n], s_in [n/128]   incoming payload (read)
 *   x_local_bf16 [n]         this rank's shard (read)
 *   q_out, s_out             outgoing payload (written)
 *   out_bf16                 NULL, or [n] BF16 materialization of the outgoing
 *                            payload (for the hop that ends at the owner). */
BQ_API bq_status bq_ring_hop_i8(const int8_t *q_in, const float *s_in, const void *x_local_bf16,
                         int64_t n, int8_t *q_out, float *s_out, void *out_bf16,
                         cudaStream_t stream);

/* BF16 [rows, cols] -> MXFP8 ("feat(pcie_dma): add INT8 and MXFP8 wire modes",
 * Summary and the mxfp8_scale_byte review comment). Row-major with leading
 * dimensions, so a 128-column-aligned slice of a wider buffer is addressed by
 * offsetting the pointers: q_e4m3 + col0 and s_e8m0 + col0/32 with col0 % 128 == 0
 * ("[II] Support staged MXFP8 linear inputs", Behavior and Compatibility).
 *   x_bf16  [rows][ld_x] BF16 (read);      ld_x >= cols, ld_x % 8 == 0
 *   q_e4m3  [rows][ld_q] bytes (written);  ld_q >= cols, ld_q % 16 == 0
 *   s_e8m0  [rows][ld_s] bytes (written);  ld_s >= cols/32, ld_s % 4 == 0 */
BQ_API bq_status bq_quant_mx(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x,
                      uint8_t *q_e4m3, int64_t ld_q, uint8_t *s_e8m0, int64_t ld_s,
                      cudaStream_t stream);

/* MXFP8 -> BF16 materialization (same page, review: dma_dequant_store_mx).
 *   q_e4m3 [rows][ld_q], s_e8m0 [rows][ld_s] (read); out_bf16 [rows][ld_out] (written),
 *   ld_out >= cols, ld_out % 8 == 0. Scale byte 255 and codes 0x7F/0xFF are NaN. */
BQ_API bq_status bq_dequant_mx(const uint8_t *q_e4m3, int64_t ld_q, const uint8_t *s_e8m0,
                        int64_t ld_s, int64_t rows, int64_t cols, void *out_bf16,
                        int64_t ld_out, cudaStream_t stream);

/* mx_a2a reduction on flat MX wires: decode every source exactly to binary32, add the
 * sources in source order in binary32, requantize per 32-value group ("feat(pcie_dma):
 * add INT8 and MXFP8 wire modes", Summary: mx_a2a on the all-to-all topology; the
 * owner materializes the payload it forwards).
 *   q_srcs, s_srcs      HOST arrays of W DEVICE pointers: [n] E4M3 codes (16-byte
 *                       aligned) and [n/32] E8M0 bytes (4-byte aligned) each; their
 *                       order is the summation order
 *   W                   1 <= W <= BQ_MAX_W
 *   q_out [n], s_out [n/32]  the requantized wire (written; same alignment)
 *   out_bf16            NULL, or [n] BF16 (16-byte aligned) receiving the
 *                       materialization of the new wire, bit-identical to
 *                       bq_dequant_mx(q_out, n, s_out, n/32, 1, n, out_bf16, n).
 * Sources may repeat or overlap one another. */
BQ_API bq_status bq_dequant_accum_mx(const uint8_t *const *q_srcs, const uint8_t *const *s_srcs,
                              int W, int64_t n, uint8_t *q_out, uint8_t *s_out, void *out_bf16,
                              cudaStream_t stream);

/* mx_ring hop on flat MX wires: decode the incoming wire, add the local BF16 shard in
 * binary32, requantize per 32-value group (same page, Summary: mx_ring).
 *   q_in [n], s_in [n/32]   incoming wire (read; 16- and 4-byte aligned)
 *   x_local_bf16 [n]        this rank's shard (read; 16-byte aligned)
 *   q_out, s_out            outgoing wire (written)
 *   out_bf16                NULL, or [n] BF16 materialization of the outgoing wire. */
BQ_API bq_status bq_ring_hop_mx(const uint8_t *q_in, const uint8_t *s_in, const void *x_local_bf16,
                         int64_t n, uint8_t *q_out, uint8_t *s_out, void *out_bf16,
                         cudaStream_t stream);

/* bq_quant_mx for an FP16 input ("[II] Support staged MXFP8 linear inputs", Behavior:
 * BF16 or FP16 feature slices). FP16 widens exactly to binary32; the arguments,
 * layout and rules are those of bq_quant_mx with x_f16 in place of x_bf16. */
BQ_API bq_status bq_quant_mx_f16(const void *x_f16, int64_t rows, int64_t cols, int64_t ld_x,
                          uint8_t *q_e4m3, int64_t ld_q, uint8_t *s_e8m0, int64_t ld_s,
                          cudaStream_t stream);

/* bq_quant_mx (BF16, or FP16 when x_is_f16 != 0) writing the E8M0 scales in the tiled
 * layout that block-scaled GEMM operands use, for a GEMM that consumes the assembled
 * MXFP8 input ("[II] Support staged MXFP8 linear inputs", Behavior: empty_input
 * allocates values and scale layouts; mm_quantized runs the GEMM on them). The pages
 * do not print this layout; it is the publicly described one that cuBLAS block-scaled
 * GEMMs read ("1D block scaling factors layout"), the same as PyTorch's to_blocked:
 * the scale matrix S [rows_total, g_total] (g_total = columns of the whole tensor / 32,
 * a multiple of 4) is cut into tiles of 128 rows x 4 scale columns, tile (R, C) stored
 * as 512 bytes at (R * g_total/4 + C) * 512, and inside a tile row r, column c at byte
 * (r % 32) * 16 + (r / 32) * 4 + c. Rows past `rows` in the last tile row are not
 * written (allocate bq_mx_tiled_scale_bytes and zero-fill if a consumer reads them).
 *   x, rows, cols, ld_x, q_e4m3, ld_q   as bq_quant_mx (a slice of a wider tensor)
 *   s_tiled    base of the whole tensor's tiled scale buffer (4-byte aligned)
 *   g_total    scale columns of the whole tensor; g0 = the slice's first scale column
 *              (column offset / 32), a multiple of 4; g0 + cols/32 <= g_total. */
BQ_API bq_status bq_quant_mx_tiled(const void *x, int x_is_f16, int64_t rows, int64_t cols, int64_t ld_x,
                            uint8_t *q_e4m3, int64_t ld_q, uint8_t *s_tiled, int64_t g_total,
                            int64_t g0, cudaStream_t stream);

/* Several staged slices quantized by one call: the bytes of bq_quant_mx (BF16, or
 * bq_quant_mx_f16 when x_is_f16 != 0) called once per slice, slice i at the
 * destination columns that follow slice i - 1's ("[II] Support staged MXFP8 linear
 * inputs", Behavior: quantize_input_slice writes a 128-column-aligned slice at its
 * offset of the assembled input). One launch covers every slice, so slices that are
 * ready together do not pay one launch's ramp and tail each.
 *   slices[i].x      [rows][slices[i].ld_x] BF16 or FP16 (read); 16-byte aligned,
 *                    ld_x % 8 == 0, ld_x >= cols
 *   slices[i].cols   a multiple of 128 (0: the slice is skipped); slice i starts at
 *                    column c_i = cols_0 + ... + cols_(i-1) of the destination
 *   nslices          1 <= nslices <= BQ_MAX_SLICES; the slices array is host memory
 *   q_e4m3, s_e8m0   the destination's first column: [rows][ld_q] and [rows][ld_s]
 *                    (written), as in bq_quant_mx, for the total of the slices'
 *                    columns; offset them for a batch that starts at another
 *                    128-column-aligned column
 * Slices may overlap one another; the outputs may overlap none of them. Errors as
 * bq_quant_mx (every slice is checked before the launch), plus BQ_ERR_SHAPE for nslices
 * outside 1..BQ_MAX_SLICES. The slice list is copied into the launch's parameters:
 * nothing is allocated, and the host array may be reused as soon as the call returns. */
typedef struct bq_mx_slice {
    const void *x;
    int64_t cols;
    int64_t ld_x;
} bq_mx_slice;
#define BQ_MAX_SLICES 16
BQ_API bq_status bq_quant_mx_slices(const bq_mx_slice *slices, int nslices, int x_is_f16, int64_t rows,
                                    uint8_t *q_e4m3, int64_t ld_q, uint8_t *s_e8m0, int64_t ld_s,
                                    cudaStream_t stream);

/* Bytes of the tiled scale layout for rows x g_total scales (rows rounded up to 128);
 * -1 if g_total is not a non-negative multiple of 4. */
BQ_API int64_t bq_mx_tiled_scale_bytes(int64_t rows, int64_t g_total);

/* The i8 mode's BF16 reduce-scatter fused with its INT8 all-gather payload
 * ("feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A", Summary: i8 =
 * BF16 reduce-scatter + INT8 all-gather): per element the W ranks' BF16 values are
 * added in rank order in binary32 and rounded once to BF16; that BF16 shard is
 * quantized as by bq_quant_i8, without writing it to memory.
 *   x_srcs     HOST array of W DEVICE pointers to [n] BF16 (16-byte aligned), rank order
 *   W          1 <= W <= BQ_MAX_W
 *   q, scales  [n] int8 payload, [n/128] FP32 scales (written)
 *   out_bf16   NULL, or [n] BF16 materialization of the payload (the owner's copy).
 * Sources may repeat or overlap one another. */
BQ_API bq_status bq_reduce_quant_i8(const void *const *x_srcs, int W, int64_t n, int8_t *q,
                             float *scales, void *out_bf16, cudaStream_t stream);

/* BF16 -> legacy E4M3 wire (same page, Summary and Why: the E4M3 codec keeps one E4M3
 * byte per value and one FP32 scale per 128 values, 132 bytes per block).
 *   x_bf16 [n] (read), q [n] E4M3 codes (written, 16-byte aligned), scales [n/128]
 *   FP32 (written, 4-byte aligned). */
BQ_API bq_status bq_quant_e4m3(const void *x_bf16, int64_t n, uint8_t *q, float *scales,
                        cudaStream_t stream);

/* Legacy E4M3 wire -> BF16: out = BF16_rne(fl(decode(code) * s)). */
BQ_API bq_status bq_dequant_e4m3(const uint8_t *q, const float *scales, int64_t n, void *out_bf16,
                          cudaStream_t stream);

/* bq_reduce_quant_i8 with the legacy E4M3 codec (the E4M3 all-gather mode). */
BQ_API bq_status bq_reduce_quant_e4m3(const void *const *x_srcs, int W, int64_t n, uint8_t *q,
                               float *scales, void *out_bf16, cudaStream_t stream);

/* Number of bounded waits inside codec kernels on the current device that ran out
 * since the previous call of this function there (the first call counts from library
 * load). Kernels that stage their inputs through shared memory (the bulk-copy ring
 * hops, a build-time alternative; the default kernels load directly and wait on
 * nothing) wait on hardware bulk-copy completions. A wait that has not completed
 * within 1 s is abandoned: that warp stops early (the outputs of the chunks it had not
 * reached are not written) and this count grows by one, instead of the kernel spinning
 * forever. The device-side counters are never reset, so a timeout that happens during
 * this call is reported by the next one, never lost.
 * Synchronizes with the current device (the counters live in device memory).
 *   count  host pointer receiving the number of abandoned waits
 * Returns BQ_ERR_CUDA if a counter cannot be read; nothing is consumed then. */
BQ_API bq_status bq_take_wait_timeouts(int64_t *count);

/* After an abandoned wait the warp gives its copies still in flight time to land, each
 * wait again bounded by 1 s, before its block exits. This is the number of such drain
 * waits that ran out too, since the previous call on the current device: each means a
 * bulk copy may have written that block's shared memory after the block exited. It is
 * 0 unless bq_take_wait_timeouts reported a timeout. Same conventions as
 * bq_take_wait_timeouts. */
BQ_API bq_status bq_take_wait_unlanded(int64_t *count);

/* The debug build (libbq_debug.so, compiled with BQ_DEBUG=1; no counterpart on the
 * pages, it is this library's own bounds checking): every kernel lists the byte ranges
 * of the buffers its arguments describe, inputs read-only and outputs writable, and each
 * global load, store and bulk copy is checked against them. An access outside every
 * listed range (or a store into an input) is not performed, a load yielding zeros, and
 * is counted; nothing traps. bq_take_index_errors returns the growth of that count on
 * the current device since its previous call (always 0 in the default build, whose
 * kernels contain no checks). Same conventions as bq_take_wait_timeouts. */
BQ_API bq_status bq_take_index_errors(int64_t *count);

/* 1 in the debug build, 0 in the default build. */
BQ_API int bq_debug_build(void);

/* Debug build only: one kernel lists the first 256 bytes of buf as its buffer and then
 * loads 16 bytes at byte 512, which the check must decline and count: the next
 * bq_take_index_errors returns 1. buf: device memory of at least 1024 bytes, 16-byte
 * aligned (its first 16 bytes are overwritten with zeros). BQ_ERR_UNSUPPORTED in the
 * default build, which launches nothing. */
BQ_API bq_status bq_selftest_index_check(void *buf, int64_t bytes, cudaStream_t stream);

/* Self-test of the bounded wait: one warp waits on a barrier that nothing completes,
 * with a 20 ms limit, so the count read by bq_take_wait_timeouts grows by exactly one.
 * Enqueued on `stream`; the device stays usable afterwards. */
BQ_API bq_status bq_selftest_wait_timeout(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BQ_H */
