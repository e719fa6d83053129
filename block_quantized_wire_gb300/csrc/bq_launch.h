// Internal launcher interface between the C ABI (bq_api.cu) and the kernels.
// Arguments are already validated; every launcher only enqueues work on `stream`
// and returns the launch's cudaError_t.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

namespace bqk {

constexpr int kThreads = 256;  // threads per CTA (8 warps) for every codec kernel
constexpr int kMaxSources = 16;

// The sources of a wire reduction: payload pointers and 4-byte scale-word pointers
// (one word per 128-value block), in accumulation order.
template <class TQ, class TS>
struct WireList {
    const TQ *q[kMaxSources];
    const TS *s[kMaxSources];
};
using SourceList = WireList<int8_t, float>;       // block INT8: one FP32 scale per block
using MxSourceList = WireList<uint8_t, uint32_t>;  // MXFP8: four E8M0 bytes per block

// Staged MX slices quantized by one launch: slice i is x[i] [rows, 128 * bpr[i]] with
// leading dimension ld_x[i], written at 128-column block cb0[i] of the destination;
// cta0 is filled by the launcher.
constexpr int kMaxSlices = 16;
struct MxSliceList {
    const uint16_t *x[kMaxSlices];
    int64_t ld_x[kMaxSlices];
    int64_t bpr[kMaxSlices];
    int64_t cb0[kMaxSlices];
    int cta0[kMaxSlices + 1];
    int n;
};

// BF16 shards of the W ranks, in rank order (the reduce of the all-gather modes).
struct Bf16List {
    const uint16_t *x[kMaxSources];
};

cudaError_t launch_quant_i8(const uint16_t *x, int64_t nblk, int8_t *q, float *s, cudaStream_t st);
cudaError_t launch_dequant_i8(const int8_t *q, const float *s, int64_t nblk, uint16_t *out,
                              cudaStream_t st);
cudaError_t launch_accum_i8(const SourceList &src, int W, int64_t nblk, int8_t *q, float *s,
                            uint16_t *out, cudaStream_t st);
cudaError_t launch_ring_hop_i8(const int8_t *q_in, const float *s_in, const uint16_t *x, int64_t nblk,
                               int8_t *q, float *s, uint16_t *out, cudaStream_t st);
cudaError_t launch_quant_mx(const uint16_t *x, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q,
                            int64_t ld_q, uint8_t *s, int64_t ld_s, cudaStream_t st);
cudaError_t launch_dequant_mx(const uint8_t *q, int64_t ld_q, const uint8_t *s, int64_t ld_s,
                              int64_t rows, int64_t cols, uint16_t *out, int64_t ld_out,
                              cudaStream_t st);
cudaError_t launch_accum_mx(const MxSourceList &src, int W, int64_t nblk, uint8_t *q, uint32_t *s,
                            uint16_t *out, cudaStream_t st);
cudaError_t launch_ring_hop_mx(const uint8_t *q_in, const uint32_t *s_in, const uint16_t *x, int64_t nblk,
                               uint8_t *q, uint32_t *s, uint16_t *out, cudaStream_t st);
cudaError_t launch_quant_mx_f16(const uint16_t *x, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q,
                                int64_t ld_q, uint8_t *s, int64_t ld_s, cudaStream_t st);
cudaError_t launch_quant_mx_tiled(const uint16_t *x, bool f16, int64_t ld_x, int64_t rows, int64_t cols, uint8_t *q,
                                  int64_t ld_q, uint8_t *s_tiled, int64_t tiles_per_row, int64_t c0, cudaStream_t st);
cudaError_t launch_quant_mx_slices(MxSliceList sl, bool f16, int64_t rows, uint8_t *q, int64_t ld_q, uint8_t *s,
                                   int64_t ld_s, cudaStream_t st);
cudaError_t launch_reduce_quant_i8(const Bf16List &src, int W, int64_t nblk, int8_t *q, float *s, uint16_t *out,
                                   cudaStream_t st);
cudaError_t launch_quant_e4m3(const uint16_t *x, int64_t nblk, uint8_t *q, float *s, cudaStream_t st);
cudaError_t launch_dequant_e4m3(const uint8_t *q, const float *s, int64_t nblk, uint16_t *out, cudaStream_t st);
cudaError_t launch_reduce_quant_e4m3(const Bf16List &src, int W, int64_t nblk, uint8_t *q, float *s, uint16_t *out,
                                     cudaStream_t st);

// Programmatic dependent launch: every codec kernel is launched with programmatic
// stream serialization and begins with griddepcontrol.wait, which returns once the
// previous grid in the stream has completed and its memory is visible. The kernel then
// allows its own dependents to launch, so the next codec call's launch and CTA
// placement overlap this kernel's tail instead of following it. Ordering against any
// other work is unchanged: a kernel that does not trigger (not one of these) is
// waited for in full.
#ifndef BQ_PDL
#define BQ_PDL 1
#endif

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_block(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t st,
                                Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = BQ_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_smem(void (*kernel)(KArgs...), int grid, size_t smem, cudaStream_t st, Args... args)
{
    return launch_kernel_block(kernel, grid, kThreads, smem, st, args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), int grid, cudaStream_t st, Args... args)
{
    return launch_kernel_smem(kernel, grid, 0, st, args...);
}

// Grid size for a grid-stride kernel over `nchunk` warp chunks with `smem` bytes of
// dynamic shared memory per CTA of `block` threads: enough CTAs to fill every SM of the
// current device at the kernel's occupancy, and no more CTAs than there are chunks. The
// first call for a kernel also raises its dynamic shared memory limit to `smem`. Returns
// the error of the device queries, if any.
cudaError_t grid_for(const void *kernel, int64_t nchunk, int *grid, size_t smem = 0, int block = kThreads);

// Each kernel translation unit's counters {wait timeouts, unlanded copies, debug index errors} (see
// g_wait_timeouts in bq_device.cuh): totals since the library was loaded, never reset.
cudaError_t read_wait_counters_i8(unsigned long long (&v)[3]);
cudaError_t read_wait_counters_mx_wire(unsigned long long (&v)[3]);
cudaError_t read_wait_counters_mx(unsigned long long (&v)[3]);
cudaError_t read_wait_counters_e4m3(unsigned long long (&v)[3]);
cudaError_t launch_wait_selftest(cudaStream_t st);
// Debug build: one listed 256-byte range of buf and one load at byte 512 (declined).
cudaError_t launch_index_selftest(void *buf, cudaStream_t st);

}  // namespace bqk
