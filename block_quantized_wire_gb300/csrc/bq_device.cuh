// Device-side building blocks shared by the codec kernels (sm_103a).
//
// Work decomposition used by every kernel: a warp owns a "chunk" of kChunkBlocks
// 128-value blocks per loop iteration. The chunk is read as kSegs warp-wide
// "segments" of 256 values: in segment j, half-warp h (lanes 16h..16h+15) holds
// block 2j+h of the chunk, each lane 8 consecutive values. So every warp-wide access
// is one contiguous run (512 B of BF16, 256 B of INT8/E4M3), block amax is a
// 16-lane shuffle reduction (4 lanes for a 32-value MX group), and the chunk's
// kChunkBlocks scales are written by lanes 0..kChunkBlocks-1 in one coalesced store.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "bq_launch.h"

namespace bqk {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kSegs = 4;                      // segments per warp iteration
constexpr int kChunkBlocks = 2 * kSegs;       // 128-value blocks per warp iteration

// ---------------------------------------------------------------- debug build
// With -DBQ_DEBUG=1 (libbq_debug.so) every global access of a codec kernel is checked
// against the buffers the kernel was given. At entry each kernel lists its buffers' byte
// ranges from its own arguments (inputs read-only, outputs writable); a load, store or
// bulk copy whose bytes do not lie inside one listed range of the right kind is not
// performed (a load yields zeros) and is counted in g_index_errors, which the host reads
// through bq_take_index_errors. Nothing traps. In the default build the checks are the
// constant true and the listing is empty, so the kernels' code is unchanged.
#ifndef BQ_DEBUG
#define BQ_DEBUG 0
#endif
static __device__ unsigned long long g_index_errors;
constexpr int kDbgMaxRanges = 2 * kMaxSources + 8;

#if BQ_DEBUG
struct DbgRanges {
    unsigned long long lo[kDbgMaxRanges], hi[kDbgMaxRanges], writable;
    int n;
};
__device__ __forceinline__ DbgRanges &dbg_ranges()
{
    __shared__ DbgRanges r;
    return r;
}
#endif

// Start of a kernel's buffer list (every thread calls it).
__device__ __forceinline__ void dbg_begin()
{
#if BQ_DEBUG
    if (threadIdx.x == 0) {
        dbg_ranges().n = 0;
        dbg_ranges().writable = 0;
    }
#endif
}

// One buffer of `bytes` bytes at p (thread 0 records it; the others ignore the call).
__device__ __forceinline__ void dbg_allow(const void *p, int64_t bytes, bool writable)
{
#if BQ_DEBUG
    DbgRanges &r = dbg_ranges();
    if (threadIdx.x == 0 && bytes > 0 && r.n < kDbgMaxRanges) {
        r.lo[r.n] = reinterpret_cast<unsigned long long>(p);
        r.hi[r.n] = r.lo[r.n] + static_cast<unsigned long long>(bytes);
        if (writable) r.writable |= 1ull << r.n;
        r.n++;
    }
#else
    (void)p, (void)bytes, (void)writable;
#endif
}

// A row-major strided buffer: rows of row_bytes, ld_bytes apart.
__device__ __forceinline__ void dbg_allow_2d(const void *p, int64_t rows, int64_t row_bytes, int64_t ld_bytes,
                                             bool writable)
{
    if (rows > 0) dbg_allow(p, (rows - 1) * ld_bytes + row_bytes, writable);
}

// End of the list: the ranges are visible to every thread of the CTA.
__device__ __forceinline__ void dbg_ready()
{
#if BQ_DEBUG
    __syncthreads();
#endif
}

// True if [p, p + bytes) lies inside one listed range (a writable one for a store).
__device__ __forceinline__ bool dbg_ok(const void *p, int64_t bytes, bool write)
{
#if BQ_DEBUG
    const unsigned long long a = reinterpret_cast<unsigned long long>(p), b = a + static_cast<unsigned long long>(bytes);
    const DbgRanges &r = dbg_ranges();
    for (int i = 0; i < r.n; i++)
        if (a >= r.lo[i] && b <= r.hi[i] && (!write || ((r.writable >> i) & 1ull))) return true;
    atomicAdd(&g_index_errors, 1ull);
    return false;
#else
    (void)p, (void)bytes, (void)write;
    return true;
#endif
}

// Listing helpers. A flat wire of 128 * nblk values: the payload (128 bytes per block)
// and the scale words (4 bytes per block); a BF16 tensor of 128 * nblk values.
__device__ __forceinline__ void dbg_wire(const void *q, const void *s, int64_t nblk, bool writable)
{
    dbg_allow(q, 128 * nblk, writable);
    dbg_allow(s, 4 * nblk, writable);
}

__device__ __forceinline__ void dbg_bf16(const void *x, int64_t nblk, bool writable)
{
    dbg_allow(x, 256 * nblk, writable);
}

template <class TQ, class TS>
__device__ __forceinline__ void dbg_sources(const WireList<TQ, TS> &src, int nsrc, int64_t nblk)
{
    for (int i = 0; i < nsrc && i < kMaxSources; i++) dbg_wire(src.q[i], src.s[i], nblk, false);
}

__device__ __forceinline__ void dbg_sources(const Bf16List &src, int nsrc, int64_t nblk)
{
    for (int i = 0; i < nsrc && i < kMaxSources; i++) dbg_bf16(src.x[i], nblk, false);
}

// ---------------------------------------------------------------- launch ordering
// First statement of every codec kernel (see launch_kernel in bq_launch.h): wait for
// the previous grid's completion and memory, then let the next grid start launching.
__device__ __forceinline__ void pdl_begin()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- bulk-copy staging
// Global -> shared bulk copies (cp.async.bulk, completed on an mbarrier by byte
// count). Every wait on a barrier is bounded in time: a wait that runs out is counted
// in g_wait_timeouts and the kernel stops early instead of spinning forever. A warp
// that gave up then waits, again bounded, for its copies still in flight; if one of
// those waits runs out too, g_wait_unlanded counts it (that block's shared memory may
// still be written by a copy after the block has exited). Both counters only grow; the
// host reports their growth since its previous read (bq_take_wait_timeouts,
// bq_take_wait_unlanded), so no count is lost between a read and a reset.
static __device__ unsigned long long g_wait_timeouts;
static __device__ unsigned long long g_wait_unlanded;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// Host side: this translation unit's counters, {timeouts, unlanded, index errors}.
static inline cudaError_t read_wait_counters(unsigned long long (&v)[3])
{
    if (cudaError_t e = cudaMemcpyFromSymbol(&v[0], g_wait_timeouts, sizeof v[0])) return e;
    if (cudaError_t e = cudaMemcpyFromSymbol(&v[1], g_wait_unlanded, sizeof v[1])) return e;
    return cudaMemcpyFromSymbol(&v[2], g_index_errors, sizeof v[2]);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    if (!dbg_ok(src, bytes, false)) return;  // the stage's barrier then runs out of time, counted too
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Orders this thread's (and, after __syncwarp, its warp's) generic shared-memory
// accesses before a following bulk copy into the same bytes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// True once the barrier's phase with the given parity has completed; false if that
// did not happen within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// ---------------------------------------------------------------- per-lane async copies
// Global -> shared copies issued by each lane for its own bytes (cp.async, 16 or 4
// bytes, bypassing L1 for 16), grouped per thread with commit_group and completed with
// wait_group. A lane reads back only bytes it copied itself, so wait_group alone makes
// them visible to it: no barrier, no mbarrier, no cross-lane synchronization. The wait
// is for this thread's own copies of valid addresses, which complete like loads.
// Both addresses aligned to the copy size.
__device__ __forceinline__ void lane_copy16(uint32_t dst, const void *src)
{
    if (!dbg_ok(src, 16, false)) return;  // the slot keeps stale bytes; counted in debug builds
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void lane_copy4(uint32_t dst, const void *src)
{
    if (!dbg_ok(src, 4, false)) return;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void lane_copy_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Returns once at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void lane_copy_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- global memory
// Inputs are read once: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    if (!dbg_ok(p, 16, false)) return make_uint4(0, 0, 0, 0);
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void *p)
{
    if (!dbg_ok(p, 8, false)) return make_uint2(0, 0);
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// 32 bytes per lane in one 256-bit access: a warp reads or writes 1 KB of whole
// sectors. The address must be 32-byte aligned; callers check the base pointer on the
// host and take 16-byte accesses otherwise.
__device__ __forceinline__ void ld_stream_v8(const void *p, uint4 &a, uint4 &b)
{
    if (!dbg_ok(p, 32, false)) {
        a = b = make_uint4(0, 0, 0, 0);
        return;
    }
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
        : "l"(p));
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p)
{
    if (!dbg_ok(p, 4, false)) return 0u;
    uint32_t r;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    if (!dbg_ok(p, 16, true)) return;
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v8(void *p, uint4 a, uint4 b)
{
    if (!dbg_ok(p, 32, true)) return;
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
                 "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint2 v)
{
    if (!dbg_ok(p, 8, true)) return;
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_u32(void *p, uint32_t v)
{
    if (!dbg_ok(p, 4, true)) return;
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- packed binary32 pairs
// A lane's eight values are held as four float2 pairs (values 2i, 2i+1) so that the
// FP32 arithmetic runs on the paired IEEE instructions of sm_100-class GPUs: each of
// add2/mul2/fma2 is two independent binary32 operations rounded to nearest even (no
// flush to zero), bit-identical to two scalar __fadd_rn/__fmul_rn/__fmaf_rn, at one
// issue slot. They are written as PTX with an explicit .rn so that no multiply is ever
// fused with a following add: the codec's definitions round every product and every
// sum separately.
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 splat(float x) { return make_float2(x, x); }

// Products that feed a sum (accumulate, ring hop) must round on their own, but the
// compiler was observed to fuse a paired multiply with a following paired add into one
// fused multiply-add, explicit .rn and --fmad=false notwithstanding (the fused result
// showed up in about 13% of random operands). A paired FMA with a +0 addend rounds the
// product exactly as a multiply does, and it cannot be rewritten into a multiply (it
// turns a -0 product into +0), so nothing can fuse it with the add that follows. The
// sign of a zero product never reaches an output here: it only feeds amax and the
// rounding of a value whose payload is 0.
__device__ __forceinline__ float2 mul2_unfused(float2 a, float2 b) { return fma2(a, b, splat(0.0f)); }

// ---------------------------------------------------------------- number formats
// Eight BF16 values (one 16-byte word) widened exactly to binary32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float2 (&v)[4])
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) v[i] = make_float2(__uint_as_float(u[i] << 16), __uint_as_float(u[i] & 0xffff0000u));
}

// Two binary32 values rounded to nearest-even BF16, packed (x in bits 0..15).
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float2 v)
{
    __nv_bfloat162 h = __float22bfloat162_rn(v);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Eight FP16 values (one 16-byte load) -> binary32, exact.
__device__ __forceinline__ void f16x8_to_f32(const uint4 w, float2 (&v)[4])
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&u[i]);
        v[i] = __half22float2(h);
    }
}

// The values of a warp chunk as a requantization reads them: seg(j, v) gives this
// lane's eight values of segment j. RegVals holds FP32 values in registers (the sums of
// the reductions). Bf16Vals holds the raw BF16 words of a quantize and widens them on
// every read: a few integer operations per read instead of 16 registers per 4 segments.
template <int SEGS>
struct RegVals {
    const float2 (&v)[SEGS][4];
    __device__ __forceinline__ void seg(int j, float2 (&o)[4]) const
    {
#pragma unroll
        for (int e = 0; e < 4; e++) o[e] = v[j][e];
    }
};

template <int SEGS>
struct Bf16Vals {
    const uint4 (&x)[SEGS];
    // volatile: each read widens anew, so the compiler cannot keep the first widening
    // alive in place of the raw words
    __device__ __forceinline__ void seg(int j, float2 (&o)[4]) const
    {
        const uint32_t u[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t lo, hi;
            asm volatile("shl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;" : "=r"(lo), "=r"(hi) : "r"(u[i]));
            o[i] = make_float2(__uint_as_float(lo), __uint_as_float(hi));
        }
    }
};

__device__ __forceinline__ uint4 f32x8_to_bf16x8(const float2 (&v)[4])
{
    return make_uint4(f32x2_to_bf16x2(v[0]), f32x2_to_bf16x2(v[1]), f32x2_to_bf16x2(v[2]), f32x2_to_bf16x2(v[3]));
}

// Low bytes of four 32-bit words, packed little-endian into one word.
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Four signed payload bytes (one word) -> their exact binary32 values. Each byte,
// offset by 128, is placed in the low mantissa bits of 2^23 and the offset removed:
// (2^23 + q + 128) - (2^23 + 128) = q exactly; q = 0 gives +0.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float2 &lo, float2 &hi)
{
    const float2 nbias = splat(-8388736.0f);  // -(2^23 + 128)
    const uint32_t u = w ^ 0x80808080u;
    lo = add2(make_float2(__uint_as_float(__byte_perm(u, 0x4b000000u, 0x7540)),
                          __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7541))), nbias);
    hi = add2(make_float2(__uint_as_float(__byte_perm(u, 0x4b000000u, 0x7542)),
                          __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7543))), nbias);
}

__device__ __forceinline__ void i8x8_to_f32(uint2 w, float2 (&v)[4])
{
    i8x4_to_f32(w.x, v[0], v[1]);
    i8x4_to_f32(w.y, v[2], v[3]);
}

// ---------------------------------------------------------------- block INT8 scale
// Per block: s = fl(amax / 127) (IEEE division), r = fl(1 / s) (IEEE reciprocal) and
// rl = fl(fl(1 - s * r) * r), so that r + rl = (1/s)(1 + O(2^-47)). A block with
// s < 2^-100 (amax below about 1e-28: tiny FP32 sums or tiny BF16 inputs) is flagged
// by r = -1 and quantized with the IEEE division x / s, because there the remainder
// of i8_quotient could fall into the subnormal range and lose bits; s == 0 gives
// r = rl = 0, for which the quotient below is 0 and the payload 0.
constexpr float kQuotientMinScale = 7.88860905e-31f;  // 2^-100

struct I8Scale {
    float s, r, rl;
};

__device__ __forceinline__ I8Scale i8_block_scale(float amax)
{
    I8Scale b;
    b.s = __fdiv_rn(amax, 127.0f);
    if (b.s >= kQuotientMinScale) {
        b.r = __frcp_rn(b.s);
        b.rl = __fmul_rn(__fmaf_rn(-b.s, b.r, 1.0f), b.r);
    } else {
        b.r = b.s > 0.0f ? -1.0f : 0.0f;
        b.rl = 0.0f;
    }
    return b;
}

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// fl(x / s) for s >= 2^-100, two values at a time, by Markstein's correction (P. W.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990): when q is within one ulp of x/s and
// r = fl(1/s), the remainder x - q*s is exact (one FMA) and fl(q + (x - q*s) * r) is
// the correctly rounded quotient. Here q = fl(x * r + fl(x * rl)) is within 1/2 ulp +
// 2^-46 relative of x/s because r + rl approximates 1/s to about 2^-47. |x / s| <=
// 127.0001, so nothing overflows; with s >= 2^-100 the remainder of a quotient >= 1/4
// is a multiple of ulp(q) * ulp(s) >= 2^-149 and so representable even when
// subnormal, and quotients below 1/4 round to payload 0 whatever their last bits.
__device__ __forceinline__ float2 i8_quotient2(float2 x, float2 r, float2 rl, float2 neg_s)
{
    const float2 q = fma2(x, r, mul2(x, rl));
    return fma2(fma2(q, neg_s, x), r, q);
}

// Quantize eight values of one block. Returns, per value, the binary32 word M + k
// (M = 1.5 * 2^23, k the payload integer): adding M to the quotient rounds it to the
// nearest integer, ties to even, and leaves k in the low mantissa bits, so the word's
// low byte is k in two's complement and k = word - M exactly. |fl(x/s)| <=
// fl(amax/s) < 127.5, so no clamp is needed there; the flagged path clamps to
// [-127, 127].
// The reciprocal path alone, for a block whose scale is known to be >= 2^-100 or 0.
__device__ __forceinline__ void i8_quant8_fast(const float2 (&v)[4], const I8Scale &b, uint32_t (&w)[8])
{
    const float2 r = splat(b.r), rl = splat(b.rl), ns = splat(-b.s), m = splat(kMagic);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 y = add2(i8_quotient2(v[i], r, rl, ns), m);
        w[2 * i] = __float_as_uint(y.x);
        w[2 * i + 1] = __float_as_uint(y.y);
    }
}

__device__ __forceinline__ void i8_quant8(const float2 (&v)[4], const I8Scale &b, uint32_t (&w)[8])
{
    if (__builtin_expect(b.r >= 0.0f, 1)) {
        i8_quant8_fast(v, b, w);
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float x = (i & 1) ? v[i >> 1].y : v[i >> 1].x;
            const float k = fminf(fmaxf(rintf(__fdiv_rn(x, b.s)), -127.0f), 127.0f);
            w[i] = __float_as_uint(__fadd_rn(k, kMagic));
        }
    }
}

__device__ __forceinline__ uint2 pack_payload8(const uint32_t (&w)[8])
{
    return make_uint2(pack_low_bytes(w[0], w[1], w[2], w[3]), pack_low_bytes(w[4], w[5], w[6], w[7]));
}

__device__ __forceinline__ float amax8(const float2 (&v)[4])
{
    float m = fmaxf(fabsf(v[0].x), fabsf(v[0].y));
#pragma unroll
    for (int i = 1; i < 4; i++) m = fmaxf(m, fmaxf(fabsf(v[i].x), fabsf(v[i].y)));
    return m;
}

// max(a, b, c) in one instruction (three-input max of sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

#ifndef BQ_MAX3
#define BQ_MAX3 1
#endif
// max |x| over a lane's 16 values (a: values 0..7, b: values 8..15)
__device__ __forceinline__ float amax16(const float2 (&a)[4], const float2 (&b)[4])
{
    if (!BQ_MAX3) return fmaxf(amax8(a), amax8(b));
    const float m0 = max3f(fabsf(a[0].x), fabsf(a[0].y), fabsf(a[1].x));
    const float m1 = max3f(fabsf(a[1].y), fabsf(a[2].x), fabsf(a[2].y));
    const float m2 = max3f(fabsf(a[3].x), fabsf(a[3].y), fabsf(b[0].x));
    const float m3 = max3f(fabsf(b[0].y), fabsf(b[1].x), fabsf(b[1].y));
    const float m4 = max3f(fabsf(b[2].x), fabsf(b[2].y), fabsf(b[3].x));
    return fmaxf(max3f(m0, m1, m2), max3f(m3, m4, fabsf(b[3].y)));
}

// max over the 16 lanes of a half-warp (xor partners stay inside the half)
__device__ __forceinline__ float halfwarp_max(float m)
{
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
    return m;
}

// BF16 of fl(k * s) for the eight payload integers held as words M + k.
__device__ __forceinline__ uint4 i8_materialize_words(const uint32_t (&w)[8], float s)
{
    const float2 nm = splat(-kMagic), s2 = splat(s);
    float2 d[4];
#pragma unroll
    for (int i = 0; i < 4; i++)
        d[i] = mul2(add2(make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1])), nm), s2);
    return f32x8_to_bf16x8(d);
}

// BF16 of fl(q * s) for eight payload integers held as binary32.
__device__ __forceinline__ uint4 i8_materialize8(const float2 (&qf)[4], float s)
{
    const float2 s2 = splat(s);
    float2 d[4];
#pragma unroll
    for (int i = 0; i < 4; i++) d[i] = mul2(qf[i], s2);
    return f32x8_to_bf16x8(d);
}

// ---------------------------------------------------------------- MXFP8
// E8M0 byte for a group: 127 for amax == 0, else the smallest e in [0, 254] with
// 2^(e-127) >= v = fl(amax / 448). From v's binary32 fields: a normal v with exponent
// field E is 2^(E-127) when its fraction is zero (e = E) and lies strictly between
// 2^(E-127) and 2^(E-126) otherwise (e = E + 1); a subnormal v is at most 2^-127
// (e = 0) when its fraction field is <= 2^22, else in (2^-127, 2^-126) (e = 1).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax)
{
    if (amax == 0.0f) return 127u;
    const uint32_t u = __float_as_uint(__fdiv_rn(amax, 448.0f));
    const uint32_t ex = u >> 23;
    const uint32_t fr = u & 0x7fffffu;
    uint32_t e = (ex == 0u) ? (fr > 0x400000u ? 1u : 0u) : ex + (fr != 0u ? 1u : 0u);
    return e > 254u ? 254u : e;
}

// 2^k as binary32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float exp2i(int k)
{
    return k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// Eight binary32 values -> eight E4M3 codes (nearest even, saturating), value i in
// byte i.
__device__ __forceinline__ uint2 f32x8_to_e4m3x8(const float2 (&y)[4])
{
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; i++) h[i] = __nv_cvt_float2_to_fp8x2(y[i], __NV_SATFINITE, __NV_E4M3);
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// Eight E4M3 codes -> binary32 fl(decode(code) * p); the decode is exact, and so is
// the product when p is a power of two.
__device__ __forceinline__ void e4m3x8_to_f32(uint2 w, float p, float2 (&v)[4])
{
    const float2 p2 = splat(p);
    const uint32_t u[2] = {w.x, w.y};
#pragma unroll
    for (int j = 0; j < 2; j++) {
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const __nv_fp8x2_storage_t c = static_cast<__nv_fp8x2_storage_t>((u[j] >> (16 * i)) & 0xffffu);
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
            const __half2 hh = *reinterpret_cast<const __half2 *>(&hr);
            v[2 * j + i] = mul2(__half22float2(hh), p2);
        }
    }
}

// ---------------------------------------------------------------- legacy E4M3 codec
// One FP32 scale s = fl(amax / 448) per 128-value block; code = E4M3 (nearest even,
// saturating, sign of zero kept) of fl(x / s). The quotient uses the same Markstein
// form as block INT8. Its remainder is exact when ulp(q) * ulp(s) >= 2^-149, i.e. when
// the exponents of q and s sum to at least -103. With s >= 2^-90 that holds for every
// quotient >= 2^-13, and smaller quotients round to E4M3 zero whatever their last bits.
// Blocks with a smaller nonzero scale divide per element.
constexpr float kE4m3QuotientMinScale = 8.07793567e-28f;  // 2^-90

__device__ __forceinline__ I8Scale e4m3_block_scale(float amax)
{
    I8Scale b;
    b.s = __fdiv_rn(amax, 448.0f);
    if (b.s >= kE4m3QuotientMinScale) {
        b.r = __frcp_rn(b.s);
        b.rl = __fmul_rn(__fmaf_rn(-b.s, b.r, 1.0f), b.r);
    } else {
        b.r = b.s > 0.0f ? -1.0f : 0.0f;  // -1: divide per element; 0: zero block
        b.rl = 0.0f;
    }
    return b;
}

// |t| with the sign of x: the correction step turns x = -0 into +0, and the sign of
// every other quotient already equals the sign of x (s > 0).
__device__ __forceinline__ float2 with_sign_of(float2 t, float2 x)
{
    return make_float2(__uint_as_float((__float_as_uint(t.x) & 0x7fffffffu) | (__float_as_uint(x.x) & 0x80000000u)),
                       __uint_as_float((__float_as_uint(t.y) & 0x7fffffffu) | (__float_as_uint(x.y) & 0x80000000u)));
}

// BF16 of fl(decode(code) * s) for eight codes of one block.
__device__ __forceinline__ uint4 e4m3_materialize8(uint2 codes, float s)
{
    float2 d[4];
    e4m3x8_to_f32(codes, s, d);
    return f32x8_to_bf16x8(d);
}

// Eight values of one block -> eight E4M3 codes (value i in byte i).
__device__ __forceinline__ uint2 e4m3_quant8(const float2 (&v)[4], const I8Scale &b)
{
    float2 t[4];
    if (__builtin_expect(b.r > 0.0f, 1)) {
        const float2 r = splat(b.r), rl = splat(b.rl), ns = splat(-b.s);
#pragma unroll
        for (int i = 0; i < 4; i++) t[i] = with_sign_of(i8_quotient2(v[i], r, rl, ns), v[i]);
    } else if (b.r < 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; i++) t[i] = make_float2(__fdiv_rn(v[i].x, b.s), __fdiv_rn(v[i].y, b.s));
    } else {
        return make_uint2(0u, 0u);  // zero block: every code 0x00
    }
    return f32x8_to_e4m3x8(t);
}

}  // namespace bqk
