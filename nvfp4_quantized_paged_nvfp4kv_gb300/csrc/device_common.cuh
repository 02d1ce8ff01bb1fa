// Device primitives shared by the kernels: mbarriers, bulk / tensor copies,
// format conversions and warp-level MMA, written as inline PTX from the PTX ISA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4kv_internal.h"

namespace nvfp4kv {

constexpr uint32_t kFullMask = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

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

// Wait for phase `parity` of a barrier, giving up after `limit` polls (none
// when limit is 0).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

// Waits (bounded) until the phases with parity pa of barrier a and pb of
// barrier b have completed, polling both in one loop.
__device__ __forceinline__ bool mbar_wait2_bounded(uint32_t a, uint32_t pa, uint32_t b, uint32_t pb, uint32_t limit)
{
    bool da = false, db = false;
    for (uint32_t i = 0; i < limit; ++i) {
        da = da || mbar_try_wait(a, pa);
        db = db || mbar_try_wait(b, pb);
        if (da && db)
            return true;
    }
    return false;
}

// ---- asynchronous copies global -> shared ---------------------------------

// Untiled bulk copy; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}


// ---- conversions --------------------------------------------------------------

// Four bytes, each two E2M1 codes (low nibble -> low half), to four f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
}

// Low 16 bits: two E4M3 bytes (low byte -> low half) to f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t lo16)
{
    uint32_t r;
    uint16_t h = static_cast<uint16_t>(lo16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

// A 32-bit word of four E4M3 bytes to two f16x2 (bytes 0,1 -> r0; 2,3 -> r1).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &r0, uint32_t &r1)
{
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(r0), "=r"(r1)
        : "r"(w));
}

// Two fp32 -> two E4M3 bytes (round to nearest even, saturating); `lo` goes to
// the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// f16x2 -> two E4M3 bytes (low half -> low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h2)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
    return r;
}

// Exact E4M3 byte -> fp32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte)
{
    uint32_t h2 = e4m3x2_to_f16x2(byte & 0xffu);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}

// max of three fp32 (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two fp32 lanes in one 64-bit register (low lane first): packed add, round
// to nearest even in each lane.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi)
{
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Eight fp32 -> one word of four E2M1 code pairs (round to nearest even,
// saturating): byte j holds e[j] in its low nibble and o[j] in its high one.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(float e0, float o0, float e1, float o1, float e2, float o2,
                                                    float e3, float o3)
{
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(e0), "f"(o0), "f"(e1), "f"(o1), "f"(e2), "f"(o2), "f"(e3), "f"(o3));
    return w;
}

__device__ __forceinline__ float f32x2_lo(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v));
}

__device__ __forceinline__ float f32x2_hi(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v >> 32));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ---- warp-level tensor-core MMA -------------------------------------------

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit values held one row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// ---- shared loads ----------------------------------------------------------
//
// Each carries a "memory" clobber: the data they read is written by bulk
// copies, TMA loads or other threads, and the loads must stay between the
// barrier wait that makes it valid and the arrive that releases the buffer
// (the compiler does not know what an asm reads and may otherwise move it
// across either).

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Orders this thread's earlier generic-proxy global writes before its (and,
// after a warp barrier, its warp's) later asynchronous bulk copies.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Orders this thread's shared-memory accesses through the generic proxy with
// the asynchronous proxy's (bulk copies, TMA, the tensor core): writes become
// visible to its reads, reads complete before its later writes.
__device__ __forceinline__ void fence_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: wait for the preceding kernel in the stream
// (no-op when the launch did not allow overlap) / let the next one start.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Tensor scale of kv head h of K or V: its per-head scale when the cache has
// per-head factors, else the uniform one.
__device__ __forceinline__ float head_tensor_scale(const HeadScales &hs, bool is_v, int h, float uniform)
{
    return hs.per_head ? (is_v ? hs.v[h] : hs.k[h]) : uniform;
}

__device__ __forceinline__ void report(int32_t *dev_status, int32_t bits)
{
    if (dev_status != nullptr)
        atomicOr(dev_status, bits);
}

} // namespace nvfp4kv
