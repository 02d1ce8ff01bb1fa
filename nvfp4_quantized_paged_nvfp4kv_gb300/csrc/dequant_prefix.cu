// Extend path: expand the cached NVFP4 prefix of each sequence into a
// contiguous FP8-E4M3 workspace ("SGLang stores KV cache in 4 bits" (LMSYS
// summary), Interpretation: the extend path dequantises the cached prefix into
// one FP8 workspace shared across layers).
//   out[kv_indptr[b] + j][h][c] = E4M3_rn_satfinite(fl32(G x E2M1(code) x E4M3(scale)))
// with G the tensor scale.  The code-scale product has at most 6 significant
// bits and lies in [2^-10, 2688], so it is exact in fp16; at G = 1 the only
// rounding is the final one to E4M3.
//
// Work unit: one page-head record (16 tokens of one kv head, K and V), grid-
// stride over (sequence, page, kv head).  A CTA of 64 threads stages the
// record of its next unit in shared memory with one bulk copy (double
// buffered) while it converts the current one.  Thread t converts K blocks
// (token t/8, block t%8) and (token t/8 + 8, block t%8), and V block t%8 of the
// token pair t/8: a V byte holds one channel of both tokens, so the pair is
// dequantised together (one cvt per channel) and split into the two tokens'
// rows when the E4M3 bytes are packed.
#include "device_common.cuh"
#include "nvfp4kv.h"

namespace nvfp4kv {

namespace {

constexpr int kPrefixThreads = 64;
constexpr int kPrefixCtasPerSm = 24;

struct PrefixUnit {
    int b, pg, h;
    int len, phys, base;
};

// Position (sequence, page, kv head) of unit u; units are numbered with the
// kv head innermost.
struct UnitPos {
    int b, pg, h;
};

__device__ __forceinline__ UnitPos unit_pos(const PrefixParams &p, long long u)
{
    UnitPos x;
    x.h = static_cast<int>(u % p.hkv);
    u /= p.hkv;
    x.pg = static_cast<int>(u % p.max_pages);
    x.b = static_cast<int>(u / p.max_pages);
    return x;
}

// x += d in the same mixed radix (d.h < hkv and d.pg < max_pages, so one
// carry per digit); the grid stride costs no division after the first unit.
__device__ __forceinline__ void advance(UnitPos &x, const UnitPos &d, const PrefixParams &p)
{
    x.h += d.h;
    int c = x.h >= p.hkv;
    x.h -= c ? p.hkv : 0;
    x.pg += d.pg + c;
    c = x.pg >= p.max_pages;
    x.pg -= c ? p.max_pages : 0;
    x.b += d.b + c;
}

__device__ __forceinline__ PrefixUnit prefix_unit(const PrefixParams &p, const UnitPos &x)
{
    PrefixUnit t;
    t.h = x.h;
    t.pg = x.pg;
    t.b = x.b;
    t.len = __ldg(p.prefix_lens + t.b);
    t.phys = __ldg(p.block_table + static_cast<size_t>(t.b) * p.max_pages + t.pg);
    t.base = __ldg(p.kv_indptr + t.b);
    return t;
}

// E4M3 bytes of the exact products in an f16x2 times the tensor scale G:
// E4M3_rn_satfinite(fl32(G * v)), which at G = 1 is the f16 conversion itself.
__device__ __forceinline__ uint32_t to_e4m3x2(uint32_t h2, float G)
{
    if (G == 1.f)
        return f16x2_to_e4m3x2(h2);
    const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
    const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
    return f32x2_to_e4m3x2(__fmul_rn(lo, G), __fmul_rn(hi, G));
}

// Four E4M3 bytes from two f16x2 (low halves first).
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t h2a, uint32_t h2b, float G)
{
    return to_e4m3x2(h2a, G) | (to_e4m3x2(h2b, G) << 16);
}

} // namespace

__global__ void __launch_bounds__(kPrefixThreads) dequant_prefix_kernel(const __grid_constant__ PrefixParams p)
{
    __shared__ __align__(128) uint8_t buf[2][kNvfp4Record];
    __shared__ __align__(8) uint64_t bars[2];
    const int t = threadIdx.x;
    const int row = t >> 3, blk = t & 7;
    const long long units = static_cast<long long>(p.batch) * p.max_pages * p.hkv;
    const int max_len = p.max_pages * kPageSize;
    const uint32_t bar0 = smem_addr(&bars[0]);
    if (t == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();                  // the records may come from the previous kernel

    // Length of the unit's sequence (clamped, reported) and whether its page
    // holds any prefix token; issues the unit's copy into buffer k if so.
    auto stage = [&](const PrefixUnit &x, int k, int &L) {
        L = x.len;
        if (L < 0 || L > max_len) {
            if (t == 0 && x.pg == 0 && x.h == 0)
                report(p.dev_status, NVFP4KV_DEV_BAD_LEN);
            L = L < 0 ? 0 : max_len;
        }
        if (x.pg * kPageSize >= L)
            return false;
        int phys = x.phys;
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_pages)) {
            if (t == 0)
                report(p.dev_status, NVFP4KV_DEV_BAD_PAGE);
            phys = 0;
        }
        if (t == 0) {
            const uint32_t bar = bar0 + 8 * k;
            mbar_arrive_expect_tx(bar, kNvfp4Record);
            bulk_g2s(smem_addr(buf[k]), p.pool + (static_cast<size_t>(phys) * p.hkv + x.h) * kNvfp4Record,
                     kNvfp4Record, bar);
        }
        return true;
    };

    long long u = blockIdx.x;
    if (u >= units)
        return;
    UnitPos pos = unit_pos(p, u);
    const UnitPos stride = unit_pos(p, gridDim.x);
    PrefixUnit cur = prefix_unit(p, pos);
    int L = 0;
    bool staged = stage(cur, 0, L);
    uint32_t parity = 0u;        // bit k: phase parity of buffer k's barrier
    int k = 0;
    for (; u < units; u += gridDim.x) {
        const long long un = u + gridDim.x;
        PrefixUnit nxt{};
        int Ln = 0;
        bool staged_n = false;
        if (un < units) {
            advance(pos, stride, p);
            nxt = prefix_unit(p, pos);
            staged_n = stage(nxt, k ^ 1, Ln);
        }
        if (staged) {
            const bool arrived = mbar_wait_bounded(bar0 + 8 * k, (parity >> k) & 1u, p.wait_limit);
            if (!__syncthreads_and(arrived)) {
                // staged data never arrived: report, let both copies in flight
                // (this unit's and the next one's) land at the default limit, stop
                if (t == 0)
                    report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
                mbar_wait_bounded(bar0 + 8 * k, (parity >> k) & 1u, kWaitLimit);
                if (staged_n)
                    mbar_wait_bounded(bar0 + 8 * (k ^ 1), (parity >> (k ^ 1)) & 1u, kWaitLimit);
                return;
            }
            parity ^= 1u << k;
            const uint32_t rec = smem_addr(buf[k]);
            const int j0 = cur.pg * kPageSize;
            const size_t rows = static_cast<size_t>(cur.base) + j0;     // output row of token 0
            // K: tokens row and row + 8, block blk (natural rows)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int tok = row + 8 * half;
                if (j0 + tok < L) {
                    const uint2 packed = lds64(rec + tok * 64 + blk * 8);
                    const uint32_t sb = lds_u8(rec + 2048 + tok * 8 + blk);
                    const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
                    uint32_t f[8];
                    e2m1x8_to_f16x2x4(packed.x, f[0], f[1], f[2], f[3]);
                    e2m1x8_to_f16x2x4(packed.y, f[4], f[5], f[6], f[7]);
                    const size_t o = ((rows + tok) * p.hkv + cur.h) * kHeadDim + blk * 16;
                    const float G = head_tensor_scale(p.hs, false, cur.h, p.gscale);
                    *reinterpret_cast<uint4 *>(p.k_out + o) = make_uint4(
                        e4m3_pair(hmul2(f[0], s2), hmul2(f[1], s2), G), e4m3_pair(hmul2(f[2], s2), hmul2(f[3], s2), G),
                        e4m3_pair(hmul2(f[4], s2), hmul2(f[5], s2), G), e4m3_pair(hmul2(f[6], s2), hmul2(f[7], s2), G));
                }
            }
            // V: tokens 2*row (low nibbles) and 2*row + 1 (high nibbles), block blk.
            // Unit g (bytes 2*blk, 2*blk + 1 of group g's chunk) holds channels
            // 16*blk + g and 16*blk + g + 8 of both tokens.
            const int t0 = 2 * row;
            if (j0 + t0 < L) {
                uint32_t unitw[4];   // units (g, g + 1) for g = 0, 2, 4, 6
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int g = 2 * q;
                    const uint32_t a = lds_u16(rec + 1024 + row * 128 + ((g + 2 * row) & 7) * 16 + 2 * blk);
                    const uint32_t c = lds_u16(rec + 1024 + row * 128 + ((g + 1 + 2 * row) & 7) * 16 + 2 * blk);
                    unitw[q] = a | (c << 16);
                }
                const uint32_t s2 = e4m3x2_to_f16x2(lds_u16(rec + 2176 + row * 16 + blk * 2));   // (s_t0, s_t1)
                // e8[r]: E4M3 bytes of channel 16*blk + r, low byte token t0, high byte t0 + 1
                uint32_t e8[16];
                const float Gv = head_tensor_scale(p.hs, true, cur.h, p.gscale);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t f0, f1, f2, f3;   // channels g, g + 8, g + 1, g + 9 (g = 2q), tokens (t0, t0 + 1)
                    e2m1x8_to_f16x2x4(unitw[q], f0, f1, f2, f3);
                    e8[2 * q] = to_e4m3x2(hmul2(f0, s2), Gv);
                    e8[2 * q + 8] = to_e4m3x2(hmul2(f1, s2), Gv);
                    e8[2 * q + 1] = to_e4m3x2(hmul2(f2, s2), Gv);
                    e8[2 * q + 9] = to_e4m3x2(hmul2(f3, s2), Gv);
                }
                uint32_t w0[4], w1[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t lo = e8[4 * q] | (e8[4 * q + 1] << 16);
                    const uint32_t hi = e8[4 * q + 2] | (e8[4 * q + 3] << 16);
                    w0[q] = __byte_perm(lo, hi, 0x6420);   // token t0: the low bytes
                    w1[q] = __byte_perm(lo, hi, 0x7531);   // token t0 + 1: the high bytes
                }
                const size_t o0 = ((rows + t0) * p.hkv + cur.h) * kHeadDim + blk * 16;
                *reinterpret_cast<uint4 *>(p.v_out + o0) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
                if (j0 + t0 + 1 < L) {
                    const size_t o1 = ((rows + t0 + 1) * p.hkv + cur.h) * kHeadDim + blk * 16;
                    *reinterpret_cast<uint4 *>(p.v_out + o1) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                }
            }
        }
        __syncthreads();         // buffer k is free for the unit after next
        cur = nxt;
        L = Ln;
        staged = staged_n;
        k ^= 1;
    }
}

cudaError_t launch_dequant_prefix_fp8(const PrefixParams &p, cudaStream_t s)
{
    const long long units = static_cast<long long>(p.batch) * p.max_pages * p.hkv;
    if (units == 0)
        return cudaSuccess;
    const int sms = sm_count();
    long long grid = static_cast<long long>(sms > 0 ? sms : 1) * kPrefixCtasPerSm;
    if (grid > units)
        grid = units;
    return launch_pdl(dequant_prefix_kernel, dim3(static_cast<unsigned>(grid)), dim3(kPrefixThreads), 0, s, p);
}

} // namespace nvfp4kv
