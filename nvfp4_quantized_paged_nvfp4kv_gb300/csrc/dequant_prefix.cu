// Extend path: expand the cached NVFP4 prefix of each sequence into a
// contiguous FP8-E4M3 workspace ("SGLang stores KV cache in 4 bits" (LMSYS
// summary), Interpretation: the extend path dequantises the cached prefix into
// one FP8 workspace shared across layers).
//   out[kv_indptr[b] + j][h][c] = E4M3_rn_satfinite(E2M1(code) x E4M3(scale))
// The product has at most 6 significant bits and lies in [2^-10, 2688], so it
// is exact in fp16; the only rounding is the final one to E4M3.
//
// Work unit: one page-head of K or V (16 tokens x 8 blocks) per 128-thread
// CTA iteration, grid-stride over (sequence, page, kv head, K|V).  Each thread
// gathers the 16 codes and the scale of one (token, block) from the record
// (layout in include/nvfp4kv.h) and writes 16 E4M3 bytes.
#include "device_common.cuh"
#include "nvfp4kv.h"

namespace nvfp4kv {

__global__ void __launch_bounds__(128) dequant_prefix_kernel(const PrefixParams p)
{
    pdl_wait();
    const int tok = threadIdx.x >> 3, blk = threadIdx.x & 7;
    const long long units = static_cast<long long>(p.batch) * p.max_pages * p.hkv * 2;
    const int max_len = p.max_pages * kPageSize;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const int kv = static_cast<int>(u & 1);
        long long r = u >> 1;
        const int h = static_cast<int>(r % p.hkv);
        r /= p.hkv;
        const int pg = static_cast<int>(r % p.max_pages);
        const int b = static_cast<int>(r / p.max_pages);
        int L = __ldg(p.prefix_lens + b);
        if (L < 0 || L > max_len) {
            if (threadIdx.x == 0 && pg == 0 && h == 0 && kv == 0)
                report(p.dev_status, NVFP4KV_DEV_BAD_LEN);
            L = L < 0 ? 0 : max_len;
        }
        if (pg * kPageSize >= L)
            continue;                                   // uniform over the CTA
        const int j = pg * kPageSize + tok;
        if (j >= L)
            continue;
        int phys = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pg);
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_pages)) {
            if (threadIdx.x == 0)
                report(p.dev_status, NVFP4KV_DEV_BAD_PAGE);
            phys = 0;
        }
        const uint8_t *rec = p.pool + (static_cast<size_t>(phys) * p.hkv + h) * kNvfp4Record;
        uint2 packed;
        uint32_t sbyte;
        if (kv == 0) {
            packed = __ldg(reinterpret_cast<const uint2 *>(rec + tok * 64 + blk * 8));
            sbyte = __ldg(rec + 2048 + tok * 8 + blk);
        } else {
            // channel 16*blk + g + 8w: row tok/2, chunk (g + 2*row) mod 8, byte
            // 2*blk + w, nibble tok & 1; repack into natural order
            const int row = tok >> 1, half = tok & 1;
            uint32_t lo = 0u, hi = 0u;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint32_t unit = __ldg(reinterpret_cast<const uint16_t *>(
                    rec + 1024 + row * 128 + ((g + 2 * row) & 7) * 16 + 2 * blk));
                const uint32_t c0 = (unit >> (4 * half)) & 15u;        // channel g
                const uint32_t c1 = (unit >> (8 + 4 * half)) & 15u;    // channel g + 8
                lo |= c0 << (4 * g);
                hi |= c1 << (4 * g);
            }
            packed = make_uint2(lo, hi);
            sbyte = __ldg(rec + 2176 + row * 16 + blk * 2 + half);
        }
        const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));
        uint32_t f[8];
        e2m1x8_to_f16x2x4(packed.x, f[0], f[1], f[2], f[3]);
        e2m1x8_to_f16x2x4(packed.y, f[4], f[5], f[6], f[7]);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = f16x2_to_e4m3x2(hmul2(f[2 * k], s2)) | (f16x2_to_e4m3x2(hmul2(f[2 * k + 1], s2)) << 16);
        const int base = __ldg(p.kv_indptr + b);
        uint8_t *out = kv ? p.v_out : p.k_out;
        const size_t orow = (static_cast<size_t>(base) + j) * p.hkv + h;
        *reinterpret_cast<uint4 *>(out + orow * kHeadDim + blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_dequant_prefix_fp8(const PrefixParams &p, cudaStream_t s)
{
    const long long units = static_cast<long long>(p.batch) * p.max_pages * p.hkv * 2;
    if (units == 0)
        return cudaSuccess;
    const int sms = sm_count();
    long long grid = static_cast<long long>(sms > 0 ? sms : 1) * 16;
    if (grid > units)
        grid = units;
    return launch_pdl(dequant_prefix_kernel, dim3(static_cast<unsigned>(grid)), dim3(128), 0, s, p);
}

} // namespace nvfp4kv
