// Extend path: expand the cached NVFP4 prefix of each sequence into a
// contiguous FP8-E4M3 workspace ("SGLang stores KV cache in 4 bits" (LMSYS
// summary), Interpretation: the extend path dequantises the cached prefix into
// one FP8 workspace shared across layers).
//   out[kv_indptr[b] + j][h][c] = E4M3_rn_satfinite(E2M1(code) x E4M3(scale))
// The product has at most 6 significant bits and lies in [2^-10, 2688], so it
// is exact in fp16; the only rounding is the final one to E4M3.
//
// Work unit: one page-head (16 tokens x 8 blocks of K and of V) per 128-thread
// CTA iteration, grid-stride over (sequence, page, kv head).  Thread (token,
// block) gathers the 16 K codes and the 16 V codes of its (token, block) from
// the record (layout in include/nvfp4kv.h) with independent loads, and writes
// 16 E4M3 bytes to each workspace.  The unit's length, block-table entry and
// output offset are read together, and those of the CTA's next unit are
// fetched while the current one is being converted.
#include "device_common.cuh"
#include "nvfp4kv.h"

namespace nvfp4kv {

namespace {

struct PrefixUnit {
    int b, pg, h;
    int len, phys, base;
};

__device__ __forceinline__ PrefixUnit prefix_unit(const PrefixParams &p, long long u)
{
    PrefixUnit t;
    long long r = u;
    t.h = static_cast<int>(r % p.hkv);
    r /= p.hkv;
    t.pg = static_cast<int>(r % p.max_pages);
    t.b = static_cast<int>(r / p.max_pages);
    t.len = __ldg(p.prefix_lens + t.b);
    t.phys = __ldg(p.block_table + static_cast<size_t>(t.b) * p.max_pages + t.pg);
    t.base = __ldg(p.kv_indptr + t.b);
    return t;
}

// 16 E2M1 codes (natural channel order) x scale -> 16 E4M3 bytes
__device__ __forceinline__ uint4 codes_to_e4m3(uint2 packed, uint32_t sbyte)
{
    const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));
    uint32_t f[8];
    e2m1x8_to_f16x2x4(packed.x, f[0], f[1], f[2], f[3]);
    e2m1x8_to_f16x2x4(packed.y, f[4], f[5], f[6], f[7]);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = f16x2_to_e4m3x2(hmul2(f[2 * k], s2)) | (f16x2_to_e4m3x2(hmul2(f[2 * k + 1], s2)) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

} // namespace

__global__ void __launch_bounds__(128) dequant_prefix_kernel(const PrefixParams p)
{
    pdl_wait();
    const int tok = threadIdx.x >> 3, blk = threadIdx.x & 7;
    const int row = tok >> 1, half = tok & 1;
    const long long units = static_cast<long long>(p.batch) * p.max_pages * p.hkv;
    const int max_len = p.max_pages * kPageSize;
    long long u = blockIdx.x;
    PrefixUnit cur{};
    if (u < units)
        cur = prefix_unit(p, u);
    for (; u < units; u += gridDim.x) {
        PrefixUnit nxt{};
        if (u + gridDim.x < units)
            nxt = prefix_unit(p, u + gridDim.x);
        int L = cur.len;
        if (L < 0 || L > max_len) {
            if (threadIdx.x == 0 && cur.pg == 0 && cur.h == 0)
                report(p.dev_status, NVFP4KV_DEV_BAD_LEN);
            L = L < 0 ? 0 : max_len;
        }
        const int j = cur.pg * kPageSize + tok;
        if (j < L) {
            int phys = cur.phys;
            if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_pages)) {
                if (tok == 0 && blk == 0)
                    report(p.dev_status, NVFP4KV_DEV_BAD_PAGE);
                phys = 0;
            }
            const uint8_t *rec = p.pool + (static_cast<size_t>(phys) * p.hkv + cur.h) * kNvfp4Record;
            // K: natural rows
            const uint2 kpacked = __ldg(reinterpret_cast<const uint2 *>(rec + tok * 64 + blk * 8));
            const uint32_t ks = __ldg(rec + 2048 + tok * 8 + blk);
            // V: channel 16*blk + g + 8w sits in row tok/2, chunk (g + 2*row) mod
            // 8, byte 2*blk + w, nibble tok & 1; repacked into natural order
            uint32_t units16[8];
#pragma unroll
            for (int g = 0; g < 8; ++g)
                units16[g] = __ldg(reinterpret_cast<const uint16_t *>(
                    rec + 1024 + row * 128 + ((g + 2 * row) & 7) * 16 + 2 * blk));
            const uint32_t vs = __ldg(rec + 2176 + row * 16 + blk * 2 + half);
            uint32_t lo = 0u, hi = 0u;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                lo |= ((units16[g] >> (4 * half)) & 15u) << (4 * g);        // channel g
                hi |= ((units16[g] >> (8 + 4 * half)) & 15u) << (4 * g);    // channel g + 8
            }
            const size_t orow = (static_cast<size_t>(cur.base) + j) * p.hkv + cur.h;
            *reinterpret_cast<uint4 *>(p.k_out + orow * kHeadDim + blk * 16) = codes_to_e4m3(kpacked, ks);
            *reinterpret_cast<uint4 *>(p.v_out + orow * kHeadDim + blk * 16) =
                codes_to_e4m3(make_uint2(lo, hi), vs);
        }
        cur = nxt;
    }
}

cudaError_t launch_dequant_prefix_fp8(const PrefixParams &p, cudaStream_t s)
{
    const long long units = static_cast<long long>(p.batch) * p.max_pages * p.hkv;
    if (units == 0)
        return cudaSuccess;
    const int sms = sm_count();
    long long grid = static_cast<long long>(sms > 0 ? sms : 1) * 16;
    if (grid > units)
        grid = units;
    return launch_pdl(dequant_prefix_kernel, dim3(static_cast<unsigned>(grid)), dim3(128), 0, s, p);
}

} // namespace nvfp4kv
