// Write side: quantise new K/V rows into the paged cache.
//
// NVFP4 ("SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation:
// 8 bytes of packed E2M1 plus one E4M3 block scale per 16 values; the tensor
// scale stays 1.0, Perspective).  For each 16-value block of a token-head row:
//   amax = max |x_i|,  S = E4M3_rn_satfinite(fl32(amax / 6)),  s = value(S),
//   q_i = E2M1_rn_satfinite(fl32(x_i / s))   (all zero when s == 0),
//   byte j = q_2j | q_2j+1 << 4.
// FP8 (the comparison cache): each value E4M3_rn_satfinite(x), scale 1.0.
//
// One thread per 16-value block; consecutive threads take consecutive blocks
// of a row, so a warp reads 2 KB (fp32) of contiguous input and writes 256
// contiguous data bytes plus 32 scale bytes.
#include "device_common.cuh"
#include "nvfp4kv.h"

namespace nvfp4kv {

template <bool kBf16>
__device__ __forceinline__ void load16(const void *src, size_t elem_off, float (&x)[16])
{
    if constexpr (kBf16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + elem_off);
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + elem_off);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 v = __ldg(p + k);
            x[4 * k] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
    }
}

// Shared front part: which block this thread owns and where it goes.
struct BlockSite {
    bool active;
    size_t src_off;     // element offset of the block in k_new / v_new
    size_t row;         // cache row: (page * hkv + h) * 16 + offset
    int blk;            // block within the row (0..7)
};

// The cache rows written here may still be read by the previous kernel in the
// stream (a decode of the last step): wait for it, then let the next start.
__device__ __forceinline__ BlockSite locate(const QuantParams &p, long long idx)
{
    pdl_wait();
    pdl_launch_dependents();
    BlockSite s{false, 0, 0, 0};
    const long long rows = static_cast<long long>(p.num_tokens) * p.hkv;
    if (idx >= rows * 8)
        return s;
    const long long th = idx >> 3;                   // token-head row of the input
    s.blk = static_cast<int>(idx & 7);
    const int t = static_cast<int>(th / p.hkv);
    const int h = static_cast<int>(th - static_cast<long long>(t) * p.hkv);
    const int slot = __ldg(p.slot_mapping + t);
    if (slot < 0)
        return s;
    if (slot >= p.num_pages * kPageSize) {
        if (s.blk == 0 && h == 0)
            report(p.dev_status, NVFP4KV_DEV_BAD_SLOT);
        return s;
    }
    const int page = slot / kPageSize, off = slot - page * kPageSize;
    s.active = true;
    s.src_off = static_cast<size_t>(th) * kHeadDim + s.blk * 16;
    s.row = (static_cast<size_t>(page) * p.hkv + h) * kPageSize + off;
    return s;
}

template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const QuantParams p)
{
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const BlockSite s = locate(p, idx);
    if (!s.active)
        return;
    const bool is_v = blockIdx.y == 1;
    float x[16];
    load16<kBf16>(is_v ? p.v_new : p.k_new, s.src_off, x);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
    const float s32 = __fdiv_rn(amax, 6.0f);
    const uint32_t S = f32x2_to_e4m3x2(s32, 0.f) & 0xffu;
    const float sc = e4m3_to_f32(S);
    uint32_t packed[2] = {0u, 0u};
    if (sc != 0.f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(x[2 * j], sc), __fdiv_rn(x[2 * j + 1], sc));
            packed[j >> 2] |= byte << (8 * (j & 3));
        }
    }
    uint8_t *data = is_v ? p.v_data : p.k_data;
    uint8_t *scale = is_v ? p.v_scale : p.k_scale;
    *reinterpret_cast<uint2 *>(data + s.row * (kHeadDim / 2) + s.blk * 8) = make_uint2(packed[0], packed[1]);
    scale[s.row * (kHeadDim / 16) + s.blk] = static_cast<uint8_t>(S);
}

template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const QuantParams p)
{
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const BlockSite s = locate(p, idx);
    if (!s.active)
        return;
    const bool is_v = blockIdx.y == 1;
    float x[16];
    load16<kBf16>(is_v ? p.v_new : p.k_new, s.src_off, x);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = f32x2_to_e4m3x2(x[4 * k], x[4 * k + 1]) | (f32x2_to_e4m3x2(x[4 * k + 2], x[4 * k + 3]) << 16);
    uint8_t *data = is_v ? p.v_data : p.k_data;
    *reinterpret_cast<uint4 *>(data + s.row * kHeadDim + s.blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <class K>
static cudaError_t launch_blocks(K kernel, const QuantParams &p, cudaStream_t s)
{
    const long long blocks = static_cast<long long>(p.num_tokens) * p.hkv * 8;
    if (blocks == 0)
        return cudaSuccess;
    const long long grid = (blocks + 255) / 256;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(grid), 2), dim3(256), 0, s, p);
}

cudaError_t launch_quantize_append_nvfp4(const QuantParams &p, cudaStream_t s)
{
    return p.in_bf16 ? launch_blocks(quantize_nvfp4_kernel<true>, p, s)
                     : launch_blocks(quantize_nvfp4_kernel<false>, p, s);
}

cudaError_t launch_quantize_append_fp8(const QuantParams &p, cudaStream_t s)
{
    return p.in_bf16 ? launch_blocks(quantize_fp8_kernel<true>, p, s)
                     : launch_blocks(quantize_fp8_kernel<false>, p, s);
}

} // namespace nvfp4kv
