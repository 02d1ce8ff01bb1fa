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
// One thread per 16-value block of one token-head row of K or V.  Records are
// laid out as documented in include/nvfp4kv.h: K rows are natural (8 bytes per
// block, one 8-byte store); V bytes hold the two tokens of a token pair in their
// two nibbles, so a V block is merged into its 8 words with atomic AND/OR on the
// thread's own nibbles (the other token of the pair may be written by another
// thread or another call).
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
    size_t record;      // byte offset of the page-head record
    int tok;            // token within the page (0..15)
    int blk;            // block within the row (0..7)
};

// The cache records written here may still be read by the previous kernel in
// the stream (a decode of the last step): wait for it, then let the next start.
__device__ __forceinline__ BlockSite locate(const QuantParams &p, long long idx, int record_bytes)
{
    pdl_wait();
    pdl_launch_dependents();
    BlockSite s{false, 0, 0, 0, 0};
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
    const int page = slot / kPageSize;
    s.tok = slot - page * kPageSize;
    s.active = true;
    s.src_off = static_cast<size_t>(th) * kHeadDim + s.blk * 16;
    s.record = (static_cast<size_t>(page) * p.hkv + h) * record_bytes;
    return s;
}

// amax -> E4M3 block scale -> 16 E2M1 codes (code i in bits 4i .. 4i+3).
__device__ __forceinline__ void quantize_block(const float (&x)[16], uint32_t &scale_byte, uint32_t (&packed)[2])
{
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
    const float s32 = __fdiv_rn(amax, 6.0f);
    scale_byte = f32x2_to_e4m3x2(s32, 0.f) & 0xffu;
    const float sc = e4m3_to_f32(scale_byte);
    packed[0] = packed[1] = 0u;
    if (sc != 0.f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(x[2 * j], sc), __fdiv_rn(x[2 * j + 1], sc));
            packed[j >> 2] |= byte << (8 * (j & 3));
        }
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const QuantParams p)
{
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const BlockSite s = locate(p, idx, kNvfp4Record);
    if (!s.active)
        return;
    const bool is_v = blockIdx.y == 1;
    float x[16];
    load16<kBf16>(is_v ? p.v_new : p.k_new, s.src_off, x);
    uint32_t S, packed[2];
    quantize_block(x, S, packed);
    uint8_t *rec = p.pool + s.record;
    if (!is_v) {
        *reinterpret_cast<uint2 *>(rec + s.tok * 64 + s.blk * 8) = make_uint2(packed[0], packed[1]);
        rec[2048 + s.tok * 8 + s.blk] = static_cast<uint8_t>(S);
        return;
    }
    // V: channel 16*blk + r (r = g + 8w) goes to row tok/2, group g at chunk
    // position (g + 2*row) mod 8, byte 2*blk + w, nibble (tok & 1).
    const int row = s.tok >> 1, half = s.tok & 1;
    const uint64_t codes = (static_cast<uint64_t>(packed[1]) << 32) | packed[0];
    const uint32_t shift = 16u * (s.blk & 1);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t c0 = static_cast<uint32_t>(codes >> (4 * g)) & 15u;        // channel 16blk + g
        const uint32_t c1 = static_cast<uint32_t>(codes >> (4 * (g + 8))) & 15u;  // channel 16blk + g + 8
        const uint32_t unit = (c0 << (4 * half)) | (c1 << (8 + 4 * half));
        const uint32_t mask = (0xFu << (4 * half)) | (0xFu << (8 + 4 * half));
        unsigned int *word = reinterpret_cast<unsigned int *>(
            rec + 1024 + row * 128 + ((g + 2 * row) & 7) * 16 + ((2 * s.blk) & ~3));
        atomicAnd(word, ~(mask << shift));
        atomicOr(word, unit << shift);
    }
    rec[2176 + row * 16 + s.blk * 2 + half] = static_cast<uint8_t>(S);
}

template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const QuantParams p)
{
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const BlockSite s = locate(p, idx, kFp8Record);
    if (!s.active)
        return;
    const bool is_v = blockIdx.y == 1;
    float x[16];
    load16<kBf16>(is_v ? p.v_new : p.k_new, s.src_off, x);
    uint8_t *rec = p.pool + s.record;
    if (!is_v) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = f32x2_to_e4m3x2(x[4 * k], x[4 * k + 1]) | (f32x2_to_e4m3x2(x[4 * k + 2], x[4 * k + 3]) << 16);
        *reinterpret_cast<uint4 *>(rec + s.tok * 128 + ((s.blk + (s.tok & 1)) & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
        return;
    }
    // V: channel 8c + i of token 2*row + half is byte 2i + half of chunk c,
    // stored at chunk position (c + f(row)) mod 16.
    const int row = s.tok >> 1, half = s.tok & 1;
    const int f = (row & 1) + 4 * ((row >> 1) & 1);
    uint8_t *vrow = rec + 2048 + row * 256;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * s.blk + cc;
        uint8_t *chunk = vrow + ((c + f) & 15) * 16;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t two = f32x2_to_e4m3x2(x[8 * cc + i], x[8 * cc + i + 1]);
            chunk[2 * i + half] = static_cast<uint8_t>(two & 0xffu);
            chunk[2 * (i + 1) + half] = static_cast<uint8_t>(two >> 8);
        }
    }
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
