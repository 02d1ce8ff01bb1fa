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
#include "nvfp4kv.h"
#include "record_write.cuh"

namespace nvfp4kv {

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
    write_nvfp4_block(p.pool + s.record, is_v, s.tok, s.blk, x);
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
    write_fp8_block(p.pool + s.record, is_v, s.tok, s.blk, x);
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
