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
// Records are laid out as documented in include/nvfp4kv.h: K rows are natural
// (8 bytes per block, one 8-byte store); V bytes hold the two tokens of a token
// pair in their two nibbles.  A pair whose two tokens are neighbours in this
// call is written whole by one thread; a lone token's V block is merged into
// its 8 words with atomic AND/OR on its own nibbles (its partner may come from
// another call).
#include "nvfp4kv.h"
#include "record_write.cuh"

namespace nvfp4kv {

// Where the block of input token t lands: the byte offset of its page-head
// record and its token within the page, or false when the slot is skipped
// (negative) or out of range (reported).
__device__ __forceinline__ bool site_of(const QuantParams &p, int slot, int h, int record_bytes, size_t &record,
                                        int &tok, bool report_bad)
{
    if (slot < 0)
        return false;
    if (slot >= p.num_pages * kPageSize) {
        if (report_bad)
            report(p.dev_status, NVFP4KV_DEV_BAD_SLOT);
        return false;
    }
    const int page = slot / kPageSize;
    tok = slot - page * kPageSize;
    record = (static_cast<size_t>(page) * p.hkv + h) * record_bytes;
    return true;
}

// NVFP4: one thread per (token pair, kv head, block) of K (blockIdx.y == 0)
// or V (y == 1), so that each thread has both tokens' loads in flight at once.
// V pairs are taken in input order, starting one token early when the first
// slot is odd, so that consecutive slots (the usual prefill order) form the
// record's token pairs; such a pair is written whole, any other token through
// the atomic nibble merge.  Data loads are issued together with the slot
// loads (the source offset does not depend on the slot).  The value and
// reciprocal of each block-scale byte come from a table in shared memory,
// filled once per CTA while the loads are in flight.  The kernel is bound by
// its instruction issue more than by memory: bf16 rows fit five CTAs to an SM
// (48 registers, no spills), fp32 rows four.
template <bool kBf16>
__global__ void __launch_bounds__(256, kBf16 ? 5 : 4) quantize_nvfp4_kernel(const __grid_constant__ QuantParams p)
{
    __shared__ float2 scale_tab[128];
    pdl_wait();                  // the records may still be read by the previous kernel
    pdl_launch_dependents();
    const unsigned idx = blockIdx.x * blockDim.x + threadIdx.x;
    const int blk = static_cast<int>(idx & 7u);
    const unsigned unit = idx >> 3;                  // pair * hkv + h
    const unsigned hk = static_cast<unsigned>(p.hkv);
    unsigned hu, pr;
    if ((hk & (hk - 1u)) == 0u) {                    // a power of two: no division
        hu = unit & (hk - 1u);
        pr = unit >> (__ffs(hk) - 1);
    } else {
        hu = unit % hk;
        pr = unit / hk;
    }
    const int h = static_cast<int>(hu);
    const bool is_v = blockIdx.y == 1;
    const int first = __ldg(p.slot_mapping);
    const int o = (is_v && first >= 0) ? (first & 1) : 0;
    const unsigned pairs = (static_cast<unsigned>(p.num_tokens) + o + 1) / 2;
    const int t0 = static_cast<int>(2 * pr) - o, t1 = t0 + 1;
    const bool live = pr < pairs;
    const bool has0 = live && t0 >= 0, has1 = live && t1 < p.num_tokens;
    const void *src = is_v ? p.v_new : p.k_new;
    RawBlock<kBf16> r0, r1;
    if (has0)
        load_raw<kBf16>(src, (static_cast<size_t>(t0) * p.hkv + h) * kHeadDim + blk * 16, r0);
    if (has1)
        load_raw<kBf16>(src, (static_cast<size_t>(t1) * p.hkv + h) * kHeadDim + blk * 16, r1);
    const int s0 = has0 ? __ldg(p.slot_mapping + t0) : -1;
    const int s1 = has1 ? __ldg(p.slot_mapping + t1) : -1;
    fill_scale_table(scale_tab);
    __syncthreads();
    if (!live)
        return;
    const ScaleTable tab{scale_tab};
    size_t rec0 = 0, rec1 = 0;
    int tok0 = 0, tok1 = 0;
    const bool rep = !is_v && blk == 0 && h == 0;
    const bool ok0 = has0 && site_of(p, s0, h, kNvfp4Record, rec0, tok0, rep);
    const bool ok1 = has1 && site_of(p, s1, h, kNvfp4Record, rec1, tok1, rep);
    float x[16];
    const TensorScale G = tensor_scale(head_tensor_scale(p.hs, is_v, h, p.gscale));
    if (is_v && ok0 && ok1 && (s0 & 1) == 0 && s1 == s0 + 1) {
        uint32_t S0, S1, c0[2], c1[2];
        unpack<kBf16>(r0, x);
        uint32_t flip = divide_by_tensor_scale(x, G);
        quantize_block(x, S0, c0, tab, flip);
        unpack<kBf16>(r1, x);
        flip = divide_by_tensor_scale(x, G);
        quantize_block(x, S1, c1, tab, flip);
        write_nvfp4_v_pair(p.pool + rec0, tok0, blk, S0, c0, S1, c1);
        return;
    }
    if (ok0) {
        unpack<kBf16>(r0, x);
        const uint32_t flip = divide_by_tensor_scale(x, G);
        write_nvfp4_block(p.pool + rec0, is_v, tok0, blk, x, tab, flip);
    }
    if (ok1) {
        unpack<kBf16>(r1, x);
        const uint32_t flip = divide_by_tensor_scale(x, G);
        write_nvfp4_block(p.pool + rec1, is_v, tok1, blk, x, tab, flip);
    }
}

// FP8: one thread per (token, kv head, block) of K (y == 0) or V (y == 1).
template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const QuantParams p)
{
    pdl_wait();
    pdl_launch_dependents();
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int blk = static_cast<int>(idx & 7);
    const long long unit = idx >> 3;
    const int h = static_cast<int>(unit % p.hkv);
    const long long tu = unit / p.hkv;
    if (tu >= p.num_tokens)
        return;
    const int t = static_cast<int>(tu);
    const bool is_v = blockIdx.y == 1;
    float x[16];
    load16<kBf16>(is_v ? p.v_new : p.k_new, (static_cast<size_t>(t) * p.hkv + h) * kHeadDim + blk * 16, x);
    size_t record;
    int tok;
    if (!site_of(p, __ldg(p.slot_mapping + t), h, kFp8Record, record, tok, !is_v && blk == 0 && h == 0))
        return;
    write_fp8_block(p.pool + record, is_v, tok, blk, x);
}

template <class K>
static cudaError_t launch_blocks(K kernel, const QuantParams &p, cudaStream_t s, bool pairs)
{
    const long long units = pairs ? (static_cast<long long>(p.num_tokens) + 2) / 2 : p.num_tokens;
    const long long blocks = units * p.hkv * 8;
    if (blocks == 0)
        return cudaSuccess;
    if (blocks >= (1LL << 32))
        return cudaErrorInvalidValue;        // thread indices are 32-bit
    const long long grid = (blocks + 255) / 256;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(grid), 2), dim3(256), 0, s, p);
}

cudaError_t launch_quantize_append_nvfp4(const QuantParams &p, cudaStream_t s)
{
    return p.in_bf16 ? launch_blocks(quantize_nvfp4_kernel<true>, p, s, true)
                     : launch_blocks(quantize_nvfp4_kernel<false>, p, s, true);
}

cudaError_t launch_quantize_append_fp8(const QuantParams &p, cudaStream_t s)
{
    return p.in_bf16 ? launch_blocks(quantize_fp8_kernel<true>, p, s, false)
                     : launch_blocks(quantize_fp8_kernel<false>, p, s, false);
}

} // namespace nvfp4kv
