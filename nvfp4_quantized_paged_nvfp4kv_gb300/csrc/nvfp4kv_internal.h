// Internal interface between the C ABI (abi.cpp) and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "nvfp4kv.h"

namespace nvfp4kv {

constexpr int kPageSize = 16;
constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 8;                 // query heads per kv head handled by one warp
constexpr int kDecodeWarps = 16;             // warps (independent workers) per decode CTA
constexpr int kDecodeCtasPerSm = 1;          // occupancy the default worker count assumes
constexpr int kPartialFloats = kMaxGroup * kHeadDim + 2 * kMaxGroup;  // O[8][128], m[8], l[8]
constexpr int kNvfp4Record = 2304;           // bytes of an NVFP4 page-head record
constexpr int kFp8Record = 4096;             // bytes of an FP8 page-head record
constexpr int kMaxBatch = NVFP4KV_MAX_BATCH; // prefix table lives in shared memory
constexpr int kMaxScaledHeads = NVFP4KV_MAX_SCALED_KV_HEADS;
// Polls before a wait for staged data (or for another role of the CTA) gives
// up and reports NVFP4KV_DEV_TIMEOUT; the launching calls pass the current
// process-wide limit (nvfp4kv_set_wait_limit) in the kernels' parameters.  A
// wait that only lets work already in flight land before the CTA exits always
// uses this default, whatever the setting.
constexpr uint32_t kWaitLimit = NVFP4KV_WAIT_LIMIT_DEFAULT;

// Per-kv-head tensor scales of K and V, fl32(G * factor), used when per_head
// is set (kernels take these parameters as __grid_constant__, so a head index
// reads them in place); otherwise every head uses the uniform scale.
struct HeadScales {
    int per_head;
    float k[kMaxScaledHeads];
    float v[kMaxScaledHeads];
};

// Split-KV decode over either cache format.
struct DecodeParams {
    const uint8_t *pool;         // page-head records [num_pages][hkv][record]
    const uint16_t *q;           // bf16 [batch][hq][128]
    void *out;                   // [batch][hq][128] bf16 or f32
    const int32_t *block_table;  // [batch][max_pages]
    const int32_t *seq_lens;     // [batch]
    int32_t *dev_status;         // nullable
    float *partials;             // [2 * num_workers][kPartialFloats]
    int batch;
    int hq;
    int hkv;
    int group;
    int max_pages;
    int num_pages;
    int out_bf16;
    int num_workers;
    float qscale;                // sm_scale * log2(e) * tensor scale
    float out_scale;             // tensor scale of V (1 for the FP8 cache)
    float gscale;                // tensor scale the fused append divides by
    // fused append: new K/V rows [batch][hkv][128] written at position
    // seq_lens[b] - 1 before the decode reads the page (append != 0)
    const void *k_new;
    const void *v_new;
    int append;
    int new_bf16;
    // multi-query decode: q_len query tokens per sequence (the last q_len
    // positions, causal among themselves); rows = group * q_len query rows
    // per kv head, taken in row groups of kMaxGroup
    int q_len;
    int rows;
    int row_groups;
    // per-head tensor scales (NVFP4): append divisors and V output scales,
    // and the query scale sm_scale * log2(e) * G_k,h of each kv head
    HeadScales hs;
    float qs[kMaxScaledHeads];
    uint32_t wait_limit;         // polls before a wait gives up (kWaitLimit by default)
};

struct QuantParams {
    const void *k_new;
    const void *v_new;
    const int32_t *slot_mapping;
    uint8_t *pool;               // page-head records [num_pages][hkv][record]
    int32_t *dev_status;
    int num_tokens;
    int hkv;
    int num_pages;
    int in_bf16;
    float gscale;                // tensor scale: blocks are taken of x / gscale
    HeadScales hs;
};

struct PrefixParams {
    const uint8_t *pool;         // NVFP4 page-head records
    const int32_t *block_table;
    const int32_t *prefix_lens;
    const int32_t *kv_indptr;
    uint8_t *k_out;
    uint8_t *v_out;
    int32_t *dev_status;
    int batch;
    int hkv;
    int max_pages;
    int num_pages;
    float gscale;                // tensor scale multiplying every value
    HeadScales hs;
    uint32_t wait_limit;         // polls before a wait gives up (kWaitLimit by default)
};

struct ExtendParams {
    const uint16_t *q;           // bf16 [q rows][hq][128]
    const int32_t *q_indptr;     // [batch + 1] chunk row ranges
    const uint8_t *k_prefix;     // E4M3 [prefix rows][hkv][128]
    const uint8_t *v_prefix;
    const int32_t *kv_indptr;    // [batch] first prefix row of each sequence
    const int32_t *prefix_lens;  // [batch]
    const void *k_chunk;         // [q rows][hkv][128]: bf16, or E4M3 bytes when chunk_e4m3
    const void *v_chunk;
    void *out;                   // [q rows][hq][128], bf16 or fp32
    int32_t *dev_status;
    int batch;
    int hq;
    int hkv;
    int group;                   // hq / hkv
    int q_rows;                  // rows of q, k_chunk, v_chunk and out
    int max_q_len;               // bound on every chunk length (sizes the grid)
    int64_t prefix_rows;         // rows of the prefix workspace
    float qscale;                // sm_scale * log2(e)
    int out_f32;
    int chunk_e4m3;              // chunk K/V are E4M3 bytes (initial prefill on FP8 K/V)
    // fused NVFP4 append of the chunk (null pool: attention only)
    uint8_t *pool;               // page-head records [num_pages][hkv][record]
    const int32_t *slot_mapping; // [q rows]
    int num_pages;
    float gscale;                // tensor scale: blocks are taken of x / gscale
    HeadScales hs;
    uint32_t wait_limit;         // polls before a wait gives up (kWaitLimit by default)
    // E4M3 chunks: tensor maps of the four E4M3 row sets as [rows][hkv][128]
    // bytes, 64-row boxes of one kv head in the 128-byte swizzle, for the
    // kernel that reads every key tile by TMA (filled by the launcher)
    CUtensorMap tm_k_prefix;
    CUtensorMap tm_v_prefix;
    CUtensorMap tm_k_chunk;
    CUtensorMap tm_v_chunk;
};

// Launch with programmatic stream serialisation allowed, so the kernel's
// prologue may overlap the tail of the previous kernel in the stream; every
// kernel launched this way calls pdl_wait() before touching data that the
// previous kernel may still write or read.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

int sm_count();                  // current device, cached
int default_num_workers();       // sm_count * kDecodeCtasPerSm * kDecodeWarps
size_t decode_workspace_bytes(int num_workers);

cudaError_t launch_quantize_append_nvfp4(const QuantParams &p, cudaStream_t s);
cudaError_t launch_quantize_append_fp8(const QuantParams &p, cudaStream_t s);
cudaError_t launch_decode_nvfp4(const DecodeParams &p, cudaStream_t s);
cudaError_t launch_decode_nvfp4_multi(const DecodeParams &p, cudaStream_t s);
cudaError_t launch_decode_fp8(const DecodeParams &p, cudaStream_t s);
cudaError_t launch_merge(const DecodeParams &p, cudaStream_t s);
cudaError_t launch_dequant_prefix_fp8(const PrefixParams &p, cudaStream_t s);
cudaError_t launch_extend_attention(const ExtendParams &p, cudaStream_t s);   // appends when p.pool != null

} // namespace nvfp4kv
