// C ABI of the library: argument validation and launches.
// The contract of every entry point is documented in include/nvfp4kv.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "nvfp4kv.h"
#include "nvfp4kv_internal.h"

using namespace nvfp4kv;

namespace {

std::atomic<uint32_t> g_wait_limit{kWaitLimit};

uint32_t wait_limit()
{
    return g_wait_limit.load(std::memory_order_relaxed);
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

cudaStream_t to_cuda(nvfp4kv_stream_t s)
{
    return reinterpret_cast<cudaStream_t>(s);
}

nvfp4kv_status from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? NVFP4KV_OK : NVFP4KV_ERR_CUDA;
}

bool normal_positive(float x)
{
    return x >= 1.17549435e-38f && x <= 3.40282347e+38f;
}

// Per-head tensor scales of a (checked) NVFP4 cache: fl32(G * factor) per kv
// head of K and V, or per_head = 0 without factors.
HeadScales head_scales_of(const nvfp4kv_cache *c)
{
    HeadScales hs{};
    if (c->head_scales == nullptr)
        return hs;
    hs.per_head = 1;
    for (int h = 0; h < c->num_kv_heads; ++h) {
        hs.k[h] = c->global_scale * c->head_scales[h];
        hs.v[h] = c->global_scale * c->head_scales[c->num_kv_heads + h];
    }
    return hs;
}

// Shared geometry checks for both cache kinds.
nvfp4kv_status check_geometry(int32_t num_pages, int32_t hkv, int32_t page_size, int32_t head_dim)
{
    if (num_pages <= 0 || hkv <= 0 || page_size <= 0 || head_dim <= 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (page_size != kPageSize || head_dim != kHeadDim)
        return NVFP4KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_pages) * hkv > (int64_t{1} << 31) - 1)
        return NVFP4KV_ERR_UNSUPPORTED;
    return NVFP4KV_OK;
}

nvfp4kv_status check_nvfp4(const nvfp4kv_cache *c)
{
    if (c == nullptr)
        return NVFP4KV_ERR_INVALID_ARG;
    nvfp4kv_status st = check_geometry(c->num_pages, c->num_kv_heads, c->page_size, c->head_dim);
    if (st != NVFP4KV_OK)
        return st;
    // a positive, normal, finite tensor scale
    if (!normal_positive(c->global_scale))
        return NVFP4KV_ERR_UNSUPPORTED;
    // optional per-head factors: each, and its product with G, positive normal
    if (c->head_scales != nullptr) {
        if (c->num_kv_heads > kMaxScaledHeads)
            return NVFP4KV_ERR_UNSUPPORTED;
        for (int i = 0; i < 2 * c->num_kv_heads; ++i) {
            const float f = c->head_scales[i];
            if (!normal_positive(f) || !normal_positive(c->global_scale * f))
                return NVFP4KV_ERR_UNSUPPORTED;
        }
    }
    if (c->pool == nullptr || !aligned16(c->pool))
        return NVFP4KV_ERR_INVALID_ARG;
    return NVFP4KV_OK;
}

nvfp4kv_status check_fp8(const fp8kv_cache *c)
{
    if (c == nullptr)
        return NVFP4KV_ERR_INVALID_ARG;
    nvfp4kv_status st = check_geometry(c->num_pages, c->num_kv_heads, c->page_size, c->head_dim);
    if (st != NVFP4KV_OK)
        return st;
    if (c->pool == nullptr || !aligned16(c->pool))
        return NVFP4KV_ERR_INVALID_ARG;
    return NVFP4KV_OK;
}

nvfp4kv_status check_append(const void *k_new, const void *v_new, nvfp4kv_dtype in_dtype, int32_t num_tokens,
                            const int32_t *slot_mapping)
{
    if (num_tokens < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (in_dtype != NVFP4KV_F32 && in_dtype != NVFP4KV_BF16)
        return NVFP4KV_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return NVFP4KV_OK;
    if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr)
        return NVFP4KV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3u))
        return NVFP4KV_ERR_INVALID_ARG;
    return NVFP4KV_OK;
}

// Decode arguments common to both cache kinds.  Fills p (except the cache
// pointers) on success.
nvfp4kv_status check_decode(int32_t hkv, int32_t num_pages, const void *q, int32_t batch, int32_t num_q_heads,
                            const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                            float sm_scale, void *out, nvfp4kv_dtype out_dtype, void *workspace,
                            size_t workspace_bytes, int32_t num_workers, int32_t *dev_status, DecodeParams &p)
{
    if (batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 || num_workers < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (out_dtype != NVFP4KV_F32 && out_dtype != NVFP4KV_BF16)
        return NVFP4KV_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale))
        return NVFP4KV_ERR_INVALID_ARG;
    if (num_q_heads % hkv != 0)
        return NVFP4KV_ERR_INVALID_ARG;
    const int group = num_q_heads / hkv;
    if (group > kMaxGroup)
        return NVFP4KV_ERR_UNSUPPORTED;
    if (batch > kMaxBatch)
        return NVFP4KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(batch) * hkv * max_pages_per_seq > (int64_t{1} << 31) - 1)
        return NVFP4KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_pages_per_seq) * kPageSize > (int64_t{1} << 30))
        return NVFP4KV_ERR_UNSUPPORTED;
    if (batch > 0) {
        if (q == nullptr || out == nullptr || block_table == nullptr || seq_lens == nullptr)
            return NVFP4KV_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
            (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
            return NVFP4KV_ERR_INVALID_ARG;
    }
    int nw = num_workers;
    if (nw == 0) {
        // automatic: the device default, but no more than one worker per four
        // page-heads of the largest possible batch
        const int64_t upper = static_cast<int64_t>(batch) * hkv * max_pages_per_seq;
        int64_t cap = upper / 4;
        if (cap < 1)
            cap = 1;
        nw = default_num_workers();
        if (nw > cap)
            nw = static_cast<int>(cap);
    }
    if (batch > 0) {
        if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return NVFP4KV_ERR_WORKSPACE;
        if (workspace_bytes < decode_workspace_bytes(nw))
            return NVFP4KV_ERR_WORKSPACE;
    }
    p = DecodeParams{};
    p.q = static_cast<const uint16_t *>(q);
    p.out = out;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.dev_status = dev_status;
    p.partials = static_cast<float *>(workspace);
    p.batch = batch;
    p.hq = num_q_heads;
    p.hkv = hkv;
    p.group = group;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.out_bf16 = out_dtype == NVFP4KV_BF16;
    p.num_workers = nw;
    p.qscale = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
    p.out_scale = 1.f;
    p.gscale = 1.f;
    p.q_len = 1;
    p.rows = group;
    p.row_groups = 1;
    p.wait_limit = wait_limit();
    return NVFP4KV_OK;
}

// The NVFP4 tensor scale G: scores see G * k, so G joins the query scale;
// outputs see G * v, so the normaliser carries it.  With per-head factors each
// kv head has its own query scale, append divisors and output scale.
void apply_tensor_scale(DecodeParams &p, float sm_scale, const nvfp4kv_cache *c)
{
    const float G = c->global_scale;
    p.qscale = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634 * static_cast<double>(G));
    p.out_scale = G;
    p.gscale = G;
    p.hs = head_scales_of(c);
    if (p.hs.per_head)
        for (int h = 0; h < c->num_kv_heads; ++h)
            p.qs[h] = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634 *
                                         static_cast<double>(p.hs.k[h]));
}

// Extend arguments common to both entry points.  Fills p (attention part)
// on success; batch == 0 or max_q_len == 0 is valid and launches nothing.
nvfp4kv_status check_extend(const void *q, const int32_t *q_indptr, int32_t q_rows, int32_t max_q_len,
                            const void *k_prefix, const void *v_prefix, const int32_t *kv_indptr,
                            const int32_t *prefix_lens, int64_t prefix_rows, const void *k_chunk,
                            const void *v_chunk, nvfp4kv_dtype chunk_dtype, int32_t batch, int32_t num_q_heads,
                            int32_t num_kv_heads, float sm_scale, void *out, nvfp4kv_dtype out_dtype,
                            int32_t *dev_status, ExtendParams &p)
{
    if (batch < 0 || q_rows < 0 || max_q_len < 0 || prefix_rows < 0 || num_q_heads <= 0 || num_kv_heads <= 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (out_dtype != NVFP4KV_F32 && out_dtype != NVFP4KV_BF16)
        return NVFP4KV_ERR_INVALID_ARG;
    if (chunk_dtype != NVFP4KV_BF16 && chunk_dtype != NVFP4KV_E4M3)
        return NVFP4KV_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale))
        return NVFP4KV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0)
        return NVFP4KV_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (group > kMaxGroup || num_kv_heads > 65535 || batch > 65535)
        return NVFP4KV_ERR_UNSUPPORTED;
    // rows of one sequence and kv head (chunk length x group) stay within
    // int32; workspace element offsets within int64
    if (static_cast<int64_t>(max_q_len) * group > (int64_t{1} << 31) - kMaxGroup * 128)
        return NVFP4KV_ERR_UNSUPPORTED;
    if (prefix_rows > (int64_t{1} << 40) / (static_cast<int64_t>(num_kv_heads) * kHeadDim))
        return NVFP4KV_ERR_UNSUPPORTED;
    if (batch == 0 || max_q_len == 0)
        return NVFP4KV_OK;
    if (q == nullptr || q_indptr == nullptr || kv_indptr == nullptr || prefix_lens == nullptr || k_chunk == nullptr ||
        v_chunk == nullptr || out == nullptr)
        return NVFP4KV_ERR_INVALID_ARG;
    if (prefix_rows > 0 && (k_prefix == nullptr || v_prefix == nullptr))
        return NVFP4KV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_chunk) || !aligned16(v_chunk) || !aligned16(out) || !aligned16(k_prefix) ||
        !aligned16(v_prefix) || (reinterpret_cast<uintptr_t>(q_indptr) & 3u) ||
        (reinterpret_cast<uintptr_t>(kv_indptr) & 3u) || (reinterpret_cast<uintptr_t>(prefix_lens) & 3u))
        return NVFP4KV_ERR_INVALID_ARG;
    p = ExtendParams{};
    p.q = static_cast<const uint16_t *>(q);
    p.q_indptr = q_indptr;
    p.k_prefix = static_cast<const uint8_t *>(k_prefix);
    p.v_prefix = static_cast<const uint8_t *>(v_prefix);
    p.kv_indptr = kv_indptr;
    p.prefix_lens = prefix_lens;
    p.k_chunk = k_chunk;
    p.v_chunk = v_chunk;
    p.chunk_e4m3 = chunk_dtype == NVFP4KV_E4M3;
    p.out = out;
    p.dev_status = dev_status;
    p.batch = batch;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.group = group;
    p.q_rows = q_rows;
    p.max_q_len = max_q_len;
    p.prefix_rows = prefix_rows;
    p.qscale = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
    p.out_f32 = out_dtype == NVFP4KV_F32;
    p.gscale = 1.f;
    p.wait_limit = wait_limit();
    return NVFP4KV_OK;
}

} // namespace

extern "C" {

nvfp4kv_status nvfp4kv_quantize_append(const nvfp4kv_cache *cache, const void *k_new, const void *v_new,
                                       nvfp4kv_dtype in_dtype, int32_t num_tokens, const int32_t *slot_mapping,
                                       int32_t *dev_status, nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_nvfp4(cache);
    if (st != NVFP4KV_OK)
        return st;
    st = check_append(k_new, v_new, in_dtype, num_tokens, slot_mapping);
    if (st != NVFP4KV_OK || num_tokens == 0)
        return st;
    QuantParams p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.pool = static_cast<uint8_t *>(cache->pool);
    p.dev_status = dev_status;
    p.num_tokens = num_tokens;
    p.hkv = cache->num_kv_heads;
    p.num_pages = cache->num_pages;
    p.in_bf16 = in_dtype == NVFP4KV_BF16;
    p.gscale = cache->global_scale;
    p.hs = head_scales_of(cache);
    return from_cuda(launch_quantize_append_nvfp4(p, to_cuda(stream)));
}

size_t nvfp4kv_decode_workspace_size(int32_t num_workers)
{
    return decode_workspace_bytes(num_workers < 0 ? 0 : num_workers);
}

nvfp4kv_status nvfp4kv_paged_decode(const nvfp4kv_cache *cache, const void *q, int32_t batch,
                                    int32_t num_q_heads, const int32_t *block_table, int32_t max_pages_per_seq,
                                    const int32_t *seq_lens, float sm_scale, void *out, nvfp4kv_dtype out_dtype,
                                    void *workspace, size_t workspace_bytes, int32_t num_workers,
                                    int32_t *dev_status, nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_nvfp4(cache);
    if (st != NVFP4KV_OK)
        return st;
    DecodeParams p;
    st = check_decode(cache->num_kv_heads, cache->num_pages, q, batch, num_q_heads, block_table,
                      max_pages_per_seq, seq_lens, sm_scale, out, out_dtype, workspace, workspace_bytes,
                      num_workers, dev_status, p);
    if (st != NVFP4KV_OK || batch == 0)
        return st;
    p.pool = static_cast<const uint8_t *>(cache->pool);
    apply_tensor_scale(p, sm_scale, cache);
    cudaError_t e = launch_decode_nvfp4(p, to_cuda(stream));
    if (e == cudaSuccess)
        e = launch_merge(p, to_cuda(stream));
    return from_cuda(e);
}

nvfp4kv_status nvfp4kv_paged_decode_multi(const nvfp4kv_cache *cache, const void *q, int32_t batch, int32_t q_len,
                                          int32_t num_q_heads, const int32_t *block_table,
                                          int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                          void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                          size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                          nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_nvfp4(cache);
    if (st != NVFP4KV_OK)
        return st;
    if (q_len < 1 || q_len > NVFP4KV_MAX_QUERY_TOKENS)
        return q_len < 1 ? NVFP4KV_ERR_INVALID_ARG : NVFP4KV_ERR_UNSUPPORTED;
    DecodeParams p;
    st = check_decode(cache->num_kv_heads, cache->num_pages, q, batch, num_q_heads, block_table,
                      max_pages_per_seq, seq_lens, sm_scale, out, out_dtype, workspace, workspace_bytes,
                      num_workers, dev_status, p);
    if (st != NVFP4KV_OK || batch == 0)
        return st;
    p.q_len = q_len;
    p.rows = p.group * q_len;
    p.row_groups = (p.rows + kMaxGroup - 1) / kMaxGroup;
    if (static_cast<int64_t>(batch) * cache->num_kv_heads * p.row_groups * max_pages_per_seq >
        (int64_t{1} << 31) - 1)
        return NVFP4KV_ERR_UNSUPPORTED;
    p.pool = static_cast<const uint8_t *>(cache->pool);
    apply_tensor_scale(p, sm_scale, cache);
    cudaError_t e = launch_decode_nvfp4_multi(p, to_cuda(stream));
    if (e == cudaSuccess)
        e = launch_merge(p, to_cuda(stream));
    return from_cuda(e);
}

nvfp4kv_status nvfp4kv_dequant_prefix_fp8(const nvfp4kv_cache *cache, const int32_t *block_table,
                                          int32_t max_pages_per_seq, const int32_t *prefix_lens,
                                          const int32_t *kv_indptr, int32_t batch, void *k_fp8_out,
                                          void *v_fp8_out, int32_t *dev_status, nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_nvfp4(cache);
    if (st != NVFP4KV_OK)
        return st;
    if (batch < 0 || max_pages_per_seq <= 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_pages_per_seq) * kPageSize > (int64_t{1} << 30))
        return NVFP4KV_ERR_UNSUPPORTED;
    if (batch == 0)
        return NVFP4KV_OK;
    if (block_table == nullptr || prefix_lens == nullptr || kv_indptr == nullptr || k_fp8_out == nullptr ||
        v_fp8_out == nullptr)
        return NVFP4KV_ERR_INVALID_ARG;
    if (!aligned16(k_fp8_out) || !aligned16(v_fp8_out) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(prefix_lens) & 3u) || (reinterpret_cast<uintptr_t>(kv_indptr) & 3u))
        return NVFP4KV_ERR_INVALID_ARG;
    PrefixParams p{};
    p.pool = static_cast<const uint8_t *>(cache->pool);
    p.block_table = block_table;
    p.prefix_lens = prefix_lens;
    p.kv_indptr = kv_indptr;
    p.k_out = static_cast<uint8_t *>(k_fp8_out);
    p.v_out = static_cast<uint8_t *>(v_fp8_out);
    p.dev_status = dev_status;
    p.batch = batch;
    p.hkv = cache->num_kv_heads;
    p.max_pages = max_pages_per_seq;
    p.num_pages = cache->num_pages;
    p.gscale = cache->global_scale;
    p.hs = head_scales_of(cache);
    p.wait_limit = wait_limit();
    return from_cuda(launch_dequant_prefix_fp8(p, to_cuda(stream)));
}

nvfp4kv_status nvfp4kv_extend_attention_fp8(const void *q, const int32_t *q_indptr, int32_t q_rows,
                                            int32_t max_q_len, const void *k_prefix, const void *v_prefix,
                                            const int32_t *kv_indptr, const int32_t *prefix_lens,
                                            int64_t prefix_rows, const void *k_chunk, const void *v_chunk,
                                            nvfp4kv_dtype chunk_dtype, int32_t batch, int32_t num_q_heads,
                                            int32_t num_kv_heads, float sm_scale, void *out,
                                            nvfp4kv_dtype out_dtype, int32_t *dev_status, nvfp4kv_stream_t stream)
{
    ExtendParams p{};
    const nvfp4kv_status st =
        check_extend(q, q_indptr, q_rows, max_q_len, k_prefix, v_prefix, kv_indptr, prefix_lens, prefix_rows,
                     k_chunk, v_chunk, chunk_dtype, batch, num_q_heads, num_kv_heads, sm_scale, out, out_dtype,
                     dev_status, p);
    if (st != NVFP4KV_OK || batch == 0 || max_q_len == 0)
        return st;
    return from_cuda(launch_extend_attention(p, to_cuda(stream)));
}

nvfp4kv_status nvfp4kv_extend_attention_fp8_append(const nvfp4kv_cache *cache, const int32_t *slot_mapping,
                                                   const void *q, const int32_t *q_indptr, int32_t q_rows,
                                                   int32_t max_q_len, const void *k_prefix, const void *v_prefix,
                                                   const int32_t *kv_indptr, const int32_t *prefix_lens,
                                                   int64_t prefix_rows, const void *k_chunk, const void *v_chunk,
                                                   nvfp4kv_dtype chunk_dtype, int32_t batch, int32_t num_q_heads,
                                                   float sm_scale, void *out, nvfp4kv_dtype out_dtype,
                                                   int32_t *dev_status, nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_nvfp4(cache);
    if (st != NVFP4KV_OK)
        return st;
    ExtendParams p{};
    st = check_extend(q, q_indptr, q_rows, max_q_len, k_prefix, v_prefix, kv_indptr, prefix_lens, prefix_rows,
                      k_chunk, v_chunk, chunk_dtype, batch, num_q_heads, cache->num_kv_heads, sm_scale, out,
                      out_dtype, dev_status, p);
    if (st != NVFP4KV_OK || batch == 0 || max_q_len == 0)
        return st;
    if (slot_mapping == nullptr || (reinterpret_cast<uintptr_t>(slot_mapping) & 3u))
        return NVFP4KV_ERR_INVALID_ARG;
    p.pool = static_cast<uint8_t *>(cache->pool);
    p.slot_mapping = slot_mapping;
    p.num_pages = cache->num_pages;
    p.gscale = cache->global_scale;
    p.hs = head_scales_of(cache);
    return from_cuda(launch_extend_attention(p, to_cuda(stream)));
}

nvfp4kv_status fp8kv_quantize_append(const fp8kv_cache *cache, const void *k_new, const void *v_new,
                                     nvfp4kv_dtype in_dtype, int32_t num_tokens, const int32_t *slot_mapping,
                                     int32_t *dev_status, nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_fp8(cache);
    if (st != NVFP4KV_OK)
        return st;
    st = check_append(k_new, v_new, in_dtype, num_tokens, slot_mapping);
    if (st != NVFP4KV_OK || num_tokens == 0)
        return st;
    QuantParams p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.pool = static_cast<uint8_t *>(cache->pool);
    p.dev_status = dev_status;
    p.num_tokens = num_tokens;
    p.hkv = cache->num_kv_heads;
    p.num_pages = cache->num_pages;
    p.in_bf16 = in_dtype == NVFP4KV_BF16;
    return from_cuda(launch_quantize_append_fp8(p, to_cuda(stream)));
}

nvfp4kv_status fp8kv_paged_decode(const fp8kv_cache *cache, const void *q, int32_t batch, int32_t num_q_heads,
                                  const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                                  float sm_scale, void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                  size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                  nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_fp8(cache);
    if (st != NVFP4KV_OK)
        return st;
    DecodeParams p;
    st = check_decode(cache->num_kv_heads, cache->num_pages, q, batch, num_q_heads, block_table,
                      max_pages_per_seq, seq_lens, sm_scale, out, out_dtype, workspace, workspace_bytes,
                      num_workers, dev_status, p);
    if (st != NVFP4KV_OK || batch == 0)
        return st;
    p.pool = static_cast<const uint8_t *>(cache->pool);
    cudaError_t e = launch_decode_fp8(p, to_cuda(stream));
    if (e == cudaSuccess)
        e = launch_merge(p, to_cuda(stream));
    return from_cuda(e);
}

nvfp4kv_status nvfp4kv_append_paged_decode(const nvfp4kv_cache *cache, const void *k_new, const void *v_new,
                                           nvfp4kv_dtype in_dtype, const void *q, int32_t batch,
                                           int32_t num_q_heads, const int32_t *block_table,
                                           int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                           void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                           size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                           nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_nvfp4(cache);
    if (st != NVFP4KV_OK)
        return st;
    st = check_append(k_new, v_new, in_dtype, batch, block_table);
    if (st != NVFP4KV_OK)
        return st;
    DecodeParams p;
    st = check_decode(cache->num_kv_heads, cache->num_pages, q, batch, num_q_heads, block_table,
                      max_pages_per_seq, seq_lens, sm_scale, out, out_dtype, workspace, workspace_bytes,
                      num_workers, dev_status, p);
    if (st != NVFP4KV_OK || batch == 0)
        return st;
    p.pool = static_cast<const uint8_t *>(cache->pool);
    apply_tensor_scale(p, sm_scale, cache);
    p.k_new = k_new;
    p.v_new = v_new;
    p.append = 1;
    p.new_bf16 = in_dtype == NVFP4KV_BF16;
    cudaError_t e = launch_decode_nvfp4(p, to_cuda(stream));
    if (e == cudaSuccess)
        e = launch_merge(p, to_cuda(stream));
    return from_cuda(e);
}

nvfp4kv_status fp8kv_append_paged_decode(const fp8kv_cache *cache, const void *k_new, const void *v_new,
                                         nvfp4kv_dtype in_dtype, const void *q, int32_t batch,
                                         int32_t num_q_heads, const int32_t *block_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                         void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                         nvfp4kv_stream_t stream)
{
    nvfp4kv_status st = check_fp8(cache);
    if (st != NVFP4KV_OK)
        return st;
    st = check_append(k_new, v_new, in_dtype, batch, block_table);
    if (st != NVFP4KV_OK)
        return st;
    DecodeParams p;
    st = check_decode(cache->num_kv_heads, cache->num_pages, q, batch, num_q_heads, block_table,
                      max_pages_per_seq, seq_lens, sm_scale, out, out_dtype, workspace, workspace_bytes,
                      num_workers, dev_status, p);
    if (st != NVFP4KV_OK || batch == 0)
        return st;
    p.pool = static_cast<const uint8_t *>(cache->pool);
    p.k_new = k_new;
    p.v_new = v_new;
    p.append = 1;
    p.new_bf16 = in_dtype == NVFP4KV_BF16;
    cudaError_t e = launch_decode_fp8(p, to_cuda(stream));
    if (e == cudaSuccess)
        e = launch_merge(p, to_cuda(stream));
    return from_cuda(e);
}

int64_t nvfp4kv_cache_bytes(int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t head_dim)
{
    if (num_pages < 0 || num_kv_heads < 0 || page_size < 0 || head_dim < 0 || head_dim % 16 != 0)
        return -1;
    const int64_t rows = static_cast<int64_t>(num_pages) * num_kv_heads * page_size;
    return 2 * rows * (head_dim / 2 + head_dim / 16);
}

int64_t fp8kv_cache_bytes(int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t head_dim)
{
    if (num_pages < 0 || num_kv_heads < 0 || page_size < 0 || head_dim < 0)
        return -1;
    return 2 * static_cast<int64_t>(num_pages) * num_kv_heads * page_size * head_dim;
}

nvfp4kv_status nvfp4kv_read_device_status(const int32_t *dev_status, nvfp4kv_stream_t stream, int32_t *bits)
{
    if (dev_status == nullptr || bits == nullptr)
        return NVFP4KV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(to_cuda(stream)) != cudaSuccess)
        return NVFP4KV_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, dev_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return NVFP4KV_ERR_CUDA;
    *bits = v;
    return v != 0 ? NVFP4KV_ERR_DEVICE_CHECK : NVFP4KV_OK;
}

uint32_t nvfp4kv_set_wait_limit(uint32_t polls)
{
    return g_wait_limit.exchange(polls, std::memory_order_relaxed);
}

const char *nvfp4kv_status_string(nvfp4kv_status status)
{
    switch (status) {
    case NVFP4KV_OK:
        return "ok";
    case NVFP4KV_ERR_INVALID_ARG:
        return "invalid argument";
    case NVFP4KV_ERR_UNSUPPORTED:
        return "unsupported geometry or option";
    case NVFP4KV_ERR_WORKSPACE:
        return "decode workspace missing, misaligned or too small";
    case NVFP4KV_ERR_CUDA:
        return "CUDA runtime error";
    case NVFP4KV_ERR_DEVICE_CHECK:
        return "a kernel reported bad device data (see the status bits)";
    }
    return "unknown status";
}

int32_t nvfp4kv_version(void)
{
    return 100;
}

} // extern "C"
