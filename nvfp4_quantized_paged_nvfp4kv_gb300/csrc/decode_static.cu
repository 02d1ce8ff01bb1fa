// NVFP4 paged decode for callers that cannot allocate device memory.
//
// A serving engine typically reserves a fixed share of device memory for
// weights and the KV cache when it starts, and hands out no further device
// memory while it decodes; some callers also run where a device allocation
// would stall or fail because that budget is already spent.  Such callers
// cannot provide the decode workspace that nvfp4kv_paged_decode asks for.
// This entry point takes its split-KV scratch (the per-worker partial softmax
// states) from one fixed array compiled into the library instead.
//
// The array below is a file-scope __device__ object.  Host code must not use
// its name as a pointer: on the host that name is only a stand-in, not a
// device address.  The device address is looked up once per device, with that
// device current, by the first call made on it (cudaGetSymbolAddress), so the
// first call on each device should come before any stream capture.  Every call
// on a device uses the same array, and it keeps whatever the last call left;
// nothing in it has to start at zero, because each call writes every partial
// it later reads.  Calls whose kernels overlap on the GPU (for example on two
// streams at once) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "nvfp4kv.h"
#include "nvfp4kv_internal.h"

namespace nvfp4kv {
namespace {

constexpr size_t kStaticScratchBytes = NVFP4KV_STATIC_SCRATCH_BYTES;
// two partial slots per worker
static_assert(kStaticScratchBytes / (2 * kPartialFloats * sizeof(float)) >= NVFP4KV_STATIC_SCRATCH_MAX_WORKERS,
              "static scratch too small for its advertised worker count");

static __device__ __align__(256) float g_decode_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

} // namespace
} // namespace nvfp4kv

using namespace nvfp4kv;

extern "C" nvfp4kv_status nvfp4kv_paged_decode_static_scratch(
    const nvfp4kv_cache *cache, const void *q, int32_t batch, int32_t num_q_heads, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale, void *out, nvfp4kv_dtype out_dtype,
    int32_t num_workers, int32_t *dev_status, nvfp4kv_stream_t stream)
{
    if (cache == nullptr || num_workers < 0 || batch < 0 || max_pages_per_seq <= 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (num_workers > NVFP4KV_STATIC_SCRATCH_MAX_WORKERS)
        return NVFP4KV_ERR_WORKSPACE;
    if (batch == 0)   // nothing to launch: the ordinary call checks the other arguments
        return nvfp4kv_paged_decode(cache, q, batch, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                    sm_scale, out, out_dtype, nullptr, 0, num_workers, dev_status, stream);
    int nw = num_workers;
    if (nw == 0) {
        // the automatic choice of nvfp4kv_paged_decode, capped by the array
        const int64_t upper = static_cast<int64_t>(batch) * (cache->num_kv_heads > 0 ? cache->num_kv_heads : 1) *
                              max_pages_per_seq;
        int64_t cap = upper / 4;
        if (cap < 1)
            cap = 1;
        nw = default_num_workers();
        if (nw > NVFP4KV_STATIC_SCRATCH_MAX_WORKERS)
            nw = NVFP4KV_STATIC_SCRATCH_MAX_WORKERS;
        if (nw > cap)
            nw = static_cast<int>(cap);
    }
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return NVFP4KV_ERR_CUDA;
    return nvfp4kv_paged_decode(cache, q, batch, num_q_heads, block_table, max_pages_per_seq, seq_lens, sm_scale,
                                out, out_dtype, scratch, kStaticScratchBytes, nw, dev_status, stream);
}
