// Split-KV merge (flash-decoding log-sum-exp combine) and the decode workspace
// arithmetic.  For a segment (sequence b, kv head h) split over workers
// wf..wl, each left (O_w, m_w, l_w) with O_w = sum_j 2^(s_j - m_w) v_j and
// l_w = sum_j 2^(s_j - m_w) (scores s in log2 units).  Then
//   M = max_w m_w,   o = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w.
#include "decode_common.cuh"

namespace nvfp4kv {

__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p)
{
    extern __shared__ int32_t msmem[];
    int32_t *scratch = msmem;
    int32_t *prefix = msmem + 8;
    build_prefix(p.seq_lens, p.batch, p.hkv, p.max_pages * kPageSize, prefix, scratch, nullptr);

    const int b = blockIdx.x / p.hkv;
    const int h = blockIdx.x - b * p.hkv;
    const int i = blockIdx.y;
    const int c = threadIdx.x;
    const int n = (prefix[b + 1] - prefix[b]) / p.hkv;
    const size_t o = (static_cast<size_t>(b) * p.hq + h * p.group + i) * kHeadDim + c;

    float result;
    if (n == 0) {
        result = 0.f;
    } else {
        const long long T = prefix[p.batch];
        const long long NW = p.num_workers;
        const int seg_begin = prefix[b] + h * n;
        const int wf = owner_of(seg_begin, T, NW);
        const int wl = owner_of(static_cast<long long>(seg_begin) + n - 1, T, NW);
        if (wf == wl)
            return;                              // written by the decode kernel
        float M = -INFINITY;
        for (int w = wf; w <= wl; ++w) {
            const float *slot = p.partials + static_cast<size_t>(partial_slot(w, seg_begin, T, NW)) * kPartialFloats;
            M = fmaxf(M, __ldcg(slot + kMaxGroup * kHeadDim + i));
        }
        float acc = 0.f, den = 0.f;
        for (int w = wf; w <= wl; ++w) {
            const float *slot = p.partials + static_cast<size_t>(partial_slot(w, seg_begin, T, NW)) * kPartialFloats;
            const float e = fast_exp2(__ldcg(slot + kMaxGroup * kHeadDim + i) - M);
            acc += e * __ldcg(slot + i * kHeadDim + c);
            den += e * __ldcg(slot + kMaxGroup * kHeadDim + kMaxGroup + i);
        }
        result = acc / den;
    }
    if (p.out_bf16)
        static_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(result);
    else
        static_cast<float *>(p.out)[o] = result;
}

cudaError_t launch_merge(const DecodeParams &p, cudaStream_t s)
{
    const size_t smem = (8 + static_cast<size_t>(p.batch) + 1) * sizeof(int32_t);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
    }
    dim3 grid(p.batch * p.hkv, p.group);
    merge_kernel<<<grid, 128, smem, s>>>(p);
    return cudaGetLastError();
}

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 0;
    if (dev < 64 && cached[dev] > 0)
        return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < 64)
        cached[dev] = n;
    return n;
}

int default_num_workers()
{
    const int sms = sm_count();
    return (sms > 0 ? sms : 1) * kDecodeCtasPerSm * kDecodeWarps;
}

size_t decode_workspace_bytes(int num_workers)
{
    if (num_workers <= 0)
        num_workers = default_num_workers();
    return static_cast<size_t>(2) * num_workers * kPartialFloats * sizeof(float);
}

} // namespace nvfp4kv
