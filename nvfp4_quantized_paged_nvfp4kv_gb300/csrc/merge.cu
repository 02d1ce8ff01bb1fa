// Split-KV merge (flash-decoding log-sum-exp combine) and the decode workspace
// arithmetic.  For a segment (sequence b, kv head h) split over workers
// wf..wl, each left (O_w, m_w, l_w) with O_w = sum_j 2^(s_j - m_w) v_j and
// l_w = sum_j 2^(s_j - m_w) (scores s in log2 units).  Then
//   M = max_w m_w,   o = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w.
#include "decode_common.cuh"

namespace nvfp4kv {

// Thread t works on channels 4*(t%32) .. +3 of the CTA's query head for the
// contributors k = t/32, t/32 + 8, ...; the 8 contributor groups are summed in
// shared memory.  Warp 0 first finds M and the denominator.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p)
{
    constexpr int kGroups = kMergeThreads / 32;
    extern __shared__ int32_t msmem[];
    __shared__ float4 part[kGroups][32];
    __shared__ float s_max, s_den;
    int32_t *scratch = msmem;
    int32_t *prefix = msmem + 32;
    build_prefix(p.seq_lens, p.batch, p.hkv, p.max_pages * kPageSize, prefix, scratch, nullptr);

    const int b = blockIdx.x / p.hkv;
    const int h = blockIdx.x - b * p.hkv;
    const int i = blockIdx.y;
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
    const int n = (prefix[b + 1] - prefix[b]) / p.hkv;
    const size_t o = (static_cast<size_t>(b) * p.hq + h * p.group + i) * kHeadDim + 4 * lane;

    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (n > 0) {
        const long long T = prefix[p.batch];
        const long long NW = p.num_workers;
        const int seg_begin = prefix[b] + h * n;
        const int wf = owner_of(seg_begin, T, NW);
        const int wl = owner_of(static_cast<long long>(seg_begin) + n - 1, T, NW);
        if (wf == wl)
            return;                              // written by the decode kernel
        pdl_wait();                              // the partials come from the decode kernel
        const int nc = wl - wf + 1;
        auto slot_of = [&](int k) {
            return p.partials + static_cast<size_t>(partial_slot(wf + k, seg_begin, T, NW)) * kPartialFloats;
        };
        if (grp == 0) {
            float M = -INFINITY;
            for (int k = lane; k < nc; k += 32)
                M = fmaxf(M, __ldcg(slot_of(k) + kMaxGroup * kHeadDim + i));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
            float den = 0.f;
            for (int k = lane; k < nc; k += 32) {
                const float *sl = slot_of(k);
                den += fast_exp2(__ldcg(sl + kMaxGroup * kHeadDim + i) - M) *
                       __ldcg(sl + kMaxGroup * kHeadDim + kMaxGroup + i);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                den += __shfl_xor_sync(kFullMask, den, off);
            if (lane == 0) {
                s_max = M;
                s_den = den;
            }
        }
        __syncthreads();
        const float M = s_max;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int k = grp; k < nc; k += kGroups) {
            const float *sl = slot_of(k);
            const float e = fast_exp2(__ldcg(sl + kMaxGroup * kHeadDim + i) - M);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(sl + i * kHeadDim) + lane);
            acc.x += e * v.x;
            acc.y += e * v.y;
            acc.z += e * v.z;
            acc.w += e * v.w;
        }
        part[grp][lane] = acc;
        __syncthreads();
        if (grp != 0)
            return;
        for (int k = 1; k < kGroups; ++k) {
            const float4 v = part[k][lane];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float r = 1.f / s_den;
        res = make_float4(acc.x * r, acc.y * r, acc.z * r, acc.w * r);
    } else if (grp != 0) {
        return;
    }
    if (p.out_bf16) {
        __nv_bfloat162 a = __floats2bfloat162_rn(res.x, res.y), c = __floats2bfloat162_rn(res.z, res.w);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + o) =
            make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&c));
    } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o) = res;
    }
}

cudaError_t launch_merge(const DecodeParams &p, cudaStream_t s)
{
    const size_t smem = (32 + static_cast<size_t>(p.batch) + 1) * sizeof(int32_t);
    if (smem > 40 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(merge_kernel, dim3(p.batch * p.hkv, p.group), dim3(kMergeThreads), smem, s, p);
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
