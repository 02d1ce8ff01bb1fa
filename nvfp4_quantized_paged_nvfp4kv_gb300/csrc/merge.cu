// Split-KV merge (flash-decoding log-sum-exp combine) and the decode workspace
// arithmetic.  For a segment (sequence b, kv head h) split over the decode
// workers wf..wl, each left one partial (O_w, m_w, l_w) with O_w = sum_j 2^(s_j - m_w) v_j and
// l_w = sum_j 2^(s_j - m_w) (scores s in log2 units).  Then
//   M = max_w m_w,   o = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w.
#include "decode_common.cuh"

namespace nvfp4kv {

// Thread t works on channels 4*(t%32) .. +3 of the CTA's query head for the
// contributors k = t/32, t/32 + G, ... (G = kThreads / 32 contributor
// groups, each loading kUnroll contributors ahead); each group keeps
// its own running maximum (one pass over the partials), and the groups are
// combined in shared memory at the end.  The segment's contributor range is
// worked out once per CTA, before the wait for the decode kernel.
template <int kThreads>
__device__ __forceinline__ void merge_segment_row(const DecodeParams &p, int32_t *msmem)
{
    constexpr int kGroups = kThreads / 32;
    constexpr int kUnroll = 8;                   // contributors a thread loads before using any
    __shared__ float4 part[kGroups][32];
    __shared__ float part_m[kGroups], part_l[kGroups];
    __shared__ int seg[3];                       // first contributor, count (-1: empty sequence), its slot
    int32_t *scratch = msmem;
    int32_t *prefix = msmem + kPrefixScratch;
    const int nseg = p.hkv * p.row_groups;       // segments per sequence (row groups of kv heads)
    build_prefix(p.seq_lens, p.batch, nseg, p.max_pages * kPageSize, prefix, scratch, nullptr);

    const int b = blockIdx.x / nseg;
    const int h = blockIdx.x - b * nseg;
    const int i = blockIdx.y;                    // row of the segment's row group
    const int hp = h / p.row_groups, row = (h - hp * p.row_groups) * kMaxGroup + i;
    if (row >= p.rows)
        return;
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        const int n = (prefix[b + 1] - prefix[b]) / nseg;
        int wf = 0, nc = -1, slot = 0;
        if (n > 0) {
            const long long T = prefix[p.batch];
            const long long NW = effective_workers(p.num_workers, T);
            const int seg_begin = prefix[b] + h * n;
            wf = owner_of(seg_begin, T, NW);
            nc = owner_of(static_cast<long long>(seg_begin) + n - 1, T, NW) - wf + 1;
            // wf reached this segment from an earlier one unless it starts at
            // seg_begin; every later contributor starts inside the segment, so
            // this is its first partial (slot 2w)
            slot = partial_slot(wf, seg_begin, T, NW);
        }
        seg[0] = wf;
        seg[1] = nc;
        seg[2] = slot;
    }
    __syncthreads();
    const int wf = seg[0], nc = seg[1], slot_wf = seg[2];
    if (nc == 1)
        return;                                  // written by the decode kernel
    const size_t o = out_row(p, b, hp, row) + 4 * lane;

    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nc > 1) {
        pdl_wait();                              // the partials come from the decode kernel
        float M = -INFINITY, den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = grp; k0 < nc; k0 += kGroups * kUnroll) {
            float mk[kUnroll], lk[kUnroll];
            float4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int k = k0 + u * kGroups;
                mk[u] = -INFINITY;
                lk[u] = 0.f;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k < nc) {
                    const int slot = k == 0 ? slot_wf : 2 * (wf + k);
                    const float *sl = p.partials + static_cast<size_t>(slot) * kPartialFloats;
                    mk[u] = __ldcg(sl + kMaxGroup * kHeadDim + i);
                    lk[u] = __ldcg(sl + kMaxGroup * kHeadDim + kMaxGroup + i);
                    v[u] = __ldcg(reinterpret_cast<const float4 *>(sl + i * kHeadDim) + lane);
                }
            }
            float mx = M;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                mx = fmaxf(mx, mk[u]);
            const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - mx);
            acc = make_float4(acc.x * a, acc.y * a, acc.z * a, acc.w * a);
            den *= a;
            M = mx;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float e = (mk[u] == -INFINITY) ? 0.f : fast_exp2(mk[u] - M);
                acc.x += e * v[u].x;
                acc.y += e * v[u].y;
                acc.z += e * v[u].z;
                acc.w += e * v[u].w;
                den += e * lk[u];
            }
        }
        part[grp][lane] = acc;
        if (lane == 0) {
            part_m[grp] = M;
            part_l[grp] = den;
        }
        __syncthreads();
        if (grp != 0)
            return;
        float Mall = part_m[0];
        for (int k = 1; k < kGroups; ++k)
            Mall = fmaxf(Mall, part_m[k]);
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        float dsum = 0.f;
        for (int k = 0; k < kGroups; ++k) {
            if (part_m[k] == -INFINITY)
                continue;                        // a group with no contributor
            const float e = fast_exp2(part_m[k] - Mall);
            const float4 v = part[k][lane];
            sum.x += e * v.x;
            sum.y += e * v.y;
            sum.z += e * v.z;
            sum.w += e * v.w;
            dsum += e * part_l[k];
        }
        const float osc = head_tensor_scale(p.hs, true, hp, p.out_scale);
        const float r = dsum > 0.f ? osc / dsum : 0.f;           // a row that saw no key: zeros
        res = make_float4(sum.x * r, sum.y * r, sum.z * r, sum.w * r);
    } else if (grp != 0) {
        return;                                  // empty sequence: zeros
    }
    if (p.out_bf16) {
        __nv_bfloat162 a = __floats2bfloat162_rn(res.x, res.y), c = __floats2bfloat162_rn(res.z, res.w);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + o) =
            make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&c));
    } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o) = res;
    }
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads == 64 ? 16 : 1) merge_kernel(const __grid_constant__ DecodeParams p)
{
    extern __shared__ int32_t msmem[];
    pdl_launch_dependents();                     // the next kernel may start its prologue
    merge_segment_row<kThreads>(p, msmem);
    // The next kernel in the stream waits for this grid only, and the decode's
    // own outputs (segments one worker covered) must be complete by then: one
    // thread of the grid always waits for the decode grid, so this grid cannot
    // complete before it, even when no segment has partials to merge.
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        pdl_wait();
}

template <int kThreads>
static cudaError_t launch_merge_width(const DecodeParams &p, cudaStream_t s)
{
    const size_t smem = (kPrefixScratch + static_cast<size_t>(p.batch) + 1) * sizeof(int32_t);
    if (smem > 40 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_kernel<kThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(merge_kernel<kThreads>,
                      dim3(p.batch * p.hkv * p.row_groups, p.rows < kMaxGroup ? p.rows : kMaxGroup),
                      dim3(kThreads), smem, s, p);
}

// Contributors per segment on average: the workers over the segments (a
// segment's page-heads are its sequence's pages; lengths are on the device,
// so equal lengths are assumed).  Each group of 32 threads loads eight
// contributors per round; the width gives about one round.
cudaError_t launch_merge(const DecodeParams &p, cudaStream_t s)
{
    const long long segments = static_cast<long long>(p.batch) * p.hkv * p.row_groups;
    const long long per_segment = segments > 0 ? (p.num_workers + segments - 1) / segments : 1;
    if (per_segment > 8 * 16)
        return launch_merge_width<1024>(p, s);
    if (per_segment > 8 * 8)
        return launch_merge_width<512>(p, s);
    if (per_segment > 8 * 4)
        return launch_merge_width<256>(p, s);
    if (per_segment > 8 * 2)
        return launch_merge_width<128>(p, s);
    return launch_merge_width<64>(p, s);
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

// Two partial slots per warp worker.
size_t decode_workspace_bytes(int num_workers)
{
    if (num_workers <= 0)
        num_workers = default_num_workers();
    return 2 * static_cast<size_t>(num_workers) * kPartialFloats * sizeof(float);
}

} // namespace nvfp4kv
