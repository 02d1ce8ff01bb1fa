// Split-KV GQA decode over a paged KV cache, shared by the NVFP4 and the FP8
// kernels (only the staging of a page-head and its dequantisation differ).
//
// Method: "SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation:
// the decode path dequantises the cached keys and values inside the attention
// kernel instead of expanding the cache first.  The split-KV scheme (partial
// softmax states merged with the log-sum-exp rule) is flash-decoding.
//
// Work decomposition.  A "page-head" is one page of one kv head of one
// sequence: 16 tokens.  Page-heads are numbered sequence-major, then kv head,
// then page, so the page-heads of one (sequence, kv head) pair -- a "segment"
// -- are contiguous.  The T page-heads are split evenly over NW warp workers:
// worker w takes [T*w/NW, T*(w+1)/NW).  Each warp stages its page-heads through
// its own ring of shared-memory buffers filled by TMA (lane 0 issues), and
// computes for the g <= 8 query heads of the kv head:
//   S^T[16 tok x 8 heads] = K[16 x 128] . Q^T          (8 x mma m16n8k16)
//   online softmax (fp32, exp2 domain, lazy rescale)
//   O^T[128 x 8]        += V^T[128 x 16] . P^T[16 x 8]  (8 x mma m16n8k16)
// with K/V dequantised to fp16 in registers (exact) and P in fp16.  A segment
// that one worker covers completely is normalised and written directly; the
// others leave (O, m, l) partials in the workspace for the merge kernel.
#pragma once

#include "device_common.cuh"
#include "nvfp4kv.h"

namespace nvfp4kv {

constexpr uint32_t kWaitLimit = 1u << 22;  // polls before a staged-data wait gives up
constexpr float kLazyRescale = 8.0f;       // rescale O only when the max grows by > 2^8

__device__ __forceinline__ int clamp_len(int L, int max_len)
{
    return L < 0 ? 0 : (L > max_len ? max_len : L);
}

// prefix[b] = sum over b' < b of hkv * ceil(len_b' / 16), for b in [0, batch].
// Whole CTA; blockDim.x a multiple of 32, at most 32 warps.
__device__ __forceinline__ void build_prefix(const int32_t *seq_lens, int batch, int hkv, int max_len,
                                             int32_t *prefix, int32_t *scratch, int32_t *dev_status)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < batch; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int v = 0;
        if (b < batch) {
            int L = seq_lens[b];
            if (L < 0 || L > max_len) {
                report(dev_status, NVFP4KV_DEV_BAD_LEN);
                L = clamp_len(L, max_len);
            }
            v = hkv * ((L + kPageSize - 1) / kPageSize);
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            scratch[warp] = x;
        __syncthreads();
        int before = 0, total = 0;
        for (int i = 0; i < nwarps; ++i) {
            const int s = scratch[i];
            total += s;
            if (i < warp)
                before += s;
        }
        if (b < batch)
            prefix[b] = carry + before + x - v;
        carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0)
        prefix[batch] = carry;
    __syncthreads();
}

// Largest b with prefix[b] <= j, for 0 <= j < prefix[batch].
__device__ __forceinline__ int find_seq(const int32_t *prefix, int batch, int j)
{
    int lo = 0, hi = batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= j)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Worker that owns page-head index x (balanced split of T over NW).
__device__ __forceinline__ int owner_of(long long x, long long T, long long NW)
{
    return static_cast<int>(((x + 1) * NW + T - 1) / T) - 1;
}

// Partial slot of worker w for the segment starting at seg_begin: its first
// segment uses slot 2w, its last one 2w + 1.
__device__ __forceinline__ int partial_slot(int w, int seg_begin, long long T, long long NW)
{
    const int lo_w = static_cast<int>((T * w) / NW);
    return 2 * w + (lo_w >= seg_begin ? 0 : 1);
}

// Logical token row -> physical token of the page (bit 0 ^= bit 1).  Used for
// both QK rows and PV columns so the two stay consistent; it spreads the rows a
// warp touches over different shared-memory banks.
__device__ __forceinline__ int tok_perm(int t)
{
    return t ^ ((t >> 1) & 1);
}

// ---- per-format page staging and dequantisation ----------------------------

// Shared-memory byte offsets a lane reads inside one stage; they depend only on
// the lane, so they are computed once.
struct LaneOffsets {
    uint32_t k[4];    // K data (NVFP4: rows A, B; FP8: rows A, A, B, B chunks)
    uint32_t ks[2];   // K scales (NVFP4)
    uint32_t v[4];    // V data of tokens t0, t1, t0+8, t1+8
    uint32_t vs[4];   // V scales (NVFP4)
    int tt[4];        // physical tokens of the V reads
    int tA;           // physical token of logical QK row gid (row gid+8 is tA+8)
};

// NVFP4: a page-head stages K data (16 rows x 64 B), V data (same), both via
// TMA with the 64-byte swizzle, and K / V scales (16 x 8 B) via bulk copies.
struct Nvfp4Format {
    static constexpr int kStages = 5;
    static constexpr int kTileBytes = 1024;
    static constexpr int kStageData = 2 * kTileBytes;
    static constexpr int kStageScale = 256;
    static constexpr uint32_t kStageTx = 2 * kTileBytes + 2 * 128;

    // Byte offset of 16-byte chunk c of 64-byte row t in a tile written with
    // the 64-byte swizzle (address bits [5:4] ^= bits [8:7]).  With tok_perm
    // the K reads (two rows of one 128-byte line per quarter warp) and the V
    // reads (rows 0,3,4,7 or 1,2,5,6 per half warp) are free of bank conflicts.
    __device__ static __forceinline__ uint32_t sw(int t, int c)
    {
        return (t << 6) + ((c ^ ((t >> 1) & 3)) << 4);
    }

    __device__ static __forceinline__ LaneOffsets offsets(int gid, int tig)
    {
        LaneOffsets o;
        o.tA = tok_perm(gid);
        const int tB = o.tA + 8;
        o.k[0] = sw(o.tA, tig);
        o.k[1] = sw(tB, tig);
        o.k[2] = o.k[3] = 0;
        o.ks[0] = o.tA * 8 + 2 * tig;
        o.ks[1] = tB * 8 + 2 * tig;
        const int t0 = tok_perm(2 * tig), t1 = tok_perm(2 * tig + 1);
        const int tt[4] = {t0, t1, t0 + 8, t1 + 8};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o.tt[i] = tt[i];
            o.v[i] = kTileBytes + sw(tt[i], gid >> 1) + ((gid & 1) << 3);
            o.vs[i] = 128 + tt[i] * 8 + gid;
        }
        return o;
    }

    // K fragments of logical rows gid (fa) and gid+8 (fb): f16x2 of channels
    // 32*tig + 2m, 2m+1 for m = 0..15.
    __device__ static __forceinline__ void load_k(uint32_t data, uint32_t scale, const LaneOffsets &o,
                                                  uint32_t (&fa)[16], uint32_t (&fb)[16])
    {
        const uint4 ka = lds128(data + o.k[0]);
        const uint4 kb = lds128(data + o.k[1]);
        const uint32_t sa = e4m3x2_to_f16x2(lds_u16(scale + o.ks[0]));
        const uint32_t sb = e4m3x2_to_f16x2(lds_u16(scale + o.ks[1]));
        const uint32_t sa0 = __byte_perm(sa, 0, 0x1010), sa1 = __byte_perm(sa, 0, 0x3232);
        const uint32_t sb0 = __byte_perm(sb, 0, 0x1010), sb1 = __byte_perm(sb, 0, 0x3232);
        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w};
        const uint32_t wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e2m1x8_to_f16x2x4(wa[i], fa[4 * i], fa[4 * i + 1], fa[4 * i + 2], fa[4 * i + 3]);
            e2m1x8_to_f16x2x4(wb[i], fb[4 * i], fb[4 * i + 1], fb[4 * i + 2], fb[4 * i + 3]);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            fa[m] = hmul2(fa[m], m < 8 ? sa0 : sa1);
            fb[m] = hmul2(fb[m], m < 8 ? sb0 : sb1);
        }
    }

    // V^T A-fragments for the 8 m-tiles: tile j, row gid <-> channel
    // 16*gid + 2j, row gid+8 <-> 16*gid + 2j + 1; columns = logical tokens
    // (2tig, 2tig+1) in a0/a1 and (2tig+8, 2tig+9) in a2/a3.
    __device__ static __forceinline__ void load_v(uint32_t data, uint32_t scale, const LaneOffsets &o,
                                                  int valid, uint32_t (&va)[8][4])
    {
        uint2 v[4];
        uint32_t s[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = lds64(data + o.v[i]);
            s[i] = lds_u8(scale + o.vs[i]);
        }
        if (valid < kPageSize) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (o.tt[i] >= valid) {
                    v[i] = make_uint2(0u, 0u);
                    s[i] = 0u;
                }
        }
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            const uint2 x = v[2 * pr], y = v[2 * pr + 1];
            const uint32_t sp = e4m3x2_to_f16x2(s[2 * pr] | (s[2 * pr + 1] << 8));
            // nibble interleave: byte k of E = (x ch 2k | y ch 2k << 4), O = odd channels
            const uint32_t E0 = (x.x & 0x0F0F0F0Fu) | ((y.x << 4) & 0xF0F0F0F0u);
            const uint32_t O0 = ((x.x >> 4) & 0x0F0F0F0Fu) | (y.x & 0xF0F0F0F0u);
            const uint32_t E1 = (x.y & 0x0F0F0F0Fu) | ((y.y << 4) & 0xF0F0F0F0u);
            const uint32_t O1 = ((x.y >> 4) & 0x0F0F0F0Fu) | (y.y & 0xF0F0F0F0u);
            uint32_t e0[4], o0[4], e1[4], o1[4];
            e2m1x8_to_f16x2x4(E0, e0[0], e0[1], e0[2], e0[3]);
            e2m1x8_to_f16x2x4(O0, o0[0], o0[1], o0[2], o0[3]);
            e2m1x8_to_f16x2x4(E1, e1[0], e1[1], e1[2], e1[3]);
            e2m1x8_to_f16x2x4(O1, o1[0], o1[1], o1[2], o1[3]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                va[k][2 * pr] = hmul2(e0[k], sp);
                va[k][2 * pr + 1] = hmul2(o0[k], sp);
                va[k + 4][2 * pr] = hmul2(e1[k], sp);
                va[k + 4][2 * pr + 1] = hmul2(o1[k], sp);
            }
        }
    }
};

// FP8: a page-head stages K and V data (16 rows x 128 B each) via TMA with the
// 128-byte swizzle (address bits [6:4] ^= bits [9:7]); values are E4M3 at
// scale 1.0.
struct Fp8Format {
    static constexpr int kStages = 3;
    static constexpr int kTileBytes = 2048;
    static constexpr int kStageData = 2 * kTileBytes;
    static constexpr int kStageScale = 0;
    static constexpr uint32_t kStageTx = 2 * kTileBytes;

    __device__ static __forceinline__ uint32_t sw(int t, int c)
    {
        return (t << 7) + ((c ^ (t & 7)) << 4);
    }

    __device__ static __forceinline__ LaneOffsets offsets(int gid, int tig)
    {
        LaneOffsets o;
        o.tA = tok_perm(gid);
        const int tB = o.tA + 8;
        o.k[0] = sw(o.tA, 2 * tig);
        o.k[1] = sw(o.tA, 2 * tig + 1);
        o.k[2] = sw(tB, 2 * tig);
        o.k[3] = sw(tB, 2 * tig + 1);
        o.ks[0] = o.ks[1] = 0;
        const int t0 = tok_perm(2 * tig), t1 = tok_perm(2 * tig + 1);
        const int tt[4] = {t0, t1, t0 + 8, t1 + 8};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o.tt[i] = tt[i];
            o.v[i] = kTileBytes + sw(tt[i], gid);
            o.vs[i] = 0;
        }
        return o;
    }

    __device__ static __forceinline__ void load_k(uint32_t data, uint32_t, const LaneOffsets &o,
                                                  uint32_t (&fa)[16], uint32_t (&fb)[16])
    {
        const uint4 a0 = lds128(data + o.k[0]), a1 = lds128(data + o.k[1]);
        const uint4 b0 = lds128(data + o.k[2]), b1 = lds128(data + o.k[3]);
        const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            e4m3x4_to_f16x2x2(wa[i], fa[2 * i], fa[2 * i + 1]);
            e4m3x4_to_f16x2x2(wb[i], fb[2 * i], fb[2 * i + 1]);
        }
    }

    __device__ static __forceinline__ void load_v(uint32_t data, uint32_t, const LaneOffsets &o, int valid,
                                                  uint32_t (&va)[8][4])
    {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = lds128(data + o.v[i]);
        if (valid < kPageSize) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (o.tt[i] >= valid)
                    v[i] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            const uint4 x = v[2 * pr], y = v[2 * pr + 1];
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo = __byte_perm(xw[k], yw[k], 0x5140);
                const uint32_t hi = __byte_perm(xw[k], yw[k], 0x7362);
                e4m3x4_to_f16x2x2(lo, va[2 * k][2 * pr], va[2 * k][2 * pr + 1]);
                e4m3x4_to_f16x2x2(hi, va[2 * k + 1][2 * pr], va[2 * k + 1][2 * pr + 1]);
            }
        }
    }
};

template <class Fmt>
__host__ __device__ constexpr size_t decode_smem_fixed()
{
    return 1024 /* alignment slack */ +
           static_cast<size_t>(kDecodeWarps) * Fmt::kStages * (Fmt::kStageData + Fmt::kStageScale + 8) +
           8 * sizeof(int32_t);
}

template <class Fmt>
size_t decode_smem_bytes(int batch)
{
    return decode_smem_fixed<Fmt>() + static_cast<size_t>(batch + 1) * sizeof(int32_t);
}

// ---- the decode kernel -------------------------------------------------------

template <class Fmt>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    constexpr int S = Fmt::kStages;
    uint8_t *data_base = smem;
    uint8_t *scale_base = data_base + kDecodeWarps * S * Fmt::kStageData;
    uint64_t *bars = reinterpret_cast<uint64_t *>(scale_base + kDecodeWarps * S * Fmt::kStageScale);
    int32_t *scratch = reinterpret_cast<int32_t *>(bars + kDecodeWarps * S);
    int32_t *prefix = scratch + 8;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const uint32_t wdata = smem_addr(data_base) + warp * S * Fmt::kStageData;
    const uint32_t wscale = smem_addr(scale_base) + warp * S * Fmt::kStageScale;
    const uint32_t wbar = smem_addr(bars) + warp * S * 8;

    if (lane == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(wbar + 8 * s, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // everything below reads data the previous kernel in the stream may write
    pdl_wait();
    const int max_len = p.max_pages * kPageSize;
    build_prefix(p.seq_lens, p.batch, p.hkv, max_len, prefix, scratch,
                 blockIdx.x == 0 ? p.dev_status : nullptr);

    const int w = blockIdx.x * kDecodeWarps + warp;
    if (w >= p.num_workers)
        return;
    const long long T = prefix[p.batch];
    const long long NW = p.num_workers;
    const int lo = static_cast<int>((T * w) / NW);
    const int hi = static_cast<int>((T * (w + 1)) / NW);
    if (lo >= hi)
        return;

    // ---- producer: page-head lookahead window, lane l holds index win + l ----
    int win = lo;
    int cur_phys = 0, cur_h = 0, nxt_phys = 0, nxt_h = 0;
    auto lookup = [&](int j, int &phys, int &hh) {
        phys = 0;
        hh = 0;
        if (j < hi) {
            const int b = find_seq(prefix, p.batch, j);
            const int r = j - prefix[b];
            const int n = (prefix[b + 1] - prefix[b]) / p.hkv;
            hh = r / n;
            const int pg = r - hh * n;
            phys = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pg);
        }
    };
    lookup(win + lane, cur_phys, cur_h);
    lookup(win + 32 + lane, nxt_phys, nxt_h);

    // Stage `st` receives page-head j (called by the whole warp, in order of j).
    auto issue = [&](int j, int st) {
        int rel = j - win;
        if (rel >= 32) {
            win += 32;
            rel -= 32;
            cur_phys = nxt_phys;
            cur_h = nxt_h;
            lookup(win + 32 + lane, nxt_phys, nxt_h);
        }
        int phys = __shfl_sync(kFullMask, cur_phys, rel);
        const int hh = __shfl_sync(kFullMask, cur_h, rel);
        if (lane == 0) {
            if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_pages)) {
                report(p.dev_status, NVFP4KV_DEV_BAD_PAGE);
                phys = 0;
            }
            const uint32_t bar = wbar + 8 * st;
            const int z = phys * p.hkv + hh;
            mbar_arrive_expect_tx(bar, Fmt::kStageTx);
            tma_load_3d(wdata + st * Fmt::kStageData, &tmap_k, 0, 0, z, bar);
            tma_load_3d(wdata + st * Fmt::kStageData + Fmt::kTileBytes, &tmap_v, 0, 0, z, bar);
            if constexpr (Fmt::kStageScale > 0) {
                bulk_g2s(wscale + st * Fmt::kStageScale, p.k_scale + static_cast<size_t>(z) * 128, 128, bar);
                bulk_g2s(wscale + st * Fmt::kStageScale + 128, p.v_scale + static_cast<size_t>(z) * 128, 128,
                         bar);
            }
        }
    };

    // ---- consumer bookkeeping (warp-uniform) ----
    int b = find_seq(prefix, p.batch, lo);
    int n = (prefix[b + 1] - prefix[b]) / p.hkv;
    int h = (lo - prefix[b]) / n;
    int pg = lo - prefix[b] - h * n;
    int L = clamp_len(p.seq_lens[b], max_len);
    int seg_begin = prefix[b] + h * n;

    const int npro = min(S, hi - lo);
    for (int j = lo; j < lo + npro; ++j)
        issue(j, j - lo);

    uint32_t qf[16];
    float m0, m1, l0, l1;
    float oacc[8][4];
    const int g = p.group;
    const LaneOffsets off = Fmt::offsets(gid, tig);

    auto start_segment = [&]() {
        if (gid < g) {
            const uint4 *qrow = reinterpret_cast<const uint4 *>(
                p.q + (static_cast<size_t>(b) * p.hq + h * g + gid) * kHeadDim + 32 * tig);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 r = __ldg(qrow + i);
                const uint32_t ww[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo_f = __uint_as_float(ww[k] << 16) * p.qscale;
                    const float hi_f = __uint_as_float(ww[k] & 0xffff0000u) * p.qscale;
                    qf[4 * i + k] = pack_f16x2(lo_f, hi_f);
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                qf[k] = 0u;
        }
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                oacc[j][e] = 0.f;
    };

    auto finish_segment = [&]() {
        float L0 = l0, L1 = l1;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            L0 += __shfl_xor_sync(kFullMask, L0, o);
            L1 += __shfl_xor_sync(kFullMask, L1, o);
        }
        const bool owned = seg_begin >= lo && seg_begin + n <= hi;
        const int hA = 2 * tig, hB = hA + 1;
        if (owned) {
            const float r0 = 1.f / L0, r1 = 1.f / L1;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const int head = which ? hB : hA;
                if (head >= g)
                    continue;
                const float r = which ? r1 : r0;
                const size_t o = (static_cast<size_t>(b) * p.hq + h * g + head) * kHeadDim + 16 * gid;
                float v[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[2 * j] = oacc[j][which] * r;
                    v[2 * j + 1] = oacc[j][2 + which] * r;
                }
                if (p.out_bf16) {
                    uint32_t pk[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                        pk[k] = *reinterpret_cast<uint32_t *>(&t);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + o);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                }
            }
        } else {
            float *slot = p.partials + static_cast<size_t>(partial_slot(w, seg_begin, T, NW)) * kPartialFloats;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const int head = which ? hB : hA;
                float4 *dst = reinterpret_cast<float4 *>(slot + head * kHeadDim + 16 * gid);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    dst[k] = make_float4(oacc[2 * k][which], oacc[2 * k][2 + which], oacc[2 * k + 1][which],
                                         oacc[2 * k + 1][2 + which]);
            }
            if (gid == 0) {
                slot[kMaxGroup * kHeadDim + hA] = m0;
                slot[kMaxGroup * kHeadDim + hB] = m1;
                slot[kMaxGroup * kHeadDim + kMaxGroup + hA] = L0;
                slot[kMaxGroup * kHeadDim + kMaxGroup + hB] = L1;
            }
        }
    };

    start_segment();

    int st = 0;            // ring stage of page-head j
    uint32_t ph = 0;       // phase parity of that stage's barrier
    for (int j = lo; j < hi; ++j) {
        // Lanes poll independently and may leave the loop at different polls;
        // the vote reconverges the warp before the warp-wide MMAs below and
        // makes the give-up decision uniform.
        const bool arrived = mbar_wait_bounded(wbar + 8 * st, ph, kWaitLimit);
        if (!__all_sync(kFullMask, arrived)) {
            // staged data never arrived: report, let the copies in flight land, stop
            if (lane == 0)
                report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
            const int pending = min(S, hi - j);
            for (int k = 0; k < pending; ++k) {
                int s2 = st + k;
                uint32_t p2 = ph;
                if (s2 >= S) {
                    s2 -= S;
                    p2 ^= 1u;
                }
                mbar_wait_bounded(wbar + 8 * s2, p2, kWaitLimit);
            }
            return;
        }
        const int valid = (pg == n - 1) ? (L - pg * kPageSize) : kPageSize;
        const uint32_t sdata = wdata + st * Fmt::kStageData;
        const uint32_t sscale = wscale + st * Fmt::kStageScale;

        // S^T = K . Q^T
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t fa[16], fb[16];
            Fmt::load_k(sdata, sscale, off, fa, fb);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_f16_16816(sc, fa[2 * s], fb[2 * s], fa[2 * s + 1], fb[2 * s + 1], qf[2 * s], qf[2 * s + 1]);
        }
        if (valid < kPageSize) {
            if (off.tA >= valid)
                sc[0] = sc[1] = -INFINITY;
            if (off.tA + 8 >= valid)
                sc[2] = sc[3] = -INFINITY;
        }
        // Online softmax, heads (2tig, 2tig+1).  The running maximum is only
        // moved when some score exceeds it by more than 2^kLazyRescale, so the
        // common page needs no cross-lane reduction; P then stays <= 2^8.
        float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
        if (__any_sync(kFullMask, (mx0 > m0 + kLazyRescale) || (mx1 > m1 + kLazyRescale))) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, o));
            }
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float a0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - n0);
            const float a1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - n1);
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                oacc[jj][0] *= a0;
                oacc[jj][1] *= a1;
                oacc[jj][2] *= a0;
                oacc[jj][3] *= a1;
            }
            m0 = n0;
            m1 = n1;
        }
        const float p0 = fast_exp2(sc[0] - m0), p1 = fast_exp2(sc[1] - m1);
        const float p2 = fast_exp2(sc[2] - m0), p3 = fast_exp2(sc[3] - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2, p3));

        // O^T += V^T . P^T
        {
            uint32_t va[8][4];
            Fmt::load_v(sdata, sscale, off, valid, va);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                mma_f16_16816(oacc[jj], va[jj][0], va[jj][1], va[jj][2], va[jj][3], pb0, pb1);
        }

        __syncwarp();
        if (j + S < hi)
            issue(j + S, st);
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }

        ++pg;
        if (pg == n || j + 1 == hi) {
            finish_segment();
            if (j + 1 < hi) {
                ++h;
                pg = 0;
                if (h == p.hkv) {
                    h = 0;
                    do {
                        ++b;
                    } while (prefix[b + 1] == prefix[b]);
                    n = (prefix[b + 1] - prefix[b]) / p.hkv;
                    L = clamp_len(p.seq_lens[b], max_len);
                }
                seg_begin = prefix[b] + h * n;
                start_segment();
            }
        }
    }
    pdl_launch_dependents();
}

// ---- split merge ---------------------------------------------------------------
// One CTA of kMergeThreads threads per (sequence, kv head, query head of the
// group).  Segments that one worker covered were written by the decode kernel;
// empty sequences get zeros here.
constexpr int kMergeThreads = 256;
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p);

} // namespace nvfp4kv
