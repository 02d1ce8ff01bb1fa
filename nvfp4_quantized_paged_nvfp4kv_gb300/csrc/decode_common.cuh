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
// worker w takes [T*w/NW, T*(w+1)/NW).  Each warp stages its page-head records
// through its own ring of shared-memory buffers, one bulk copy per record
// (lane 0 issues), and computes for the g <= 8 query heads of the kv head:
//   S^T[16 tok x 8 heads] = K[16 x 128] . Q^T          (8 x mma m16n8k16)
//   online softmax (fp32, exp2 domain, lazy rescale)
//   O^T[128 x 8]        += V^T[128 x 16] . P^T[16 x 8]  (8 x mma m16n8k16)
// with K/V dequantised to fp16 in registers (exact) and P in fp16.  A segment
// that one worker covers completely is normalised and written directly; the
// others leave (O, m, l) partials in the workspace for the merge kernel.
#pragma once

#include <type_traits>

#include "device_common.cuh"
#include "nvfp4kv.h"
#include "record_write.cuh"

namespace nvfp4kv {

// The running max is moved only when a score exceeds it by more than this
// (log2 units), so P <= 2^7 and its fp16 rounding stays relative (far from the
// fp16 overflow and subnormal ranges for the terms that matter).
constexpr float kLazyRescale = 7.0f;

__device__ __forceinline__ int clamp_len(int L, int max_len)
{
    return L < 0 ? 0 : (L > max_len ? max_len : L);
}

// Slots of the warp-sum scratch that build_prefix needs: one per warp of the
// CTA, for any CTA of up to 32 warps.
constexpr int kPrefixScratch = 32;
static_assert(kDecodeWarps <= kPrefixScratch, "build_prefix takes one scratch slot per warp");

// prefix[b] = sum over b' < b of hkv * ceil(len_b' / 16), for b in [0, batch].
// Whole CTA; blockDim.x a multiple of 32, at most 32 warps; scratch holds
// kPrefixScratch slots and must not overlap prefix.
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

// Workers that take part: never more than there are page-heads, so that every
// worker's range [T*w/NW, T*(w+1)/NW) is non-empty and the contributors to a
// segment are exactly the workers owner_of(first) .. owner_of(last).
__device__ __forceinline__ long long effective_workers(int num_workers, long long T)
{
    return num_workers < T ? num_workers : (T > 0 ? T : 1);
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

// ---- per-format page staging and dequantisation ----------------------------
//
// A warp stages one whole page-head record (layout in include/nvfp4kv.h) with a
// single bulk copy and reads it from shared memory.  Lane (gid = lane/4,
// tig = lane%4) holds the MMA fragments:
//   QK^T  A = K rows gid and gid+8 (tokens), channels 32*tig .. 32*tig + 31;
//         B = Q^T, the same 32 channels of query head gid.
//   PV    A = V^T, columns (tokens) 2tig, 2tig+1 (a0/a1) and 2tig+8, 2tig+9
//         (a2/a3); the channel of m-tile j, row r is Fmt::channel(j, r).
// The record arrangement (chosen by the writer) makes every shared-memory read
// below conflict-free and hands cvt.f16x2 the two tokens of a V column pair in
// one byte (NVFP4) or one 16-bit unit (FP8).

struct LaneOffsets {
    uint32_t k[4];    // K data (NVFP4: rows gid, gid+8; FP8: rows gid, gid+8, two chunks each)
    uint32_t ks[2];   // K scales of rows gid, gid+8 (NVFP4)
    uint32_t v[4];    // V data (NVFP4: rows tig, tig+4; FP8: two chunks of each)
    uint32_t vs[2];   // V scale rows tig, tig+4 (NVFP4)
};

struct Nvfp4Format {
    static constexpr int kStages = 5;
    static constexpr int kRecord = 2304;

    // x as left by divide_by_tensor_scale, whose code flip comes with it
    __device__ static __forceinline__ void write_block(uint8_t *rec, bool is_v, int tok, int blk,
                                                       const float (&x)[16], uint32_t flip)
    {
        write_nvfp4_block(rec, is_v, tok, blk, x, ScaleOfByte(), flip);
    }

    // m-tile j, row r (0..15) is channel 16j + r: each m-tile is one scale block.
    __device__ static __forceinline__ int channel(int j, int gid, int w) { return 16 * j + gid + 8 * w; }

    __device__ static __forceinline__ LaneOffsets offsets(int gid, int tig)
    {
        LaneOffsets o;
        o.k[0] = gid * 64 + 16 * tig;
        o.k[1] = o.k[0] + 512;
        o.k[2] = o.k[3] = 0;
        o.ks[0] = 2048 + gid * 8 + 2 * tig;
        o.ks[1] = o.ks[0] + 64;
        o.v[0] = 1024 + tig * 128 + ((gid + 2 * tig) & 7) * 16;
        o.v[1] = o.v[0] + 512;                           // row tig + 4, same chunk position
        o.v[2] = o.v[3] = 0;
        o.vs[0] = 2176 + tig * 16;
        o.vs[1] = o.vs[0] + 64;
        return o;
    }

    // K fragments of rows gid (fa) and gid+8 (fb): f16x2 of channels
    // 32*tig + 2m, 2m+1 for m = 0..15, scaled exactly.
    __device__ static __forceinline__ void load_k(uint32_t rec, const LaneOffsets &o, uint32_t (&fa)[16],
                                                  uint32_t (&fb)[16])
    {
        const uint4 ka = lds128(rec + o.k[0]);
        const uint4 kb = lds128(rec + o.k[1]);
        const uint32_t sa = e4m3x2_to_f16x2(lds_u16(rec + o.ks[0]));
        const uint32_t sb = e4m3x2_to_f16x2(lds_u16(rec + o.ks[1]));
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

    // V^T fragments, dequantised exactly: the E2M1 value (at most two
    // significant bits) times the E4M3 block scale (four) is exact in fp16.
    // va[j][0..1] hold tokens 2tig, 2tig+1 and va[j][2..3] tokens 2tig+8,
    // 2tig+9 of m-tile j, which is scale block j; the scales of those token
    // pairs come as f16x2 from one cvt each.
    __device__ static __forceinline__ void load_v(uint32_t rec, const LaneOffsets &o, int tig, int valid,
                                                  uint32_t (&va)[8][4])
    {
        uint4 x = lds128(rec + o.v[0]), y = lds128(rec + o.v[1]);
        uint4 s0 = lds128(rec + o.vs[0]), s1 = lds128(rec + o.vs[1]);
        if (valid < kPageSize) {
            // tokens at or past `valid` read as zero codes with zero scales
            auto keep = [&](int t0, uint32_t &nib, uint32_t &byt) {
                nib = (t0 >= valid) ? 0u : ((t0 + 1 >= valid) ? 0x0F0F0F0Fu : 0xFFFFFFFFu);
                byt = (t0 >= valid) ? 0u : ((t0 + 1 >= valid) ? 0x00FF00FFu : 0xFFFFFFFFu);
            };
            uint32_t n0, b0, n1, b1;
            keep(2 * tig, n0, b0);
            keep(2 * tig + 8, n1, b1);
            x = make_uint4(x.x & n0, x.y & n0, x.z & n0, x.w & n0);
            y = make_uint4(y.x & n1, y.y & n1, y.z & n1, y.w & n1);
            s0 = make_uint4(s0.x & b0, s0.y & b0, s0.z & b0, s0.w & b0);
            s1 = make_uint4(s1.x & b1, s1.y & b1, s1.z & b1, s1.w & b1);
        }
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
        const uint32_t s0w[4] = {s0.x, s0.y, s0.z, s0.w}, s1w[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // bytes 4k .. 4k+3 = (m-tile 2k, w 0), (2k, 1), (2k+1, 0), (2k+1, 1)
            e2m1x8_to_f16x2x4(xw[k], va[2 * k][0], va[2 * k][1], va[2 * k + 1][0], va[2 * k + 1][1]);
            e2m1x8_to_f16x2x4(yw[k], va[2 * k][2], va[2 * k][3], va[2 * k + 1][2], va[2 * k + 1][3]);
            uint32_t sa, sb, sc, sd;   // scale pairs of m-tiles 2k, 2k+1 for the two token pairs
            e4m3x4_to_f16x2x2(s0w[k], sa, sb);
            e4m3x4_to_f16x2x2(s1w[k], sc, sd);
            va[2 * k][0] = hmul2(va[2 * k][0], sa);
            va[2 * k][1] = hmul2(va[2 * k][1], sa);
            va[2 * k + 1][0] = hmul2(va[2 * k + 1][0], sb);
            va[2 * k + 1][1] = hmul2(va[2 * k + 1][1], sb);
            va[2 * k][2] = hmul2(va[2 * k][2], sc);
            va[2 * k][3] = hmul2(va[2 * k][3], sc);
            va[2 * k + 1][2] = hmul2(va[2 * k + 1][2], sd);
            va[2 * k + 1][3] = hmul2(va[2 * k + 1][3], sd);
        }
    }
};

struct Fp8Format {
    static constexpr int kStages = 3;
    static constexpr int kRecord = 4096;

    // (the FP8 cache has no tensor scale: x is the row itself, flip kCodeFlip)
    __device__ static __forceinline__ void write_block(uint8_t *rec, bool is_v, int tok, int blk,
                                                       const float (&x)[16], uint32_t)
    {
        write_fp8_block(rec, is_v, tok, blk, x);
    }

    // m-tile j: row gid is channel 16*gid + 2j, row gid+8 is 16*gid + 2j + 1.
    __device__ static __forceinline__ int channel(int j, int gid, int w) { return 16 * gid + 2 * j + w; }

    __device__ static __forceinline__ LaneOffsets offsets(int gid, int tig)
    {
        LaneOffsets o;
        const int par = gid & 1;
        o.k[0] = gid * 128 + ((2 * tig + par) & 7) * 16;
        o.k[1] = gid * 128 + ((2 * tig + 1 + par) & 7) * 16;
        o.k[2] = o.k[0] + 1024;                          // row gid + 8, same parity
        o.k[3] = o.k[1] + 1024;
        o.ks[0] = o.ks[1] = 0;
        const int f = (tig & 1) + 4 * ((tig >> 1) & 1);  // rows tig and tig+4 share f
        o.v[0] = 2048 + tig * 256 + ((2 * gid + f) & 15) * 16;
        o.v[1] = 2048 + tig * 256 + ((2 * gid + 1 + f) & 15) * 16;
        o.v[2] = o.v[0] + 1024;
        o.v[3] = o.v[1] + 1024;
        o.vs[0] = o.vs[1] = 0;
        return o;
    }

    __device__ static __forceinline__ void load_k(uint32_t rec, const LaneOffsets &o, uint32_t (&fa)[16],
                                                  uint32_t (&fb)[16])
    {
        const uint4 a0 = lds128(rec + o.k[0]), a1 = lds128(rec + o.k[1]);
        const uint4 b0 = lds128(rec + o.k[2]), b1 = lds128(rec + o.k[3]);
        const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            e4m3x4_to_f16x2x2(wa[i], fa[2 * i], fa[2 * i + 1]);
            e4m3x4_to_f16x2x2(wb[i], fb[2 * i], fb[2 * i + 1]);
        }
    }

    __device__ static __forceinline__ void load_v(uint32_t rec, const LaneOffsets &o, int tig, int valid,
                                                  uint32_t (&va)[8][4])
    {
        uint4 x0 = lds128(rec + o.v[0]), x1 = lds128(rec + o.v[1]);
        uint4 y0 = lds128(rec + o.v[2]), y1 = lds128(rec + o.v[3]);
        if (valid < kPageSize) {
            auto keep = [&](int t0) {
                return (t0 >= valid) ? 0u : ((t0 + 1 >= valid) ? 0x00FF00FFu : 0xFFFFFFFFu);
            };
            const uint32_t m0 = keep(2 * tig), m1 = keep(2 * tig + 8);
            x0 = make_uint4(x0.x & m0, x0.y & m0, x0.z & m0, x0.w & m0);
            x1 = make_uint4(x1.x & m0, x1.y & m0, x1.z & m0, x1.w & m0);
            y0 = make_uint4(y0.x & m1, y0.y & m1, y0.z & m1, y0.w & m1);
            y1 = make_uint4(y1.x & m1, y1.y & m1, y1.z & m1, y1.w & m1);
        }
        const uint32_t x0w[4] = {x0.x, x0.y, x0.z, x0.w}, x1w[4] = {x1.x, x1.y, x1.z, x1.w};
        const uint32_t y0w[4] = {y0.x, y0.y, y0.z, y0.w}, y1w[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // word k: channels 16gid + 2k (tokens t0, t1) and 16gid + 2k + 1
            e4m3x4_to_f16x2x2(x0w[k], va[k][0], va[k][1]);
            e4m3x4_to_f16x2x2(x1w[k], va[k + 4][0], va[k + 4][1]);
            e4m3x4_to_f16x2x2(y0w[k], va[k][2], va[k][3]);
            e4m3x4_to_f16x2x2(y1w[k], va[k + 4][2], va[k + 4][3]);
        }
    }
};

template <class Fmt>
__host__ __device__ constexpr size_t decode_smem_fixed()
{
    return 128 /* alignment slack */ + static_cast<size_t>(kDecodeWarps) * Fmt::kStages * (Fmt::kRecord + 8) +
           kPrefixScratch * sizeof(int32_t);
}

template <class Fmt>
size_t decode_smem_bytes(int batch)
{
    return decode_smem_fixed<Fmt>() + static_cast<size_t>(batch + 1) * sizeof(int32_t);
}

// one CTA per SM: the staging rings of all its warps plus the largest prefix table
static_assert(decode_smem_fixed<Nvfp4Format>() + (kMaxBatch + 1) * sizeof(int32_t) <= 227 * 1024,
              "NVFP4 decode shared memory");
static_assert(decode_smem_fixed<Fp8Format>() + (kMaxBatch + 1) * sizeof(int32_t) <= 227 * 1024,
              "FP8 decode shared memory");

// ---- the decode kernel -------------------------------------------------------

// Output element offset of query row r (0 .. rows-1) of kv head hp, sequence b:
// row r is query token r / group, head r % group of the kv head's group.
__device__ __forceinline__ size_t out_row(const DecodeParams &p, int b, int hp, int r)
{
    const int t = r / p.group, i = r - t * p.group;
    return ((static_cast<size_t>(b) * p.q_len + t) * p.hq + hp * p.group + i) * kHeadDim;
}

// kMulti: several query tokens per sequence.  A segment is then one row group
// of one kv head ("virtual heads" hkv * row_groups per sequence), numbered
// with the row group innermost so that the row groups of a kv head read the
// same pages close together in time.
template <class Fmt, bool kMulti = false>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeCtasPerSm) decode_kernel(const __grid_constant__ DecodeParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((128u - (raw_addr & 127u)) & 127u);
    constexpr int S = Fmt::kStages;
    constexpr int R = Fmt::kRecord;
    uint8_t *data_base = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(data_base + kDecodeWarps * S * R);
    int32_t *scratch = reinterpret_cast<int32_t *>(bars + kDecodeWarps * S);
    int32_t *prefix = scratch + kPrefixScratch;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const uint32_t wdata = smem_addr(data_base) + warp * S * R;
    const uint32_t wbar = smem_addr(bars) + warp * S * 8;

    if (lane == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(wbar + 8 * s, 1);
        fence_mbar_init();
    }
    // The merge kernel that follows may start its own prologue meanwhile.
    pdl_launch_dependents();
    // The work split and the block-table lookups read only the lengths and the
    // block table, which no kernel of this library writes; they run before the
    // wait for the previous kernel in the stream, overlapping its tail.  The
    // cache records, q, the new K/V, the output and the workspace are touched
    // only after the wait.
    const int max_len = p.max_pages * kPageSize;
    const int nseg = kMulti ? p.hkv * p.row_groups : p.hkv;   // segments per sequence
    build_prefix(p.seq_lens, p.batch, nseg, max_len, prefix, scratch,
                 blockIdx.x == 0 ? p.dev_status : nullptr);

    const int w = blockIdx.x * kDecodeWarps + warp;
    const long long T = prefix[p.batch];
    const long long NW = effective_workers(p.num_workers, T);
    const int lo = w < NW ? static_cast<int>((T * w) / NW) : 0;
    const int hi = w < NW ? static_cast<int>((T * (w + 1)) / NW) : 0;

    // The worker: this warp's page-heads [lo, hi).
    auto run_worker = [&]() {
    if (lo >= hi)
        return;

    // ---- producer: page-head lookahead window, lane l holds index win + l ----
    // Lane l looks up page-head win + l of the current window and of the next
    // one; a window's entries are checked and turned into record indices
    // (page * hkv + head) when it becomes current, long after its block-table
    // reads were issued.
    int win = lo;
    int nxt_phys = 0, nxt_h = 0;
    uint32_t cur_rec = 0;
    auto lookup = [&](int j, int &phys, int &hh) {
        phys = 0;
        hh = 0;
        if (j < hi) {
            const int b = find_seq(prefix, p.batch, j);
            const int r = j - prefix[b];
            const int n = (prefix[b + 1] - prefix[b]) / nseg;
            hh = r / n;
            const int pg = r - hh * n;
            if constexpr (kMulti)
                hh /= p.row_groups;                  // the kv head of the row group
            phys = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pg);
        }
    };
    auto record_of = [&](int phys, int hh, int j) {
        if (j < hi && static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_pages)) {
            report(p.dev_status, NVFP4KV_DEV_BAD_PAGE);
            phys = 0;
        }
        return static_cast<uint32_t>(phys) * static_cast<uint32_t>(p.hkv) + static_cast<uint32_t>(hh);
    };
    {
        int phys, hh;
        lookup(win + lane, phys, hh);
        lookup(win + 32 + lane, nxt_phys, nxt_h);
        cur_rec = record_of(phys, hh, win + lane);
    }

    // Stage `st` receives page-head j (called by the whole warp, in order of j).
    auto issue = [&](int j, int st) {
        int rel = j - win;
        if (rel >= 32) {
            win += 32;
            rel -= 32;
            cur_rec = record_of(nxt_phys, nxt_h, win + lane);
            lookup(win + 32 + lane, nxt_phys, nxt_h);
        }
        const uint32_t z = __shfl_sync(kFullMask, cur_rec, rel);
        if (lane == 0) {
            const uint32_t bar = wbar + 8 * st;
            mbar_arrive_expect_tx(bar, R);
            bulk_g2s(wdata + st * R, p.pool + static_cast<size_t>(z) * R, R, bar);
        }
    };

    // ---- consumer bookkeeping (warp-uniform) ----
    int b = find_seq(prefix, p.batch, lo);
    int n = (prefix[b + 1] - prefix[b]) / nseg;
    int h = (lo - prefix[b]) / n;                 // segment (kv head, or row group) in the sequence
    int pg = lo - prefix[b] - h * n;
    int L = clamp_len(p.seq_lens[b], max_len);
    int seg_begin = prefix[b] + h * n;

    pdl_wait();
    // The first two records go out at once, the rest of the ring once the
    // first has landed: when every warp asks for its whole ring together,
    // each warp's first record would arrive late in that burst.  With the
    // fused append, the records before the first page that receives a new
    // token (the last page-head of the first segment, if the warp reaches
    // it) go out before the append, so the warps that append do not start
    // streaming later than the others.
    const int npro = min(S, hi - lo);
    const int app_first = (!kMulti && p.append && seg_begin + n - 1 < hi) ? seg_begin + n - 1 : hi;
    const int npre = min(min(2, npro), app_first - lo);
    for (int x = lo; x < lo + npre; ++x)
        issue(x, x - lo);
    if (!kMulti && p.append) {
        // Fused append: the warp that streams the last page-head of a segment
        // first writes that sequence's new token (position seq_len - 1) into
        // it, one 16-value block per lane, before any copy of that page.
        for (int idx = lo; idx < hi;) {
            const int bb = find_seq(prefix, p.batch, idx);
            const int nn = (prefix[bb + 1] - prefix[bb]) / p.hkv;
            const int hh = (idx - prefix[bb]) / nn;
            const int last = prefix[bb] + hh * nn + nn - 1;
            if (last < hi && lane < 16) {
                int phys = __ldg(p.block_table + static_cast<size_t>(bb) * p.max_pages + nn - 1);
                if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_pages)) {
                    if (lane == 0)
                        report(p.dev_status, NVFP4KV_DEV_BAD_PAGE);
                } else {
                    const int tok = (clamp_len(p.seq_lens[bb], max_len) - 1) & (kPageSize - 1);
                    const bool is_v = lane >= 8;
                    const int blk = lane & 7;
                    const size_t src = (static_cast<size_t>(bb) * p.hkv + hh) * kHeadDim + blk * 16;
                    float x[16];
                    if (p.new_bf16)
                        load16<true>(is_v ? p.v_new : p.k_new, src, x);
                    else
                        load16<false>(is_v ? p.v_new : p.k_new, src, x);
                    const uint32_t flip = divide_by_tensor_scale(x, head_tensor_scale(p.hs, is_v, hh, p.gscale));
                    Fmt::write_block(const_cast<uint8_t *>(p.pool) + (static_cast<size_t>(phys) * p.hkv + hh) * R,
                                     is_v, tok, blk, x, flip);
                    fence_proxy_async_global();
                }
            }
            idx = last + 1;
        }
        __syncwarp();
    }
    for (int x = lo + npre; x < lo + min(2, npro); ++x)
        issue(x, x - lo);

    uint32_t qf[16];
    float m0, m1, l0, l1;
    float oacc[8][4];
    const int g = p.group;
    const LaneOffsets off = Fmt::offsets(gid, tig);

    // multi-query: the segment's kv head and row group, and the number of
    // keys visible to this lane's two score columns (rows 2tig, 2tig + 1)
    int hp = h, rg = 0, limA = 0, limB = 0;
    auto start_segment = [&]() {
        bool has_row = gid < g;
        const uint16_t *qsrc = p.q + (static_cast<size_t>(b) * p.hq + h * g + gid) * kHeadDim;
        if constexpr (kMulti) {
            hp = h / p.row_groups;
            rg = h - hp * p.row_groups;
            const int r = rg * kMaxGroup + gid;
            has_row = r < p.rows;
            qsrc = p.q + out_row(p, b, hp, has_row ? r : 0);
            // row r is query token t = r / g at position L - q_len + t
            const int rA = rg * kMaxGroup + 2 * tig, rB = rA + 1;
            limA = rA < p.rows ? L - p.q_len + rA / g + 1 : 0;
            limB = rB < p.rows ? L - p.q_len + rB / g + 1 : 0;
        }
        if (has_row) {
            const float qsc = p.hs.per_head ? p.qs[kMulti ? hp : h] : p.qscale;
            const uint4 *qrow = reinterpret_cast<const uint4 *>(qsrc + 32 * tig);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 r = __ldg(qrow + i);
                const uint32_t ww[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo_f = __uint_as_float(ww[k] << 16) * qsc;
                    const float hi_f = __uint_as_float(ww[k] & 0xffff0000u) * qsc;
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
            // (a row that saw no key at all -- a multi-query row before its
            // first visible key -- has l = 0 and gets zeros)
            const float osc = head_tensor_scale(p.hs, true, kMulti ? hp : h, p.out_scale);
            const float r0 = L0 > 0.f ? osc / L0 : 0.f, r1 = L1 > 0.f ? osc / L1 : 0.f;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const int head = which ? hB : hA;
                size_t o = (static_cast<size_t>(b) * p.hq + h * g + head) * kHeadDim;
                if constexpr (kMulti) {
                    const int row = rg * kMaxGroup + head;   // rows beyond the group are later tokens
                    if (row >= p.rows)
                        continue;
                    o = out_row(p, b, hp, row);
                } else if (head >= g) {
                    continue;
                }
                const float r = which ? r1 : r0;
                if (p.out_bf16) {
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + o;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        dst[Fmt::channel(j, gid, 0)] = __float2bfloat16_rn(oacc[j][which] * r);
                        dst[Fmt::channel(j, gid, 1)] = __float2bfloat16_rn(oacc[j][2 + which] * r);
                    }
                } else {
                    float *dst = static_cast<float *>(p.out) + o;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        dst[Fmt::channel(j, gid, 0)] = oacc[j][which] * r;
                        dst[Fmt::channel(j, gid, 1)] = oacc[j][2 + which] * r;
                    }
                }
            }
        } else {
            float *slot = p.partials + static_cast<size_t>(2 * w + (lo >= seg_begin ? 0 : 1)) * kPartialFloats;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                float *dst = slot + (which ? hB : hA) * kHeadDim;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    dst[Fmt::channel(j, gid, 0)] = oacc[j][which];
                    dst[Fmt::channel(j, gid, 1)] = oacc[j][2 + which];
                }
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
    if (npro > 2) {
        // (a wait that gives up here gives up again, reported, in the loop)
        mbar_wait_bounded(wbar, 0, p.wait_limit);
        __syncwarp();
        for (int x = lo + 2; x < lo + npro; ++x)
            issue(x, x - lo);
    }

    // One step handles one page-head, or two of the same segment.
    auto step = [&](auto npc, uint32_t rec0, uint32_t rec1, int last_valid, int pos0) {
        constexpr int NP = decltype(npc)::value;
        // S^T = K . Q^T
        // (two accumulators per page-head halve the dependent MMA chain)
        float sc[NP][4];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            uint32_t fa[16], fb[16];
            Fmt::load_k(q == 0 ? rec0 : rec1, off, fa, fb);
            float sd[4] = {0.f, 0.f, 0.f, 0.f};
            sc[q][0] = sc[q][1] = sc[q][2] = sc[q][3] = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_f16_16816((s & 1) ? sd : sc[q], fa[2 * s], fb[2 * s], fa[2 * s + 1], fb[2 * s + 1], qf[2 * s],
                              qf[2 * s + 1]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[q][e] += sd[e];
        }
        if constexpr (kMulti) {
            // key pos0 + 16q + token against each column's visible count
            if (pos0 + NP * kPageSize > min(limA, limB)) {
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const int k0 = pos0 + q * kPageSize + gid, k1 = k0 + 8;
                    if (k0 >= limA)
                        sc[q][0] = -INFINITY;
                    if (k0 >= limB)
                        sc[q][1] = -INFINITY;
                    if (k1 >= limA)
                        sc[q][2] = -INFINITY;
                    if (k1 >= limB)
                        sc[q][3] = -INFINITY;
                }
            }
        } else if (last_valid < kPageSize) {
            if (gid >= last_valid)
                sc[NP - 1][0] = sc[NP - 1][1] = -INFINITY;
            if (gid + 8 >= last_valid)
                sc[NP - 1][2] = sc[NP - 1][3] = -INFINITY;
        }
        // Online softmax, heads (2tig, 2tig+1).  The running maximum is only
        // moved when some score exceeds it by more than kLazyRescale, so the
        // common step needs no cross-lane reduction.
        float mx0 = fmaxf(sc[0][0], sc[0][2]), mx1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
        for (int q = 1; q < NP; ++q) {
            mx0 = fmaxf(mx0, fmaxf(sc[q][0], sc[q][2]));
            mx1 = fmaxf(mx1, fmaxf(sc[q][1], sc[q][3]));
        }
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
        uint32_t pb[NP][2];
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            float p0 = fast_exp2(sc[q][0] - m0), p1 = fast_exp2(sc[q][1] - m1);
            float p2 = fast_exp2(sc[q][2] - m0), p3 = fast_exp2(sc[q][3] - m1);
            if constexpr (kMulti) {
                // a masked score against a maximum that is still -inf
                p0 = sc[q][0] == -INFINITY ? 0.f : p0;
                p1 = sc[q][1] == -INFINITY ? 0.f : p1;
                p2 = sc[q][2] == -INFINITY ? 0.f : p2;
                p3 = sc[q][3] == -INFINITY ? 0.f : p3;
            }
            ls0 += p0 + p2;
            ls1 += p1 + p3;
            pb[q][0] = movmatrix_trans(pack_f16x2(p0, p1));
            pb[q][1] = movmatrix_trans(pack_f16x2(p2, p3));
        }
        l0 += ls0;
        l1 += ls1;
        // O^T += V^T . P^T (V arrives scaled)
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            uint32_t va[8][4];
            Fmt::load_v(q == 0 ? rec0 : rec1, off, tig, q == NP - 1 ? last_valid : kPageSize, va);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                mma_f16_16816(oacc[jj], va[jj][0], va[jj][1], va[jj][2], va[jj][3], pb[q][0], pb[q][1]);
        }
    };

    int st = 0;            // ring stage of page-head j
    uint32_t ph = 0;       // phase parity of that stage's barrier
    int j = lo;
    while (j < hi) {
        const int np = (j + 1 < hi && pg + 1 < n) ? 2 : 1;
        int st1 = st + 1;
        uint32_t ph1 = ph;
        if (st1 == S) {
            st1 = 0;
            ph1 ^= 1u;
        }
        // Lanes poll independently and may leave the loop at different polls;
        // the vote reconverges the warp before the warp-wide MMAs below and
        // makes the give-up decision uniform.
        const bool arrived = np == 2 ? mbar_wait2_bounded(wbar + 8 * st, ph, wbar + 8 * st1, ph1, p.wait_limit)
                                     : mbar_wait_bounded(wbar + 8 * st, ph, p.wait_limit);
        if (!__all_sync(kFullMask, arrived)) {
            // staged data never arrived: report, let the copies in flight land
            // (at the default limit, whatever p.wait_limit is), stop
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
        const int plast = pg + np - 1;
        const int last_valid = (plast == n - 1) ? (L - plast * kPageSize) : kPageSize;
        if (np == 2)
            step(std::integral_constant<int, 2>(), wdata + st * R, wdata + st1 * R, last_valid, pg * kPageSize);
        else
            step(std::integral_constant<int, 1>(), wdata + st * R, wdata + st * R, last_valid, pg * kPageSize);

        __syncwarp();
        if (j + S < hi)
            issue(j + S, st);
        if (np == 2 && j + 1 + S < hi)
            issue(j + 1 + S, st1);
        st += np;
        if (st >= S) {
            st -= S;
            ph ^= 1u;
        }

        j += np;
        pg += np;
        if (pg == n || j == hi) {
            finish_segment();
            if (j < hi) {
                ++h;
                pg = 0;
                if (h == nseg) {
                    h = 0;
                    do {
                        ++b;
                    } while (prefix[b + 1] == prefix[b]);
                    n = (prefix[b + 1] - prefix[b]) / nseg;
                    L = clamp_len(p.seq_lens[b], max_len);
                }
                seg_begin = prefix[b] + h * n;
                start_segment();
            }
        }
    }
    };  // run_worker
    run_worker();
}

// ---- split merge ---------------------------------------------------------------
// One CTA per (sequence, kv head, query head of the group), of kThreads
// threads: 32 per contributor group.  Segments that one worker covered were
// written by the decode kernel; empty sequences get zeros here.  The launch
// picks the CTA width from the contributors a segment has on average: 64
// threads while two groups take them in one round of loads -- capped at 64
// registers, such a CTA fits beside a decode CTA (61,440 of an SM's 65,536
// registers), so merge CTAs become resident while the decode runs and the next
// step's decode CTA need not wait for them to leave; 128 threads while four
// groups do (seven CTAs to an SM once the decode CTA has left); wider CTAs for
// the few long segments of a small batch at a long context.
template <int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads == 64 ? 16 : 1) merge_kernel(const __grid_constant__ DecodeParams p);

} // namespace nvfp4kv
