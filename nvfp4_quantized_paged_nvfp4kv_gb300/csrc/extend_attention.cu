// Extend attention on the fifth-generation tensor cores (tcgen05).
//
// "SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation: on the
// extend path the cached prefix is dequantised into one FP8 workspace and the
// new chunk attends over it and over itself; chunk token t of a sequence with
// prefix length P sees the P prefix keys and chunk keys 0 .. t.
//
// One CTA owns 128 rows of one sequence and one kv head, a row being a
// (chunk token, query head of the group) pair taken token-major.  Per key
// tile of 64:
//   S = Q K^T     tcgen05.mma M128 N64 K16 x 8 into tensor memory (two S
//                 buffers, so Q K^T of tile i+1 runs during the softmax of i)
//   softmax       one thread per row reads its S row from tensor memory,
//                 masks, takes exp2 against a running maximum that is only
//                 raised when it grows by more than 2^8 (then the O row in
//                 tensor memory is rescaled), writes P (f16) back to tensor
//                 memory
//   O += P V      tcgen05.mma M128 N128 K16 x 4 with P read from tensor
//                 memory, O resident in tensor memory
// Warps 0-3 run the softmax, warps 4-7 convert key tiles (E4M3 prefix rows,
// and bf16 or E4M3 chunk rows) to f16 in the 128-byte-swizzled operand
// layout, warp 8 allocates tensor memory and issues the MMAs.  E4M3 chunk
// rows are initial prefill as the same paragraph describes it: attention on
// the current prompt's FP8 keys and values.  mbarriers order the roles;
// every wait is bounded and a timeout is reported.
//
// The appending variant also writes the chunk's K/V into the NVFP4 cache
// ("SGLang stores KV cache in 4 bits", Interpretation: prefill quantises the
// new K/V into the cache): each chunk key tile has one owning CTA, whose
// converter warps quantise it after their last key tile.
#include <cudaTypedefs.h>

#include <mutex>

#include "record_write.cuh"
#include "tcgen05.cuh"

namespace nvfp4kv {
namespace {

constexpr int kTcRows = 128;                  // M: rows per CTA
constexpr int kTcKeys = 64;                   // keys per tile
constexpr int kSoftmaxThreads = 128;          // warps 0-3
constexpr int kProducerThreads = 128;         // warps 4-7
constexpr int kMmaWarp = 8;
constexpr int kTcThreads = kSoftmaxThreads + kProducerThreads + 32;
constexpr float kRescaleLog2 = 8.f;           // raise the running maximum only past this margin

constexpr uint32_t kQBytes = kTcRows * kHeadDim * 2;   // 32 KB
constexpr uint32_t kKVBytes = kTcKeys * kHeadDim * 2;  // 16 KB per K or V tile
constexpr uint32_t kOffQ = 0;
constexpr int kKvStages = 2;                           // converted key tiles in flight
constexpr uint32_t kOffK = kOffQ + kQBytes;            // kKvStages buffers
constexpr uint32_t kOffV = kOffK + kKvStages * kKVBytes;
constexpr uint32_t kOffBar = kOffV + kKvStages * kKVBytes;
// kv_full / kv_empty per key-tile stage; s_full, p_full, pv_done per S / P buffer
enum { kBarKvFull = 0, kBarKvEmpty = 4, kBarSFull = 8, kBarPFull = 10, kBarPvDone = 12, kBarDone = 14, kNumBars = 15 };
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffFail = kOffTmemSlot + 4;
constexpr uint32_t kTcSmem = kOffFail + 4 + 1024;      // + slack to align the base to 1024 bytes
// tensor-memory columns: O, S[2] (fp32); P[b] (f16 pairs) overwrites the first
// 32 columns of S[b] once the softmax has read them.  The MMAs of a CTA run in
// issue order, so Q K^T of tile i + 2 (into S[b]) follows P V of tile i.
constexpr uint32_t kColO = 0, kColS = 128, kColP = 128;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColPStride = kTcKeys;                // P[b] at kColP + b * kColPStride

static_assert(kTcSmem <= 227 * 1024, "shared memory");
// two CTAs per SM, no more: their 2 x 256 tensor-memory columns are then
// always free
static_assert(2 * kTcSmem <= 228 * 1024 && 3 * kTcSmem > 228 * 1024, "two CTAs per SM");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle atoms");

// Byte offset of 16-byte chunk c (f16 columns 8c .. 8c + 7) of row r in a
// 128-byte-swizzled tile of `rows` rows: 64-column blocks of rows x 128
// bytes, eight-row atoms of 1024 bytes, chunk position c ^ (r mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t rows, uint32_t r, uint32_t c)
{
    return (c >> 3) * rows * 128u + r * 128u + (((c & 7u) ^ (r & 7u)) << 4);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_nc(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float s)
{
    return pack_f16x2(__uint_as_float(w << 16) * s, __uint_as_float(w & 0xffff0000u) * s);
}

__device__ __forceinline__ bool wait_or_fail(uint32_t bar, uint32_t parity, volatile int *fail, int32_t *dev_status,
                                             uint32_t limit)
{
    if (*fail)
        return false;
    if (mbar_wait_bounded(bar, parity, limit))
        return true;
    *fail = 1;
    report(dev_status, NVFP4KV_DEV_TIMEOUT);
    return false;
}

struct TcCta {
    int c0, C, P;
    int64_t p0;
    int n_pre, n_tiles;
};

// Producer thread pt (0..127): load key tile i, wait until its stage is free,
// convert it to f16 in the 128-byte-swizzled layout and signal the MMA warp.
// FP8 tiles (every prefix tile; chunk tiles when kChunk8): 64 keys x 8 pieces
// of 16 bytes per K and per V, four pieces a thread each, loaded together.  bf16 chunk tiles: 64 keys x 16
// pieces per K and per V; thread pt owns piece pt mod 16 of keys pt / 16 + 8 j
// (j = 0..7), K then V (eight loads in flight a thread keep the register count
// low); its offsets repeat from tile to tile and are taken once.  Keys past
// the end are zeros.
struct ChunkLanes {
    int key;                         // first key of the thread's bf16 pieces
    uint32_t src;                    // its element offset inside a chunk tile's first row
    uint32_t dst;                    // swizzled f16 offset of its piece of key `key`
};

__device__ __forceinline__ ChunkLanes chunk_lanes(const ExtendParams &p, int pt)
{
    ChunkLanes l;
    const uint32_t piece = pt & 15;
    l.key = pt >> 4;
    l.src = static_cast<uint32_t>(l.key * p.hkv * kHeadDim) + 8 * piece;
    l.dst = sw128(kTcKeys, l.key, piece);
    return l;
}

template <bool kChunk8>
__device__ __forceinline__ bool produce_tile(const ExtendParams &p, const TcCta &c, int h, int i, int pt,
                                             const ChunkLanes &l, uint32_t base, volatile int *fail)
{
    const int st = i % kKvStages;
    const uint32_t kdst = base + kOffK + st * kKVBytes, vdst = base + kOffV + st * kKVBytes;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const size_t row_elems = static_cast<size_t>(p.hkv) * kHeadDim;   // one key's bf16 row
    const uint16_t *k_chunk = static_cast<const uint16_t *>(p.k_chunk);
    const uint16_t *v_chunk = static_cast<const uint16_t *>(p.v_chunk);
    uint4 raw[8];
    const bool pre = i < c.n_pre;
    const bool e4m3 = kChunk8 || pre;
    const int k0 = (pre ? i : i - c.n_pre) * kTcKeys;
    if (e4m3) {
        const uint8_t *kb = pre ? p.k_prefix : static_cast<const uint8_t *>(p.k_chunk);
        const uint8_t *vb = pre ? p.v_prefix : static_cast<const uint8_t *>(p.v_chunk);
        const int64_t r0 = pre ? c.p0 + k0 : static_cast<int64_t>(c.c0) + k0;
        const int lim = pre ? c.P : c.C;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = pt + kProducerThreads * (u & 3);
            const int key = idx >> 3, piece = idx & 7;
            const uint8_t *src = (u < 4 ? kb : vb) + ((r0 + key) * p.hkv + h) * kHeadDim + 16 * piece;
            raw[u] = k0 + key < lim ? ldg_nc(src) : zero;
        }
    } else {
        const size_t tile = (static_cast<size_t>(c.c0 + k0) * p.hkv + h) * kHeadDim + l.src;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            raw[u] = k0 + l.key + 8 * u < c.C ? ldg_nc(k_chunk + tile + u * 8 * row_elems) : zero;
    }
    // stage st was last read by the MMAs of tile i - kKvStages
    if (i >= kKvStages && !wait_or_fail(base + kOffBar + 8 * (kBarKvEmpty + st), ((i / kKvStages) - 1) & 1, fail,
                                        p.dev_status, p.wait_limit))
        return false;
    if (e4m3) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = pt + kProducerThreads * (u & 3);
            const uint32_t key = idx >> 3, piece = idx & 7;
            uint4 lo, hi;
            e4m3x4_to_f16x2x2(raw[u].x, lo.x, lo.y);
            e4m3x4_to_f16x2x2(raw[u].y, lo.z, lo.w);
            e4m3x4_to_f16x2x2(raw[u].z, hi.x, hi.y);
            e4m3x4_to_f16x2x2(raw[u].w, hi.z, hi.w);
            const uint32_t dst = u < 4 ? kdst : vdst;
            // pieces 4..7 store their high half first: eight lanes, eight bank groups
            const uint32_t first = (piece >> 2) & 1u;
            sts128(dst + sw128(kTcKeys, key, 2 * piece + first), first ? hi : lo);
            sts128(dst + sw128(kTcKeys, key, 2 * piece + 1 - first), first ? lo : hi);
        }
    } else {
        const size_t tile = (static_cast<size_t>(c.c0 + k0) * p.hkv + h) * kHeadDim + l.src;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half == 1) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    raw[u] = k0 + l.key + 8 * u < c.C ? ldg_nc(v_chunk + tile + u * 8 * row_elems) : zero;
            }
            const uint32_t dst = (half ? vdst : kdst) + l.dst;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                uint4 f;
                f.x = bf16x2_to_f16x2(raw[u].x, 1.f);
                f.y = bf16x2_to_f16x2(raw[u].y, 1.f);
                f.z = bf16x2_to_f16x2(raw[u].z, 1.f);
                f.w = bf16x2_to_f16x2(raw[u].w, 1.f);
                sts128(dst + 1024u * u, f);     // keys chunk_key + 8 u: 8 u rows below, same swizzle
            }
        }
    }
    fence_async_shared();
    mbar_arrive(base + kOffBar + 8 * (kBarKvFull + st));
    return true;
}

// ---- fused NVFP4 append of the chunk ----------------------------------------

// Page-head record and token of a chunk token's slot; false when the slot is
// skipped (negative) or out of range (reported when `rep`).
__device__ __forceinline__ bool append_site(const ExtendParams &p, int slot, int h, size_t &rec, int &tok, bool rep)
{
    if (slot < 0)
        return false;
    if (slot >= p.num_pages * kPageSize) {
        if (rep)
            report(p.dev_status, NVFP4KV_DEV_BAD_SLOT);
        return false;
    }
    const int page = slot / kPageSize;
    tok = slot - page * kPageSize;
    rec = (static_cast<size_t>(page) * p.hkv + h) * kNvfp4Record;
    return true;
}

// One 16-value block of a chunk row as loaded: two 16-byte pieces of bf16, or
// one of E4M3 codes (kChunk8).
template <bool kChunk8>
struct ChunkBlock {
    uint4 v[kChunk8 ? 1 : 2];
};

template <bool kChunk8>
__device__ __forceinline__ void load_raw(const void *src, size_t elem_off, ChunkBlock<kChunk8> &r)
{
    if constexpr (kChunk8) {
        r.v[0] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(src) + elem_off));
    } else {
        RawBlock<true> b;
        load_raw<true>(src, elem_off, b);
        r.v[0] = b.v[0];
        r.v[1] = b.v[1];
    }
}

// The block's values as fp32, exactly (bf16 widened; E4M3 through f16, which
// holds every E4M3 value).
template <bool kChunk8>
__device__ __forceinline__ void unpack(const ChunkBlock<kChunk8> &r, float (&x)[16])
{
    if constexpr (kChunk8) {
        const uint32_t w[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t lo, hi;
            e4m3x4_to_f16x2x2(w[k], lo, hi);
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
            const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
            x[4 * k] = a.x;
            x[4 * k + 1] = a.y;
            x[4 * k + 2] = b.x;
            x[4 * k + 3] = b.y;
        }
    } else {
        RawBlock<true> b;
        b.v[0] = r.v[0];
        b.v[1] = r.v[1];
        unpack<true>(b, x);
    }
}

// Producer thread pt quantises chunk keys k0 .. k0 + 63 of kv head h into the
// cache, reading the chunk rows (bf16, or E4M3 when kChunk8) from global
// memory (each group of loads issued together).  K: 64 keys x 8 blocks, four a
// thread.  V: 32 key pairs x 8 blocks, two a thread; a pair on an even slot
// and its successor is written whole, any other token through the atomic
// nibble merge.
template <bool kChunk8>
__device__ __forceinline__ void append_chunk_tile(const ExtendParams &p, const TcCta &c, int h, int k0, int pt)
{
    auto offset = [&](int key, int blk) {
        return (static_cast<size_t>(c.c0 + key) * p.hkv + h) * kHeadDim + blk * 16;
    };
    const TensorScale Gk = tensor_scale(head_tensor_scale(p.hs, false, h, p.gscale));
    const TensorScale Gv = tensor_scale(head_tensor_scale(p.hs, true, h, p.gscale));
    ChunkBlock<kChunk8> r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int item = pt + kProducerThreads * u;
        const int key = k0 + (item >> 3), blk = item & 7;
        if (key < c.C)
            load_raw<kChunk8>(p.k_chunk, offset(key, blk), r[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int item = pt + kProducerThreads * u;
        const int key = k0 + (item >> 3), blk = item & 7;
        size_t rec;
        int tok;
        if (key >= c.C || !append_site(p, p.slot_mapping[c.c0 + key], h, rec, tok, blk == 0))
            continue;
        float x[16];
        unpack<kChunk8>(r[u], x);
        const uint32_t flip = divide_by_tensor_scale(x, Gk);
        write_nvfp4_block(p.pool + rec, false, tok, blk, x, ScaleOfByte(), flip);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int item = pt + kProducerThreads * u;
        const int key0 = k0 + 2 * (item >> 3), blk = item & 7;
        if (key0 < c.C)
            load_raw<kChunk8>(p.v_chunk, offset(key0, blk), r[2 * u]);
        if (key0 + 1 < c.C)
            load_raw<kChunk8>(p.v_chunk, offset(key0 + 1, blk), r[2 * u + 1]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int item = pt + kProducerThreads * u;
        const int key0 = k0 + 2 * (item >> 3), blk = item & 7;
        const bool has0 = key0 < c.C, has1 = key0 + 1 < c.C;
        const int s0 = has0 ? p.slot_mapping[c.c0 + key0] : -1;
        const int s1 = has1 ? p.slot_mapping[c.c0 + key0 + 1] : -1;
        size_t rec0 = 0, rec1 = 0;
        int tok0 = 0, tok1 = 0;
        const bool ok0 = has0 && append_site(p, s0, h, rec0, tok0, false);
        const bool ok1 = has1 && append_site(p, s1, h, rec1, tok1, false);
        float x[16];
        if (ok0 && ok1 && (s0 & 1) == 0 && s1 == s0 + 1) {
            uint32_t S0, S1, q0[2], q1[2];
            unpack<kChunk8>(r[2 * u], x);
            uint32_t flip = divide_by_tensor_scale(x, Gv);
            quantize_block(x, S0, q0, ScaleOfByte(), flip);
            unpack<kChunk8>(r[2 * u + 1], x);
            flip = divide_by_tensor_scale(x, Gv);
            quantize_block(x, S1, q1, ScaleOfByte(), flip);
            write_nvfp4_v_pair(p.pool + rec0, tok0, blk, S0, q0, S1, q1);
            continue;
        }
        if (ok0) {
            unpack<kChunk8>(r[2 * u], x);
            const uint32_t flip = divide_by_tensor_scale(x, Gv);
            write_nvfp4_block(p.pool + rec0, true, tok0, blk, x, ScaleOfByte(), flip);
        }
        if (ok1) {
            unpack<kChunk8>(r[2 * u + 1], x);
            const uint32_t flip = divide_by_tensor_scale(x, Gv);
            write_nvfp4_block(p.pool + rec1, true, tok1, blk, x, ScaleOfByte(), flip);
        }
    }
}

// Softmax thread of row `row` (tensor-memory lane base lane_base): O / l to
// the output row, once the last value product has landed (the warp together:
// tensor-memory loads are warp-wide).
__device__ __forceinline__ void store_out_row(const ExtendParams &p, const TcCta &c, int h, int row, int R, int g,
                                              int t, uint32_t lane_base, float l)
{
    tc_fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const bool store = row < R;
    const int64_t off = (static_cast<int64_t>(c.c0 + t) * p.hq + h * g + (min(row, R - 1) - t * g)) * kHeadDim;
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t o[32];
        tmem_ld32(lane_base + kColO + 32 * cb, o);
        tmem_wait_ld();
        if (!store)
            continue;
        if (p.out_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off + 32 * cb);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                     __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + off + 32 * cb);
            auto bf2 = [&](int j) {
                const __nv_bfloat162 two =
                    __floats2bfloat162_rn(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
                return *reinterpret_cast<const uint32_t *>(&two);
            };
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dst[k] = make_uint4(bf2(8 * k), bf2(8 * k + 2), bf2(8 * k + 4), bf2(8 * k + 6));
        }
    }
}

template <bool kAppend, bool kChunk8>
__global__ void __launch_bounds__(kTcThreads, 2) extend_tc_kernel(const __grid_constant__ ExtendParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw_addr);
    volatile int *fail = reinterpret_cast<volatile int *>(gbase + kOffFail);
    const uint32_t bar = base + kOffBar;

    const int b_seq = blockIdx.z;
    const int h = blockIdx.y;
    const int tile = static_cast<int>(gridDim.x - 1 - blockIdx.x);  // later rows see more keys: start them first
    const int tid = threadIdx.x;
    const int warp = tid >> 5;

    TcCta c;
    c.c0 = p.q_indptr[b_seq];
    const int c1 = p.q_indptr[b_seq + 1];
    c.P = p.prefix_lens[b_seq];
    const int kv0 = p.kv_indptr[b_seq];
    if (c.c0 < 0 || c1 < c.c0 || c1 > p.q_rows || c1 - c.c0 > p.max_q_len || c.P < 0 || kv0 < 0 ||
        static_cast<int64_t>(kv0) + c.P > p.prefix_rows) {
        if (tid == 0)
            report(p.dev_status, NVFP4KV_DEV_BAD_LEN);
        return;
    }
    c.C = c1 - c.c0;
    c.p0 = kv0;
    const int g = p.group;
    const int R = c.C * g;
    const int row0 = tile * kTcRows;
    if (row0 >= R)
        return;
    const int t_max = (min(row0 + kTcRows, R) - 1) / g;
    c.n_pre = (c.P + kTcKeys - 1) / kTcKeys;
    c.n_tiles = c.n_pre + t_max / kTcKeys + 1;

    // Q tile: rows past the end are zeros; sm_scale * log2 e folded in
    for (int idx = tid; idx < kTcRows * 16; idx += kTcThreads) {
        const int r = idx >> 4, piece = idx & 15;
        const int row = row0 + r;
        uint4 f = make_uint4(0, 0, 0, 0);
        if (row < R) {
            const int t = row / g;
            const uint4 w = ldg_nc(p.q + (static_cast<int64_t>(c.c0 + t) * p.hq + h * g + (row - t * g)) * kHeadDim +
                                   8 * piece);
            f.x = bf16x2_to_f16x2(w.x, p.qscale);
            f.y = bf16x2_to_f16x2(w.y, p.qscale);
            f.z = bf16x2_to_f16x2(w.z, p.qscale);
            f.w = bf16x2_to_f16x2(w.w, p.qscale);
        }
        sts128(base + kOffQ + sw128(kTcRows, r, piece), f);
    }
    if (tid == 0) {
        for (int k = 0; k < kKvStages; ++k) {
            mbar_init(bar + 8 * (kBarKvFull + k), kProducerThreads);
            mbar_init(bar + 8 * (kBarKvEmpty + k), 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(bar + 8 * (kBarSFull + k), 1);
            mbar_init(bar + 8 * (kBarPFull + k), kSoftmaxThreads);
            mbar_init(bar + 8 * (kBarPvDone + k), 1);
        }
        mbar_init(bar + 8 * kBarDone, 1);
        *fail = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp)
        tmem_alloc(base + kOffTmemSlot, kTmemCols);
    fence_async_shared();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + kOffTmemSlot);

    if (warp == kMmaWarp) {
        if ((tid & 31) == 0) {
            constexpr uint32_t i_qk = idesc_f16(kTcRows, kTcKeys, false);
            constexpr uint32_t i_pv = idesc_f16(kTcRows, kHeadDim, true);
            bool ok = true;
            auto qk = [&](int i) {
                const int b = i & 1, st = i % kKvStages;
                tc_fence_after_sync();
                const uint32_t kb = base + kOffK + st * kKVBytes;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    umma_f16(tmem + kColS + b * kTcKeys,
                             smem_desc(base + kOffQ + (s >> 2) * (kTcRows * 128) + (s & 3) * 32, 16, 1024),
                             smem_desc(kb + (s >> 2) * (kTcKeys * 128) + (s & 3) * 32, 16, 1024), i_qk, s > 0);
                umma_commit(bar + 8 * (kBarSFull + b));
            };
            auto pv = [&](int i) {
                const int b = i & 1;
                tc_fence_after_sync();
                const uint32_t vb = base + kOffV + (i % kKvStages) * kKVBytes;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    umma_f16_ts(tmem + kColO, tmem + kColP + b * kColPStride + s * 8,
                                smem_desc(vb + s * 2048, kTcKeys * 128, 1024), i_pv, i > 0 || s > 0);
                umma_commit(bar + 8 * (kBarPvDone + b));
                umma_commit(bar + 8 * (kBarKvEmpty + i % kKvStages));
            };
            // Q K^T of tile j may be issued once its keys are in and S buffer
            // j mod 2 is free (tile j - 2's P V issued), P V of tile i once its
            // P is in.  Whichever is ready first goes first, so a value product
            // never waits behind the conversion of the next key tile.  P V of
            // tile i always precedes Q K^T of tile i + 2 (the P aliasing).
            int next_qk = 0;
            for (int i = 0; ok && i < c.n_tiles; ++i) {
                const int b = i & 1;
                bool pv_done = false;
                for (uint64_t polls = 0; !pv_done;) {
                    bool progress = false;
                    if (next_qk <= i + 1 && next_qk < c.n_tiles &&
                        mbar_test_wait(bar + 8 * (kBarKvFull + next_qk % kKvStages), (next_qk / kKvStages) & 1)) {
                        qk(next_qk++);
                        progress = true;
                    }
                    if (next_qk > i && mbar_test_wait(bar + 8 * (kBarPFull + b), (i >> 1) & 1)) {
                        pv(i);
                        pv_done = progress = true;
                    }
                    if (progress)
                        continue;
                    if (++polls > 64ull * p.wait_limit || *fail) {
                        if (!*fail) {
                            *fail = 1;
                            report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
                        }
                        ok = false;
                        break;
                    }
                }
            }
            // nothing of this thread's may still run when tensor memory is freed
            // (waited for at the default limit, whatever p.wait_limit is)
            umma_commit(bar + 8 * kBarDone);
            if (!mbar_wait_bounded(bar + 8 * kBarDone, 0, kWaitLimit))
                report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= kSoftmaxThreads / 32) {
        const int pt = tid - kSoftmaxThreads;
        const ChunkLanes lanes = chunk_lanes(p, pt);
        for (int i = 0; i < c.n_tiles; ++i)
            if (!produce_tile<kChunk8>(p, c, h, i, pt, lanes, base, fail))
                break;
        if constexpr (kAppend) {
            // the chunk key tiles whose first key's first row (64 kt g) falls in
            // this CTA's rows; done while the last tiles are still in the MMAs
            const int per = kTcKeys * g;
            for (int kt = (row0 + per - 1) / per; kt < (row0 + kTcRows + per - 1) / per && kt * kTcKeys < c.C; ++kt)
                append_chunk_tile<kChunk8>(p, c, h, kt * kTcKeys, pt);
        }
    } else {
        // softmax: thread r owns row row0 + r, tensor-memory lane r
        const int r = tid;
        const int row = row0 + r;
        const int t = min(row, R - 1) / g;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // the warp leaves together: its tensor-memory accesses are warp-wide
        auto wait_warp = [&](uint32_t bar_addr, uint32_t parity) {
            return __all_sync(kFullMask, wait_or_fail(bar_addr, parity, fail, p.dev_status, p.wait_limit));
        };
        for (int i = 0; i < c.n_tiles; ++i) {
            const int b = i & 1;
            if (!(ok = wait_warp(bar + 8 * (kBarSFull + b), (i >> 1) & 1)))
                break;
            tc_fence_after_sync();
            uint32_t sr0[32], sr1[32];
            tmem_ld32(lane_base + kColS + b * kTcKeys, sr0);
            tmem_ld32(lane_base + kColS + b * kTcKeys + 32, sr1);
            tmem_wait_ld();
            float s[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                s[j] = __uint_as_float(sr0[j]);
                s[j + 32] = __uint_as_float(sr1[j]);
            }
            const int lim = i < c.n_pre ? c.P - i * kTcKeys : t + 1 - (i - c.n_pre) * kTcKeys;
            if (lim < kTcKeys) {
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j >= lim)
                        s[j] = -INFINITY;
            }
            // eight independent partial maxima (three-input max) and packed
            // two-lane subtractions and sums keep the chains and counts short
            float pm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                pm[k] = fmax3(fmax3(s[8 * k], s[8 * k + 1], s[8 * k + 2]), fmax3(s[8 * k + 3], s[8 * k + 4], s[8 * k + 5]),
                              fmaxf(s[8 * k + 6], s[8 * k + 7]));
            const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
            const bool need = mx > m_used + kRescaleLog2;
            const float m_new = need ? mx : m_used;
            const float mbase = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = need ? fast_exp2(m_used - mbase) : 1.f;
            const uint64_t neg2 = f32x2_pack(-mbase, -mbase);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint64_t d = add_f32x2(f32x2_pack(s[2 * j], s[2 * j + 1]), neg2);
                s[2 * j] = fast_exp2(f32x2_lo(d));
                s[2 * j + 1] = fast_exp2(f32x2_hi(d));
                acc[j & 3] = add_f32x2(acc[j & 3], f32x2_pack(s[2 * j], s[2 * j + 1]));
            }
            const uint64_t a01 = add_f32x2(acc[0], acc[1]), a23 = add_f32x2(acc[2], acc[3]);
            const uint64_t a = add_f32x2(a01, a23);
            const float sum = f32x2_lo(a) + f32x2_hi(a);
            l = l * alpha + sum;
            m_used = m_new;
            // P row into tensor memory, f16 pairs, the A operand of the value
            // product.  P[b] was last read by the value product of tile i - 2,
            // which ran before Q K^T of tile i (in issue order): it is free.
            {
                uint32_t pw[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    pw[j] = pack_f16x2(s[2 * j], s[2 * j + 1]);
                tmem_st32(lane_base + kColP + b * kColPStride, pw);
            }
            // a raised maximum: rescale the O rows of the warp once the value
            // product of tile i - 1 has landed
            if (__any_sync(kFullMask, need) && i >= 1) {
                const int pb = (i - 1) & 1;
                if (!(ok = wait_warp(bar + 8 * (kBarPvDone + pb), ((i - 1) >> 1) & 1)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + 32 * cb, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(lane_base + kColO + 32 * cb, o);
                }
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(bar + 8 * (kBarPFull + b));
        }
        if (ok) {
            const int last = c.n_tiles - 1;
            ok = wait_warp(bar + 8 * (kBarPvDone + (last & 1)), (last >> 1) & 1);
        }
        if (ok)
            store_out_row(p, c, h, row, R, g, t, lane_base, l);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- all keys in E4M3: Q K^T on kind::f8f6f4 with the key tiles from TMA ----
//
// When the chunk's keys and values are E4M3 too (initial prefill and extends
// on FP8 K/V), every key tile is E4M3 bytes, one 128-byte row per key: the
// TMA unit loads a 64-key tile of one kv head straight into the 128-byte
// swizzle the MMA reads, and S = Q K^T runs as tcgen05.mma kind::f8f6f4 with
// Q split into two E4M3 terms (hi, lo), both accumulated into S.  Each row of
// the bf16 Q is first multiplied by a power of two 2^e_r that puts its largest
// element in [128, 256); the softmax takes S * 2^-e_r * sm_scale.  A bf16
// value has eight significant bits: hi = E4M3(x) keeps the first four, and the
// remainder x - hi is a multiple of x's last place no larger than hi's half
// place, so lo = E4M3(x - hi) holds it exactly wherever it is not below
// E4M3's subnormal step 2^-9 (scaled elements of at least 1/4); smaller
// elements keep an error of at most 2^-10, under 2^-17 of the row's largest.
// Values stay on the f16 path: the TMA unit loads the E4M3 value tile into a
// staging ring, the converter warps turn it into the f16 operand of P V (rows
// past the sequence's keys become zeros), and P V runs on kind::f16 as in the
// kernel above.  Warp 9 issues the TMA loads: key tiles into a ring of three
// stages, value tiles into a ring of two, so that a tile's load latency is
// covered by the work on the tiles before it.
//
// With a bf16 chunk (kChunkBf16) the prefix tiles run as above and the chunk
// tiles come from the converter warps: each bf16 key tile is multiplied by a
// power of two 2^f that puts its largest element in [128, 256) and split, as
// Q is, into hi and lo E4M3 terms (exact for bf16 under the same bound); hi
// goes to the key stage, lo to the idle value staging stage, and Q K^T
// accumulates the four products of the terms.  The tile's 2^-f reaches the
// softmax through a small ring in shared memory with its own barriers.  The
// values are converted bf16 -> f16 as in the kernel above.
constexpr int kF8Threads = kTcThreads + 32;                 // + the TMA warp
constexpr int kF8TmaWarp = 9;
constexpr int kF8QTerms = 2;
constexpr int kF8KStages = 3;                               // E4M3 key tiles
constexpr int kF8VrawStages = 2;                            // E4M3 value tiles
constexpr uint32_t kF8QTerm = kTcRows * kHeadDim;           // 16 KB per E4M3 term
constexpr uint32_t kF8KBytes = kTcKeys * kHeadDim;          // 8 KB per E4M3 key or value tile
constexpr uint32_t kF8OffQ = 0;
constexpr uint32_t kF8OffK = kF8OffQ + kF8QTerms * kF8QTerm;
constexpr uint32_t kF8OffV = kF8OffK + kF8KStages * kF8KBytes;     // two f16 stages (kKVBytes each)
constexpr uint32_t kF8OffVraw = kF8OffV + 2 * kKVBytes;
constexpr uint32_t kF8OffBar = kF8OffVraw + kF8VrawStages * kF8KBytes;
// K stages are released after their Q K^T (kF8KEmpty), staged value tiles
// after their conversion (kF8VrawEmpty), f16 V stages after their P V
// (kF8VEmpty)
enum {
    kF8KFull = 0, kF8KEmpty = kF8KFull + kF8KStages, kF8VrawFull = kF8KEmpty + kF8KStages,
    kF8VrawEmpty = kF8VrawFull + kF8VrawStages, kF8VFull = kF8VrawEmpty + kF8VrawStages, kF8VEmpty = kF8VFull + 2,
    kF8SFull = kF8VEmpty + 2, kF8PFull = kF8SFull + 2, kF8PvDone = kF8PFull + 2, kF8Done = kF8PvDone + 2,
    // bf16 chunk tiles: the low key term's stage released by Q K^T, the
    // tile scale ring filled by the converters, and two converter-only
    // barriers (the tile maximum exchanged; every term stored), each used by
    // alternate chunk tiles
    kF8KloEmpty = kF8Done + 1, kF8KScale = kF8KloEmpty + 2, kF8KRed = kF8KScale + 8, kF8KTerm = kF8KRed + 2,
    kF8NumBars = kF8KTerm + 2
};
constexpr int kF8KScaleRing = 8;                            // converters run at most ~5 tiles ahead
constexpr uint32_t kF8OffRowInv = (kF8OffBar + 8 * kF8NumBars + 15) / 16 * 16;
constexpr uint32_t kF8OffKScale = kF8OffRowInv + 4 * kTcRows;      // 2^-f of chunk tiles [ring]
constexpr uint32_t kF8OffKRed = kF8OffKScale + 4 * kF8KScaleRing;  // converter warps' maxima [2][4]
constexpr uint32_t kF8OffTmemSlot = kF8OffKRed + 4 * 8;
constexpr uint32_t kF8OffFail = kF8OffTmemSlot + 4;
constexpr uint32_t kF8Smem = kF8OffFail + 4 + 1024;
static_assert(kF8OffRowInv % 16 == 0, "row scale table alignment");
static_assert(kF8OffK % 1024 == 0 && kF8OffV % 1024 == 0 && kF8OffVraw % 1024 == 0, "swizzle atoms");
static_assert(2 * (kF8Smem + 1024) <= 228 * 1024, "two CTAs per SM");

// Two fp32 -> E4M3 bytes and back to fp32, exactly (the decode is exact).
__device__ __forceinline__ float2 e4m3x2_value(uint32_t two)
{
    const uint32_t h = e4m3x2_to_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

template <bool kAppend, bool kChunkBf16>
__global__ void __launch_bounds__(kF8Threads, 2) extend_f8_kernel(const __grid_constant__ ExtendParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw_addr);
    volatile int *fail = reinterpret_cast<volatile int *>(gbase + kF8OffFail);
    float *rowinv = reinterpret_cast<float *>(gbase + kF8OffRowInv);
    const uint32_t bar = base + kF8OffBar;
    auto B = [&](int k) { return bar + 8 * k; };

    const int b_seq = blockIdx.z;
    const int h = blockIdx.y;
    const int tile = static_cast<int>(gridDim.x - 1 - blockIdx.x);  // later rows see more keys: start them first
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    TcCta c;
    c.c0 = p.q_indptr[b_seq];
    const int c1 = p.q_indptr[b_seq + 1];
    c.P = p.prefix_lens[b_seq];
    const int kv0 = p.kv_indptr[b_seq];
    if (c.c0 < 0 || c1 < c.c0 || c1 > p.q_rows || c1 - c.c0 > p.max_q_len || c.P < 0 || kv0 < 0 ||
        static_cast<int64_t>(kv0) + c.P > p.prefix_rows) {
        if (tid == 0)
            report(p.dev_status, NVFP4KV_DEV_BAD_LEN);
        return;
    }
    c.C = c1 - c.c0;
    c.p0 = kv0;
    const int g = p.group;
    const int R = c.C * g;
    const int row0 = tile * kTcRows;
    if (row0 >= R)
        return;
    const int t_max = (min(row0 + kTcRows, R) - 1) / g;
    c.n_pre = (c.P + kTcKeys - 1) / kTcKeys;
    c.n_tiles = c.n_pre + t_max / kTcKeys + 1;

    // Q as two E4M3 terms, each row scaled by a power of two first (the
    // softmax scale is applied to S).  Sixteen consecutive lanes hold one row
    // (eight channels each): the CTA's threads cover the 2,048 pieces in whole
    // warps, so the row maximum is a shuffle over those lanes.
    for (int idx0 = warp * 32; idx0 < kTcRows * 16; idx0 += kF8Threads) {
        const int idx = idx0 + lane;
        const int r = idx >> 4, piece = idx & 15;
        const int row = row0 + r;
        float x[8];
        if (row < R) {
            const int t = row / g;
            const uint4 w = ldg_nc(p.q + (static_cast<int64_t>(c.c0 + t) * p.hq + h * g + (row - t * g)) * kHeadDim +
                                   8 * piece);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[2 * k] = __uint_as_float(ww[k] << 16);
                x[2 * k + 1] = __uint_as_float(ww[k] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                x[k] = 0.f;
        }
        float am = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            am = fmaxf(am, fabsf(x[k]));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
            am = fmaxf(am, __shfl_xor_sync(kFullMask, am, o));
        // 2^e with amax * 2^e in [128, 256); rows of (almost) zeros keep scale 1
        int e = 0;
        if (am >= 1e-30f)
            e = 7 - (static_cast<int>((__float_as_uint(am) >> 23) & 0xffu) - 127);
        const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        if (piece == 0)
            rowinv[r] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23) * p.qscale;
        uint32_t term[kF8QTerms][2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float a = x[2 * k] * sc, b = x[2 * k + 1] * sc;
#pragma unroll
            for (int t = 0; t < kF8QTerms; ++t) {
                const uint32_t two = f32x2_to_e4m3x2(a, b);
                const float2 v = e4m3x2_value(two);
                a -= v.x;                         // exact: the remainder of an E4M3 rounding
                b -= v.y;
                if (k & 1)
                    term[t][k >> 1] |= two << 16;
                else
                    term[t][k >> 1] = two;
            }
        }
        const uint32_t off = r * 128u + ((static_cast<uint32_t>(piece >> 1) ^ (r & 7u)) << 4) + (piece & 1) * 8u;
#pragma unroll
        for (int t = 0; t < kF8QTerms; ++t)
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(base + kF8OffQ + t * kF8QTerm + off),
                         "r"(term[t][0]), "r"(term[t][1])
                         : "memory");
    }
    if (tid == 0) {
        for (int k = 0; k < kF8KStages; ++k) {
            mbar_init(B(kF8KFull + k), 1);
            mbar_init(B(kF8KEmpty + k), 1);
        }
        for (int k = 0; k < kF8VrawStages; ++k) {
            mbar_init(B(kF8VrawFull + k), 1);
            mbar_init(B(kF8VrawEmpty + k), kProducerThreads);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(B(kF8VEmpty + k), 1);
            mbar_init(B(kF8VFull + k), kProducerThreads);
            mbar_init(B(kF8SFull + k), 1);
            mbar_init(B(kF8PFull + k), kSoftmaxThreads);
            mbar_init(B(kF8PvDone + k), 1);
        }
        mbar_init(B(kF8Done), 1);
        if constexpr (kChunkBf16) {
            for (int k = 0; k < 2; ++k)
                mbar_init(B(kF8KloEmpty + k), 1);
            for (int k = 0; k < kF8KScaleRing; ++k)
                mbar_init(B(kF8KScale + k), 1);
            for (int k = 0; k < 2; ++k) {
                mbar_init(B(kF8KRed + k), kProducerThreads);
                mbar_init(B(kF8KTerm + k), kProducerThreads);
            }
        }
        *fail = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp)
        tmem_alloc(base + kF8OffTmemSlot, kTmemCols);
    fence_async_shared();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + kF8OffTmemSlot);

    if (warp == kF8TmaWarp) {
        if (lane == 0) {
            // key tile i: K into stage i % kF8KStages, V into staging stage
            // i % kF8VrawStages
            int nk = 0, nv = 0;                  // loads issued
            const int n_tma = kChunkBf16 ? c.n_pre : c.n_tiles;     // bf16 chunk tiles come from the converters
            for (int i = 0; i < n_tma; ++i) {
                const int sk = i % kF8KStages, sv = i % kF8VrawStages;
                const bool pre = i < c.n_pre;
                const int rowc = pre ? static_cast<int>(c.p0) + i * kTcKeys : c.c0 + (i - c.n_pre) * kTcKeys;
                // the K stage was last read by Q K^T of tile i - kF8KStages
                if (i >= kF8KStages &&
                    !wait_or_fail(B(kF8KEmpty + sk), (i / kF8KStages - 1) & 1, fail, p.dev_status, p.wait_limit))
                    break;
                mbar_arrive_expect_tx(B(kF8KFull + sk), kF8KBytes);
                tma_load_3d(base + kF8OffK + sk * kF8KBytes, pre ? &p.tm_k_prefix : &p.tm_k_chunk, 0, h, rowc,
                            B(kF8KFull + sk));
                ++nk;
                // the staging stage was last read by the converters for tile
                // i - kF8VrawStages
                if (i >= kF8VrawStages && !wait_or_fail(B(kF8VrawEmpty + sv), (i / kF8VrawStages - 1) & 1, fail,
                                                        p.dev_status, p.wait_limit))
                    break;
                mbar_arrive_expect_tx(B(kF8VrawFull + sv), kF8KBytes);
                tma_load_3d(base + kF8OffVraw + sv * kF8KBytes, pre ? &p.tm_v_prefix : &p.tm_v_chunk, 0, h, rowc,
                            B(kF8VrawFull + sv));
                ++nv;
            }
            // nothing issued may still be in flight when the CTA exits: the
            // last loads of each ring (earlier ones were waited for before
            // their stage was reused)
            for (int i = max(0, nk - kF8KStages); i < nk; ++i)
                if (!mbar_wait_bounded(B(kF8KFull + i % kF8KStages), (i / kF8KStages) & 1, kWaitLimit))
                    report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
            for (int i = max(0, nv - kF8VrawStages); i < nv; ++i)
                if (!mbar_wait_bounded(B(kF8VrawFull + i % kF8VrawStages), (i / kF8VrawStages) & 1, kWaitLimit))
                    report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t i_qk = idesc_f16(kTcRows, kTcKeys, false);   // E4M3 x E4M3 -> f32 (same bits)
            constexpr uint32_t i_pv = idesc_f16(kTcRows, kHeadDim, true);
            bool ok = true;
            auto qk = [&](int i) {
                const int b = i & 1, st = i % kF8KStages;
                tc_fence_after_sync();
                const uint32_t kb = base + kF8OffK + st * kF8KBytes;
#pragma unroll
                for (int t = 0; t < kF8QTerms; ++t)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_f8(tmem + kColS + b * kTcKeys,
                                smem_desc(base + kF8OffQ + t * kF8QTerm + ks * 32, 16, 1024),
                                smem_desc(kb + ks * 32, 16, 1024), i_qk, t > 0 || ks > 0);
                if (kChunkBf16 && i >= c.n_pre) {
                    // the chunk tile's low key term, in the staging stage
                    const int sl = (i - c.n_pre) & 1;
                    const uint32_t klo = base + kF8OffVraw + sl * kF8KBytes;
#pragma unroll
                    for (int t = 0; t < kF8QTerms; ++t)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            umma_f8(tmem + kColS + b * kTcKeys,
                                    smem_desc(base + kF8OffQ + t * kF8QTerm + ks * 32, 16, 1024),
                                    smem_desc(klo + ks * 32, 16, 1024), i_qk, true);
                    umma_commit(B(kF8KloEmpty + sl));
                }
                umma_commit(B(kF8SFull + b));
                umma_commit(B(kF8KEmpty + st));
            };
            auto pv = [&](int i) {
                const int b = i & 1, st = i & 1;
                tc_fence_after_sync();
                const uint32_t vb = base + kF8OffV + st * kKVBytes;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    umma_f16_ts(tmem + kColO, tmem + kColP + b * kColPStride + s * 8,
                                smem_desc(vb + s * 2048, kTcKeys * 128, 1024), i_pv, i > 0 || s > 0);
                umma_commit(B(kF8PvDone + b));
                umma_commit(B(kF8VEmpty + st));
            };
            // Q K^T of tile j once its keys are in and tile j - 2's P V is
            // issued; P V of tile i once its P and its converted values are
            // in; whichever is ready first goes first.
            int next_qk = 0;
            for (int i = 0; ok && i < c.n_tiles; ++i) {
                const int b = i & 1;
                bool pv_done = false;
                for (uint64_t polls = 0; !pv_done;) {
                    bool progress = false;
                    if (next_qk <= i + 1 && next_qk < c.n_tiles &&
                        mbar_test_wait(B(kF8KFull + next_qk % kF8KStages), (next_qk / kF8KStages) & 1)) {
                        qk(next_qk++);
                        progress = true;
                    }
                    if (next_qk > i && mbar_test_wait(B(kF8PFull + b), (i >> 1) & 1) &&
                        mbar_test_wait(B(kF8VFull + b), (i >> 1) & 1)) {
                        pv(i);
                        pv_done = progress = true;
                    }
                    if (progress)
                        continue;
                    if (++polls > 64ull * p.wait_limit || *fail) {
                        if (!*fail) {
                            *fail = 1;
                            report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
                        }
                        ok = false;
                        break;
                    }
                }
            }
            // nothing of this thread's may still run when tensor memory is freed
            // (waited for at the default limit, whatever p.wait_limit is)
            umma_commit(B(kF8Done));
            if (!mbar_wait_bounded(B(kF8Done), 0, kWaitLimit))
                report(p.dev_status, NVFP4KV_DEV_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= kSoftmaxThreads / 32) {
        // converters: thread pt turns half a row of the staged E4M3 value tile
        // (key pt % 64, channels 64 (pt / 64) .. + 63) into f16.  A warp takes
        // 32 consecutive keys of one half, so each eight lanes of a 16-byte
        // load or store meet eight different bank groups (the chunk index is
        // xored with the key's low three bits).
        const int pt = tid - kSoftmaxThreads;
        const int key = pt & 63, half = pt >> 6;
        // bf16 chunk tile i (kChunkBf16): thread pt takes channels 64 half ..
        // + 63 of key pt % 64 for K, then for V.  The converters meet only on
        // mbarriers with bounded waits (a thread that gave up elsewhere stops
        // arriving, and the others' waits give up after it).  Returns false
        // when a wait gave up.
        auto chunk_tile = [&](int i) {
            const int cc = i - c.n_pre, sk = i % kF8KStages, sl = cc & 1, st = i & 1;
            const bool live = cc * kTcKeys + key < c.C;
            const size_t src =
                (static_cast<size_t>(c.c0 + cc * kTcKeys + key) * p.hkv + h) * kHeadDim + 64 * half;
            const uint16_t *kc = static_cast<const uint16_t *>(p.k_chunk);
            const uint16_t *vc = static_cast<const uint16_t *>(p.v_chunk);
            const uint4 zero = make_uint4(0, 0, 0, 0);
            uint4 kr[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                kr[j] = live ? ldg_nc(kc + src + 8 * j) : zero;
            // the tile's largest |k| (bf16 magnitudes compare as integers)
            uint32_t m2 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                m2 = __vmaxu2(m2, kr[j].x & 0x7fff7fffu);
                m2 = __vmaxu2(m2, kr[j].y & 0x7fff7fffu);
                m2 = __vmaxu2(m2, kr[j].z & 0x7fff7fffu);
                m2 = __vmaxu2(m2, kr[j].w & 0x7fff7fffu);
            }
            float am = __uint_as_float(max(m2 & 0xffffu, m2 >> 16) << 16);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                am = fmaxf(am, __shfl_xor_sync(kFullMask, am, o));
            float *kred = reinterpret_cast<float *>(gbase + kF8OffKRed) + 4 * sl;
            if (lane == 0)
                kred[warp - kSoftmaxThreads / 32] = am;
            mbar_arrive(B(kF8KRed + sl));
            if (!wait_or_fail(B(kF8KRed + sl), (cc >> 1) & 1, fail, p.dev_status, p.wait_limit))
                return false;
            am = fmaxf(fmaxf(kred[0], kred[1]), fmaxf(kred[2], kred[3]));
            int e = 0;
            if (am >= 1e-30f)
                e = 7 - (static_cast<int>((__float_as_uint(am) >> 23) & 0xffu) - 127);
            const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
            // the key stage was last read by Q K^T of tile i - 3, the low-term
            // stage by Q K^T of chunk tile cc - 2
            if (i >= kF8KStages &&
                !wait_or_fail(B(kF8KEmpty + sk), (i / kF8KStages - 1) & 1, fail, p.dev_status, p.wait_limit))
                return false;
            if (cc >= 2 &&
                !wait_or_fail(B(kF8KloEmpty + sl), ((cc >> 1) - 1) & 1, fail, p.dev_status, p.wait_limit))
                return false;
            const uint32_t khi = base + kF8OffK + sk * kF8KBytes, klo = base + kF8OffVraw + sl * kF8KBytes;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t w[4] = {kr[j].x, kr[j].y, kr[j].z, kr[j].w};
                uint32_t th[2], tl[2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float a = __uint_as_float(w[k] << 16) * sc, bb = __uint_as_float(w[k] & 0xffff0000u) * sc;
                    const uint32_t hi2 = f32x2_to_e4m3x2(a, bb);
                    const float2 v = e4m3x2_value(hi2);
                    const uint32_t lo2 = f32x2_to_e4m3x2(a - v.x, bb - v.y);   // exact remainders
                    if (k & 1) {
                        th[k >> 1] |= hi2 << 16;
                        tl[k >> 1] |= lo2 << 16;
                    } else {
                        th[k >> 1] = hi2;
                        tl[k >> 1] = lo2;
                    }
                }
                const uint32_t off =
                    key * 128u + ((static_cast<uint32_t>(4 * half + (j >> 1)) ^ (key & 7u)) << 4) + (j & 1) * 8u;
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(khi + off), "r"(th[0]), "r"(th[1]) : "memory");
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(klo + off), "r"(tl[0]), "r"(tl[1]) : "memory");
            }
            fence_async_shared();
            mbar_arrive(B(kF8KTerm + sl));
            if (pt == 0) {
                // every converter's terms are stored: publish the tile
                if (!wait_or_fail(B(kF8KTerm + sl), (cc >> 1) & 1, fail, p.dev_status, p.wait_limit))
                    return false;
                reinterpret_cast<float *>(gbase + kF8OffKScale)[cc % kF8KScaleRing] =
                    __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                mbar_arrive(B(kF8KScale + cc % kF8KScaleRing));
                mbar_arrive(B(kF8KFull + sk));
            }
            // values: bf16 -> f16 into stage st (last read by P V of tile i - 2)
            uint4 vr[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                vr[j] = live ? ldg_nc(vc + src + 8 * j) : zero;
            if (i >= 2 && !wait_or_fail(B(kF8VEmpty + st), ((i >> 1) - 1) & 1, fail, p.dev_status, p.wait_limit))
                return false;
            const uint32_t dst = base + kF8OffV + st * kKVBytes;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 f;
                f.x = bf16x2_to_f16x2(vr[j].x, 1.f);
                f.y = bf16x2_to_f16x2(vr[j].y, 1.f);
                f.z = bf16x2_to_f16x2(vr[j].z, 1.f);
                f.w = bf16x2_to_f16x2(vr[j].w, 1.f);
                sts128(dst + sw128(kTcKeys, key, 8 * half + j), f);
            }
            fence_async_shared();
            mbar_arrive(B(kF8VFull + st));
            return true;
        };
        for (int i = 0; i < c.n_tiles; ++i) {
            if constexpr (kChunkBf16) {
                if (i >= c.n_pre) {
                    if (!chunk_tile(i))
                        break;
                    continue;
                }
            }
            const int st = i & 1, sv = i % kF8VrawStages;
            const int lim = i < c.n_pre ? c.P - i * kTcKeys : c.C - (i - c.n_pre) * kTcKeys;
            if (!wait_or_fail(B(kF8VrawFull + sv), (i / kF8VrawStages) & 1, fail, p.dev_status, p.wait_limit))
                break;
            uint4 raw[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                raw[jj] = lds128(base + kF8OffVraw + sv * kF8KBytes + key * 128u +
                                 ((static_cast<uint32_t>(4 * half + jj) ^ (key & 7u)) << 4));
            // a later TMA load (async proxy) overwrites the staging tile these
            // generic-proxy reads come from: a proxy fence orders the reads
            // before the release, as a plain arrive does not across proxies
            fence_async_shared();
            mbar_arrive(B(kF8VrawEmpty + sv));
            // the f16 stage was last read by P V of tile i - 2
            if (i >= 2 && !wait_or_fail(B(kF8VEmpty + st), ((i >> 1) - 1) & 1, fail, p.dev_status, p.wait_limit))
                break;
            const uint32_t dst = base + kF8OffV + st * kKVBytes;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                if (key < lim) {
                    e4m3x4_to_f16x2x2(raw[jj].x, lo.x, lo.y);
                    e4m3x4_to_f16x2x2(raw[jj].y, lo.z, lo.w);
                    e4m3x4_to_f16x2x2(raw[jj].z, hi.x, hi.y);
                    e4m3x4_to_f16x2x2(raw[jj].w, hi.z, hi.w);
                }
                const int cch = 8 * half + 2 * jj;       // 16-byte f16 chunk index over the 128 channels
                sts128(dst + sw128(kTcKeys, key, cch), lo);
                sts128(dst + sw128(kTcKeys, key, cch + 1), hi);
            }
            fence_async_shared();
            mbar_arrive(B(kF8VFull + st));
        }
        if constexpr (kAppend) {
            const int per = kTcKeys * g;
            for (int kt = (row0 + per - 1) / per; kt < (row0 + kTcRows + per - 1) / per && kt * kTcKeys < c.C; ++kt)
                append_chunk_tile<!kChunkBf16>(p, c, h, kt * kTcKeys, pt);
        }
    } else {
        // softmax: thread r owns row row0 + r, tensor-memory lane r; scores are
        // S * 2^-e_r (times 2^-f for a bf16 chunk tile)
        const int r = tid;
        const int row = row0 + r;
        const int t = min(row, R - 1) / g;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float inv_row = rowinv[r];
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        auto wait_warp = [&](uint32_t bar_addr, uint32_t parity) {
            return __all_sync(kFullMask, wait_or_fail(bar_addr, parity, fail, p.dev_status, p.wait_limit));
        };
        for (int i = 0; i < c.n_tiles; ++i) {
            const int b = i & 1;
            if (!(ok = wait_warp(B(kF8SFull + b), (i >> 1) & 1)))
                break;
            float inv = inv_row;
            if (kChunkBf16 && i >= c.n_pre) {
                // the chunk tile's key scale 2^-f, published with its terms
                const int cc = i - c.n_pre;
                if (!(ok = wait_warp(B(kF8KScale + cc % kF8KScaleRing), (cc / kF8KScaleRing) & 1)))
                    break;
                inv *= reinterpret_cast<const volatile float *>(gbase + kF8OffKScale)[cc % kF8KScaleRing];
            }
            const uint64_t inv2 = f32x2_pack(inv, inv);
            tc_fence_after_sync();
            uint32_t sr0[32], sr1[32];
            tmem_ld32(lane_base + kColS + b * kTcKeys, sr0);
            tmem_ld32(lane_base + kColS + b * kTcKeys + 32, sr1);
            tmem_wait_ld();
            float s[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                s[j] = __uint_as_float(sr0[j]);
                s[j + 32] = __uint_as_float(sr1[j]);
            }
            const int lim = i < c.n_pre ? c.P - i * kTcKeys : t + 1 - (i - c.n_pre) * kTcKeys;
            if (lim < kTcKeys) {
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j >= lim)
                        s[j] = -INFINITY;
            }
            float pm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                pm[k] = fmax3(fmax3(s[8 * k], s[8 * k + 1], s[8 * k + 2]), fmax3(s[8 * k + 3], s[8 * k + 4], s[8 * k + 5]),
                              fmaxf(s[8 * k + 6], s[8 * k + 7]));
            const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7])) * inv;
            const bool need = mx > m_used + kRescaleLog2;
            const float m_new = need ? mx : m_used;
            const float mbase = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = need ? fast_exp2(m_used - mbase) : 1.f;
            const uint64_t neg2 = f32x2_pack(-mbase, -mbase);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint64_t d = fma_f32x2(f32x2_pack(s[2 * j], s[2 * j + 1]), inv2, neg2);
                s[2 * j] = fast_exp2(f32x2_lo(d));
                s[2 * j + 1] = fast_exp2(f32x2_hi(d));
                acc[j & 3] = add_f32x2(acc[j & 3], f32x2_pack(s[2 * j], s[2 * j + 1]));
            }
            const uint64_t a01 = add_f32x2(acc[0], acc[1]), a23 = add_f32x2(acc[2], acc[3]);
            const uint64_t a = add_f32x2(a01, a23);
            const float sum = f32x2_lo(a) + f32x2_hi(a);
            l = l * alpha + sum;
            m_used = m_new;
            {
                uint32_t pw[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    pw[j] = pack_f16x2(s[2 * j], s[2 * j + 1]);
                tmem_st32(lane_base + kColP + b * kColPStride, pw);
            }
            if (__any_sync(kFullMask, need) && i >= 1) {
                const int pb = (i - 1) & 1;
                if (!(ok = wait_warp(B(kF8PvDone + pb), ((i - 1) >> 1) & 1)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + kColO + 32 * cb, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(lane_base + kColO + 32 * cb, o);
                }
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(B(kF8PFull + b));
        }
        if (ok) {
            const int last = c.n_tiles - 1;
            ok = wait_warp(B(kF8PvDone + (last & 1)), (last >> 1) & 1);
        }
        if (ok)
            store_out_row(p, c, h, row, R, g, t, lane_base, l);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

} // namespace

namespace {

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// E4M3 rows [rows][hkv][128] as a 3-D tensor (bytes, head, row), read in
// boxes of 64 rows of one head in the 128-byte swizzle; rows outside read as
// zeros.
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *base, int64_t rows, int hkv)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(hkv),
                                static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(hkv) * kHeadDim};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 1u, static_cast<cuuint32_t>(kTcKeys)};
    const cuuint32_t elem[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor maps of the all-E4M3 kernel, or false when that kernel cannot
// run (no encoder, or row coordinates beyond 32 bits).
bool fill_tensor_maps(ExtendParams &q)
{
    constexpr int64_t kMaxRows = (int64_t{1} << 31) - 2 * kTcKeys;
    if (q.prefix_rows >= kMaxRows || q.q_rows >= kMaxRows || q.q_rows < 1)
        return false;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr)
        return false;
    // with no prefix rows no prefix tile is ever loaded: the chunk rows stand in
    const bool has_prefix = q.prefix_rows > 0;
    const void *kp = has_prefix ? static_cast<const void *>(q.k_prefix) : q.k_chunk;
    const void *vp = has_prefix ? static_cast<const void *>(q.v_prefix) : q.v_chunk;
    const int64_t prows = has_prefix ? q.prefix_rows : q.q_rows;
    return encode_rows(enc, &q.tm_k_prefix, kp, prows, q.hkv) && encode_rows(enc, &q.tm_v_prefix, vp, prows, q.hkv) &&
           encode_rows(enc, &q.tm_k_chunk, q.k_chunk, q.q_rows, q.hkv) &&
           encode_rows(enc, &q.tm_v_chunk, q.v_chunk, q.q_rows, q.hkv);
}

} // namespace

constexpr int64_t kMixedPrefixRatio = 8;

cudaError_t launch_extend_attention(const ExtendParams &p, cudaStream_t s)
{
    const int64_t rows = static_cast<int64_t>(p.max_q_len) * p.group;
    const dim3 grid(static_cast<unsigned>((rows + kTcRows - 1) / kTcRows), p.hkv, p.batch);
    if (p.chunk_e4m3 || p.prefix_rows >= kMixedPrefixRatio * static_cast<int64_t>(p.q_rows)) {
        // E4M3 prefix tiles (and chunk tiles, when E4M3 too): the TMA +
        // kind::f8f6f4 kernel; bf16 chunk tiles go through its converters,
        // at a higher cost per tile than on the kind::f16 kernel, so a bf16
        // chunk takes this kernel only when the prefix rows outnumber the
        // chunk rows by kMixedPrefixRatio.
        ExtendParams q = p;
        if (fill_tensor_maps(q)) {
            const auto kernel = p.chunk_e4m3 ? (q.pool != nullptr ? extend_f8_kernel<true, false>
                                                                  : extend_f8_kernel<false, false>)
                                             : (q.pool != nullptr ? extend_f8_kernel<true, true>
                                                                  : extend_f8_kernel<false, true>);
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
            if (e != cudaSuccess)
                return e;
            kernel<<<grid, kF8Threads, kF8Smem, s>>>(q);
            return cudaGetLastError();
        }
    }
    const auto kernel = p.chunk_e4m3 ? (p.pool != nullptr ? extend_tc_kernel<true, true> : extend_tc_kernel<false, true>)
                                     : (p.pool != nullptr ? extend_tc_kernel<true, false> : extend_tc_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess)
        return e;
    kernel<<<grid, kTcThreads, kTcSmem, s>>>(p);
    return cudaGetLastError();
}

} // namespace nvfp4kv
