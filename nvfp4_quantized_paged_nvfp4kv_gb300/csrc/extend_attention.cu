// Extend attention over the FP8 prefix workspace and the current chunk.
//
// "SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation: on the
// extend path the cached prefix is dequantised into one FP8 workspace and the
// new chunk attends over it and over itself.  Chunk token t of a sequence
// with prefix length P sees the P prefix keys and chunk keys 0 .. t.
//
// One CTA owns 128 rows of one sequence and one kv head, a row being a
// (chunk token, query head of the group) pair taken token-major, so the g
// query heads that share a kv head read each key tile once.  Eight warps own
// 16 rows each and run a flash-attention forward over key tiles of 64:
// S = Q K^T and O += P V on mma.sync m16n8k16 (f16 operands, fp32
// accumulators), online softmax in base 2 with sm_scale * log2(e) folded
// into Q.  The CTA converts every key tile once into f16 shared memory
// (E4M3 -> f16 and bf16 -> f16, both exact in range), double buffered, while
// the next tile's raw bytes are in flight by cp.async.
//
// The appending variant also writes the chunk's K/V into the NVFP4 cache
// ("SGLang stores KV cache in 4 bits", Interpretation: prefill quantises the
// new K/V into the cache): each chunk key tile has one owning CTA, which
// stages it through shared memory and quantises it before its attention loop.
// Every row tile of a kv head reads the same chunk tiles, so the chunk stays
// in L2 and no separate pass over it is needed.
#include "record_write.cuh"

namespace nvfp4kv {
namespace {

constexpr int kExtWarps = 8;
constexpr int kExtThreads = 32 * kExtWarps;
constexpr int kExtRows = 16 * kExtWarps;                  // rows per CTA
constexpr int kExtKeys = 64;                              // keys per tile
constexpr uint32_t kTileBytes = kExtKeys * kHeadDim * 2;  // one f16 K or V tile
constexpr uint32_t kF16Bytes = 2 * 2 * kTileBytes;        // [buffer][K, V] f16 tiles

static_assert(kExtKeys * kHeadDim / 16 == 2 * kExtThreads, "FP8 tile: two 16-byte pieces a thread");
static_assert(kExtKeys * kHeadDim / 8 == 4 * kExtThreads, "bf16 tile: four 16-byte pieces a thread");

// Byte offset of 16-byte chunk c (channels 8c .. 8c + 7) of key row `key` in
// an f16 tile: 256-byte rows, chunks XOR-swizzled by the row's low three bits
// so that eight rows read at one chunk index hit eight different bank groups.
__device__ __forceinline__ uint32_t tile_off(uint32_t key, uint32_t c)
{
    return key * 256u + ((c ^ (key & 7u)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Two bf16 (low half first) to f16x2, round to nearest even.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t bf16x2_scaled_f16x2(uint32_t w, float s)
{
    return pack_f16x2(__uint_as_float(w << 16) * s, __uint_as_float(w & 0xffff0000u) * s);
}

// Where the CTA is in its sequence and which tiles it visits.
struct ExtCta {
    int c0;          // first chunk row of the sequence
    int C;           // chunk length
    int P;           // prefix length
    int64_t p0;      // first prefix row of the sequence
    int n_pre;       // prefix tiles
    int n_tiles;     // prefix tiles + chunk tiles
    int t_min;       // smallest chunk token among the CTA's rows
};

// Raw bytes of one key tile are staged with cp.async into a per-thread slot
// array: piece u of thread tid sits at stage + (u * kExtThreads + tid) * 16.
// FP8 prefix tiles use pieces 0..3 (K, K, V, V), bf16 chunk tiles 0..7 (K x4,
// V x4).  Each thread converts only the pieces it copied, so a wait on its own
// copies is enough before the conversion.
constexpr uint32_t kStageBytes = 8 * kExtThreads * 16;
constexpr uint32_t kExtSmem = kF16Bytes + kStageBytes;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Start the copies of tile i; keys past the prefix or chunk read as zeros.
__device__ __forceinline__ void load_tile(const ExtendParams &p, const ExtCta &c, int h, int i, uint32_t stage)
{
    const int tid = threadIdx.x;
    if (i < c.n_pre) {
        const int k0 = i * kExtKeys;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + kExtThreads * (u & 1);
            const int key = idx >> 3, piece = idx & 7;
            const uint8_t *base = u < 2 ? p.k_prefix : p.v_prefix;
            const bool ok = k0 + key < c.P;
            const uint8_t *src = ok ? base + ((c.p0 + k0 + key) * p.hkv + h) * kHeadDim + 16 * piece : base;
            cp_async16(stage + (u * kExtThreads + tid) * 16u, src, ok);
        }
    } else {
        const int k0 = (i - c.n_pre) * kExtKeys;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = tid + kExtThreads * (u & 3);
            const int key = idx >> 4, piece = idx & 15;
            const uint16_t *base = u < 4 ? p.k_chunk : p.v_chunk;
            const bool ok = k0 + key < c.C;
            const uint16_t *src =
                ok ? base + (static_cast<int64_t>(c.c0 + k0 + key) * p.hkv + h) * kHeadDim + 8 * piece : base;
            cp_async16(stage + (u * kExtThreads + tid) * 16u, src, ok);
        }
    }
    cp_async_commit();
}

// Wait for this thread's copies of tile i, convert them to f16 and store them
// into buffer `buf` (K tile at buf, V tile at buf + kTileBytes).
__device__ __forceinline__ void store_tile(const ExtCta &c, int i, uint32_t stage, uint32_t buf)
{
    const int tid = threadIdx.x;
    cp_async_wait_all();
    if (i < c.n_pre) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + kExtThreads * (u & 1);
            const uint32_t key = idx >> 3, piece = idx & 7;
            const uint32_t dst = buf + (u < 2 ? 0u : kTileBytes);
            const uint4 w = lds128(stage + (u * kExtThreads + tid) * 16u);
            uint4 lo, hi;
            e4m3x4_to_f16x2x2(w.x, lo.x, lo.y);
            e4m3x4_to_f16x2x2(w.y, lo.z, lo.w);
            e4m3x4_to_f16x2x2(w.z, hi.x, hi.y);
            e4m3x4_to_f16x2x2(w.w, hi.z, hi.w);
            // the upper four pieces of a row store their high half first, so
            // each group of eight lanes covers all eight bank groups
            const uint32_t first = (piece >> 2) & 1u;
            sts128(dst + tile_off(key, 2 * piece + first), first ? hi : lo);
            sts128(dst + tile_off(key, 2 * piece + 1 - first), first ? lo : hi);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = tid + kExtThreads * (u & 3);
            const uint32_t key = idx >> 4, piece = idx & 15;
            const uint32_t dst = buf + (u < 4 ? 0u : kTileBytes);
            const uint4 w = lds128(stage + (u * kExtThreads + tid) * 16u);
            uint4 h;
            h.x = bf16x2_to_f16x2(w.x);
            h.y = bf16x2_to_f16x2(w.y);
            h.z = bf16x2_to_f16x2(w.z);
            h.w = bf16x2_to_f16x2(w.w);
            sts128(dst + tile_off(key, piece), h);
        }
    }
}

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

__device__ __forceinline__ void staged_block(const uint8_t *src, float (&x)[16], float G)
{
    RawBlock<true> r;
    r.v[0] = *reinterpret_cast<const uint4 *>(src);
    r.v[1] = *reinterpret_cast<const uint4 *>(src + 16);
    unpack<true>(r, x);
    divide_by_tensor_scale(x, G);
}

// Quantise chunk keys k0 .. k0 + 63 of kv head h from the staged raw tile (K
// rows at `raw`, V rows at raw + 64 * 256, 256 bytes a key) into the cache.
// K: 64 keys x 8 blocks, two a thread.  V: 32 key pairs x 8 blocks, one a
// thread; a pair on an even slot and its successor is written whole, any
// other token through the atomic nibble merge.
__device__ __forceinline__ void append_tile(const ExtendParams &p, const ExtCta &c, int h, int k0, const uint8_t *raw)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int item = tid + kExtThreads * u;
        const int key = item >> 3, blk = item & 7;
        if (k0 + key >= c.C)
            continue;
        size_t rec;
        int tok;
        if (!append_site(p, p.slot_mapping[c.c0 + k0 + key], h, rec, tok, blk == 0))
            continue;
        float x[16];
        staged_block(raw + key * 256 + blk * 32, x, p.gscale);
        write_nvfp4_block(p.pool + rec, false, tok, blk, x);
    }
    const int key0 = 2 * (tid >> 3), blk = tid & 7;
    const uint8_t *vraw = raw + kExtKeys * 256;
    const bool has0 = k0 + key0 < c.C, has1 = k0 + key0 + 1 < c.C;
    const int s0 = has0 ? p.slot_mapping[c.c0 + k0 + key0] : -1;
    const int s1 = has1 ? p.slot_mapping[c.c0 + k0 + key0 + 1] : -1;
    size_t rec0 = 0, rec1 = 0;
    int tok0 = 0, tok1 = 0;
    const bool ok0 = has0 && append_site(p, s0, h, rec0, tok0, false);
    const bool ok1 = has1 && append_site(p, s1, h, rec1, tok1, false);
    float x[16];
    if (ok0 && ok1 && (s0 & 1) == 0 && s1 == s0 + 1) {
        uint32_t S0, S1, c0[2], c1[2];
        staged_block(vraw + key0 * 256 + blk * 32, x, p.gscale);
        quantize_block(x, S0, c0);
        staged_block(vraw + (key0 + 1) * 256 + blk * 32, x, p.gscale);
        quantize_block(x, S1, c1);
        write_nvfp4_v_pair(p.pool + rec0, tok0, blk, S0, c0, S1, c1);
        return;
    }
    if (ok0) {
        staged_block(vraw + key0 * 256 + blk * 32, x, p.gscale);
        write_nvfp4_block(p.pool + rec0, true, tok0, blk, x);
    }
    if (ok1) {
        staged_block(vraw + (key0 + 1) * 256 + blk * 32, x, p.gscale);
        write_nvfp4_block(p.pool + rec1, true, tok1, blk, x);
    }
}

// One key tile for one warp's 16 rows.  lim_a / lim_b: keys of the tile that
// rows a (lane / 4) and b (lane / 4 + 8) see, counted from the tile's start;
// only read when `masked`.
__device__ __forceinline__ void tile_step(uint32_t kbuf, uint32_t vbuf, const uint32_t (&qa)[8][4],
                                          float (&o)[16][4], float &m_a, float &m_b, float &l_a, float &l_b,
                                          bool masked, int lim_a, int lim_b)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t rr = lane & 7u, mi = lane >> 3;

    // S = Q K^T: eight n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t chunk = 2 * ks + (mi & 1u);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            const uint32_t key = 16 * np + 8 * (mi >> 1) + rr;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbuf + key * 256u + ((chunk ^ rr) << 4), b0, b1, b2, b3);
            mma_f16_16816(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            mma_f16_16816(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
    }

    if (masked) {
        const int q2 = 2 * static_cast<int>(lane & 3u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = 8 * j + q2 + (e & 1);
                if (key >= (e < 2 ? lim_a : lim_b))
                    s[j][e] = -INFINITY;
            }
        }
    }

    // online softmax, base 2 (Q carries sm_scale * log2 e)
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        mx_a = fmaxf(mx_a, fmaxf(s[j][0], s[j][1]));
        mx_b = fmaxf(mx_b, fmaxf(s[j][2], s[j][3]));
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    // a row that has seen no key yet keeps zero weights
    const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
    const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float al_a = fast_exp2(m_a - base_a), al_b = fast_exp2(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        s[j][0] = fast_exp2(s[j][0] - base_a);
        s[j][1] = fast_exp2(s[j][1] - base_a);
        s[j][2] = fast_exp2(s[j][2] - base_b);
        s[j][3] = fast_exp2(s[j][3] - base_b);
        sum_a += s[j][0] + s[j][1];
        sum_b += s[j][2] + s[j][3];
    }
    l_a = l_a * al_a + sum_a;
    l_b = l_b * al_b + sum_b;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        o[j][0] *= al_a;
        o[j][1] *= al_a;
        o[j][2] *= al_b;
        o[j][3] *= al_b;
    }

    // O += P V: four k-steps of 16 keys, sixteen n-tiles of 8 channels
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint32_t a0 = pack_f16x2(s[2 * kk][0], s[2 * kk][1]);
        const uint32_t a1 = pack_f16x2(s[2 * kk][2], s[2 * kk][3]);
        const uint32_t a2 = pack_f16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        const uint32_t a3 = pack_f16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
        const uint32_t key = 16 * kk + 8 * (mi & 1u) + rr;
#pragma unroll
        for (int cp = 0; cp < 8; ++cp) {
            const uint32_t chunk = 2 * cp + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vbuf + key * 256u + ((chunk ^ rr) << 4), b0, b1, b2, b3);
            mma_f16_16816(o[2 * cp], a0, a1, a2, a3, b0, b1);
            mma_f16_16816(o[2 * cp + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

template <bool kAppend>
__global__ void __launch_bounds__(kExtThreads, 1) extend_kernel(const ExtendParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int b = blockIdx.z;
    const int h = blockIdx.y;
    const int tile = static_cast<int>(gridDim.x - 1 - blockIdx.x);  // later rows see more keys: start them first
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    ExtCta c;
    c.c0 = p.q_indptr[b];
    const int c1 = p.q_indptr[b + 1];
    c.P = p.prefix_lens[b];
    const int kv0 = p.kv_indptr[b];
    if (c.c0 < 0 || c1 < c.c0 || c1 > p.q_rows || c1 - c.c0 > p.max_q_len || c.P < 0 || kv0 < 0 ||
        static_cast<int64_t>(kv0) + c.P > p.prefix_rows) {
        if (threadIdx.x == 0)
            report(p.dev_status, NVFP4KV_DEV_BAD_LEN);
        return;
    }
    c.C = c1 - c.c0;
    c.p0 = kv0;
    const int g = p.group;
    const int R = c.C * g;                 // rows of this sequence and kv head
    const int row0 = tile * kExtRows;
    if (row0 >= R)
        return;
    const int row_end = min(row0 + kExtRows, R);
    c.t_min = row0 / g;
    const int t_max = (row_end - 1) / g;
    c.n_pre = (c.P + kExtKeys - 1) / kExtKeys;
    c.n_tiles = c.n_pre + t_max / kExtKeys + 1;
    // chunk key tiles this CTA appends: those whose first key's first row
    // (64 kt g) falls in its row range
    const int own_lo = (row0 + kExtKeys * g - 1) / (kExtKeys * g);
    const int own_hi = (row0 + kExtRows + kExtKeys * g - 1) / (kExtKeys * g);

    // this lane's two rows; rows past the end repeat the last row and are not stored
    const int r_a = row0 + 16 * warp + (lane >> 2);
    const int r_b = r_a + 8;
    const bool warp_live = row0 + 16 * warp < R;
    const int t_a = min(r_a, R - 1) / g, t_b = min(r_b, R - 1) / g;
    const int hq_a = h * g + (min(r_a, R - 1) - t_a * g);
    const int hq_b = h * g + (min(r_b, R - 1) - t_b * g);
    const int t_warp_max = min(row0 + 16 * warp + 15, R - 1) / g;

    // Q fragments, scaled by sm_scale * log2 e and rounded to f16
    uint32_t qa[8][4];
    {
        const int q2 = 2 * (lane & 3);
        const uint16_t *qa_row = p.q + (static_cast<int64_t>(c.c0 + t_a) * p.hq + hq_a) * kHeadDim + q2;
        const uint16_t *qb_row = p.q + (static_cast<int64_t>(c.c0 + t_b) * p.hq + hq_b) * kHeadDim + q2;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t wa0 = *reinterpret_cast<const uint32_t *>(qa_row + 16 * ks);
            const uint32_t wb0 = *reinterpret_cast<const uint32_t *>(qb_row + 16 * ks);
            const uint32_t wa1 = *reinterpret_cast<const uint32_t *>(qa_row + 16 * ks + 8);
            const uint32_t wb1 = *reinterpret_cast<const uint32_t *>(qb_row + 16 * ks + 8);
            qa[ks][0] = bf16x2_scaled_f16x2(wa0, p.qscale);
            qa[ks][1] = bf16x2_scaled_f16x2(wb0, p.qscale);
            qa[ks][2] = bf16x2_scaled_f16x2(wa1, p.qscale);
            qa[ks][3] = bf16x2_scaled_f16x2(wb1, p.qscale);
        }
    }

    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    const uint32_t sbase = smem_addr(smem);
    const uint32_t stage = sbase + kF16Bytes;
    if constexpr (kAppend) {
        // the chunk key tiles this CTA owns go into the cache first, staged
        // through the same area; the attention below reads them from L2
        for (int kt = own_lo; kt < own_hi && kt * kExtKeys < c.C; ++kt) {
            load_tile(p, c, h, c.n_pre + kt, stage);
            cp_async_wait_all();
            __syncthreads();
            append_tile(p, c, h, kt * kExtKeys, smem + kF16Bytes);
            __syncthreads();
        }
    }
    load_tile(p, c, h, 0, stage);
    store_tile(c, 0, stage, sbase);
    __syncthreads();

    for (int i = 0; i < c.n_tiles; ++i) {
        const uint32_t buf = sbase + static_cast<uint32_t>(i & 1) * 2u * kTileBytes;
        if (i + 1 < c.n_tiles)
            load_tile(p, c, h, i + 1, stage);
        if (warp_live) {
            if (i < c.n_pre) {
                const int lim = c.P - i * kExtKeys;
                tile_step(buf, buf + kTileBytes, qa, o, m_a, m_b, l_a, l_b, lim < kExtKeys, lim, lim);
            } else {
                const int k0 = (i - c.n_pre) * kExtKeys;
                if (k0 <= t_warp_max) {
                    const bool masked = k0 + kExtKeys - 1 > c.t_min;
                    tile_step(buf, buf + kTileBytes, qa, o, m_a, m_b, l_a, l_b, masked, t_a + 1 - k0,
                              t_b + 1 - k0);
                }
            }
        }
        if (i + 1 < c.n_tiles)
            store_tile(c, i + 1, stage, sbase + static_cast<uint32_t>((i + 1) & 1) * 2u * kTileBytes);
        __syncthreads();
    }

    if (!warp_live)
        return;
    l_a += __shfl_xor_sync(kFullMask, l_a, 1);
    l_a += __shfl_xor_sync(kFullMask, l_a, 2);
    l_b += __shfl_xor_sync(kFullMask, l_b, 1);
    l_b += __shfl_xor_sync(kFullMask, l_b, 2);
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
    const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    const int q2 = 2 * (lane & 3);
    const int64_t off_a = (static_cast<int64_t>(c.c0 + t_a) * p.hq + hq_a) * kHeadDim + q2;
    const int64_t off_b = (static_cast<int64_t>(c.c0 + t_b) * p.hq + hq_b) * kHeadDim + q2;
    const bool st_a = r_a < R, st_b = r_b < R;
    if (p.out_f32) {
        float *out = static_cast<float *>(p.out);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (st_a)
                *reinterpret_cast<float2 *>(out + off_a + 8 * j) = make_float2(o[j][0] * inv_a, o[j][1] * inv_a);
            if (st_b)
                *reinterpret_cast<float2 *>(out + off_b + 8 * j) = make_float2(o[j][2] * inv_b, o[j][3] * inv_b);
        }
    } else {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (st_a)
                *reinterpret_cast<__nv_bfloat162 *>(out + off_a + 8 * j) =
                    __floats2bfloat162_rn(o[j][0] * inv_a, o[j][1] * inv_a);
            if (st_b)
                *reinterpret_cast<__nv_bfloat162 *>(out + off_b + 8 * j) =
                    __floats2bfloat162_rn(o[j][2] * inv_b, o[j][3] * inv_b);
        }
    }
}

} // namespace

cudaError_t launch_extend_attention(const ExtendParams &p, cudaStream_t s)
{
    static_assert(kExtSmem <= 227 * 1024, "shared memory");
    if (p.pool == nullptr)
        return launch_extend_attention_tc(p, s);
    const auto kernel = extend_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kExtSmem);
    if (e != cudaSuccess)
        return e;
    const int64_t rows = static_cast<int64_t>(p.max_q_len) * p.group;
    const dim3 grid(static_cast<unsigned>((rows + kExtRows - 1) / kExtRows), p.hkv, p.batch);
    kernel<<<grid, kExtThreads, kExtSmem, s>>>(p);
    return cudaGetLastError();
}

} // namespace nvfp4kv
