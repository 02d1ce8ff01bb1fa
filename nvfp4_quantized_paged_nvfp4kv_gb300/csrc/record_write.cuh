// Writing one 16-value block of a token-head row into a page-head record
// (layout in include/nvfp4kv.h), shared by the quantize-append kernels and the
// append step of the fused append + decode kernel.
#pragma once

#include "device_common.cuh"

namespace nvfp4kv {

// One 16-value block of an input row, as loaded (fp32 or bf16 bits).
template <bool kBf16>
struct RawBlock {
    uint4 v[kBf16 ? 2 : 4];
};

template <bool kBf16>
__device__ __forceinline__ void load_raw(const void *src, size_t elem_off, RawBlock<kBf16> &r)
{
    const uint4 *p = kBf16 ? reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + elem_off)
                           : reinterpret_cast<const uint4 *>(static_cast<const float *>(src) + elem_off);
#pragma unroll
    for (int i = 0; i < (kBf16 ? 2 : 4); ++i)
        r.v[i] = __ldg(p + i);
}

template <bool kBf16>
__device__ __forceinline__ void unpack(const RawBlock<kBf16> &r, float (&x)[16])
{
    if constexpr (kBf16) {
        const uint32_t w[8] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w, r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[4 * k] = __uint_as_float(r.v[k].x);
            x[4 * k + 1] = __uint_as_float(r.v[k].y);
            x[4 * k + 2] = __uint_as_float(r.v[k].z);
            x[4 * k + 3] = __uint_as_float(r.v[k].w);
        }
    }
}

template <bool kBf16>
__device__ __forceinline__ void load16(const void *src, size_t elem_off, float (&x)[16])
{
    RawBlock<kBf16> r;
    load_raw<kBf16>(src, elem_off, r);
    unpack<kBf16>(r, x);
}

// A tensor scale G and r = RN(1/G); r = 0 where G lies outside [2^-32, 2^32]
// (every quotient then takes the IEEE division) and at G = 1 (no division).
struct TensorScale {
    float G, r;
};

__device__ __forceinline__ TensorScale tensor_scale(float G)
{
    return {G, (G != 1.f && G >= 0x1p-32f && G <= 0x1p32f) ? __frcp_rn(G) : 0.f};
}

// Values relative to the tensor scale G: the block procedure runs on the
// correctly rounded quotients y = fl32(x / G) (nothing to do at G = 1).
// Returns the code flip quantize_block must apply: kCodeFlip when x now
// holds y, 0 when it holds -y (the division-free path, which ends on the
// negated quotients; quantize_block negates its input anyway).
//
// No division per element.  With r = RN(1/G), q0 = RN(x r) is within two ulps
// of x / G; one correction step, q1 = RN(q0 + (x - q0 G) r) with the
// remainder through an FMA, brings it within one ulp, and a second gives
// RN(x / G) exactly (Markstein's theorem: a quotient within one ulp, corrected
// once with the correctly rounded reciprocal, is the correctly rounded
// quotient when nothing underflows or overflows).  G in [2^-32, 2^32] and
// |x| < 2^64 keep every step finite and r normal.  The remainder can lose
// bits only for |x| < 2^-80, and there |x / G| < 2^-48: no such value decides
// a code or a scale (a block of them has scale 0; beside a larger value,
// whose scale is at least 2^-9, they give a zero code), and the steps keep
// its sign.  A block with a larger value takes the IEEE division.  The steps
// run on the negated terms -- q0' = RN(x (-r)), e = RN(x + q0' G) = x - q0 G,
// q' = RN(q0' + e (-r)) = -q, twice -- so that a zero quotient keeps the sign
// of x (a remainder that cancels is +0, and -0 + -0 stays -0) and x needs no
// negation.
constexpr uint32_t kCodeFlip = 0x88888888u;

__device__ __forceinline__ uint32_t divide_by_tensor_scale(float (&x)[16], TensorScale ts)
{
    if (ts.G == 1.f)
        return kCodeFlip;
    const float m = fmaxf(fmax3(fmax3(fabsf(x[0]), fabsf(x[1]), fabsf(x[2])),
                                fmax3(fabsf(x[3]), fabsf(x[4]), fabsf(x[5])),
                                fmax3(fabsf(x[6]), fabsf(x[7]), fabsf(x[8]))),
                          fmax3(fmax3(fabsf(x[9]), fabsf(x[10]), fabsf(x[11])),
                                fmax3(fabsf(x[12]), fabsf(x[13]), fabsf(x[14])), fabsf(x[15])));
    if (ts.r != 0.f && m < 0x1p64f) {
        const uint64_t nr2 = f32x2_pack(-ts.r, -ts.r), g2 = f32x2_pack(ts.G, ts.G);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint64_t v2 = f32x2_pack(x[2 * j], x[2 * j + 1]);
            uint64_t q = mul_f32x2(v2, nr2);
            q = fma_f32x2(fma_f32x2(q, g2, v2), nr2, q);
            q = fma_f32x2(fma_f32x2(q, g2, v2), nr2, q);
            x[2 * j] = f32x2_lo(q);
            x[2 * j + 1] = f32x2_hi(q);
        }
        return 0u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
        x[i] = __fdiv_rn(x[i], ts.G);
    return kCodeFlip;
}

__device__ __forceinline__ uint32_t divide_by_tensor_scale(float (&x)[16], float G)
{
    return G != 1.f ? divide_by_tensor_scale(x, tensor_scale(G)) : kCodeFlip;
}

// The value s of an E4M3 block-scale byte S (0 .. 126) and RN(1/s) (0 for
// s = 0), computed on the spot ...
struct ScaleOfByte {
    __device__ __forceinline__ float2 operator()(uint32_t S) const
    {
        const float sc = e4m3_to_f32(S);
        return make_float2(sc, sc != 0.f ? __frcp_rn(sc) : 0.f);
    }
};

// ... or read from a table of all 128 bytes in shared memory, filled by
// fill_scale_table (the same values, computed once per CTA).
struct ScaleTable {
    const float2 *t;
    __device__ __forceinline__ float2 operator()(uint32_t S) const { return t[S]; }
};

// Whole CTA (at least 128 threads' worth of entries are filled in a loop);
// the caller synchronises the CTA before the first read.
__device__ __forceinline__ void fill_scale_table(float2 *t)
{
    for (uint32_t i = threadIdx.x; i < 128u; i += blockDim.x)
        t[i] = i < 127u ? ScaleOfByte()(i) : make_float2(0.f, 0.f);
}

// amax -> E4M3 block scale -> 16 E2M1 codes (code i in bits 4i .. 4i+3).
//
// The scale is decided on fl32(amax / 6) and each code on the IEEE quotient
// fl32(x / s).  Both are computed without a division per element: with
// r = RN(1/s), q0 = RN(x r) is within an ulp of x / s, the remainder x - q0 s
// is exact through one FMA, and RN(q0 + (x - q0 s) r) is the correctly
// rounded quotient (Markstein's correction step).  s has at most four
// significant bits, so only eight mantissas occur; every fp32 quotient in the
// range that decides a code is compared against an IEEE division for all eight
// in the GPU tests.  The step runs on the negated terms -- q0' = RN(x (-r)),
// e = RN(x + q0' s), q' = RN(q0' + e (-r)) = -RN(x / s) exactly -- because then
// a zero quotient keeps the sign of x (a remainder that cancels to zero is +0,
// and -0 + -0 is -0 where +0 + -0 would lose it); E2M1 rounding is symmetric,
// so the codes of -q' are those of q' with each sign bit flipped (flip =
// kCodeFlip).  Given x = -y (flip = 0), the same steps end on RN(y / s) and
// its codes need no flip.
template <class ScaleFn = ScaleOfByte>
__device__ __forceinline__ void quantize_block(const float (&x)[16], uint32_t &scale_byte, uint32_t (&packed)[2],
                                               ScaleFn scale_of = ScaleFn(), uint32_t flip = kCodeFlip)
{
    // amax with three-input maxima (a NaN element is ignored, as by fmaxf);
    // capped at the largest finite float so the quotient below stays finite
    // (any amax above 6 * 448 saturates the scale the same way)
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        a[i] = fabsf(x[i]);
    const float m = fmaxf(fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmax3(a[6], a[7], a[8])),
                          fmax3(fmax3(a[9], a[10], a[11]), fmax3(a[12], a[13], a[14]), a[15]));
    const float amax = fminf(fmaxf(m, 0.f), 3.40282347e+38f);   // an all-NaN block has amax 0
    // fl32(amax / 6) by the same correction step as the elements below, with
    // RN(1/6) = 0x3E2AAAAB
    const float sixth = __uint_as_float(0x3E2AAAABu);
    const float d0 = __fmul_rn(amax, sixth);
    const float s32 = __fmaf_rn(__fmaf_rn(-d0, 6.0f, amax), sixth, d0);
    scale_byte = f32x2_to_e4m3x2(s32, 0.f) & 0xffu;
    const float2 sr = scale_of(scale_byte);
    const float sc = sr.x;
    packed[0] = packed[1] = 0u;
    if (sc != 0.f) {
        // the quotient step two lanes at a time (packed fp32, each lane IEEE)
        const uint64_t nr2 = f32x2_pack(-sr.y, -sr.y), sc2 = f32x2_pack(sc, sc);
        float q[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint64_t v2 = f32x2_pack(x[2 * j], x[2 * j + 1]);
            const uint64_t q0 = mul_f32x2(v2, nr2);
            const uint64_t qq = fma_f32x2(fma_f32x2(q0, sc2, v2), nr2, q0);
            q[2 * j] = f32x2_lo(qq);
            q[2 * j + 1] = f32x2_hi(qq);
        }
        packed[0] = f32x8_to_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]) ^ flip;
        packed[1] = f32x8_to_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]) ^ flip;
    }
}

// NVFP4: quantise x (block blk of token tok of the record) and write it.  K
// rows are natural (one 8-byte store); a V block is merged into the 8 words
// that hold its token pair with atomic AND/OR on the thread's own nibbles.
template <class ScaleFn = ScaleOfByte>
__device__ __forceinline__ void write_nvfp4_block(uint8_t *rec, bool is_v, int tok, int blk, const float (&x)[16],
                                                  ScaleFn scale_of = ScaleFn(), uint32_t flip = kCodeFlip)
{
    uint32_t S, packed[2];
    quantize_block(x, S, packed, scale_of, flip);
    if (!is_v) {
        *reinterpret_cast<uint2 *>(rec + tok * 64 + blk * 8) = make_uint2(packed[0], packed[1]);
        rec[2048 + tok * 8 + blk] = static_cast<uint8_t>(S);
        return;
    }
    // channel 16*blk + r (r = g + 8w) goes to row tok/2, group g at chunk
    // position (g + 2*row) mod 8, byte 2*blk + w, nibble (tok & 1).
    const int row = tok >> 1, half = tok & 1;
    const uint64_t codes = (static_cast<uint64_t>(packed[1]) << 32) | packed[0];
    const uint32_t shift = 16u * (blk & 1);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t c0 = static_cast<uint32_t>(codes >> (4 * g)) & 15u;        // channel 16blk + g
        const uint32_t c1 = static_cast<uint32_t>(codes >> (4 * (g + 8))) & 15u;  // channel 16blk + g + 8
        const uint32_t unit = (c0 << (4 * half)) | (c1 << (8 + 4 * half));
        const uint32_t mask = (0xFu << (4 * half)) | (0xFu << (8 + 4 * half));
        unsigned int *word = reinterpret_cast<unsigned int *>(
            rec + 1024 + row * 128 + ((g + 2 * row) & 7) * 16 + ((2 * blk) & ~3));
        atomicAnd(word, ~(mask << shift));
        atomicOr(word, unit << shift);
    }
    rec[2176 + row * 16 + blk * 2 + half] = static_cast<uint8_t>(S);
}

// NVFP4, V block blk of both tokens of a token pair (tok0 even, tok0 + 1), from
// their scale bytes and codes: every byte of theirs is written whole, no atomics.
// Byte 2*blk of chunk group g holds channel 16blk + g (low nibble token tok0,
// high nibble tok0 + 1) and byte 2*blk + 1 channel 16blk + g + 8.  The nibble
// pairs are formed a word at a time: from the codes a (tok0) and b (tok0 + 1)
// of eight channels, (a & 0x0F0F0F0F) | ((b << 4) & 0xF0F0F0F0) holds the even
// channels' bytes and ((a >> 4) & 0x0F0F0F0F) | (b & 0xF0F0F0F0) the odd ones';
// one byte permutation then pairs the low and high channel bytes of two groups.
__device__ __forceinline__ void write_nvfp4_v_pair(uint8_t *rec, int tok0, int blk, uint32_t S0,
                                                   const uint32_t (&p0)[2], uint32_t S1, const uint32_t (&p1)[2])
{
    const int row = tok0 >> 1;
    constexpr uint32_t kLo = 0x0F0F0F0Fu;
    const uint32_t el = (p0[0] & kLo) | ((p1[0] << 4) & ~kLo);     // groups 0,2,4,6: channel 16blk + g
    const uint32_t ol = ((p0[0] >> 4) & kLo) | (p1[0] & ~kLo);     // groups 1,3,5,7
    const uint32_t eh = (p0[1] & kLo) | ((p1[1] << 4) & ~kLo);     // the same groups, channel 16blk + g + 8
    const uint32_t oh = ((p0[1] >> 4) & kLo) | (p1[1] & ~kLo);
    const uint32_t w[4] = {__byte_perm(el, eh, 0x5140), __byte_perm(ol, oh, 0x5140),   // groups {0,2}, {1,3}
                           __byte_perm(el, eh, 0x7362), __byte_perm(ol, oh, 0x7362)};  // groups {4,6}, {5,7}
    uint8_t *base = rec + 1024 + row * 128 + 2 * blk;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t word = w[(g & 1) | ((g >> 2) << 1)];
        const uint32_t v = ((g >> 1) & 1) ? (word >> 16) : word;
        *reinterpret_cast<uint16_t *>(base + ((g + 2 * row) & 7) * 16) = static_cast<uint16_t>(v);
    }
    *reinterpret_cast<uint16_t *>(rec + 2176 + row * 16 + blk * 2) = static_cast<uint16_t>(S0 | (S1 << 8));
}

// FP8: each value E4M3_rn_satfinite(x); K chunk blk of row tok sits at position
// (blk + (tok & 1)) mod 8; V channel 8c + i of token 2*row + half is byte
// 2i + half of chunk c, at chunk position (c + f(row)) mod 16.
__device__ __forceinline__ void write_fp8_block(uint8_t *rec, bool is_v, int tok, int blk, const float (&x)[16])
{
    if (!is_v) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = f32x2_to_e4m3x2(x[4 * k], x[4 * k + 1]) | (f32x2_to_e4m3x2(x[4 * k + 2], x[4 * k + 3]) << 16);
        *reinterpret_cast<uint4 *>(rec + tok * 128 + ((blk + (tok & 1)) & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
        return;
    }
    const int row = tok >> 1, half = tok & 1;
    const int f = (row & 1) + 4 * ((row >> 1) & 1);
    uint8_t *vrow = rec + 2048 + row * 256;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * blk + cc;
        uint8_t *chunk = vrow + ((c + f) & 15) * 16;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t two = f32x2_to_e4m3x2(x[8 * cc + i], x[8 * cc + i + 1]);
            chunk[2 * i + half] = static_cast<uint8_t>(two & 0xffu);
            chunk[2 * (i + 1) + half] = static_cast<uint8_t>(two >> 8);
        }
    }
}

} // namespace nvfp4kv
