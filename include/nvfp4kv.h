/*
 * nvfp4kv -- NVFP4 paged KV cache for GQA decode on one GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  Every device pointer is a CUDA
 * device address owned by the caller; the library allocates no device memory
 * and keeps no state between calls except a per-device cache of the SM count
 * and the fixed scratch array of nvfp4kv_paged_decode_static_scratch.
 * Every launching call is asynchronous on the given stream: it validates its
 * arguments on the host first (returning an error and launching nothing when
 * they are bad), then enqueues its kernels and returns.  A NULL stream is the
 * legacy default stream.
 *
 * The method (from the pages this library implements; cited by title and
 * section):
 *   "SGLang stores KV cache in 4 bits: long-context decode throughput rises
 *   26-30%, ..." (summary of the LMSYS post "Accelerating Long-Context and
 *   Agentic Inference with NVFP4 KV Cache"), Interpretation: the KV cache is
 *   paged; each block of 16 values is 8 bytes of packed 4-bit data plus one
 *   byte of block scale; decode dequantises inside the attention kernel; the
 *   extend path dequantises the cached prefix into an FP8 workspace; prefill
 *   quantises the new K/V into the cache.  Perspective: the per-tensor FP32
 *   global scale is left at 1.0.
 *   "NVFP4-KV-Cache auf der NVIDIA RTX PRO 6000 Blackwell Server Edition",
 *   "Bytes pro Token": E2M1 elements (1 sign, 2 exponent, 1 mantissa bit),
 *   one FP8-E4M3 scale per 16 values, an FP32 tensor scale above them;
 *   "Unterstuetzung in den Engines": the FP8-E4M3 cache is the baseline.
 *
 * Formats (readings where the pages are silent):
 *   E2M1 code: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 *     magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   E4M3 (OCP "FN"): bias 7, subnormals m/8 * 2^-6, max 448, 0x7F = NaN.
 *   Tensor scale G (nvfp4kv_cache.global_scale, FP32; the pages run with
 *     G = 1.0 and name its calibration as the next step): a cached value is
 *     G * E4M3 block scale * E2M1 code.
 *   Block of 16 consecutive channels of one token-head, y_i = fl32(x_i / G)
 *     (y = x at G = 1):
 *     S = E4M3_rn_satfinite(fl32(amax_i |y_i| / 6)), s = value(S),
 *     q_i = E2M1_rn_satfinite(fl32(y_i / s)), or 0 for all i if s == 0.
 *     Packed byte j = q_{2j} | q_{2j+1} << 4 (low nibble = even channel).
 *
 * Cache layout.  The cache is one pool of page-head records: the record of
 * kv head h of physical page P starts at byte (P * num_kv_heads + h) * R and
 * holds the 16 tokens of that page for that head (token t of the page is the
 * one at slot P * 16 + t).  The pages give only the storage cost (8 packed
 * bytes + 1 scale byte per 16 values); the arrangement inside a record is this
 * library's, chosen so the decode stages a record with one bulk copy and reads
 * it without shared-memory bank conflicts.
 *
 * NVFP4 record, R = NVFP4KV_RECORD_BYTES = 2304:
 *   [0, 1024)     K data: 16 rows of 64 bytes, row t = token t; byte 8*b + i
 *                 of a row holds channels 16*b + 2i (low nibble) and
 *                 16*b + 2i + 1 (high nibble).
 *   [1024, 2048)  V data: 8 rows of 128 bytes; row p holds tokens 2p (low
 *                 nibbles) and 2p + 1 (high nibbles) of the same channel.  A row
 *                 is 8 chunks of 16 bytes; group g (0..7) sits in the chunk at
 *                 position (g + 2p) mod 8, and byte 2j + w of group g is
 *                 channel 16j + g + 8w.
 *   [2048, 2176)  K scales: [16 tokens][8 blocks] E4M3 (block b = channels
 *                 16b .. 16b + 15).
 *   [2176, 2304)  V scales: [8 rows p][8 blocks][2]; byte (p, b, w) is the scale
 *                 of token 2p + w, block b.
 * FP8 record, R = FP8KV_RECORD_BYTES = 4096 (E4M3 at scale 1.0):
 *   [0, 2048)     K: 16 rows of 128 bytes, row t = token t; the 16-byte chunk
 *                 at position (c + (t mod 2)) mod 8
 *                 holds channels 16c .. 16c + 15.
 *   [2048, 4096)  V: 8 rows of 256 bytes, row p = tokens 2p and 2p + 1; the
 *                 16-byte chunk at position (c + f(p)) mod 16, with
 *                 f(p) = (p mod 2) + 4 * (floor(p / 2) mod 2), holds channels
 *                 8c .. 8c + 7, byte 2i + w being channel 8c + i of token 2p + w.
 *
 * Supported geometry: head_dim 128, page_size 16, num_q_heads a multiple of
 * num_kv_heads with group g = num_q_heads / num_kv_heads in 1..8,
 * global_scale a positive normal finite fp32.  Anything else returns
 * NVFP4KV_ERR_UNSUPPORTED.
 *
 * Device-side checks: kernels that read page ids, slots or lengths from
 * device memory check them and, instead of faulting, OR a bit into the
 * optional caller-owned device word *dev_status (int32, may be NULL) and
 * treat the item as described per call.  Read it after synchronising.
 */
#ifndef NVFP4KV_H
#define NVFP4KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (the same object as cudaStream_t). */
typedef struct CUstream_st *nvfp4kv_stream_t;

typedef enum {
    NVFP4KV_OK = 0,
    NVFP4KV_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size ... */
    NVFP4KV_ERR_UNSUPPORTED = 2,  /* valid but outside the supported geometry   */
    NVFP4KV_ERR_WORKSPACE = 3,    /* decode workspace smaller than required     */
    NVFP4KV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed       */
    NVFP4KV_ERR_DEVICE_CHECK = 5  /* a kernel set bits in the device status word */
} nvfp4kv_status;

/* Bits ORed into *dev_status by the kernels. */
#define NVFP4KV_DEV_BAD_PAGE 0x1  /* block-table entry outside [0, num_pages)     */
#define NVFP4KV_DEV_BAD_SLOT 0x2  /* slot outside [0, num_pages * page_size)      */
#define NVFP4KV_DEV_BAD_LEN 0x4   /* length < 0 or > max_pages_per_seq*page_size  */
#define NVFP4KV_DEV_TIMEOUT 0x8   /* a bounded wait for staged data gave up        */

/* Element types of caller buffers.  NVFP4KV_E4M3 (OCP FP8 E4M3FN bytes at
 * scale 1.0) is accepted only where a call says so: the chunk K/V of the
 * extend calls. */
typedef enum { NVFP4KV_F32 = 0, NVFP4KV_BF16 = 1, NVFP4KV_E4M3 = 2 } nvfp4kv_dtype;

#define NVFP4KV_RECORD_BYTES 2304
#define FP8KV_RECORD_BYTES 4096

/* NVFP4 cache: pool of num_pages * num_kv_heads records laid out as above,
 * 16-byte aligned; global_scale is the tensor scale G described above.
 * head_scales (optional, may be NULL): a HOST array of 2 * num_kv_heads
 * per-head factors, K then V.  With it, kv head h of K uses the tensor scale
 * G_h = fl32(global_scale * head_scales[h]) and of V fl32(global_scale *
 * head_scales[num_kv_heads + h]) wherever G appears above (a refinement of the
 * pages' single tensor scale; this library's).  Each factor and each product
 * must be a positive normal finite float, and num_kv_heads at most
 * NVFP4KV_MAX_SCALED_KV_HEADS, else calls return NVFP4KV_ERR_UNSUPPORTED.  The
 * values are read on the host during each call. */
#define NVFP4KV_MAX_SCALED_KV_HEADS 128

typedef struct {
    void *pool;
    int32_t num_pages;
    int32_t num_kv_heads;
    int32_t page_size;
    int32_t head_dim;
    float global_scale;
    const float *head_scales;
} nvfp4kv_cache;

/* FP8-E4M3 comparison cache (scale 1.0): pool of records as above, 16-byte
 * aligned. */
typedef struct {
    void *pool;
    int32_t num_pages;
    int32_t num_kv_heads;
    int32_t page_size;
    int32_t head_dim;
} fp8kv_cache;

/* Write side ("SGLang stores KV cache in 4 bits", Interpretation ¶2: prefill
 * quantises the new K/V into the NVFP4 cache).
 * k_new, v_new: [num_tokens][num_kv_heads][head_dim] contiguous, fp32 or bf16
 *   (in_dtype), 16-byte aligned; read only.
 * slot_mapping: int32[num_tokens] device array; slot < 0 skips the token; a
 *   slot >= num_pages * page_size is skipped and sets NVFP4KV_DEV_BAD_SLOT.
 *   Slots must be distinct (two tokens writing one slot is a data race).
 * Writes the data and scale bytes of every (token, kv head) row of K and V.
 * Inputs must be finite (non-finite values give unspecified codes). */
nvfp4kv_status nvfp4kv_quantize_append(const nvfp4kv_cache *cache, const void *k_new,
                                       const void *v_new, nvfp4kv_dtype in_dtype,
                                       int32_t num_tokens, const int32_t *slot_mapping,
                                       int32_t *dev_status, nvfp4kv_stream_t stream);

/* Largest batch one decode call takes (the per-sequence page-head offsets are
 * kept in shared memory next to the staging ring); a larger batch returns
 * NVFP4KV_ERR_UNSUPPORTED. */
#define NVFP4KV_MAX_BATCH 8192

/* Bytes of decode workspace needed by nvfp4kv_paged_decode / fp8kv_paged_decode
 * when called with the same num_workers on the current device (num_workers 0 =
 * the automatic choice, whose need is bounded by this value).  Host only; the
 * result depends on the current device's SM count.  A library utility: the
 * pages describe no workspace (the split-KV scratch is this library's
 * design). */
size_t nvfp4kv_decode_workspace_size(int32_t num_workers);

/* Decode attention over the NVFP4 cache ("SGLang stores KV cache in 4 bits",
 * Interpretation ¶2: the decode path dequantises inside the attention kernel;
 * "NVFP4-KV-Cache auf der ...", "Geschwindigkeit": bf16 queries against
 * NVFP4 keys and values).
 * For sequence b and query head i (kv head h = i / g):
 *   o[b][i] = sum_j softmax_j(sm_scale * q[b][i] . k_j) v_j over the
 *   seq_lens[b] tokens j of sequence b, token j in page block_table[b][j/16]
 *   at offset j%16; no causal mask (the query sees all cached tokens).
 * q: bf16 [batch][num_q_heads][128], 16-byte aligned.  Computation: q is
 *   multiplied by sm_scale*log2(e)*G (G the tensor scale) and rounded to fp16
 *   (|q * sm_scale * G| must stay below 4.5e4); K and V are dequantised
 *   exactly to fp16 (block scale times code) and the output is multiplied by
 *   G; QK^T and PV run
 *   on tensor cores with fp32 accumulation; softmax in fp32.
 * block_table: int32 [batch][max_pages_per_seq]; only the first
 *   ceil(seq_lens[b]/16) entries of row b are read; an entry outside
 *   [0, num_pages) reads page 0 instead and sets NVFP4KV_DEV_BAD_PAGE.
 * seq_lens: int32[batch]; a length outside [0, max_pages_per_seq*16] is
 *   clamped into it and sets NVFP4KV_DEV_BAD_LEN.  Length 0 gives zeros.
 * out: [batch][num_q_heads][128] in out_dtype, 16-byte aligned.
 * workspace: device scratch of workspace_bytes >= the size above, 256-byte
 *   aligned; its contents need no initialisation and are overwritten.  Two
 *   calls in flight at once must not share a workspace.
 * num_workers: 0 = automatic; otherwise the number of warp workers the
 *   page-heads are balanced over (results agree up to rounding for any
 *   value).
 * Launches two kernels (split-KV attention, then the split merge), both with
 * programmatic dependent launch allowed, so each may start its prologue while
 * the previous kernel in the stream drains.  seq_lens and block_table are read
 * in that prologue: a kernel earlier in the stream that writes them must not
 * let its dependents start before it has written them (no kernel of this
 * library writes them). */
nvfp4kv_status nvfp4kv_paged_decode(const nvfp4kv_cache *cache, const void *q,
                                    int32_t batch, int32_t num_q_heads,
                                    const int32_t *block_table, int32_t max_pages_per_seq,
                                    const int32_t *seq_lens, float sm_scale, void *out,
                                    nvfp4kv_dtype out_dtype, void *workspace,
                                    size_t workspace_bytes, int32_t num_workers,
                                    int32_t *dev_status, nvfp4kv_stream_t stream);

/* One decode step: append each sequence's newest token, then attend
 * ("SGLang stores KV cache in 4 bits", Interpretation: new K/V are written to
 * the cache in NVFP4 and the decode path dequantises inside attention; doing
 * both in one launch is this library's fusion, not described on the pages).
 * For every sequence b with seq_lens[b] > 0, the K and V rows k_new[b],
 * v_new[b] ([batch][num_kv_heads][128], fp32 or bf16 per in_dtype, 16-byte
 * aligned) are quantised into the cache at position seq_lens[b] - 1 (page
 * block_table[b][(seq_lens[b]-1)/16], offset (seq_lens[b]-1)%16) exactly as
 * nvfp4kv_quantize_append would, and then the decode of nvfp4kv_paged_decode
 * runs over all seq_lens[b] tokens, including the new one.  The append is done
 * inside the decode kernel by the warp that streams that page, so the step is
 * two kernels instead of three.  The page that receives a sequence's new
 * token must not appear in another sequence's block table in the same call.
 * Other arguments and results as for nvfp4kv_paged_decode. */
nvfp4kv_status nvfp4kv_append_paged_decode(const nvfp4kv_cache *cache, const void *k_new, const void *v_new,
                                           nvfp4kv_dtype in_dtype, const void *q, int32_t batch,
                                           int32_t num_q_heads, const int32_t *block_table,
                                           int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                           void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                           size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                           nvfp4kv_stream_t stream);

/* Multi-query decode (several new tokens per sequence at once, as in
 * multi-token prediction or speculative decoding; "NVFP4-KV-Cache auf der
 * ...", "Unterstuetzung in den Engines": the engines' NVFP4 decode paths are
 * judged on speculative decoding with multi-token prediction): q_len query tokens per
 * sequence sit at the last q_len positions and attend causally, token t
 * (0-based) over the seq_lens[b] - q_len + t + 1 first cached tokens (the
 * new tokens must already be in the cache, e.g. by nvfp4kv_quantize_append).
 * Same arguments as nvfp4kv_paged_decode except
 * q: bf16 [batch][q_len][num_q_heads][128] and out: [batch][q_len][num_q_heads]
 *   [128]; 1 <= q_len <= NVFP4KV_MAX_QUERY_TOKENS (a larger value returns
 *   NVFP4KV_ERR_UNSUPPORTED).  A query that sees no cached token gets zeros.
 * The group * q_len query rows of a kv head are processed in row groups of
 * 8; each row group streams the kv head's pages (the row groups of one kv
 * head run close together, so the repeats mostly hit L2).  The workspace is
 * sized as for nvfp4kv_paged_decode. */
#define NVFP4KV_MAX_QUERY_TOKENS 8
nvfp4kv_status nvfp4kv_paged_decode_multi(const nvfp4kv_cache *cache, const void *q, int32_t batch,
                                          int32_t q_len, int32_t num_q_heads, const int32_t *block_table,
                                          int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                          void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                          size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                          nvfp4kv_stream_t stream);

/* Decode without a caller-provided workspace, for callers that cannot
 * allocate device memory (for example a serving engine whose device memory is
 * all reserved for weights and KV cache at start-up).  The pages have no
 * counterpart to this call; it exists for such callers.
 * Same arguments and result as nvfp4kv_paged_decode, minus the workspace: the
 * split-KV scratch comes from one array of NVFP4KV_STATIC_SCRATCH_BYTES that
 * the library keeps on every device that loads it, until the process exits.
 * num_workers may be at most NVFP4KV_STATIC_SCRATCH_MAX_WORKERS (a larger
 * value returns NVFP4KV_ERR_WORKSPACE); 0 picks the automatic count, capped at
 * that maximum.  The first call on a device looks the array up with that
 * device current, so make it before any stream capture.  All calls on a
 * device share the array: calls whose kernels can overlap on the GPU race and
 * must be serialised (for example, issue them on one stream).  Allocates no
 * memory. */
#define NVFP4KV_STATIC_SCRATCH_BYTES (24u << 20)
#define NVFP4KV_STATIC_SCRATCH_MAX_WORKERS 3024
nvfp4kv_status nvfp4kv_paged_decode_static_scratch(const nvfp4kv_cache *cache, const void *q, int32_t batch,
                                                   int32_t num_q_heads, const int32_t *block_table,
                                                   int32_t max_pages_per_seq, const int32_t *seq_lens,
                                                   float sm_scale, void *out, nvfp4kv_dtype out_dtype,
                                                   int32_t num_workers, int32_t *dev_status,
                                                   nvfp4kv_stream_t stream);

/* Extend path ("SGLang stores KV cache in 4 bits", Interpretation ¶2: the
 * cached prefix is dequantised into one FP8 workspace shared across layers).
 * For sequence b, token j < prefix_lens[b], kv head h, channel c:
 *   out[kv_indptr[b] + j][h][c] = E4M3_rn_satfinite(fl32(E2M1 x scale x G))
 * for K into k_fp8_out and V into v_fp8_out (each [rows][num_kv_heads][128]
 * uint8, 16-byte aligned; the caller sizes it to cover every row written).
 * kv_indptr: int32[batch] row offsets; prefix_lens: int32[batch].
 * Page-id and length checks as in nvfp4kv_paged_decode. */
nvfp4kv_status nvfp4kv_dequant_prefix_fp8(const nvfp4kv_cache *cache,
                                          const int32_t *block_table,
                                          int32_t max_pages_per_seq,
                                          const int32_t *prefix_lens,
                                          const int32_t *kv_indptr, int32_t batch,
                                          void *k_fp8_out, void *v_fp8_out,
                                          int32_t *dev_status, nvfp4kv_stream_t stream);

/* Extend attention over the FP8 prefix workspace and the current chunk
 * ("SGLang stores KV cache in 4 bits", Interpretation: the extend path
 * dequantises the cached prefix into one FP8 workspace and attends over it
 * together with the new chunk).  For sequence b with chunk rows
 * [q_indptr[b], q_indptr[b+1]) and prefix length P = prefix_lens[b], chunk
 * token t (row q_indptr[b] + t) and query head i (kv head h = i / g):
 *   keys   = k_prefix[kv_indptr[b] + j][h] for j < P, then k_chunk[q_indptr[b] + u][h] for u <= t
 *   values = the same rows of v_prefix / v_chunk
 *   out[q_indptr[b] + t][i] = softmax_j(sm_scale * q . key_j) . value_j
 * Prefix keys and values are E4M3 bytes (the workspace written by
 * nvfp4kv_dequant_prefix_fp8, with the same kv_indptr and prefix_lens); q is
 * bf16; chunk keys and values are bf16 or E4M3 (chunk_dtype).  E4M3 chunk K/V
 * are initial prefill as "SGLang stores KV cache in 4 bits", Interpretation
 * ¶2 describes it: attention reads the current prompt's FP8 keys and values
 * directly (prefix length 0 there; a prefix is allowed too).
 *   q        bf16 [q_rows][num_q_heads][128]
 *   k_chunk, v_chunk  [q_rows][num_kv_heads][128], chunk_dtype NVFP4KV_BF16
 *            (bf16) or NVFP4KV_E4M3 (uint8 E4M3 codes at scale 1.0); anything
 *            else returns NVFP4KV_ERR_INVALID_ARG
 *   out      [q_rows][num_q_heads][128], out_dtype bf16 or fp32; rows outside
 *            every [q_indptr[b], q_indptr[b+1]) are not written
 *   k_prefix, v_prefix  uint8 E4M3 [prefix_rows][num_kv_heads][128]
 *   q_indptr int32 [batch + 1] (device), kv_indptr and prefix_lens int32
 *            [batch] (device)
 *   max_q_len  host bound on every q_indptr[b+1] - q_indptr[b]; it sizes the
 *            launch
 * Arithmetic.  With E4M3 chunk K/V, or bf16 ones behind prefix_rows of at
 * least 8 * q_rows: q meets the keys as two E4M3 terms of its bf16 values,
 * each row multiplied by a power of two first (exact for every element but
 * those below 2^-10 of the row's largest, whose error stays under 2^-17 of
 * it), and sm_scale * log2(e) is applied to the fp32 scores; bf16 chunk keys
 * are split the same way per 64-key tile.  Otherwise q * sm_scale * log2(e)
 * and bf16 chunk keys are rounded to fp16 (exact for bf16 values of magnitude
 * 2^-14 .. 65504; the caller keeps |q * sm_scale| below 65504).  Values: E4M3
 * to fp16 is exact, bf16 chunk values are rounded to fp16 (kept below 65504
 * by the caller).  Scores and outputs accumulate in fp32, softmax weights are
 * rounded to fp16 for the value product.
 * Pointers 16-byte aligned (index arrays 4-byte).  Group g = num_q_heads /
 * num_kv_heads in 1..8; batch and num_kv_heads at most 65535.  Device check:
 * a sequence whose q_indptr range is not inside [0, q_rows] or longer than
 * max_q_len, or whose prefix rows are not inside [0, prefix_rows), sets
 * NVFP4KV_DEV_BAD_LEN and its output rows are not written.  A sequence with
 * an empty chunk writes nothing; with an empty prefix it is causal
 * attention over the chunk alone. */
nvfp4kv_status nvfp4kv_extend_attention_fp8(const void *q, const int32_t *q_indptr, int32_t q_rows,
                                            int32_t max_q_len, const void *k_prefix,
                                            const void *v_prefix, const int32_t *kv_indptr,
                                            const int32_t *prefix_lens, int64_t prefix_rows,
                                            const void *k_chunk, const void *v_chunk,
                                            nvfp4kv_dtype chunk_dtype, int32_t batch,
                                            int32_t num_q_heads, int32_t num_kv_heads, float sm_scale,
                                            void *out, nvfp4kv_dtype out_dtype, int32_t *dev_status,
                                            nvfp4kv_stream_t stream);

/* Extend attention fused with the NVFP4 write of the chunk ("SGLang stores KV
 * cache in 4 bits", Interpretation: prefill quantises the new K/V into the
 * cache; the fusion removes the separate read of the chunk).  Computes out
 * exactly as nvfp4kv_extend_attention_fp8 (num_kv_heads taken from the cache)
 * and writes chunk row r's K and V into slot slot_mapping[r] of the cache, as
 * nvfp4kv_quantize_append would given the chunk's values (bf16 as they are;
 * E4M3 codes as the fp32 values they stand for: the same data the attention
 * reads, as initial prefill does) -- same blocks, same bytes, same tensor
 * scale; slot < 0 skips the token, a slot >= num_pages * page_size is skipped
 * and sets NVFP4KV_DEV_BAD_SLOT.  slot_mapping: int32
 * [q_rows] (device, 4-byte aligned), read only for rows inside a sequence's
 * q_indptr range; slots must be distinct.  The prefix workspace must not
 * overlap the cache. */
nvfp4kv_status nvfp4kv_extend_attention_fp8_append(const nvfp4kv_cache *cache,
                                                   const int32_t *slot_mapping, const void *q,
                                                   const int32_t *q_indptr, int32_t q_rows,
                                                   int32_t max_q_len, const void *k_prefix,
                                                   const void *v_prefix, const int32_t *kv_indptr,
                                                   const int32_t *prefix_lens, int64_t prefix_rows,
                                                   const void *k_chunk, const void *v_chunk,
                                                   nvfp4kv_dtype chunk_dtype,
                                                   int32_t batch, int32_t num_q_heads, float sm_scale,
                                                   void *out, nvfp4kv_dtype out_dtype,
                                                   int32_t *dev_status, nvfp4kv_stream_t stream);

/* FP8-E4M3 comparison cache, written and read the same way ("NVFP4-KV-Cache
 * auf der ...", "Unterstuetzung in den Engines": the FP8 baseline runs with
 * --kv-cache-dtype fp8_e4m3; "Bytes pro Token": scales 1.0 uncalibrated).
 * Each value is E4M3_rn_satfinite(x).  Arguments as for the NVFP4 calls. */
nvfp4kv_status fp8kv_quantize_append(const fp8kv_cache *cache, const void *k_new,
                                     const void *v_new, nvfp4kv_dtype in_dtype,
                                     int32_t num_tokens, const int32_t *slot_mapping,
                                     int32_t *dev_status, nvfp4kv_stream_t stream);

nvfp4kv_status fp8kv_paged_decode(const fp8kv_cache *cache, const void *q, int32_t batch,
                                  int32_t num_q_heads, const int32_t *block_table,
                                  int32_t max_pages_per_seq, const int32_t *seq_lens,
                                  float sm_scale, void *out, nvfp4kv_dtype out_dtype,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t num_workers, int32_t *dev_status,
                                  nvfp4kv_stream_t stream);

/* The same fused step over the FP8 comparison cache (the FP8 baseline of
 * "NVFP4-KV-Cache auf der ...", "Unterstuetzung in den Engines", run through
 * the same append-then-decode step for a like-for-like comparison). */
nvfp4kv_status fp8kv_append_paged_decode(const fp8kv_cache *cache, const void *k_new, const void *v_new,
                                         nvfp4kv_dtype in_dtype, const void *q, int32_t batch,
                                         int32_t num_q_heads, const int32_t *block_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens, float sm_scale,
                                         void *out, nvfp4kv_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, int32_t num_workers, int32_t *dev_status,
                                         nvfp4kv_stream_t stream);

/* Bytes of an NVFP4 pool (K and V data and scales) for a geometry:
 * num_pages * num_kv_heads * page_size * 2 * (head_dim/2 + head_dim/16),
 * i.e. 9 bytes per 16 values ("SGLang stores KV cache in 4 bits",
 * Interpretation); for the supported geometry that is num_pages *
 * num_kv_heads * NVFP4KV_RECORD_BYTES.  Returns -1 for invalid arguments.
 * Host only. */
int64_t nvfp4kv_cache_bytes(int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                            int32_t head_dim);

/* Bytes of an FP8 pool: num_pages * num_kv_heads * page_size * 2 * head_dim,
 * one byte per value ("NVFP4-KV-Cache auf der ...", "Bytes pro Token: FP8
 * gegenueber NVFP4": 16 bytes per 16 values in FP8).  Returns -1 for invalid
 * arguments.  Host only. */
int64_t fp8kv_cache_bytes(int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                          int32_t head_dim);

/* A library utility with no counterpart on the pages: read a device status
 * word once the work on `stream` has finished:
 * synchronises the stream, copies *dev_status (device int32) into *bits
 * (host) and returns NVFP4KV_ERR_DEVICE_CHECK when any bit is set, NVFP4KV_OK
 * when none is (NVFP4KV_ERR_CUDA if the synchronisation or copy fails).  The
 * word is not reset.  Null pointers return NVFP4KV_ERR_INVALID_ARG. */
nvfp4kv_status nvfp4kv_read_device_status(const int32_t *dev_status, nvfp4kv_stream_t stream,
                                          int32_t *bits);

/* Failure detection (a library utility with no counterpart on the pages).
 * Every kernel wait for staged data, or for another part of the same CTA,
 * gives up after a number of polls, sets NVFP4KV_DEV_TIMEOUT in *dev_status,
 * lets whatever it already started (bulk copies, tensor-core operations)
 * finish and returns, so a wait that can never be satisfied costs a short
 * delay and a status bit, not a hung GPU.  This sets that number for the
 * calls made from now on in this process (0 = give up without polling;
 * NVFP4KV_WAIT_LIMIT_DEFAULT is the default) and returns the previous value.
 * The waits for work already in flight always use the default.  Host only,
 * thread-safe; a small limit makes ordinary calls report timeouts. */
#define NVFP4KV_WAIT_LIMIT_DEFAULT 4194304u
uint32_t nvfp4kv_set_wait_limit(uint32_t polls);

/* Static description of a status code (library utility). */
const char *nvfp4kv_status_string(nvfp4kv_status status);

/* Library version: major * 10000 + minor * 100 + patch (library utility). */
int32_t nvfp4kv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4KV_H */
