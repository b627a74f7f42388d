/*
 * fp4idx.h -- C ABI of libfp4idx.so, the fused FP4 indexer pre-pass of a
 * DeepSeek-style sparse-attention (DSA) indexer, as CUDA kernels for one
 * GB300 GPU (sm_103a).
 *
 * What it computes (sources are web pages, cited by title and section):
 *   (the pre-pass; the FP4 scorer that reads its bytes is declared last)
 *   "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656), Summary: keys
 *   get RMSNorm, RoPE, two quantisation stages to the per-32 UE8M0 E2M1 grid
 *   (round half to even) and a paged-cache store of the 68-byte index-K slot
 *   (64 e2m1 bytes + 4 block exponents); queries get the same RoPE and
 *   quantisation plus fp32 head weights in the same launch.
 *   "[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR
 *   5484), API: head_dim 128, rope_dim 64, group 32, kv_block 64; q_out is
 *   u8 [T, H, 64]; weights carry the plain weight, nothing folded in.
 *
 * Fixed geometry (anything else is not representable in these calls):
 *   head_dim 128, RoPE on dims 0..63, groups of 32 (4 per row), 64 slots per
 *   cache page.
 *
 * Numerics, per 128-element row (all fp32 steps round to nearest even, no
 * fused multiply-add, subnormals kept):
 *   RMSNorm (keys only): sum of squares in a fixed order (16 partial sums of
 *     8 consecutive squares, then pairwise at distances 8, 4, 2, 1),
 *     r = 1 / sqrt(sum/128 + eps) (correctly rounded sqrt, then correctly
 *     rounded reciprocal), y = bf16((x * r) * gamma).
 *   RoPE: pair i in 0..31 is (i, i+32) for NeoX or (2i, 2i+1) interleaved,
 *     a' = bf16(a*c - b*s), b' = bf16(b*c + a*s) with c, s = cos/sin[pos][i].
 *   Quantisation, per group of 32 (both stages): e = biased exponent of
 *     ceil_pow2(max(amax/6, 2^-126)); code = nearest of
 *     {0,.5,1,1.5,2,3,4,6} to |z| * 2^(127-e), ties to the even code; sign
 *     bit only on a non-zero code.  Stage 1 dequantises; stage 2 packs.
 *   Slot: payload byte 16g+j = nib[32g+2j] | nib[32g+2j+1] << 4; exponent
 *     word byte g = stage-2 exponent of group g.
 *   Weights: weights[t,h] = fp32(w[t,h]) * weight_scale (one rounding).
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers (cudaMalloc / torch CUDA memory)
 *     on the current device, except where fp4idx_indexer_prepass_host says
 *     HOST.  bf16 tensors are passed as const void*.
 *   - The caller owns every buffer.  The library allocates nothing, keeps no
 *     per-call state, never synchronises, and enqueues one kernel on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream);
 *     fp4idx_indexer_prepass_host enqueues one per chunk, on streams of its
 *     own that it orders after and before `stream`.
 *   - Host-side checks run before anything is enqueued; a failing check
 *     returns its status and enqueues nothing.  num_tokens == 0 returns
 *     FP4IDX_OK and enqueues nothing.
 *   - Device-side range checks: a position outside [0, max_pos) or a slot
 *     >= num_blocks*64 never causes an out-of-bounds access; the token is
 *     skipped (its outputs are left untouched) and, if err_flags is not
 *     NULL, the matching FP4IDX_ERRFLAG_* bit is OR-ed into *err_flags.
 *   - Inputs must keep every intermediate finite: |x| below ~1.8e19 for
 *     keys (the fp32 sum of squares), and every 32-element group of the
 *     rotated row with amax <= 6*2^125 (the stage-1 dequantised values);
 *     outputs for non-finite intermediates are unspecified.
 *   - Calls are asynchronous; errors of the kernel itself surface at the
 *     caller's next synchronisation.  FP4IDX_ERR_CUDA reports a failed
 *     launch (cudaGetLastError right after it).
 */
#ifndef FP4IDX_H
#define FP4IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp4idx_status {
  FP4IDX_OK = 0,
  FP4IDX_ERR_NULL = 1,  /* a required pointer is NULL (num_tokens > 0)      */
  FP4IDX_ERR_SHAPE = 2, /* num_tokens < 0, num_heads < 1, max_pos < 1,
                           num_blocks < 1, or a size product overflows      */
  FP4IDX_ERR_ALIGN = 3, /* a pointer or stride breaks its alignment rule    */
  FP4IDX_ERR_ARG = 4,   /* bad rope_style, eps not finite and > 0, a
                           non-finite weight_scale, or a bad option          */
  FP4IDX_ERR_CUDA = 5,  /* the kernel launch failed                          */
  FP4IDX_ERR_SCRATCH = 6 /* the request needs more than the library's static
                            scratch (fp4idx_indexer_prepass_host_static)     */
} fp4idx_status;

enum {
  FP4IDX_ROPE_NEOX = 0,        /* pairs (i, i+32)  */
  FP4IDX_ROPE_INTERLEAVED = 1  /* pairs (2i, 2i+1) */
};

enum {
  FP4IDX_HEAD_DIM = 128,
  FP4IDX_ROPE_DIM = 64,
  FP4IDX_GROUP = 32,
  FP4IDX_KV_BLOCK = 64,
  FP4IDX_SLOT_PAYLOAD_BYTES = 64,
  FP4IDX_SLOT_EXP_BYTES = 4,
  FP4IDX_PAGE_BYTES = 64 * 68, /* 4352 */
  FP4IDX_FP8_PAGE_BYTES = 64 * (128 + 4) /* 8448: FP8 output mode */
};

enum {
  FP4IDX_OUTPUT_FP4 = 0, /* packed E2M1 + per-32 UE8M0 exponents (default) */
  FP4IDX_OUTPUT_FP8 = 1  /* E4M3 codes + one power-of-two scale per row   */
};

/* Bits OR-ed into *err_flags by the device-side checks. */
#define FP4IDX_ERRFLAG_POSITION 0x1u /* a position outside [0, max_pos)     */
#define FP4IDX_ERRFLAG_SLOT 0x2u     /* a slot >= num_blocks * 64           */
#define FP4IDX_ERRFLAG_TIMEOUT 0x4u  /* an input copy did not arrive within
                                        1 s; that warp's remaining rows were
                                        left unwritten                       */
#define FP4IDX_ERRFLAG_PAGE 0x8u     /* scorer: a block-table entry outside
                                        [0, num_blocks) for a token below its
                                        context length; its logits are -inf */

/*
 * Keys: RMSNorm -> RoPE -> two-stage FP4 -> 68-byte slot -> paged cache.
 * Source: "dsv4.1: RoPE and FP4 packing kernels", Summary
 * (index_k_norm_rope_pack_store fuses RMSNorm, RoPE, both quantisation
 * stages and the paged cache store).
 *
 *   k            bf16, row t at k + t*k_token_stride elements, 128 elements
 *                each.  16-byte aligned; k_token_stride a multiple of 8.
 *   gamma        bf16 [128], 16-byte aligned.
 *   eps          RMSNorm epsilon, finite and > 0.
 *   positions    int64 [num_tokens]; the RoPE row of token t.
 *   cos_cache,   fp32 [max_pos, 32] each, dense, 16-byte aligned.
 *   sin_cache
 *   rope_style   FP4IDX_ROPE_NEOX or FP4IDX_ROPE_INTERLEAVED.
 *   slot_mapping int64 [num_tokens]; slot < 0 skips the token (nothing is
 *                written); otherwise page slot/64, offset o = slot%64.
 *                Slots must be distinct (duplicates: unspecified winner).
 *   kv_cache     bytes [num_blocks, 4352], 16-byte aligned, updated in
 *                place: the slot's 64-byte payload at page + o*64 and its
 *                4-byte exponent word at page + 4096 + o*4.  Every other
 *                byte is left untouched.
 *   err_flags    optional device uint32 (NULL: no reporting).
 *   stream       cudaStream_t.
 */
fp4idx_status fp4idx_k_norm_rope_pack_store(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, const int64_t* slot_mapping,
    uint8_t* kv_cache, int64_t num_blocks, int64_t num_tokens,
    uint32_t* err_flags, void* stream);

/*
 * Queries: RoPE -> two-stage FP4 -> pack, plus fp32 head weights, in one
 * launch.  Source: "dsv4.1: RoPE and FP4 packing kernels", Summary
 * (index_q_rope_pack_weights); "[HIP] Add FP4 output mode to
 * indexer_qk_rope_quant_and_cache", API (q_out u8 [T, H, 64]; weights carry
 * the plain weight).
 *
 *   q            bf16, row (t,h) at q + t*q_token_stride + h*q_head_stride
 *                elements, 128 elements each.  16-byte aligned; both strides
 *                multiples of 8.
 *   w            bf16, w[t,h] at w + t*w_token_stride + h elements.
 *   weight_scale finite fp32; the pages' value is H^-1/2 * D^-1/2 (D = 128).
 *   positions, cos_cache, sin_cache, max_pos, rope_style: as for keys.
 *   q_fp4        bytes [num_tokens, num_heads, 64], dense, 16-byte aligned.
 *   q_scale      bytes [num_tokens, num_heads, 4], dense, 4-byte aligned
 *                (one exponent word per row, group g in byte g).
 *   weights_out  fp32 [num_tokens, num_heads], dense, 4-byte aligned.
 *   err_flags    optional device uint32 (NULL: no reporting).
 *   stream       cudaStream_t.
 */
fp4idx_status fp4idx_q_rope_pack_weights(
    const void* q, int64_t q_token_stride, int64_t q_head_stride,
    const void* w, int64_t w_token_stride, float weight_scale,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, uint8_t* q_fp4, uint8_t* q_scale,
    float* weights_out, int64_t num_tokens, int64_t num_heads,
    uint32_t* err_flags, void* stream);

/*
 * Both halves of the pre-pass in ONE launch: exactly the two calls above
 * (same arguments, same results, same checks), with the key rows and the
 * query tokens scheduled over one grid so that the step pays one launch and
 * one tail.  Source: "dsv4.1: RoPE and FP4 packing kernels", Summary (the
 * key and query ops of the indexer pre-pass).  positions, cos_cache,
 * sin_cache, max_pos and rope_style are shared by both halves.
 */
fp4idx_status fp4idx_indexer_prepass(
    /* keys */
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_blocks,
    /* queries */
    const void* q, int64_t q_token_stride, int64_t q_head_stride,
    const void* w, int64_t w_token_stride, float weight_scale,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, int64_t num_heads,
    /* shared */
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, int64_t num_tokens, uint32_t* err_flags,
    void* stream);

/*
 * Stated variants of the same two operations, selected by an options block
 * (NULL = the defaults, identical to the calls above).
 *
 *   compress_ratio  1 (default), 2 or 4.  Compressed index keys take their
 *                   RoPE at the first position of their group of
 *                   compress_ratio consecutive positions: a key at position
 *                   p is rotated with table row p - p % compress_ratio.
 *                   Queries are never moved.  Source: "dsv4.1: RoPE and FP4
 *                   packing kernels" (sglang PR 39656), Summary (RoPE at the
 *                   group's first position) and Verification (compress
 *                   ratios 1, 2, 4).
 *   hadamard        0 (default) or 1.  After RoPE, every key and query row is
 *                   rotated by the normalised 128-point Walsh-Hadamard
 *                   transform (Sylvester order) before quantisation:
 *                   fast-transform butterflies h = 1, 2, ..., 64 in fp32,
 *                   each (a, b) -> (rn(a + b), rn(a - b)), then one product
 *                   with rn32(1/sqrt(128)) and a bf16 rounding.  Rotating
 *                   both sides keeps every query-key dot product.  Source:
 *                   "DeepSeek-V4 FP4: fused_compress FP4 scatter +
 *                   rmsnorm_rope_rotate FP4 KV-cache kernel" (aiter PR 4029),
 *                   Changes (RMSNorm + RoPE + optional Hadamard rotate + FP4
 *                   quant + paged KV-cache write).
 *   output_mode     FP4IDX_OUTPUT_FP4 (default) or FP4IDX_OUTPUT_FP8: the
 *                   FP8 contract that the FP4 mode extends ("[HIP] Add FP4
 *                   output mode to indexer_qk_rope_quant_and_cache" (aiter
 *                   PR 5484), Summary and API: the FP8 path folds its
 *                   per-(token, head) query scale into the head weights).
 *                   Every 128-element row gets one power-of-two scale
 *                   s = 2^(e-127) = ceil_pow2(max(rn32(amax/448), 2^-126))
 *                   and E4M3 (e4m3fn) codes of x / s (an exact division),
 *                   rounded half to even, saturating at 448, sign of zero
 *                   kept.  Then:
 *                     kv_cache is [num_blocks, 8448]: page b holds 64 code
 *                       rows of 128 bytes at o*128, then 64 fp32 scales s at
 *                       8192 + o*4 (page-split, like the FP4 pages);
 *                     q_fp4 receives the codes, [num_tokens, num_heads, 128]
 *                       bytes (16-byte aligned); q_scale is not written and
 *                       may be NULL;
 *                     weights_out[t,h] = rn(fp32(w[t,h]) * weight_scale) * s
 *                       (s folded in; the product by s is exact).
 * Any other value returns FP4IDX_ERR_ARG.  All other arguments, checks and
 * results are those of the corresponding call above.
 */
typedef struct fp4idx_options {
  int32_t compress_ratio;
  int32_t hadamard;
  int32_t output_mode;
} fp4idx_options;

fp4idx_status fp4idx_k_norm_rope_pack_store_ex(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, const int64_t* slot_mapping,
    uint8_t* kv_cache, int64_t num_blocks, int64_t num_tokens,
    const fp4idx_options* options, uint32_t* err_flags, void* stream);

fp4idx_status fp4idx_q_rope_pack_weights_ex(
    const void* q, int64_t q_token_stride, int64_t q_head_stride,
    const void* w, int64_t w_token_stride, float weight_scale,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, uint8_t* q_fp4, uint8_t* q_scale,
    float* weights_out, int64_t num_tokens, int64_t num_heads,
    const fp4idx_options* options, uint32_t* err_flags, void* stream);

fp4idx_status fp4idx_indexer_prepass_ex(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_blocks,
    const void* q, int64_t q_token_stride, int64_t q_head_stride,
    const void* w, int64_t w_token_stride, float weight_scale,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, int64_t num_heads,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, int64_t num_tokens,
    const fp4idx_options* options, uint32_t* err_flags, void* stream);

/*
 * fp4idx_indexer_prepass for inputs and query outputs in HOST memory.  The
 * operation is fp4idx_indexer_prepass (same source, same results, bytes
 * identical); the pages give no host-memory form of it, so this call only
 * adds the copies.  The tokens go through in chunks of chunk_tokens: the
 * upload of chunk c+1, the fused launch of chunk c and the download of chunk
 * c-1 overlap on three streams that the library creates once per device and
 * keeps.  Every copy is one cudaMemcpyAsync.
 *
 *   k, q, w      HOST bf16, dense: k [num_tokens, 128], q [num_tokens,
 *                num_heads, 128], w [num_tokens, num_heads].
 *   slot_mapping, positions   HOST int64 [num_tokens].
 *   q_fp4, q_scale, weights_out   HOST outputs, dense, as for
 *                fp4idx_q_rope_pack_weights.
 *                Host buffers should be page-locked (cudaHostAlloc or
 *                cudaHostRegister) for the copies to overlap; pageable
 *                memory works, without overlap.
 *   gamma, kv_cache, cos_cache, sin_cache, err_flags   DEVICE, as for
 *                fp4idx_indexer_prepass.
 *   staging      DEVICE scratch of fp4idx_host_staging_bytes(chunk_tokens,
 *                num_heads) bytes, 256-byte aligned, owned by the caller (the
 *                library allocates nothing).  Its contents are not kept.
 *   stream       the caller's stream: the pipeline starts after the work
 *                already queued on it, and the work queued on it after this
 *                call runs once every launch and download is done.  The host
 *                outputs are complete, and the host inputs may be reused,
 *                once the caller's stream has reached that point.
 *
 * Calls are serialised by a lock while they enqueue, and a call's first
 * chunks wait until the previous call on the same device no longer reads or
 * writes its staging buffer.  Checks: those of fp4idx_indexer_prepass (run before anything is
 * enqueued), chunk_tokens >= 1 and num_heads * chunk_tokens below 2^30
 * (FP4IDX_ERR_SHAPE), staging NULL (FP4IDX_ERR_NULL) or misaligned
 * (FP4IDX_ERR_ALIGN).  FP4IDX_ERR_CUDA: a stream, event or copy call failed;
 * what was enqueued before it stays enqueued.
 */
size_t fp4idx_host_staging_bytes(int64_t chunk_tokens, int64_t num_heads);

fp4idx_status fp4idx_indexer_prepass_host(
    const void* k, const int64_t* slot_mapping, const void* gamma, float eps,
    uint8_t* kv_cache, int64_t num_blocks, const void* q, const void* w,
    int64_t num_heads, float weight_scale, uint8_t* q_fp4, uint8_t* q_scale,
    float* weights_out, const int64_t* positions, const float* cos_cache,
    const float* sin_cache, int64_t max_pos, int rope_style, int64_t num_tokens,
    int64_t chunk_tokens, void* staging, uint32_t* err_flags, void* stream);

/*
 * fp4idx_indexer_prepass_host with the device staging in a static buffer of
 * the library instead of one the caller passes.  The pages have no
 * counterpart: this is a convenience form of the host-buffer call for
 * callers that own no device scratch.  It allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine): the staging is one file-scope
 * __device__ array of FP4IDX_STATIC_STAGING_BYTES per device, whose address
 * is looked up once per device (cudaGetSymbolAddress).  The array occupies
 * device memory from the time the library's module is loaded on a device:
 * with the CUDA runtime's lazy module loading (its default), the first call
 * of this function there; with eager loading, context creation.
 *
 * Arguments, results and checks are those of fp4idx_indexer_prepass_host
 * without `staging`.  A request whose staging
 * (fp4idx_host_staging_bytes(chunk_tokens, num_heads)) exceeds the static
 * buffer returns FP4IDX_ERR_SCRATCH before anything is enqueued: choose
 * chunk_tokens with chunk_tokens * (660 * num_heads + 544) + 4096 <=
 * FP4IDX_STATIC_STAGING_BYTES (e.g. 1,536 tokens at 64 heads).  A failed
 * symbol lookup returns FP4IDX_ERR_CUDA.  Nothing in the buffer needs to
 * start at zero: every chunk's inputs are uploaded before its launch reads
 * them, and its outputs written before they are downloaded.
 *
 * Overlapping calls would race on the one buffer.  The library orders them
 * instead: calls enqueue under a lock, and each call's first uploads wait
 * until the previous call on the device no longer reads or writes the
 * staging, so concurrent callers run one after the other on the GPU.
 */
enum { FP4IDX_STATIC_STAGING_BYTES = 64 << 20 };

fp4idx_status fp4idx_indexer_prepass_host_static(
    const void* k, const int64_t* slot_mapping, const void* gamma, float eps,
    uint8_t* kv_cache, int64_t num_blocks, const void* q, const void* w,
    int64_t num_heads, float weight_scale, uint8_t* q_fp4, uint8_t* q_scale,
    float* weights_out, const int64_t* positions, const float* cos_cache,
    const float* sin_cache, int64_t max_pos, int rope_style, int64_t num_tokens,
    int64_t chunk_tokens, uint32_t* err_flags, void* stream);

/*
 * Torch-shaped fake quantisation: RoPE, then every value replaced by its
 * dequantised FP4 value, written as bf16.  Source: "dsv4.1: RoPE and FP4
 * packing kernels" (sglang PR 39656), Summary (the RoPE tail plus FP4
 * fake-quant of the torch-shaped path, per-32 UE8M0 by default and per-16
 * E4M3 for compressed KV, keeping the bf16 round trip after RoPE and round
 * half to even).
 *
 *   x            bf16 rows, row r at x + r*row_stride elements (16-byte
 *                aligned, row_stride a multiple of 8 and >= 128).
 *   rows_per_token  row r takes positions[r / rows_per_token] (1 for keys
 *                [T,128], H for queries [T,H,128]).
 *   positions, cos_cache, sin_cache, max_pos, rope_style: as above; RoPE
 *                on dims 0..63 with the bf16 round trip.
 *   scale_mode   FP4IDX_FAKE_QUANT_UE8M0_32: groups of 32 with the
 *                pre-pass's stage-1 scale (the values its stage 1 produces);
 *                FP4IDX_FAKE_QUANT_E4M3_16: groups of 16 with the scale
 *                s = E4M3(rn32(amax/6)) (round half to even, saturating at
 *                448), codes the nearest E2M1 of rn32(x/s) (ties to even,
 *                saturating at 6), values code*s; a group whose s rounds to
 *                0 becomes zeros.  No output is -0.  Rows holding an inf
 *                or NaN give unspecified values.
 *   out          bf16 [num_rows, 128], dense, 16-byte aligned.
 *   err_flags    FP4IDX_ERRFLAG_POSITION for a row whose position is out of
 *                range (that row is left untouched).
 */
enum {
  FP4IDX_FAKE_QUANT_UE8M0_32 = 0,
  FP4IDX_FAKE_QUANT_E4M3_16 = 1
};

fp4idx_status fp4idx_rope_fake_quant(
    const void* x, int64_t row_stride, int64_t rows_per_token,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, int scale_mode, void* out,
    int64_t num_rows, uint32_t* err_flags, void* stream);

/*
 * FP4 paged MQA-logits scorer: the consumer of the bytes written above.
 * Sources: "[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache"
 * (aiter PR 5484), Verification (the paged FP4 MQA-logits scorer reads the
 * packed keys and their e8m0 exponents from the paged cache; GLM-5.2 shapes
 * H = 32, kv_block 64, next_n 1 and 4); "[ROCm][Perf] Enabled FP4Indexer for
 * DSV4" (vLLM PR 42908), Code Review (block-scaled E2M1 dot products of
 * packed queries and keys, ReLU, head weights, sum over heads).
 *
 * Query row t = b*next_n + j (sequence b, its j-th query token) scores every
 * cached token s of sequence b:
 *   logits[t, s] = sum_h weights[t,h] * max(0, sum_d q[t,h,d] * k_s[d])
 *     for s < min(context_lens[b], max_context),
 *   logits[t, s] = -inf for context_lens[b] <= s < max_context,
 * with q and k the FP4 values (E2M1 grid value * 2^(e-127), e the row's
 * exponent byte for the group d/32) and k_s the slot of token s: page
 * block_table[b, s/64], offset s%64, in the layout fp4idx_k_norm_rope_pack_store
 * writes.  The products are exact; sums are fp32 (tensor-core accumulation
 * over d, then the weighted head sum in fixed-order packed chains), so a
 * logit is within 2^-17 * sum_h |weights[t,h]| * sum_d |q[t,h,d] k_s[d]| of
 * the exact value (a bound from the fp32 roundings of the tensor core's sum
 * of 128 products and of the head sum, whose chains are at most 15
 * additions deep; the tests hold every logit to it).
 *
 *   q_fp4        bytes [batch*next_n, num_heads, 64], dense, 16-byte aligned
 *                (the q_fp4 output of the calls above).
 *   q_scale      bytes [batch*next_n, num_heads, 4], dense, 16-byte aligned.
 *   weights      fp32 [batch*next_n, num_heads], dense.
 *   kv_cache     bytes [num_blocks, 4352], 16-byte aligned, read only.
 *                Exponent bytes must be <= 254 (255 is NaN on the tensor
 *                core); the pre-pass writes 1..252.
 *   block_table  int32, entry (b, p) at b*block_table_stride + p; read for
 *                p < ceil(min(context_lens[b], max_context) / 64) only.
 *                block_table_stride >= ceil(max_context / 64).
 *   context_lens int32 [batch]; values < 0 count as 0.
 *   logits       fp32, row t at logits + t*logits_stride, columns
 *                [0, max_context) written, the rest untouched;
 *                logits_stride >= max_context.
 *   batch >= 0, next_n >= 1, num_heads one of 32, 64, 96, 128 (a sequence
 *   whose next_n * num_heads query rows exceed 128 is scored in groups of
 *   128 / num_heads tokens, each group reading the sequence's keys once),
 *   0 <= max_context < 2^30, batch * next_n * num_heads < 2^31.
 *   err_flags    optional device uint32: FP4IDX_ERRFLAG_PAGE for a bad
 *                block-table entry (those logits are -inf, nothing is read),
 *                FP4IDX_ERRFLAG_TIMEOUT if a copy or the tensor core did not
 *                finish within 1 s (that CTA's remaining logits unwritten).
 * batch == 0 or max_context == 0 returns FP4IDX_OK and enqueues nothing.
 */
fp4idx_status fp4idx_paged_mqa_logits(
    const uint8_t* q_fp4, const uint8_t* q_scale, const float* weights,
    const uint8_t* kv_cache, int64_t num_blocks, const int32_t* block_table,
    int64_t block_table_stride, const int32_t* context_lens, float* logits,
    int64_t logits_stride, int64_t batch, int64_t next_n, int64_t num_heads,
    int64_t max_context, uint32_t* err_flags, void* stream);

/*
 * The prefill variant of the scorer: query tokens of a prefill chunk against
 * the chunk's keys, each token over its own key range.  Source: "[HIP] Add
 * FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR 5484),
 * Summary (the FP4 paged scorer "and its prefill variant" read the packed
 * keys straight out of the cache).  The page prints no signature; reading
 * taken: the keys are consecutive -- key s is the slot at page s/64, offset
 * s%64 of kv_cache, which is what fp4idx_k_norm_rope_pack_store writes with
 * slot_mapping[s] = s -- so there is no block table, and query token t
 * scores the keys in [ks[t], ke[t]):
 *   logits[t, s] = sum_h weights[t,h] * max(0, sum_d q[t,h,d] * k_s[d])
 *     for max(ks[t], 0) <= s < min(ke[t], num_keys),
 *   logits[t, s] = -inf for every other s < num_keys
 * (an empty range gives a row of -inf), with the decode scorer's arithmetic
 * and error bound.
 *
 *   q_fp4, q_scale, weights  as above, [num_tokens, num_heads, ...].
 *   kv_cache     bytes [num_blocks, 4352], 16-byte aligned, read only;
 *                num_keys <= num_blocks * 64.  Exponent bytes <= 254.
 *   ks, ke       int32 [num_tokens].
 *   logits       fp32, row t at logits + t*logits_stride, columns
 *                [0, num_keys) written, the rest untouched;
 *                logits_stride >= num_keys.
 *   num_heads one of 32, 64, 96, 128; 0 <= num_keys < 2^30;
 *   num_tokens * num_heads < 2^31.
 *   err_flags    optional: FP4IDX_ERRFLAG_TIMEOUT as above.
 * num_tokens == 0 or num_keys == 0 returns FP4IDX_OK and enqueues nothing.
 */
fp4idx_status fp4idx_mqa_logits_prefill(
    const uint8_t* q_fp4, const uint8_t* q_scale, const float* weights,
    const uint8_t* kv_cache, int64_t num_blocks, int64_t num_keys,
    const int32_t* ks, const int32_t* ke, float* logits, int64_t logits_stride,
    int64_t num_tokens, int64_t num_heads, uint32_t* err_flags, void* stream);

/*
 * The head-weight scale the pages use: H^-1/2 * D^-1/2 with D = 128,
 * evaluated in double and rounded once to fp32 (0 when num_heads < 1).  Pass
 * it as weight_scale to the query calls above.  Sources: "[HIP] Add FP4
 * output mode to indexer_qk_rope_quant_and_cache" (aiter PR 5484), API (the
 * head weights carry the plain weight; the scorer applies its own scalar);
 * "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656), Summary (the
 * indexer head weights of the query op).
 */
float fp4idx_default_weight_scale(int64_t num_heads);

/*
 * Testing hook for the bounded waits (no counterpart in the pages: it exists
 * so that the timeout path can be exercised without faulting the GPU).  The
 * next launch of the given kernel, on any thread, leaves out the copies of
 * one work item of its first CTA: a 64-row unit of the streaming pre-pass
 * kernel (FP4IDX_TEST_PREPASS; units count key units first, then query
 * units; head counts that are a multiple of 16), or a 128-key tile of the
 * scorers (FP4IDX_TEST_SCORER; tiles count in that CTA's order, and a tile's
 * partner in its stage pair is left out with it).  The waits for it then
 * run out after their 1 s limit: that launch raises FP4IDX_ERRFLAG_TIMEOUT,
 * leaves part of its outputs unwritten, drains its copies in flight and
 * returns; later launches are unaffected.  The hook is taken by that one
 * launch (an index past the CTA's work withholds nothing).  Returns
 * FP4IDX_ERR_ARG for an unknown kernel or a negative index.
 */
enum { FP4IDX_TEST_PREPASS = 0, FP4IDX_TEST_SCORER = 1 };
fp4idx_status fp4idx_test_withhold_next(int kernel, int64_t index);

/* Static, NUL-terminated description of a status code. */
const char* fp4idx_status_string(fp4idx_status status);

/* Static version string of the library ("fp4idx <semver> sm_103a"). */
const char* fp4idx_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP4IDX_H */
