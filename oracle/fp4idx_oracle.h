/*
 * fp4idx_oracle.h -- plain scalar CPU oracle for the fused FP4 indexer
 * pre-pass.  TEST INFRASTRUCTURE ONLY: nothing on the product path may link,
 * load or call this library.  Only the test suite, the smoke check and the
 * bench's CPU-baseline / reference legs use it.
 *
 * It shares no code, header, table or constant with the CUDA library.  Every
 * buffer is a HOST pointer to a dense, row-major array.  bf16 values are
 * passed as their 16-bit patterns (uint16_t).
 *
 * Sources (web pages on FP4 DSA-indexer keys and queries):
 *   [sgl]  "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656):
 *          Summary; Verification; review comment on clear_negative_zero,
 *          index_pack_exponent and inv_scale_ue8m0.
 *   [aiter] "[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache"
 *          (aiter PR 5484): API; Verification; One deliberate deviation.
 *   [csa]  "DeepSeek-V4 FP4: fused_compress FP4 scatter + rmsnorm_rope_rotate
 *          FP4 KV-cache kernel" (aiter PR 4029): Changes (optional Hadamard
 *          rotation before the FP4 quantisation).
 *
 * Where the pages leave a step open, the reading used is stated beside the
 * function that takes it.
 *
 * Parity unpinned: two readings have no page fact to pin them, so the tests
 * fix the oracle's behaviour under them but cannot confirm them: the
 * summation order of the sum of squares in oracle_rmsnorm_row, and the
 * placement of a slot's 68 bytes in a 4352-byte cache page (64 payload
 * bytes at 64 o, the exponent word at 4096 + 4 o) in the cache store.
 */
#ifndef FP4IDX_ORACLE_H
#define FP4IDX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* RoPE pairing styles. */
#define ORACLE_ROPE_NEOX 0        /* pairs (i, i+32), i in 0..31 */
#define ORACLE_ROPE_INTERLEAVED 1 /* pairs (2i, 2i+1), i in 0..31 */

/* ---- single steps, exported so the tests can pin each one ---- */

/* fp32 -> bf16 bit pattern, round to nearest, ties to even (finite input). */
uint16_t oracle_f32_to_bf16(float x);

/* RMSNorm of one 128-element key row, bf16 in / bf16 out. */
void oracle_rmsnorm_row(const uint16_t* x, const uint16_t* gamma, float eps,
                        uint16_t* y);

/* In-place RoPE of the first 64 dims of a 128-element bf16 row. */
void oracle_rope_row(uint16_t* y, const float* cos_row, const float* sin_row,
                     int rope_style);

/* Quantise one 32-element group z (fp32 values) with scale floor `floor_`.
 * Writes 32 nibbles (bit 3 sign, bits 2..0 E2M1 code) and returns the
 * biased UE8M0 exponent. */
int oracle_quant_group(const float* z, float floor_, uint8_t* nibbles);

/* The same with a floor on the amax (before the division by 6) and one on
 * the quotient (after it); 0 means no floor.  Stage 1 of the pre-pass uses
 * the amax floor, stage 2 the quotient floor. */
int oracle_quant_group_floors(const float* z, float amax_floor, float quot_floor,
                              uint8_t* nibbles);

/* Dequantise a nibble with biased exponent e (exact in fp32). */
float oracle_dequant(uint8_t nibble, int e);

/* Both quantisation stages + pack for one 128-element bf16 row:
 * 64 payload bytes and 4 exponent bytes (group g -> byte g).
 * If stage1_e / stage2_e are non-NULL they receive the 4 exponents of each
 * stage; stage1_codes (128 nibbles) likewise, for invariant tests. */
void oracle_quant_pack_row(const uint16_t* row, uint8_t* payload64,
                           uint8_t* exp4, int* stage1_e, int* stage2_e,
                           uint8_t* stage1_nibbles);

/* The pack with explicit floors: stage-1 amax and quotient floors, stage-2
 * amax and quotient floors (the pre-pass: 2^-126, 0, 0, 2^-126). */
void oracle_quant_pack_row_floors(const uint16_t* row, float s1_amax, float s1_quot,
                                  float s2_amax, float s2_quot, uint8_t* payload64,
                                  uint8_t* exp4, int* stage1_e, int* stage2_e,
                                  uint8_t* stage1_nibbles);

/* ---- the two operations of the pre-pass ---- */

/* Keys: RMSNorm -> RoPE -> two-stage FP4 -> 68-byte slot -> paged cache.
 *   k          [T,128] bf16      gamma [128] bf16
 *   positions  [T] int64         cos_cache, sin_cache [max_pos,32] fp32
 *   slot_mapping [T] int64 (<0: skip the token)
 *   kv_cache   [num_blocks, 4352] bytes: page b holds 64 payloads of 64 B
 *              at b*4352 + o*64, then 64 exponent words at b*4352+4096+o*4.
 * Returns 0, or -1 if a position or slot is out of range (that row is
 * skipped, the others are still written). */
int oracle_k_norm_rope_pack_store(const uint16_t* k, const uint16_t* gamma,
                                  float eps, const int64_t* positions,
                                  const float* cos_cache,
                                  const float* sin_cache, int64_t max_pos,
                                  int rope_style, const int64_t* slot_mapping,
                                  uint8_t* kv_cache, int64_t num_blocks,
                                  int64_t num_tokens);

/* Queries: RoPE -> two-stage FP4 -> pack, plus fp32 head weights.
 *   q [T,H,128] bf16, w [T,H] bf16
 *   q_fp4 [T,H,64] bytes, q_scale [T,H,4] bytes, weights [T,H] fp32
 *   weights[t,h] = w[t,h] * H^-1/2 * D^-1/2 (D = 128), rounded once.
 * Returns 0, or -1 if a position is out of range (that token's outputs are
 * left untouched). */
int oracle_q_rope_pack_weights(const uint16_t* q, const uint16_t* w,
                               const int64_t* positions,
                               const float* cos_cache, const float* sin_cache,
                               int64_t max_pos, int rope_style,
                               uint8_t* q_fp4, uint8_t* q_scale,
                               float* weights, int64_t num_tokens,
                               int64_t num_heads);

/* ---- stated variants of the same two operations ---- */

/* In-place normalised 128-point Walsh-Hadamard rotation of a bf16 row:
 * fast-transform butterflies h = 1..64 in fp32, times rn32(1/sqrt(128)),
 * rounded to bf16. */
void oracle_hadamard_row(uint16_t* y);

/* Keys with the variants: compress_ratio (1, 2 or 4) moves the RoPE to the
 * group's first position, pos - pos % ratio; hadamard != 0 rotates the row
 * after RoPE.  compress_ratio 1 and hadamard 0 is the call above. */
int oracle_k_norm_rope_pack_store_ex(const uint16_t* k, const uint16_t* gamma,
                                     float eps, const int64_t* positions,
                                     const float* cos_cache,
                                     const float* sin_cache, int64_t max_pos,
                                     int rope_style, const int64_t* slot_mapping,
                                     uint8_t* kv_cache, int64_t num_blocks,
                                     int64_t num_tokens, int compress_ratio,
                                     int hadamard);

/* Queries with the rotation variant (hadamard != 0: after RoPE). */
int oracle_q_rope_pack_weights_ex(const uint16_t* q, const uint16_t* w,
                                  const int64_t* positions,
                                  const float* cos_cache, const float* sin_cache,
                                  int64_t max_pos, int rope_style,
                                  uint8_t* q_fp4, uint8_t* q_scale,
                                  float* weights, int64_t num_tokens,
                                  int64_t num_heads, int hadamard);

/* ---- FP8 output mode (E4M3 codes, one power-of-two scale per row) ---- */

float oracle_e4m3_to_f32(uint8_t c);
/* Nearest E4M3, ties to even mantissa, |v| > 448 saturates, sign kept. */
uint8_t oracle_f32_to_e4m3(float v);
/* 128 codes of one bf16 row; returns the biased exponent e of the row's
 * scale 2^(e-127) = ceil_pow2(max(amax/448, 2^-126)). */
int oracle_fp8_quant_row(const uint16_t* row, uint8_t* codes);
/* Keys -> FP8 paged cache [num_blocks, 8448]: page b holds 64 code rows of
 * 128 bytes at o*128, then 64 fp32 scales at 8192 + o*4. */
int oracle_k_norm_rope_fp8_store(const uint16_t* k, const uint16_t* gamma,
                                 float eps, const int64_t* positions,
                                 const float* cos_cache, const float* sin_cache,
                                 int64_t max_pos, int rope_style,
                                 const int64_t* slot_mapping, uint8_t* kv_cache,
                                 int64_t num_blocks, int64_t num_tokens,
                                 int compress_ratio, int hadamard);
/* Queries -> q_out [T,H,128] E4M3 codes and weights [T,H] fp32 with the
 * row's scale folded in: w * H^-1/2 * D^-1/2 * 2^(e-127), rounded once. */
int oracle_q_rope_fp8_weights(const uint16_t* q, const uint16_t* w,
                              const int64_t* positions, const float* cos_cache,
                              const float* sin_cache, int64_t max_pos,
                              int rope_style, uint8_t* q_out, float* weights,
                              int64_t num_tokens, int64_t num_heads,
                              int hadamard);

/* ---- Torch-shaped fake quantisation (bf16 in, dequantised bf16 out) ---- */

/* One 128-element bf16 row: mode 0 = per-32 UE8M0 (stage 1 of the pack),
 * mode 1 = per-16 groups with E4M3 scales E4M3(amax/6). */
void oracle_fake_quant_row(const uint16_t* row, int mode, uint16_t* out);
/* RoPE (as in the pre-pass) then fake quantisation of rows x [num_rows,128];
 * row r takes positions[r / rows_per_token].  Returns 0, or -1 if a position
 * is out of range (that row's output is left untouched). */
int oracle_rope_fake_quant(const uint16_t* x, int64_t rows_per_token,
                           const int64_t* positions, const float* cos_cache,
                           const float* sin_cache, int64_t max_pos,
                           int rope_style, int mode, uint16_t* out,
                           int64_t num_rows);

/* FP4 paged MQA-logits scorer (the consumer of the packed queries and the
 * paged index-K cache).  Query row t = b*next_n + j of sequence b scores
 * every cached token s < context_lens[b]:
 *   logits[t, s] = sum_h weights[t,h] * max(0, sum_d q[t,h,d] * k_s[d])
 * with q, k the dequantised FP4 values (grid value * 2^(e-127)) and k_s the
 * slot at page block_table[b, s/64], offset s%64 (page-split layout).
 * Positions context_lens[b] <= s < max_context get -inf.  Sums in double,
 * rounded to fp32 once.  Returns 0, or -1 if a page index is out of range
 * (those logits are -inf). */
int oracle_paged_mqa_logits(const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* weights, const uint8_t* kv_cache,
                            int64_t num_blocks, const int32_t* block_table,
                            int64_t block_table_stride,
                            const int32_t* context_lens, float* logits,
                            int64_t logits_stride, int64_t batch,
                            int64_t next_n, int64_t num_heads,
                            int64_t max_context);

/* Prefill scorer: query token t (rows t*H .. t*H+H-1 of q_fp4/q_scale,
 * weights[t, :]) against the consecutive keys s = 0 .. num_keys-1 (page
 * s/64, offset s%64 of kv_cache [>= ceil(num_keys/64), 4352]):
 * logits[t*logits_stride + s] = sum_h w * max(0, q . k_s) for
 * ks[t] <= s < ke[t], -inf for the other s < num_keys.  Returns 0. */
int oracle_mqa_logits_prefill(const uint8_t* q_fp4, const uint8_t* q_scale,
                              const float* weights, const uint8_t* kv_cache,
                              int64_t num_keys, const int32_t* ks, const int32_t* ke,
                              float* logits, int64_t logits_stride, int64_t num_tokens,
                              int64_t num_heads);

/* Host threads used by the token / row loops (default 1), and the number
 * the machine offers (1 when built without OpenMP). */
void oracle_set_threads(int n);
int oracle_get_threads(void);
int oracle_threads_available(void);

#ifdef __cplusplus
}
#endif
#endif /* FP4IDX_ORACLE_H */
