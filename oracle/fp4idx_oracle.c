/*
 * fp4idx_oracle.c -- plain, slow, scalar CPU oracle for the fused FP4
 * indexer pre-pass.  TEST INFRASTRUCTURE ONLY (see fp4idx_oracle.h).
 *
 * Build with no floating-point contraction and no fast-math so that every
 * fp32 operation below is one IEEE round-to-nearest-even step:
 *     gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (fp32 expressions are evaluated in fp32 on x86-64 SSE and on aarch64.)
 *
 * Notation used in the comments: rn32(.) is one fp32 rounding, bf16(.) one
 * fp32 -> bf16 rounding, both to nearest with ties to even.
 */
#include "fp4idx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Tokens (and scorer rows) are independent, so the top-level loops may run
 * on several host threads; the arithmetic of each row is the same scalar
 * code whatever the thread count.  Default: one thread. */
static int g_threads = 1;

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

int oracle_get_threads(void) { return g_threads; }

int oracle_threads_available(void) {
#ifdef _OPENMP
  return omp_get_num_procs();
#else
  return 1;
#endif
}

enum {
  HEAD_DIM = 128,     /* [aiter] API: head_dim = 128 */
  ROPE_DIM = 64,      /* [aiter] API: rope_dim = 64, dims 0..63 */
  GROUP = 32,         /* [aiter] API: group_size = 32 (per-32 UE8M0 scales) */
  KV_BLOCK = 64,      /* [aiter] API: kv_block_size = 64 */
  PAYLOAD_BYTES = 64, /* [sgl] Summary: 64 e2m1 bytes ... */
  EXP_BYTES = 4,      /* ... plus four block exponents = 68-byte slot */
  PAGE_BYTES = KV_BLOCK * (PAYLOAD_BYTES + EXP_BYTES) /* 4352 */
};

/* The E2M1 grid: magnitude code m in 0..7 encodes GRID[m]. */
static const double GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Scale floors of the two quantisation stages.
 *   Stage 1 is the fake quantisation (fake_quant_fp4 / fp4::block_scale).
 *     Its floor guards the amax of an all-zero group BEFORE the division by
 *     6 ([csa] review: the FP4 quantiser's amax has an all-zero-group eps
 *     floor).
 *   Stage 2 is the indexer packer.  It divides first and floors the
 *     quotient ([sgl] review: index_pack_exponent keeps amax / 6.0f and a
 *     post-divide floor rather than reusing fp4::block_scale).
 * So the two scale floors differ, as the [sgl] review states (the packer
 * "has a different scale floor from fake_quant_fp4"): one acts on the amax,
 * the other on amax/6.  Neither value is printed.  Reading taken: both
 * constants are 2^-126, the smallest normal fp32 -- the smallest floor that
 * does the one job the pages give it (an all-zero group).
 * Which bytes hang on this reading: none, for any amax floor in
 * (0, 6 * 2^-126] and any quotient floor in (0, 2^-126].  Every quotient at
 * or below 2^-126 already has biased exponent 1 after the ceiling (and 1 is
 * the clamp's lower bound), so every such floor pair gives every group the
 * same exponent.  A larger floor F would change exactly the groups whose
 * stage amax is below 6 * F. */
static const float STAGE1_AMAX_FLOOR = 1.17549435082228750797e-38f; /* 2^-126 */
static const float STAGE2_QUOT_FLOOR = 1.17549435082228750797e-38f; /* 2^-126 */
/* The FP8 row scale's floor (reading F2: ceil_pow2(max(amax/448, 2^-126))). */
static const float FP8_QUOT_FLOOR = 1.17549435082228750797e-38f; /* 2^-126 */

static uint32_t f2u(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}
static float u2f(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static float bf16_to_f32(uint16_t b) { return u2f((uint32_t)b << 16); }

/* fp32 -> bf16, round to nearest, ties to even, written from the definition:
 * take the two bf16 neighbours of |x| (truncation, and one bf16 ulp above
 * it), keep the nearer one, and on a tie the one whose last bit is 0.  The
 * distances are exact in double.  Finite inputs only. */
uint16_t oracle_f32_to_bf16(float x) {
  uint32_t u = f2u(x);
  uint32_t sign = u & 0x80000000u;
  uint32_t mag = u & 0x7fffffffu;
  uint32_t lo = mag & 0xffff0000u;   /* bf16 neighbour toward zero */
  uint32_t hi = lo + 0x00010000u;    /* next bf16 magnitude up     */
  double m = (double)u2f(mag);
  double d_lo = m - (double)u2f(lo);
  double d_hi = (double)u2f(hi) - m;
  uint32_t pick;
  if (d_lo < d_hi)
    pick = lo;
  else if (d_hi < d_lo)
    pick = hi;
  else
    pick = ((lo >> 16) & 1u) ? hi : lo; /* tie: even last bit */
  return (uint16_t)((sign | pick) >> 16);
}

/* RMSNorm of an index-key row ([sgl] Summary: the key kernel fuses RMSNorm
 * ahead of RoPE), y = bf16(rn32(rn32(x * r) * gamma)).
 * Readings (pages silent): fp32 arithmetic, x*r before *gamma, one bf16
 * rounding at the end (the bf16 round trip after RMSNorm); r is a correctly
 * rounded sqrt followed by a correctly rounded reciprocal.  The sum of squares
 * uses one fixed order: 16 partial sums of 8 consecutive squares, accumulated
 * left to right, then combined pairwise at distances 8, 4, 2, 1 (partial c
 * plus partial c^d), the total being partial 0. */
void oracle_rmsnorm_row(const uint16_t* xb, const uint16_t* gamma, float eps,
                        uint16_t* y) {
  float x[HEAD_DIM];
  for (int i = 0; i < HEAD_DIM; ++i) x[i] = bf16_to_f32(xb[i]);

  float p[16];
  for (int c = 0; c < 16; ++c) {
    float acc = x[8 * c] * x[8 * c];
    for (int j = 1; j < 8; ++j) {
      float sq = x[8 * c + j] * x[8 * c + j];
      acc = acc + sq;
    }
    p[c] = acc;
  }
  for (int d = 8; d >= 1; d >>= 1) {
    float nxt[16];
    for (int c = 0; c < 16; ++c) nxt[c] = p[c] + p[c ^ d];
    memcpy(p, nxt, sizeof p);
  }
  float sum = p[0];
  float ms = sum / 128.0f;
  float den = ms + eps;
  float root = sqrtf(den);
  float r = 1.0f / root;
  for (int i = 0; i < HEAD_DIM; ++i) {
    float xr = x[i] * r;
    float xg = xr * bf16_to_f32(gamma[i]);
    y[i] = oracle_f32_to_bf16(xg);
  }
}

/* RoPE on dims 0..63 ([aiter] API: rope_dim = 64 and the is_neox switch;
 * [sgl] Summary: the bf16 round trip after RoPE).  Pair i (0..31) uses
 * cos_row[i], sin_row[i]:
 *   NeoX:        (a, b) = (y[i], y[i+32])
 *   interleaved: (a, b) = (y[2i], y[2i+1])
 *   a' = bf16(rn32(rn32(a*c) - rn32(b*s))),  b' = bf16(rn32(rn32(b*c) + rn32(a*s)))
 * Dims 64..127 pass through unchanged. */
void oracle_rope_row(uint16_t* y, const float* cos_row, const float* sin_row,
                     int rope_style) {
  for (int i = 0; i < ROPE_DIM / 2; ++i) {
    int ia, ib;
    if (rope_style == ORACLE_ROPE_NEOX) {
      ia = i;
      ib = i + ROPE_DIM / 2;
    } else {
      ia = 2 * i;
      ib = 2 * i + 1;
    }
    float a = bf16_to_f32(y[ia]);
    float b = bf16_to_f32(y[ib]);
    float c = cos_row[i];
    float s = sin_row[i];
    float ac = a * c, bs = b * s, bc = b * c, as = a * s;
    float na = ac - bs;
    float nb = bc + as;
    y[ia] = oracle_f32_to_bf16(na);
    y[ib] = oracle_f32_to_bf16(nb);
  }
}

/* Nearest E2M1 code of a magnitude v >= 0, by brute force over the grid;
 * on an exact tie the even code wins (round half to even, [sgl] Summary and
 * [aiter] One deliberate deviation).  Values above 6 land on code 7.  The
 * distances are exact in double for every v that can sit near a midpoint. */
static int e2m1_nearest_code(double v) {
  int best = 0;
  double best_d = fabs(v - GRID[0]);
  for (int m = 1; m < 8; ++m) {
    double d = fabs(v - GRID[m]);
    if (d < best_d || (d == best_d && (m % 2) == 0 && (best % 2) != 0)) {
      best = m;
      best_d = d;
    }
  }
  return best;
}

/* One per-32 UE8M0 group ([sgl] review, index_pack_exponent and
 * clear_negative_zero):
 *   A = max(max|z|, amax_floor);  t = max(rn32(A / 6), quot_floor)
 *   e = (bits(t) >> 23) + (mantissa(t) != 0), clamped to [1, 254]
 *       i.e. the biased exponent of the power of two ceil_pow2(t)
 *   code = nearest grid point to |z| / 2^(e-127), ties to even
 *   nibble = code | 8 if z < 0 and code != 0  (no -0 codes).
 * A floor of 0 is no floor. */
int oracle_quant_group_floors(const float* z, float amax_floor, float quot_floor,
                              uint8_t* nibbles) {
  float amax = 0.0f;
  for (int i = 0; i < GROUP; ++i) {
    float a = fabsf(z[i]);
    if (a > amax) amax = a;
  }
  if (amax < amax_floor) amax = amax_floor;
  float t = amax / 6.0f;
  if (t < quot_floor) t = quot_floor;
  uint32_t bits = f2u(t);
  int e = (int)(bits >> 23) + ((bits & 0x7fffffu) != 0u ? 1 : 0);
  if (e < 1) e = 1;
  if (e > 254) e = 254;
  double scale = ldexp(1.0, e - 127);
  for (int i = 0; i < GROUP; ++i) {
    double v = fabs((double)z[i]) / scale;
    int m = e2m1_nearest_code(v);
    int neg = (z[i] < 0.0f) && (m != 0);
    nibbles[i] = (uint8_t)(m | (neg ? 8 : 0));
  }
  return e;
}

/* The same group quantiser with only a quotient floor (the packer's form). */
int oracle_quant_group(const float* z, float floor_, uint8_t* nibbles) {
  return oracle_quant_group_floors(z, 0.0f, floor_, nibbles);
}

float oracle_dequant(uint8_t nibble, int e) {
  double v = GRID[nibble & 7] * ldexp(1.0, e - 127);
  if (nibble & 8) v = -v;
  return (float)v; /* exact: at most two significant bits */
}

/* Stage 1 fake-quantises the row to the per-32 UE8M0 E2M1 grid (dequantised
 * back to bf16, which is exact); stage 2 runs the indexer packer on that
 * result with its own floor ([sgl] review: "Keep both quantization stages").
 * Pack: payload byte 16g+j = nibble[32g+2j] | nibble[32g+2j+1] << 4, and
 * exponent byte g = stage-2 exponent of group g.
 * Readings (pages silent): even element in the low nibble; group g in byte g
 * of the little-endian exponent word. */
/* The pack with the four floors as arguments (stage-1 amax and quotient
 * floors, stage-2 amax and quotient floors): lets the tests show which
 * floor readings give the same bytes.  The pre-pass uses
 * (STAGE1_AMAX_FLOOR, 0, 0, STAGE2_QUOT_FLOOR). */
void oracle_quant_pack_row_floors(const uint16_t* row, float s1_amax, float s1_quot,
                                  float s2_amax, float s2_quot, uint8_t* payload64,
                                  uint8_t* exp4, int* stage1_e, int* stage2_e,
                                  uint8_t* stage1_nibbles) {
  for (int g = 0; g < HEAD_DIM / GROUP; ++g) {
    float z[GROUP];
    for (int i = 0; i < GROUP; ++i) z[i] = bf16_to_f32(row[GROUP * g + i]);

    uint8_t n1[GROUP];
    int e1 = oracle_quant_group_floors(z, s1_amax, s1_quot, n1);
    float u[GROUP];
    for (int i = 0; i < GROUP; ++i) {
      float dq = oracle_dequant(n1[i], e1);
      u[i] = bf16_to_f32(oracle_f32_to_bf16(dq));
    }

    uint8_t n2[GROUP];
    int e2 = oracle_quant_group_floors(u, s2_amax, s2_quot, n2);

    for (int j = 0; j < GROUP / 2; ++j)
      payload64[16 * g + j] = (uint8_t)(n2[2 * j] | (n2[2 * j + 1] << 4));
    exp4[g] = (uint8_t)e2;
    if (stage1_e) stage1_e[g] = e1;
    if (stage2_e) stage2_e[g] = e2;
    if (stage1_nibbles) memcpy(stage1_nibbles + GROUP * g, n1, GROUP);
  }
}

void oracle_quant_pack_row(const uint16_t* row, uint8_t* payload64,
                           uint8_t* exp4, int* stage1_e, int* stage2_e,
                           uint8_t* stage1_nibbles) {
  oracle_quant_pack_row_floors(row, STAGE1_AMAX_FLOOR, 0.0f, 0.0f, STAGE2_QUOT_FLOOR,
                               payload64, exp4, stage1_e, stage2_e, stage1_nibbles);
}

/* Optional rotation of a row before quantisation ([csa] Changes: the
 * fused kv-cache kernel does RMSNorm + RoPE + optional Hadamard rotate + FP4
 * quant).  Reading: the normalised 128-point Walsh-Hadamard transform in
 * Sylvester order, y' = bf16(rn32(H y) * rn32(1/sqrt(128))), with H y formed
 * by the fast transform's butterfly stages h = 1, 2, 4, ..., 64, each pair
 * (j, j+h) (bit h of j clear) becoming (rn32(a+b), rn32(a-b)). */
void oracle_hadamard_row(uint16_t* y) {
  float x[HEAD_DIM];
  for (int i = 0; i < HEAD_DIM; ++i) x[i] = bf16_to_f32(y[i]);
  for (int h = 1; h < HEAD_DIM; h *= 2)
    for (int i = 0; i < HEAD_DIM; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        float a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
  const float norm = (float)(1.0 / sqrt((double)HEAD_DIM));
  for (int i = 0; i < HEAD_DIM; ++i) y[i] = oracle_f32_to_bf16(x[i] * norm);
}

/* Keys ([sgl] Summary: RMSNorm, RoPE, both quantisation stages and the paged
 * cache store in one op).  Slot s >= 0 goes to page s/64, offset s%64.
 * Readings: a negative slot means "skip" (slot 0 is an ordinary slot); the
 * 68 bytes of a slot are split inside the 4352-byte page into the 64-byte
 * payload at o*64 and the 4-byte exponent word at 4096 + o*4. */
static int fp8_quant_row(const uint16_t* row, uint8_t* codes);

/* Both output modes share every step up to the quantisation: fp8 = 0 packs
 * the FP4 slot (4352-byte pages), fp8 = 1 the FP8 slot (8448-byte pages). */
static int key_pass(const uint16_t* k, const uint16_t* gamma, float eps,
                    const int64_t* positions, const float* cos_cache,
                    const float* sin_cache, int64_t max_pos, int rope_style,
                    const int64_t* slot_mapping, uint8_t* kv_cache,
                    int64_t num_blocks, int64_t num_tokens, int compress_ratio,
                    int hadamard, int fp8) {
  /* Each token's slot bytes are formed first (in parallel when threads are
   * enabled), then stored in token order, so a repeated slot keeps the last
   * token's bytes whatever the thread count. */
  enum { REC = HEAD_DIM + 4 }; /* 132 >= 68 */
  uint8_t* rec = (uint8_t*)malloc((size_t)(num_tokens > 0 ? num_tokens : 1) * REC);
  signed char* state = (signed char*)malloc((size_t)(num_tokens > 0 ? num_tokens : 1));
  if (!rec || !state) {
    free(rec);
    free(state);
    return -2;
  }
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 64)
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    state[t] = 0; /* skipped */
    if (slot < 0) continue;
    int64_t pos = positions[t];
    if (pos < 0 || pos >= max_pos || slot >= num_blocks * KV_BLOCK) {
      state[t] = -1;
      continue;
    }
    /* [sgl] Summary: RoPE at the group's first position; with groups of
     * compress_ratio consecutive positions that is pos - pos % ratio. */
    int64_t rope_pos = pos - pos % compress_ratio;
    uint16_t y[HEAD_DIM];
    oracle_rmsnorm_row(k + t * HEAD_DIM, gamma, eps, y);
    oracle_rope_row(y, cos_cache + rope_pos * (ROPE_DIM / 2),
                    sin_cache + rope_pos * (ROPE_DIM / 2), rope_style);
    if (hadamard) oracle_hadamard_row(y);
    uint8_t* r = rec + t * REC;
    if (fp8) {
      int e = fp8_quant_row(y, r);
      float scale = (float)ldexp(1.0, e - 127);
      memcpy(r + HEAD_DIM, &scale, 4);
    } else {
      oracle_quant_pack_row(y, r, r + PAYLOAD_BYTES, NULL, NULL, NULL);
    }
    state[t] = 1;
  }
  int status = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    if (state[t] < 0) status = -1;
    if (state[t] <= 0) continue;
    int64_t slot = slot_mapping[t];
    int64_t b = slot / KV_BLOCK, o = slot % KV_BLOCK;
    const uint8_t* r = rec + t * REC;
    if (fp8) {
      uint8_t* page = kv_cache + b * (int64_t)KV_BLOCK * (HEAD_DIM + 4);
      memcpy(page + o * HEAD_DIM, r, HEAD_DIM);
      memcpy(page + KV_BLOCK * HEAD_DIM + o * 4, r + HEAD_DIM, 4);
      continue;
    }
    uint8_t* page = kv_cache + b * PAGE_BYTES;
    memcpy(page + o * PAYLOAD_BYTES, r, PAYLOAD_BYTES);
    memcpy(page + KV_BLOCK * PAYLOAD_BYTES + o * EXP_BYTES, r + PAYLOAD_BYTES, EXP_BYTES);
  }
  free(rec);
  free(state);
  return status;
}

int oracle_k_norm_rope_pack_store_ex(const uint16_t* k, const uint16_t* gamma,
                                     float eps, const int64_t* positions,
                                     const float* cos_cache,
                                     const float* sin_cache, int64_t max_pos,
                                     int rope_style, const int64_t* slot_mapping,
                                     uint8_t* kv_cache, int64_t num_blocks,
                                     int64_t num_tokens, int compress_ratio,
                                     int hadamard) {
  return key_pass(k, gamma, eps, positions, cos_cache, sin_cache, max_pos,
                  rope_style, slot_mapping, kv_cache, num_blocks, num_tokens,
                  compress_ratio, hadamard, 0);
}

int oracle_k_norm_rope_pack_store(const uint16_t* k, const uint16_t* gamma,
                                  float eps, const int64_t* positions,
                                  const float* cos_cache,
                                  const float* sin_cache, int64_t max_pos,
                                  int rope_style, const int64_t* slot_mapping,
                                  uint8_t* kv_cache, int64_t num_blocks,
                                  int64_t num_tokens) {
  return oracle_k_norm_rope_pack_store_ex(k, gamma, eps, positions, cos_cache,
                                          sin_cache, max_pos, rope_style,
                                          slot_mapping, kv_cache, num_blocks,
                                          num_tokens, 1, 0);
}

/* Queries ([sgl] Summary: the query op rotates, quantises and packs the same
 * way and computes the head weights in the same launch; [aiter] API: weights
 * carry the plain weight, fp32 here, nothing folded in). */
/* fp8 = 0: packed FP4 queries, exponent words and plain weights; fp8 = 1:
 * E4M3 codes, the row's scale folded into its weight ([aiter] Summary: the
 * FP8 path folds its per-(token, head) q_scale into the weights). */
static int query_pass(const uint16_t* q, const uint16_t* w,
                      const int64_t* positions, const float* cos_cache,
                      const float* sin_cache, int64_t max_pos, int rope_style,
                      uint8_t* q_out, uint8_t* q_scale, float* weights,
                      int64_t num_tokens, int64_t num_heads, int hadamard,
                      int fp8) {
  int status = 0;
  double wscale = 1.0 / sqrt((double)num_heads * (double)HEAD_DIM);
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 16) reduction(min : status)
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t pos = positions[t];
    if (pos < 0 || pos >= max_pos) {
      status = -1;
      continue;
    }
    for (int64_t h = 0; h < num_heads; ++h) {
      int64_t r = t * num_heads + h;
      uint16_t y[HEAD_DIM];
      memcpy(y, q + r * HEAD_DIM, sizeof y);
      oracle_rope_row(y, cos_cache + pos * (ROPE_DIM / 2),
                      sin_cache + pos * (ROPE_DIM / 2), rope_style);
      if (hadamard) oracle_hadamard_row(y);
      double folded = 1.0;
      if (fp8)
        folded = ldexp(1.0, fp8_quant_row(y, q_out + r * HEAD_DIM) - 127);
      else
        oracle_quant_pack_row(y, q_out + r * PAYLOAD_BYTES,
                              q_scale + r * EXP_BYTES, NULL, NULL, NULL);
      weights[r] = (float)((double)bf16_to_f32(w[r]) * wscale * folded);
    }
  }
  return status;
}

int oracle_q_rope_pack_weights_ex(const uint16_t* q, const uint16_t* w,
                                  const int64_t* positions,
                                  const float* cos_cache, const float* sin_cache,
                                  int64_t max_pos, int rope_style,
                                  uint8_t* q_fp4, uint8_t* q_scale,
                                  float* weights, int64_t num_tokens,
                                  int64_t num_heads, int hadamard) {
  return query_pass(q, w, positions, cos_cache, sin_cache, max_pos, rope_style,
                    q_fp4, q_scale, weights, num_tokens, num_heads, hadamard, 0);
}

int oracle_q_rope_pack_weights(const uint16_t* q, const uint16_t* w,
                               const int64_t* positions,
                               const float* cos_cache, const float* sin_cache,
                               int64_t max_pos, int rope_style,
                               uint8_t* q_fp4, uint8_t* q_scale,
                               float* weights, int64_t num_tokens,
                               int64_t num_heads) {
  return oracle_q_rope_pack_weights_ex(q, w, positions, cos_cache, sin_cache,
                                       max_pos, rope_style, q_fp4, q_scale,
                                       weights, num_tokens, num_heads, 0);
}

/* ---- FP8 output mode ([aiter] Summary and API: the FP8 contract that the
 * FP4 mode extends; the FP8 path folds its per-(token, head) query scale
 * into the head weights).  Readings: E4M3 codes (the e4m3fn format: bias 7,
 * 3 mantissa bits, no infinities, largest finite 448, subnormals m * 2^-9),
 * one power-of-two (UE8M0) scale per 128-element row, and a key slot of 128
 * code bytes plus the scale as an fp32 value, page-split like the FP4 slots
 * (64 x 128 code bytes, then 64 x 4 scale bytes: 8448-byte pages). ---- */

float oracle_e4m3_to_f32(uint8_t c) {
  int sign = c >> 7, ex = (c >> 3) & 15, man = c & 7;
  if (ex == 15 && man == 7) return NAN;
  double v = ex == 0 ? ldexp((double)man, -9) : ldexp(1.0 + man / 8.0, ex - 7);
  return (float)(sign ? -v : v);
}

/* Nearest finite E4M3 value by brute force over the 127 non-negative finite
 * codes; a tie goes to the code with an even mantissa (round half to even);
 * magnitudes above 448 saturate to 448; the sign is kept, zero included. */
uint8_t oracle_f32_to_e4m3(float v) {
  double a = fabs((double)v);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c < 127; ++c) {
    double d = fabs((double)oracle_e4m3_to_f32((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c % 2) == 0 && (best % 2) != 0)) {
      best = c;
      best_d = d;
    }
  }
  if (a > 448.0) best = 126;
  return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* One 128-element row: e = biased exponent of ceil_pow2(max(amax/448,
 * 2^-126)) (the same power-of-two rounding and floor as the FP4 scales),
 * codes of x * 2^(127 - e).  Returns e. */
int oracle_fp8_quant_row(const uint16_t* row, uint8_t* codes) {
  return fp8_quant_row(row, codes);
}

static int fp8_quant_row(const uint16_t* row, uint8_t* codes) {
  float amax = 0.0f;
  for (int i = 0; i < HEAD_DIM; ++i) {
    float a = fabsf(bf16_to_f32(row[i]));
    if (a > amax) amax = a;
  }
  float t = amax / 448.0f;
  if (t < FP8_QUOT_FLOOR) t = FP8_QUOT_FLOOR;
  uint32_t bits = f2u(t);
  int e = (int)(bits >> 23) + (int)((bits & 0x7fffffu) != 0u);
  if (e < 1) e = 1;
  if (e > 254) e = 254;
  for (int i = 0; i < HEAD_DIM; ++i) {
    double x = (double)bf16_to_f32(row[i]) * ldexp(1.0, 127 - e);
    codes[i] = oracle_f32_to_e4m3((float)x);
  }
  return e;
}

enum { FP8_PAGE_BYTES = KV_BLOCK * (HEAD_DIM + 4) /* 8448 */ };

int oracle_k_norm_rope_fp8_store(const uint16_t* k, const uint16_t* gamma,
                                 float eps, const int64_t* positions,
                                 const float* cos_cache, const float* sin_cache,
                                 int64_t max_pos, int rope_style,
                                 const int64_t* slot_mapping, uint8_t* kv_cache,
                                 int64_t num_blocks, int64_t num_tokens,
                                 int compress_ratio, int hadamard) {
  return key_pass(k, gamma, eps, positions, cos_cache, sin_cache, max_pos,
                  rope_style, slot_mapping, kv_cache, num_blocks, num_tokens,
                  compress_ratio, hadamard, 1);
}

int oracle_q_rope_fp8_weights(const uint16_t* q, const uint16_t* w,
                              const int64_t* positions, const float* cos_cache,
                              const float* sin_cache, int64_t max_pos,
                              int rope_style, uint8_t* q_out, float* weights,
                              int64_t num_tokens, int64_t num_heads,
                              int hadamard) {
  return query_pass(q, w, positions, cos_cache, sin_cache, max_pos, rope_style,
                    q_out, NULL, weights, num_tokens, num_heads, hadamard, 1);
}

/* ---- Torch-shaped fake quantisation ([sgl] Summary: the RoPE tail plus
 * FP4 fake-quant of the torch-shaped path, per-32 UE8M0 by default and
 * per-16 E4M3 for compressed KV, keeping the bf16 round trip after RoPE and
 * round half to even).  Reading: RoPE as in the pre-pass (dims 0..63, bf16
 * output), then every value is replaced by its dequantised FP4 value, as
 * bf16 (exact: at most 6 significant bits).
 *   mode 0 (per-32 UE8M0): stage 1 of the pre-pass.
 *   mode 1 (per-16 E4M3): s = E4M3(rn32(amax/6)) (the scale rounded to
 *     E4M3, saturating at 448); code = nearest E2M1 of rn32(x / s) (ties to
 *     even, saturating at 6); value = code * s; a group whose s rounds to 0
 *     is all zeros; no -0 (as in the packed path). ---- */

static void fake_quant_group16(const float* z, float* out) {
  float amax16 = 0.0f;
  for (int i = 0; i < 16; ++i) amax16 = fmaxf(amax16, fabsf(z[i]));
  float t16 = amax16 / 6.0f;
  float sc = oracle_e4m3_to_f32(oracle_f32_to_e4m3(t16));
  for (int i = 0; i < 16; ++i) {
    if (sc == 0.0f) {
      out[i] = 0.0f;
      continue;
    }
    float v = z[i] / sc;
    int m = e2m1_nearest_code(fabs((double)v));
    double d = GRID[m] * (double)sc;
    out[i] = (float)((v < 0.0f && m != 0) ? -d : d);
  }
}

void oracle_fake_quant_row(const uint16_t* row, int mode, uint16_t* out) {
  float z[HEAD_DIM], q[HEAD_DIM];
  for (int i = 0; i < HEAD_DIM; ++i) z[i] = bf16_to_f32(row[i]);
  if (mode == 1) {
    for (int g = 0; g < HEAD_DIM / 16; ++g) fake_quant_group16(z + 16 * g, q + 16 * g);
  } else {
    for (int g = 0; g < HEAD_DIM / GROUP; ++g) {
      uint8_t nib[GROUP];
      int e = oracle_quant_group_floors(z + GROUP * g, STAGE1_AMAX_FLOOR, 0.0f, nib);
      for (int i = 0; i < GROUP; ++i) q[GROUP * g + i] = oracle_dequant(nib[i], e);
    }
  }
  for (int i = 0; i < HEAD_DIM; ++i) out[i] = oracle_f32_to_bf16(q[i]);
}

int oracle_rope_fake_quant(const uint16_t* x, int64_t rows_per_token,
                           const int64_t* positions, const float* cos_cache,
                           const float* sin_cache, int64_t max_pos,
                           int rope_style, int mode, uint16_t* out,
                           int64_t num_rows) {
  int status = 0;
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 256) reduction(min : status)
  for (int64_t r = 0; r < num_rows; ++r) {
    int64_t pos = positions[r / rows_per_token];
    if (pos < 0 || pos >= max_pos) {
      status = -1;
      continue;
    }
    uint16_t y[HEAD_DIM];
    memcpy(y, x + r * HEAD_DIM, sizeof y);
    oracle_rope_row(y, cos_cache + pos * (ROPE_DIM / 2),
                    sin_cache + pos * (ROPE_DIM / 2), rope_style);
    oracle_fake_quant_row(y, mode, out + r * HEAD_DIM);
  }
  return status;
}

/* The scorer ([aiter] Verification, End-to-end: the FP4 paged MQA-logits
 * scorer reads the kernel's own bytes; [vllm] Code Review: the scaled E2M1
 * dot product of packed queries and packed keys with their per-32 block
 * scales).  The DSA indexer score of a query row against a key is the
 * head-weighted sum of ReLU'd dot products.  Readings (pages silent): no
 * causal mask between the next_n rows of one sequence (every row scores
 * [0, context_len)), -inf for the padding columns, and no extra scalar
 * (the head weights already carry H^-1/2 D^-1/2). */
static double dequant_d(uint8_t nibble, int e) {
  double v = GRID[nibble & 7] * ldexp(1.0, e - 127);
  return (nibble & 8) ? -v : v;
}

/* The dequantised key of one 68-byte slot (payload at pg + o*64, exponent
 * word at pg + 4096 + o*4). */
static void key_values(const uint8_t* pg, int64_t o, double* kv) {
  for (int d = 0; d < HEAD_DIM; ++d) {
    uint8_t kbyte = pg[o * PAYLOAD_BYTES + d / 2];
    uint8_t knib = (d % 2) ? (kbyte >> 4) : (kbyte & 15);
    int ke = pg[KV_BLOCK * PAYLOAD_BYTES + o * EXP_BYTES + d / GROUP];
    kv[d] = dequant_d(knib, ke);
  }
}

/* sum_h w[h] * max(0, q_h . k) in fp64 over the H query rows starting at
 * query row r0 (each product of two E2M1 values with power-of-two scales is
 * exact in fp64; the sums round in fp64). */
static double score(const uint8_t* q_fp4, const uint8_t* q_scale, const float* weights,
                    int64_t r0, int64_t num_heads, const double* kv) {
  double qv[HEAD_DIM];
  double acc = 0.0;
  for (int64_t h = 0; h < num_heads; ++h) {
    int64_t r = r0 + h;
    for (int d = 0; d < HEAD_DIM; ++d) {
      uint8_t qbyte = q_fp4[r * PAYLOAD_BYTES + d / 2];
      uint8_t qnib = (d % 2) ? (qbyte >> 4) : (qbyte & 15);
      qv[d] = dequant_d(qnib, q_scale[r * EXP_BYTES + d / GROUP]);
    }
    double dot = 0.0;
    for (int d = 0; d < HEAD_DIM; ++d) dot += qv[d] * kv[d];
    if (dot > 0.0) acc += (double)weights[r] * dot;
  }
  return acc;
}

int oracle_paged_mqa_logits(const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* weights, const uint8_t* kv_cache,
                            int64_t num_blocks, const int32_t* block_table,
                            int64_t block_table_stride,
                            const int32_t* context_lens, float* logits,
                            int64_t logits_stride, int64_t batch,
                            int64_t next_n, int64_t num_heads,
                            int64_t max_context) {
  int status = 0;
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 1) reduction(min : status)
  for (int64_t t = 0; t < batch * next_n; ++t) {
    int64_t b = t / next_n;
    int64_t ctx = context_lens[b];
    double kv[HEAD_DIM];
    for (int64_t s = 0; s < max_context; ++s) {
      float* out = logits + t * logits_stride + s;
      if (s >= ctx) {
        *out = -INFINITY;
        continue;
      }
      int64_t page = block_table[b * block_table_stride + s / KV_BLOCK];
      if (page < 0 || page >= num_blocks) {
        *out = -INFINITY;
        status = -1;
        continue;
      }
      int64_t o = s % KV_BLOCK;
      key_values(kv_cache + page * PAGE_BYTES, o, kv);
      *out = (float)score(q_fp4, q_scale, weights, t * num_heads, num_heads, kv);
    }
  }
  return status;
}

/* The prefill variant of the scorer ([aiter] Summary: the FP4 paged scorer
 * "and its prefill variant" read the packed keys straight out of the
 * cache).  Readings (pages silent on its arguments): the keys of the
 * prefill chunk are consecutive -- key s sits in page s/64 at offset s%64,
 * which is what the key op writes with slot_mapping[s] = s -- so there is
 * no block table; query token t scores the keys s with ks[t] <= s < ke[t];
 * every other column of [0, num_keys) is -inf.  The score is the decode
 * scorer's: sum_h w * max(0, q . k). */
int oracle_mqa_logits_prefill(const uint8_t* q_fp4, const uint8_t* q_scale,
                              const float* weights, const uint8_t* kv_cache,
                              int64_t num_keys, const int32_t* ks, const int32_t* ke,
                              float* logits, int64_t logits_stride, int64_t num_tokens,
                              int64_t num_heads) {
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 1)
  for (int64_t t = 0; t < num_tokens; ++t) {
    double kv[HEAD_DIM];
    for (int64_t s = 0; s < num_keys; ++s) {
      float* out = logits + t * logits_stride + s;
      if (s < ks[t] || s >= ke[t]) {
        *out = -INFINITY;
        continue;
      }
      key_values(kv_cache + (s / KV_BLOCK) * PAGE_BYTES, s % KV_BLOCK, kv);
      *out = (float)score(q_fp4, q_scale, weights, t * num_heads, num_heads, kv);
    }
  }
  return 0;
}
