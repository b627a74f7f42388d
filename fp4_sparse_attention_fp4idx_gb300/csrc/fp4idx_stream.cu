// fp4idx_stream.cu -- the streaming kernel of the fused FP4 indexer pre-pass
// (sm_103a): the path taken, in both output modes and with or without the
// Hadamard rotation, when the head count is a multiple of 16 (or only keys
// are processed).
//
// Sources (web pages, by title and section): "dsv4.1: RoPE and FP4 packing
// kernels" (sglang PR 39656), Summary (key op = RMSNorm + RoPE + both
// quantisation stages + paged store; query op = RoPE + quantisation + head
// weights in one launch); "[HIP] Add FP4 output mode to
// indexer_qk_rope_quant_and_cache" (aiter PR 5484), API (geometry, q_out
// layout, plain weights), One deliberate deviation (round half to even) and
// Summary (the FP8 contract, its query scale folded into the weights);
// "DeepSeek-V4 FP4: fused_compress FP4 scatter + rmsnorm_rope_rotate FP4
// KV-cache kernel" (aiter PR 4029), Changes (the optional Hadamard rotation
// between RoPE and quantisation).
// The arithmetic is fp4idx.cu's, operation for operation (the same closed
// form of the two quantisation stages, the same explicitly rounded fp32
// steps); only the distribution of the work differs.
//
// ---------------------------------------------------------------- design
// The pass moves ~336 bytes per query row and costs a few dozen instructions
// per row, so on a 152-SM part it is bound by HBM only if the issue slots
// per row stay small.  The layout is chosen for that:
//
//  * Work units of 64 rows: a query unit is 64 consecutive rows of the
//    flattened (token, head) row space, a key unit 64 consecutive tokens.
//    Every CTA takes an equal contiguous slice of each list, key units first.
//  * kProducers producer warps per CTA fill a ring of kStagesS shared-memory
//    stages (kShortStages on a short step) with cp.async.bulk (producer p
//    owns units p, p + kProducers, ...
//    and so every kProducers-th stage): a unit's rows (one 16 KB copy when
//    they are contiguous in memory) and, for a query unit, the cos/sin rows
//    of each distinct token.  A warp waits a few hundred cycles for each bulk
//    copy it issues, so the copies per unit are kept few (4 for H >= 64) and
//    spread over more than one warp.  The 32 lanes of a producer look up the
//    positions of the 4 slices of its next 8 units with one load, a batch
//    ahead.  Where the
//    layout allows it, the producer also stages a full query unit's 64 head
//    weights and a full key unit's positions and slots, so that no consumer
//    waits on a global load.
//  * Consumer warps claim 16-row slices (unit i, slice k) in order from a
//    shared counter, so a warp that stalls holds back one slice, not a share
//    of the ring.  A slice is two passes of 8 rows.
//  * Four lanes own a row.  Lane j holds four 8-element parts: dims 8j..8j+7
//    (part 0), 32+8j.. (part 1), 64+8j.. (part 2), 96+8j.. (part 3), i.e. one
//    piece of each of the four 32-element quantisation groups.  A NeoX RoPE
//    pair (i, i+32) is parts 0 and 1 of one lane and an interleaved pair is
//    one bf16x2 word, so RoPE needs no shuffle; the four group maxima travel
//    as two bf16x2 words (two shuffles each); the RMSNorm partial sums of the
//    fixed summation order (runs j, 4+j, 8+j, 12+j) combine in-lane for the
//    distance-8 and distance-4 steps.
//  * Rows are 256 bytes, so the two rows that share a quarter-warp of a
//    128-bit shared load would hit the same banks.  Lanes of odd rows take
//    their parts in the order 1, 0, 3, 2 (register p holds part p ^ parity),
//    which puts the two rows in different halves of the 128-byte bank
//    window.  The swap is undone where it shows: the NeoX sine sign, the
//    interleaved coefficients, the exponent byte order and the store offsets.
//  * The rotation and the FP8 output mode are template flags on the same
//    layout.  The 128-point Walsh-Hadamard butterflies (rotate4) need lane
//    shuffles only at distances 8 and 16; the FP8 quantiser (quant4_fp8)
//    reduces one amax per row over its 4 lanes and stores 8 code bytes per
//    part.
//  * Every wait is bounded (1 s); a timeout sets FP4IDX_ERRFLAG_TIMEOUT and
//    the CTA drains its copies in flight before it exits.

#include <atomic>
#include <mutex>

#include "fp4idx_common.cuh"

namespace fp4idx_impl {
namespace {

#ifndef FP4IDX_STREAM_CONSUMERS
#define FP4IDX_STREAM_CONSUMERS 16
#endif
#ifndef FP4IDX_STREAM_STAGES
#define FP4IDX_STREAM_STAGES 12
#endif
#ifndef FP4IDX_STREAM_SHORT_STAGES
#define FP4IDX_STREAM_SHORT_STAGES 8
#endif
#ifndef FP4IDX_STREAM_PRODUCERS
#define FP4IDX_STREAM_PRODUCERS 4
#endif
#ifndef FP4IDX_STREAM_UNIT_ROWS
#define FP4IDX_STREAM_UNIT_ROWS 64
#endif

constexpr int kUnitRows = FP4IDX_STREAM_UNIT_ROWS;
constexpr int kSliceRows = 16;
constexpr int kSlices = kUnitRows / kSliceRows;
constexpr int kConsumers = FP4IDX_STREAM_CONSUMERS;
constexpr int kProducers = FP4IDX_STREAM_PRODUCERS;
constexpr int kThreadsS = (kConsumers + kProducers) * 32;
constexpr int kStagesS = FP4IDX_STREAM_STAGES;
// A producer's share of units up to which no rows go out ahead of the first
// metadata.
constexpr int kShortShare = 32;
// The largest producer share of a launch up to which the ring is
// kShortStages deep instead of kStagesS.  On a short step the first units'
// copies then queue behind fewer rows (T=8192 at 64 heads, shares of 14:
// 35.2 against 35.6 us; MTP, shares of 4: 16.8 against 17.1 us); from
// shares of ~28 up the deeper ring keeps HBM busier (T=16384: 61.9 against
// 60.9 us; T=65536: 212.5 against 217.3 us with 8 stages throughout).
constexpr int kShallowShare = 16;
constexpr int kShortStages = FP4IDX_STREAM_SHORT_STAGES;
static_assert(kStagesS % kProducers == 0 && kShortStages % kProducers == 0 &&
                  kShortStages >= kProducers && kShortStages <= kStagesS,
              "each producer owns a whole number of stages");
// Stage: rows | a cos row and a sin row per token of a query unit (at most
// 4: slices never straddle tokens), or 64 positions and 64 slots (key unit)
// | header | 64 head weights (query unit).
constexpr int kCoefOff = kUnitRows * kRowBytes;
constexpr int kHdrOff = kCoefOff + kSlices * 256;  // {unit << 2 | kind, first, rows, flags}
constexpr int kWOff = kHdrOff + 16;
constexpr int kStageBytesS = kWOff + kUnitRows * 2;  // 17552 for 64-row units
constexpr int kSmemS = kStagesS * kStageBytesS;
constexpr int kBatch = 32 / kSlices;  // units per position lookup
constexpr int kSlotsOff = kCoefOff + kUnitRows * 8;  // key unit: slots after positions
static_assert(kUnitRows % kSliceRows == 0 && kSlices <= 4 && 32 % kSlices == 0,
              "a unit is 1, 2 or 4 slices");
static_assert(2 * kUnitRows * 8 <= kSlices * 256, "key positions and slots fit the area");
static_assert(kSmemS <= 227 * 1024, "the ring must fit in shared memory");
static_assert(kStageBytesS % 16 == 0, "bulk-copy destinations must be 16-byte aligned");

enum : uint32_t { kUnitKey = 1, kUnitQuery = 2 };
constexpr uint32_t kNoUnit = 0xffffffffu;  // header word 0 before a stage's first unit
// Header flags: bits 0..3 = slice k's position is valid (query unit); bit 4 =
// the unit's weights (query) or positions and slots (key) are in the stage.
constexpr uint32_t kInStage = 1u << 4;

struct SWork {
  int32_t T, H;
  int32_t TH;      // query rows (T * H; 0 without queries)
  int32_t nk, nq;  // key units, query units
  FastDiv hdiv;    // n / H
  int q_mode;      // 0: all query rows contiguous, 1: heads of a token contiguous, 2: per row
  int k_contig;    // key rows contiguous
  int w_bulk;      // head weights dense ([T, H]) and 16-byte aligned
  int meta_bulk;   // positions and slots 16-byte aligned
  int withhold;    // testing: a unit of CTA 0 whose copies are not issued (-1: none)
  int stages;      // ring depth S of this launch: kShortStages or kStagesS
  uint32_t smul;   // ceil(2^32 / S)
};

// Uses of unit i's stage before unit i, i / S (the stage is i - uses * S):
// S * ceil(2^32 / S) = 2^32 + d with d < S, so the high word of i * smul is
// the quotient for every i below 2^32 / S, far above any unit count.
__device__ __forceinline__ uint32_t stage_uses(int i, const SWork& wk) {
  return __umulhi((uint32_t)i, wk.smul);
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ int64_t lds_s64(uint32_t addr) {
  int64_t v;
  asm volatile("ld.shared.s64 %0, [%1];" : "=l"(v) : "r"(addr));
  return v;
}

// --------------------------------------------------------------- helpers
// (r0, r1) = (rn(a0-b0), rn(a1-b1)).
__device__ __forceinline__ void diff2(float& r0, float& r1, float a0, float a1, float b0,
                                      float b1) {
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Bounded wait for a phase, the same answer in every lane of the warp (all
// 32 lanes call): false if the time limit ran out or the CTA is aborting.
__device__ __forceinline__ bool lane_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort != 0 || global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              const volatile int* abort) {
  return __all_sync(kFull, lane_wait(bar, parity, abort));
}

__device__ __forceinline__ uint32_t lds_volatile(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// A consumer's wait for unit i in stage `stage` (all 32 lanes call).  Slices
// are claimed ahead of the producers, so the stage may still be waiting for
// unit i - stages or older; a parity wait alone would then alias an older
// phase.  So first wait (bounded) until the producer has tagged the stage's
// header with i -- it does so only after the previous unit in the stage was
// released, i.e. once the stage's barrier is in unit i's phase -- and only
// then wait for that phase.
__device__ __forceinline__ bool wait_unit(uint32_t stage, uint32_t bar, int i, const SWork& wk,
                                          const volatile int* abort) {
  bool ok = (lds_volatile(stage + kHdrOff) >> 2) == (uint32_t)i;
  if (!ok) {
    const unsigned long long t0 = global_ns();
    for (;;) {
      __nanosleep(64);
      if ((lds_volatile(stage + kHdrOff) >> 2) == (uint32_t)i) {
        ok = true;
        break;
      }
      if (*abort != 0 || global_ns() - t0 > kWaitLimitNs) break;
    }
  }
  if (!__all_sync(kFull, ok)) return false;
  return wait_or_abort(bar, stage_uses(i, wk) & 1u, abort);
}

// RoPE coefficients of one lane, in the order of its registers A (parts
// 0 ^ par) and B (part 1 ^ par).
//   NeoX: pair e of A/B (element e of the 8) uses c[e], s[e] (the pair's
//   frequency 8j+e); for odd rows (A = part 1) s is negated, so that both
//   parities compute A' = A c - B s, B' = B c + A s.
//   Interleaved: word k of A is the pair fA+k with fA = 4j + 16 par (B: the
//   other half); c[0..3], s[0..3] are A's cos/sin, c[4..7], s[4..7] B's,
//   and sn = -s.
template <int kStyle>
struct Coef {
  float c[8], s[8], sn[8];
  __device__ __forceinline__ void neox_finish(bool par) {
    if (par) {
#pragma unroll
      for (int e = 0; e < 8; ++e) s[e] = -s[e];
    }
  }
  __device__ __forceinline__ void interleaved_finish() {
#pragma unroll
    for (int e = 0; e < 8; ++e) sn[e] = -s[e];
  }
  // NeoX from a cos/sin row at `cos_row`/`sin_row` (shared memory).
  __device__ __forceinline__ void load_smem(uint32_t cos_row, uint32_t sin_row, int j, bool par) {
    if (kStyle == FP4IDX_ROPE_NEOX) {
      const float4 c0 = lds_f4(cos_row + 32u * j), c1 = lds_f4(cos_row + 32u * j + 16u);
      const float4 s0 = lds_f4(sin_row + 32u * j), s1 = lds_f4(sin_row + 32u * j + 16u);
      set8(c0, c1, s0, s1);
      neox_finish(par);
    } else {
      const uint32_t oa = 16u * j + (par ? 64u : 0u), ob = 16u * j + (par ? 0u : 64u);
      set8(lds_f4(cos_row + oa), lds_f4(cos_row + ob), lds_f4(sin_row + oa),
           lds_f4(sin_row + ob));
      interleaved_finish();
    }
  }
  __device__ __forceinline__ void load_global(const float* cos_row, const float* sin_row, int j,
                                              bool par) {
    if (kStyle == FP4IDX_ROPE_NEOX) {
      set8(ld_f4(cos_row + 8 * j), ld_f4(cos_row + 8 * j + 4), ld_f4(sin_row + 8 * j),
           ld_f4(sin_row + 8 * j + 4));
      neox_finish(par);
    } else {
      const int oa = 4 * j + (par ? 16 : 0), ob = 4 * j + (par ? 0 : 16);
      set8(ld_f4(cos_row + oa), ld_f4(cos_row + ob), ld_f4(sin_row + oa), ld_f4(sin_row + ob));
      interleaved_finish();
    }
  }
  // NeoX: c = (c0, c1), s = (s0, s1).  Interleaved: c[0..3] = A's cos,
  // c[4..7] = B's cos, likewise s.
  __device__ __forceinline__ void set8(const float4& c0, const float4& c1, const float4& s0,
                                       const float4& s1) {
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
    c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
    s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
  }
};

// RoPE of registers A and B (see Coef).  Each result is
// rn(rn(x*c) -/+ rn(y*s)) rounded to bf16; the products come from prod2
// (exactly rounded, never fused with the sum).
template <int kStyle>
__device__ __forceinline__ void rope4(uint32_t (&a)[4], uint32_t (&b)[4], const Coef<kStyle>& cf,
                                      float z) {
  if (kStyle == FP4IDX_ROPE_NEOX) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a0 = bf16_lo(a[k]), a1 = bf16_hi(a[k]);
      const float b0 = bf16_lo(b[k]), b1 = bf16_hi(b[k]);
      const float c0 = cf.c[2 * k], c1 = cf.c[2 * k + 1];
      const float s0 = cf.s[2 * k], s1 = cf.s[2 * k + 1];
      float ac0, ac1, bs0, bs1, bc0, bc1, as0, as1, r0, r1, q0, q1;
      prod2(ac0, ac1, a0, a1, c0, c1, z);
      prod2(bs0, bs1, b0, b1, s0, s1, z);
      prod2(bc0, bc1, b0, b1, c0, c1, z);
      prod2(as0, as1, a0, a1, s0, s1, z);
      diff2(r0, r1, ac0, ac1, bs0, bs1);
      sum2(q0, q1, bc0, bc1, as0, as1);
      a[k] = pack_bf16x2(r0, r1);
      b[k] = pack_bf16x2(q0, q1);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t(&x)[4] = h == 0 ? a : b;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = bf16_lo(x[k]), x1 = bf16_hi(x[k]);
        const float c = cf.c[4 * h + k];
        float m0, m1, n0, n1, r0, r1;
        prod2(m0, m1, x0, x1, c, c, z);
        prod2(n0, n1, x1, x0, cf.sn[4 * h + k], cf.s[4 * h + k], z);
        sum2(r0, r1, m0, m1, n0, n1);  // (x0 c - x1 s, x1 c + x0 s)
        x[k] = pack_bf16x2(r0, r1);
      }
    }
  }
}

__device__ __forceinline__ void unpack8(const uint32_t (&x)[4], float (&v)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = bf16_lo(x[k]);
    v[2 * k + 1] = bf16_hi(x[k]);
  }
}

// x = bf16(rn(v * rn32(1/sqrt(128)))), the rotation's normalisation; the
// products packed over the element pairs (i, i + PS).
template <int PS>
__device__ __forceinline__ void scale_pack8(const float (&v)[8], uint32_t (&x)[4]) {
  const float norm = 0.08838834764831845f;
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (!(i & PS)) mul2(y[i], y[i + PS], v[i], v[i + PS], norm, norm);
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = pack_bf16x2(y[2 * k], y[2 * k + 1]);
}

// (r0, r1) = (rn(a0*s + c0), rn(a1*s + c1)) for s = +-1: exactly rn(c +- a).
__device__ __forceinline__ void pm2(float& r0, float& r1, float a0, float a1, float s, float c0,
                                    float c1) {
  asm("{\n\t.reg .b64 ra, rs, rc, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rs, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %6};\n\t"
      "fma.rn.f32x2 rr, ra, rs, rc;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(s), "f"(c0), "f"(c1));
}

// The rotation's packed fp32 operations pair elements (i, i + kPairStride)
// of a part in every stage, so that each pair stays in one aligned register
// pair throughout; the stage h == kPairStride runs on scalars.  (Pairing
// differently in one stage costs register moves: 9% of the rotated
// pre-pass's time.)
constexpr int kPairStride = 1;

// In-lane butterfly stage h of one 8-element part; packed over the element
// pairs (i, i + PS), scalar for h == PS.
template <int PS>
__device__ __forceinline__ void part_stage(float (&v)[8], int h) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i & h) continue;
    if (h == PS) {
      const float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    } else if (!(i & PS)) {
      float s0, s1, d0, d1;
      sum2(s0, s1, v[i], v[i + PS], v[i + h], v[i + h + PS]);
      diff2(d0, d1, v[i], v[i + PS], v[i + h], v[i + h + PS]);
      v[i] = s0;
      v[i + PS] = s1;
      v[i + h] = d0;
      v[i + h + PS] = d1;
    }
  }
}

// Normalised 128-point Walsh-Hadamard rotation of a row held by 4 lanes
// (register p = part p ^ par, part q = dims 32q + 8j .. 32q + 8j + 7).  The
// butterfly stages run in the order h = 1, 2, ..., 64, each pair (lower,
// upper) becoming (rn(lower + upper), rn(lower - upper)): h = 1, 2, 4 inside
// a part, h = 8 and 16 with lanes j^1 and j^2 (a lane computes rn(partner
// +- own) as one exact-product fma), h = 32 between registers 0/1 and 2/3
// (the part swap of odd rows folded into the sign), h = 64 between
// registers 0/2 and 1/3.  Then one product with rn32(1/sqrt(128)) and the
// bf16 rounding.  All 32 lanes call (shuffles).
__device__ __forceinline__ void rotate4(uint32_t (&x0)[4], uint32_t (&x1)[4], uint32_t (&x2)[4],
                                        uint32_t (&x3)[4], int j, bool par) {
  constexpr int PS = kPairStride;
  float v[4][8];
  unpack8(x0, v[0]);
  unpack8(x1, v[1]);
  unpack8(x2, v[2]);
  unpack8(x3, v[3]);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    part_stage<PS>(v[q], 1);
    part_stage<PS>(v[q], 2);
    part_stage<PS>(v[q], 4);
  }
#pragma unroll
  for (int m = 1; m <= 2; m *= 2) {  // h = 8, 16: lower lane own + other, upper other - own
    const float sg = (j & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i & PS) continue;
        const float o0 = __shfl_xor_sync(kFull, v[q][i], m);
        const float o1 = __shfl_xor_sync(kFull, v[q][i + PS], m);
        pm2(v[q][i], v[q][i + PS], v[q][i], v[q][i + PS], sg, o0, o1);
      }
  }
  {  // h = 32: register 0 is the lower part for even rows, the upper for odd
    const float sg = par ? -1.0f : 1.0f;
#pragma unroll
    for (int q = 0; q < 4; q += 2)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i & PS) continue;
        const float a0 = v[q][i], a1 = v[q][i + PS], b0 = v[q + 1][i], b1 = v[q + 1][i + PS];
        pm2(v[q][i], v[q][i + PS], a0, a1, sg, b0, b1);           // rn(b +- a)
        pm2(v[q + 1][i], v[q + 1][i + PS], b0, b1, -sg, a0, a1);  // rn(a -+ b)
      }
  }
#pragma unroll
  for (int q = 0; q < 2; ++q)  // h = 64: registers 0/1 lower, 2/3 upper
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & PS) continue;
      float s0, s1, d0, d1;
      sum2(s0, s1, v[q][i], v[q][i + PS], v[q + 2][i], v[q + 2][i + PS]);
      diff2(d0, d1, v[q][i], v[q][i + PS], v[q + 2][i], v[q + 2][i + PS]);
      v[q][i] = s0;
      v[q][i + PS] = s1;
      v[q + 2][i] = d0;
      v[q + 2][i + PS] = d1;
    }
  scale_pack8<PS>(v[0], x0);
  scale_pack8<PS>(v[1], x1);
  scale_pack8<PS>(v[2], x2);
  scale_pack8<PS>(v[3], x3);
}

// Lane-local max(|x|) of two 8-element parts, packed: low half = part x,
// high half = part y (bf16 bits; the sign bits are garbage).
__device__ __forceinline__ uint32_t pair_amax(const uint32_t (&x)[4], const uint32_t (&y)[4]) {
  const uint32_t mx = hmax_abs(hmax_abs(x[0], x[1]), hmax_abs(x[2], x[3]));
  const uint32_t my = hmax_abs(hmax_abs(y[0], y[1]), hmax_abs(y[2], y[3]));
  return hmax_abs(prmt(mx, my, 0x5410u), prmt(mx, my, 0x7632u));
}

// Stage-1 scale, stage-2 decision and stored exponent of two groups whose
// bf16 amax bits are the halves of m (see the closed form in fp4idx.cu):
// sa/sb = 2^(127-e1) per group, ha/hb = 0x11111111 where stage 2 halves the
// scale, e2 = e1 - halve per 16-bit half.
__device__ __forceinline__ void group_exps(uint32_t m, float& sa, float& sb, uint32_t& ha,
                                           uint32_t& hb, uint32_t& e2) {
  const uint32_t ep = ((m + 0x003f003fu) >> 7) & 0x01ff01ffu;
  const uint32_t ie = umin16x2(0x01000100u - ep, 0x00fd00fdu);  // 254 - e1 per half
  sa = __uint_as_float(ie << 23);
  sb = __uint_as_float((ie >> 16) << 23);
  const uint32_t mq = uadd16x2(m & 0x007f007fu, 0xffbfffbfu);  // mantissa - 65
  const bool a2 = (mq & 0xffffu) < 31u && (ie & 0xffffu) < 253u;
  const bool b2 = (mq >> 16) < 31u && (ie >> 16) < 253u;
  ha = a2 ? 0x11111111u : 0u;
  hb = b2 ? 0x11111111u : 0u;
  e2 = 0x00fe00feu - ie - (a2 ? 1u : 0u) - (b2 ? 0x10000u : 0u);
}

// Stage-1 nibbles p -> final codes.  With hk = 0x11111111 (stage 2 halves
// the scale) every magnitude m (m <= 5) becomes m + min(m, 2): m + 2 when
// m >= 2, 2m when m < 2.  Sign bits survive only on non-zero magnitudes (no
// -0 codes).  No nibble carries: results stay <= 15.
__device__ __forceinline__ uint32_t finish4(uint32_t p, uint32_t hk) {
  const uint32_t mag = p & 0x77777777u;
  const uint32_t sgn = p & (mag + 0x77777777u) & 0x88888888u;  // bit 3 iff mag != 0
  const uint32_t g = ((mag >> 1) | (mag >> 2)) & hk;            // m >= 2
  const uint32_t b0 = mag & ~g & hk;                            // m == 1
  return mag + sgn + b0 + (g << 1);
}

__device__ __forceinline__ uint32_t codes8(const uint32_t (&x)[4], float s, uint32_t hk) {
  float v[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) mul2(v[2 * k], v[2 * k + 1], bf16_lo(x[k]), bf16_hi(x[k]), s, s);
  return finish4(e2m1x8(v), hk);
}

// Both quantisation stages of one row held by 4 lanes (all 32 lanes call:
// shuffles).  x[p] is part p ^ par.  Returns the lane's four code words in
// register order and the row's exponent word in group order.
__device__ __forceinline__ void quant4(const uint32_t (&x0)[4], const uint32_t (&x1)[4],
                                       const uint32_t (&x2)[4], const uint32_t (&x3)[4], bool par,
                                       uint32_t (&code)[4], uint32_t& ew) {
  uint32_t m01 = pair_amax(x0, x1), m23 = pair_amax(x2, x3);
  m01 = hmax_abs(m01, __shfl_xor_sync(kFull, m01, 1));
  m23 = hmax_abs(m23, __shfl_xor_sync(kFull, m23, 1));
  m01 = hmax_abs(m01, __shfl_xor_sync(kFull, m01, 2));
  m23 = hmax_abs(m23, __shfl_xor_sync(kFull, m23, 2));
  float s0, s1, s2, s3;
  uint32_t h0, h1, h2, h3, e01, e23;
  group_exps(m01 & 0x7fff7fffu, s0, s1, h0, h1, e01);
  group_exps(m23 & 0x7fff7fffu, s2, s3, h2, h3, e23);
  code[0] = codes8(x0, s0, h0);
  code[1] = codes8(x1, s1, h1);
  code[2] = codes8(x2, s2, h2);
  code[3] = codes8(x3, s3, h3);
  ew = prmt(e01, e23, par ? 0x4602u : 0x6420u);
}

// The 8 E4M3 codes of one 8-element part: x * inv (an exact product by a
// power of two), round half to even, saturating at 448.
__device__ __forceinline__ uint2 codes8_fp8(const uint32_t (&x)[4], float inv) {
  float v[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) mul2(v[2 * k], v[2 * k + 1], bf16_lo(x[k]), bf16_hi(x[k]), inv, inv);
  return make_uint2(e4m3x4(v[0], v[1], v[2], v[3]), e4m3x4(v[4], v[5], v[6], v[7]));
}

// FP8 output mode for a row held by 4 lanes (all 32 lanes call): the row's
// amax over its 128 elements, one power-of-two scale 2^(e-127) =
// ceil_pow2(max(rn(amax/448), 2^-126)), and the E4M3 codes of x * 2^(127-e),
// 8 bytes per register.
__device__ __forceinline__ void quant4_fp8(const uint32_t (&x0)[4], const uint32_t (&x1)[4],
                                           const uint32_t (&x2)[4], const uint32_t (&x3)[4],
                                           uint2 (&code)[4], uint32_t& e) {
  uint32_t m = hmax_abs(pair_amax(x0, x1), pair_amax(x2, x3));
  m = hmax_abs(m, prmt(m, m, 0x1032u));  // both halves
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 1));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 2));
  const float amax = __uint_as_float((m & 0x7fffu) << 16);
  const float t = fmaxf(__fdiv_rn(amax, 448.0f), 1.17549435082228750797e-38f);
  const uint32_t tb = __float_as_uint(t);
  e = (tb >> 23) + ((tb & 0x7fffffu) != 0u ? 1u : 0u);  // 1 .. 248 for finite bf16
  const float inv = __uint_as_float((254u - e) << 23);  // 2^(127-e), a normal float
  code[0] = codes8_fp8(x0, inv);
  code[1] = codes8_fp8(x1, inv);
  code[2] = codes8_fp8(x2, inv);
  code[3] = codes8_fp8(x3, inv);
}

// Sum of the squares of 8 elements, left to right, each step rounded.
__device__ __forceinline__ float sumsq8(const uint32_t (&x)[4]) {
  float acc = __fmul_rn(bf16_lo(x[0]), bf16_lo(x[0]));
  acc = __fadd_rn(acc, __fmul_rn(bf16_hi(x[0]), bf16_hi(x[0])));
#pragma unroll
  for (int k = 1; k < 4; ++k) {
    acc = __fadd_rn(acc, __fmul_rn(bf16_lo(x[k]), bf16_lo(x[k])));
    acc = __fadd_rn(acc, __fmul_rn(bf16_hi(x[k]), bf16_hi(x[k])));
  }
  return acc;
}

// x <- bf16(rn(rn(x * r) * gamma)) for one 8-element part.
__device__ __forceinline__ void norm8(uint32_t (&x)[4], float r, const uint4 g) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float u0, u1, y0, y1;
    mul2(u0, u1, bf16_lo(x[k]), bf16_hi(x[k]), r, r);
    mul2(y0, y1, u0, u1, bf16_lo(gw[k]), bf16_hi(gw[k]));
    x[k] = pack_bf16x2(y0, y1);
  }
}

// Per-lane geometry of the part swap: shared-memory offsets of registers
// 0/1 (+128 for 2/3) within a row, and payload offsets of registers 0/1 (+32
// for 2/3) within a 64-byte slot.
struct Lanes {
  int lane, j;
  bool par;
  uint32_t lds_a, lds_b, st_a, st_b;
  __device__ __forceinline__ Lanes() {
    lane = threadIdx.x & 31;
    j = lane & 3;
    par = ((lane >> 2) & 1) != 0;
    lds_a = 16u * j + (par ? 64u : 0u);
    lds_b = 16u * j + (par ? 0u : 64u);
    st_a = 4u * j + (par ? 16u : 0u);
    st_b = 4u * j + (par ? 0u : 16u);
  }
  __device__ __forceinline__ void load(uint32_t row, uint32_t (&x0)[4], uint32_t (&x1)[4],
                                       uint32_t (&x2)[4], uint32_t (&x3)[4]) const {
    lds128(row + lds_a, x0);
    lds128(row + lds_b, x1);
    lds128(row + 128u + lds_a, x2);
    lds128(row + 128u + lds_b, x3);
  }
  __device__ __forceinline__ void store(uint8_t* slot, const uint32_t (&code)[4]) const {
    *reinterpret_cast<uint32_t*>(slot + st_a) = code[0];
    *reinterpret_cast<uint32_t*>(slot + st_b) = code[1];
    *reinterpret_cast<uint32_t*>(slot + 32 + st_a) = code[2];
    *reinterpret_cast<uint32_t*>(slot + 32 + st_b) = code[3];
  }
  // FP8 codes of register p (part p ^ par) at bytes 32 (p ^ par) + 8j of a
  // 128-byte code row.
  __device__ __forceinline__ void store8(uint8_t* row, const uint2 (&code)[4]) const {
    const uint32_t a = 2u * st_a, b = 2u * st_b;
    *reinterpret_cast<uint2*>(row + a) = code[0];
    *reinterpret_cast<uint2*>(row + b) = code[1];
    *reinterpret_cast<uint2*>(row + 64 + a) = code[2];
    *reinterpret_cast<uint2*>(row + 64 + b) = code[3];
  }
};

// --------------------------------------------------------- consumer side
// Rows 16*sl .. of a query unit (first flattened row row0, n rows).
template <int kStyle, bool kRotate, bool kFp8>
__device__ __forceinline__ void query_slice(uint32_t stage, int32_t row0, int n, uint32_t flags,
                                            int sl, const SWork& wk, const QArgs& qa,
                                            const Shared& sh) {
  const Lanes ln;
  const int r_first = kSliceRows * sl;
  if (r_first >= n) return;  // uniform
  const int ns = min(kSliceRows, n - r_first);
  const int32_t rs = row0 + r_first;  // the slice's first row; one token
  if (((flags >> sl) & 1u) == 0u) {
    if (ln.lane == 0) flag_error(sh.err, FP4IDX_ERRFLAG_POSITION);
    return;  // the token's position is out of range: its rows are skipped
  }
  const int32_t t = (int32_t)wk.hdiv.div((uint32_t)rs);
  const int32_t h0 = rs - t * wk.H;
  uint32_t wb = 0;
  if (ln.lane < ns)
    wb = (flags & kInStage) ? lds_u16(stage + kWOff + 2u * (r_first + ln.lane))
                            : __ldg(qa.w + (int64_t)t * qa.w_tstride + h0 + ln.lane);

  Coef<kStyle> cf;
  const uint32_t coef =
      stage + kCoefOff + 256u * (uint32_t)(t - (int32_t)wk.hdiv.div((uint32_t)row0));
  cf.load_smem(coef, coef + 128u, ln.j, ln.par);
  // Both passes unconditionally (rows past the unit's end read stale
  // shared memory and are not stored), so that they can overlap.
#pragma unroll
  for (int pass = 0; pass < kSliceRows / 8; ++pass) {
    const int r = 8 * pass + (ln.lane >> 2);
    uint32_t x0[4], x1[4], x2[4], x3[4];
    ln.load(stage + (uint32_t)(r_first + r) * kRowBytes, x0, x1, x2, x3);
    rope4<kStyle>(x0, x1, cf, sh.neg_zero);
    if constexpr (kRotate) rotate4(x0, x1, x2, x3, ln.j, ln.par);
    if constexpr (kFp8) {
      // codes at q_fp4 + row*128; the row's scale folded into its weight
      uint2 code[4];
      uint32_t e;
      quant4_fp8(x0, x1, x2, x3, code, e);
      const float wr = __uint_as_float(__shfl_sync(kFull, wb, r) << 16);
      if (r < ns) {
        const int64_t row = rs + r;
        ln.store8(qa.q_fp4 + row * FP4IDX_HEAD_DIM, code);
        if (ln.j == 0)
          qa.weights[row] = __fmul_rn(__fmul_rn(wr, qa.wscale), __uint_as_float(e << 23));
      }
    } else {
      uint32_t code[4], ew;
      quant4(x0, x1, x2, x3, ln.par, code, ew);
      if (r < ns) {
        const int64_t row = rs + r;
        ln.store(qa.q_fp4 + row * kPayloadBytes, code);
        if (ln.j == 0) *reinterpret_cast<uint32_t*>(qa.q_scale + row * 4) = ew;
      }
    }
  }
  if (!kFp8 && ln.lane < ns)
    qa.weights[rs + ln.lane] = __fmul_rn(__uint_as_float(wb << 16), qa.wscale);
}

// Rows 16*sl .. of a key unit (tokens t0 .. t0 + n - 1).
template <int kStyle, bool kRotate, bool kFp8>
__device__ __forceinline__ void key_slice(uint32_t stage, int32_t t0, int n, uint32_t flags,
                                          int sl, const KArgs& ka, const Shared& sh) {
  const Lanes ln;
  const int r_first = kSliceRows * sl;
  if (r_first >= n) return;  // uniform
  const int ns = min(kSliceRows, n - r_first);
#pragma unroll 1
  for (int pass = 0; pass < kSliceRows / 8; ++pass) {
    if (8 * pass >= ns) break;  // uniform
    const int r = r_first + 8 * pass + (ln.lane >> 2);
    const bool have = r < r_first + ns;
    int64_t pos = 0, slot = -1;
    if (have) {
      if (flags & kInStage) {
        pos = lds_s64(stage + kCoefOff + 8u * r);
        slot = lds_s64(stage + kSlotsOff + 8u * r);
      } else {
        pos = __ldg(sh.pos + t0 + r);
        slot = __ldg(ka.slots + t0 + r);
      }
    }
    bool live = slot >= 0;
    if (live) {
      const bool pos_ok = pos >= 0 && pos < sh.max_pos;
      const bool slot_ok = slot < ka.num_blocks * kKvBlock;
      if (!(pos_ok && slot_ok)) {
        if (ln.j == 0)
          flag_error(sh.err, (pos_ok ? 0u : FP4IDX_ERRFLAG_POSITION) |
                                 (slot_ok ? 0u : FP4IDX_ERRFLAG_SLOT));
        live = false;
      }
    }
    if (!live) pos = 0;
    pos &= ka.pos_mask;
    Coef<kStyle> cf;
    cf.load_global(sh.cos + pos * kRopeHalf, sh.sin + pos * kRopeHalf, ln.j, ln.par);

    uint32_t x0[4], x1[4], x2[4], x3[4];
    ln.load(stage + (uint32_t)r * kRowBytes, x0, x1, x2, x3);
    // RMSNorm.  Register p holds run 4(p ^ par) + j of the fixed summation
    // order; registers 0/2 and 1/3 are the distance-8 pairs, their two sums
    // the distance-4 pair, lanes j^2 and j^1 the rest.
    float ss = __fadd_rn(__fadd_rn(sumsq8(x0), sumsq8(x2)), __fadd_rn(sumsq8(x1), sumsq8(x3)));
    ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 2));
    ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 1));
    const float ms = __fmul_rn(ss, 0.0078125f);  // /128, exact scaling
    const float rr = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, ka.eps)));
    const uint4* g = reinterpret_cast<const uint4*>(ka.gamma);
    const int pa = ln.par ? 1 : 0;
    norm8(x0, rr, __ldg(g + 4 * (0 ^ pa) + ln.j));
    norm8(x1, rr, __ldg(g + 4 * (1 ^ pa) + ln.j));
    norm8(x2, rr, __ldg(g + 4 * (2 ^ pa) + ln.j));
    norm8(x3, rr, __ldg(g + 4 * (3 ^ pa) + ln.j));
    rope4<kStyle>(x0, x1, cf, sh.neg_zero);
    if constexpr (kRotate) rotate4(x0, x1, x2, x3, ln.j, ln.par);
    if constexpr (kFp8) {
      // a 128-byte code row at o*128 of the page, the fp32 scale at 8192 + o*4
      uint2 code[4];
      uint32_t e;
      quant4_fp8(x0, x1, x2, x3, code, e);
      if (live) {
        uint8_t* page = ka.cache + (slot / kKvBlock) * (int64_t)kFp8PageBytes;
        const int64_t o = slot % kKvBlock;
        ln.store8(page + o * FP4IDX_HEAD_DIM, code);
        if (ln.j == 0) *reinterpret_cast<uint32_t*>(page + kFp8ScaleOffset + 4 * o) = e << 23;
      }
      continue;
    }
    uint32_t code[4], ew;
    quant4(x0, x1, x2, x3, ln.par, code, ew);
    if (live) {
      uint8_t* page = ka.cache + (slot / kKvBlock) * (int64_t)kPageBytes;
      const int64_t o = slot % kKvBlock;
      ln.store(page + o * kPayloadBytes, code);
      if (ln.j == 0) *reinterpret_cast<uint32_t*>(page + kExpOffset + 4 * o) = ew;
    }
  }
}

// --------------------------------------------------------- producer side
// Unit i of this CTA: key units first, then query units.
struct Units {
  int32_t k_lo, nk, q_lo, nq;
  __device__ __forceinline__ int total() const { return nk + nq; }
};

// The rows of unit i into its stage (no arrive).
__device__ __forceinline__ void issue_rows(int i, const Units& u, const SWork& wk,
                                           const KArgs& ka, const QArgs& qa, uint32_t stage,
                                           uint32_t bar) {
  const int lane = threadIdx.x & 31;
  if (i < u.nk) {
    const int32_t t0 = (u.k_lo + i) * kUnitRows;
    const int n = min(kUnitRows, wk.T - t0);
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)n * kRowBytes);
    if (wk.k_contig) {
      if (lane == 0)
        bulk_g2s(stage, ka.k + (int64_t)t0 * ka.k_stride, (uint32_t)n * kRowBytes, bar);
    } else {
      for (int r = lane; r < n; r += 32)
        bulk_g2s(stage + (uint32_t)r * kRowBytes, ka.k + (int64_t)(t0 + r) * ka.k_stride,
                 kRowBytes, bar);
    }
    return;
  }
  const int32_t row0 = (u.q_lo + i - u.nk) * kUnitRows;
  const int n = min(kUnitRows, wk.TH - row0);
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)n * kRowBytes);
  if (wk.q_mode == 0) {
    if (lane == 0)
      bulk_g2s(stage, qa.q + (int64_t)row0 * FP4IDX_HEAD_DIM, (uint32_t)n * kRowBytes, bar);
  } else if (wk.q_mode == 1) {
    if (lane < kSlices && kSliceRows * lane < n) {
      const int32_t row = row0 + kSliceRows * lane;
      const int32_t t = (int32_t)wk.hdiv.div((uint32_t)row);
      const int32_t h = row - t * wk.H;
      bulk_g2s(stage + (uint32_t)(kSliceRows * lane) * kRowBytes,
               qa.q + (int64_t)t * qa.q_tstride + (int64_t)h * FP4IDX_HEAD_DIM,
               (uint32_t)min(kSliceRows, n - kSliceRows * lane) * kRowBytes, bar);
    }
  } else {
    for (int r = lane; r < n; r += 32) {
      const int32_t row = row0 + r;
      const int32_t t = (int32_t)wk.hdiv.div((uint32_t)row);
      const int32_t h = row - t * wk.H;
      bulk_g2s(stage + (uint32_t)r * kRowBytes,
               qa.q + (int64_t)t * qa.q_tstride + (int64_t)h * qa.q_hstride, kRowBytes, bar);
    }
  }
}

// Position of this lane's slice in producer p's batch of own units mb ..
// mb + kBatch - 1 (unit i = p + kProducers * m; lane = 4 * (m - mb) + slice);
// 0 where there is none.
__device__ __forceinline__ int64_t slice_pos(int p, int mb, const Units& u, const SWork& wk,
                                             const Shared& sh) {
  const int lane = threadIdx.x & 31;
  const int i = p + kProducers * (mb + lane / kSlices);
  if (i < u.nk || i >= u.total()) return 0;
  const int32_t row = (u.q_lo + i - u.nk) * kUnitRows + kSliceRows * (lane % kSlices);
  if (row >= wk.TH) return 0;
  return __ldg(sh.pos + wk.hdiv.div((uint32_t)row));
}

// The rest of unit i: the cos/sin rows of a query unit's slices, the header
// and the producer's arrive.
// `kb` is unit i's index in its producer's batch.
__device__ __forceinline__ void issue_meta(int i, int kb, const Units& u, const SWork& wk,
                                           const KArgs& ka, const QArgs& qa, const Shared& sh,
                                           int64_t pos, uint32_t stage, uint32_t bar) {
  const int lane = threadIdx.x & 31;
  if (i < u.nk) {
    if (lane == 0) {
      const int32_t t0 = (u.k_lo + i) * kUnitRows;
      const int n = min(kUnitRows, wk.T - t0);
      const bool meta = wk.meta_bulk && n == kUnitRows;
      if (meta) {
        bulk_g2s(stage + kCoefOff, sh.pos + t0, kUnitRows * 8u, bar);
        bulk_g2s(stage + kSlotsOff, ka.slots + t0, kUnitRows * 8u, bar);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stage + kHdrOff),
                   "r"(((uint32_t)i << 2) | kUnitKey), "r"(t0), "r"(n),
                   "r"(meta ? kInStage : 0u)
                   : "memory");
      mbar_arrive_expect_tx(bar, meta ? 2u * kUnitRows * 8u : 0u);
    }
    return;
  }
  const int32_t row0 = (u.q_lo + i - u.nk) * kUnitRows;
  const int n = min(kUnitRows, wk.TH - row0);
  const int nsl = (n + kSliceRows - 1) / kSliceRows;
  const bool mine = lane / kSlices == kb;
  const int sl = lane % kSlices;
  const bool ok = pos >= 0 && pos < sh.max_pos;
  // One cos/sin pair per token: the slice that starts a token (or the
  // unit) copies it into token slot t - t(row0).
  const int32_t t_first = (int32_t)wk.hdiv.div((uint32_t)row0);
  const int32_t rsl = row0 + kSliceRows * sl;
  const int32_t tsl = (int32_t)wk.hdiv.div((uint32_t)rsl);
  if (mine && sl < nsl && (sl == 0 || rsl == tsl * wk.H)) {
    const int64_t prow = ok ? pos : 0;
    const uint32_t dst = stage + kCoefOff + 256u * (uint32_t)(tsl - t_first);
    bulk_g2s(dst, sh.cos + prow * kRopeHalf, 128u, bar);
    bulk_g2s(dst + 128u, sh.sin + prow * kRopeHalf, 128u, bar);
  }
  const uint32_t okbits =
      (__ballot_sync(kFull, mine && ok) >> (kSlices * kb)) & ((1u << kSlices) - 1u);
  if (lane == 0) {
    const int32_t ntok =
        (int32_t)wk.hdiv.div((uint32_t)(row0 + kSliceRows * (nsl - 1))) - t_first + 1;
    const bool wst = wk.w_bulk && n == kUnitRows;
    if (wst) bulk_g2s(stage + kWOff, qa.w + row0, kUnitRows * 2u, bar);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stage + kHdrOff),
                 "r"(((uint32_t)i << 2) | kUnitQuery), "r"(row0), "r"(n),
                 "r"(okbits | (wst ? kInStage : 0u))
                 : "memory");
    mbar_arrive_expect_tx(bar, (uint32_t)ntok * 256u + (wst ? kUnitRows * 2u : 0u));
  }
}

// ------------------------------------------------------------------ kernel
template <int kStyle, bool kRotate, bool kFp8>
__global__ void __launch_bounds__(kThreadsS, 1)
    stream_kernel(KArgs ka, QArgs qa, Shared sh, SWork wk) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStagesS], empty[kStagesS];
  __shared__ int abort_flag, next_slice;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Units u;
  u.k_lo = (int32_t)((int64_t)blockIdx.x * wk.nk / gridDim.x);
  u.nk = (int32_t)((int64_t)(blockIdx.x + 1) * wk.nk / gridDim.x) - u.k_lo;
  u.q_lo = (int32_t)((int64_t)blockIdx.x * wk.nq / gridDim.x);
  u.nq = (int32_t)((int64_t)(blockIdx.x + 1) * wk.nq / gridDim.x) - u.q_lo;
  const uint32_t ring = smem_addr(smem);
  const uint32_t full0 = smem_addr(&full[0]), empty0 = smem_addr(&empty[0]);
  // The producers' first position lookups go out before anything else: the
  // cos/sin copies of the first units depend on them, and once the row
  // copies of every SM are queued a load waits behind all of them.
  int64_t pos_first = 0;
  if (warp >= kConsumers) pos_first = slice_pos(warp - kConsumers, 0, u, wk, sh);
  if (threadIdx.x == 0) {
    for (int s = 0; s < wk.stages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, kSlices);
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(ring + (uint32_t)s * kStageBytesS + kHdrOff),
                   "r"(kNoUnit)
                   : "memory");
    }
    abort_flag = 0;
    next_slice = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int n_units = u.total();
  const int S = wk.stages;

  if (warp >= kConsumers) {
    // ---------------- producers: producer p issues units p, p + kProducers, ...
    const int p = warp - kConsumers;
    const int n_own = n_units > p ? (n_units - p + kProducers - 1) / kProducers : 0;
    int issued = 0;  // own units issued
    int64_t pos_cur = pos_first, pos_next = 0;
    // On a long share the first own unit's rows go out at once; every other
    // unit's rows go out together with its metadata.  The first metadata
    // waits for the positions and should not queue behind a ring of rows; on
    // a short share (a prefill-sized step) not even behind one unit's rows
    // (T=8192: 36.0 against 36.4 us; T=65536 keeps the early rows, 0.6%).
    // (testing hook, see fp4idx_test_withhold_next: a withheld unit's copies
    // and arrival are skipped, so the waits for it run out)
    const int held = blockIdx.x == 0 ? wk.withhold : -1;
    const int rows_first = n_own > kShortShare ? 1 : 0;  // own units whose rows go out first
    if (rows_first && p != held)
      issue_rows(p, u, wk, ka, qa, ring + (uint32_t)p * kStageBytesS, full0 + 8u * p);
    for (int m = 0; m < n_own; ++m) {
      if (m % kBatch == 0) {
        if (m > 0) pos_cur = pos_next;
        pos_next = slice_pos(p, m + kBatch, u, wk, sh);
      }
      const int i = p + kProducers * m;
      const uint32_t ph = stage_uses(i, wk);
      const int s = i - (int)ph * S;
      const uint32_t stage = ring + (uint32_t)s * kStageBytesS, bar = full0 + 8u * s;
      if (ph > 0) {
        if (!wait_or_abort(empty0 + 8u * s, (ph - 1) & 1u, &abort_flag)) {
          if (lane == 0) {
            flag_error(sh.err, FP4IDX_ERRFLAG_TIMEOUT);
            abort_flag = 1;
          }
          break;
        }
      }
      if (m >= rows_first && i != held) issue_rows(i, u, wk, ka, qa, stage, bar);
      if (i != held) issue_meta(i, m % kBatch, u, wk, ka, qa, sh, pos_cur, stage, bar);
      issued = m + 1;
    }
    __syncwarp();
    // Drain: the last phase of each own stage that was used must complete
    // before the CTA's shared memory is released (bounded).  Every unit whose
    // rows were issued also had its metadata issued: the loop can stop only
    // at an empty-stage wait, which precedes both.
    // The drain ignores the abort flag: only the time limit ends it.
    __syncthreads();
    const int no_abort = 0;
    for (int m = max(issued - S / kProducers, 0); m < issued; ++m) {
      const int i = p + kProducers * m;
      const uint32_t ph = stage_uses(i, wk);
      wait_or_abort(full0 + 8u * (uint32_t)(i - (int)ph * S), ph & 1u, &no_abort);
    }
    return;
  }

  // ---------------- consumers: slices (unit i, slice sl) claimed in order
  for (;;) {
    int k = 0;
    if (lane == 0) k = atomicAdd(&next_slice, 1);
    k = __shfl_sync(kFull, k, 0);
    const int i = k / kSlices, sl = k % kSlices;
    if (i >= n_units) break;
    const uint32_t ph = stage_uses(i, wk);
    const int s = i - (int)ph * wk.stages;
    const uint32_t stage = ring + (uint32_t)s * kStageBytesS;
    if (!wait_unit(stage, full0 + 8u * s, i, wk, &abort_flag)) {
      if (lane == 0) {
        flag_error(sh.err, FP4IDX_ERRFLAG_TIMEOUT);
        abort_flag = 1;
      }
      break;
    }
    uint32_t hdr[4];
    lds128(stage + kHdrOff, hdr);
    if ((hdr[0] & 3u) == kUnitKey)
      key_slice<kStyle, kRotate, kFp8>(stage, (int32_t)hdr[1], (int)hdr[2], hdr[3], sl, ka, sh);
    else
      query_slice<kStyle, kRotate, kFp8>(stage, (int32_t)hdr[1], (int)hdr[2], hdr[3], sl, wk, qa, sh);
    __syncwarp();
    // (the stage's index again from its address: one register fewer live
    // across the slice, which one variant would otherwise spill)
    if (lane == 0) mbar_arrive(empty0 + 8u * ((stage - ring) / (uint32_t)kStageBytesS));
  }
  __syncthreads();
}

// --------------------------------------------------------------- host side
constexpr int kMaxDevicesS = 64;
// 0: not set up yet (a failed set-up is retried); published with release
// once the kernel attributes are set, under g_sms_mutex
std::atomic<int> g_sms[kMaxDevicesS];
std::mutex g_sms_mutex;

template <int kStyle, bool kRotate, bool kFp8>
bool setup_stream() {
  auto kern = stream_kernel<kStyle, kRotate, kFp8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemS) !=
      cudaSuccess)
    return false;
  int n = 0;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreadsS, kSmemS) ==
             cudaSuccess &&
         n >= 1;
}

template <int kStyle>
bool setup_style() {
  return setup_stream<kStyle, false, false>() && setup_stream<kStyle, false, true>() &&
         setup_stream<kStyle, true, false>() && setup_stream<kStyle, true, true>();
}

// The kernel for (rotate, fp8); returns the launch's own status.
template <int kStyle>
cudaError_t launch_style(unsigned grid, cudaStream_t s, const KArgs& ka, const QArgs& qa,
                         const Shared& sh, const SWork& wk, int rotate, int fp8) {
  auto kern = !rotate && !fp8 ? stream_kernel<kStyle, false, false>
              : !rotate       ? stream_kernel<kStyle, false, true>
              : !fp8          ? stream_kernel<kStyle, true, false>
                              : stream_kernel<kStyle, true, true>;
  return launch_kernel(kern, grid, kThreadsS, (unsigned)(wk.stages * kStageBytesS), s, ka, qa,
                       sh, wk);
}

// Testing hook: the unit of CTA 0 whose copies the next launch withholds
// (-1: none), taken once.
std::atomic<int64_t> g_stream_withhold{-1};

int stream_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesS) return 0;
  const int known = g_sms[dev].load(std::memory_order_acquire);
  if (known != 0) return known;
  std::lock_guard<std::mutex> lock(g_sms_mutex);
  if (g_sms[dev].load(std::memory_order_relaxed) == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        !setup_style<FP4IDX_ROPE_NEOX>() || !setup_style<FP4IDX_ROPE_INTERLEAVED>())
      return 0;
    g_sms[dev].store(sms, std::memory_order_release);
  }
  return g_sms[dev].load(std::memory_order_relaxed);
}

}  // namespace

void stream_withhold_next(int64_t index) { g_stream_withhold.store(index); }

bool stream_eligible(bool queries, int64_t H) { return !queries || H % kSliceRows == 0; }

fp4idx_status launch_stream(const KArgs& ka, const QArgs& qa, const Shared& sh, bool keys,
                            bool queries, int rope_style, int rotate, int fp8, void* stream) {
  const int64_t H = queries ? qa.H : 0;
  if (sh.T >= (1 << 30) || H >= (1 << 30) || sh.T * H >= (1 << 30)) return FP4IDX_ERR_SHAPE;
  SWork wk;
  wk.T = (int32_t)sh.T;
  wk.H = queries ? (int32_t)H : 1;
  wk.TH = (int32_t)(sh.T * H);
  wk.nk = keys ? (wk.T + kUnitRows - 1) / kUnitRows : 0;
  wk.nq = queries ? (wk.TH + kUnitRows - 1) / kUnitRows : 0;
  wk.hdiv = make_fastdiv((uint32_t)wk.H);
  wk.q_mode = !queries || qa.q_hstride != FP4IDX_HEAD_DIM         ? 2
              : qa.q_tstride == (int64_t)H * FP4IDX_HEAD_DIM ? 0
                                                             : 1;
  wk.k_contig = keys && ka.k_stride == FP4IDX_HEAD_DIM ? 1 : 0;
  wk.w_bulk = queries && qa.w_tstride == H && (reinterpret_cast<uintptr_t>(qa.w) % 16) == 0;
  wk.meta_bulk = keys && (reinterpret_cast<uintptr_t>(sh.pos) % 16) == 0 &&
                 (reinterpret_cast<uintptr_t>(ka.slots) % 16) == 0;
  {
    const int64_t w = g_stream_withhold.exchange(-1);
    wk.withhold = w >= 0 && w < (1ll << 30) ? (int32_t)w : -1;
  }
  const int64_t total = (int64_t)wk.nk + wk.nq;
  if (total == 0) return FP4IDX_OK;
  const int sms = stream_sms();
  if (sms <= 0) return FP4IDX_ERR_CUDA;
  const unsigned grid = (unsigned)(total < sms ? total : sms);
  // the largest producer share of this launch decides the ring depth
  const int64_t per_cta = (total + grid - 1) / grid;
  wk.stages = (per_cta + kProducers - 1) / kProducers <= kShallowShare ? kShortStages : kStagesS;
  wk.smul = (uint32_t)(((1ull << 32) + (uint64_t)wk.stages - 1) / (uint64_t)wk.stages);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      rope_style == FP4IDX_ROPE_NEOX
          ? launch_style<FP4IDX_ROPE_NEOX>(grid, s, ka, qa, sh, wk, rotate, fp8)
          : launch_style<FP4IDX_ROPE_INTERLEAVED>(grid, s, ka, qa, sh, wk, rotate, fp8);
  return e == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}

}  // namespace fp4idx_impl
