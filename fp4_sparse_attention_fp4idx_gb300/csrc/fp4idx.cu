// fp4idx.cu -- CUDA kernels (sm_103a) and C ABI of the fused FP4 indexer
// pre-pass.  The operation, its numerics and the argument contract are
// described in include/fp4idx.h.
//
// Sources (web pages, by title and section):
//   "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656): Summary (key op
//   = RMSNorm + RoPE + both quantisation stages + paged store; query op =
//   RoPE + quantisation + head weights in one launch), review (packed -0
//   clearing, UE8M0 exponent of ceil_pow2(amax/6) with a post-divide floor,
//   exact inverse scale).
//   "[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR
//   5484): API (geometry, q_out layout, plain weights), One deliberate
//   deviation (round half to even at midpoints).
//
// ---------------------------------------------------------------- design
// Routing: this file's pre-pass kernel (prepass_kernel) serves query calls
// whose head count is not a multiple of 16; every other launch runs the
// streaming kernel of fp4idx_stream.cu, which performs the same operations
// in the same order (shared helpers in fp4idx_common.cuh).
//
// The pass is HBM-bound (about 2.6 bytes moved per element and a few dozen
// integer/fp32 operations), so the kernel is organised around two limits:
// bytes in flight and issue slots per element.
//
// Data movement: one persistent grid of 24-warp CTAs; the warps of a CTA
// claim work items from shared counters, each warp with a private ring of
// kStages shared-memory stages.  A work item is a chunk of up to kChunkRows
// (16) rows of 128 bf16 (4 KB): up to 16 heads of one query token, or the key
// rows of 16 consecutive tokens.  Lane 0 of the warp fetches items
// kStages ahead with cp.async.bulk (the Blackwell bulk-copy engine), together
// with the query token's cos/sin rows, and an mbarrier per stage counts the
// bytes in.  So the bytes in flight cost no registers and no load
// instructions, and the warp only computes.
//
// Compute layout: 8 lanes own a row.  Lane j holds dims 8j..8j+7 (the RoPE
// half) AND dims 64+8j..64+8j+7 (the pass-through half) as two 16-byte words,
// so every lane does the same RoPE work (no idle lanes), and every lane sits
// in two 32-element quantisation groups: group j/4 (dims 0..63) and group
// 2+j/4 (dims 64..127).  The two group maxima travel as one packed bf16x2
// word, so both reductions take two shuffles.  A warp works on 4 rows at a
// time.
//
// Bit-exactness: fp32 steps use explicit round-to-nearest operations (scalar
// intrinsics or packed f32x2 .rn instructions), which are never fused into
// FMA; subnormals are kept (no FTZ anywhere).
//
// Quantisation in closed form (derived from the two-stage definition):
//   * stage-1 exponent: for a bf16 amax with bits h = E<<7 | m (E biased),
//     ceil_pow2(amax/6) is 2^(E-129) if m <= 64 (1.m <= 1.5) and 2^(E-128)
//     otherwise; amax/6 rounded to fp32 never crosses a power of two for a
//     bf16 amax.  So e1 = max(((h + 63) >> 7) - 2, 1), no division.
//   * stage-1 codes: the hardware e2m1x2 conversion rounds to nearest even
//     and saturates, i.e. exactly the grid rule (it may emit -0 codes, which
//     are cleared at the end).
//   * stage 2: with e1 > 1 the group's largest scaled value is 1.m * 4 (m <=
//     64, code 6 or 7) or 1.m * 2 (m > 64); it lands on code 5 (3.0) exactly
//     when 64 < m < 96.  Then stage 2 halves the scale (e2 = e1 - 1) and each
//     code m <= 5 becomes the code of 2*grid[m], i.e. m + min(m, 2);
//     otherwise (and always when e1 == 1, where the floor holds) stage 2
//     reproduces stage 1.

#include <atomic>
#include <mutex>

#include "fp4idx_common.cuh"

namespace {

// Build-time tuning knobs (rows per work item, ring depth, CTAs per SM).
#ifndef FP4IDX_CHUNK_ROWS
#define FP4IDX_CHUNK_ROWS 16
#endif
#ifndef FP4IDX_STAGES
#define FP4IDX_STAGES 2
#endif
#ifndef FP4IDX_MIN_BLOCKS
#define FP4IDX_MIN_BLOCKS 1
#endif
#ifndef FP4IDX_WARPS
#define FP4IDX_WARPS 24
#endif

using namespace fp4idx_impl;

constexpr int kWarps = FP4IDX_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kChunkRows = FP4IDX_CHUNK_ROWS;  // rows per work item (multiple of 4)
constexpr int kStages = FP4IDX_STAGES;
constexpr int kStageCos = kChunkRows * kRowBytes;  // 32 fp32 cos values (query item)
constexpr int kStageSin = kStageCos + 128;         // 32 fp32 sin values (query item)
constexpr int kStageHdr = kStageSin + 128;         // 4-byte header
constexpr int kStageBytes = kStageHdr + 16;        // 16-byte multiple
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kSmemBytes = kWarps * kRingBytes;
constexpr int kMinBlocksPerSm = FP4IDX_MIN_BLOCKS;
static_assert(kChunkRows % 4 == 0 && kChunkRows <= 16, "chunk rows: multiple of 4, at most 16");
// A key item reuses the cos/sin area for its tokens' positions and slots.
static_assert(kChunkRows * 8 <= 128, "positions/slots of a key item must fit in 128 bytes");


// Stage-2 fix-up of eight stage-1 nibbles: if `halve`, every magnitude m
// (m <= 5) becomes m + min(m, 2); then sign bits survive only on non-zero
// magnitudes (no -0 codes).
__device__ __forceinline__ uint32_t finish_codes(uint32_t p, bool halve) {
  const uint32_t ge2 = ((p >> 1) | (p >> 2)) & 0x11111111u;  // magnitude >= 2
  const uint32_t b0 = p & 0x11111111u;                        // magnitude bit 0
  uint32_t mag = p & 0x77777777u;
  if (halve) mag += (ge2 << 1) | (b0 & ~ge2);
  return (p & ((ge2 | b0) << 3)) | mag;
}

// Both stages for this lane's two 8-element parts: a = its slice of group
// j/4 (dims 8j..8j+7), b = its slice of group 2+j/4 (dims 64+8j..).  All 32
// lanes must call (shuffles).  Returns the two payload words and the row's
// exponent word (valid in lanes 0 and 4 of each 8-lane row group).
// The two groups' exponent arithmetic runs packed, one group per 16 bits.
__device__ __forceinline__ void quant_lane(const uint32_t (&a)[4], const uint32_t (&b)[4], int j,
                                           uint32_t& pa, uint32_t& pb, uint32_t& ew) {
  const uint32_t ma = hmax_abs(hmax_abs(a[0], a[1]), hmax_abs(a[2], a[3]));
  const uint32_t mb = hmax_abs(hmax_abs(b[0], b[1]), hmax_abs(b[2], b[3]));
  uint32_t m = hmax_abs(prmt(ma, mb, 0x5410u), prmt(ma, mb, 0x7632u));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 1));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 2));
  m &= 0x7fff7fffu;  // bf16 amax bits h of (group a, group b)

  // Per half: E' = (h + 63) >> 7 is e1 + 2 before the floor, so
  // 254 - e1 = min(256 - E', 253); it is the biased exponent of 2^(127-e1).
  const uint32_t ep = ((m + 0x003f003fu) >> 7) & 0x01ff01ffu;
  const uint32_t ie = umin16x2(0x01000100u - ep, 0x00fd00fdu);
  const float ia = __uint_as_float(ie << 23);
  const float ib = __uint_as_float((ie >> 16) << 23);
  // Stage 2 halves the scale when e1 > 1 (254 - e1 < 253) and the amax
  // mantissa lies in (64, 96), i.e. the top stage-1 code is 5.
  const uint32_t mq = uadd16x2(m & 0x007f007fu, 0xffbfffbfu);  // mantissa - 65
  const bool ha2 = (mq & 0xffffu) < 31u && (ie & 0xffffu) < 253u;
  const bool hb2 = (mq >> 16) < 31u && (ie >> 16) < 253u;

  float va[8], vb[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mul2(va[2 * k], va[2 * k + 1], bf16_lo(a[k]), bf16_hi(a[k]), ia, ia);
    mul2(vb[2 * k], vb[2 * k + 1], bf16_lo(b[k]), bf16_hi(b[k]), ib, ib);
  }
  pa = finish_codes(e2m1x8(va), ha2);
  pb = finish_codes(e2m1x8(vb), hb2);
  // e2 = e1 - halve, one group per 16 bits (each fits in a byte).
  const uint32_t e2 = 0x00fe00feu - ie - (ha2 ? 1u : 0u) - (hb2 ? 0x10000u : 0u);
  const uint32_t x = e2 << (8 * (j >> 2));
  ew = x | __shfl_xor_sync(kFull, x, 4);
}

// FP8 mode for this lane's two 8-element parts of its row (a = dims
// 8j..8j+7, b = dims 64+8j..64+8j+7).  All 32 lanes must call (shuffles).
// The row's scale is 2^(e-127) = ceil_pow2(max(rn(amax/448), 2^-126)); the
// codes are E4M3 of x * 2^(127-e) (an exact product).  Returns the codes of
// a and b (8 bytes each) and e.
__device__ __forceinline__ void quant_lane_fp8(const uint32_t (&a)[4], const uint32_t (&b)[4],
                                               uint2& ca, uint2& cb, uint32_t& e) {
  uint32_t m = hmax_abs(hmax_abs(hmax_abs(a[0], a[1]), hmax_abs(a[2], a[3])),
                        hmax_abs(hmax_abs(b[0], b[1]), hmax_abs(b[2], b[3])));
  m = hmax_abs(m, prmt(m, m, 0x1032u));  // both halves
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 1));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 2));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 4));
  const float amax = __uint_as_float((m & 0x7fffu) << 16);
  const float t = fmaxf(__fdiv_rn(amax, 448.0f), 1.17549435082228750797e-38f);
  const uint32_t tb = __float_as_uint(t);
  e = (tb >> 23) + ((tb & 0x7fffffu) != 0u ? 1u : 0u);  // 1 .. 248 for finite bf16
  const float inv = __uint_as_float((254u - e) << 23);  // 2^(127-e), a normal float
  float va[8], vb[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mul2(va[2 * k], va[2 * k + 1], bf16_lo(a[k]), bf16_hi(a[k]), inv, inv);
    mul2(vb[2 * k], vb[2 * k + 1], bf16_lo(b[k]), bf16_hi(b[k]), inv, inv);
  }
  ca = make_uint2(e4m3x4(va[0], va[1], va[2], va[3]), e4m3x4(va[4], va[5], va[6], va[7]));
  cb = make_uint2(e4m3x4(vb[0], vb[1], vb[2], vb[3]), e4m3x4(vb[4], vb[5], vb[6], vb[7]));
}

// RoPE coefficients of lane j for one position, as fp32 pairs.
//   NeoX: lane j owns dims 8j..8j+7, pair index i = 8(j&3)+k; lanes 0..3
//   hold the first member of each pair and use -sin, so every lane computes
//   own*cos + partner*sin'.
//   Interleaved: word k of lane j is the pair i = 4j+k; c = (cos_i, cos_i),
//   s = (-sin_i, sin_i) so that (a, b)*c + (b, a)*s = (a', b').
template <int kStyle>
struct RopeCoef {
  float c[8];
  float s[8];
  __device__ __forceinline__ void set(const float4& c0, const float4& c1, const float4& s0,
                                      const float4& s1, int j) {
    if (kStyle == FP4IDX_ROPE_NEOX) {
      const float sg = j < 4 ? -1.0f : 1.0f;
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
      s[0] = sg * s0.x; s[1] = sg * s0.y; s[2] = sg * s0.z; s[3] = sg * s0.w;
      s[4] = sg * s1.x; s[5] = sg * s1.y; s[6] = sg * s1.z; s[7] = sg * s1.w;
    } else {
      c[0] = c0.x; c[1] = c0.x; c[2] = c0.y; c[3] = c0.y;
      c[4] = c0.z; c[5] = c0.z; c[6] = c0.w; c[7] = c0.w;
      s[0] = -s0.x; s[1] = s0.x; s[2] = -s0.y; s[3] = s0.y;
      s[4] = -s0.z; s[5] = s0.z; s[6] = -s0.w; s[7] = s0.w;
    }
  }
  // From a cos/sin row pair in shared memory.
  __device__ __forceinline__ void load_smem(uint32_t cos_row, uint32_t sin_row, int j) {
    if (kStyle == FP4IDX_ROPE_NEOX) {
      const uint32_t off = 32u * (uint32_t)(j & 3);
      set(lds_f4(cos_row + off), lds_f4(cos_row + off + 16), lds_f4(sin_row + off),
          lds_f4(sin_row + off + 16), j);
    } else {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      set(lds_f4(cos_row + 16u * j), z, lds_f4(sin_row + 16u * j), z, j);
    }
  }
  // From the global cos/sin tables.
  __device__ __forceinline__ void load_global(const float* cos_row, const float* sin_row, int j) {
    if (kStyle == FP4IDX_ROPE_NEOX) {
      const int off = 8 * (j & 3);
      set(ld_f4(cos_row + off), ld_f4(cos_row + off + 4), ld_f4(sin_row + off),
          ld_f4(sin_row + off + 4), j);
    } else {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      set(ld_f4(cos_row + 4 * j), z, ld_f4(sin_row + 4 * j), z, j);
    }
  }
};

// In-place RoPE of the lane's RoPE-half word group `a`.  All 32 lanes must
// call (the NeoX partner exchange is a shuffle).  Each result is
// rn(rn(x*c) + rn(y*s')): the products come from prod2 (exactly rounded,
// never fused with the sum), then one rounded packed addition.
template <int kStyle>
__device__ __forceinline__ void rope_lane(uint32_t (&a)[4], const RopeCoef<kStyle>& rc, float z) {
  if (kStyle == FP4IDX_ROPE_NEOX) {
    uint32_t p[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = __shfl_xor_sync(kFull, a[k], 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float m0, m1, n0, n1, r0, r1;
      prod2(m0, m1, bf16_lo(a[k]), bf16_hi(a[k]), rc.c[2 * k], rc.c[2 * k + 1], z);
      prod2(n0, n1, bf16_lo(p[k]), bf16_hi(p[k]), rc.s[2 * k], rc.s[2 * k + 1], z);
      sum2(r0, r1, m0, m1, n0, n1);
      a[k] = pack_bf16x2(r0, r1);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float x0 = bf16_lo(a[k]), x1 = bf16_hi(a[k]);
      float m0, m1, n0, n1, r0, r1;
      prod2(m0, m1, x0, x1, rc.c[2 * k], rc.c[2 * k + 1], z);
      prod2(n0, n1, x1, x0, rc.s[2 * k], rc.s[2 * k + 1], z);
      sum2(r0, r1, m0, m1, n0, n1);
      a[k] = pack_bf16x2(r0, r1);
    }
  }
}

// Normalised 128-point Walsh-Hadamard rotation of the row held by the 8
// lanes of a row group (lane j: a = dims 8j..8j+7, b = dims 64+8j..64+8j+7).
// Butterfly stages h = 1, 2, 4 stay inside a lane's 8-element runs, h = 8,
// 16, 32 pair lane j with lane j ^ (h/8), h = 64 pairs a with b; each
// butterfly turns (lower, upper) into (rn(lower + upper), rn(lower - upper)).
// Then one product with rn32(1/sqrt(128)) and the bf16 rounding.  All 32
// lanes must call (shuffles).
__device__ __forceinline__ void hadamard_lane(uint32_t (&a)[4], uint32_t (&b)[4], int j) {
  float x[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = bf16_lo(a[k]);
    x[2 * k + 1] = bf16_hi(a[k]);
    x[8 + 2 * k] = bf16_lo(b[k]);
    x[8 + 2 * k + 1] = bf16_hi(b[k]);
  }
#pragma unroll
  for (int h = 1; h < 8; h *= 2)
#pragma unroll
    for (int run = 0; run < 16; run += 8)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (!(i & h)) {
          const float u = x[run + i], v = x[run + i + h];
          x[run + i] = __fadd_rn(u, v);
          x[run + i + h] = __fsub_rn(u, v);
        }
#pragma unroll
  for (int m = 1; m < 8; m *= 2) {
    const bool upper = (j & m) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float other = __shfl_xor_sync(kFull, x[i], m);
      x[i] = upper ? __fsub_rn(other, x[i]) : __fadd_rn(x[i], other);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float u = x[i], v = x[8 + i];
    x[i] = __fadd_rn(u, v);
    x[8 + i] = __fsub_rn(u, v);
  }
  const float norm = 0.08838834764831845f;  // rn32(1/sqrt(128))
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a[k] = pack_bf16x2(__fmul_rn(x[2 * k], norm), __fmul_rn(x[2 * k + 1], norm));
    b[k] = pack_bf16x2(__fmul_rn(x[8 + 2 * k], norm), __fmul_rn(x[8 + 2 * k + 1], norm));
  }
}


// The work of one launch, in two item lists: key items (kChunkRows
// consecutive tokens each) and query items (token t, heads h0 .. h0 +
// kChunkRows - 1; cpt items per token).  Every CTA gets an equal slice of
// each list; inside a CTA the warps claim items one at a time from two
// shared-memory counters (key items first), so a warp that runs ahead
// simply takes more items.  All indices fit in 32 bits: the host rejects
// T * H >= 2^30, which no query tensor that fits in memory reaches.
struct Work {
  int32_t T, H;
  int32_t nk;   // key items
  int32_t nq;   // query items = T * cpt
  int32_t cpt;  // query items per token = ceil(H / kChunkRows)
  FastDiv cpt_div;
};

enum : uint32_t { kItemNone = 0, kItemKey = 1, kItemQuery = 2 };

// --------------------------------------------------------- producer side
// Lane 0's view of the items it will issue next: A is ready to issue (its
// token position was requested one step earlier), B is claimed.
struct Producer {
  uint32_t a_kind, b_kind;
  int32_t a_t, a_h0, b_idx;
  int64_t a_pos;
  bool k_done;

  __device__ __forceinline__ void claim(int32_t* sk, int32_t* sq, int32_t k_hi, int32_t q_hi) {
    if (!k_done) {
      const int32_t k = atomicAdd(sk, 1);
      if (k < k_hi) {
        b_kind = kItemKey;
        b_idx = k;
        return;
      }
      k_done = true;
    }
    const int32_t q = atomicAdd(sq, 1);
    b_kind = q < q_hi ? kItemQuery : kItemNone;
    b_idx = q;
  }
  // A <- B (decode it and request its position), then claim a new B.
  __device__ __forceinline__ void advance(const Work& wk, const Shared& sh, int32_t* sk,
                                          int32_t* sq, int32_t k_hi, int32_t q_hi) {
    a_kind = b_kind;
    if (a_kind == kItemKey) {
      a_t = b_idx * kChunkRows;
      a_h0 = 0;
    } else if (a_kind == kItemQuery) {
      a_t = (int32_t)wk.cpt_div.div((uint32_t)b_idx);
      a_h0 = (b_idx - a_t * wk.cpt) * kChunkRows;
      a_pos = __ldg(sh.pos + a_t);
    }
    if (a_kind != kItemNone) claim(sk, sq, k_hi, q_hi);
  }
};

// Issues item A into a stage: its header (kind, token, first head, position
// ok) and its bulk copies.  Lane 0 only.
__device__ __forceinline__ void issue_item(const Producer& pr, const Work& wk, const KArgs& ka,
                                           const QArgs& qa, const Shared& sh, uint32_t stage,
                                           uint32_t bar) {
  if (pr.a_kind == kItemKey) {
    const int n = min(wk.T - pr.a_t, kChunkRows);
    const bool meta = ka.meta_bulk && n == kChunkRows;
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(stage + kStageHdr), "r"(kItemKey),
                 "r"(pr.a_t)
                 : "memory");
    mbar_arrive_expect_tx(bar, (uint32_t)n * kRowBytes + (meta ? 2u * kChunkRows * 8u : 0u));
    const uint16_t* src = ka.k + (int64_t)pr.a_t * ka.k_stride;
    if (ka.k_stride == FP4IDX_HEAD_DIM) {
      bulk_g2s(stage, src, (uint32_t)n * kRowBytes, bar);
    } else {
      for (int r = 0; r < n; ++r)
        bulk_g2s(stage + (uint32_t)r * kRowBytes, src + r * ka.k_stride, kRowBytes, bar);
    }
    if (meta) {
      bulk_g2s(stage + kStageCos, sh.pos + pr.a_t, kChunkRows * 8u, bar);
      bulk_g2s(stage + kStageSin, ka.slots + pr.a_t, kChunkRows * 8u, bar);
    }
    return;
  }
  // Query item: the row copies go out before the token's position is
  // needed; the header and the arrive come last, so the consumer sees the
  // header once the phase completes.  An out-of-range position copies table
  // row 0 instead (the consumer skips the token).
  const int n = min(wk.H - pr.a_h0, kChunkRows);
  mbar_expect_tx(bar, (uint32_t)n * kRowBytes + 256u);
  const uint16_t* src = qa.q + (int64_t)pr.a_t * qa.q_tstride + (int64_t)pr.a_h0 * qa.q_hstride;
  if (qa.q_hstride == FP4IDX_HEAD_DIM) {
    bulk_g2s(stage, src, (uint32_t)n * kRowBytes, bar);
  } else {
    for (int r = 0; r < n; ++r)
      bulk_g2s(stage + (uint32_t)r * kRowBytes, src + r * qa.q_hstride, kRowBytes, bar);
  }
  const bool ok = pr.a_pos >= 0 && pr.a_pos < sh.max_pos;
  const int64_t row = ok ? pr.a_pos : 0;
  bulk_g2s(stage + kStageCos, sh.cos + row * kRopeHalf, 128u, bar);
  bulk_g2s(stage + kStageSin, sh.sin + row * kRopeHalf, 128u, bar);
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stage + kStageHdr),
               "r"(kItemQuery), "r"(pr.a_t), "r"(pr.a_h0), "r"(ok ? 1u : 0u)
               : "memory");
  mbar_arrive(bar);
}

// --------------------------------------------------------- consumer side
__device__ __forceinline__ int64_t lds_s64(uint32_t addr) {
  int64_t v;
  asm volatile("ld.shared.s64 %0, [%1];" : "=l"(v) : "r"(addr));
  return v;
}

// A query item: heads h0 .. h0 + kChunkRows - 1 of token t, rows in the
// stage; `ok` says whether the token's position was in range.
template <int kStyle, bool kRotate, bool kFp8>
__device__ __forceinline__ void query_chunk(int32_t t, int32_t h0, bool ok, const Work& wk,
                                            const QArgs& qa, const Shared& sh, uint32_t stage) {
  const int lane = threadIdx.x & 31, j = lane & 7, rg = lane >> 3;
  const int n = min(wk.H - h0, kChunkRows);
  if (!ok) {
    if (lane == 0) flag_error(sh.err, FP4IDX_ERRFLAG_POSITION);
    return;  // the whole token is skipped; uniform over the warp
  }
  const int32_t row0 = t * wk.H + h0;
  uint16_t wb = 0;
  if (lane < n) wb = __ldg(qa.w + (int64_t)t * qa.w_tstride + h0 + lane);

  RopeCoef<kStyle> rc;
  rc.load_smem(stage + kStageCos, stage + kStageSin, j);
  uint8_t* const out = qa.q_fp4 + (int64_t)row0 * kPayloadBytes + 4 * j;
  uint8_t* const scl = qa.q_scale + (int64_t)row0 * 4;
  const uint32_t rows = stage + 16u * j;
#pragma unroll
  for (int r0 = 0; r0 < kChunkRows; r0 += 4) {
    if (r0 >= n) break;  // uniform over the warp
    const int r = r0 + rg;
    uint32_t a[4], b[4];
    lds128(rows + (uint32_t)r * kRowBytes, a);
    lds128(rows + (uint32_t)r * kRowBytes + 128u, b);
    rope_lane<kStyle>(a, rc, sh.neg_zero);
    if constexpr (kRotate) hadamard_lane(a, b, j);
    if constexpr (kFp8) {
      // codes at q_out + row*128; the row's scale folded into its weight
      uint2 ca, cb;
      uint32_t e;
      quant_lane_fp8(a, b, ca, cb, e);
      const float wr = __uint_as_float((uint32_t)__shfl_sync(kFull, (uint32_t)wb, r) << 16);
      if (r < n) {
        uint8_t* q8 = qa.q_fp4 + (int64_t)(row0 + r) * FP4IDX_HEAD_DIM + 8 * j;
        *reinterpret_cast<uint2*>(q8) = ca;
        *reinterpret_cast<uint2*>(q8 + 64) = cb;
        if (j == 0)
          qa.weights[row0 + r] = __fmul_rn(__fmul_rn(wr, qa.wscale), __uint_as_float(e << 23));
      }
    } else {
      uint32_t pa, pb, ew;
      quant_lane(a, b, j, pa, pb, ew);
      if (r < n) {
        *reinterpret_cast<uint32_t*>(out + r * kPayloadBytes) = pa;
        *reinterpret_cast<uint32_t*>(out + r * kPayloadBytes + 32) = pb;
        if (j == 0) *reinterpret_cast<uint32_t*>(scl + 4 * r) = ew;
      }
    }
  }
  if (!kFp8 && lane < n)
    qa.weights[row0 + lane] = __fmul_rn(__uint_as_float((uint32_t)wb << 16), qa.wscale);
}

// Slot and position of one key row (r < n), validated; live = false for a
// skipped or out-of-range row (then pos = 0, a safe table row).
struct KeyMeta {
  int64_t slot, pos;
  bool live;
};

__device__ __forceinline__ KeyMeta key_meta(int32_t t0, const KArgs& ka, const Shared& sh,
                                            uint32_t stage, int r, int n, bool meta, int j) {
  KeyMeta m{-1, 0, false};
  if (r < n) {
    if (meta) {
      m.pos = lds_s64(stage + kStageCos + 8u * r);
      m.slot = lds_s64(stage + kStageSin + 8u * r);
    } else {
      m.pos = __ldg(sh.pos + t0 + r);
      m.slot = __ldg(ka.slots + t0 + r);
    }
    m.live = m.slot >= 0;
  }
  if (m.live) {
    const bool pos_ok = m.pos >= 0 && m.pos < sh.max_pos;
    const bool slot_ok = m.slot < ka.num_blocks * kKvBlock;
    if (!(pos_ok && slot_ok)) {
      if (j == 0)
        flag_error(sh.err, (pos_ok ? 0u : FP4IDX_ERRFLAG_POSITION) |
                               (slot_ok ? 0u : FP4IDX_ERRFLAG_SLOT));
      m.live = false;
    }
  }
  if (!m.live) m.pos = 0;
  m.pos &= ka.pos_mask;
  return m;
}

// A key item: tokens t0 .. t0 + kChunkRows - 1, rows in the stage.
template <int kStyle, bool kRotate, bool kFp8>
__device__ __forceinline__ void key_chunk(int32_t t0, const Work& wk, const KArgs& ka,
                                          const Shared& sh, uint32_t stage) {
  const int lane = threadIdx.x & 31, j = lane & 7, rg = lane >> 3;
  const int n = min(wk.T - t0, kChunkRows);
  const bool meta = ka.meta_bulk && n == kChunkRows;  // uniform
#pragma unroll 1
  for (int r0 = 0; r0 < n; r0 += 4) {  // uniform over the warp
    const int r = r0 + rg;
    const KeyMeta km = key_meta(t0, ka, sh, stage, r, n, meta, j);
    RopeCoef<kStyle> rc;
    rc.load_global(sh.cos + km.pos * kRopeHalf, sh.sin + km.pos * kRopeHalf, j);

    uint32_t a[4], b[4];
    const uint32_t rowaddr = stage + (uint32_t)r * kRowBytes + 16u * j;
    lds128(rowaddr, a);
    lds128(rowaddr + 128u, b);
    // RMSNorm.  Lane j holds the 8-element runs j and 8+j of the fixed
    // summation order; the butterfly's distance-8 step is the local add.
    float sa = __fmul_rn(bf16_lo(a[0]), bf16_lo(a[0]));
    float sb = __fmul_rn(bf16_lo(b[0]), bf16_lo(b[0]));
    sa = __fadd_rn(sa, __fmul_rn(bf16_hi(a[0]), bf16_hi(a[0])));
    sb = __fadd_rn(sb, __fmul_rn(bf16_hi(b[0]), bf16_hi(b[0])));
#pragma unroll
    for (int k = 1; k < 4; ++k) {
      sa = __fadd_rn(sa, __fmul_rn(bf16_lo(a[k]), bf16_lo(a[k])));
      sa = __fadd_rn(sa, __fmul_rn(bf16_hi(a[k]), bf16_hi(a[k])));
      sb = __fadd_rn(sb, __fmul_rn(bf16_lo(b[k]), bf16_lo(b[k])));
      sb = __fadd_rn(sb, __fmul_rn(bf16_hi(b[k]), bf16_hi(b[k])));
    }
    float ss = __fadd_rn(sa, sb);                       // distance 8
    ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 4));  // distance 4
    ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 2));  // distance 2
    ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 1));  // distance 1
    const float ms = __fmul_rn(ss, 0.0078125f);         // /128, exact scaling
    const float rr = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, ka.eps)));
    const uint4 ga = __ldg(reinterpret_cast<const uint4*>(ka.gamma) + j);
    const uint4 gb = __ldg(reinterpret_cast<const uint4*>(ka.gamma) + 8 + j);
    const uint32_t gwa[4] = {ga.x, ga.y, ga.z, ga.w}, gwb[4] = {gb.x, gb.y, gb.z, gb.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float u0, u1, y0, y1;
      mul2(u0, u1, bf16_lo(a[k]), bf16_hi(a[k]), rr, rr);
      mul2(y0, y1, u0, u1, bf16_lo(gwa[k]), bf16_hi(gwa[k]));
      a[k] = pack_bf16x2(y0, y1);
      mul2(u0, u1, bf16_lo(b[k]), bf16_hi(b[k]), rr, rr);
      mul2(y0, y1, u0, u1, bf16_lo(gwb[k]), bf16_hi(gwb[k]));
      b[k] = pack_bf16x2(y0, y1);
    }
    rope_lane<kStyle>(a, rc, sh.neg_zero);
    if constexpr (kRotate) hadamard_lane(a, b, j);
    if constexpr (kFp8) {
      uint2 ca, cb;
      uint32_t e;
      quant_lane_fp8(a, b, ca, cb, e);
      if (km.live) {
        uint8_t* page = ka.cache + (km.slot / kKvBlock) * (int64_t)kFp8PageBytes;
        const int64_t o = km.slot % kKvBlock;
        uint8_t* dst = page + o * FP4IDX_HEAD_DIM + 8 * j;
        *reinterpret_cast<uint2*>(dst) = ca;
        *reinterpret_cast<uint2*>(dst + 64) = cb;
        if (j == 0) *reinterpret_cast<uint32_t*>(page + kFp8ScaleOffset + 4 * o) = e << 23;
      }
      continue;
    }
    uint32_t pa, pb, ew;
    quant_lane(a, b, j, pa, pb, ew);
    if (km.live) {
      uint8_t* page = ka.cache + (km.slot / kKvBlock) * (int64_t)kPageBytes;
      const int64_t o = km.slot % kKvBlock;
      uint8_t* dst = page + o * kPayloadBytes + 4 * j;
      *reinterpret_cast<uint32_t*>(dst) = pa;
      *reinterpret_cast<uint32_t*>(dst + 32) = pb;
      if (j == 0) *reinterpret_cast<uint32_t*>(page + kExpOffset + 4 * o) = ew;
    }
  }
}

// ------------------------------------------------------------------ kernel
template <int kStyle, bool kRotate, bool kFp8>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm)
    prepass_kernel(KArgs ka, QArgs qa, Shared sh, Work wk) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps * kStages];
  __shared__ int32_t next_k, next_q;  // this CTA's claim counters
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t k_hi = (int32_t)((int64_t)(blockIdx.x + 1) * wk.nk / gridDim.x);
  const int32_t q_hi = (int32_t)((int64_t)(blockIdx.x + 1) * wk.nq / gridDim.x);
  if (threadIdx.x == 0) {
    next_k = (int32_t)((int64_t)blockIdx.x * wk.nk / gridDim.x);
    next_q = (int32_t)((int64_t)blockIdx.x * wk.nq / gridDim.x);
  }
  const uint32_t ring = smem_addr(smem) + (uint32_t)warp * kRingBytes;
  const uint32_t bar0 = smem_addr(&bars[warp * kStages]);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8u * s, 1);
    fence_mbar_init();
  }
  __syncthreads();

  Producer pr;  // meaningful in lane 0 only
  pr.k_done = false;
  pr.b_kind = kItemNone;
  if (lane == 0) {
    pr.claim(&next_k, &next_q, k_hi, q_hi);
    pr.advance(wk, sh, &next_k, &next_q, k_hi, q_hi);
  }
  uint32_t valid = 0;  // bit s: stage s holds an item
  for (int s = 0; s < kStages; ++s) {
    bool v = false;
    if (lane == 0 && pr.a_kind != kItemNone) {
      issue_item(pr, wk, ka, qa, sh, ring + s * kStageBytes, bar0 + 8u * s);
      pr.advance(wk, sh, &next_k, &next_q, k_hi, q_hi);
      v = true;
    }
    valid |= (uint32_t)__shfl_sync(kFull, v ? 1 : 0, 0) << s;
  }

  int s = 0;
  uint32_t phase = 0;
  while (valid & (1u << s)) {
    const uint32_t stage = ring + (uint32_t)s * kStageBytes;
    const uint32_t bar = bar0 + 8u * s;
    if (!mbar_wait_bounded(bar, phase)) {
      // Give up: report, then wait (bounded) for this warp's other copies so
      // none is still writing shared memory when the CTA exits.
      if (lane == 0) flag_error(sh.err, FP4IDX_ERRFLAG_TIMEOUT);
      for (int k = 1; k < kStages; ++k) {
        const int s2 = (s + k) % kStages;
        if (valid & (1u << s2)) mbar_wait_bounded(bar0 + 8u * s2, phase ^ (s + k >= kStages ? 1u : 0u));
      }
      return;
    }
    uint32_t hdr[4];
    lds128(stage + kStageHdr, hdr);
    if (hdr[0] == kItemKey)
      key_chunk<kStyle, kRotate, kFp8>((int32_t)hdr[1], wk, ka, sh, stage);
    else
      query_chunk<kStyle, kRotate, kFp8>((int32_t)hdr[1], (int32_t)hdr[2], hdr[3] != 0, wk, qa,
                                         sh, stage);
    __syncwarp();
    bool v = false;
    if (lane == 0 && pr.a_kind != kItemNone) {
      issue_item(pr, wk, ka, qa, sh, stage, bar);
      pr.advance(wk, sh, &next_k, &next_q, k_hi, q_hi);
      v = true;
    }
    valid = (valid & ~(1u << s)) | ((uint32_t)__shfl_sync(kFull, v ? 1 : 0, 0) << s);
    if (++s == kStages) {
      s = 0;
      phase ^= 1u;
    }
  }
}

// ----------------------------------------------------- torch-shaped fake quant
// RoPE then FP4 fake quantisation of bf16 rows, written back as the
// dequantised bf16 values.  Source: "dsv4.1: RoPE and FP4 packing kernels"
// (sglang PR 39656), Summary (the RoPE tail plus FP4 fake-quant of the
// torch-shaped path: per-32 UE8M0 by default, per-16 E4M3 for compressed
// KV; bf16 round trip after RoPE; round half to even).

struct FQArgs {
  const uint16_t* x;
  int64_t row_stride;       // elements
  uint32_t rows_per_token;
  uint32_t N;               // rows
  const int64_t* pos;
  const float* cos;
  const float* sin;
  int64_t max_pos;
  uint16_t* out;            // dense [N, 128]
  uint32_t* err;
  float neg_zero;
};

// Eight packed E2M1 codes (element 0 in the low nibble) -> fp32 values at
// scale 2^0, exactly, by the hardware E2M1 -> f16 conversion.
__device__ __forceinline__ void e2m1x8_values(uint32_t p, float (&v)[8]) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(p));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __half2float(__ushort_as_half((unsigned short)(h[k] & 0xffffu)));
    v[2 * k + 1] = __half2float(__ushort_as_half((unsigned short)(h[k] >> 16)));
  }
}

// fp32 -> E4M3 (round half to even, saturating) -> fp32, exactly.
__device__ __forceinline__ float e4m3_round(float t) {
  uint32_t h;
  asm("{\n\t.reg .b16 c;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c, %1, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h)
      : "f"(t));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// Dequantised values of eight codes times `scale` (an exact product),
// packed as four bf16x2 words.  Codes with a zero magnitude carry no sign.
__device__ __forceinline__ void dequant8(uint32_t p, float scale, uint32_t (&o)[4]) {
  float v[8];
  e2m1x8_values(finish_codes(p, false), v);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    o[k] = pack_bf16x2(__fmul_rn(v[2 * k], scale), __fmul_rn(v[2 * k + 1], scale));
}

// Per-32 UE8M0 (stage 1 of the pack) for this lane's two parts; all 32
// lanes must call (shuffles).
__device__ __forceinline__ void fake_quant_ue8m0(uint32_t (&a)[4], uint32_t (&b)[4]) {
  const uint32_t ma = hmax_abs(hmax_abs(a[0], a[1]), hmax_abs(a[2], a[3]));
  const uint32_t mb = hmax_abs(hmax_abs(b[0], b[1]), hmax_abs(b[2], b[3]));
  uint32_t m = hmax_abs(prmt(ma, mb, 0x5410u), prmt(ma, mb, 0x7632u));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 1));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 2));
  m &= 0x7fff7fffu;
  const uint32_t ep = ((m + 0x003f003fu) >> 7) & 0x01ff01ffu;
  const uint32_t ie = umin16x2(0x01000100u - ep, 0x00fd00fdu);  // 254 - e1 per half
  const float ia = __uint_as_float(ie << 23), ib = __uint_as_float((ie >> 16) << 23);
  const float sa = __uint_as_float((254u - (ie & 0xffffu)) << 23);  // 2^(e1 - 127)
  const float sb = __uint_as_float((254u - (ie >> 16)) << 23);
  float va[8], vb[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mul2(va[2 * k], va[2 * k + 1], bf16_lo(a[k]), bf16_hi(a[k]), ia, ia);
    mul2(vb[2 * k], vb[2 * k + 1], bf16_lo(b[k]), bf16_hi(b[k]), ib, ib);
  }
  dequant8(e2m1x8(va), sa, a);
  dequant8(e2m1x8(vb), sb, b);
}

// Per-16 E4M3: a group of 16 is lanes j and j^1 of one part; all 32 lanes
// must call (shuffles).
__device__ __forceinline__ void fake_quant_e4m3_16(uint32_t (&a)[4], uint32_t (&b)[4]) {
  const uint32_t ma = hmax_abs(hmax_abs(a[0], a[1]), hmax_abs(a[2], a[3]));
  const uint32_t mb = hmax_abs(hmax_abs(b[0], b[1]), hmax_abs(b[2], b[3]));
  uint32_t m = hmax_abs(prmt(ma, mb, 0x5410u), prmt(ma, mb, 0x7632u));
  m = hmax_abs(m, __shfl_xor_sync(kFull, m, 1));
  m &= 0x7fff7fffu;
  // rn(amax / 6) and rn(x / s) through the corrected reciprocal quotient
  // (exact for these operands: bf16 numerators, E4M3 or 6 divisors)
  constexpr float kSixth = 1.0f / 6.0f;
  const float sa = e4m3_round(div_rcp(__uint_as_float(m << 16), 6.0f, kSixth));
  const float sb = e4m3_round(div_rcp(__uint_as_float(m & 0xffff0000u), 6.0f, kSixth));
  // A zero scale takes a zero reciprocal: every quotient is then +-0 (finite
  // x), so the group is all zeros.
  const float ra = sa == 0.0f ? 0.0f : rcp_approx(sa), rb = sb == 0.0f ? 0.0f : rcp_approx(sb);
  float va[8], vb[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    div_rcp2(va[2 * k], va[2 * k + 1], bf16_lo(a[k]), bf16_hi(a[k]), sa, ra);
    div_rcp2(vb[2 * k], vb[2 * k + 1], bf16_lo(b[k]), bf16_hi(b[k]), sb, rb);
  }
  dequant8(e2m1x8(va), sa, a);
  dequant8(e2m1x8(vb), sb, b);
}

template <int kStyle, int kMode>
__global__ void __launch_bounds__(256) fake_quant_kernel(FQArgs fa) {
  const int lane = threadIdx.x & 31, j = lane & 7, rg = lane >> 3;
  const uint32_t nwarps = gridDim.x * (blockDim.x / 32);
  const uint32_t warp = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  for (uint32_t r0 = 4 * warp; r0 < fa.N; r0 += 4 * nwarps) {  // uniform over the warp
    const uint32_t row = r0 + rg;
    const bool in = row < fa.N;
    int64_t pos = 0;
    bool ok = false;
    if (in) {
      pos = __ldg(fa.pos + row / fa.rows_per_token);
      ok = pos >= 0 && pos < fa.max_pos;
      if (!ok && j == 0) flag_error(fa.err, FP4IDX_ERRFLAG_POSITION);
    }
    if (!ok) pos = 0;
    RopeCoef<kStyle> rc;
    rc.load_global(fa.cos + pos * kRopeHalf, fa.sin + pos * kRopeHalf, j);
    uint32_t a[4] = {0u, 0u, 0u, 0u}, b[4] = {0u, 0u, 0u, 0u};
    if (ok) {
      const uint4* src = reinterpret_cast<const uint4*>(fa.x + (int64_t)row * fa.row_stride);
      const uint4 va = __ldg(src + j), vb = __ldg(src + 8 + j);
      a[0] = va.x; a[1] = va.y; a[2] = va.z; a[3] = va.w;
      b[0] = vb.x; b[1] = vb.y; b[2] = vb.z; b[3] = vb.w;
    }
    rope_lane<kStyle>(a, rc, fa.neg_zero);
    if (kMode == FP4IDX_FAKE_QUANT_E4M3_16)
      fake_quant_e4m3_16(a, b);
    else
      fake_quant_ue8m0(a, b);
    if (ok) {
      uint4* dst = reinterpret_cast<uint4*>(fa.out + (int64_t)row * FP4IDX_HEAD_DIM);
      dst[j] = make_uint4(a[0], a[1], a[2], a[3]);
      dst[8 + j] = make_uint4(b[0], b[1], b[2], b[3]);
    }
  }
}

// --------------------------------------------------------------- host side
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  std::atomic<int> sm_count{0};     // published (release) after blocks_per_sm
  int blocks_per_sm[2][2][2] = {};  // [style][rotate][fp8]
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_setup_mutex;  // one thread sets a device up; the others wait

template <int kStyle, bool kRotate, bool kFp8>
int setup_kernel() {
  auto kern = prepass_kernel<kStyle, kRotate, kFp8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, kSmemBytes) !=
      cudaSuccess)
    return 0;
  return n;
}

// CTAs that fit on the device at once, cached per device; 0 on a CUDA error.
int resident_ctas(int style, int rotate, int fp8) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  DeviceInfo& di = g_devices[dev];
  if (di.sm_count.load(std::memory_order_acquire) == 0) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (di.sm_count.load(std::memory_order_relaxed) != 0)
      return di.sm_count.load(std::memory_order_relaxed) * di.blocks_per_sm[style][rotate][fp8];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    const int n[2][2][2] = {
        {{setup_kernel<FP4IDX_ROPE_NEOX, false, false>(),
          setup_kernel<FP4IDX_ROPE_NEOX, false, true>()},
         {setup_kernel<FP4IDX_ROPE_NEOX, true, false>(),
          setup_kernel<FP4IDX_ROPE_NEOX, true, true>()}},
        {{setup_kernel<FP4IDX_ROPE_INTERLEAVED, false, false>(),
          setup_kernel<FP4IDX_ROPE_INTERLEAVED, false, true>()},
         {setup_kernel<FP4IDX_ROPE_INTERLEAVED, true, false>(),
          setup_kernel<FP4IDX_ROPE_INTERLEAVED, true, true>()}}};
    for (int a = 0; a < 2; ++a)
      for (int b = 0; b < 2; ++b)
        for (int c = 0; c < 2; ++c) {
          if (n[a][b][c] < 1) return 0;
          di.blocks_per_sm[a][b][c] = n[a][b][c];
        }
    di.sm_count.store(sms, std::memory_order_release);
  }
  return di.sm_count.load(std::memory_order_acquire) * di.blocks_per_sm[style][rotate][fp8];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fp4idx_status check_shared(const int64_t* positions, const float* cos_cache,
                           const float* sin_cache, int64_t max_pos, int rope_style) {
  if (!positions || !cos_cache || !sin_cache) return FP4IDX_ERR_NULL;
  if (max_pos < 1 || max_pos > (INT64_MAX / 4) / kRopeHalf) return FP4IDX_ERR_SHAPE;
  if (rope_style != FP4IDX_ROPE_NEOX && rope_style != FP4IDX_ROPE_INTERLEAVED)
    return FP4IDX_ERR_ARG;
  if (!aligned(positions, 8) || !aligned(cos_cache, 16) || !aligned(sin_cache, 16))
    return FP4IDX_ERR_ALIGN;
  return FP4IDX_OK;
}

fp4idx_status check_keys(const void* k, int64_t k_stride, const void* gamma, float eps,
                         const int64_t* slots, const uint8_t* cache, int64_t num_blocks) {
  if (!k || !gamma || !slots || !cache) return FP4IDX_ERR_NULL;
  if (num_blocks < 1 || num_blocks > INT64_MAX / kFp8PageBytes) return FP4IDX_ERR_SHAPE;
  if (!(eps > 0.0f) || !isfinite(eps)) return FP4IDX_ERR_ARG;
  if (!aligned(k, 16) || (k_stride % 8) != 0 || !aligned(gamma, 16) || !aligned(slots, 8) ||
      !aligned(cache, 16))
    return FP4IDX_ERR_ALIGN;
  return FP4IDX_OK;
}

// q_scale is not written in the FP8 mode (fp8 != 0) and may be NULL there.
fp4idx_status check_queries(const void* q, int64_t q_tstride, int64_t q_hstride, const void* w,
                            float wscale, const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* weights, int64_t num_tokens, int64_t num_heads,
                            int fp8 = 0) {
  if (!q || !w || !q_fp4 || (!q_scale && !fp8) || !weights) return FP4IDX_ERR_NULL;
  if (num_heads < 1 ||
      num_heads > INT64_MAX / FP4IDX_HEAD_DIM / (num_tokens > 0 ? num_tokens : 1))
    return FP4IDX_ERR_SHAPE;
  if (!isfinite(wscale)) return FP4IDX_ERR_ARG;
  if (!aligned(q, 16) || (q_tstride % 8) != 0 || (q_hstride % 8) != 0 || !aligned(w, 2) ||
      !aligned(q_fp4, 16) || (!fp8 && !aligned(q_scale, 4)) || !aligned(weights, 4))
    return FP4IDX_ERR_ALIGN;
  return FP4IDX_OK;
}

template <int kStyle, bool kRotate, bool kFp8>
cudaError_t launch_one(unsigned grid, cudaStream_t s, const KArgs& ka, const QArgs& qa,
                       const Shared& sh, const Work& wk) {
  return launch_kernel(prepass_kernel<kStyle, kRotate, kFp8>, grid, kThreads, kSmemBytes, s, ka,
                       qa, sh, wk);
}

fp4idx_status launch(const KArgs& ka, const QArgs& qa, const Shared& sh, bool keys, bool queries,
                     int rope_style, int rotate, int fp8, void* stream) {
  if (stream_eligible(queries, qa.H))
    return launch_stream(ka, qa, sh, keys, queries, rope_style, rotate, fp8, stream);
  // 32-bit indices: T * H and T itself below 2^30.
  const int64_t H = queries ? qa.H : 1;
  if (sh.T >= (1 << 30) || H >= (1 << 30) || sh.T * H >= (1 << 30)) return FP4IDX_ERR_SHAPE;
  Work wk;
  wk.T = (int32_t)sh.T;
  wk.H = (int32_t)H;
  wk.cpt = (int32_t)((H + kChunkRows - 1) / kChunkRows);
  wk.cpt_div = make_fastdiv((uint32_t)wk.cpt);
  wk.nk = keys ? (wk.T + kChunkRows - 1) / kChunkRows : 0;
  wk.nq = queries ? wk.T * wk.cpt : 0;
  const int64_t total = (int64_t)wk.nk + wk.nq;
  const int64_t resident = resident_ctas(rope_style, rotate, fp8);
  if (resident <= 0) return FP4IDX_ERR_CUDA;
  const int64_t want = (total + kWarps - 1) / kWarps;  // at least one item per warp
  const int64_t grid = want < resident ? want : resident;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned g = (unsigned)grid;
  const int which = (rope_style == FP4IDX_ROPE_NEOX ? 0 : 4) + (rotate ? 2 : 0) + (fp8 ? 1 : 0);
  cudaError_t e;
  switch (which) {
    case 0: e = launch_one<FP4IDX_ROPE_NEOX, false, false>(g, s, ka, qa, sh, wk); break;
    case 1: e = launch_one<FP4IDX_ROPE_NEOX, false, true>(g, s, ka, qa, sh, wk); break;
    case 2: e = launch_one<FP4IDX_ROPE_NEOX, true, false>(g, s, ka, qa, sh, wk); break;
    case 3: e = launch_one<FP4IDX_ROPE_NEOX, true, true>(g, s, ka, qa, sh, wk); break;
    case 4: e = launch_one<FP4IDX_ROPE_INTERLEAVED, false, false>(g, s, ka, qa, sh, wk); break;
    case 5: e = launch_one<FP4IDX_ROPE_INTERLEAVED, false, true>(g, s, ka, qa, sh, wk); break;
    case 6: e = launch_one<FP4IDX_ROPE_INTERLEAVED, true, false>(g, s, ka, qa, sh, wk); break;
    default: e = launch_one<FP4IDX_ROPE_INTERLEAVED, true, true>(g, s, ka, qa, sh, wk); break;
  }
  return e == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}

// Options: NULL means the defaults (compress ratio 1, no rotation, FP4).
fp4idx_status check_options(const fp4idx_options* o, int64_t& pos_mask, int& rotate, int& fp8) {
  pos_mask = -1;
  rotate = 0;
  fp8 = 0;
  if (o == nullptr) return FP4IDX_OK;
  if (o->compress_ratio != 1 && o->compress_ratio != 2 && o->compress_ratio != 4)
    return FP4IDX_ERR_ARG;
  if (o->hadamard != 0 && o->hadamard != 1) return FP4IDX_ERR_ARG;
  if (o->output_mode != FP4IDX_OUTPUT_FP4 && o->output_mode != FP4IDX_OUTPUT_FP8)
    return FP4IDX_ERR_ARG;
  pos_mask = ~(int64_t)(o->compress_ratio - 1);
  rotate = o->hadamard;
  fp8 = o->output_mode == FP4IDX_OUTPUT_FP8 ? 1 : 0;
  return FP4IDX_OK;
}

}  // namespace

namespace fp4idx_impl {
fp4idx_status prepass_check(const void* k, int64_t k_token_stride, const void* gamma, float eps,
                            const int64_t* slot_mapping, const uint8_t* kv_cache,
                            int64_t num_blocks, const void* q, int64_t q_token_stride,
                            int64_t q_head_stride, const void* w, float weight_scale,
                            const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* weights_out, int64_t num_heads,
                            const int64_t* positions, const float* cos_cache,
                            const float* sin_cache, int64_t max_pos, int rope_style,
                            int64_t num_tokens, const uint32_t* err_flags, int fp8) {
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  st = check_keys(k, k_token_stride, gamma, eps, slot_mapping, kv_cache, num_blocks);
  if (st != FP4IDX_OK) return st;
  st = check_queries(q, q_token_stride, q_head_stride, w, weight_scale, q_fp4, q_scale,
                     weights_out, num_tokens, num_heads, fp8);
  if (st != FP4IDX_OK) return st;
  if (err_flags && !aligned(err_flags, 4)) return FP4IDX_ERR_ALIGN;
  return FP4IDX_OK;
}
}  // namespace fp4idx_impl

// ------------------------------------------------------------------- C ABI
extern "C" {

fp4idx_status fp4idx_k_norm_rope_pack_store_ex(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, const int64_t* slot_mapping, uint8_t* kv_cache,
    int64_t num_blocks, int64_t num_tokens, const fp4idx_options* options,
    uint32_t* err_flags, void* stream) {
  if (num_tokens < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  st = check_keys(k, k_token_stride, gamma, eps, slot_mapping, kv_cache, num_blocks);
  if (st != FP4IDX_OK) return st;
  int64_t pos_mask;
  int rotate, fp8;
  st = check_options(options, pos_mask, rotate, fp8);
  if (st != FP4IDX_OK) return st;
  if (err_flags && !aligned(err_flags, 4)) return FP4IDX_ERR_ALIGN;

  KArgs ka{static_cast<const uint16_t*>(k), k_token_stride, static_cast<const uint16_t*>(gamma),
           eps, slot_mapping, kv_cache, num_blocks,
           aligned(positions, 16) && aligned(slot_mapping, 16) ? 1 : 0, pos_mask};
  QArgs qa{};
  qa.H = 1;
  Shared sh{positions, cos_cache, sin_cache, max_pos, num_tokens, err_flags, -0.0f};
  return launch(ka, qa, sh, true, false, rope_style, rotate, fp8, stream);
}

fp4idx_status fp4idx_k_norm_rope_pack_store(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, const int64_t* slot_mapping, uint8_t* kv_cache,
    int64_t num_blocks, int64_t num_tokens, uint32_t* err_flags, void* stream) {
  return fp4idx_k_norm_rope_pack_store_ex(k, k_token_stride, gamma, eps, positions, cos_cache,
                                          sin_cache, max_pos, rope_style, slot_mapping, kv_cache,
                                          num_blocks, num_tokens, nullptr, err_flags, stream);
}

fp4idx_status fp4idx_q_rope_pack_weights_ex(
    const void* q, int64_t q_token_stride, int64_t q_head_stride, const void* w,
    int64_t w_token_stride, float weight_scale, const int64_t* positions,
    const float* cos_cache, const float* sin_cache, int64_t max_pos, int rope_style,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, int64_t num_tokens,
    int64_t num_heads, const fp4idx_options* options, uint32_t* err_flags, void* stream) {
  if (num_tokens < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  int64_t pos_mask;
  int rotate, fp8;
  st = check_options(options, pos_mask, rotate, fp8);
  if (st != FP4IDX_OK) return st;
  st = check_queries(q, q_token_stride, q_head_stride, w, weight_scale, q_fp4, q_scale,
                     weights_out, num_tokens, num_heads, fp8);
  if (st != FP4IDX_OK) return st;
  if (err_flags && !aligned(err_flags, 4)) return FP4IDX_ERR_ALIGN;

  KArgs ka{};
  ka.pos_mask = -1;
  QArgs qa{static_cast<const uint16_t*>(q), q_token_stride, q_head_stride,
           static_cast<const uint16_t*>(w), w_token_stride, weight_scale, q_fp4, q_scale,
           weights_out, num_heads};
  Shared sh{positions, cos_cache, sin_cache, max_pos, num_tokens, err_flags, -0.0f};
  return launch(ka, qa, sh, false, true, rope_style, rotate, fp8, stream);
}

fp4idx_status fp4idx_q_rope_pack_weights(
    const void* q, int64_t q_token_stride, int64_t q_head_stride, const void* w,
    int64_t w_token_stride, float weight_scale, const int64_t* positions,
    const float* cos_cache, const float* sin_cache, int64_t max_pos, int rope_style,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, int64_t num_tokens,
    int64_t num_heads, uint32_t* err_flags, void* stream) {
  return fp4idx_q_rope_pack_weights_ex(q, q_token_stride, q_head_stride, w, w_token_stride,
                                       weight_scale, positions, cos_cache, sin_cache, max_pos,
                                       rope_style, q_fp4, q_scale, weights_out, num_tokens,
                                       num_heads, nullptr, err_flags, stream);
}

fp4idx_status fp4idx_indexer_prepass_ex(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_blocks, const void* q,
    int64_t q_token_stride, int64_t q_head_stride, const void* w, int64_t w_token_stride,
    float weight_scale, uint8_t* q_fp4, uint8_t* q_scale, float* weights_out,
    int64_t num_heads, const int64_t* positions, const float* cos_cache,
    const float* sin_cache, int64_t max_pos, int rope_style, int64_t num_tokens,
    const fp4idx_options* options, uint32_t* err_flags, void* stream) {
  if (num_tokens < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  int64_t pos_mask;
  int rotate, fp8;
  fp4idx_status st = check_options(options, pos_mask, rotate, fp8);
  if (st != FP4IDX_OK) return st;
  st = prepass_check(k, k_token_stride, gamma, eps, slot_mapping, kv_cache, num_blocks, q,
                     q_token_stride, q_head_stride, w, weight_scale, q_fp4, q_scale,
                     weights_out, num_heads, positions, cos_cache, sin_cache, max_pos,
                     rope_style, num_tokens, err_flags, fp8);
  if (st != FP4IDX_OK) return st;

  KArgs ka{static_cast<const uint16_t*>(k), k_token_stride, static_cast<const uint16_t*>(gamma),
           eps, slot_mapping, kv_cache, num_blocks,
           aligned(positions, 16) && aligned(slot_mapping, 16) ? 1 : 0, pos_mask};
  QArgs qa{static_cast<const uint16_t*>(q), q_token_stride, q_head_stride,
           static_cast<const uint16_t*>(w), w_token_stride, weight_scale, q_fp4, q_scale,
           weights_out, num_heads};
  Shared sh{positions, cos_cache, sin_cache, max_pos, num_tokens, err_flags, -0.0f};
  return launch(ka, qa, sh, true, true, rope_style, rotate, fp8, stream);
}

fp4idx_status fp4idx_indexer_prepass(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_blocks, const void* q,
    int64_t q_token_stride, int64_t q_head_stride, const void* w, int64_t w_token_stride,
    float weight_scale, uint8_t* q_fp4, uint8_t* q_scale, float* weights_out,
    int64_t num_heads, const int64_t* positions, const float* cos_cache,
    const float* sin_cache, int64_t max_pos, int rope_style, int64_t num_tokens,
    uint32_t* err_flags, void* stream) {
  return fp4idx_indexer_prepass_ex(k, k_token_stride, gamma, eps, slot_mapping, kv_cache,
                                   num_blocks, q, q_token_stride, q_head_stride, w,
                                   w_token_stride, weight_scale, q_fp4, q_scale, weights_out,
                                   num_heads, positions, cos_cache, sin_cache, max_pos,
                                   rope_style, num_tokens, nullptr, err_flags, stream);
}

fp4idx_status fp4idx_rope_fake_quant(const void* x, int64_t row_stride, int64_t rows_per_token,
                                     const int64_t* positions, const float* cos_cache,
                                     const float* sin_cache, int64_t max_pos, int rope_style,
                                     int scale_mode, void* out, int64_t num_rows,
                                     uint32_t* err_flags, void* stream) {
  if (num_rows < 0) return FP4IDX_ERR_SHAPE;
  if (num_rows == 0) return FP4IDX_OK;
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  if (!x || !out) return FP4IDX_ERR_NULL;
  if (rows_per_token < 1 || num_rows >= (1ll << 31) || rows_per_token >= (1ll << 31) ||
      row_stride < FP4IDX_HEAD_DIM)
    return FP4IDX_ERR_SHAPE;
  if (scale_mode != FP4IDX_FAKE_QUANT_UE8M0_32 && scale_mode != FP4IDX_FAKE_QUANT_E4M3_16)
    return FP4IDX_ERR_ARG;
  if (!aligned(x, 16) || (row_stride % 8) != 0 || !aligned(out, 16) ||
      (err_flags && !aligned(err_flags, 4)))
    return FP4IDX_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FP4IDX_ERR_CUDA;
  FQArgs fa{static_cast<const uint16_t*>(x), row_stride, (uint32_t)rows_per_token,
            (uint32_t)num_rows, positions, cos_cache, sin_cache, max_pos,
            static_cast<uint16_t*>(out), err_flags, -0.0f};
  const int64_t quads = (num_rows + 3) / 4;  // one warp-iteration per 4 rows
  int64_t grid = (quads + 7) / 8;
  if (grid > (int64_t)sms * 8) grid = (int64_t)sms * 8;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int which = (rope_style == FP4IDX_ROPE_NEOX ? 0 : 2) + scale_mode;
  auto kern = which == 0   ? fake_quant_kernel<FP4IDX_ROPE_NEOX, 0>
              : which == 1 ? fake_quant_kernel<FP4IDX_ROPE_NEOX, 1>
              : which == 2 ? fake_quant_kernel<FP4IDX_ROPE_INTERLEAVED, 0>
                           : fake_quant_kernel<FP4IDX_ROPE_INTERLEAVED, 1>;
  return launch_kernel(kern, (unsigned)grid, 256, 0, s, fa) == cudaSuccess ? FP4IDX_OK
                                                                            : FP4IDX_ERR_CUDA;
}

const char* fp4idx_status_string(fp4idx_status status) {
  switch (status) {
    case FP4IDX_OK: return "ok";
    case FP4IDX_ERR_NULL: return "a required pointer is NULL";
    case FP4IDX_ERR_SHAPE: return "invalid size (negative count, zero heads/blocks/positions, or overflow)";
    case FP4IDX_ERR_ALIGN: return "a pointer or stride breaks its alignment rule";
    case FP4IDX_ERR_ARG: return "invalid argument (rope_style, eps, weight_scale or an option)";
    case FP4IDX_ERR_CUDA: return "CUDA launch failed";
    case FP4IDX_ERR_SCRATCH: return "the request needs more than the library's static scratch";
  }
  return "unknown status";
}

const char* fp4idx_version(void) { return "fp4idx 0.5.0 sm_103a"; }

// H^-1/2 * D^-1/2 with D = 128, evaluated in double and rounded once to fp32;
// 0 for a non-positive head count.
fp4idx_status fp4idx_test_withhold_next(int kernel, int64_t index) {
  if (index < 0) return FP4IDX_ERR_ARG;
  if (kernel == FP4IDX_TEST_PREPASS)
    fp4idx_impl::stream_withhold_next(index);
  else if (kernel == FP4IDX_TEST_SCORER)
    fp4idx_impl::scorer_withhold_next(index);
  else
    return FP4IDX_ERR_ARG;
  return FP4IDX_OK;
}

float fp4idx_default_weight_scale(int64_t num_heads) {
  if (num_heads < 1) return 0.0f;
  return (float)(1.0 / sqrt((double)num_heads * (double)FP4IDX_HEAD_DIM));
}

}  // extern "C"
