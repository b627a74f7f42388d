// fp4idx_scorer.cu -- FP4 MQA-logits scorers on the block-scaled FP4 tensor
// cores of sm_103a (tcgen05.mma kind::mxf4): the paged decode scorer and its
// prefill variant.  They consume the bytes the pre-pass writes: packed E2M1
// queries with their per-32 UE8M0 exponent words, and the 68-byte index-K
// slots of the paged cache.  The operations and argument contracts are in
// include/fp4idx.h.
//
// Sources (web pages, by title and section):
//   "[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR
//   5484), Summary and Verification: the paged FP4 MQA-logits scorer "and its
//   prefill variant" read the packed E2M1 keys and their e8m0 exponents
//   straight out of the cache; GLM-5.2 shapes (H = 32, D = 128, kv_block =
//   64), next_n 1 and 4.
//   "[ROCm][Perf] Enabled FP4Indexer for DSV4" (vLLM PR 42908), Code Review:
//   the score of a key is the block-scaled E2M1 dot product with each query
//   head, through ReLU, times the head weight, summed over the heads.
//   "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656), Summary: the
//   68-byte slot (64 payload bytes + 4 exponent bytes).
//
// Work.  A segment is a set of query rows sharing one key range: a sequence
// (next_n tokens) in the decode scorer, a block of consecutive query tokens
// in the prefill scorer; R = tokens x H <= 128 rows form the MMA's N (a
// sequence with more rows is split into groups of 128 / H tokens).  A tile
// is 128 consecutive keys (two 64-slot pages) of a segment's range.  The
// persistent grid splits the list of all (segment, tile) work items into
// equal contiguous shares, one per CTA, from the context lengths / key
// ranges alone; a share may span several segments.  Columns outside the
// ranges (-inf) are split the same way.
//
// MMA.  Keys are A (M = 128), the segment's query rows B (N = R), K = 128 as
// two MMAs of K = 64 into an fp32 TMEM accumulator.  Each exponent word of a
// slot is exactly one TMEM scale-factor cell (group g in byte g; the K halves
// use bytes 0-1 and 2-3).
//
// Roles (16 warps, four per SM sub-partition, so 128 registers a thread).
// The tile rate of a one-CTA-per-SM pipeline is set by the longest serial
// chain of dependent instructions that one warp runs per tile, not by the
// copy latency: an mbarrier operation costs one thread on the order of a
// hundred cycles, and one warp's copies are accepted at about one 8.7 KB
// tile per thousand cycles whatever their number or kind.  So four
// consecutive tiles share one stage and one full / empty barrier pair, the
// stages alternate between two producer warps, the tiles between two issuer
// warps, and accumulator m and epilogue group m form a pipeline for the
// tiles k = m (mod 3).
//   warps 2-3    producers: stage j belongs to producer j % 2.  For its next
//                four stages, a batch ahead, a producer's lanes describe the
//                batch's 16 tiles in parallel (page ids, a header word per
//                tile, the segment's first query row).  Per stage, lane 0
//                waits for it, writes the four header words, at a segment's
//                first tile loads the segment's query operand and scale
//                words into a query buffer (the loads into one buffer in
//                segment order, whichever producer makes them) and makes the
//                buffer releases of the issuers that have no tile in the
//                segment, then issues the TMA tensor copies of the page
//                payloads (64-byte swizzled, the layout the MMA reads) and
//                the bulk copies of their exponent words.  Between stages the
//                warp writes its share of the -inf columns outside every
//                segment's range.
//   warps 0-1    issuers: tile k belongs to issuer k % 2 and accumulator
//                k % 3.  Once the stage has landed, the warp transposes the
//                tile's 128 exponent words (and at its first tile of a
//                segment the queries' words) into the 32 x 128-bit blocks
//                tcgen05.cp reads; lane 0 then issues tcgen05.cp into TMEM,
//                the two MMAs into the accumulator and commits that mark the
//                accumulator full, after its last tile of a stage its share
//                of the stage free and, after its last tile of a segment, its
//                share of the segment's query buffer free (a buffer is free
//                once two releases came).
//   warps 4-15   epilogue: group m = (w - 4) / 4 reads accumulator m; each
//                warp of the group waits for it; warp w of the group reads TMEM lane
//                quadrant w % 4 (keys 32(w%4) .. +31 of the tile, one per
//                thread) over every query row, frees the accumulator once its
//                loads are done, then forms and stores the logits.
// Every wait is bounded (1 s) and a shared abort flag stops every role;
// copies and MMAs in flight are waited for before TMEM and shared memory are
// released.  Each E2M1 product is exact; the tensor core accumulates in
// fp32, and the weighted head sum is fp32.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fp4idx.h"

namespace {

// Warp roles.  The warps on a tile's critical chains (issuer, stager,
// producers) take the lowest warp ids: among ready warps the schedulers
// favour the oldest, so the epilogue's bulk work does not delay them.
constexpr int kIssuers = 2;                               // tile k: issuer k % 2
constexpr int kIssuerWarp = 0;                            // warps 0-1
constexpr int kProducers = 2;                             // stage j: producer j % 2
constexpr int kProducerWarp = kIssuerWarp + kIssuers;     // warps 2-3
constexpr int kEpiWarp = kProducerWarp + kProducers;      // warps 4-15
constexpr int kEpiGroups = 3;                             // one per accumulator
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kWarps = kEpiWarp + kEpiWarps;              // 16: four per SM sub-partition
constexpr int kThreads = kWarps * 32;                    // 512
constexpr int kTile = 128;                               // keys per tile (MMA M)
constexpr int kKvBlock = FP4IDX_KV_BLOCK;
constexpr int kPageBytes = FP4IDX_PAGE_BYTES;
constexpr int kPayloadBytes = kKvBlock * FP4IDX_SLOT_PAYLOAD_BYTES;  // 4096
constexpr int kExpBytes = kKvBlock * FP4IDX_SLOT_EXP_BYTES;          // 256
constexpr int kMaxRows = 128;                  // query rows per segment (MMA N)
constexpr int kMaxChunks = kMaxRows / 32;
constexpr int kMaxTps = kMaxRows / 32;         // query tokens per segment (H >= 32)
constexpr int kMaxAccs = kEpiGroups;           // TMEM accumulators
constexpr int kQBufs = 4;                      // query operand buffers
constexpr int kTps = 4;                        // tiles per stage
constexpr int kMaxStages = 4;                  // stages (kTps tiles each)
constexpr int kSegTab = 512;                   // segment ranges kept in shared memory
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCols = 8;                // TMEM columns per scale-word slot
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
static_assert(kMaxStages % kProducers == 0, "stage slots are split evenly between the producers");
static_assert(kIssuers >= 2 && kIssuers <= kMaxAccs && (kIssuers == kMaxAccs || kIssuers == 2),
              "an accumulator is used by one issuer, or by two in turn");
// Each issuer releases a stage once, after its last tile there, when the
// issuers split every stage evenly; otherwise every tile releases its share.
constexpr bool kReleasePerIssuer = kTps % kIssuers == 0;
constexpr int kStageReleases = kReleasePerIssuer ? kIssuers : kTps;
static_assert(kReleasePerIssuer, "an issuer handles its tiles of a stage together");
static_assert(kQBufs == 4, "a header word holds the query buffer in two bits");
static_assert(kMaxAccs * kMaxRows + (kMaxAccs + kIssuers * kQBufs) * kSfCols <= kTmemCols,
              "accumulators and scale words fit the TMEM columns");

// Offsets inside a stage: tiles h = 0 .. kTps-1 share one stage, one full
// and one empty barrier.
constexpr uint32_t kTilePayload = 2 * kPayloadBytes;  // 8192: tile h's two swizzled payloads at +8192h
constexpr uint32_t kPsExp = kTps * kTilePayload;      // tile h's 2 x 256 exponent words at +512h
constexpr uint32_t kPsSfa = kPsExp + kTps * 512;      // tile h's keys' words, transposed, at +512h
constexpr uint32_t kPsSfb = kPsSfa + kTps * 512;      // tile h's queries' words, transposed, at +512h
constexpr uint32_t kPsHdr = kPsSfb + kTps * 512;      // one header word per tile
constexpr uint32_t kStageBytes = (kPsHdr + 4 * kTps + 1023) / 1024 * 1024;  // a multiple of 1024
// A tile's header word (written by the producer, read by the tile's issuer):
// query buffer (bits 0-1), its fill parity (bit 2), the issuer's first
// (bit 3) and last (bit 4) tile of the segment here, the segment's first
// tile here (bit 5), the number of issuers with tiles in the segment here
// (bits 6-7), the segment's query rows (bits 8-15), the segment's ordinal in
// this CTA modulo 2^16 (bits 16-31; the buffer is its low two bits).
constexpr uint32_t kHdrFirst = 1u << 3, kHdrLast = 1u << 4, kHdrSegFirst = 1u << 5;

enum { kModeDecode = 0, kModePrefill = 1 };

struct ScorerParams {
  const uint8_t* q_scale;
  const float* weights;
  const uint8_t* cache;
  const int32_t* block_table;  // decode
  const int32_t* ctx_lens;     // decode
  const int32_t* ks;           // prefill
  const int32_t* ke;           // prefill
  float* logits;
  uint32_t* err;
  int64_t num_blocks;
  int64_t bt_stride;
  int64_t logits_stride;
  int32_t mode;
  int32_t nseg;         // segments
  int32_t tps;          // query tokens per segment (at most; R = tps * H <= 128)
  int32_t next_n;       // decode: query tokens per sequence
  int32_t ngroups;      // decode: segments per sequence, ceil(next_n / tps)
  int32_t num_q;        // query tokens
  int32_t H;
  int32_t R;            // tps * H
  int32_t ncols;        // logits columns (decode max_context, prefill key count)
  int32_t tiles_total;  // ceil(ncols / 128)
  int32_t stages;       // stages of kTps tiles
  int32_t withhold;     // testing: a tile of CTA 0 whose copies are not issued (-1: none)
};

struct Layout {
  uint32_t q, qs, w, tab, bars, misc, total;
};

// mbarriers: full and empty per stage; full per accumulator and two empty
// ones (for its even and its odd uses); empty and full per query buffer.
__host__ __device__ constexpr int kBarriers(int P) { return 2 * P + 3 * kMaxAccs + 2 * kQBufs; }

__host__ __device__ inline Layout make_layout(int P, int R) {
  Layout L;
  L.q = (uint32_t)P * kStageBytes;                   // kQBufs x R x 64 swizzled queries
  L.qs = L.q + (uint32_t)kQBufs * R * 64;           // kQBufs x 128 query scale words
  L.w = L.qs + (uint32_t)kQBufs * 512u;             // per epilogue warp: kMaxRows weights
  L.tab = L.w + (uint32_t)kEpiWarps * kMaxRows * 4u;  // kSegTab x (lo, hi, lim)
  L.bars = L.tab + (uint32_t)kSegTab * 12u;
  L.misc = L.bars + 8u * (uint32_t)kBarriers(P);
  L.total = L.misc + 128u;
  return L;
}


// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (false)
// when another role has raised *abort, or after 1 s, raising *abort itself.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 8; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort = 1u;
      return false;
    }
  }
}

// Waits until *w == v (a word another warp of the CTA writes); gives up like
// wait_phase.
__device__ __forceinline__ bool wait_word(volatile uint32_t* w, uint32_t v,
                                          volatile uint32_t* abort) {
  if (*w == v) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    if (*w == v) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort = 1u;
      return false;
    }
  }
}

// The same wait with no abort flag: used while draining after an abort.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 64-byte
// swizzled layout: rows of 64 bytes, 8-row groups 512 bytes apart.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused here)
  d |= (uint64_t)(512 >> 4) << 32;         // stride byte offset: 8 rows
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)4 << 61;                  // 64-byte swizzle
  return d;
}

// Instruction descriptor of kind::mxf4: E2M1 A and B, UE8M0 scales, both
// K-major, M = 128, N = R, with the scale-factor byte ids of A and B.
__device__ __forceinline__ uint32_t mxf4_idesc(int R, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(R >> 3) << 17) | (1u << 23) |
         (1u << 27) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a tcgen05.cp source without swizzle: rows of
// 16 bytes, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t cp_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)(128 >> 4) << 16;         // leading byte offset
  d |= (uint64_t)(128 >> 4) << 32;         // stride byte offset: 8 rows
  d |= (uint64_t)1 << 46;                  // descriptor version
  return d;                                // no swizzle
}

// 32 rows x 128 bits from shared memory into TMEM columns taddr .. taddr+3
// of every lane quadrant (row l -> lane 32q + l): the scale-word layout the
// block-scaled MMA reads (row r's word at lane r, column r / 32).
__device__ __forceinline__ void cp_32x128b_x4(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Packed fp32 pair: (a.x * b.x + c.x, a.y * b.y + c.y), each rounded once.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// sum over 32 columns of w[i] * max(x[i], 0): four packed chains, then a
// fixed combining order.
__device__ __forceinline__ float weighted_relu_sum(const uint32_t (&x)[32], const float* w) {
  float2 a0 = make_float2(0.0f, 0.0f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 w0 = reinterpret_cast<const float4*>(w)[2 * i];
    const float4 w1 = reinterpret_cast<const float4*>(w)[2 * i + 1];
    const uint32_t* v = x + 8 * i;
    a0 = fma2(make_float2(w0.x, w0.y),
              make_float2(fmaxf(__uint_as_float(v[0]), 0.0f), fmaxf(__uint_as_float(v[1]), 0.0f)),
              a0);
    a1 = fma2(make_float2(w0.z, w0.w),
              make_float2(fmaxf(__uint_as_float(v[2]), 0.0f), fmaxf(__uint_as_float(v[3]), 0.0f)),
              a1);
    a2 = fma2(make_float2(w1.x, w1.y),
              make_float2(fmaxf(__uint_as_float(v[4]), 0.0f), fmaxf(__uint_as_float(v[5]), 0.0f)),
              a2);
    a3 = fma2(make_float2(w1.z, w1.w),
              make_float2(fmaxf(__uint_as_float(v[6]), 0.0f), fmaxf(__uint_as_float(v[7]), 0.0f)),
              a3);
  }
  return __fadd_rn(__fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y)),
                   __fadd_rn(__fadd_rn(a2.x, a2.y), __fadd_rn(a3.x, a3.y)));
}

// ---------------------------------------------------------------- segments
// A segment's work tiles [lo, hi) and its column limit: decode -- tiles
// below the effective context c = clamp(ctx, 0, max_context), limit c;
// prefill -- the tiles covering the union of its tokens' clamped key
// ranges, limit the key count.
struct SegRange {
  int lo, hi, lim;
};

// The query tokens of segment g: decode -- tokens j0 .. j0 + ntok - 1 of
// sequence b = g / ngroups (j0 = (g % ngroups) * tps), whose key range and
// block-table row it uses; prefill -- tokens g*tps .. of the chunk.
struct SegQ {
  int b, qt0, ntok;  // key-range owner (decode: sequence), first query token, tokens
};

__device__ __forceinline__ SegQ seg_q(const ScorerParams& p, int g) {
  SegQ q;
  if (p.mode == kModeDecode) {
    q.b = g / p.ngroups;
    const int j0 = (g - q.b * p.ngroups) * p.tps;
    q.qt0 = q.b * p.next_n + j0;
    q.ntok = min(p.tps, p.next_n - j0);
  } else {
    q.b = g;
    q.qt0 = g * p.tps;
    q.ntok = min(p.tps, p.num_q - q.qt0);
  }
  return q;
}

__device__ __forceinline__ SegRange seg_load(const ScorerParams& p, int g) {
  SegRange r;
  if (p.mode == kModeDecode) {
    const int c = min(max(__ldg(p.ctx_lens + g / p.ngroups), 0), p.ncols);
    r.lo = 0;
    r.hi = (c + kTile - 1) / kTile;
    r.lim = c;
  } else {
    int mn = p.ncols, mx = 0;
    const int t0 = g * p.tps;
    for (int j = 0; j < p.tps; ++j) {
      const int t = t0 + j;
      if (t >= p.num_q) break;
      const int a = min(max(__ldg(p.ks + t), 0), p.ncols);
      const int b = min(max(__ldg(p.ke + t), 0), p.ncols);
      if (a < b) {
        mn = min(mn, a);
        mx = max(mx, b);
      }
    }
    if (mn < mx) {
      r.lo = mn / kTile;
      r.hi = (mx + kTile - 1) / kTile;
    } else {
      r.lo = r.hi = 0;
    }
    r.lim = p.ncols;
  }
  return r;
}

struct SegTable {
  const int* tab;  // kSegTab x (lo, hi, lim) for segments g0 .. g0 + kSegTab - 1
  int g0;
  __device__ __forceinline__ SegRange get(const ScorerParams& p, int g) const {
    const int i = g - g0;
    if (i >= 0 && i < kSegTab) {
      SegRange r;
      r.lo = tab[3 * i];
      r.hi = tab[3 * i + 1];
      r.lim = tab[3 * i + 2];
      return r;
    }
    if (g >= p.nseg) return SegRange{0, 0, 0};
    return seg_load(p, g);
  }
  // the next segment after g with work tiles (p.nseg if none)
  __device__ __forceinline__ int next(const ScorerParams& p, int g, SegRange& r) const {
    for (++g; g < p.nseg; ++g) {
      r = get(p, g);
      if (r.lo < r.hi) return g;
    }
    r = SegRange{0, 0, 0};
    return p.nseg;
  }
};

// Walks a CTA's work tiles in order: segment g, tile t in [lo, hi), the
// segment's ordinal qi in this CTA (its query buffer is qi % qbufs) and
// whether t is the first tile of the segment in this CTA.
struct Walk {
  int g, t, hi, lim, qi, pos;  // pos: tiles of the segment before t in this CTA
  SegQ q;
  bool first;
  __device__ __forceinline__ void init(const ScorerParams& p, const SegTable& st, int g0,
                                       int toff) {
    const SegRange r = st.get(p, g0);
    g = g0;
    t = r.lo + toff;
    hi = r.hi;
    lim = r.lim;
    qi = 0;
    pos = 0;
    q = seg_q(p, g0);
    first = true;
  }
  // Only called while tiles remain, so a later segment with work exists.
  __device__ __forceinline__ void advance(const ScorerParams& p, const SegTable& st) {
    first = false;
    ++pos;
    if (++t < hi) return;
    SegRange r;
    g = st.next(p, g, r);
    t = r.lo;
    hi = r.hi;
    lim = r.lim;
    ++qi;
    pos = 0;
    q = seg_q(p, g);
    first = true;
  }
};

// Writes -inf over a CTA's share of the tiles outside every segment's range
// (for each such (segment, tile): the segment's query rows x 128 columns),
// a few tiles at a time, one warp.
struct Filler {
  int g, off, left;
  SegRange r;
  __device__ __forceinline__ void init(const ScorerParams& p, const SegTable& st, int g0,
                                       int off0, int count) {
    g = g0;
    off = off0;
    left = count;
    if (count > 0) r = st.get(p, g);
  }
  // write (store) or step over (!store) the next `items` tiles
  __device__ __forceinline__ void run(const ScorerParams& p, const SegTable& st, int items,
                                      int lane, bool store = true) {
    for (; items > 0 && left > 0; --items, --left) {
      int np = p.tiles_total - (r.hi - r.lo);
      while (off >= np && g + 1 < p.nseg) {  // the next segment with -inf tiles
        off = 0;
        r = st.get(p, ++g);
        np = p.tiles_total - (r.hi - r.lo);
      }
      if (off >= np) {
        left = 0;
        return;
      }
      const int tile = off < r.lo ? off : r.hi + (off - r.lo);
      const SegQ q = seg_q(p, g);
      for (int j = 0; j < q.ntok && store; ++j) {
        float* const out = p.logits + (int64_t)(q.qt0 + j) * p.logits_stride;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int s = tile * kTile + 32 * m + lane;
          if (s < p.ncols) __stcs(out + s, -INFINITY);
        }
      }
      ++off;
    }
  }
};

// Inclusive warp scan of two 64-bit values.
__device__ __forceinline__ void warp_scan2(long long& a, long long& b, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long ya = __shfl_up_sync(0xffffffffu, a, o);
    const long long yb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) {
      a += ya;
      b += yb;
    }
  }
}

// ---------------------------------------------------------------- the kernel
// CPJ: accumulator chunks of 32 columns per query token, H / 32.
template <int CPJ, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    scorer_kernel(const __grid_constant__ ScorerParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages, R = p.R;
  constexpr int A = kMaxAccs, QB = kQBufs;
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Layout L = make_layout(S, R);
  uint8_t* const sQ = smem + L.q;
  const uint32_t* const sQs = reinterpret_cast<const uint32_t*>(smem + L.qs);
  float* const sW = reinterpret_cast<float*>(smem + L.w);
  int* const tab = reinterpret_cast<int*>(smem + L.tab);
  const uint32_t bars = smem_addr(smem + L.bars);
  uint32_t* const misc = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile uint32_t* const abort = misc + 1;
  volatile uint32_t* const qseq = misc + 24;  // per query buffer: loads made (mod 2^14)
  int32_t* const start = reinterpret_cast<int32_t*>(misc + 2);  // g0, toff, n, pg0, poff, pn
  auto stage = [&](int s) { return smem + (uint32_t)s * kStageBytes; };
  auto bar_full = [&](int s) { return bars + 8u * (uint32_t)s; };
  auto bar_empty = [&](int s) { return bars + 8u * (uint32_t)(S + s); };
  auto bar_accf = [&](int a) { return bars + 8u * (uint32_t)(2 * S + a); };
  // Accumulator a's readout of its use v arrives on bar_acce(a, v & 1): the
  // two issuers take turns on an accumulator, and one barrier per use parity
  // keeps every wait on it within one phase of the barrier's state.
  auto bar_acce = [&](int a, int par) {
    return bars + 8u * (uint32_t)(2 * S + kMaxAccs + 2 * a + par);
  };
  auto bar_qempty = [&](int b) { return bars + 8u * (uint32_t)(2 * S + 3 * kMaxAccs + b); };
  auto bar_qfull = [&](int b) {
    return bars + 8u * (uint32_t)(2 * S + 3 * kMaxAccs + kQBufs + b);
  };

  // ---- this CTA's shares of the work tiles and of the -inf tiles ----------
  // (the scan scratch lives in the stage area, unused until the copies start)
  long long* const scanw = reinterpret_cast<long long*>(smem);   // kWarps (prefix of work)
  long long* const scanp = scanw + 32;                           // kWarps (prefix of pads)
  {
    const int per = (p.nseg + kThreads - 1) / kThreads;
    const int g_lo = min(p.nseg, tid * per), g_hi = min(p.nseg, g_lo + per);
    long long wpart = 0, ppart = 0;
    for (int g = g_lo; g < g_hi; ++g) {
      const SegRange r = seg_load(p, g);
      wpart += r.hi - r.lo;
      ppart += p.tiles_total - (r.hi - r.lo);
    }
    long long wi = wpart, pi = ppart;
    warp_scan2(wi, pi, lane);
    if (tid == 0) {
      *abort = 0u;
      start[2] = 0;
      start[5] = 0;
      for (int m = 0; m < kIssuers; ++m) misc[8 + m] = 0u;
      for (int b = 0; b < kQBufs; ++b) misc[24 + b] = 0u;
    }
    if (lane == 31) {
      scanw[warp] = wi;
      scanp[warp] = pi;
    }
    __syncthreads();
    if (warp == 0) {
      long long a = lane < kWarps ? scanw[lane] : 0, b = lane < kWarps ? scanp[lane] : 0;
      const long long a0 = a, b0 = b;
      warp_scan2(a, b, lane);
      __syncwarp();
      if (lane < kWarps) {
        scanw[lane] = a - a0;  // exclusive prefix of each warp
        scanp[lane] = b - b0;
      }
      if (lane == kWarps - 1) {
        scanw[kWarps] = a;  // totals
        scanp[kWarps] = b;
      }
    }
    __syncthreads();
    const long long wex = scanw[warp] + wi - wpart, pex = scanp[warp] + pi - ppart;
    const long long W = scanw[kWarps], P = scanp[kWarps];
    const long long lo = W * blockIdx.x / gridDim.x, hi = W * (blockIdx.x + 1) / gridDim.x;
    if (lo < hi && wex <= lo && lo < wex + wpart) {
      long long acc = wex;
      for (int g = g_lo; g < g_hi; ++g) {
        const SegRange r = seg_load(p, g);
        if (lo < acc + (r.hi - r.lo)) {
          start[0] = g;
          start[1] = (int)(lo - acc);
          start[2] = (int)(hi - lo);
          break;
        }
        acc += r.hi - r.lo;
      }
    }
    const long long plo = P * blockIdx.x / gridDim.x, phi = P * (blockIdx.x + 1) / gridDim.x;
    if (plo < phi && pex <= plo && plo < pex + ppart) {
      long long acc = pex;
      for (int g = g_lo; g < g_hi; ++g) {
        const SegRange r = seg_load(p, g);
        const int np = p.tiles_total - (r.hi - r.lo);
        if (plo < acc + np) {
          start[3] = g;
          start[4] = (int)(plo - acc);
          start[5] = (int)(phi - plo);
          break;
        }
        acc += np;
      }
    }
    __syncthreads();
  }
  const int n = start[2];
  SegTable st;
  st.tab = tab;
  st.g0 = n > 0 ? start[0] : -2 * kSegTab;  // no table without work tiles
  for (int i = tid; i < kSegTab; i += kThreads) {
    const int g = st.g0 + i;
    SegRange r = SegRange{0, 0, 0};
    if (n > 0 && g < p.nseg) r = seg_load(p, g);
    tab[3 * i] = r.lo;
    tab[3 * i + 1] = r.hi;
    tab[3 * i + 2] = r.lim;
  }

  uint32_t tmem = 0;
  if (n > 0) {
    if (tid == 0) {
      for (int i = 0; i < kBarriers(S); ++i) {
        // a stage's empty takes one arrival per issuer, acc_empty one per
        // warp of its epilogue group, a query buffer's empty one per issuer
        const int j = i - 2 * S;
        const int cnt = i >= S && i < 2 * S                             ? kStageReleases
                        : j >= kMaxAccs && j < 3 * kMaxAccs                ? 4
                        : j >= 3 * kMaxAccs && j < 3 * kMaxAccs + kQBufs ? kIssuers
                                                                         : 1;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bars + 8u * i), "r"(cnt)
                     : "memory");
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kIssuerWarp) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_addr(misc)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  }
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (n > 0) tmem = misc[0];
  // TMEM columns: accumulator a at a*R; the keys' scale words of
  // accumulator a at A*R + 8a; the queries' words of buffer b for issuer m
  // at A*R + 8A + 8(m*QB + b) (each issuer copies its own).
  const uint32_t sfa_col0 = (uint32_t)A * R, sfb_col0 = sfa_col0 + kMaxAccs * kSfCols;
  int last_issued = -1;  // producer: the last stage use whose copies were issued
  int q_issued[4] = {-1, -1, -1, -1};  // producers: parity of the last query copy per buffer

  if (n > 0 && warp >= kProducerWarp && warp < kProducerWarp + kProducers) {
    // ---- producers: stage j (tiles kTps*j ..) belongs to producer j % 2 ------
    // Per batch of the producer's next four stages, a batch ahead, lane L
    // describes half L % 2 of the batch's tile L / 2: the page to read (or
    // none), the tile's header word and the first query row of its segment.
    // Lane 0 then issues every copy of a stage itself: one warp's copies are
    // accepted at a bounded rate, and a loop in one lane beats lanes that
    // each issue one.
    const int pr = warp - kProducerWarp;
    Walk lw;  // this lane's walker, at its tile of the batch being described
    lw.init(p, st, start[0], start[1]);
    int lk = 0;  // lw's tile index
    struct Desc {
      int32_t page;  // page to read; -1: none (past the context, or a bad entry)
      uint32_t hdr;
      int32_t qrow;
    };
    // first stage of the producer's batch b; tile of slot s (0..15) in it
    auto batch_stage = [&](int b) { return pr + kProducers * 4 * b; };
    auto describe = [&](int b) -> Desc {
      const int sl = lane >> 1;
      const int m = kTps * (batch_stage(b) + kProducers * (sl / kTps)) + sl % kTps;
      Desc dsc = {-1, 0u, 0};
      if (m < n) {
        if (m > lk && lw.t + (m - lk) < lw.hi) {  // the common case: the same segment
          lw.t += m - lk;
          lw.pos += m - lk;
          lw.first = false;
          lk = m;
        }
        for (; lk < m; ++lk) lw.advance(p, st);
        const int pidx = lw.t * 2 + (lane & 1);
        if (pidx * kKvBlock < lw.lim) {
          const int32_t id = MODE == kModeDecode
                                 ? __ldg(p.block_table + (int64_t)lw.q.b * p.bt_stride + pidx)
                                 : pidx;
          if (id >= 0 && id < p.num_blocks)
            dsc.page = id;
          else
            flag_error(p.err, FP4IDX_ERRFLAG_PAGE);  // not read: those keys score -inf
        }
        const int left = min(lw.hi - 1 - lw.t, n - 1 - m);  // the segment's tiles here after m
        const int owners = min(kIssuers, left + 1);           // at its first tile here
        dsc.hdr = (uint32_t)(lw.qi % QB) | ((((uint32_t)(lw.qi / QB)) & 1u) << 2) |
                  (lw.pos < kIssuers ? kHdrFirst : 0u) | (left < kIssuers ? kHdrLast : 0u) |
                  (lw.first ? kHdrSegFirst : 0u) | ((uint32_t)owners << 6) |
                  ((uint32_t)(lw.q.ntok * p.H) << 8) | ((uint32_t)(lw.qi & 0xFFFF) << 16);
        dsc.qrow = lw.q.qt0 * p.H;
      }
      return dsc;
    };
    const uint32_t q_bytes = (uint32_t)R * 64u;
    // A segment's first tile here: its query operand and scale words, on the
    // query buffer's own barrier; then the releases of the buffer that
    // issuers without a tile in the segment will not make.  The loads into a
    // buffer go in segment order, whichever producer makes them: a load
    // first waits until the buffer's previous segment has been loaded, so the
    // release it then waits for is the barrier's current phase, never one
    // two phases back (which the parity alone cannot tell apart).
    auto load_q = [&](uint32_t hdr, int32_t qrow) -> bool {
      const int qb = (int)(hdr & 3u);
      const uint32_t qpar = (hdr >> 2) & 1u, use = (hdr >> 18) & 0x3FFFu;
      if (!wait_word(qseq + qb, use, abort)) return false;
      if (!wait_phase(bar_qempty(qb), qpar ^ 1u, abort)) return false;
      const uint32_t qf = bar_qfull(qb);
      const uint32_t sw_bytes = ((hdr >> 8) & 0xFFu) * 4u;
      mbar_expect_tx(qf, q_bytes + sw_bytes);
      tma_2d(smem_addr(sQ + (uint32_t)qb * q_bytes), &qmap, 0, qrow, qf);
      bulk_copy(smem_addr(sQs + qb * 128), p.q_scale + (int64_t)qrow * 4, sw_bytes, qf);
      q_issued[qb] = (int)qpar;
      for (int o = (int)((hdr >> 6) & 3u); o < kIssuers; ++o) mbar_arrive(bar_qempty(qb));
      qseq[qb] = (use + 1u) & 0x3FFFu;
      return true;
    };
    // This producer's share of the CTA's -inf tiles, spread over its stages
    // (the producers run well ahead of the tensor cores, the epilogue does
    // not).
    const int pn_all = start[5];
    const int f_lo = (int)((long long)pn_all * pr / kProducers);
    const int f_hi = (int)((long long)pn_all * (pr + 1) / kProducers), pn = f_hi - f_lo;
    const int n_st = ((n + kTps - 1) / kTps - pr + kProducers - 1) / kProducers;  // its stages
    Filler fill;
    fill.init(p, st, start[3], start[4], f_hi);
    fill.run(p, st, f_lo, lane, false);  // step over the other producer's share
    int facc = 0;  // Bresenham: f_hi - f_lo tiles over n_st stages, without a division
    Desc cur = describe(0), nxt = {-1, 0u, 0};
    bool stop = false;
    for (int b = 0; !stop && kTps * batch_stage(b) < n; ++b) {
      if (kTps * batch_stage(b + 1) < n) nxt = describe(b + 1);
      for (int i = 0; i < 4; ++i) {
        const int j = batch_stage(b) + kProducers * i, k = kTps * j;
        if (k >= n) break;
        const int nt = min(kTps, n - k);  // tiles in this stage
        const int ps = j % S;
        const uint32_t ph = (uint32_t)(j / S) & 1u;
        int32_t page[kTps][2];
        uint32_t hdr[kTps];
        int32_t qrow[kTps];
#pragma unroll
        for (int t = 0; t < kTps; ++t) {
          page[t][0] = __shfl_sync(0xffffffffu, cur.page, 2 * (kTps * i + t));
          page[t][1] = __shfl_sync(0xffffffffu, cur.page, 2 * (kTps * i + t) + 1);
          hdr[t] = __shfl_sync(0xffffffffu, cur.hdr, 2 * (kTps * i + t));
          qrow[t] = __shfl_sync(0xffffffffu, cur.qrow, 2 * (kTps * i + t));
        }
        int ok = 1;
        if (lane == 0) {
          ok = wait_phase(bar_empty(ps), ph ^ 1u, abort);
          // testing hook (see fp4idx_test_withhold_next): this stage's copies
          // and its arrival are withheld, so the waits for it run out
          const bool withheld = blockIdx.x == 0 && p.withhold >= k && p.withhold < k + nt;
          if (ok && !withheld) {
#pragma unroll
            for (int t = 0; t < kTps; ++t)
              if (ok && t < nt && (hdr[t] & kHdrSegFirst)) ok = load_q(hdr[t], qrow[t]);
          }
          if (ok && !withheld) {
            uint8_t* const sp = stage(ps);
            uint32_t reads = 0;
#pragma unroll
            for (int t = 0; t < kTps; ++t) {
              reinterpret_cast<uint32_t*>(sp + kPsHdr)[t] = hdr[t];
              reads += (t < nt && page[t][0] >= 0) + (t < nt && page[t][1] >= 0);
            }
            const uint32_t fb = bar_full(ps);
            mbar_expect_tx(fb, reads * (kPayloadBytes + kExpBytes));
#pragma unroll
            for (int t = 0; t < kTps; ++t)
#pragma unroll
              for (int pg = 0; pg < 2; ++pg)
                if (t < nt && page[t][pg] >= 0) {
                  const int32_t id = page[t][pg];
                  tma_3d(smem_addr(sp + t * kTilePayload + pg * kPayloadBytes), &kmap, 0, 0, id, fb);
                  bulk_copy(smem_addr(sp + kPsExp + t * 512 + pg * kExpBytes),
                            p.cache + (int64_t)id * kPageBytes + kPayloadBytes, kExpBytes, fb);
                }
            last_issued = j;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        int items = 0;
        for (facc += pn; facc >= n_st; facc -= n_st) ++items;
        fill.run(p, st, items, lane);
      }
      cur = nxt;
    }
    fill.run(p, st, pn, lane);  // any left (an aborted loop)
  } else if (n > 0 && warp >= kIssuerWarp && warp < kIssuerWarp + kIssuers) {
    // ---- issuers: tile k belongs to issuer k % 2 and accumulator k % 3 -------
    const int m = warp - kIssuerWarp;
    const uint32_t id0 = mxf4_idesc(R, 0), id1 = mxf4_idesc(R, 2);
    const uint32_t q_bytes = (uint32_t)R * 64u;
    int issued = 0;  // tiles issued by this issuer
    // tile k's accumulator a = k % 3 and its use k / 3; its stage j = k / kTps
    // (slot ps = j % S, parity ph) and place h = k % kTps there, all stepped
    // along with k
    int a = m % kMaxAccs, use = m / kMaxAccs, h = m % kTps, ps = (m / kTps) % S;
    uint32_t ph = (uint32_t)((m / kTps) / S) & 1u;
    for (int k = m; k < n; k += kIssuers) {
      const uint32_t d = tmem + (uint32_t)a * (uint32_t)R;
      const uint32_t sfa = tmem + sfa_col0 + kSfCols * (uint32_t)a;
      uint8_t* const sp = stage(ps);
      // At its first tile of a stage the issuer waits for the stage (every
      // lane, which reads the landed words, observes the completed phase
      // itself: acquire) and transposes the keys' words of both its tiles
      // there; row l of a tile's block holds tokens l, l+32, l+64, l+96.
      const bool stage_first = h < kIssuers;
      int ok = 1;
      if (stage_first) {
        ok = __all_sync(0xffffffffu, wait_phase(bar_full(ps), ph, abort));
        if (!ok) break;
#pragma unroll
        for (int t = 0; t < kTps / kIssuers; ++t) {
          const int ht = h + kIssuers * t;
          if (t == 0 || k + kIssuers * t < n) {
            const uint32_t* ew = reinterpret_cast<const uint32_t*>(sp + kPsExp + 512 * ht);
            *reinterpret_cast<uint4*>(sp + kPsSfa + 512 * ht + 16 * lane) =
                make_uint4(ew[lane], ew[lane + 32], ew[lane + 64], ew[lane + 96]);
          }
        }
      }
      const uint32_t hdr = *reinterpret_cast<const uint32_t*>(sp + kPsHdr + 4 * h);
      const int qb = (int)(hdr & 3u);
      const bool first = (hdr & kHdrFirst) != 0;
      if (first) {  // this issuer's first tile of the segment: the queries' words
        const uint32_t qpar = (hdr >> 2) & 1u;
        ok = __all_sync(0xffffffffu, wait_phase(bar_qfull(qb), qpar, abort));
        if (!ok) break;
        const int rows = (int)(hdr >> 8) & 0xFF;
        const uint32_t* qw = sQs + qb * 128;
        uint32_t v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = 32 * c + lane < rows ? qw[32 * c + lane] : 0x7F7F7F7Fu;
        *reinterpret_cast<uint4*>(sp + kPsSfb + 512 * h + 16 * lane) = make_uint4(v[0], v[1], v[2], v[3]);
      }
      // generic-proxy writes, read next by tcgen05.cp (async proxy)
      if (stage_first || first) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        // accumulator a has been read out (its previous use, tile k - 3, which
        // the other issuer made).  That barrier cannot be two phases behind:
        // this issuer made tile k - 6 only after the readout of tile k - 9.
        ok = use == 0 || wait_phase(bar_acce(a, (use - 1) & 1), (uint32_t)((use - 1) >> 1) & 1u,
                                    abort);
        if (ok) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t sfb = tmem + sfb_col0 + kSfCols * (uint32_t)(m * QB + qb);
          cp_32x128b_x4(sfa, cp_desc(smem_addr(sp + kPsSfa + 512 * h)));
          if (first) cp_32x128b_x4(sfb, cp_desc(smem_addr(sp + kPsSfb + 512 * h)));
          // operand descriptors built from the buffers' own addresses
          const uint64_t adesc = sw64_desc(smem_addr(sp + h * kTilePayload));
          const uint64_t qdesc = sw64_desc(smem_addr(sQ + (uint32_t)qb * q_bytes));
          mma_mxf4(d, adesc, qdesc, id0, sfa, sfb, 0u);
          mma_mxf4(d, adesc + 2, qdesc + 2, id1, sfa, sfb, 1u);
          // Each commit tracks every earlier MMA of this thread: the
          // accumulator is full, this tile's share of the stage can be
          // refilled, and after this issuer's last tile of the segment, its
          // share of the query buffer is released.
          mma_commit(bar_accf(a));
          // the stage is free once both issuers' tiles there are done: each
          // releases it after its last one (the stage's empty barrier takes
          // kIssuers arrivals; a partial last stage is never refilled)
          if (!kReleasePerIssuer || h >= kTps - kIssuers) mma_commit(bar_empty(ps));
          if (hdr & kHdrLast) mma_commit(bar_qempty(qb));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++issued;
      a += kIssuers;
      if (a >= kMaxAccs) {
        a -= kMaxAccs;
        ++use;
      }
      h += kIssuers;
      if (h >= kTps) {
        h -= kTps;
        if (++ps == S) {
          ps = 0;
          ph ^= 1u;
        }
      }
    }
    // for the drain after an abort: 1 + this issuer's last tile issued
    if (lane == 0) misc[8 + m] = issued > 0 ? (uint32_t)(m + kIssuers * (issued - 1) + 1) : 0u;
  } else if (n > 0 && warp >= kEpiWarp) {
    // ---- epilogue ---------------------------------------------------------------
    // Group j (warps 4+4j .. 7+4j) reads accumulator j, i.e. tiles k = j
    // (mod 3); its warp w reads TMEM lane quadrant w % 4 (tile keys
    // 32(w%4) .. +31, one per thread) across every query row of the segment.
    const int grp = (warp - kEpiWarp) >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // the tile's key = TMEM lane
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* const wts = sW + (warp - kEpiWarp) * kMaxRows;  // this warp's copy of the weights
    Walk w;
    w.init(p, st, start[0], start[1]);
    int wk = 0;                        // w's tile
    int cur_g = -1;                    // segment whose weights are in wts
    float* rowp = p.logits;            // the segment's first logits row
    const int32_t* btrow = p.block_table;  // decode: the segment's block-table row
    int ac[kMaxTps] = {0, 0, 0, 0}, bc[kMaxTps] = {0, 0, 0, 0};  // prefill key ranges
    uint32_t pu = 0;                   // parity of this group's next use of accumulator grp
    int j_own = 0;
    for (int k = grp; k < n; k += kEpiGroups) {
      if (k > wk && w.t + (k - wk) < w.hi) {  // the common case: the same segment
        w.t += k - wk;
        w.pos += k - wk;
        w.first = false;
        wk = k;
      }
      for (; wk < k; ++wk) w.advance(p, st);
      const int ntok = w.q.ntok;
      if (w.g != cur_g) {  // a new segment: its weights (and key ranges)
        rowp = p.logits + (int64_t)w.q.qt0 * p.logits_stride;
        if (MODE == kModeDecode) btrow = p.block_table + (int64_t)w.q.b * p.bt_stride;
        float wr[kMaxChunks];
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
          const int r = 32 * c + lane;
          wr[c] = r < ntok * p.H ? __ldg(p.weights + (int64_t)w.q.qt0 * p.H + r) : 0.0f;
        }
        if (MODE == kModePrefill) {
#pragma unroll
          for (int t = 0; t < kMaxTps; ++t) {
            const bool in = t < ntok;
            ac[t] = in ? min(max(__ldg(p.ks + w.q.qt0 + t), 0), p.ncols) : 0;
            bc[t] = in ? min(max(__ldg(p.ke + w.q.qt0 + t), 0), p.ncols) : 0;
          }
        }
        __syncwarp();  // the previous segment's reads of wts are done
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) wts[32 * c + lane] = wr[c];
        __syncwarp();
        cur_g = w.g;
      }
      // decode: this warp's page of the tile (-1 past the context), loaded
      // before the wait so that its latency is hidden behind it
      int32_t pid = 0;
      if (MODE == kModeDecode) {
        const int pidx = w.t * 2 + (quad >> 1);
        pid = pidx * kKvBlock < w.lim
                  ? __ldg(btrow + pidx)
                  : -1;
      }
      // Every warp of the group waits for the accumulator itself (a warp
      // suspended in mbarrier.try_wait takes no issue slots) and so observes
      // its completion (acquire).
      if (!__all_sync(0xffffffffu, wait_phase(bar_accf(grp), pu, abort))) break;
      pu ^= 1u;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int nv = ntok * CPJ;  // accumulator chunks holding this segment's rows
      const uint32_t col = tmem + lane_base + (uint32_t)grp * (uint32_t)R;
      float v[kMaxTps] = {0.0f, 0.0f, 0.0f, 0.0f};
      // chunk c's weighted head sum, added to its query token's score
      auto take = [&](int c, const uint32_t(&x)[32]) {
        const float sc = weighted_relu_sum(x, wts + 32 * c);
        v[c / CPJ] = c % CPJ == 0 ? sc : __fadd_rn(v[c / CPJ], sc);
      };
      // every load of the tile has landed: the accumulator is free
      auto release = [&]() {
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acce(grp, j_own & 1));
      };
      // Chunk c + 1 is loaded while chunk c is summed; tcgen05.wait::ld waits
      // for every load in flight, so each wait follows the sum before it.
      uint32_t xa[32], xb[32];
      tmem_ld32(col, xa);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int c = 0; c < kMaxChunks; c += 2) {
        if (c < nv) {  // xa holds chunk c
          if (c + 1 < nv)
            tmem_ld32(col + 32u * (c + 1), xb);
          else
            release();
          take(c, xa);
          if (c + 1 < nv) {
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (c + 2 < nv)
              tmem_ld32(col + 32u * (c + 2), xa);
            else
              release();
            take(c + 1, xb);
            if (c + 2 < nv) asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          }
        }
      }
      const int s_tok = w.t * kTile + row;
      const bool pok = pid >= 0 && pid < p.num_blocks;
#pragma unroll
      for (int t = 0; t < kMaxTps; ++t) {
        if (t < ntok && s_tok < p.ncols) {
          const bool valid = MODE == kModeDecode ? (s_tok < w.lim && pok)
                                                   : (s_tok >= ac[t] && s_tok < bc[t]);
          __stcs(rowp + (int64_t)t * p.logits_stride + s_tok, valid ? v[t] : -INFINITY);
        }
      }
      ++j_own;
    }
  } else if (n == 0 && warp == kProducerWarp) {
    // ---- no work tiles: only this CTA's share of the -inf tiles -------------
    Filler fill;
    fill.init(p, st, start[3], start[4], start[5]);
    fill.run(p, st, start[5], lane);
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (n > 0) {
    if (*abort) {  // every role has stopped: let copies in flight land first
      if (warp >= kProducerWarp && warp < kProducerWarp + kProducers && lane == 0) {
        for (int q = last_issued; q >= 0 && q > last_issued - S; q -= kProducers)
          wait_phase_drain(bar_full(q % S), (uint32_t)(q / S) & 1u);
        for (int b = 0; b < QB; ++b)
          if (q_issued[b] >= 0) wait_phase_drain(bar_qfull(b), (uint32_t)q_issued[b]);
      }
      // MMAs in flight land before TMEM is released: an issuer's last
      // commit tracks all its earlier MMAs, and that accumulator cannot be
      // two phases behind it (its previous use was read out before the tile
      // was issued).
      if (warp >= kIssuerWarp && warp < kIssuerWarp + kIssuers && lane == 0) {
        const int last = (int)misc[8 + (warp - kIssuerWarp)] - 1;
        if (last >= 0)
          wait_phase_drain(bar_accf(last % kMaxAccs), (uint32_t)(last / kMaxAccs) & 1u);
      }
      if (tid == 0) flag_error(p.err, FP4IDX_ERRFLAG_TIMEOUT);
      __syncthreads();
    }
    __syncwarp();
    if (warp == kIssuerWarp)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
  }
}

// ---------------------------------------------------------------- host side
bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

typedef void (*ScorerKernel)(ScorerParams, CUtensorMap, CUtensorMap);
// [mode][H / 32 - 1]
constexpr ScorerKernel kKernels[2][4] = {
    {scorer_kernel<1, kModeDecode>, scorer_kernel<2, kModeDecode>, scorer_kernel<3, kModeDecode>,
     scorer_kernel<4, kModeDecode>},
    {scorer_kernel<1, kModePrefill>, scorer_kernel<2, kModePrefill>,
     scorer_kernel<3, kModePrefill>, scorer_kernel<4, kModePrefill>}};

bool set_smem_limits(int bytes) {
  for (const auto& row : kKernels)
    for (ScorerKernel k : row)
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
          cudaSuccess)
        return false;
  return true;
}

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
};

std::mutex g_setup_mutex;
DeviceInfo g_info[64];
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

// One-time per-device set-up (SM count, shared-memory opt-in) and the driver
// entry point of cuTensorMapEncodeTiled, under a lock.
fp4idx_status device_setup(DeviceInfo& out, EncodeTiledFn& enc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4IDX_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_encode_tried) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(f);
    g_encode_tried = true;
  }
  DeviceInfo& di = g_info[dev];
  if (!di.ready) {
    DeviceInfo t;
    if (cudaDeviceGetAttribute(&t.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        !set_smem_limits(t.smem_optin))
      return FP4IDX_ERR_CUDA;
    t.ready = true;
    di = t;
  }
  out = di;
  enc = g_encode;
  return enc ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}

// Testing hook: the tile of CTA 0 whose copies the next scorer launch
// withholds (-1: none), taken once.
std::atomic<int64_t> g_withhold{-1};

// Heads both scorers accept: a multiple of 32, at most 128 (a segment holds
// at least one query token's heads).
bool heads_ok(int64_t H) { return H >= 32 && H % 32 == 0 && H <= kMaxRows; }

// Fills the launch-shape fields of p (stages, tiles) and launches.
fp4idx_status launch(ScorerParams& p, const uint8_t* q_fp4, const uint8_t* kv_cache,
                     cudaStream_t stream) {
  DeviceInfo di;
  EncodeTiledFn encode = nullptr;
  const fp4idx_status ds = device_setup(di, encode);
  if (ds != FP4IDX_OK) return ds;
  const int R = p.R;  // <= 128: 3 accumulators + scale words fit 512 TMEM columns
  // a multiple of the producer count: producer j % kProducers owns the
  // stage slots j % S, so no slot is shared between producers
  int S = kMaxStages;
  while (S > kProducers && (int)make_layout(S, R).total + 1024 > di.smem_optin) S -= kProducers;
  if ((int)make_layout(S, R).total + 1024 > di.smem_optin) return FP4IDX_ERR_SHAPE;
  p.stages = S;
  const int smem_bytes = (int)make_layout(S, R).total + 1024;
  p.tiles_total = (p.ncols + kTile - 1) / kTile;
  {
    const int64_t w = g_withhold.exchange(-1);
    p.withhold = w >= 0 && w < (1ll << 30) ? (int32_t)w : -1;
  }

  // The cache as a 3-D byte tensor: 64 payload bytes x 64 slots x pages.
  alignas(64) CUtensorMap kmap;
  {
    const cuuint64_t gdim[3] = {64, 64, (cuuint64_t)p.num_blocks};
    const cuuint64_t gstride[2] = {64, (cuuint64_t)kPageBytes};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(kv_cache), gdim,
               gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return FP4IDX_ERR_CUDA;
  }
  // The queries as rows of 64 bytes; a segment's R rows are one box (rows
  // past the last query row read as zeros).
  alignas(64) CUtensorMap qmap;
  {
    const cuuint64_t gdim[2] = {64, (cuuint64_t)p.num_q * (cuuint64_t)p.H};
    const cuuint64_t gstride[1] = {64};
    const cuuint32_t box[2] = {64, (cuuint32_t)R};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q_fp4), gdim,
               gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return FP4IDX_ERR_CUDA;
  }
  const auto kern = kKernels[p.mode == kModePrefill ? 1 : 0][p.H / 32 - 1];
  // cudaLaunchKernelEx reports this launch's own status, without reading or
  // clearing an error that the caller's own work left in the runtime
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)di.sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, p, kmap, qmap) == cudaSuccess ? FP4IDX_OK
                                                                        : FP4IDX_ERR_CUDA;
}

}  // namespace

extern "C" fp4idx_status fp4idx_paged_mqa_logits(
    const uint8_t* q_fp4, const uint8_t* q_scale, const float* weights, const uint8_t* kv_cache,
    int64_t num_blocks, const int32_t* block_table, int64_t block_table_stride,
    const int32_t* context_lens, float* logits, int64_t logits_stride, int64_t batch,
    int64_t next_n, int64_t num_heads, int64_t max_context, uint32_t* err_flags, void* stream) {
  if (batch < 0 || max_context < 0) return FP4IDX_ERR_SHAPE;
  if (batch == 0 || max_context == 0) return FP4IDX_OK;
  if (!q_fp4 || !q_scale || !weights || !kv_cache || !block_table || !context_lens || !logits)
    return FP4IDX_ERR_NULL;
  if (next_n < 1 || !heads_ok(num_heads) || num_blocks < 1 || num_blocks >= (1ll << 31) ||
      max_context >= (1 << 30) || next_n >= (1 << 20) ||
      batch * next_n >= (1ll << 31) / num_heads ||
      logits_stride < max_context ||
      block_table_stride < (max_context + kKvBlock - 1) / kKvBlock)
    return FP4IDX_ERR_SHAPE;
  if (!aligned(q_fp4, 16) || !aligned(q_scale, 16) || !aligned(weights, 4) ||
      !aligned(kv_cache, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4) ||
      !aligned(logits, 4) || (err_flags && !aligned(err_flags, 4)))
    return FP4IDX_ERR_ALIGN;
  ScorerParams p = {};
  p.q_scale = q_scale;
  p.weights = weights;
  p.cache = kv_cache;
  p.block_table = block_table;
  p.ctx_lens = context_lens;
  p.logits = logits;
  p.err = err_flags;
  p.num_blocks = num_blocks;
  p.bt_stride = block_table_stride;
  p.logits_stride = logits_stride;
  p.mode = kModeDecode;
  // A sequence's next_n tokens form one segment when their rows fit the MMA's
  // N = 128, otherwise groups of 128 / H tokens sharing the sequence's keys.
  p.tps = (int32_t)(next_n * num_heads <= kMaxRows ? next_n : kMaxRows / num_heads);
  p.next_n = (int32_t)next_n;
  p.ngroups = (int32_t)((next_n + p.tps - 1) / p.tps);
  p.nseg = (int32_t)(batch * p.ngroups);
  p.num_q = (int32_t)(batch * next_n);
  p.H = (int32_t)num_heads;
  p.R = p.tps * p.H;
  p.ncols = (int32_t)max_context;
  return launch(p, q_fp4, kv_cache, static_cast<cudaStream_t>(stream));
}

extern "C" fp4idx_status fp4idx_mqa_logits_prefill(
    const uint8_t* q_fp4, const uint8_t* q_scale, const float* weights, const uint8_t* kv_cache,
    int64_t num_blocks, int64_t num_keys, const int32_t* ks, const int32_t* ke, float* logits,
    int64_t logits_stride, int64_t num_tokens, int64_t num_heads, uint32_t* err_flags,
    void* stream) {
  if (num_tokens < 0 || num_keys < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0 || num_keys == 0) return FP4IDX_OK;
  if (!q_fp4 || !q_scale || !weights || !kv_cache || !ks || !ke || !logits)
    return FP4IDX_ERR_NULL;
  if (!heads_ok(num_heads) || num_blocks < 1 ||
      num_blocks >= (1ll << 31) || num_keys >= (1 << 30) ||
      num_keys > num_blocks * (int64_t)kKvBlock || num_tokens >= (1ll << 31) / num_heads ||
      logits_stride < num_keys)
    return FP4IDX_ERR_SHAPE;
  if (!aligned(q_fp4, 16) || !aligned(q_scale, 16) || !aligned(weights, 4) ||
      !aligned(kv_cache, 16) || !aligned(ks, 4) || !aligned(ke, 4) || !aligned(logits, 4) ||
      (err_flags && !aligned(err_flags, 4)))
    return FP4IDX_ERR_ALIGN;
  ScorerParams p = {};
  p.q_scale = q_scale;
  p.weights = weights;
  p.cache = kv_cache;
  p.ks = ks;
  p.ke = ke;
  p.logits = logits;
  p.err = err_flags;
  p.num_blocks = num_blocks;
  p.logits_stride = logits_stride;
  p.mode = kModePrefill;
  p.tps = (int32_t)(kMaxRows / num_heads);  // query tokens per segment
  p.next_n = p.tps;
  p.ngroups = 1;
  p.nseg = (int32_t)((num_tokens + p.tps - 1) / p.tps);
  p.num_q = (int32_t)num_tokens;
  p.H = (int32_t)num_heads;
  p.R = p.tps * p.H;
  p.ncols = (int32_t)num_keys;
  return launch(p, q_fp4, kv_cache, static_cast<cudaStream_t>(stream));
}

// The testing hook's scorer half (the C entry point, in fp4idx.cu, routes
// here): the next scorer launch withholds the copies of tile `index` of CTA 0.
namespace fp4idx_impl {
void scorer_withhold_next(int64_t index) { g_withhold.store(index); }
}  // namespace fp4idx_impl
