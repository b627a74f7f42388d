// fp4idx_scorer.cu -- FP4 paged MQA-logits scorer on the block-scaled FP4
// tensor cores of sm_103a (tcgen05.mma kind::mxf4).  It consumes the bytes
// the pre-pass writes: packed E2M1 queries with their per-32 UE8M0 exponent
// words, and the paged 68-byte index-K slots.  The operation and the argument
// contract are in include/fp4idx.h.
//
// Sources (web pages, by title and section):
//   "[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR
//   5484), Verification: the paged FP4 MQA-logits scorer reads the packed
//   E2M1 keys and their e8m0 block exponents straight from the paged cache,
//   at GLM-5.2 shapes (H = 32, D = 128, kv_block = 64) with next_n 1 and 4.
//   "[ROCm][Perf] Enabled FP4Indexer for DSV4" (vLLM PR 42908), Code Review:
//   the score of a key is the block-scaled E2M1 dot product with each query
//   head, through ReLU, times the head weight, summed over the heads.
//   "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656), Summary: the
//   68-byte slot (64 payload bytes + 4 exponent bytes).
//
// Work.  A tile is 128 consecutive tokens (two 64-slot pages) of one
// sequence; only tiles holding a token below the sequence's context are
// work.  The persistent grid splits the list of all work tiles (sequence by
// sequence) into equal contiguous shares, one per CTA, from the context
// lengths alone; a CTA's share may span several sequences ("segments").
// Logits of tiles past the context are -inf, written in a final phase.
//
// MMA.  Keys are A (M = 128 tokens), the sequence's R = next_n * H query rows
// are B (N = R), K = 128 as two MMAs of K = 64.  Each exponent word of a slot
// is exactly one TMEM scale-factor cell: group g sits in byte g; the MMA over
// groups {0,1} takes bytes 0-1 (scale-factor id 0), the one over {2,3} bytes
// 2-3 (id 2).  Row r's cell is TMEM column base + r/32; the key side reads
// lane r, the query side lane r%32 (written to every lane quadrant).
//
// Roles (17 + P warps, P = kProducers producer warps).
//   producers (warps 16 .. 16+P-1): TMA tensor copies of the page payloads
//     (64 tokens x 64 bytes, in the 64-byte swizzled layout the MMA reads)
//     and bulk copies of the exponent words into a ring of S stages;
//     producer i issues tiles i, i+P, ...; each warp fetches the page ids
//     of 16 of its tiles per load, one batch ahead;
//   MMA issuer (warp 16+P): per tile it waits for the data and for a free
//     accumulator, stages the keys' exponent words (and, at the first tile
//     of a segment, the segment's query operand and query scale words) in
//     shared memory as a 32 x 128-bit transpose, and lane 0 issues
//     tcgen05.cp of those words into the scale-factor columns of TMEM, the
//     two MMAs into accumulator k % 3 and the commits -- all in order in
//     the tensor pipe, so no thread waits for the copies;
//   two epilogue groups of 8 warps (0-7, 8-15), group e owning the tiles k
//     with k % 2 == e.  Warps q and q+4 of a group share TMEM lane quadrant q
//     and split the accumulator's 32-column chunks.  Per tile a warp reads
//     its chunks one at a time (thread = token = TMEM lane), releases the
//     accumulator (acc_empty) and stores sum_h w * max(D, 0) per query
//     token; a page's validity comes from the block table, fetched a tile
//     ahead.  Each warp holds its own copy of the segment's head weights.
// Every wait is bounded (1 s) and a shared abort flag stops every role; in
// flight copies and MMAs are waited for before TMEM and shared memory are
// released.  Each E2M1 product is exact; the tensor core accumulates in fp32.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fp4idx.h"

namespace {

constexpr int kEpiWarps = 16;                // two groups of eight
constexpr int kGroupWarps = 8;
#ifndef FP4IDX_SCORER_PRODUCERS
#define FP4IDX_SCORER_PRODUCERS 1
#endif
constexpr int kProducers = FP4IDX_SCORER_PRODUCERS;  // producer warps
constexpr int kProducerWarp = 16;                    // the first of them
constexpr int kMmaWarp = kProducerWarp + kProducers;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kMaxNext = 4;                  // next_n <= kMaxRows / 32
constexpr int kAccs = 3;                     // TMEM accumulators (tile k: k % 3)
constexpr int kQBufs = 4;                    // query operands (segment g: g % 4)
constexpr int kTile = 128;                   // key tokens per tile (MMA M)
constexpr int kKvBlock = FP4IDX_KV_BLOCK;
constexpr int kPageBytes = FP4IDX_PAGE_BYTES;
constexpr int kPayloadBytes = kKvBlock * FP4IDX_SLOT_PAYLOAD_BYTES;  // 4096
constexpr int kExpBytes = kKvBlock * FP4IDX_SLOT_EXP_BYTES;          // 256
constexpr int kStageA = 2 * kPayloadBytes;                           // 8192
constexpr int kStageE = 2 * kExpBytes;                               // 512
constexpr int kMaxRows = 128;                // query rows per sequence (MMA N)
constexpr int kMaxStages = 16;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

struct ScorerParams {
  const uint8_t* q_fp4;
  const uint8_t* q_scale;
  const float* weights;
  const uint8_t* cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  float* logits;
  uint32_t* err;
  int64_t num_blocks;
  int64_t bt_stride;
  int64_t logits_stride;
  int32_t batch;
  int32_t next_n;
  int32_t H;
  int32_t R;
  int32_t max_context;
  int32_t tiles_total;     // ceil(max_context / 128) tiles per sequence
  int32_t stages;
  uint32_t tmem_cols;      // power of two >= 3R + 40
};

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
struct Layout {
  uint32_t a, q, e, w, x, sf, bars, ok, misc, scan, total;
};

// Barrier indices: full[S], empty[S], then the ones below.
__host__ __device__ inline int bar_full(int s) { return s; }
__host__ __device__ inline int bar_empty(int S, int s) { return S + s; }
// acc_full[k % 6]: the MMAs of tile k are complete.  Tile k uses accumulator
// k % 3 and belongs to group k % 2, so each of the six barriers is waited on
// by one group only, one phase after another.
__host__ __device__ inline int bar_accf(int S, int k6) { return 2 * S + k6; }
// acc_empty[a]: the group that read accumulator a has its values (8 arrivals).
__host__ __device__ inline int bar_acce(int S, int a) { return 2 * S + 6 + a; }
// Partial-sum hand-off between the two warps of a lane quadrant (group e,
// quadrant q, buffer b), used when a query token's heads span both halves.
__host__ __device__ inline int bar_xch(int S, int e, int q, int b) {
  return 2 * S + 9 + (e * 4 + q) * 2 + b;
}
constexpr int kExtraBars = 6 + 3 + 16;

__host__ __device__ inline Layout make_layout(int S, int R) {
  Layout L;
  L.a = 0;                                     // S x 8192, swizzled payloads
  L.q = L.a + (uint32_t)S * kStageA;           // 4 x R x 64, swizzled queries
  L.e = L.q + (uint32_t)kQBufs * R * 64;       // S x 512 exponent words
  L.w = L.e + (uint32_t)S * kStageE;           // 16 epilogue warps x R weights
  L.x = L.w + (uint32_t)kEpiWarps * R * 4;     // partial sums: 2 groups x 2 x next_n x 128
  L.sf = L.x + 2u * 2u * kMaxNext * kTile * 4u;  // scale-word copy sources
  L.bars = L.sf + (uint32_t)(kAccs + kQBufs) * 512u;  // 2S + extra mbarriers
  L.ok = L.bars + 8u * (uint32_t)(2 * S + kExtraBars);
  L.misc = L.ok;                               // tmem base, abort, b/t/n start
  L.scan = L.misc + 32;                        // kThreads + 1 partial sums (int64)
  L.total = L.scan + 8u * (kThreads + 1);
  return L;
}

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

// The same wait with no abort flag: used while draining after an abort.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

// Byte offset of 16-byte chunk c of row r in the 64-byte swizzled layout.
__device__ __forceinline__ uint32_t sw64_chunk(int r, int c) {
  return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
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

__device__ __forceinline__ int ctx_eff(const ScorerParams& p, int b) {
  return min(max(__ldg(p.ctx_lens + b), 0), p.max_context);
}

__device__ __forceinline__ int work_tiles(int ctx) { return (ctx + kTile - 1) / kTile; }

// Chunks [C0, C1) of an accumulator (this thread's TMEM lane, 32 columns
// each), one chunk in registers at a time: part[c - C0] = sum over chunk c's
// columns of w * max(D, 0).  Returns once every TMEM load has completed.
template <int C0, int C1>
struct HalfAcc {
  __device__ __forceinline__ void run(uint32_t acc, const float* wts, float* part) const {
#pragma unroll
    for (int c = C0; c < C1; ++c) {
      uint32_t r[32];
      tmem_ld32(acc + 32u * c, r);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      // two independent packed chains, then a fixed combining order
      float2 a0 = make_float2(0.0f, 0.0f), a1 = a0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 ww = reinterpret_cast<const float4*>(wts + 32 * c)[i];
        const uint32_t* x = r + 4 * i;
        a0 = fma2(make_float2(ww.x, ww.y),
                  make_float2(fmaxf(__uint_as_float(x[0]), 0.0f),
                              fmaxf(__uint_as_float(x[1]), 0.0f)),
                  a0);
        a1 = fma2(make_float2(ww.z, ww.w),
                  make_float2(fmaxf(__uint_as_float(x[2]), 0.0f),
                              fmaxf(__uint_as_float(x[3]), 0.0f)),
                  a1);
      }
      part[c - C0] = __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y));
    }
  }
};

template <int C0, int C1>
struct HalfAccT : HalfAcc<C0, C1> {
  static constexpr int kC0 = C0, kC1 = C1;
};

// Walks a CTA's tiles in order: sequence b, tile t, its context, and the
// segment index g (how many times b has changed since the first tile).
struct Walker {
  int b, t, ctx, g;
  __device__ void init(const ScorerParams& p, int b0, int t0) {
    b = b0;
    t = t0;
    ctx = ctx_eff(p, b0);
    g = 0;
  }
  __device__ void advance(const ScorerParams& p) {
    ++t;
    while (t >= work_tiles(ctx) && b + 1 < p.batch) {
      ++b;
      t = 0;
      ctx = ctx_eff(p, b);
      ++g;
    }
  }
};

template <int NCHUNK>
__global__ void __launch_bounds__(kThreads, 1)
    scorer_kernel(const __grid_constant__ ScorerParams p, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.stages, R = p.R;
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Layout L = make_layout(S, R);
  uint8_t* const sA = smem + L.a;
  uint8_t* const sQ = smem + L.q;
  uint8_t* const sE = smem + L.e;
  float* const sW = reinterpret_cast<float*>(smem + L.w);
  const uint32_t bars = smem_addr(smem + L.bars);
  uint32_t* const misc = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile uint32_t* const abort = misc + 1;
  int32_t* const start = reinterpret_cast<int32_t*>(misc + 2);  // b, t, n
  long long* const scan = reinterpret_cast<long long*>(smem + L.scan);
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  // ---- this CTA's share of the work tiles --------------------------------
  const int per = (p.batch + kThreads - 1) / kThreads;
  const int b_lo = min(p.batch, tid * per), b_hi = min(p.batch, b_lo + per);
  long long part = 0;
  for (int b = b_lo; b < b_hi; ++b) part += work_tiles(ctx_eff(p, b));
  scan[tid] = part;
  if (tid == 0) {
    *abort = 0u;
    start[2] = 0;
  }
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int i = 0; i < kThreads; ++i) {
      const long long v = scan[i];
      scan[i] = run;
      run += v;
    }
    scan[kThreads] = run;
  }
  __syncthreads();
  const long long W = scan[kThreads];
  const long long lo = W * blockIdx.x / gridDim.x, hi = W * (blockIdx.x + 1) / gridDim.x;
  if (lo < hi && scan[tid] <= lo && lo < scan[tid] + part) {
    long long acc = scan[tid];
    for (int b = b_lo; b < b_hi; ++b) {
      const int wt = work_tiles(ctx_eff(p, b));
      if (lo < acc + wt) {
        start[0] = b;
        start[1] = (int)(lo - acc);
        start[2] = (int)(hi - lo);
        break;
      }
      acc += wt;
    }
  }
  __syncthreads();
  const int n = start[2];

  if (n > 0) {
    const int b0 = start[0], t0 = start[1];
    if (tid == 0) {
      for (int i = 0; i < 2 * S + kExtraBars; ++i) {
        // acc_empty takes one arrival per epilogue warp of a group
        const int cnt = (i >= bar_acce(S, 0) && i < bar_acce(S, kAccs)) ? kGroupWarps : 1;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar(i)), "r"(cnt)
                     : "memory");
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_addr(misc)),
                   "r"(p.tmem_cols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = misc[0];
    // TMEM columns: accumulators [0, R) and [R, 2R); key scale words of
    // group e at 2R + 8e; query scale words of segment g at 2R + 16 + 8(g%2).
    // TMEM columns: accumulator a at aR (a < 3); the keys' scale words of
    // accumulator a's tile at 3R + 8a; the query scale words of segment g at
    // 3R + 24 + 8(g%4).
    const uint32_t sfa_col0 = (uint32_t)kAccs * R, sfb_col0 = (uint32_t)kAccs * R + 24u;
    uint8_t* const sSF = smem + L.sf;  // copy sources: 3 key + 4 query, 512 B each
    int issued = 0;  // producer: tiles whose copies were issued

    if (warp >= kProducerWarp && warp < kMmaWarp) {
      // Producer pi issues the tiles k = pi, pi + kProducers, ... and so owns
      // the stages s = k % S (S is a multiple of kProducers).  A warp waits a
      // few hundred cycles for each copy it issues, so the copies are spread
      // over several warps.  The page ids of 16 of its tiles are fetched by
      // the whole warp in one load (lane L: own tile L/2, page L%2), a batch
      // ahead of the tiles issued.
      const int pi = warp - kProducerWarp;
      const int n_own = n > pi ? (n - pi + kProducers - 1) / kProducers : 0;
      Walker fw;  // at tile fk
      fw.init(p, b0, t0);
      int fk = 0;
      auto fetch = [&](int m0, int32_t& id, bool& inctx) {
        const int mine = lane >> 1;
        int cb = 0, ct = 0, cctx = 0;
        for (int i = 0; i < 16 && m0 + i < n_own; ++i) {
          const int k = pi + kProducers * (m0 + i);
          while (fk < k) {
            fw.advance(p);
            ++fk;
          }
          if (i == mine) {
            cb = fw.b;
            ct = fw.t;
            cctx = fw.ctx;
          }
        }
        const int pidx = ct * 2 + (lane & 1);
        inctx = m0 + mine < n_own && pidx * kKvBlock < cctx;
        id = inctx ? __ldg(p.block_table + (int64_t)cb * p.bt_stride + pidx) : -1;
      };
      int32_t cur_id, nxt_id = -1;
      bool cur_in, nxt_in = false;
      fetch(0, cur_id, cur_in);
      bool stop = false;
      for (int m0 = 0; m0 < n_own && !stop; m0 += 16) {
        if (m0 + 16 < n_own) fetch(m0 + 16, nxt_id, nxt_in);
        for (int i = 0; i < 16 && m0 + i < n_own; ++i) {
          const int k = pi + kProducers * (m0 + i), s = k % S;
          int32_t page[2];
          bool in[2];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            page[half] = __shfl_sync(0xffffffffu, cur_id, 2 * i + half);
            in[half] = __shfl_sync(0xffffffffu, (int)cur_in, 2 * i + half) != 0;
          }
          int ok = 1;
          if (lane == 0) {
            ok = wait_phase(bar(bar_empty(S, s)), ((uint32_t)(k / S) & 1u) ^ 1u, abort);
            if (ok) {
              uint32_t bytes = 0;
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                if (!in[half]) {
                  page[half] = -1;
                } else if (page[half] < 0 || page[half] >= p.num_blocks) {
                  flag_error(p.err, FP4IDX_ERRFLAG_PAGE);
                  page[half] = -1;
                } else {
                  bytes += kPayloadBytes + kExpBytes;
                }
              }
              const uint32_t fb = bar(bar_full(s));
              asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                           "r"(bytes)
                           : "memory");
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                if (page[half] < 0) continue;
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
                    "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(sA + s * kStageA +
                                                                      half * kPayloadBytes)),
                    "l"(&tmap), "r"(0), "r"(0), "r"(page[half]), "r"(fb)
                    : "memory");
                const uint8_t* src = p.cache + (int64_t)page[half] * kPageBytes + kPayloadBytes;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
                    "[%1], %2, [%3];" ::"r"(smem_addr(sE + s * kStageE + half * kExpBytes)),
                    "l"(src), "r"(kExpBytes), "r"(fb)
                    : "memory");
              }
              issued = k + 1;
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            stop = true;
            break;
          }
        }
        cur_id = nxt_id;
        cur_in = nxt_in;
      }
    } else if (warp == kMmaWarp) {
      // The whole warp waits (a warp-uniform loop wakes promptly) and stages
      // the scale words; lane 0 issues the copies into TMEM, the MMAs and the
      // commits, in that order in the tensor pipe.
      Walker wk;
      wk.init(p, b0, t0);
      const uint32_t id0 = mxf4_idesc(R, 0), id1 = mxf4_idesc(R, 2);
      // descriptor start addresses advance in 16-byte units
      const uint64_t a_desc0 = sw64_desc(smem_addr(sA)), q_desc0 = sw64_desc(smem_addr(sQ));
      int done = 0;
      for (int k = 0; k < n; ++k) {
        const int s = k % S, a = k % kAccs, gq = wk.g % kQBufs;
        // Tile k's data, and accumulator a free again: tile k-3 read out,
        // which also means every MMA up to tile k-3 -- and the copies and
        // operands those MMAs used -- is complete.
        bool ok = wait_phase(bar(bar_full(s)), (uint32_t)(k / S) & 1u, abort) &&
                  (k < kAccs ||
                   wait_phase(bar(bar_acce(S, a)), (uint32_t)(k / kAccs - 1) & 1u, abort));
        if (!__all_sync(0xffffffffu, ok)) break;
        const bool seg_start = k == 0 || wk.t == 0;
        if (seg_start) {
          // The segment's query operand and query scale words.  Buffer gq was
          // last used by segment g-4, whose tiles all precede tile k-3.
          const int64_t row0 = ((int64_t)wk.b * p.next_n) * p.H;  // first query row of b
          uint8_t* dst = sQ + gq * R * 64;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = lane + 32 * i;
            if (r < R) {
              const uint4* src = reinterpret_cast<const uint4*>(p.q_fp4 + (row0 + r) * 64);
#pragma unroll
              for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(dst + sw64_chunk(r, c)) = __ldg(src + c);
            }
          }
          uint32_t v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 32 * j + lane;
            v[j] = r < R ? __ldg(reinterpret_cast<const uint32_t*>(p.q_scale) + row0 + r)
                         : 0x7F7F7F7Fu;
          }
          *reinterpret_cast<uint4*>(sSF + (kAccs + gq) * 512 + 16 * lane) =
              make_uint4(v[0], v[1], v[2], v[3]);
        }
        {  // the keys' exponent words, token 32c + l at row l, column c
          const uint32_t* ew = reinterpret_cast<const uint32_t*>(sE + s * kStageE);
          *reinterpret_cast<uint4*>(sSF + a * 512 + 16 * lane) =
              make_uint4(ew[lane], ew[lane + 32], ew[lane + 64], ew[lane + 96]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (lane == 0) {
          const uint32_t sfa = tmem + sfa_col0 + 8u * (uint32_t)a;
          const uint32_t sfb = tmem + sfb_col0 + 8u * (uint32_t)gq;
          cp_32x128b_x4(sfa, cp_desc(smem_addr(sSF + a * 512)));
          if (seg_start) cp_32x128b_x4(sfb, cp_desc(smem_addr(sSF + (kAccs + gq) * 512)));
          const uint64_t adesc = a_desc0 + (uint64_t)(s * (kStageA >> 4));
          const uint64_t qdesc = q_desc0 + (uint64_t)(gq * R * (64 >> 4));
          const uint32_t d = tmem + (uint32_t)a * (uint32_t)R;
          mma_mxf4(d, adesc, qdesc, id0, sfa, sfb, 0u);
          mma_mxf4(d, adesc + 2, qdesc + 2, id1, sfa, sfb, 1u);
          mma_commit(bar(bar_accf(S, k % 6)));
          mma_commit(bar(bar_empty(S, s)));
        }
        __syncwarp();
        done = k + 1;
        wk.advance(p);
      }
      if (done > 0 && lane == 0)  // the last commits land before the memory is released
        wait_phase_drain(bar(bar_empty(S, (done - 1) % S)), (uint32_t)((done - 1) / S) & 1u);
    } else {
      // ---- epilogue group e (warps 8e .. 8e+7): tiles k = e, e+2, ... --------
      // Warps q and q+4 of a group share TMEM lane quadrant q (tokens
      // 32q .. 32q+31) and split the accumulator's 32-column chunks: the
      // lower half takes chunks [0, kC1), the upper half [kC1, NCHUNK).  Per
      // tile a warp reads and reduces its chunks, releases the accumulator
      // (acc_empty) and stores the logits.
      constexpr int kC1 = (NCHUNK + 1) / 2;
      const int e = warp / kGroupWarps, gw = warp % kGroupWarps;
      const int quad = gw & 3, half = gw >> 2;
      const int row = quad * 32 + lane;  // token of the tile = TMEM lane
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      float* const wts = sW + warp * R;  // this warp's head weights
      float* const xch = reinterpret_cast<float*>(smem + L.x) + e * 2 * kMaxNext * kTile;
      const int cpj = p.H / 32;          // chunks per query token
      // a query token whose heads span both halves (its partial sums are
      // handed from the upper to the lower warp through shared memory)
      const bool split = kC1 < NCHUNK && kC1 % cpj != 0;
      const int js = kC1 / cpj;

      // The validity of this warp's page of tile (w.b, w.t) -- the same rule
      // the producer applies: inside the context and a page id in range.
      auto page_id = [&](const Walker& w) -> int32_t {
        const int pidx = w.t * 2 + (quad >> 1);
        return pidx * kKvBlock < w.ctx
                   ? __ldg(p.block_table + (int64_t)w.b * p.bt_stride + pidx)
                   : -1;
      };

      // Tile k, chunks [C0, C1) of accumulator k % 3: load and reduce chunk
      // by chunk, release the accumulator, store (or hand off) the logits.
      auto tile = [&](auto acc, int k, const Walker& w, bool page_ok, bool& live) {
        constexpr int C0 = decltype(acc)::kC0, C1 = decltype(acc)::kC1;
        const int a = k % kAccs;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        float part[C1 > C0 ? C1 - C0 : 1];
        acc.run(tmem + lane_base + (uint32_t)a * (uint32_t)R, wts, part);
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bar_acce(S, a)));
        const int s_tok = w.t * kTile + row;
        const bool valid = s_tok < w.ctx && page_ok;
        float* const xb = xch + ((k >> 1) & 1) * kMaxNext * kTile;
        const uint32_t xbar = bar(bar_xch(S, e, quad, (k >> 1) & 1));
        float* const out = p.logits + ((int64_t)w.b * p.next_n) * p.logits_stride + s_tok;
#pragma unroll
        for (int j = 0; j < kMaxNext; ++j) {
          if (j >= p.next_n) break;
          float v = 0.0f;
          bool any = false;
#pragma unroll
          for (int c = C0; c < C1; ++c)
            if (c / cpj == j) {
              v = any ? __fadd_rn(v, part[c - C0]) : part[c - C0];
              any = true;
            }
          if (split && j == js) {
            if (half == 1) {  // hand the upper part to the lower warp
              xb[j * kTile + row] = v;
              __syncwarp();
              if (lane == 0) mbar_arrive(xbar);
              continue;
            }
            if (!__all_sync(0xffffffffu, wait_phase(xbar, (uint32_t)(k >> 2) & 1u, abort))) {
              live = false;
              return;
            }
            v = __fadd_rn(v, xb[j * kTile + row]);
          } else if (!any) {
            continue;
          }
          if (s_tok < p.max_context) out[(int64_t)j * p.logits_stride] = valid ? v : -INFINITY;
        }
      };

      Walker wk;
      wk.init(p, b0, t0);
      if (e == 1) wk.advance(p);
      Walker nw = wk;
      nw.advance(p);
      nw.advance(p);
      int32_t pid = e < n ? page_id(wk) : -1, pid_next = -1;
      bool live = true;
      int wg = -1;  // segment of the weights held
      for (int k = e; k < n && live; k += 2) {
        if (k + 2 < n) pid_next = page_id(nw);  // a tile ahead
        if (!__all_sync(0xffffffffu,
                        wait_phase(bar(bar_accf(S, k % 6)), (uint32_t)(k / 6) & 1u, abort)))
          break;
        if (wk.g != wg) {  // this warp's copy of the segment's head weights
          const int64_t row0 = ((int64_t)wk.b * p.next_n) * p.H;
          for (int i = lane; i < R; i += 32) wts[i] = __ldg(p.weights + row0 + i);
          __syncwarp();
          wg = wk.g;
        }
        const bool page_ok = pid >= 0 && pid < p.num_blocks;
        if (half == 0)
          tile(HalfAccT<0, kC1>(), k, wk, page_ok, live);
        else
          tile(HalfAccT<kC1, NCHUNK>(), k, wk, page_ok, live);
        pid = pid_next;
        wk = nw;
        nw.advance(p);
        nw.advance(p);
      }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (*abort) {  // every role has stopped: let copies in flight land first
      if (warp >= kProducerWarp && warp < kMmaWarp && lane == 0)  // its own stages
        for (int q = issued - 1; q >= 0 && q >= issued - S; q -= kProducers)
          wait_phase_drain(bar(bar_full(q % S)), (uint32_t)(q / S) & 1u);
      if (tid == 0) flag_error(p.err, FP4IDX_ERRFLAG_TIMEOUT);
      __syncthreads();
    }
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(p.tmem_cols)
                   : "memory");
  }

  // ---- -inf for tiles past each context, spread over the grid's warps ------
  const long long items = (long long)p.batch * p.tiles_total;
  const int gwarps = gridDim.x * (kThreads / 32);
  for (long long it = (long long)blockIdx.x * (kThreads / 32) + warp; it < items; it += gwarps) {
    const int b = (int)(it / p.tiles_total), t = (int)(it % p.tiles_total);
    if (t < work_tiles(ctx_eff(p, b))) continue;
    for (int j = 0; j < p.next_n; ++j) {
      float* out = p.logits + ((int64_t)b * p.next_n + j) * p.logits_stride;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int s = t * kTile + 32 * m + lane;
        if (s < p.max_context) out[s] = -INFINITY;
      }
    }
  }
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    tried = true;
  }
  return fn;
}

typedef void (*ScorerKernel)(ScorerParams, CUtensorMap);

ScorerKernel kernel_for(int nchunk) {
  switch (nchunk) {
    case 1: return scorer_kernel<1>;
    case 2: return scorer_kernel<2>;
    case 3: return scorer_kernel<3>;
    default: return scorer_kernel<4>;
  }
}

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
};

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
  if (next_n < 1 || num_heads < 32 || num_heads % 32 != 0 || next_n * num_heads > kMaxRows ||
      num_blocks < 1 || num_blocks >= (1ll << 31) || max_context >= (1 << 30) ||
      batch >= (1 << 30) || logits_stride < max_context ||
      block_table_stride < (max_context + kKvBlock - 1) / kKvBlock)
    return FP4IDX_ERR_SHAPE;
  if (!aligned(q_fp4, 16) || !aligned(q_scale, 4) || !aligned(weights, 4) ||
      !aligned(kv_cache, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4) ||
      !aligned(logits, 4) || (err_flags && !aligned(err_flags, 4)))
    return FP4IDX_ERR_ALIGN;

  static DeviceInfo info[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4IDX_ERR_CUDA;
  DeviceInfo& di = info[dev];
  if (!di.ready) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return FP4IDX_ERR_CUDA;
    for (int c = 1; c <= 4; ++c)
      if (cudaFuncSetAttribute(kernel_for(c), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               di.smem_optin) != cudaSuccess)
        return FP4IDX_ERR_CUDA;
    di.ready = true;
  }
  EncodeTiledFn encode = encode_fn();
  if (encode == nullptr) return FP4IDX_ERR_CUDA;

  ScorerParams p;
  p.q_fp4 = q_fp4;
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
  p.batch = (int32_t)batch;
  p.next_n = (int32_t)next_n;
  p.H = (int32_t)num_heads;
  p.R = (int32_t)(next_n * num_heads);
  p.max_context = (int32_t)max_context;
  p.tiles_total = (int32_t)((max_context + kTile - 1) / kTile);
  uint32_t cols = 32;
  while (cols < (uint32_t)kAccs * (uint32_t)p.R + 24u + 8u * kQBufs) cols <<= 1;
  p.tmem_cols = cols;
  // As many stages as fit in one CTA's shared memory (one CTA per SM).
  int S = kMaxStages - kMaxStages % kProducers;  // a multiple of the producer count
  while (S > kProducers && (int)make_layout(S, p.R).total + 1024 > di.smem_optin)
    S -= kProducers;
  if ((int)make_layout(S, p.R).total + 1024 > di.smem_optin) return FP4IDX_ERR_SHAPE;
  p.stages = S;
  const int smem_bytes = (int)make_layout(S, p.R).total + 1024;

  // The cache as a 3-D byte tensor: 64 payload bytes x 64 slots x pages.
  alignas(64) CUtensorMap tmap;
  const cuuint64_t gdim[3] = {64, 64, (cuuint64_t)num_blocks};
  const cuuint64_t gstride[2] = {64, (cuuint64_t)kPageBytes};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(kv_cache), gdim,
             gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return FP4IDX_ERR_CUDA;

  kernel_for(p.R / 32)<<<(unsigned)di.sms, kThreads, smem_bytes,
                          static_cast<cudaStream_t>(stream)>>>(p, tmap);
  return cudaGetLastError() == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}
