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
// Design.  A CTA (4 warps) owns one sequence b and a contiguous range of
// 128-token key tiles; a tile is two 64-slot cache pages.  The MMA has the
// keys as A (M = 128 tokens) and the sequence's R = next_n * H query rows as
// B (N = R), K = 128 as two MMAs of K = 64:
//   - the page payloads (64 tokens x 64 bytes) arrive by TMA tensor copies in
//     the 64-byte swizzled layout the MMA reads, and the exponent words by a
//     bulk copy, into a ring of stages (one mbarrier each);
//   - each exponent word is exactly one TMEM scale-factor cell: group g sits
//     in byte g, and the MMA over groups {0,1} takes bytes 0-1 (scale-factor
//     id 0), the one over {2,3} bytes 2-3 (id 2).  Row r's cell is TMEM
//     column base + r/32; the key side reads lane r, the query side lane
//     r%32 (written to every lane quadrant);
//   - the accumulator D[token, query row] (R fp32 columns) stays in TMEM;
//     thread t of the CTA owns token t of the tile (TMEM lane t) and forms
//     sum_h w * max(D, 0) for each of the next_n query tokens in registers,
//     so the head sum needs no data exchange between threads.
// Each E2M1 product is exact; the tensor core accumulates in fp32.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fp4idx.h"

namespace {

constexpr int kThreads = 128;          // 4 warps = the 128 TMEM lanes
constexpr int kTile = 128;             // key tokens per tile (MMA M)
constexpr int kKvBlock = FP4IDX_KV_BLOCK;
constexpr int kPageBytes = FP4IDX_PAGE_BYTES;
constexpr int kPayloadBytes = kKvBlock * FP4IDX_SLOT_PAYLOAD_BYTES;  // 4096
constexpr int kExpBytes = kKvBlock * FP4IDX_SLOT_EXP_BYTES;          // 256
constexpr int kStageA = 2 * kPayloadBytes;                           // 8192
constexpr int kStageE = 2 * kExpBytes;                               // 512
constexpr int kMaxRows = 128;          // query rows per sequence (MMA N)
constexpr int kMaxStages = 12;
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
  int32_t next_n;
  int32_t H;
  int32_t R;
  int32_t max_context;
  int32_t tiles;           // ceil(max_context / 128)
  int32_t tiles_per_cta;
  int32_t splits;          // CTAs per sequence
  int32_t stages;
  uint32_t tmem_cols;      // power of two >= R + 12
};

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
struct Layout {
  uint32_t a, b, e, w, bars, ok, tmem_slot, total;
};

__host__ __device__ inline Layout make_layout(int stages, int R) {
  Layout L;
  L.a = 0;                                              // stages x 8192, swizzled
  L.b = L.a + (uint32_t)stages * kStageA;               // R x 64, swizzled
  L.e = L.b + (uint32_t)R * 64;                         // stages x 512
  L.w = L.e + (uint32_t)stages * kStageE;               // R floats
  L.bars = (L.w + (uint32_t)R * 4 + 7u) & ~7u;          // stages + 1 mbarriers
  L.ok = L.bars + 8u * (uint32_t)(stages + 1);          // stages words
  L.tmem_slot = L.ok + 4u * (uint32_t)stages;
  L.total = L.tmem_slot + 4u;
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

// Waits for the phase with the given parity to complete; gives up after 1 s.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 16; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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

// -inf for every column of tiles [t0, t1) below max_context.
__device__ void write_padding(const ScorerParams& p, int b, int t0, int t1) {
  for (int t = t0; t < t1; ++t) {
    const int s = t * kTile + (int)threadIdx.x;
    if (s >= p.max_context) continue;
    for (int j = 0; j < p.next_n; ++j)
      p.logits[((int64_t)b * p.next_n + j) * p.logits_stride + s] = -INFINITY;
  }
}

__global__ void __launch_bounds__(kThreads) scorer_kernel(const __grid_constant__ ScorerParams p,
                                                          const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int b = blockIdx.x / p.splits;
  const int split = blockIdx.x - b * p.splits;
  const int t_lo = split * p.tiles_per_cta;
  const int t_hi = min(p.tiles, t_lo + p.tiles_per_cta);
  if (t_lo >= t_hi) return;  // uniform over the CTA
  const int ctx = min(max(__ldg(p.ctx_lens + b), 0), p.max_context);
  const int work_hi = min(t_hi, (ctx + kTile - 1) / kTile);  // tiles holding a token < ctx
  if (work_hi <= t_lo) {  // nothing to score: padding only
    write_padding(p, b, t_lo, t_hi);
    return;
  }
  const int nwork = work_hi - t_lo;

  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Layout L = make_layout(p.stages, p.R);
  uint8_t* const sA = smem + L.a;
  uint8_t* const sB = smem + L.b;
  uint8_t* const sE = smem + L.e;
  float* const sW = reinterpret_cast<float*>(smem + L.w);
  const uint32_t bars = smem_addr(smem + L.bars);  // full[0..S-1], then the MMA barrier
  const uint32_t mma_bar = bars + 8u * (uint32_t)p.stages;
  volatile uint32_t* const stage_ok = reinterpret_cast<volatile uint32_t*>(smem + L.ok);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);

  if (tid == 0) {
    for (int s = 0; s <= p.stages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * s) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t sfa_col = (uint32_t)p.R, sfb_col = (uint32_t)p.R + 8u;

  // Producer state (thread 0): tiles issued so far.
  int issued = 0;
  auto issue = [&](int k) {  // tile t_lo + k into stage k % S
    const int stage = k % p.stages;
    const int tile = t_lo + k;
    uint32_t okmask = 0, bytes = 0;
    int32_t page[2];
    for (int half = 0; half < 2; ++half) {
      const int pidx = tile * 2 + half;
      page[half] = -1;
      if (pidx * kKvBlock < ctx) {
        const int32_t id = __ldg(p.block_table + (int64_t)b * p.bt_stride + pidx);
        if (id >= 0 && id < p.num_blocks) {
          page[half] = id;
          okmask |= 1u << half;
          bytes += kPayloadBytes + kExpBytes;
        } else {
          flag_error(p.err, FP4IDX_ERRFLAG_PAGE);
        }
      }
    }
    stage_ok[stage] = okmask;
    const uint32_t bar = bars + 8u * stage;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    for (int half = 0; half < 2; ++half) {
      if (page[half] < 0) continue;
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
          "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(sA + stage * kStageA +
                                                            half * kPayloadBytes)),
          "l"(&tmap), "r"(0), "r"(0), "r"(page[half]), "r"(bar)
          : "memory");
      const uint8_t* src = p.cache + (int64_t)page[half] * kPageBytes + kPayloadBytes;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
          "[%3];" ::"r"(smem_addr(sE + stage * kStageE + half * kExpBytes)),
          "l"(src), "r"(kExpBytes), "r"(bar)
          : "memory");
    }
    issued = k + 1;
  };
  if (tid == 0)
    for (int k = 0; k < min(p.stages, nwork); ++k) issue(k);

  // Query rows of sequence b (rows b*R .. b*R+R-1 of q_fp4), their weights,
  // and their scale words (row 32j+i in column sfb_col+j, lane i of every
  // quadrant).
  const int64_t row0 = (int64_t)b * p.R;
  if (tid < p.R) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q_fp4 + (row0 + tid) * 64);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(sB + sw64_chunk(tid, c)) = __ldg(src + c);
    sW[tid] = __ldg(p.weights + row0 + tid);
  }
  {
    const int i = tid & 31;
    uint32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 32 * j + i;
      v[j] = r < p.R ? __ldg(reinterpret_cast<const uint32_t*>(p.q_scale) + row0 + r)
                     : 0x7F7F7F7Fu;
    }
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                     tmem + lane_base + sfb_col),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // sB -> tensor core

  const uint32_t id0 = mxf4_idesc(p.R, 0), id1 = mxf4_idesc(p.R, 2);
  const uint32_t a_base = smem_addr(sA), b_base = smem_addr(sB);
  float* const out0 = p.logits + (int64_t)b * p.next_n * p.logits_stride;
  bool failed = false, mma_pending = false;
  int k = 0;
  for (; k < nwork; ++k) {
    const int stage = k % p.stages;
    const uint32_t parity = (uint32_t)(k / p.stages) & 1u;
    const bool ok = mbar_wait_bounded(bars + 8u * stage, parity);
    uint32_t okmask = 0;
    if (ok) {
      okmask = stage_ok[stage];
      const uint32_t word = reinterpret_cast<const uint32_t*>(sE + stage * kStageE)[tid];
      asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(
                       tmem + lane_base + sfa_col + (uint32_t)warp),
                   "r"(word)
                   : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t a = a_base + (uint32_t)stage * kStageA;
      mma_mxf4(tmem, sw64_desc(a), sw64_desc(b_base), id0, tmem + sfa_col, tmem + sfb_col, 0u);
      mma_mxf4(tmem, sw64_desc(a + 32), sw64_desc(b_base + 32), id1, tmem + sfa_col,
               tmem + sfb_col, 1u);
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              mma_bar)
          : "memory");
    }
    mma_pending = true;
    const bool done = mbar_wait_bounded(mma_bar, (uint32_t)k & 1u);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (__syncthreads_or(!done)) {
      failed = true;
      break;
    }
    mma_pending = false;
    if (tid == 0 && k + p.stages < nwork) issue(k + p.stages);

    // Epilogue: token s of this thread, one logit per query token j.
    const int s = (t_lo + k) * kTile + tid;
    const bool valid = s < ctx && ((okmask >> (tid >> 6)) & 1u);
    for (int j = 0; j < p.next_n; ++j) {
      float2 acc = make_float2(0.0f, 0.0f);
      for (int c0 = j * p.H; c0 < (j + 1) * p.H; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + (uint32_t)c0, r);
        const float4* w4 = reinterpret_cast<const float4*>(sW + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 w = w4[i];
          const float2 x0 = make_float2(fmaxf(__uint_as_float(r[4 * i]), 0.0f),
                                        fmaxf(__uint_as_float(r[4 * i + 1]), 0.0f));
          const float2 x1 = make_float2(fmaxf(__uint_as_float(r[4 * i + 2]), 0.0f),
                                        fmaxf(__uint_as_float(r[4 * i + 3]), 0.0f));
          acc = fma2(make_float2(w.x, w.y), x0, acc);
          acc = fma2(make_float2(w.z, w.w), x1, acc);
        }
      }
      if (s < p.max_context)
        out0[(int64_t)j * p.logits_stride + s] = valid ? __fadd_rn(acc.x, acc.y) : -INFINITY;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  }

  if (failed) {
    // Let every copy and the MMA in flight land before the CTA's shared
    // memory and TMEM are released.  The logits of this CTA's remaining
    // tiles are left unwritten.
    if (tid == 0) {
      flag_error(p.err, FP4IDX_ERRFLAG_TIMEOUT);
      for (int q = k; q < issued; ++q)
        mbar_wait_bounded(bars + 8u * (q % p.stages), (uint32_t)(q / p.stages) & 1u);
      if (mma_pending) mbar_wait_bounded(mma_bar, (uint32_t)k & 1u);
    }
  } else {
    write_padding(p, b, work_hi, t_hi);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(p.tmem_cols)
                 : "memory");
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

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int smem_per_sm = 0;
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
        cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return FP4IDX_ERR_CUDA;
    if (cudaFuncSetAttribute(scorer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  p.next_n = (int32_t)next_n;
  p.H = (int32_t)num_heads;
  p.R = (int32_t)(next_n * num_heads);
  p.max_context = (int32_t)max_context;
  p.tiles = (int32_t)((max_context + kTile - 1) / kTile);
  uint32_t cols = 32;
  while (cols < (uint32_t)p.R + 12u) cols <<= 1;
  p.tmem_cols = cols;

  // Stages: the fewest (>= 4) with which shared memory, not TMEM, limits the
  // CTAs resident on an SM to what TMEM (512 columns) can hold at once.
  const int tmem_ctas = 512 / (int)cols;
  const int reserve = 1024;  // per-CTA shared memory the system keeps
  int stages = 4;
  for (;; ++stages) {
    const int bytes = (int)make_layout(stages, p.R).total + 1024;  // + base alignment
    if (bytes > di.smem_optin) {
      --stages;
      break;
    }
    if (di.smem_per_sm / (bytes + reserve) <= tmem_ctas || stages == kMaxStages) break;
  }
  if (stages < 2) return FP4IDX_ERR_SHAPE;
  p.stages = stages;
  const int smem_bytes = (int)make_layout(stages, p.R).total + 1024;
  int ctas = di.smem_per_sm / (smem_bytes + reserve);
  if (ctas > tmem_ctas) ctas = tmem_ctas;
  if (ctas < 1) ctas = 1;

  // Split each sequence's tiles so that the grid covers about four waves.
  const int64_t want = (int64_t)di.sms * ctas * 4;
  int64_t per = (batch * p.tiles + want - 1) / want;
  if (per < 1) per = 1;
  p.tiles_per_cta = (int32_t)per;
  p.splits = (int32_t)((p.tiles + per - 1) / per);
  const int64_t grid = batch * p.splits;
  if (grid >= (1ll << 31)) return FP4IDX_ERR_SHAPE;

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

  scorer_kernel<<<(unsigned)grid, kThreads, smem_bytes, static_cast<cudaStream_t>(stream)>>>(p,
                                                                                            tmap);
  return cudaGetLastError() == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}
