// fp4idx_common.cuh -- constants, PTX wrappers, arithmetic helpers and
// argument blocks shared by the pre-pass kernels (fp4idx.cu and
// fp4idx_stream.cu) and the host-buffer pipeline (fp4idx_host.cu).  Internal to the library; the public contract is
// include/fp4idx.h.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <utility>

#include <cuda_fp16.h>

#include "fp4idx.h"

namespace fp4idx_impl {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRowBytes = 256;
constexpr int kRopeHalf = FP4IDX_ROPE_DIM / 2;     // 32 cos/sin entries per row
constexpr int kKvBlock = FP4IDX_KV_BLOCK;
constexpr int kPageBytes = FP4IDX_PAGE_BYTES;
constexpr int kPayloadBytes = FP4IDX_SLOT_PAYLOAD_BYTES;
constexpr int kExpOffset = kKvBlock * kPayloadBytes;  // 4096
// FP8 output mode: slots of 128 E4M3 codes + a 4-byte fp32 scale, page-split
// (64 x 128 code bytes, then 64 scales).
constexpr int kFp8PageBytes = FP4IDX_FP8_PAGE_BYTES;             // 8448
constexpr int kFp8ScaleOffset = kKvBlock * FP4IDX_HEAD_DIM;      // 8192
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per stage wait

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Adds to the stage's expected byte count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Arrives (release): everything this thread wrote before is visible to a
// thread whose wait observes the completed phase.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for a stage with a time limit; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&w)[4]) {
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr));
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 ld_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// ---------------------------------------------------- arithmetic helpers
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// x / s rounded to nearest even, given rs = rn(1/s): q = rn(x * rs), the
// residual x - q*s (exact in one fma), then q + residual * rs rounded once
// (Markstein's correction of a reciprocal quotient, "IA-64 and Elementary
// Functions", 2000).  For every bf16 x and every positive E4M3 s (and for
// s = 6), the result equals the correctly rounded quotient; the GPU tests
// check all of those pairs against the IEEE division.
__device__ __forceinline__ float div_rcp(float x, float s, float rs) {
  const float q = __fmul_rn(x, rs);
  const float r = __fmaf_rn(-q, s, x);
  return __fmaf_rn(r, rs, q);
}

// The hardware's approximate reciprocal (rcp.approx.ftz.f32).  With it as
// rs, div_rcp still gives the correctly rounded x / s for the quantiser's
// operands (bf16 x, positive E4M3 s): the GPU tests check every such pair.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// (x0 / s, x1 / s) by div_rcp's three steps on f32x2 pairs (the residual as
// rn(q * -s + x), the same exact value).
__device__ __forceinline__ void div_rcp2(float& r0, float& r1, float x0, float x1, float s,
                                         float rs) {
  asm("{\n\t.reg .b64 rx, rr, rm, rq, rd, ro;\n\t"
      "mov.b64 rx, {%2, %3};\n\t"
      "mov.b64 rr, {%5, %5};\n\t"
      "mov.b64 rm, {%4, %4};\n\t"
      "mul.rn.f32x2 rq, rx, rr;\n\t"
      "fma.rn.f32x2 rd, rq, rm, rx;\n\t"
      "fma.rn.f32x2 ro, rd, rr, rq;\n\t"
      "mov.b64 {%0, %1}, ro;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(-s), "f"(rs));
}

// fp32 pair -> bf16x2 word (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// (r0, r1) = (a0*b0, a1*b1), each rounded to nearest even.  Used only where
// no addition consumes the products (the compiler may fuse a packed
// multiply with a following packed add).
__device__ __forceinline__ void mul2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (r0, r1) = (rn(a0*b0 + z), rn(a1*b1 + z)) with z = -0 supplied at run time:
// exactly the rounded products rn(a*b) (x + -0 = x, and +0 + -0 = +0).
// Because z is unknown to the compiler, the products can never be merged
// with a following addition into one fused operation.
__device__ __forceinline__ void prod2(float& r0, float& r1, float a0, float a1, float b0, float b1,
                                      float z) {
  asm("{\n\t.reg .b64 ra, rb, rz, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rz, {%6, %6};\n\t"
      "fma.rn.f32x2 rr, ra, rb, rz;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(z));
}

// (r0, r1) = (rn(a0+b0), rn(a1+b1)).
__device__ __forceinline__ void sum2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Per half: max(|a|, |b|) of two bf16 (sign bit = xor of the signs, ignored).
__device__ __forceinline__ uint32_t hmax_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t umin16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t uadd16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four fp32 values -> four E4M3 codes (round half to even, saturating at
// 448), element 0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint32_t w;
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
      "mov.b32 %0, {h0, h1};\n\t}"
      : "=r"(w)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return w;
}

// Eight fp32 values -> eight E2M1 nibbles (element 2k in the low nibble of
// byte k), round to nearest even, saturating at 6.  The conversion writes
// its first source operand to the high nibble.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
        "f"(v[7]));
  return w;
}
__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// ---------------------------------------------------------------- arguments
struct KArgs {
  const uint16_t* k;
  int64_t k_stride;
  const uint16_t* gamma;
  float eps;
  const int64_t* slots;
  uint8_t* cache;
  int64_t num_blocks;
  int meta_bulk;  // positions and slots 16-byte aligned: a full key item's
                  // positions/slots travel with its rows in the bulk copy
  int64_t pos_mask;  // ~(compress_ratio - 1): a key takes the RoPE of its
                     // group's first position, pos - pos % ratio
};

struct QArgs {
  const uint16_t* q;
  int64_t q_tstride;
  int64_t q_hstride;
  const uint16_t* w;
  int64_t w_tstride;
  float wscale;
  uint8_t* q_fp4;
  uint8_t* q_scale;
  float* weights;
  int64_t H;
};

struct Shared {
  const int64_t* pos;
  const float* cos;
  const float* sin;
  int64_t max_pos;
  int64_t T;
  uint32_t* err;
  float neg_zero;  // -0.0f, passed at run time (see prod2)
};

// Unsigned 32-bit division by a run-time invariant d >= 1 with one
// multiply-high and two shifts (Granlund and Montgomery, "Division by
// Invariant Integers using Multiplication", PLDI 1994, section 4):
//   l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
//   t = mulhi(m, n), q = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0).
struct FastDiv {
  uint32_t m, s1, s2;
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> s1)) >> s2;
  }
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 1 ? l - 1 : 0;
  return f;
}

}  // namespace fp4idx_impl

namespace fp4idx_impl {
// Launches kern on stream s and returns this launch's own status:
// cudaLaunchKernelEx reports its result directly, without reading or
// clearing an error that the caller's own work left in the runtime.
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(Params...), unsigned grid, unsigned block,
                                 size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The streaming kernel (fp4idx_stream.cu): every output mode, with or
// without the rotation; for queries a head count that is a multiple of 16.
bool stream_eligible(bool queries, int64_t H);
fp4idx_status launch_stream(const KArgs& ka, const QArgs& qa, const Shared& sh, bool keys,
                            bool queries, int rope_style, int rotate, int fp8, void* stream);
// The testing hook (fp4idx_test_withhold_next): the next launch of the
// streaming kernel, or of a scorer, withholds the copies of work item `index`
// of CTA 0 (a 64-row unit; a 128-key tile).
void stream_withhold_next(int64_t index);
void scorer_withhold_next(int64_t index);

// The host-side checks of fp4idx_indexer_prepass(_ex) without the launch
// (fp8: the FP8 output mode, where q_scale may be NULL).
fp4idx_status prepass_check(const void* k, int64_t k_token_stride, const void* gamma, float eps,
                            const int64_t* slot_mapping, const uint8_t* kv_cache,
                            int64_t num_blocks, const void* q, int64_t q_token_stride,
                            int64_t q_head_stride, const void* w, float weight_scale,
                            const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* weights_out, int64_t num_heads,
                            const int64_t* positions, const float* cos_cache,
                            const float* sin_cache, int64_t max_pos, int rope_style,
                            int64_t num_tokens, const uint32_t* err_flags, int fp8);
}  // namespace fp4idx_impl
