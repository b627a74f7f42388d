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
// Mapping onto the GPU.  A half-warp owns one 128-element row: lane j holds
// elements 8j..8j+7 as one 16-byte load, so a 32-element quantisation group
// is four adjacent lanes and the group amax is two xor-shuffles.  Each lane
// then produces one 32-bit word of eight nibbles, so the 64-byte payload of a
// row is one coalesced 64-byte store per half-warp (128 bytes per warp).
// Queries are processed one token per CTA iteration (the RoPE coefficients
// are loaded once per token and reused for all heads); each half-warp keeps
// four 256-byte rows in flight.  Keys are one row per half-warp.
//
// Bit-exactness.  Every fp32 step uses an explicit round-to-nearest
// intrinsic (__fmul_rn, __fadd_rn, __fsqrt_rn, __frcp_rn), which the compiler
// never fuses into FMA, and the build keeps subnormals (no FTZ).
//
// Quantisation shortcut (derived from the two-stage definition):
//   * stage-1 exponent: for a bf16 amax A = 1.m * 2^(E-127) (E its biased
//     exponent field), ceil_pow2(A/6) = 2^(E-129) if 1.m <= 1.5 and 2^(E-128)
//     otherwise; A/6 rounded to fp32 never crosses a power of two for a bf16
//     A, so e1 = max(E - 2 + (mantissa > 0x400000), 1) without a division.
//   * stage-1 codes: the hardware e2m1x2 conversion rounds to nearest even
//     and saturates, i.e. exactly the grid rule; it may emit -0 codes, which
//     are cleared at the end.
//   * stage 2: with e1 > 1 the stage-1 top code is 5, 6 or 7.  If it is 5
//     (3.0, i.e. A*2^(127-e1) < 3.5) stage 2 halves the scale (e2 = e1 - 1)
//     and every code m <= 5 maps exactly to the code of 2*grid[m], which is
//     m + min(m, 2); otherwise (and whenever e1 == 1, where the floor holds)
//     stage 2 reproduces stage 1.  The dequantised values never change.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fp4idx.h"

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;             // 8 warps = 16 half-warp row engines
constexpr int kEngines = kThreads / 16;   // rows processed side by side
constexpr int kQRowsInFlight = 4;         // rows per half-warp per batch
constexpr int kRopeHalf = FP4IDX_ROPE_DIM / 2;  // 32 cos/sin entries per row
constexpr int kKvBlock = FP4IDX_KV_BLOCK;
constexpr int kPageBytes = FP4IDX_PAGE_BYTES;
constexpr int kPayloadBytes = FP4IDX_SLOT_PAYLOAD_BYTES;
constexpr int kExpOffset = kKvBlock * kPayloadBytes;  // 4096

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 pair -> bf16x2 word (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// 16-byte streaming load of data read exactly once (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float4 ld_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
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
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
        "f"(v[6]), "f"(v[7]));
  return w;
}

// Per nibble: magnitude m (m <= 5) -> m + min(m, 2), the code of 2*grid[m];
// sign bits unchanged.
__device__ __forceinline__ uint32_t double_codes(uint32_t p) {
  const uint32_t mag = p & 0x77777777u;
  const uint32_t ge2 = ((mag >> 1) | (mag >> 2)) & 0x11111111u;  // m >= 2
  const uint32_t add = (ge2 << 1) | (mag & 0x11111111u & ~ge2);   // min(m,2)
  return (p & 0x88888888u) | (mag + add);
}

// Keep a nibble's sign bit only when its magnitude is non-zero.
__device__ __forceinline__ uint32_t clear_negative_zero(uint32_t p) {
  const uint32_t nz = (p | (p >> 1) | (p >> 2)) & 0x11111111u;
  return p & (0x77777777u | (nz << 3));
}

// Both quantisation stages for this lane's 8 elements (bf16-exact fp32
// values z).  Must be called by all 32 lanes (group amax uses shuffles).
// Returns the lane's payload word; *e2 receives the group's exponent.
__device__ __forceinline__ uint32_t quant_pack_lane(const uint32_t (&w)[4], uint32_t* e2) {
  float z[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    z[2 * k] = bf16_lo(w[k]);
    z[2 * k + 1] = bf16_hi(w[k]);
  }
  float a = fabsf(z[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, fabsf(z[i]));
  a = fmaxf(a, __shfl_xor_sync(kFull, a, 1));
  a = fmaxf(a, __shfl_xor_sync(kFull, a, 2));

  const uint32_t ab = __float_as_uint(a);
  int e1 = (int)(ab >> 23) - 2 + ((ab & 0x7fffffu) > 0x400000u ? 1 : 0);
  e1 = e1 < 1 ? 1 : e1;
  const float inv1 = __uint_as_float((uint32_t)(254 - e1) << 23);  // 2^(127-e1)

  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(z[i], inv1);
  uint32_t p = e2m1x8(v);

  const bool halve = (e1 > 1) && (__fmul_rn(a, inv1) < 3.5f);
  if (halve) p = double_codes(p);
  *e2 = (uint32_t)(e1 - (halve ? 1 : 0));
  return clear_negative_zero(p);
}

// Exponent word of the row: byte g = exponent of group g (lanes 4g..4g+3).
__device__ __forceinline__ uint32_t exponent_word(uint32_t e, int j) {
  uint32_t x = e << (8 * (j >> 2));
  x |= __shfl_xor_sync(kFull, x, 4);
  x |= __shfl_xor_sync(kFull, x, 8);
  return x;
}

// RoPE coefficients of this lane for one position.  NeoX: lanes 0..7 hold
// cos/sin[8(j&3) .. +7]; lanes 0..3 own the first element of each pair and
// take -sin so both halves compute own*c + partner*s.  Interleaved: lanes
// 0..7 hold cos/sin[4j .. 4j+3].  Lanes 8..15 hold nothing.
template <int kStyle>
struct RopeCoef {
  float c[8];
  float s[8];
  __device__ __forceinline__ void load(const float* cos_row, const float* sin_row, int j) {
    if (j >= 8) return;
    if (kStyle == FP4IDX_ROPE_NEOX) {
      const int b = 8 * (j & 3);
      const float4 c0 = ld_f4(cos_row + b), c1 = ld_f4(cos_row + b + 4);
      const float4 s0 = ld_f4(sin_row + b), s1 = ld_f4(sin_row + b + 4);
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
      s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
      if (j < 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i] = -s[i];
      }
    } else {
      const float4 c0 = ld_f4(cos_row + 4 * j), s0 = ld_f4(sin_row + 4 * j);
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
    }
  }
};

// In-place RoPE of this lane's words.  Must be called by all 32 lanes (the
// NeoX partner exchange is a shuffle); only lanes j < 8 change their data.
template <int kStyle>
__device__ __forceinline__ void rope_lane(uint32_t (&w)[4], const RopeCoef<kStyle>& rc, int j) {
  if (kStyle == FP4IDX_ROPE_NEOX) {
    uint32_t p[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = __shfl_xor_sync(kFull, w[k], 4);
    if (j < 8) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float r0 = __fadd_rn(__fmul_rn(bf16_lo(w[k]), rc.c[2 * k]),
                                   __fmul_rn(bf16_lo(p[k]), rc.s[2 * k]));
        const float r1 = __fadd_rn(__fmul_rn(bf16_hi(w[k]), rc.c[2 * k + 1]),
                                   __fmul_rn(bf16_hi(p[k]), rc.s[2 * k + 1]));
        w[k] = pack_bf16x2(r0, r1);
      }
    }
  } else {
    if (j < 8) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = bf16_lo(w[k]), x1 = bf16_hi(w[k]);
        const float r0 = __fsub_rn(__fmul_rn(x0, rc.c[k]), __fmul_rn(x1, rc.s[k]));
        const float r1 = __fadd_rn(__fmul_rn(x1, rc.c[k]), __fmul_rn(x0, rc.s[k]));
        w[k] = pack_bf16x2(r0, r1);
      }
    }
  }
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
};

// ------------------------------------------------------------- key rows
// 16 consecutive key rows [row0, row0 + 16), one per half-warp engine.
template <int kStyle>
__device__ __forceinline__ void key_rows(const KArgs& ka, const Shared& sh, int64_t row0,
                                         const float (&g)[8]) {
  const int j = threadIdx.x & 15;
  const int64_t t = row0 + (threadIdx.x >> 4);
  bool live = t < sh.T;
  int64_t slot = -1, pos = 0;
  if (live) {
    slot = __ldg(ka.slots + t);
    live = slot >= 0;
  }
  uint4 raw = make_uint4(0u, 0u, 0u, 0u);
  if (live) {
    pos = __ldg(sh.pos + t);
    raw = ld_stream_v4(ka.k + t * ka.k_stride + 8 * j);
    const bool pos_ok = pos >= 0 && pos < sh.max_pos;
    const bool slot_ok = slot < ka.num_blocks * kKvBlock;
    if (!(pos_ok && slot_ok)) {
      if (j == 0) flag_error(sh.err, (pos_ok ? 0u : FP4IDX_ERRFLAG_POSITION) |
                                         (slot_ok ? 0u : FP4IDX_ERRFLAG_SLOT));
      live = false;
      pos = 0;
    }
  }
  RopeCoef<kStyle> rc{};
  if (live) rc.load(sh.cos + pos * kRopeHalf, sh.sin + pos * kRopeHalf, j);

  // RMSNorm: 8 sequential squares per lane, then the xor butterfly 8,4,2,1.
  uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = bf16_lo(w[k]);
    x[2 * k + 1] = bf16_hi(w[k]);
  }
  float ss = __fmul_rn(x[0], x[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(x[i], x[i]));
  ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 8));
  ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 4));
  ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 2));
  ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, 1));
  const float ms = __fmul_rn(ss, 0.0078125f);  // /128, exact scaling
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, ka.eps)));
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = pack_bf16x2(__fmul_rn(__fmul_rn(x[2 * k], r), g[2 * k]),
                       __fmul_rn(__fmul_rn(x[2 * k + 1], r), g[2 * k + 1]));

  rope_lane<kStyle>(w, rc, j);
  uint32_t e2;
  const uint32_t payload = quant_pack_lane(w, &e2);
  const uint32_t ex = exponent_word(e2, j);
  if (live) {
    uint8_t* page = ka.cache + (slot / kKvBlock) * (int64_t)kPageBytes;
    const int64_t o = slot % kKvBlock;
    *reinterpret_cast<uint32_t*>(page + o * kPayloadBytes + 4 * j) = payload;
    if (j == 0) *reinterpret_cast<uint32_t*>(page + kExpOffset + 4 * o) = ex;
  }
}

template <int kStyle>
__device__ __forceinline__ void load_gamma(const KArgs& ka, float (&g)[8]) {
  const int j = threadIdx.x & 15;
  const uint4 gr = __ldg(reinterpret_cast<const uint4*>(ka.gamma) + j);
  const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    g[2 * k] = bf16_lo(gw[k]);
    g[2 * k + 1] = bf16_hi(gw[k]);
  }
}

// ----------------------------------------------------------- query tokens
template <int kStyle>
__device__ __forceinline__ void query_token(const QArgs& qa, const Shared& sh, int64_t t) {
  const int j = threadIdx.x & 15;
  const int engine = threadIdx.x >> 4;
  const int64_t pos = __ldg(sh.pos + t);
  if (pos < 0 || pos >= sh.max_pos) {  // uniform over the CTA
    if (threadIdx.x == 0) flag_error(sh.err, FP4IDX_ERRFLAG_POSITION);
    return;
  }
  for (int64_t h = threadIdx.x; h < qa.H; h += blockDim.x) {
    const uint16_t wb = __ldg(qa.w + t * qa.w_tstride + h);
    qa.weights[t * qa.H + h] = __fmul_rn(__uint_as_float((uint32_t)wb << 16), qa.wscale);
  }
  RopeCoef<kStyle> rc;
  rc.load(sh.cos + pos * kRopeHalf, sh.sin + pos * kRopeHalf, j);

  const uint16_t* qt = qa.q + t * qa.q_tstride + 8 * j;
  for (int64_t base = 0; base < qa.H; base += kEngines * kQRowsInFlight) {
    uint4 raw[kQRowsInFlight];
#pragma unroll
    for (int i = 0; i < kQRowsInFlight; ++i) {
      const int64_t h = base + engine + kEngines * i;
      raw[i] = h < qa.H ? ld_stream_v4(qt + h * qa.q_hstride) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kQRowsInFlight; ++i) {
      const int64_t h = base + engine + kEngines * i;
      uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
      rope_lane<kStyle>(w, rc, j);
      uint32_t e2;
      const uint32_t payload = quant_pack_lane(w, &e2);
      const uint32_t ex = exponent_word(e2, j);
      if (h < qa.H) {
        const int64_t row = t * qa.H + h;
        *reinterpret_cast<uint32_t*>(qa.q_fp4 + row * kPayloadBytes + 4 * j) = payload;
        if (j == 0) *reinterpret_cast<uint32_t*>(qa.q_scale + row * 4) = ex;
      }
    }
  }
}

// ------------------------------------------------------------------ kernels
template <int kStyle>
__global__ void __launch_bounds__(kThreads) k_kernel(KArgs ka, Shared sh) {
  float g[8];
  load_gamma<kStyle>(ka, g);
  for (int64_t row0 = (int64_t)blockIdx.x * kEngines; row0 < sh.T;
       row0 += (int64_t)gridDim.x * kEngines)
    key_rows<kStyle>(ka, sh, row0, g);
}

template <int kStyle>
__global__ void __launch_bounds__(kThreads) q_kernel(QArgs qa, Shared sh) {
  for (int64_t t = blockIdx.x; t < sh.T; t += gridDim.x) query_token<kStyle>(qa, sh, t);
}

// One grid over both halves: work items [0, nk) are groups of 16 key rows,
// items [nk, nk + T) are query tokens.
template <int kStyle>
__global__ void __launch_bounds__(kThreads) prepass_kernel(KArgs ka, QArgs qa, Shared sh) {
  float g[8];
  load_gamma<kStyle>(ka, g);
  const int64_t nk = (sh.T + kEngines - 1) / kEngines;
  const int64_t total = nk + sh.T;
  for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
    if (item < nk)
      key_rows<kStyle>(ka, sh, item * kEngines, g);
    else
      query_token<kStyle>(qa, sh, item - nk);
  }
}

// --------------------------------------------------------------- host side
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  int sm_count = 0;
  int occupancy[3][2] = {{0, 0}, {0, 0}, {0, 0}};  // [kernel][style]
};
DeviceInfo g_devices[kMaxDevices];

template <typename Kernel>
int occupancy_of(Kernel kern) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

// Resident CTAs for a persistent grid (SM count x blocks per SM), cached per
// device; 0 on a CUDA error.
int persistent_grid(int which, int style) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  DeviceInfo& di = g_devices[dev];
  if (di.sm_count == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    di.occupancy[0][0] = occupancy_of(k_kernel<FP4IDX_ROPE_NEOX>);
    di.occupancy[0][1] = occupancy_of(k_kernel<FP4IDX_ROPE_INTERLEAVED>);
    di.occupancy[1][0] = occupancy_of(q_kernel<FP4IDX_ROPE_NEOX>);
    di.occupancy[1][1] = occupancy_of(q_kernel<FP4IDX_ROPE_INTERLEAVED>);
    di.occupancy[2][0] = occupancy_of(prepass_kernel<FP4IDX_ROPE_NEOX>);
    di.occupancy[2][1] = occupancy_of(prepass_kernel<FP4IDX_ROPE_INTERLEAVED>);
    di.sm_count = sms;
  }
  return di.sm_count * di.occupancy[which][style];
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
  if (num_blocks < 1 || num_blocks > INT64_MAX / kPageBytes) return FP4IDX_ERR_SHAPE;
  if (!(eps > 0.0f) || !isfinite(eps)) return FP4IDX_ERR_ARG;
  if (!aligned(k, 16) || (k_stride % 8) != 0 || !aligned(gamma, 16) || !aligned(slots, 8) ||
      !aligned(cache, 16))
    return FP4IDX_ERR_ALIGN;
  return FP4IDX_OK;
}

fp4idx_status check_queries(const void* q, int64_t q_tstride, int64_t q_hstride, const void* w,
                            float wscale, const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* weights, int64_t num_tokens, int64_t num_heads) {
  if (!q || !w || !q_fp4 || !q_scale || !weights) return FP4IDX_ERR_NULL;
  if (num_heads < 1 || num_heads > INT64_MAX / kPayloadBytes / (num_tokens > 0 ? num_tokens : 1))
    return FP4IDX_ERR_SHAPE;
  if (!isfinite(wscale)) return FP4IDX_ERR_ARG;
  if (!aligned(q, 16) || (q_tstride % 8) != 0 || (q_hstride % 8) != 0 || !aligned(w, 2) ||
      !aligned(q_fp4, 16) || !aligned(q_scale, 4) || !aligned(weights, 4))
    return FP4IDX_ERR_ALIGN;
  return FP4IDX_OK;
}

fp4idx_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}

int64_t grid_for(int64_t items, int which, int style) {
  const int64_t resident = persistent_grid(which, style);
  if (resident <= 0) return 0;
  return items < resident ? items : resident;
}

}  // namespace

// ------------------------------------------------------------------- C ABI
extern "C" {

fp4idx_status fp4idx_k_norm_rope_pack_store(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* positions, const float* cos_cache, const float* sin_cache,
    int64_t max_pos, int rope_style, const int64_t* slot_mapping, uint8_t* kv_cache,
    int64_t num_blocks, int64_t num_tokens, uint32_t* err_flags, void* stream) {
  if (num_tokens < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  st = check_keys(k, k_token_stride, gamma, eps, slot_mapping, kv_cache, num_blocks);
  if (st != FP4IDX_OK) return st;
  if (err_flags && !aligned(err_flags, 4)) return FP4IDX_ERR_ALIGN;

  KArgs ka{static_cast<const uint16_t*>(k), k_token_stride, static_cast<const uint16_t*>(gamma),
           eps, slot_mapping, kv_cache, num_blocks};
  Shared sh{positions, cos_cache, sin_cache, max_pos, num_tokens, err_flags};
  const int64_t grid = grid_for((num_tokens + kEngines - 1) / kEngines, 0, rope_style);
  if (grid <= 0) return FP4IDX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rope_style == FP4IDX_ROPE_NEOX)
    k_kernel<FP4IDX_ROPE_NEOX><<<(unsigned)grid, kThreads, 0, s>>>(ka, sh);
  else
    k_kernel<FP4IDX_ROPE_INTERLEAVED><<<(unsigned)grid, kThreads, 0, s>>>(ka, sh);
  return launch_status();
}

fp4idx_status fp4idx_q_rope_pack_weights(
    const void* q, int64_t q_token_stride, int64_t q_head_stride, const void* w,
    int64_t w_token_stride, float weight_scale, const int64_t* positions,
    const float* cos_cache, const float* sin_cache, int64_t max_pos, int rope_style,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, int64_t num_tokens,
    int64_t num_heads, uint32_t* err_flags, void* stream) {
  if (num_tokens < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  st = check_queries(q, q_token_stride, q_head_stride, w, weight_scale, q_fp4, q_scale,
                     weights_out, num_tokens, num_heads);
  if (st != FP4IDX_OK) return st;
  if (err_flags && !aligned(err_flags, 4)) return FP4IDX_ERR_ALIGN;

  QArgs qa{static_cast<const uint16_t*>(q), q_token_stride, q_head_stride,
           static_cast<const uint16_t*>(w), w_token_stride, weight_scale, q_fp4, q_scale,
           weights_out, num_heads};
  Shared sh{positions, cos_cache, sin_cache, max_pos, num_tokens, err_flags};
  const int64_t grid = grid_for(num_tokens, 1, rope_style);
  if (grid <= 0) return FP4IDX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rope_style == FP4IDX_ROPE_NEOX)
    q_kernel<FP4IDX_ROPE_NEOX><<<(unsigned)grid, kThreads, 0, s>>>(qa, sh);
  else
    q_kernel<FP4IDX_ROPE_INTERLEAVED><<<(unsigned)grid, kThreads, 0, s>>>(qa, sh);
  return launch_status();
}

fp4idx_status fp4idx_indexer_prepass(
    const void* k, int64_t k_token_stride, const void* gamma, float eps,
    const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_blocks, const void* q,
    int64_t q_token_stride, int64_t q_head_stride, const void* w, int64_t w_token_stride,
    float weight_scale, uint8_t* q_fp4, uint8_t* q_scale, float* weights_out,
    int64_t num_heads, const int64_t* positions, const float* cos_cache,
    const float* sin_cache, int64_t max_pos, int rope_style, int64_t num_tokens,
    uint32_t* err_flags, void* stream) {
  if (num_tokens < 0) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  fp4idx_status st = check_shared(positions, cos_cache, sin_cache, max_pos, rope_style);
  if (st != FP4IDX_OK) return st;
  st = check_keys(k, k_token_stride, gamma, eps, slot_mapping, kv_cache, num_blocks);
  if (st != FP4IDX_OK) return st;
  st = check_queries(q, q_token_stride, q_head_stride, w, weight_scale, q_fp4, q_scale,
                     weights_out, num_tokens, num_heads);
  if (st != FP4IDX_OK) return st;
  if (err_flags && !aligned(err_flags, 4)) return FP4IDX_ERR_ALIGN;

  KArgs ka{static_cast<const uint16_t*>(k), k_token_stride, static_cast<const uint16_t*>(gamma),
           eps, slot_mapping, kv_cache, num_blocks};
  QArgs qa{static_cast<const uint16_t*>(q), q_token_stride, q_head_stride,
           static_cast<const uint16_t*>(w), w_token_stride, weight_scale, q_fp4, q_scale,
           weights_out, num_heads};
  Shared sh{positions, cos_cache, sin_cache, max_pos, num_tokens, err_flags};
  const int64_t items = (num_tokens + kEngines - 1) / kEngines + num_tokens;
  const int64_t grid = grid_for(items, 2, rope_style);
  if (grid <= 0) return FP4IDX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rope_style == FP4IDX_ROPE_NEOX)
    prepass_kernel<FP4IDX_ROPE_NEOX><<<(unsigned)grid, kThreads, 0, s>>>(ka, qa, sh);
  else
    prepass_kernel<FP4IDX_ROPE_INTERLEAVED><<<(unsigned)grid, kThreads, 0, s>>>(ka, qa, sh);
  return launch_status();
}

const char* fp4idx_status_string(fp4idx_status status) {
  switch (status) {
    case FP4IDX_OK: return "ok";
    case FP4IDX_ERR_NULL: return "a required pointer is NULL";
    case FP4IDX_ERR_SHAPE: return "invalid size (negative count, zero heads/blocks/positions, or overflow)";
    case FP4IDX_ERR_ALIGN: return "a pointer or stride breaks its alignment rule";
    case FP4IDX_ERR_ARG: return "invalid argument (rope_style, eps or weight_scale)";
    case FP4IDX_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

const char* fp4idx_version(void) { return "fp4idx 0.1.0 sm_103a"; }

}  // extern "C"
