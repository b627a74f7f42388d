// Exhaustive check of the library's corrected reciprocal quotient (div_rcp
// and its packed form div_rcp2 in fp4idx_common.cuh, the latter on the pair
// (x, -x), each with the reciprocal the quantiser passes) against the IEEE
// division (__fdiv_rn): every finite
// bf16 numerator by every positive finite E4M3 scale (126 values) and by 6,
// wherever the IEEE quotient is below 2^120 in magnitude.  The fake
// quantisation only meets such pairs: |x| <= amax and s = E4M3(rn(amax/6))
// give |x/s| <= 9 unless s saturates at 448, and then |x/s| < 2^128 / 448.
// Below 2^-60 the residual x - q*s can underflow, so the quotient may be
// one ulp off there; such quotients are far below the smallest E2M1 rounding
// boundary (0.25), so the code is the same.  Prints "checked N mismatches M
// skipped K tiny T codes C": M quotients differ, T of them below 2^-60 in
// magnitude, C pairs give a different E2M1 code (ties to even, saturating at
// 6), P pairs where the packed form differs from the scalar one (printed as
// "packed P"); K pairs have a larger or non-finite quotient.  Then the operands of the
// first few mismatches at or above 2^-60.  Test infrastructure: built and
// run by tests/test_division_gpu.py.
#include <stdio.h>
#include <stdint.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include "fp4idx_common.cuh"

using fp4idx_impl::div_rcp;
using fp4idx_impl::div_rcp2;

__device__ float e4m3_value(uint32_t code) {  // code 1 .. 126: positive finite e4m3fn
  uint32_t h;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h) : "r"(code));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// E2M1 code of v (round half to even, saturating), as the quantiser takes
// it: a zero magnitude carries no sign (the quantiser drops it, so -0 and +0
// quotients give the same value).
__device__ uint32_t e2m1_code(float v) {
  uint32_t c;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %1;\n\tcvt.u32.u8 %0, b;\n\t}"
      : "=r"(c) : "f"(v));
  c &= 0xfu;
  return (c & 7u) ? c : 0u;
}

__device__ bool same(float a, float b) {
  return (__float_as_uint(a) == __float_as_uint(b)) || (a != a && b != b);
}

__global__ void check(unsigned long long* count, unsigned long long* bad, uint32_t* first,
                      unsigned long long* skipped, unsigned long long* tiny,
                      unsigned long long* codes, unsigned long long* packed) {
  const uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x;  // 127 divisors x 65536 numerators
  if (idx >= 127u * 65536u) return;
  const uint32_t di = idx >> 16, xb = idx & 0xffffu;
  const float x = __uint_as_float(xb << 16);
  const float s = di < 126 ? e4m3_value(di + 1) : 6.0f;
  // the reciprocal the quantiser uses: the hardware approximation for an
  // E4M3 scale, rn(1/6) for the scale's own divisor
  const float rs = di < 126 ? fp4idx_impl::rcp_approx(s) : 1.0f / 6.0f;
  float got = div_rcp(x, s, rs), g0, g1;
  div_rcp2(g0, g1, x, -x, s, rs);
  const float want = __fdiv_rn(x, s);
  if (!(fabsf(x) < INFINITY) || !(fabsf(want) < 0x1p120f)) {
    atomicAdd(skipped, 1ull);
    return;
  }
  atomicAdd(count, 1ull);
  // the packed form gives the scalar's results (and -x / s = -(x / s))
  if (__float_as_uint(g0) != __float_as_uint(got) ||
      (__float_as_uint(g1) != (__float_as_uint(got) ^ 0x80000000u) && !(got == 0.0f && g1 == 0.0f)))
    atomicAdd(packed, 1ull);
  if (e2m1_code(got) != e2m1_code(want)) atomicAdd(codes, 1ull);
  if (!same(got, want)) {
    atomicAdd(bad, 1ull);
    if (fabsf(want) < 0x1p-60f) {
      atomicAdd(tiny, 1ull);
      return;
    }
    const unsigned long long k = atomicAdd(first + 24, 1u);
    if (k < 8) {
      first[3 * k] = xb;
      first[3 * k + 1] = __float_as_uint(s);
      first[3 * k + 2] = __float_as_uint(got);
    }
  }
}

int main() {
  unsigned long long *c, *b, *k, *t, *cd, *pk;
  uint32_t* f;
  if (cudaMalloc(&c, 8) || cudaMalloc(&b, 8) || cudaMalloc(&k, 8) || cudaMalloc(&t, 8) ||
      cudaMalloc(&cd, 8) || cudaMalloc(&pk, 8) || cudaMalloc(&f, 25 * 4))
    return 2;
  cudaMemset(pk, 0, 8);
  cudaMemset(c, 0, 8);
  cudaMemset(b, 0, 8);
  cudaMemset(k, 0, 8);
  cudaMemset(t, 0, 8);
  cudaMemset(cd, 0, 8);
  cudaMemset(f, 0, 25 * 4);
  const uint32_t n = 127u * 65536u;
  check<<<(n + 255) / 256, 256>>>(c, b, f, k, t, cd, pk);
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  unsigned long long hc, hb, hk, ht, hcd, hpk;
  uint32_t hf[25];
  cudaMemcpy(&hc, c, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(&hb, b, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(&hk, k, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(&ht, t, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(&hcd, cd, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(&hpk, pk, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(hf, f, sizeof hf, cudaMemcpyDeviceToHost);
  printf("checked %llu mismatches %llu skipped %llu tiny %llu codes %llu packed %llu\n", hc, hb, hk,
         ht, hcd, hpk);
  for (unsigned long long k = 0; k < hf[24] && k < 8; ++k)
    printf("x=0x%04x s=0x%08x got=0x%08x\n", hf[3 * k], hf[3 * k + 1], hf[3 * k + 2]);
  return 0;
}
