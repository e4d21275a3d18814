// norm.cuh — the RMSNorm arithmetic of the fused projection (sm_103a):
// x^ = x / sqrt(mean(x^2) + eps) * g rounded once to bf16.
//
// x is bf16, so every x*x is exact in fp32 and a row's sum of squares is
// carried as an unevaluated (hi, lo) pair of floats (TwoSum); the scale
// 1 / sqrt(ss / D + eps) is formed as a float pair as well (relative error
// ~2^-40), and x^ is the correctly rounded bf16 value of x * scale * g (the
// product evaluated with its exact error).  fp32 only: fp64 is slow on this
// part.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace dllm {

// s + e == a + b exactly (Knuth's TwoSum), with the additions pinned to
// round-to-nearest so that the compiler cannot contract or reorder them.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Add the exact squares of 8 bf16 values to the pair (hi, lo).
__device__ __forceinline__ void sumsq_pair_add(const uint4& u, float& hi, float& lo) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    float e;
    two_sum(hi, __fmul_rn(f.x, f.x), hi, e);
    lo = __fadd_rn(lo, e);
    two_sum(hi, __fmul_rn(f.y, f.y), hi, e);
    lo = __fadd_rn(lo, e);
  }
}

// (hi, lo) += (oh, ol)
__device__ __forceinline__ void pair_add(float& hi, float& lo, float oh, float ol) {
  float e;
  two_sum(hi, oh, hi, e);
  lo = __fadd_rn(lo, __fadd_rn(e, ol));
}

// 1 / sqrt(ss / D + eps) as an unevaluated pair (hi, lo) of floats, from the
// sum of squares (ss_hi, ss_lo).  The quotient and the sum are carried as
// float pairs (the division remainder by FMA is exact); the reciprocal square
// root is one Newton-Raphson step y1 = y0 - y0 (s y0^2 - 1) / 2 from the
// hardware estimate y0 (relative error e0 < 2^-21), with the residual
// s y0^2 - 1 formed from an exact product y0^2 and FMAs.  Newton's error
// (3/2) e0^2 and the rounding of the residual leave |y1 / y - 1| below about
// 2^-40, far inside the 2^-9 spacing that the bf16 rounding of x^ resolves.
__device__ __forceinline__ void rsqrt_pair(float ss_hi, float ss_lo, int D, float eps, float& y_hi, float& y_lo) {
  const float fd = static_cast<float>(D);
  const float q_hi = __fdiv_rn(ss_hi, fd);
  const float rem = __fmaf_rn(-q_hi, fd, ss_hi);  // exact: ss_hi - q_hi * D
  const float q_lo = __fdiv_rn(__fadd_rn(rem, ss_lo), fd);
  float s_hi, e;
  two_sum(q_hi, eps, s_hi, e);
  const float s_lo = __fadd_rn(e, q_lo);
  const float y0 = rsqrtf(s_hi);
  const float p = __fmul_rn(y0, y0);
  const float pe = __fmaf_rn(y0, y0, -p);  // y0^2 = p + pe exactly
  const float u = __fmaf_rn(s_hi, p, -1.f);
  const float t = __fadd_rn(u, __fmaf_rn(s_hi, pe, __fmul_rn(s_lo, p)));  // s y0^2 - 1
  const float corr = __fmul_rn(__fmul_rn(-0.5f, y0), t);
  two_sum(y0, corr, y_hi, y_lo);
}

// x^ = x * (s_hi + s_lo) * g for 8 consecutive elements (bf16 x, g),
// correctly rounded to bf16 without branches.  t = x * g is exact in fp32
// (two 8-bit significands); t * s is formed as p + e with p = fl(t * s_hi)
// and e = (t * s_hi - p) (exact, FMA) + t * s_lo.  p alone decides the bf16
// rounding unless p sits exactly on a bf16 midpoint (its 16 discarded bits
// are 0x8000), in which case the sign of e does (|e| is below half an fp32
// step of p).
__device__ __forceinline__ uint4 normalise8(const uint4& u, const uint4& gu, float s_hi, float s_lo) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w}, gw[4] = {gu.x, gu.y, gu.z, gu.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t half[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float xf = __uint_as_float(h ? (w[i] & 0xFFFF0000u) : (w[i] << 16));
      const float gv = __uint_as_float(h ? (gw[i] & 0xFFFF0000u) : (gw[i] << 16));
      const float t = __fmul_rn(xf, gv);  // exact
      const float p = __fmul_rn(t, s_hi);
      const float e = __fmaf_rn(t, s_lo, __fmaf_rn(t, s_hi, -p));
      const uint32_t bits = __float_as_uint(p);
      const uint32_t rn = __bfloat16_as_ushort(__float2bfloat16_rn(p));
      const bool tie = (bits & 0xFFFFu) == 0x8000u && e != 0.f;
      const uint32_t away = ((e > 0.f) == (p > 0.f)) ? 1u : 0u;
      half[h] = tie ? (bits >> 16) + away : rn;
    }
    o[i] = (half[0] & 0xFFFFu) | (half[1] << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace dllm
