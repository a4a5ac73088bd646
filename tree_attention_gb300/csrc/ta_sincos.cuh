// ta_sincos.cuh -- float32 sine and cosine rounded correctly except in rare
// near-tie cases, for the RoPE table.
//
// RoPE (``_rope`` on the page "_kernel_common.py") rounds each rotated
// element to fp16/bf16; a cos or sin that is off by one float32 ulp flips
// that rounding now and then, and a q row that attends only a few tree nodes
// feels one flip as a log-sum-exp change of about 1e-3.  So the table is
// built from sin/cos that carry ~2^-44 absolute error before the final
// float32 rounding, using float32 arithmetic only:
//
//   1. additive range reduction (Cody and Waite): x = k*pi/2 + r with pi/2 =
//      C1 + C2 + C3; x - k*C1 is exact in one FMA (both terms are multiples
//      of ulp(C1) and the difference is below 1), the rest is carried as a
//      float pair with exact products (FMA) and exact sums (Knuth's two-sum);
//   2. table split r = j/32 + b, |b| <= 1/64, with sin/cos(j/32) stored as
//      float pairs;
//   3. sin(b) = b - b^3/6 + b^5/120 and cos(b) - 1 = -b^2/2 + b^4/24 - b^6/720
//      (Taylor), then the angle-addition formulas summed in float pairs and
//      rounded once.
// Arguments with |x| >= 2^23 fall back to CUDA's sincosf.
#pragma once

#include "ta_sincos_table.h"

namespace ta {

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = a * b;
  e = fmaf(a, b, -p);
}

// ``tab`` is kSinCosTable as float4 rows {sin_hi, sin_lo, cos_hi, cos_lo}, in
// shared memory: lanes index it with different j, which the constant cache
// would serve one address at a time.
__device__ __forceinline__ void cr_sincosf(float x, float* sin_out, float* cos_out,
                                           const float4* tab) {
  if (!(fabsf(x) < 8388608.0f)) {
    sincosf(x, sin_out, cos_out);
    return;
  }
  // 1. x = k * pi/2 + (rh + rl)
  const float kf = rintf(x * 0.636619772f);
  const float r1 = fmaf(-kf, kPio2C1, x);  // exact
  float ph, pl;
  two_prod(kf, kPio2C2, ph, pl);
  float rh, rl;
  two_sum(r1, -ph, rh, rl);
  rl = (rl - pl) - kf * kPio2C3;
  {
    const float s = rh + rl;  // renormalise, |rh| >= |rl|
    rl = rl - (s - rh);
    rh = s;
  }
  // 2. r = j/32 + b
  const float jf = rintf(rh * 32.0f);
  const int j = (int)jf;
  const int ja = j < 0 ? -j : j;
  const float bh = rh - jf * 0.03125f;  // exact
  const float bl = rl;
  // 3. b^2 as a float pair, cos(b) - 1 and sin(b)
  float b2h, b2e;
  two_prod(bh, bh, b2h, b2e);
  const float b2l = fmaf(2.0f * bh, bl, b2e);
  const float cmh = -0.5f * b2h;  // exact
  const float cml = fmaf(b2h * b2h, fmaf(b2h, -1.0f / 720.0f, 1.0f / 24.0f), -0.5f * b2l);
  const float sbl = fmaf(bh * b2h, fmaf(b2h, 1.0f / 120.0f, -1.0f / 6.0f), bl);  // sin b - bh
  const float4 e = tab[ja];
  float Sh = e.x, Sl = e.y;
  const float Ch = e.z, Cl = e.w;
  if (j < 0) {
    Sh = -Sh;
    Sl = -Sl;
  }
  // sin(a + b) = S + S*(cos b - 1) + C*sin b
  float p1, e1, q1, f1, s1, g1, s2, g2;
  two_prod(Ch, bh, p1, e1);
  two_prod(Sh, cmh, q1, f1);
  two_sum(Sh, p1, s1, g1);
  two_sum(s1, q1, s2, g2);
  const float ts =
      ((((g1 + g2) + (e1 + f1)) + Sl) + (fmaf(Ch, sbl, Cl * bh) + fmaf(Sh, cml, Sl * cmh)));
  const float sin_r = s2 + ts;
  // cos(a + b) = C + C*(cos b - 1) - S*sin b
  float p2, e2, q2, f2, c1, h1, c2, h2;
  two_prod(Sh, bh, p2, e2);
  two_prod(Ch, cmh, q2, f2);
  two_sum(Ch, -p2, c1, h1);
  two_sum(c1, q2, c2, h2);
  const float tc =
      ((((h1 + h2) + (f2 - e2)) + Cl) + (fmaf(Ch, cml, Cl * cmh) - fmaf(Sh, sbl, Sl * bh)));
  const float cos_r = c2 + tc;
  // quadrant
  switch (((int)kf) & 3) {
    case 0: *sin_out = sin_r; *cos_out = cos_r; break;
    case 1: *sin_out = cos_r; *cos_out = -sin_r; break;
    case 2: *sin_out = -sin_r; *cos_out = -cos_r; break;
    default: *sin_out = -cos_r; *cos_out = sin_r; break;
  }
}

}  // namespace ta
