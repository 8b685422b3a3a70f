// qk_codes.cuh -- INT8 codes of Q and K for one 32-token block scale, shared
// by the quantisation pass and the attention kernel's in-kernel Q quantiser.
// Codes are clamp(rint(x / sc), -127, 127) with x / sc the fp32 quotient
// rounded to nearest even (diffusers issue #15014, kernel contract: "Q/K are
// quantized per 32-row block"), formed on the packed FP32 pipe.
#pragma once

#include "sm103_ptx.cuh"

namespace sage {

// Rounding and code stores without the XU pipe (int/half conversions and
// frnd there cap this HBM-bound kernel): y + 1.5*2^23 - 1.5*2^23 is y rounded
// to the nearest integer, ties to even, exactly for |y| < 2^22, and the low
// bits of y + 1.5*2^23 are that integer.
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23

// Integer code of x for block scale sc, as a float: bit-identical to
// clamp(rint(x / sc), -127, 127) with x / sc rounded to nearest even in fp32.
// While 1/sc is a normal float (sc in [2^-125, 2^125]), y = x * fl(1/sc) is
// within |x/sc| * 2^-23 <= 1.6e-5 of x/sc (|x/sc| <= 127) and fl(x/sc)
// within 7.6e-6, so both round to the same integer unless y lies within
// 2^-15 of a half-integer; only then, or for extreme scales, divide.
static __device__ __noinline__ float code_by_division(float x, float sc) {
  const float y = __fdiv_rn(x, sc);
  return fminf(fmaxf((y + kRoundMagic) - kRoundMagic, -127.0f), 127.0f);
}

// Eight codes at once on the packed FP32 pipe, for a block scale sc in
// [2^-125, 2^125] (rcp = fl(1/sc)).  No clamp: |x| <= amax = 127 sc (1 + 2^-24)
// at most, so |y| < 127.5 and the rounded code is within [-127, 127].
// Returns false when some y lies within 2^-15 of a half-integer (or is not
// finite); the caller then divides, value by value.
__device__ __forceinline__ bool codes8_fast(const float (&x)[8], float rcp, float (&c)[8]) {
  constexpr float kTieLimit = 0.5f - 0x1p-15f;
  const float2 m2 = make_float2(kRoundMagic, kRoundMagic), r2 = make_float2(rcp, rcp);
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 y = fmul2v(make_float2(x[2 * i], x[2 * i + 1]), r2);
    const float2 r = fsub2v(fadd2v(y, m2), m2);
    const float2 d = fsub2v(y, r);
    ok &= (fabsf(d.x) <= kTieLimit) & (fabsf(d.y) <= kTieLimit);
    c[2 * i] = r.x;
    c[2 * i + 1] = r.y;
  }
  return ok;
}

// Codes of eight values of one block with scale sc (rcp = fl(1/sc)).
__device__ __forceinline__ void codes8(const float (&x)[8], float sc, float rcp, bool fast_sc, float (&c)[8]) {
  if (sc == 0.0f) {
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = 0.0f;
  } else if (!(fast_sc && codes8_fast(x, rcp, c))) {
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = code_by_division(x[e], sc);
  }
}

}  // namespace sage
