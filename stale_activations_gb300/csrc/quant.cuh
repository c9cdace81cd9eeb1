// The residual quantiser of one 128-element block ("A way to reduce bandwidth
// requirement for xDiT": only the compressed residual fresh - stale is sent), shared by
// the refresh kernel and the projection epilogue that refreshes K and V as it stores
// them, so that both produce the same codes and values bit for bit.
//
//   s = absmax(d) / 127 (IEEE division), q = rint(d / s) (ties to even, clamped to
//   +-127, 0 when s == 0), new = fmaf(q, s, stale).
#pragma once
#include "common.cuh"

namespace dpp {

// Rounding without conversion instructions: for |t| < 2^22 the fp32 sum t + 1.5 * 2^23
// (round to nearest, ties to even) is exactly 1.5 * 2^23 + rint(t) with rint's ties to
// even (the constant is even), so subtracting it back gives rint(t) as a float and the
// low byte of the sum's bits is rint(t) as a two's-complement int8.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ int quantise(float d, float s) {
  if (s == 0.0f) return 0;
  float t = __fdiv_rn(d, s);                 // IEEE division, as on the CPU
  int q = __float2int_rn(t);                 // round to nearest, ties to even
  return max(-127, min(127, q));
}

// Per-block constants: the scale and, when 1/s is a finite normal number, its rounded
// reciprocal.
struct QuantBlock {
  float s, rc;
  bool fast;
};

__device__ __forceinline__ QuantBlock quant_block(float absmax) {
  QuantBlock b;
  b.s = __fdiv_rn(absmax, 127.0f);
  b.fast = b.s >= 1.17549435e-38f;  // FLT_MIN: a zero or subnormal s takes the IEEE rule
  b.rc = b.fast ? __frcp_rn(b.s) : 0.0f;
  return b;
}

// One element, the same rule as quant8 with a branch per element: returns
// kRoundMagic + q and sets the new value.
__device__ __forceinline__ float quant_elem(const QuantBlock& b, float d, float sv, float& nv) {
  float tm;
  if (b.fast) {
    const float t = d * b.rc;
    tm = t + kRoundMagic;
    if (0.5f - fabsf(t - (tm - kRoundMagic)) < 1e-4f) tm = __fdiv_rn(d, b.s) + kRoundMagic;
  } else {
    tm = (float)quantise(d, b.s) + kRoundMagic;
  }
  tm = fminf(fmaxf(tm, kRoundMagic - 127.0f), kRoundMagic + 127.0f);  // clamp to +-127
  nv = __fmaf_rn(tm - kRoundMagic, b.s, sv);
  return tm;
}

// Eight elements: codes (kRoundMagic + q per element, its low byte the code) and new
// values.  With r = rn(1/s), t = rn(d*r) lies within 2e-5 of rn(d/s) (|d/s| <= 127.0001
// and three roundings of relative size 2^-24), so both round to the same integer unless
// t is within 1e-4 of a half-integer; only for such elements (rare: no branch per
// element) is the IEEE quotient formed.  A block with a zero or subnormal s takes the
// IEEE rule for every element.
__device__ __forceinline__ void quant8(const QuantBlock& b, const float (&d)[8],
                                       const float (&sv)[8], float (&tm)[8], float (&nv)[8]) {
  uint32_t slow = 0;
  if (b.fast) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float t = d[e] * b.rc;
      tm[e] = t + kRoundMagic;
      slow |= (0.5f - fabsf(t - (tm[e] - kRoundMagic)) < 1e-4f ? 1u : 0u) << e;
    }
    if (slow) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if ((slow >> e) & 1u) tm[e] = __fdiv_rn(d[e], b.s) + kRoundMagic;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) tm[e] = (float)quantise(d[e], b.s) + kRoundMagic;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    tm[e] = fminf(fmaxf(tm[e], kRoundMagic - 127.0f), kRoundMagic + 127.0f);  // +-127
    nv[e] = __fmaf_rn(tm[e] - kRoundMagic, b.s, sv[e]);
  }
}

// The eight code bytes (low bytes of tm's bits) packed into two words.
__device__ __forceinline__ uint2 pack_codes(const float (&tm)[8]) {
  constexpr uint32_t kSel[4] = {0x3214u, 0x3240u, 0x3410u, 0x4210u};
  uint32_t c0 = 0, c1 = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    c0 = __byte_perm(c0, __float_as_uint(tm[e]), kSel[e]);
    c1 = __byte_perm(c1, __float_as_uint(tm[4 + e]), kSel[e]);
  }
  return make_uint2(c0, c1);
}

}  // namespace dpp
