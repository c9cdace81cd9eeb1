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

// Per-block constants: the scale and, when s >= 2^-96, its rounded reciprocal.
struct QuantBlock {
  float s, rc;
  bool fast;
};

__device__ __forceinline__ QuantBlock quant_block(float absmax) {
  QuantBlock b;
  b.s = __fdiv_rn(absmax, 127.0f);
  b.fast = b.s >= 1.2621774e-29f;  // 2^-96: below it (and for s == 0) the IEEE rule
  b.rc = b.fast ? __frcp_rn(b.s) : 0.0f;
  return b;
}

// Eight elements: codes (kRoundMagic + q per element, its low byte the code) and new
// values.  The quotient rn(d/s) is formed without a division by one correction step
// (Markstein's theorem): with rc = rn(1/s) and t0 = rn(d rc), which lies within one ulp
// of d/s, the residual r = d - t0 s is exact as an FMA, and rn(t0 + r rc) is the
// correctly rounded quotient -- the same bits as the IEEE division, as long as r does not
// underflow, which s >= 2^-96 guarantees for every quotient that rounds to a non-zero
// code (|d/s| >= 1/2).  Checked against exact rational division on 4e5 cases (random,
// near half-integers, extreme significands of s, block maxima); blocks with a smaller s
// take the IEEE division per element.
__device__ __forceinline__ void quant8(const QuantBlock& b, const float (&d)[8],
                                       const float (&sv)[8], float (&tm)[8], float (&nv)[8]) {
  if (b.fast) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float t0 = __fmul_rn(d[e], b.rc);
      const float q = __fmaf_rn(__fmaf_rn(-t0, b.s, d[e]), b.rc, t0);
      tm[e] = __fadd_rn(q, kRoundMagic);
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
