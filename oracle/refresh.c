/*
 * CPU oracle: compressed-residual refresh of a stale buffer (test infrastructure
 * only; nothing in the product links this file).
 *
 * Follows the CompactFusion idea quoted on the raylight issue page ("A way to
 * reduce bandwidth requirement for xDiT", first comment): transmit only the
 * compressed residual, i.e. the change fresh - stale.  The pages give no
 * quantiser; the one used here is the stated workload's: contiguous blocks of
 * 128 elements of the flat buffer, one fp32 scale per block, int8 codes, and
 * stale += dequant(codes).
 *
 * Exact fp32 semantics, one block at a time (a partial last block is allowed):
 *   d_i   = float(fresh_i) - float(stale_i)            (fp32 subtraction)
 *   a     = max_i |d_i|
 *   s     = a / 127                                    (IEEE fp32 division)
 *   q_i   = s == 0 ? 0 : clamp(rint(d_i / s), -127, 127)   (ties to even)
 *   new_i = fmaf(q_i, s, float(stale_i))               (one rounding)
 *   bf16 storage: stale_i = bf16_rne(new_i); fp32 storage: stale_i = new_i
 * A block whose delta is all zero gets s = 0, q = 0 and stays unchanged.
 *
 * Built with -O2 -ffp-contract=off so that no other fused multiply-add is formed.
 * Inputs must be finite; |fresh - stale| must not overflow fp32.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even of a finite fp32 value to bf16 (top 16 bits). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float load(const void* p, int64_t i, int is_bf16) {
  if (is_bf16) return bf16_bits_to_f32(((const uint16_t*)p)[i]);
  return ((const float*)p)[i];
}

/* One block [i0, i1).  Returns nothing; writes codes, the scale and stale. */
static void refresh_block(const void* fresh, void* stale, int8_t* codes, float* scale,
                          int64_t i0, int64_t i1, int is_bf16) {
  float a = 0.0f;
  for (int64_t i = i0; i < i1; ++i) {
    float d = load(fresh, i, is_bf16) - load(stale, i, is_bf16);
    float ad = fabsf(d);
    if (ad > a) a = ad;
  }
  float s = a / 127.0f;
  *scale = s;
  for (int64_t i = i0; i < i1; ++i) {
    float st = load(stale, i, is_bf16);
    float d = load(fresh, i, is_bf16) - st;
    int q = 0;
    if (s != 0.0f) {
      float t = d / s;
      float r = nearbyintf(t); /* default rounding mode: to nearest, ties to even */
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q = (int)r;
    }
    codes[i] = (int8_t)q;
    float nv = fmaf((float)q, s, st);
    if (is_bf16)
      ((uint16_t*)stale)[i] = f32_to_bf16_rne(nv);
    else
      ((float*)stale)[i] = nv;
  }
}

/* Refresh the flat buffer of n elements in place.  dtype: 0 = fp32, 1 = bf16
 * (raw bit patterns).  codes[n], scales[ceil(n/128)].  Returns 0, or 1 on bad
 * arguments. */
int oracle_refresh_residual(const void* fresh, void* stale, int8_t* codes, float* scales,
                            int64_t n, int dtype) {
  if (n < 0 || (dtype != 0 && dtype != 1)) return 1;
  if (n == 0) return 0;
  if (!fresh || !stale || !codes || !scales) return 1;
  int64_t nblk = (n + 127) / 128;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int64_t b = 0; b < nblk; ++b) {
    int64_t i0 = b * 128, i1 = i0 + 128;
    if (i1 > n) i1 = n;
    refresh_block(fresh, stale, codes, &scales[b], i0, i1, dtype == 1);
  }
  return 0;
}

/* Receiver side of the same message: stale_i = store(fmaf(codes[i], scales[i/128],
 * f32(stale_i))).  Used to emulate ranks that each hold their own stale copy. */
int oracle_apply_residual(void* stale, const int8_t* codes, const float* scales, int64_t n,
                          int dtype) {
  if (n < 0 || (dtype != 0 && dtype != 1)) return 1;
  if (n == 0) return 0;
  if (!stale || !codes || !scales) return 1;
  for (int64_t i = 0; i < n; ++i) {
    float st = load(stale, i, dtype == 1);
    float nv = fmaf((float)codes[i], scales[i / 128], st);
    if (dtype == 1)
      ((uint16_t*)stale)[i] = f32_to_bf16_rne(nv);
    else
      ((float*)stale)[i] = nv;
  }
  return 0;
}
