// Compressed-residual refresh of stale buffers ("A way to reduce bandwidth
// requirement for xDiT": send only the compressed residual fresh - stale).
//
// Quantiser: contiguous 128-element blocks of each flat buffer, one fp32 scale
// s = absmax(delta)/127 per block, int8 codes q = rint(delta/s) (ties to even,
// clamped to +-127, 0 when s == 0), stale <- store(fmaf(q, s, stale)).
//
// HBM-bound streaming kernel: one block of 128 elements per 16 lanes, 8
// elements (one or two 128-bit accesses) per lane; the block maximum is a
// 16-lane xor-shuffle reduction.  Algorithmic traffic per element: read fresh
// and stale, write stale and the int8 code, plus 4 bytes of scale per 128.
#include "refresh.cuh"

namespace dpp {

__device__ __forceinline__ int quantise(float d, float s) {
  if (s == 0.0f) return 0;
  float t = __fdiv_rn(d, s);                 // IEEE division, as on the CPU
  int q = __float2int_rn(t);                 // round to nearest, ties to even
  return max(-127, min(127, q));
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
  uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
  unpack16(u, f);
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
  uint4 a = __ldcs(reinterpret_cast<const uint4*>(p));
  uint4 b = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
  float fa[4], fb[4];
  unpack16(a, fa);
  unpack16(b, fb);
#pragma unroll
  for (int i = 0; i < 4; ++i) { f[i] = fa[i]; f[4 + i] = fb[i]; }
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&f)[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&f)[8]) {
  __stcs(reinterpret_cast<uint4*>(p), pack16(f));
}
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&f)[8]) {
  float a[4] = {f[0], f[1], f[2], f[3]}, b[4] = {f[4], f[5], f[6], f[7]};
  __stcs(reinterpret_cast<uint4*>(p), pack16(a));
  __stcs(reinterpret_cast<uint4*>(p) + 1, pack16(b));
}

template <typename T>
__global__ void __launch_bounds__(256) refresh_kernel(const __grid_constant__ RefreshTable tab) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;                 // lane within the 16-lane block group
  const long long group = (long long)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 2 +
                          (lane >> 4);
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5) * 2;
  const long long total = tab.blk_start[tab.nseg];
  int seg = 0;
  for (long long gb = group; gb < total; gb += stride) {
    while (gb >= tab.blk_start[seg + 1]) ++seg;  // gb only grows: segments in order
    const RefreshSeg& sg = tab.seg[seg];
    const long long j = gb - tab.blk_start[seg];    // block within the segment
    const long long e0 = j * 128;
    const int nb = (int)min(128ll, sg.n - e0);
    const T* fr = reinterpret_cast<const T*>(sg.fresh) + e0;
    T* st = reinterpret_cast<T*>(sg.stale) + e0;
    int8_t* cd = sg.codes + e0;
    const bool vec = nb == 128 && sg.vec_ok;
    float d[8], sv[8];
    float a = 0.0f;
    if (vec) {
      float fv[8];
      load8<T>(fr + sub * 8, fv);
      load8<T>(st + sub * 8, sv);
#pragma unroll
      for (int i = 0; i < 8; ++i) { d[i] = fv[i] - sv[i]; a = fmaxf(a, fabsf(d[i])); }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = sub + 16 * i;               // strided so that any nb is covered
        if (e < nb) {
          sv[i] = to_f32(st[e]);
          d[i] = to_f32(fr[e]) - sv[i];
          a = fmaxf(a, fabsf(d[i]));
        } else {
          sv[i] = 0.0f; d[i] = 0.0f;
        }
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float s = __fdiv_rn(a, 127.0f);
    if (sub == 0) sg.scales[j] = s;
    if (vec) {
      float nv[8];
      uint32_t c0 = 0, c1 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = quantise(d[i], s);
        nv[i] = __fmaf_rn((float)q, s, sv[i]);
        const uint32_t b = (uint32_t)(q & 0xFF);
        if (i < 4) c0 |= b << (8 * i); else c1 |= b << (8 * (i - 4));
      }
      store8<T>(st + sub * 8, nv);
      __stcs(reinterpret_cast<uint2*>(cd + sub * 8), make_uint2(c0, c1));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = sub + 16 * i;
        if (e < nb) {
          const int q = quantise(d[i], s);
          st[e] = from_f32<T>(__fmaf_rn((float)q, s, sv[i]));
          cd[e] = (int8_t)q;
        }
      }
    }
  }
}

int launch_refresh(const RefreshTable& tab, int dtype, cudaStream_t stream) {
  const long long total = tab.blk_start[tab.nseg];
  if (total == 0) return DPP_OK;
  const int threads = 256;
  const long long groups_per_cta = threads / 32 * 2;
  long long want = (total + groups_per_cta - 1) / groups_per_cta;
  const long long cap = (long long)dpp_host::sm_count() * 8;  // 8 CTAs of 256 per SM
  const int grid = (int)(want < cap ? want : cap);
  if (dtype == DPP_BF16)
    refresh_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(tab);
  else
    refresh_kernel<float><<<grid, threads, 0, stream>>>(tab);
  return cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

}  // namespace dpp
