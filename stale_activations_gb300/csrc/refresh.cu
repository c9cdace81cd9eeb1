// Compressed-residual refresh of stale buffers ("A way to reduce bandwidth
// requirement for xDiT": send only the compressed residual fresh - stale).
//
// Quantiser: contiguous 128-element blocks of each flat buffer, one fp32 scale
// s = absmax(delta)/127 per block, int8 codes q = rint(delta/s) (ties to even,
// clamped to +-127, 0 when s == 0), stale <- store(fmaf(q, s, stale)).
//
// HBM-bound streaming kernel: one block of 128 elements per half warp, 8
// elements (one or two 128-bit accesses) per lane, two blocks in flight per half
// warp; the block maximum is a 16-lane xor-shuffle reduction.  Algorithmic
// traffic per element: read fresh and stale, write stale and the int8 code, plus
// 4 bytes of scale per 128.
#include "refresh.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace dpp {

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

// One 128-element block, done by the 16 lanes of a half warp (`hmask` names them):
// elements strided by 16 so that any length nb <= 128 is covered.  Used for ragged
// last blocks and misaligned segments only (the scalar pass after the streaming loop).
template <typename T>
__device__ __forceinline__ void refresh_block_scalar(const T* fr, const T* st, T* out, int8_t* cd,
                                                  float* scale, int nb, int sub,
                                                  unsigned hmask) {
  float d[8], sv[8];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = sub + 16 * i;
    sv[i] = e < nb ? to_f32(st[e]) : 0.0f;
    d[i] = e < nb ? to_f32(fr[e]) - sv[i] : 0.0f;
    a = fmaxf(a, fabsf(d[i]));
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(hmask, a, o));
  const float s = __fdiv_rn(a, 127.0f);
  if (sub == 0) *scale = s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = sub + 16 * i;
    if (e < nb) {
      const int q = quantise(d[i], s);
      out[e] = from_f32<T>(__fmaf_rn((float)q, s, sv[i]));
      cd[e] = (int8_t)q;
    }
  }
}

// A full, aligned block: each lane holds 8 consecutive elements as raw 128-bit vectors.
struct VecBlock {
  uint4 fr[2], st[2];
  void* out;  // where the refreshed values go
  int8_t* codes;
  float* scale;
  bool live;
};

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 (&u)[2], float (&f)[8]);
template <>
__device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4 (&u)[2], float (&f)[8]) {
  unpack16(u[0], f);
}
template <>
__device__ __forceinline__ void unpack8<float>(const uint4 (&u)[2], float (&f)[8]) {
  float a[4], b[4];
  unpack16(u[0], a);
  unpack16(u[1], b);
#pragma unroll
  for (int i = 0; i < 4; ++i) { f[i] = a[i]; f[4 + i] = b[i]; }
}

// Looks up block gb and, if it is a full block of an aligned segment, issues its
// loads (returned in v); other blocks are left to the scalar pass.
template <typename T>
__device__ __forceinline__ void start_block(const RefreshTable& tab, long long gb, long long total,
                                            int& seg, int sub, VecBlock& v) {
  v.live = false;
  if (gb >= total) return;
  while (gb >= tab.blk_start[seg + 1]) ++seg;  // gb only grows: segments in order
  const RefreshSeg& sg = tab.seg[seg];
  const long long j = gb - tab.blk_start[seg];
  const long long e0 = j * 128;
  if (!sg.vec_ok || sg.n - e0 < 128) return;
  // the whole block and its scale (the same for the 16 lanes, which shuffle together)
  if (!DPP_IN(e0, 128, sg.n) || !DPP_IN(j, 1, (sg.n + 127) / 128)) return;
  const T* fr = reinterpret_cast<const T*>(sg.fresh) + e0;
  T* st = reinterpret_cast<T*>(sg.stale) + e0;
  constexpr int NV = 8 / Vec<T>::N;  // 16-byte vectors per lane: 1 (bf16) or 2 (fp32)
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    v.fr[k] = __ldcs(reinterpret_cast<const uint4*>(fr + sub * 8) + k);
    v.st[k] = __ldcs(reinterpret_cast<const uint4*>(st + sub * 8) + k);
  }
  v.out = static_cast<T*>(sg.out) + e0 + sub * 8;
  v.codes = sg.codes + e0 + sub * 8;
  v.scale = sg.scales + j;
  v.live = true;
}

template <typename T>
__device__ __forceinline__ void finish_block(const VecBlock& v, int sub, unsigned hmask) {
  float f[8], sv[8], d[8];
  unpack8<T>(v.fr, f);
  unpack8<T>(v.st, sv);
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) { d[i] = f[i] - sv[i]; a = fmaxf(a, fabsf(d[i])); }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(hmask, a, o));
  const QuantBlock qb = quant_block(a);
  if (sub == 0) *v.scale = qb.s;
  float tm[8], nv[8];
  quant8(qb, d, sv, tm, nv);
  store8<T>(static_cast<T*>(v.out), nv);
  __stcs(reinterpret_cast<uint2*>(v.codes), pack_codes(tm));
}

// Each half warp takes two blocks per pass, issuing all four 128-bit loads before
// finishing either block, to keep more bytes in flight per thread.  Blocks that are
// ragged (the last of a segment) or in a misaligned segment are refreshed by a
// second, scalar pass, so that the streaming loop holds no call.
template <typename T>
__global__ void __launch_bounds__(256, 4) refresh_kernel(const __grid_constant__ RefreshTable tab) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;
  const unsigned hmask = 0xFFFFu << (lane & 16);
  const long long group = (long long)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 2 +
                          (lane >> 4);
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5) * 2;
  const long long total = tab.blk_start[tab.nseg];
  if (!tab.early) ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < tab.copy_n; i += blockDim.x) tab.copy_dst[i] = tab.copy_src[i];
  int seg = 0;
  for (long long gb = group; gb < total; gb += 2 * stride) {
    VecBlock v0, v1;
    start_block<T>(tab, gb, total, seg, sub, v0);
    start_block<T>(tab, gb + stride, total, seg, sub, v1);
    if (v0.live) finish_block<T>(v0, sub, hmask);
    if (v1.live) finish_block<T>(v1, sub, hmask);
  }
  // scalar pass: every block of a misaligned segment, the ragged last block of others
  for (int k = 0; k < tab.nseg; ++k) {
    const RefreshSeg& sg = tab.seg[k];
    const long long nblk = tab.blk_start[k + 1] - tab.blk_start[k];
    for (long long j = (sg.vec_ok ? sg.n / 128 : 0) + group; j < nblk; j += stride) {
      const long long e0 = j * 128;
      if (!DPP_IN(e0, min(128ll, sg.n - e0), sg.n) || !DPP_IN(j, 1, (sg.n + 127) / 128))
        continue;  // the same for the 16 lanes
      refresh_block_scalar<T>(reinterpret_cast<const T*>(sg.fresh) + e0,
                              reinterpret_cast<const T*>(sg.stale) + e0,
                              reinterpret_cast<T*>(sg.out) + e0, sg.codes + e0, sg.scales + j,
                              (int)min(128ll, sg.n - e0), sub, hmask);
    }
  }
  if (tab.early) ptx::grid_dep_wait();
}

int launch_refresh(const RefreshTable& tab, int dtype, cudaStream_t stream) {
  const long long total = tab.blk_start[tab.nseg];
  if (total == 0 && tab.copy_n == 0) return DPP_OK;
  const int threads = 256;
  const long long groups_per_cta = threads / 32 * 2 * 2;  // two blocks per group and pass
  long long want = (total + groups_per_cta - 1) / groups_per_cta;
  const long long cap = (long long)dpp_host::sm_count() * 4;  // 4 resident CTAs of 256 per SM
  const int grid = (int)(want < 1 ? 1 : want < cap ? want : cap);  // >= 1 for the side copy
  const cudaError_t e =
      dtype == DPP_BF16
          ? dpp_host::launch_pdl(refresh_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0,
                                 stream, tab)
          : dpp_host::launch_pdl(refresh_kernel<float>, dim3(grid), dim3(threads), 0, stream, tab);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

// ------------------------------------------------------------------ receiver side
// One 128-element block per half warp, 8 elements per lane (codes as one 8-byte load),
// stale streamed in and out.  The code byte becomes an exact float without a
// conversion: the bits of 1.5 * 2^23 plus q (|q| <= 127) are the float 1.5 * 2^23 + q.
template <typename T>
__device__ __forceinline__ void apply8(const int8_t* cd, float s, T* st) {
  const uint2 c = *reinterpret_cast<const uint2*>(cd);
  float sv[8], nv[8];
  if constexpr (sizeof(T) == 2) {
    unpack16(__ldcs(reinterpret_cast<const uint4*>(st)), sv);
  } else {
    float a[4], b[4];
    unpack16(__ldcs(reinterpret_cast<const uint4*>(st)), a);
    unpack16(__ldcs(reinterpret_cast<const uint4*>(st) + 1), b);
#pragma unroll
    for (int i = 0; i < 4; ++i) { sv[i] = a[i]; sv[4 + i] = b[i]; }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int q = (int)(int8_t)((i < 4 ? c.x : c.y) >> (8 * (i & 3)));
    const float qf = __int_as_float(0x4B400000 + q) - kRoundMagic;
    nv[i] = __fmaf_rn(qf, s, sv[i]);
  }
  store8<T>(st, nv);
}

template <typename T>
__global__ void __launch_bounds__(256) apply_kernel(const __grid_constant__ ApplyTable tab) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;
  const long long group = (long long)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 2 +
                          (lane >> 4);
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5) * 2;
  const long long total = tab.blk_start[tab.nseg];
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < tab.copy_n; i += blockDim.x) tab.copy_dst[i] = tab.copy_src[i];
  int seg = 0;
  for (long long gb = group; gb < total; gb += stride) {
    while (gb >= tab.blk_start[seg + 1]) ++seg;
    const ApplySeg& sg = tab.seg[seg];
    const long long j = gb - tab.blk_start[seg];
    const long long e0 = j * 128;
    const int nb = (int)min(128ll, sg.n - e0);
    if (!DPP_IN(j, 1, (sg.n + 127) / 128) || !DPP_IN(e0, nb, sg.n)) continue;
    const float s = sg.scales[j];
    T* st = static_cast<T*>(sg.stale) + e0;
    const int8_t* cd = sg.codes + e0;
    if (nb == 128 && sg.vec_ok) {
      apply8<T>(cd + sub * 8, s, st + sub * 8);
    } else {  // ragged or misaligned: element by element, strided by 16
      for (int e = sub; e < nb; e += 16)
        st[e] = from_f32<T>(__fmaf_rn((float)cd[e], s, to_f32(st[e])));
    }
  }
}

DPP_BOUNDS_READER(bounds_refresh)

int launch_apply(const ApplyTable& tab, int dtype, cudaStream_t stream) {
  const long long total = tab.blk_start[tab.nseg];
  if (total == 0 && tab.copy_n == 0) return DPP_OK;
  const int threads = 256;
  const long long groups_per_cta = threads / 32 * 2 * 4;  // ~4 blocks per half warp
  long long want = (total + groups_per_cta - 1) / groups_per_cta;
  const long long cap = (long long)dpp_host::sm_count() * 8;
  const int grid = (int)(want < 1 ? 1 : want < cap ? want : cap);
  const cudaError_t e =
      dtype == DPP_BF16
          ? dpp_host::launch_pdl(apply_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0, stream,
                                 tab)
          : dpp_host::launch_pdl(apply_kernel<float>, dim3(grid), dim3(threads), 0, stream, tab);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

}  // namespace dpp
