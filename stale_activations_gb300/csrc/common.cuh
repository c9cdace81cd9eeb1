// Shared device/host helpers of the displaced-patch layer library (sm_103a).
#pragma once
#include <utility>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dpp.h"

namespace dpp {

constexpr int kNumSMs = 152;              // GB300: 2 dies x 76 SMs (grid sizing hint)
// Bounded waits: no legitimate wait in these kernels lasts more than microseconds.
// Each try may suspend the waiting thread for up to ~20 us (it wakes as soon as
// the phase completes), so 2^16 tries bound a wait to about a second.
constexpr long long kDefaultWaitLimit = 1ll << 16;  // bounded-wait iterations
constexpr long long kDrainWaitLimit = 1ll << 16;    // waits for own copies before exit

// ------------------------------------------------------------ storage types
template <typename T> struct Vec;  // 16-byte vector of T
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Unpack a 16-byte vector of T into fp32 values.
__device__ __forceinline__ void unpack16(const uint4& u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack16(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint4 pack16(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Record a device-side failure: the first code wins.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ index checks
// In a library built with -DDPP_DEBUG_BOUNDS every kernel checks each global-memory index
// it computes against the extent of the tensor it addresses, as the call's shapes give it
// (TMA copies are clipped to their tensor maps by the copy engine itself and are not
// checked): DPP_IN(i, n, extent) is true when elements [i, i + n) lie in [0, extent);
// otherwise the access is skipped and the first such index of this translation unit is
// recorded (source line, index, extent) for dpp_debug_bounds().  Without the flag DPP_IN
// is the constant true and the checks compile away.
#ifdef DPP_DEBUG_BOUNDS
namespace {  // one record per translation unit
__device__ long long g_bounds[3];  // source line (0: none), index, extent
__device__ int g_bounds_claim;
__device__ __noinline__ bool bounds_violation(long long i, long long ext, int line) {
  if (atomicCAS(&g_bounds_claim, 0, 1) == 0) {
    g_bounds[1] = i;
    g_bounds[2] = ext;
    __threadfence();
    atomicExch(reinterpret_cast<unsigned long long*>(&g_bounds[0]), (unsigned long long)line);
  }
  return false;
}
__device__ __forceinline__ bool in_extent(long long i, long long n, long long ext, int line) {
  return (i >= 0 && n >= 0 && i + n <= ext) ? true : bounds_violation(i, ext, line);
}
}  // namespace
#define DPP_IN(i, n, ext) \
  ::dpp::in_extent((long long)(i), (long long)(n), (long long)(ext), __LINE__)
// The host reader of this translation unit's record: rec = {line, index, extent}.
#define DPP_BOUNDS_READER(fn)                                                           \
  int fn(long long* rec, int reset) {                                                   \
    if (cudaMemcpyFromSymbol(rec, g_bounds, sizeof(g_bounds)) != cudaSuccess)          \
      return DPP_ERR_CUDA;                                                              \
    if (reset) {                                                                        \
      const long long z[3] = {0, 0, 0};                                                 \
      const int zi = 0;                                                                 \
      if (cudaMemcpyToSymbol(g_bounds, z, sizeof(z)) != cudaSuccess ||                  \
          cudaMemcpyToSymbol(g_bounds_claim, &zi, sizeof(zi)) != cudaSuccess)          \
        return DPP_ERR_CUDA;                                                            \
    }                                                                                   \
    return DPP_OK;                                                                      \
  }
#else
#define DPP_IN(i, n, ext) true
#define DPP_BOUNDS_READER(fn)
#endif

}  // namespace dpp

// ------------------------------------------------------------ host helpers
namespace dpp_host {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
long long wait_limit_from_env();  // DPP_DEBUG_WAIT_LIMIT, else the default
// DPP_DEBUG_SKIP_LOAD=<kind>:<i> (kind "attn", "conv" or "linear"): a test hook that makes the TMA
// producer of every CTA of that kernel kind leave its i-th load unissued, so that the
// kernel's bounded waits give up and report DPP_ERR_TIMEOUT; -1 when unset
int skip_load_from_env(const char* kind);
int sm_count();                   // SMs of the current device (cached per device)

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialization (the kernel calls ptx::grid_dep_wait before its first dependent
// memory access).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dpp_host

#define DPP_CUDA_CHECK(expr)                 \
  do {                                       \
    cudaError_t _e = (expr);                 \
    if (_e != cudaSuccess) return DPP_ERR_CUDA; \
  } while (0)
