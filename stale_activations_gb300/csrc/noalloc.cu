// patch_layer_step_noalloc: the layer step for callers that cannot allocate
// device memory when they run a layer.
//
// Such callers exist: a plugin inside a host framework that owns every byte of
// device memory through its own allocator and budget (a foreign cudaMalloc would
// bypass its accounting or fail against its limit), or a latency-critical loop in
// which cudaMalloc's implicit synchronisation and unbounded latency are not
// allowed.  They still pass inputs, weights, state and outputs; the workspace that
// patch_layer_step normally takes from the caller comes from one fixed array of
// device memory that this file owns.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes.  Every
// GPU that loads this part of the library keeps it until the process exits.  The
// host never uses the array's name as an address: once per device, with that
// device current, the first call looks up its device address with
// cudaGetSymbolAddress and caches it.
//
// The library has no counterpart of this entry point on the pages it follows; it
// exists only for the allocation constraint above.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 80ull << 20;  // 80 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on first use).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DPP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DPP_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DPP_OK;
}

}  // namespace

extern "C" int patch_layer_step_noalloc(const dpp_layer_params* prm,
                                        const dpp_layer_weights* wts,
                                        const dpp_layer_state* st, const void* x, void* out,
                                        int mode, void* stream) {
  dpp_workspace_layout lo;
  int rc = dpp_workspace_query(prm, &lo);
  if (rc) return rc;
  if (lo.total > kNoAllocScratchBytes) return DPP_ERR_SCRATCH_LIMIT;
  if (!wts || !st || !x || !out) return DPP_ERR_NULL;
  if (mode != DPP_SYNC && mode != DPP_STALE) return DPP_ERR_ARG;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  // patch_layer_step zeroes the status word at offset 0 in its first kernel; every
  // other workspace byte is written before it is read within the same call.
  return patch_layer_step(prm, wts, st, x, out, mode, scratch, stream);
}

// The device status word of the last patch_layer_step_noalloc on the current device
// (offset 0 of the fixed scratch, zeroed at the start of each call and set by a kernel
// whose bounded wait gave up): synchronizes `stream` and returns it, like
// dpp_read_device_status does for a caller's workspace.  Allocates nothing.
extern "C" int dpp_noalloc_read_status(void* stream) {
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  int v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DPP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DPP_ERR_CUDA;
  return v;
}
