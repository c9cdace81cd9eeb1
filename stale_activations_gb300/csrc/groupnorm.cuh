#pragma once
#include "common.cuh"

namespace dpp {

struct GnDims {
  int B, H, W, C, P, G;
  int Hp;              // rows per patch
  int nchunk;          // pixel chunks per (batch, patch)
  long long chunk_pix; // pixels per chunk
};

GnDims make_gn_dims(int B, int H, int W, int C, int P, int G);
size_t gn_partial_bytes(const GnDims& g);

// Launches the stats and apply kernels.  mode: DPP_GN_SPLICED, DPP_GN_SYNC (every patch
// fresh; the synchronous step) or DPP_GN_PREVIOUS; stale_stats may be NULL under
// DPP_GN_SYNC.
// fresh_out (may be NULL) receives the [B,P,G,2] fresh sums.  The stats kernel
// zeroes *status_to_zero first (if non-NULL), and the nzero ints at zero_ints (the next
// kernels' counters).  params_out (may be NULL): [B][P][3][C] fp32 mean, rstd * gamma,
// beta per channel.  vstale (bf16, not with halo_only; may be NULL): also the max |V| of
// this stale [B, H*W, C] tensor per (batch, head of 64 channels), into vmax [B][heads] as
// fp32 bits by atomicMax (vmax zeroed by the stats kernel, as part of zero_ints).
// halo_only: y is written only for each band's first and last rows
// (the rows the neighbouring bands read as halos), the rest being applied by a fused
// consumer.
int launch_gn(const void* x, void* y, float* partial, const float* stale_stats, float* fresh_out,
              const float* gamma, const float* beta, const GnDims& g, float eps, int mode,
              int dtype, int* status_to_zero, int* zero_ints, int nzero, float* params_out,
              int halo_only, const void* vstale, unsigned* vmax, int heads,
              cudaStream_t stream);

}  // namespace dpp
