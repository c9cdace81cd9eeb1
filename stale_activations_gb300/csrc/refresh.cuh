// Segment table of one refresh launch: several flat buffers refreshed together.
#pragma once
#include "common.cuh"

namespace dpp {

constexpr int kMaxRefreshSegs = 48;

struct RefreshSeg {
  const void* fresh;  // [n] elements of the storage type
  void* stale;        // [n], refreshed in place
  int8_t* codes;      // [n]
  float* scales;      // [ceil(n/128)]
  long long n;
  int vec_ok;         // fresh/stale/codes 16-byte aligned: 128-bit path for full blocks
  int pad_;
};

struct RefreshTable {
  RefreshSeg seg[kMaxRefreshSegs];
  long long blk_start[kMaxRefreshSegs + 1];  // prefix sums of ceil(n/128)
  int nseg;
  // an exact fp32 copy done on the side by CTA 0 (the layer's GroupNorm sums), or none
  int copy_n;
  const float* copy_src;
  float* copy_dst;
};

// Launches one refresh over all segments of `tab` (blk_start filled by caller).
int launch_refresh(const RefreshTable& tab, int dtype, cudaStream_t stream);

}  // namespace dpp
