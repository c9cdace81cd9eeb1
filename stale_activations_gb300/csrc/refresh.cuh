// Segment table of one refresh launch: several flat buffers refreshed together.
#pragma once
#include "common.cuh"

namespace dpp {

constexpr int kMaxRefreshSegs = 48;

struct RefreshSeg {
  const void* fresh;  // [n] elements of the storage type
  void* stale;        // [n] the stale values
  int8_t* codes;      // [n]
  float* scales;      // [ceil(n/128)]
  long long n;
  int vec_ok;         // fresh/stale/out/codes 16-byte aligned: 128-bit path for full blocks
  int pad_;
  void* out;          // [n] where the refreshed values go (== stale: in place)
};

struct RefreshTable {
  RefreshSeg seg[kMaxRefreshSegs];
  long long blk_start[kMaxRefreshSegs + 1];  // prefix sums of ceil(n/128)
  int nseg;
  // an exact fp32 copy done on the side by CTA 0 (the layer's GroupNorm sums), or none
  int copy_n;
  const float* copy_src;
  float* copy_dst;
  // 1 when the kernel launched just before this one neither reads nor writes any buffer
  // of the table, and every kernel that does has completed before that one started
  // (its griddepcontrol.wait returned): the refresh then runs alongside it and waits
  // for it only at the end, which keeps completion ordered down the stream
  int early;
};

// Launches one refresh over all segments of `tab` (blk_start filled by caller).
int launch_refresh(const RefreshTable& tab, int dtype, cudaStream_t stream);

// The receiver's half: stale <- store(fmaf(q, s, stale)) from a message (codes, one
// scale per 128-element block), the same arithmetic as the sender's refresh, so a copy
// fed only the messages stays bit-identical to the sender's.
struct ApplySeg {
  const int8_t* codes;  // [n]
  const float* scales;  // [ceil(n/128)]
  void* stale;          // [n] elements of the storage type, updated in place
  long long n;
  int vec_ok;           // codes/stale 16-byte aligned: 8 elements per lane for full blocks
  int pad_;
};

struct ApplyTable {
  ApplySeg seg[kMaxRefreshSegs];
  long long blk_start[kMaxRefreshSegs + 1];  // prefix sums of ceil(n/128)
  int nseg;
  int copy_n;  // an exact fp32 copy done on the side by CTA 0, or none
  const float* copy_src;
  float* copy_dst;
};

int launch_apply(const ApplyTable& tab, int dtype, cudaStream_t stream);

}  // namespace dpp
