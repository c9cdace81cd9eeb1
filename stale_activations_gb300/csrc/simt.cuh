#pragma once
#include "common.cuh"

namespace dpp {

// Output of a GEMM whose N columns are split into equal column blocks, each
// written to its own [M, ncols] buffer (Q, K, V of the packed projection).
struct SimtOut {
  void* ptr[3];
  int ncols;
};

int launch_simt_linear(const void* a, const void* w, const SimtOut& out, long long M, int N, int K,
                       int dtype, cudaStream_t stream);
int launch_simt_conv(const void* yf, const void* ys, const void* w, void* out, int B, int H, int W,
                     int Cin, int Cout, int P, int dtype, cudaStream_t stream);
int launch_simt_attention(const void* q, const void* kf, const void* vf, const void* ks,
                          const void* vs, void* o, int B, int L, int heads, int P, int dtype,
                          cudaStream_t stream);

}  // namespace dpp
