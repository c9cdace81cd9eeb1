// Tensor-core (tcgen05 + TMA) kernels of the bf16 path.
#pragma once
#include "common.cuh"

namespace dpp {

// Shape checks (host).
bool tc_conv_supported(int B, int H, int W, int Cin, int Cout, int P);
bool tc_linear_supported(long long M, int C);

// out[M, N] = a[M, K] * w[N, K]^T (bf16, fp32 accumulation).  If o1/o2 are
// non-NULL, N is split into three equal column blocks written to o0, o1, o2.
int launch_tc_linear(const void* a, const void* w, void* o0, void* o1, void* o2, long long M,
                     int N, int K, int* status, long long wait_limit, cudaStream_t s);

// The packed Q, K, V projection (N = 3 * ncols, ncols a multiple of 128, 128-wide tiles)
// with the compressed-residual refresh of K and V in its epilogue: besides storing fresh
// K and V (o1, o2), each K / V row block is quantised against k_stale / v_stale and the
// refreshed values go to k_out / v_out (which must not alias the stale inputs: the
// attention still reads them), the codes to codes (K then V, flat) and the block scales
// to scales (the same order) -- the same message and values as the refresh kernel.
// The shapes the GroupNorm-fused conv (gn_par) takes: W % 128 == 0 or 128 % W == 0,
// and (H/P)*W % 128 == 0.
bool tc_conv_gn_supported(int H, int W, int P);

int launch_tc_linear_refresh(const void* a, const void* w, void* o0, void* o1, void* o2,
                             long long M, int N, int K, const void* k_stale, const void* v_stale,
                             void* k_out, void* v_out, int8_t* codes, float* scales,
                             int* status, long long wait_limit, cudaStream_t s);

// Implicit-GEMM halo conv3x3 (see halo_conv3x3 in dpp.h).  With gn_par non-NULL, yf is
// the raw GroupNorm input x and the kernel applies GroupNorm to its in-band rows on the
// fly (gn_par: [B][P][3][Cin] fp32 mean, rstd * gamma, beta); ys is the stale y.
int launch_tc_conv(const void* yf, const void* ys, const void* w, void* out, int B, int H, int W,
                   int Cin, int Cout, int P, const float* gn_par, int* status,
                   long long wait_limit, cudaStream_t s);

// Stale-KV flash attention (see stale_kv_attention in dpp.h), head_dim 64.  With
// `partials` non-NULL the units that do not divide evenly over the CTAs are shared key
// tile by key tile and merged in the kernel; partial_bytes must then be at least
// tc_attention_partial_bytes() (0 when the units divide evenly).  The buffer starts
// with tc_attention_counters() ints that must be zero when the kernel starts: the
// launch zeroes them unless counters_zeroed says an earlier kernel of the stream did
// (the kernel leaves them zero).
int launch_tc_attention(const void* q, const void* kf, const void* vf, const void* ks,
                        const void* vs, void* o, int B, int L, int heads, int P, void* partials,
                        size_t partial_bytes, bool counters_zeroed, int* status,
                        long long wait_limit, cudaStream_t s);
size_t tc_attention_partial_bytes(int B, int L, int heads, int P);
int tc_attention_counters(int B, int L, int heads, int P);

}  // namespace dpp
