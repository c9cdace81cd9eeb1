// Tensor-core (tcgen05 + TMA) kernels of the bf16 path.
#pragma once
#include "common.cuh"

namespace dpp {

// Shape checks (host).
bool tc_conv_supported(int B, int H, int W, int Cin, int Cout, int P);
bool tc_linear_supported(long long M, int C);

// out[M, N] = a[M, K] * w[N, K]^T (bf16, fp32 accumulation).  If o1/o2 are
// non-NULL, N is split into three equal column blocks written to o0, o1, o2.
// With vmax non-NULL (three-way split only, vmax_L a multiple of 128): also the max |o2|
// per (batch of vmax_L rows, 64-column head) into vmax [batches][vmax_heads] as fp32 bits
// by atomicMax (vmax zeroed before the launch).
int launch_tc_linear(const void* a, const void* w, void* o0, void* o1, void* o2, long long M,
                     int N, int K, int* status, long long wait_limit, cudaStream_t s,
                     unsigned* vmax = nullptr, int vmax_L = 0, int vmax_heads = 0);

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
// vstale (bf16 [B, H*W, vs_C], may be NULL, not with gn_par): the launch also takes its
// max |.| per (batch, head of 64 channels) into vmax [B][heads] as fp32 bits by atomicMax
// (vmax zeroed before the launch): with extra CTAs on the SMs the tiles leave idle, or by
// the epilogue warps while the first accumulator fills.
int launch_tc_conv(const void* yf, const void* ys, const void* w, void* out, int B, int H, int W,
                   int Cin, int Cout, int P, const float* gn_par, int* status,
                   long long wait_limit, cudaStream_t s, const void* vstale = nullptr,
                   int vs_C = 0, unsigned* vmax = nullptr, int heads = 0);

// Stale-KV flash attention (see stale_kv_attention in dpp.h), head_dim 64.  `scratch`
// (tc_attention_scratch_bytes() bytes) holds the per-(batch, head) maxima of |V| that
// set V's fp16 scaling and, with `split`, the counters and partial records of the units
// shared key tile by key tile; its first tc_attention_zero_ints() ints must be zero when
// the launch runs: the launch zeroes them unless scratch_zeroed says an earlier kernel of
// the stream did (the kernel leaves the counters zero, not the maxima).  Launches a
// small max|V| pass, then the attention kernel.  skip_load (test hook, normally -1):
// the producer of every CTA leaves the K/V tile of that step unloaded, so the kernel's
// bounded waits give up with DPP_ERR_TIMEOUT.
// vmax_ready: the maxima at the start of the scratch were already computed by earlier
// kernels of the stream (then the max |V| pass is not launched; scratch_zeroed must hold).
int launch_tc_attention(const void* q, const void* kf, const void* vf, const void* ks,
                        const void* vs, void* o, int B, int L, int heads, int P, bool split,
                        void* scratch, size_t scratch_bytes, bool scratch_zeroed,
                        bool vmax_ready, int* status, long long wait_limit, int skip_load,
                        cudaStream_t s);
size_t tc_attention_scratch_bytes(int B, int L, int heads, int P, bool split);
int tc_attention_zero_ints(int B, int L, int heads, int P, bool split);

}  // namespace dpp
