// GroupNorm with spliced stale statistics ("OTIL for SDXL on 4x L40S", What is
// implemented where: DistriGroupNorm carries stale context; GroupNorm sync
// without the rest: two scalars per group).
//
// gn_stats: per (batch, patch, chunk of the patch's pixels) the fp32 sums
//   (sum x, sum x^2) of every group.  Each thread owns one 16-byte channel
//   vector and walks pixels, so loads are 128-bit and coalesced along C; the
//   per-channel sums are reduced across the block in shared memory and then
//   folded into groups in a fixed order (deterministic, no atomics).
// gn_apply: patch p's statistics = its own fresh sums (summed over chunks) +
//   the other patches' stale sums (fresh ones at the synchronous step and under
//   DPP_GN_SYNC; under DPP_GN_PREVIOUS its own sums are the stale ones too);
//   mu = S1/N, var = max(S2/N - mu^2, 0), y = (x - mu) * rstd * gamma + beta.
// Both are HBM-bound streams: stats reads 1 element, apply reads 1 and writes 1.
#include "groupnorm.cuh"
#include "ptx.cuh"

namespace dpp {

// Threads that share one sum in a 256-thread block reducing `nsum` sums: the largest
// power of two <= min(32, 256 / nsum), at least 1 (lanes of one warp, aligned).
__device__ __forceinline__ int lanes_per_sum(int nsum) {
  int t = nsum >= 256 ? 1 : 256 / nsum;
  if (t > 32) t = 32;
  while (t & (t - 1)) t &= t - 1;
  return t;
}

// Pixels a thread loads before it uses any of them (one batch in flight).
constexpr int kGnBatch = 8;

template <typename T>
__global__ void __launch_bounds__(256) gn_stats_kernel(const T* __restrict__ x,
                                                       float* __restrict__ partial, GnDims g,
                                                       int* status_to_zero, int* zero_ints,
                                                       int nzero) {
  constexpr int VEC = Vec<T>::N;
  extern __shared__ float red[];  // [2][PIX][C]
  const int chunk = blockIdx.x, p = blockIdx.y, b = blockIdx.z;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (chunk == 0 && p == 0 && b == 0) {
    if (status_to_zero && threadIdx.x == 0) *status_to_zero = 0;
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero_ints[i] = 0;
  }
  const int NV = g.C / VEC;
  const int PIX = 256 / NV;
  const int tid = threadIdx.x;
  const int pl = tid / NV, v = tid % NV;
  const long long band_pix = (long long)g.Hp * g.W;
  const long long p0 = (long long)chunk * g.chunk_pix;
  const long long p1 = min(band_pix, p0 + g.chunk_pix);
  float s1[VEC], s2[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) { s1[i] = 0.f; s2[i] = 0.f; }
  const long long act = (long long)g.B * g.H * g.W * g.C;  // elements of x
  if (pl < PIX) {
    const long long xo = (((long long)b * g.H + (long long)p * g.Hp) * g.W) * g.C + v * VEC;
    const T* base = x + xo;
    for (long long px = p0 + pl; px < p1; px += kGnBatch * PIX) {
      uint4 u[kGnBatch];
#pragma unroll
      for (int k = 0; k < kGnBatch; ++k)
        if (px + k * PIX < p1 && DPP_IN(xo + (px + k * PIX) * g.C, VEC, act))
          u[k] = __ldg(reinterpret_cast<const uint4*>(base + (px + k * PIX) * g.C));
#pragma unroll
      for (int k = 0; k < kGnBatch; ++k) {
        if (px + k * PIX >= p1) break;
        float f[VEC];
        unpack16(u[k], f);
#pragma unroll
        for (int i = 0; i < VEC; ++i) { s1[i] += f[i]; s2[i] = fmaf(f[i], f[i], s2[i]); }
      }
    }
    float* r1 = red + (long long)pl * g.C + v * VEC;
    float* r2 = red + (long long)PIX * g.C + (long long)pl * g.C + v * VEC;
#pragma unroll
    for (int i = 0; i < VEC; ++i) { r1[i] = s1[i]; r2[i] = s2[i]; }
  }
  __syncthreads();
  // fold channels into groups: tpg threads per group, each summing a fixed stride of the
  // group's (pixel lane, channel) values, then a shuffle tree over the tpg lanes (a
  // fixed order, so the sums are deterministic)
  const int cg = g.C / g.G;
  const int tpg = lanes_per_sum(g.G);
  const int n = PIX * cg;
  for (int t0 = 0; t0 < g.G * tpg; t0 += blockDim.x) {
    const int t = t0 + tid, gi = t / tpg, part = t % tpg;
    float a = 0.f, q = 0.f;
    if (gi < g.G)
      for (int j = part; j < n; j += tpg) {
        const int k = j / cg, c = gi * cg + (j - k * cg);
        a += red[(long long)k * g.C + c];
        q += red[(long long)PIX * g.C + (long long)k * g.C + c];
      }
    for (int m = tpg >> 1; m > 0; m >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, m);
      q += __shfl_xor_sync(0xffffffffu, q, m);
    }
    const long long po = ((((long long)b * g.P + p) * g.nchunk + chunk) * g.G + gi) * 2;
    if (gi < g.G && part == 0 && DPP_IN(po, 2, (long long)g.B * g.P * g.nchunk * g.G * 2)) {
      partial[po] = a;
      partial[po + 1] = q;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) gn_apply_kernel(const T* __restrict__ x, T* __restrict__ y,
                                                       const float* __restrict__ partial,
                                                       const float* __restrict__ stale_stats,
                                                       float* __restrict__ fresh_out,
                                                       const float* __restrict__ gamma,
                                                       const float* __restrict__ beta, GnDims g,
                                                       float eps, int mode,
                                                       float* __restrict__ params_out,
                                                       int halo_only, const T* __restrict__ vstale,
                                                       unsigned* __restrict__ vmax, int heads) {
  constexpr int VEC = Vec<T>::N;
  __shared__ unsigned s_hmax[32];  // max |V_stale| bits per head of this block
  extern __shared__ float sm[];  // group sums [P][G][2], then mean and rstd [G][2]
  const bool all_fresh = mode == DPP_GN_SYNC;
  const int G2 = g.G * 2;
  float* s_tot = sm;  // own patch fresh, the others fresh or stale
  float* s_grp = sm + g.P * G2;
  const int chunk = blockIdx.x, p = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  // each thread keeps one 16-byte channel vector (and its parameters in registers) and
  // walks the block's pixels
  const int NV = g.C / VEC;
  const int PIX = 256 / NV;
  const int pl = tid / NV, v = tid % NV;
  const bool active = pl < PIX;
  const long long band_pix = (long long)g.Hp * g.W;
  long long p0 = (long long)chunk * g.chunk_pix;
  long long p1 = min(band_pix, p0 + g.chunk_pix);
  bool rows = true;
  if (halo_only) {  // block 0: the band's first row (p > 0), block 1: its last (p < P-1)
    rows = !((chunk == 0 && p == 0) || (chunk == 1 && p == g.P - 1));
    p0 = chunk == 0 ? 0 : (long long)(g.Hp - 1) * g.W;
    p1 = p0 + g.W;
  }
  const long long base = (((long long)b * g.H + (long long)p * g.Hp) * g.W) * g.C + v * VEC;
  const long long act = (long long)g.B * g.H * g.W * g.C;  // elements of x, y and the stale V
  const long long nstat = (long long)g.B * g.P * G2;       // [B, P, G, 2] sums

  // What does not depend on the stats kernel is fetched before waiting for it: the first
  // batch of x, this thread's gamma and beta, the stale sums.  (Every block of the
  // stats kernel has passed its own wait for the kernels before it when this grid
  // starts, so their outputs are complete.)
  uint4 u[kGnBatch];
  long long px = p0 + pl;
  if (active && rows) {
#pragma unroll
    for (int k = 0; k < kGnBatch; ++k)
      if (px + k * PIX < p1 && DPP_IN(base + (px + k * PIX) * g.C, VEC, act))
        u[k] = __ldcs(reinterpret_cast<const uint4*>(x + base + (px + k * PIX) * g.C));
  }
  float ga[VEC], be[VEC];
  if (active && DPP_IN(v * VEC, VEC, g.C)) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      ga[k] = __ldg(gamma + v * VEC + k);
      be[k] = __ldg(beta + v * VEC + k);
    }
  }
  if (!all_fresh)
    for (int idx = tid; idx < g.P * G2; idx += blockDim.x)
      if (idx / G2 != p && DPP_IN((long long)b * g.P * G2 + idx, 1, nstat))
        s_tot[idx] = stale_stats[(long long)b * g.P * G2 + idx];
  // The stale V has x's layout ([B, H*W, C]): its max |V| per (batch, head) over this
  // block's pixels, for the attention's fp16 scaling of V.  It is state written before the
  // stats kernel started, so it is read before the wait; the per-(batch, head) maxima are
  // zeroed by the stats kernel, so they are updated after it.
  if (vstale) {
    if (tid < 32) s_hmax[tid] = 0;
    __syncthreads();
    unsigned vm = 0;
    if (active) {
      for (long long q = p0 + pl; q < p1; q += 4 * PIX) {
        uint4 w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (q + k * PIX < p1 && DPP_IN(base + (q + k * PIX) * g.C, VEC, act))
            w[k] = __ldcs(reinterpret_cast<const uint4*>(vstale + base + (q + k * PIX) * g.C));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (q + k * PIX < p1) {
            const uint32_t h4[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              vm = max(vm, max(h4[e] & 0x7FFFu, (h4[e] >> 16) & 0x7FFFu));
          }
      }
      if (vm) atomicMax(&s_hmax[(v * VEC) / 64], vm);
    }
    __syncthreads();
  }
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (vstale && tid < heads && s_hmax[tid] &&
      DPP_IN((long long)b * heads + tid, 1, (long long)g.B * heads))
    atomicMax(vmax + (long long)b * heads + tid, s_hmax[tid] << 16);  // bf16 -> fp32 bits
  // fresh sums over chunks, for own patch (and every patch when all are fresh): tps
  // threads per sum, each a fixed stride of chunks with eight loads in flight, then a
  // shuffle tree (fixed order)
  const int nq = all_fresh ? g.P : 1;
  const int tps = lanes_per_sum(nq * G2);
  for (int t0 = 0; t0 < nq * G2 * tps; t0 += blockDim.x) {
    const int t = t0 + tid, si = t / tps, part = t % tps;
    const int q = all_fresh ? si / G2 : p, r = si % G2;
    float val = 0.f;
    if (si < nq * G2) {
      const long long so = (((long long)b * g.P + q) * g.nchunk) * G2 + r;
      const long long npart = (long long)g.B * g.P * g.nchunk * G2;
      const float* src = partial + so;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      int c = part;
      for (; c + 7 * tps < g.nchunk; c += 8 * tps) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (DPP_IN(so + (long long)(c + k * tps) * G2, 1, npart))
            acc[k] += src[(long long)(c + k * tps) * G2];
      }
#pragma unroll
      for (int k = 0; k < 7; ++k)
        if (c + k * tps < g.nchunk && DPP_IN(so + (long long)(c + k * tps) * G2, 1, npart))
          acc[k] += src[(long long)(c + k * tps) * G2];
      val = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    }
    for (int m = tps >> 1; m > 0; m >>= 1) val += __shfl_xor_sync(0xffffffffu, val, m);
    if (si < nq * G2 && part == 0) s_tot[q * G2 + r] = val;
  }
  __syncthreads();
  if (chunk == 0 && fresh_out)
    for (int r = tid; r < G2; r += blockDim.x)
      if (DPP_IN(((long long)b * g.P + p) * G2 + r, 1, nstat))
        fresh_out[((long long)b * g.P + p) * G2 + r] = s_tot[p * G2 + r];
  // group statistics: own patch first (its previous-step sums under DPP_GN_PREVIOUS),
  // then the others in order; mu = S1/N, var = max(S2/N - mu^2, 0)
  const int cg = g.C / g.G;
  const double invN = 1.0 / ((double)g.H * g.W * cg);
  const float* own = mode == DPP_GN_PREVIOUS ? stale_stats + ((long long)b * g.P + p) * G2
                                             : s_tot + p * G2;
  for (int gi = tid; gi < g.G; gi += blockDim.x) {
    float S1 = 0.f, S2 = 0.f;
    if (mode != DPP_GN_PREVIOUS || DPP_IN(((long long)b * g.P + p) * G2 + gi * 2, 2, nstat)) {
      S1 = own[gi * 2];
      S2 = own[gi * 2 + 1];
    }
    for (int q = 0; q < g.P; ++q)
      if (q != p) { S1 += s_tot[q * G2 + gi * 2]; S2 += s_tot[q * G2 + gi * 2 + 1]; }
    const float mu = (float)(S1 * invN);
    const float var = fmaxf((float)(S2 * invN) - mu * mu, 0.f);
    s_grp[gi * 2] = mu;
    s_grp[gi * 2 + 1] = rsqrtf(var + eps);
  }
  __syncthreads();
  if (!active) return;
  float mu[VEC], sc[VEC];
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int gi = (v * VEC + k) / cg;
    mu[k] = s_grp[gi * 2];
    sc[k] = s_grp[gi * 2 + 1] * ga[k];
  }
  if (params_out && chunk == 0 && pl == 0 &&  // the per-channel parameters, for a fused consumer
      DPP_IN(((long long)b * g.P + p) * 3 * g.C + v * VEC, 2 * g.C + VEC,
             (long long)g.B * g.P * 3 * g.C)) {
    float* dst = params_out + ((long long)b * g.P + p) * 3 * g.C + v * VEC;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      dst[k] = mu[k];
      dst[g.C + k] = sc[k];
      dst[2 * g.C + k] = be[k];
    }
  }
  if (!rows) return;
  for (;;) {
#pragma unroll
    for (int k = 0; k < kGnBatch; ++k) {
      if (px + k * PIX >= p1) break;
      float f[VEC];
      unpack16(u[k], f);
#pragma unroll
      for (int i = 0; i < VEC; ++i) f[i] = fmaf(f[i] - mu[i], sc[i], be[i]);
      if (DPP_IN(base + (px + k * PIX) * g.C, VEC, act))
        *reinterpret_cast<uint4*>(y + base + (px + k * PIX) * g.C) = pack16(f);
    }
    px += kGnBatch * PIX;
    if (px >= p1) break;
#pragma unroll
    for (int k = 0; k < kGnBatch; ++k)
      if (px + k * PIX < p1 && DPP_IN(base + (px + k * PIX) * g.C, VEC, act))
        u[k] = __ldcs(reinterpret_cast<const uint4*>(x + base + (px + k * PIX) * g.C));
  }
}

DPP_BOUNDS_READER(bounds_groupnorm)

GnDims make_gn_dims(int B, int H, int W, int C, int P, int G) {
  GnDims g;
  g.B = B; g.H = H; g.W = W; g.C = C; g.P = P; g.G = G;
  g.Hp = H / P;
  const long long band_pix = (long long)g.Hp * W;
  // two blocks per SM in one wave (the apply kernel holds a batch of x in registers,
  // which allows two 256-thread blocks per SM); long per-thread pixel runs stream best
  long long nchunk = (2ll * kNumSMs + (long long)B * P - 1) / ((long long)B * P);
  if (nchunk > band_pix) nchunk = band_pix;
  if (nchunk < 1) nchunk = 1;
  g.chunk_pix = (band_pix + nchunk - 1) / nchunk;
  g.nchunk = (int)((band_pix + g.chunk_pix - 1) / g.chunk_pix);
  return g;
}

size_t gn_partial_bytes(const GnDims& g) {
  return (size_t)g.B * g.P * g.nchunk * g.G * 2 * sizeof(float);
}

int launch_gn(const void* x, void* y, float* partial, const float* stale_stats, float* fresh_out,
              const float* gamma, const float* beta, const GnDims& g, float eps, int mode,
              int dtype, int* status_to_zero, int* zero_ints, int nzero, float* params_out,
              int halo_only, const void* vstale, unsigned* vmax, int heads,
              cudaStream_t stream) {
  dim3 grid(g.nchunk, g.P, g.B);
  const dim3 agrid = halo_only ? dim3(2, g.P, g.B) : grid;
  const int VEC = dtype == DPP_BF16 ? 8 : 4;
  const int NV = g.C / VEC;
  const int PIX = 256 / NV;
  const size_t red_bytes = 2ull * PIX * g.C * sizeof(float);
  const size_t app_bytes = (2ull * g.P * g.G + 2ull * g.G) * sizeof(float);
  using dpp_host::launch_pdl;
  cudaError_t e;
  if (dtype == DPP_BF16) {
    auto* xs = static_cast<const __nv_bfloat16*>(x);
    e = launch_pdl(gn_stats_kernel<__nv_bfloat16>, grid, dim3(256), red_bytes, stream, xs, partial,
                   g, status_to_zero, zero_ints, nzero);
    if (e == cudaSuccess)
      e = launch_pdl(gn_apply_kernel<__nv_bfloat16>, agrid, dim3(256), app_bytes, stream, xs,
                     static_cast<__nv_bfloat16*>(y), (const float*)partial, stale_stats, fresh_out,
                     gamma, beta, g, eps, mode, params_out, halo_only,
                     static_cast<const __nv_bfloat16*>(vstale), vmax, heads);
  } else {
    auto* xs = static_cast<const float*>(x);
    e = launch_pdl(gn_stats_kernel<float>, grid, dim3(256), red_bytes, stream, xs, partial, g,
                   status_to_zero, zero_ints, nzero);
    if (e == cudaSuccess)
      e = launch_pdl(gn_apply_kernel<float>, agrid, dim3(256), app_bytes, stream, xs,
                     static_cast<float*>(y), (const float*)partial, stale_stats, fresh_out, gamma,
                     beta, g, eps, mode, params_out, halo_only, nullptr, nullptr, 0);
  }
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

}  // namespace dpp
