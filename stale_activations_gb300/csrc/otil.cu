// OTIL selective latent transmit on P virtual ranks of one device ("OTIL for SDXL on
// 4x L40S", What is implemented where: each rank scores the K sub-blocks of its own
// slice, sends the top k -- unvisited first, then the highest cosine dissimilarity,
// i.e. topk(dissimilarity + 10 * unvisited, k) -- and every receiver copies them into
// its copy with index_copy_; Self-tests: the local slice is exact, a remote position is
// a received sub-block or stale memory, never a blend; finalize gives every rank the
// exact latent).
//
// The latent (the noise prediction) is [B, C, H, W]; rank p owns rows [p*H/P,
// (p+1)*H/P).  views holds every rank's copy, [P][B, C, H, W].  A sub-block is a
// bh x bw tile of a band over all B and C, numbered row-major over the band.  The
// peers' copy of band p is the same on every receiver (they all applied the same
// messages), so rank (p+1) % P's copy is the one rank p scores against.
//
// otil_step_kernel: one CTA per sender p (it alone writes band p of every view).
//   1. a warp per sub-block: fp32 sums of x.s, x.x, s.s in a fixed order (plane by
//      plane, row by row, lanes across the columns, then an xor-shuffle tree);
//      d = 1 - x.s / sqrt(x.x * s.s) (cos = 0 when a norm is 0); score = d + 10 if the
//      block was not sent since the last reset.
//   2. one thread: k passes of argmax (ties to the lower index), flags set, the
//      selection written in index order.
//   3. the CTA copies the selected blocks into the message and into every other rank's
//      view, and the whole fresh band into its own view.  Copies only.
#include "otil.cuh"
#include "ptx.cuh"

namespace dpp {

namespace {

constexpr int kOtilThreads = 512;

struct OtilDims {
  int B, C, H, W, P, bh, bw, k, Hp, nbc, K;
  long long belem;  // elements of one sub-block: B * C * bh * bw
};

// Offset in a [B, C, H, W] tensor of the top-left element of sub-block i of band p in
// plane (b, ch) = 0.
__device__ __forceinline__ long long block_origin(const OtilDims& d, int p, int i) {
  const int br = i / d.nbc, bc = i - br * d.nbc;
  return ((long long)p * d.Hp + (long long)br * d.bh) * d.W + (long long)bc * d.bw;
}

template <typename T>
__global__ void __launch_bounds__(kOtilThreads) otil_step_kernel(const T* __restrict__ fresh,
                                                                 T* __restrict__ views,
                                                                 uint8_t* __restrict__ visited,
                                                                 int32_t* __restrict__ sel,
                                                                 T* __restrict__ msg, OtilDims d) {
  __shared__ float s_score[kOtilMaxBlocks];
  __shared__ uint8_t s_taken[kOtilMaxBlocks];
  __shared__ int s_sel[kOtilMaxK];
  const int p = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const long long img = (long long)d.B * d.C * d.H * d.W;
  const long long peer0 = (long long)((p + 1) % d.P) * img;  // offset of the peer's view
  const T* peer = views + peer0;
  // 1. scores
  const long long plane = (long long)d.H * d.W;
  const int planes = d.B * d.C;
  for (int i = warp; i < d.K; i += nwarps) {
    float xs = 0.f, xx = 0.f, ss = 0.f;
    const long long o0 = block_origin(d, p, i);
    for (int pl = 0; pl < planes; ++pl)  // plane, row, then lanes across the columns
#pragma unroll 8
      for (int rr = 0; rr < d.bh; ++rr) {
        const long long row = pl * plane + o0 + (long long)rr * d.W;
        for (int cc = lane; cc < d.bw; cc += 32) {
          if (!DPP_IN(row + cc, 1, img) || !DPP_IN(peer0 + row + cc, 1, d.P * img)) continue;
          const float x = to_f32(fresh[row + cc]), s = to_f32(peer[row + cc]);
          xs = fmaf(x, s, xs);
          xx = fmaf(x, x, xx);
          ss = fmaf(s, s, ss);
        }
      }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      xs += __shfl_xor_sync(0xffffffffu, xs, m);
      xx += __shfl_xor_sync(0xffffffffu, xx, m);
      ss += __shfl_xor_sync(0xffffffffu, ss, m);
    }
    if (lane == 0) {
      const float den = sqrtf(xx) * sqrtf(ss);
      const float dis = den > 0.f ? 1.f - xs / den : 1.f;
      const bool seen = DPP_IN((long long)p * d.K + i, 1, (long long)d.P * d.K) &&
                        visited[(long long)p * d.K + i];
      s_score[i] = dis + (seen ? 0.f : 10.f);
      s_taken[i] = 0;
    }
  }
  __syncthreads();
  // 2. top k, ties to the lower index, written in index order
  if (threadIdx.x == 0) {
    for (int j = 0; j < d.k; ++j) {  // k <= K, so some block is always left
      int best = -1;
      for (int i = 0; i < d.K; ++i)
        if (!s_taken[i] && (best < 0 || s_score[i] > s_score[best])) best = i;
      s_sel[j] = best;
      s_taken[best] = 1;
    }
    for (int j = 1; j < d.k; ++j)  // insertion sort by index
      for (int m = j; m > 0 && s_sel[m - 1] > s_sel[m]; --m) {
        const int t = s_sel[m - 1];
        s_sel[m - 1] = s_sel[m];
        s_sel[m] = t;
      }
    for (int j = 0; j < d.k; ++j) {
      if (DPP_IN((long long)p * d.k + j, 1, (long long)d.P * d.k)) sel[(long long)p * d.k + j] = s_sel[j];
      if (DPP_IN((long long)p * d.K + s_sel[j], 1, (long long)d.P * d.K))
        visited[(long long)p * d.K + s_sel[j]] = 1;
    }
  }
  __syncthreads();
  // 3. copies: a warp per (selected block, plane, row), lanes across the columns; the
  // message keeps the block's [B, C, bh, bw] order
  const long long per = (long long)d.k * d.belem;
  const int rows = d.k * planes * d.bh;
#pragma unroll 4
  for (int q = warp; q < rows; q += nwarps) {
    const int j = q / (planes * d.bh), rem = q - j * planes * d.bh;
    const int pl = rem / d.bh, rr = rem - pl * d.bh;
    const long long row = pl * plane + block_origin(d, p, s_sel[j]) + (long long)rr * d.W;
    const long long m0 =
        (long long)p * per + (long long)j * d.belem + ((long long)pl * d.bh + rr) * d.bw;
    T* mrow = msg + m0;
    for (int cc = lane; cc < d.bw; cc += 32) {
      if (!DPP_IN(row + cc, 1, img) || !DPP_IN(m0 + cc, 1, d.P * per)) continue;
      const T v = fresh[row + cc];
      mrow[cc] = v;
      for (int r = 0; r < d.P; ++r)
        if (r != p && DPP_IN((long long)r * img + row + cc, 1, d.P * img))
          views[(long long)r * img + row + cc] = v;
    }
  }
  // own band in full (rows [p*Hp, (p+1)*Hp) of every (b, ch) plane): a warp per
  // (plane, row)
  T* own = views + (long long)p * img;
#pragma unroll 4
  for (int q = warp; q < planes * d.Hp; q += nwarps) {
    const int pl = q / d.Hp, rr = q - pl * d.Hp;
    const long long row = pl * plane + ((long long)p * d.Hp + rr) * d.W;
    for (int cc = lane; cc < d.W; cc += 32)
      if (DPP_IN(row + cc, 1, img) && DPP_IN((long long)p * img + row + cc, 1, d.P * img))
        own[row + cc] = fresh[row + cc];
  }
}

// Every view := fresh; with reset, the unvisited flags are set again.
template <typename T>
__global__ void __launch_bounds__(256) otil_finalize_kernel(const T* __restrict__ fresh,
                                                            T* __restrict__ views,
                                                            uint8_t* __restrict__ visited,
                                                            long long img, int P, int nflags,
                                                            int reset) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const long long n = img * P;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n;
       q += (long long)gridDim.x * blockDim.x)
    views[q] = fresh[q % img];
  if (reset && blockIdx.x == 0)
    for (int i = threadIdx.x; i < nflags; i += blockDim.x) visited[i] = 0;
}

OtilDims dims(const dpp_otil_params& p) {
  OtilDims d{};
  d.B = p.B; d.C = p.C; d.H = p.H; d.W = p.W; d.P = p.P; d.bh = p.bh; d.bw = p.bw; d.k = p.k;
  d.Hp = p.H / p.P;
  d.nbc = p.W / p.bw;
  d.K = (d.Hp / p.bh) * d.nbc;
  d.belem = (long long)p.B * p.C * p.bh * p.bw;
  return d;
}

}  // namespace

DPP_BOUNDS_READER(bounds_otil)

int otil_check(const dpp_otil_params* p) {
  if (!p) return DPP_ERR_NULL;
  if (p->dtype != DPP_BF16 && p->dtype != DPP_F32) return DPP_ERR_DTYPE;
  if (p->B <= 0 || p->C <= 0 || p->H <= 0 || p->W <= 0 || p->P < 2 || p->bh <= 0 || p->bw <= 0)
    return DPP_ERR_SHAPE;
  if (p->H % p->P || (p->H / p->P) % p->bh || p->W % p->bw) return DPP_ERR_SHAPE;
  const long long K = (long long)(p->H / p->P / p->bh) * (p->W / p->bw);
  if (K > kOtilMaxBlocks || p->k < 1 || p->k > K || p->k > kOtilMaxK) return DPP_ERR_SHAPE;
  if ((long long)p->B * p->C * p->H * p->W * p->P >= (1ll << 40)) return DPP_ERR_SHAPE;
  return DPP_OK;
}

int otil_blocks(const dpp_otil_params* p) {
  if (otil_check(p)) return -1;
  return dims(*p).K;
}

int launch_otil_step(const dpp_otil_params& p, const void* fresh, void* views, uint8_t* visited,
                     int32_t* sel, void* msg, cudaStream_t s) {
  const OtilDims d = dims(p);
  cudaError_t e;
  if (p.dtype == DPP_BF16)
    e = dpp_host::launch_pdl(otil_step_kernel<__nv_bfloat16>, dim3(p.P), dim3(kOtilThreads), 0, s,
                             static_cast<const __nv_bfloat16*>(fresh),
                             static_cast<__nv_bfloat16*>(views), visited, sel,
                             static_cast<__nv_bfloat16*>(msg), d);
  else
    e = dpp_host::launch_pdl(otil_step_kernel<float>, dim3(p.P), dim3(kOtilThreads), 0, s,
                             static_cast<const float*>(fresh), static_cast<float*>(views),
                             visited, sel, static_cast<float*>(msg), d);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

int launch_otil_finalize(const dpp_otil_params& p, const void* fresh, void* views,
                         uint8_t* visited, int reset, cudaStream_t s) {
  const OtilDims d = dims(p);
  const long long img = (long long)p.B * p.C * p.H * p.W;
  const long long want = (img * p.P + 255) / 256;
  const int grid = (int)(want < 4ll * dpp_host::sm_count() ? want : 4ll * dpp_host::sm_count());
  cudaError_t e;
  if (p.dtype == DPP_BF16)
    e = dpp_host::launch_pdl(otil_finalize_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s,
                             static_cast<const __nv_bfloat16*>(fresh),
                             static_cast<__nv_bfloat16*>(views), visited, img, p.P, p.P * d.K,
                             reset);
  else
    e = dpp_host::launch_pdl(otil_finalize_kernel<float>, dim3(grid), dim3(256), 0, s,
                             static_cast<const float*>(fresh), static_cast<float*>(views),
                             visited, img, p.P, p.P * d.K, reset);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

}  // namespace dpp
