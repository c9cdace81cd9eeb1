// fp32 SIMT kernels: the arithmetic path of fp32-storage layers (tcgen05 has no
// full-precision fp32 kind, and TF32 cannot meet fp32 tolerances).
//
// simt_gemm: C[m, n] = sum_k A[m, k] * Wt[n, k] with a 64x64 output tile per
//   block, 16-wide K slices staged in shared memory, 4x4 outputs per thread.
//   A is either a plain row-major matrix (projections) or the implicit im2col
//   view of the halo conv: row m = pixel (b, r, c), column k = (tap, cin), the
//   tap's source row taken from the fresh map inside r's band, from the stale
//   map for the band's two halo rows, zero outside the image ("Benchmarking
//   DistVAE", Glossary: halo rows of a sharded convolution).
// simt_attention: one warp per query row of one patch and head (lanes split the keys);
//   64-key tiles of the spliced K/V (own patch fresh, other rows stale) in shared
//   memory; online softmax in fp32.
#include "simt.cuh"

namespace dpp {

// The A operand seen by one thread: a fixed set of rows (prepared once per row, no
// divisions afterwards) and a column k that advances by 16 per K slice.
struct ALinear {
  const void* a;
  int K;
#ifdef DPP_DEBUG_BOUNDS
  long long n_a;  // elements of A (M * K), for the index checks
#endif
  struct Row {
    long long m;
    bool ok;
  };
  __device__ __forceinline__ Row row(long long m, long long M) const { return Row{m, m < M}; }
  struct Col {
    int k;
  };
  __device__ __forceinline__ Col col(int k) const { return Col{k}; }
  __device__ __forceinline__ void advance(Col& c, int step) const { c.k += step; }
  template <typename T>
  __device__ __forceinline__ float load(const Row& r, const Col& c) const {
#ifdef DPP_DEBUG_BOUNDS
    if (r.ok && c.k < K && !DPP_IN(r.m * K + c.k, 1, n_a)) return 0.f;
#endif
    return r.ok && c.k < K ? to_f32(static_cast<const T*>(a)[r.m * K + c.k]) : 0.f;
  }
};

struct AConv {
  const void* yf;
  const void* ys;
  int H, W, Cin, Hp;
#ifdef DPP_DEBUG_BOUNDS
  long long n_y;  // elements of each input map (B * H * W * Cin), for the index checks
#endif
  struct Row {  // pixel (b, r, c) and its band [lo, lo + Hp)
    long long img;  // offset of image b
    int r, c, lo;
    bool ok;
  };
  __device__ __forceinline__ Row row(long long m, long long M) const {
    Row x{};
    x.ok = m < M;
    const long long hw = (long long)H * W;
    const long long b = x.ok ? m / hw : 0;
    const int rem = (int)(m - b * hw);
    x.r = rem / W;
    x.c = rem - x.r * W;
    x.lo = (x.r / Hp) * Hp;
    x.img = b * hw;
    return x;
  }
  struct Col {  // k = tap * Cin + ci, tap = (di + 1) * 3 + (dj + 1)
    int k, ci, di, dj;
  };
  __device__ __forceinline__ Col col(int k) const {
    const int tap = k / Cin;
    return Col{k, k - tap * Cin, tap / 3 - 1, tap % 3 - 1};
  }
  __device__ __forceinline__ void advance(Col& c, int step) const {
    c.k += step;
    c.ci += step;
    while (c.ci >= Cin) {  // next tap
      c.ci -= Cin;
      if (++c.dj == 2) {
        c.dj = -1;
        ++c.di;
      }
    }
  }
  template <typename T>
  __device__ __forceinline__ float load(const Row& x, const Col& k) const {
    if (!x.ok || k.di > 1) return 0.f;  // past the last tap: K's ragged end
    const int rr = x.r + k.di, cc = x.c + k.dj;
    if (rr < 0 || rr >= H || cc < 0 || cc >= W) return 0.f;
    const bool own = rr >= x.lo && rr < x.lo + Hp;
    const T* src = static_cast<const T*>(own ? yf : ys);
    const long long i = (x.img + (long long)rr * W + cc) * Cin + k.ci;
    return DPP_IN(i, 1, n_y) ? to_f32(src[i]) : 0.f;
  }
};

// 64 x 64 output tile per block, 16-wide K slices in shared memory, 4 x 4 outputs per
// thread; each thread fetches the same 4 rows of A (and of W) in every slice, so their
// coordinates are prepared once, and the next slice's values are loaded into registers
// while the current one is multiplied.
template <typename T, typename ALoad>
__global__ void __launch_bounds__(256) simt_gemm_kernel(ALoad A, const T* __restrict__ Wt,
                                                        SimtOut out, long long M, int N, int K) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long long m0 = (long long)blockIdx.y * 64;
  const int n0 = blockIdx.x * 64;
  const int kk = threadIdx.x & 15;  // this thread's column within a slice
  typename ALoad::Row rows[4];
  bool nok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int mm = (threadIdx.x >> 4) + 16 * i;
    rows[i] = A.row(m0 + mm, M);
    nok[i] = n0 + mm < N;
  }
  typename ALoad::Col ac = A.col(kk);
  float ra[4], rb[4];
  auto fetch = [&](int k) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ra[i] = A.template load<T>(rows[i], ac);
      const int n = n0 + (threadIdx.x >> 4) + 16 * i;
      rb[i] = nok[i] && k < K && DPP_IN((long long)n * K + k, 1, (long long)N * K)
                  ? to_f32(Wt[(long long)n * K + k])
                  : 0.f;
    }
  };
  fetch(kk);
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      As[kk][(threadIdx.x >> 4) + 16 * i] = ra[i];
      Bs[kk][(threadIdx.x >> 4) + 16 * i] = rb[i];
    }
    __syncthreads();
    if (k0 + 16 < K) {  // the next slice's values, in flight during this slice's products
      A.advance(ac, 16);
      fetch(k0 + 16 + kk);
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      float a[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[q][ty * 4 + i]; bv[i] = Bs[q][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      const int which = n / out.ncols;
      const int col = n - which * out.ncols;
      if (DPP_IN(m * out.ncols + col, 1, M * out.ncols))
        static_cast<T*>(out.ptr[which])[m * out.ncols + col] = from_f32<T>(acc[i][j]);
    }
  }
}

// One warp per query row (8 rows per block), each lane taking keys kk = lane and
// lane + 32 of every 64-key tile with its own online-softmax state (m, l, acc[64]); the
// lanes' states are merged once at the end (warp maximum of m, then warp sums of the
// rescaled l and acc).  Padded shared rows keep the lanes' reads of 32 different keys on
// 32 different banks.
template <typename T>
__global__ void __launch_bounds__(256) simt_attention_kernel(const T* __restrict__ q,
                                                             const T* __restrict__ kf,
                                                             const T* __restrict__ vf,
                                                             const T* __restrict__ ks,
                                                             const T* __restrict__ vs,
                                                             T* __restrict__ o, int L, int heads,
                                                             int P) {
  constexpr int D = 64, KT = 64, ROWS = 8;
  __shared__ float Ks[KT][D + 1];
  __shared__ float Vs[KT][D + 1];
  const int Lp = L / P;
  const int blocks_per_patch = (Lp + ROWS - 1) / ROWS;
  const int p = blockIdx.x / blocks_per_patch;
  const int qb = blockIdx.x - p * blocks_per_patch;
  const int h = blockIdx.y, b = blockIdx.z;
  const int C = heads * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_in_patch = qb * ROWS + warp;
  const bool valid = row_in_patch < Lp;
  const long long rowbase = (long long)b * L;
  const long long t = rowbase + p * Lp + (valid ? row_in_patch : 0);
  const long long nel = (long long)gridDim.z * L * C;  // elements of Q, K, V and O
  const bool q_in = DPP_IN(t * C + h * D, D, nel);
  float qr[D], acc[D];
#pragma unroll
  for (int e = 0; e < D; ++e) {
    qr[e] = q_in ? to_f32(q[t * C + h * D + e]) * 0.125f : 0.f;  // 1/sqrt(64), exact
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  // tile loads: thread -> key row tid / 4 of the tile, 16 of its 64 dimensions, all 32
  // loads in flight before the stores; own patch's rows fresh, the others stale
  const int lk = threadIdx.x >> 2, le = (threadIdx.x & 3) * 16;
  const int own_lo = p * Lp, own_hi = own_lo + Lp;
  float kv[16], vv[16];
  auto fetch = [&](int s) {
    if (s < L && DPP_IN((rowbase + s) * C + h * D + le, 16, nel)) {
      const bool own = s >= own_lo && s < own_hi;
      const T* kp = (own ? kf : ks) + (rowbase + s) * C + h * D + le;
      const T* vp = (own ? vf : vs) + (rowbase + s) * C + h * D + le;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        kv[e] = to_f32(kp[e]);
        vv[e] = to_f32(vp[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) kv[e] = vv[e] = 0.f;
    }
  };
  fetch(lk);
  for (int s0 = 0; s0 < L; s0 += KT) {
    __syncthreads();  // the previous tile's products are done
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      Ks[lk][le + e] = kv[e];
      Vs[lk][le + e] = vv[e];
    }
    __syncthreads();
    if (s0 + KT < L) fetch(s0 + KT + lk);  // the next tile, in flight during this one
    float sc[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int kk = lane + 32 * j;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) dot = fmaf(qr[e], Ks[kk][e], dot);
      sc[j] = s0 + kk < L ? dot : -INFINITY;
    }
    const float mt = fmaxf(m, fmaxf(sc[0], sc[1]));
    if (mt == -INFINITY) continue;  // no valid key for this lane yet
    const float corr = expf(m - mt);  // m = -inf before the lane's first key gives 0
    const float p0 = expf(sc[0] - mt), p1 = expf(sc[1] - mt);
    l = fmaf(l, corr, p0 + p1);
#pragma unroll
    for (int e = 0; e < D; ++e)
      acc[e] = fmaf(p1, Vs[lane + 32][e], fmaf(p0, Vs[lane][e], acc[e] * corr));
    m = mt;
  }
  // merge the 32 lanes' states
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float f = m == -INFINITY ? 0.f : expf(m - M);
  l *= f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  float mine[2] = {0.f, 0.f};  // outputs e = lane and lane + 32
#pragma unroll
  for (int e = 0; e < D; ++e) {
    float a = acc[e] * f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (e == lane) mine[0] = a;
    if (e == lane + 32) mine[1] = a;
  }
  if (valid && DPP_IN(t * C + h * D, D, nel)) {
    const float inv = 1.f / l;
    o[t * C + h * D + lane] = from_f32<T>(mine[0] * inv);
    o[t * C + h * D + lane + 32] = from_f32<T>(mine[1] * inv);
  }
}

DPP_BOUNDS_READER(bounds_simt)

int launch_simt_linear(const void* a, const void* w, const SimtOut& out, long long M, int N, int K,
                       int dtype, cudaStream_t stream) {
  dim3 grid((N + 63) / 64, (unsigned)((M + 63) / 64));
  ALinear A{a, K};
#ifdef DPP_DEBUG_BOUNDS
  A.n_a = M * K;
#endif
  if (dtype == DPP_BF16)
    simt_gemm_kernel<__nv_bfloat16, ALinear><<<grid, 256, 0, stream>>>(
        A, static_cast<const __nv_bfloat16*>(w), out, M, N, K);
  else
    simt_gemm_kernel<float, ALinear><<<grid, 256, 0, stream>>>(A, static_cast<const float*>(w),
                                                               out, M, N, K);
  return cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

int launch_simt_conv(const void* yf, const void* ys, const void* w, void* out, int B, int H, int W,
                     int Cin, int Cout, int P, int dtype, cudaStream_t stream) {
  const long long M = (long long)B * H * W;
  const int K = 9 * Cin;
  dim3 grid((Cout + 63) / 64, (unsigned)((M + 63) / 64));
  AConv A{yf, ys, H, W, Cin, H / P};
#ifdef DPP_DEBUG_BOUNDS
  A.n_y = M * Cin;
#endif
  SimtOut o{};
  o.ptr[0] = out;
  o.ncols = Cout;
  if (dtype == DPP_BF16)
    simt_gemm_kernel<__nv_bfloat16, AConv><<<grid, 256, 0, stream>>>(
        A, static_cast<const __nv_bfloat16*>(w), o, M, Cout, K);
  else
    simt_gemm_kernel<float, AConv><<<grid, 256, 0, stream>>>(A, static_cast<const float*>(w), o,
                                                             M, Cout, K);
  return cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

int launch_simt_attention(const void* q, const void* kf, const void* vf, const void* ks,
                          const void* vs, void* o, int B, int L, int heads, int P, int dtype,
                          cudaStream_t stream) {
  const int Lp = L / P;
  dim3 grid(P * ((Lp + 7) / 8), heads, B);  // 8 query rows (one warp each) per block
  if (dtype == DPP_BF16) {
    using T = __nv_bfloat16;
    simt_attention_kernel<T><<<grid, 256, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(kf), static_cast<const T*>(vf),
        static_cast<const T*>(ks), static_cast<const T*>(vs), static_cast<T*>(o), L, heads, P);
  } else {
    simt_attention_kernel<float><<<grid, 256, 0, stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(kf),
        static_cast<const float*>(vf), static_cast<const float*>(ks),
        static_cast<const float*>(vs), static_cast<float*>(o), L, heads, P);
  }
  return cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

}  // namespace dpp
