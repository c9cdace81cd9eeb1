// Stale-KV flash attention on tcgen05 tensor cores (bf16 inputs, head_dim 64).
//
// ("OTIL for SDXL on 4x L40S", item 3 and Periodic layer-context refresh: the
// cross-slice attention K/V are stale; Self-tests: a rank's own slice is fresh,
// other positions stale, never a blend.)  Query token t of patch p attends over
// all L keys; key row s comes from the fresh K/V if s lies in patch p, else
// from the stale K/V.
//
// Work unit = two 128-row query tiles of one (batch, head, patch) against all key
// tiles.  The kernel is persistent (one CTA per SM): CTA c first takes whole units
// c, c+G, c+2G, ... (G CTAs; consecutive CTAs work on neighbouring units, which
// share their K/V in L2), and when the units do not divide evenly the remaining
// U mod G units are shared by all CTAs key tile by key tile ("split" schedule):
// each CTA takes an equal contiguous run of their (unit, key tile) steps, a unit
// cut between CTAs leaves one partial result per piece (O/l in fp16, the running
// maximum m and sum l in fp32); for each 32-row warp of a query tile, the warp that
// finishes the unit's last piece (an atomic count per unit, query tile and warp) merges
// its rows of all of them in CTA order, so the result does not depend on which piece
// finished last.
//
// A CTA's steps run through one pipeline: the next unit's Q is loaded into the second
// Q buffer while the current unit finishes, and its first S = Q K^T is issued right
// after the last P V.
// Per CTA, 12 warps:
//   warps 0-3 / 4-7  softmax of query tile 0 / 1 (thread = query row = TMEM lane):
//                    read S_t from TMEM, write fp16 P_t back to TMEM.
//   warp 8           TMA producer: Q tiles per unit (two buffers), a 5-stage ring of K and V
//                    tiles; each 128-key tile is fetched in sub-boxes of g rows
//                    (g = largest power of two <= 128 dividing L/P), each sub-box
//                    from the fresh or the stale tensor map -- the splice.  A stage is
//                    refilled once the tile-1 softmax warps have seen P_1 V of its step
//                    complete (every MMA that reads the stage is older than that one).
//   warp 9           MMA issuer (one thread) and TMEM owner.  Per key tile j and
//                    query tile t, once softmax t has written P_t(j):
//                    S_t = Q_t K(j+1)^T (M=128, N=128, K=16 steps over d=64), then
//                    O_t += P_t(j) V(j) (M=128, N=64, K=16 steps over keys, P from
//                    TMEM), each with its own commit.  The scores come first because the
//                    softmax waits for them, while P V only has to finish before the next
//                    P store; the two query tiles alternate, so the tensor pipe works on
//                    one tile while the other's softmax runs (one batch for both tiles
//                    after both P were written measured slower: the two softmaxes then
//                    run in step and contend for the exponential unit).  All MMAs of the
//                    CTA come from this one thread: issuing tcgen05.mma from two warps of
//                    one CTA at once faulted the GPU (an illegal memory access) in two
//                    independent implementations.
//   warps 10-11      widen each landed V tile from bf16 to fp16 in place (half a tile
//                    each), times the (batch, head) power of two, and report V(v) ready
//                    only once K(v+1) has landed too; the MMA thread waits for this
//                    before the step's MMAs.  The single MMA thread is the pipeline's
//                    bottleneck (each P is ready 700-1000 cycles before it is free), and each
//                    barrier test or commit it executes delays the next MMA batch; so
//                    the K wait and the stage release are done by warps with slack.
// P is rounded to fp16, not bf16: its 11-bit significand keeps the rounding of the
// probabilities well inside the 2e-3 output tolerance (bf16's 8 bits would not), and
// V is widened to fp16 so that P V runs as kind::f16 with both operands fp16.  fp16
// covers [2^-14, 65504] at full precision; V is brought into that range by a power of
// two 2^e per (batch, head), from max |V| over the fresh and stale V (taken by the
// kernels that write or read them before this one inside the layer step, by a small pass
// before the kernel for the standalone calls; e = 0 when max|V| lies in [2^-6, 2^15), the
// usual case), applied in the widening and removed again from O in the epilogue.
// Online softmax in the log2 domain with a lazily moved reference maximum: the row
// maximum of a unit's first key tile is the reference, later tiles are exponentiated
// against it without a maximum pass, and the reference moves (O and l rescaled, P
// recomputed from the scores still in TMEM) only for a row whose tile sum of P reaches
// 2^15, before any P could exceed fp16's range.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ptx.cuh"
#include "tc.cuh"

namespace dpp {

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn();  // tc_gemm.cu

namespace {

constexpr int D = 64;                   // head dim
constexpr int QT = 128;                 // query rows per tile
constexpr int KT = 128;                 // keys per tile
constexpr int KV_STAGES = 5;
constexpr int TILE_BYTES = KT * D * 2;  // 16 KB (K or V tile, Q tile)
constexpr int ATTN_THREADS = 384;
constexpr int NUM_CONVERTERS = 2;       // warps 10 and 11, half a V tile each
// smem: two Q buffers (Q0 Q1 each) | (K V) x stages | barriers.  TMEM (512 columns):
// S0 S1 (128 each), O0 O1 (64 each), P0 P1 (64 each: 128 fp16 probabilities per row,
// two per column).
constexpr int OFF_Q = 0;
constexpr int OFF_KV = 4 * TILE_BYTES;
constexpr int OFF_BAR = OFF_KV + KV_STAGES * 2 * TILE_BYTES;
constexpr int ATTN_SMEM = OFF_BAR + 512 + 1024;
// The first step of every CTA's tail run, tail_bound(c) for c = 0..G (split schedule), in
// static shared memory (a fixed address: no register holds a pointer to it).
constexpr int MAX_G = 159;
static_assert(ATTN_SMEM + (MAX_G + 1) * 4 <= 227 * 1024, "shared memory per CTA");
static_assert(ATTN_SMEM <= 227 * 1024, "shared memory per CTA");
constexpr float kScaleLog2 = 0.18033688011112042f;  // log2(e) / sqrt(64)
// A key tile whose probabilities (against the row's reference maximum) sum to 2^15 or
// more moves the reference: below that every P < 2^15 fits fp16 (max 65504).
constexpr float kRefSum = 32768.0f;
// Partial result of one piece of a cut unit: O/l as fp16 [2 tiles][128 rows][64],
// then the reference maximum m (log2 units) and the sum l, fp32 [2][128] each.
constexpr int REC_M = 2 * QT * D * 2;
constexpr int REC_L = REC_M + 2 * QT * 4;
constexpr int REC_BYTES = REC_L + 2 * QT * 4;

struct AttnArgs {
  int L, heads, P, Lp, g, n_pairs, nkt;
  int* cnt;         // split: [tail unit][query tile][warp] pieces finished (zero before the call)
  int U;            // units (batch, head, patch, pair of query tiles), pair fastest
  int G;            // CTAs
  int W;            // split: whole units per CTA (c, c+G, ...); 0 otherwise
  int split;        // 1: units W*G .. U-1 are shared key tile by key tile
  long long tailT;  // split: their (unit, key tile) steps
  int tq, tr;       // tailT = tq * G + tr (tail_bound(c) = c tq + c tr / G in 32 bits)
  __nv_bfloat16* o;
  uint8_t* part;    // split: G + (U - W*G) partial records
  const unsigned* vmax;  // [B*heads] fp32 bits of max |V| over the fresh and stale V
  int* status;
  long long wait_limit;
  int skip_load;    // test hook: the producer never loads the K/V tile of this step (-1)
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[KV_STAGES], v_full[KV_STAGES], v_conv[KV_STAGES], kv_empty[KV_STAGES];
  uint64_t s_full[2], p_full[2], pv_done[2], drain;
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier area");

// The steps of CTA c: nfull whole units (c, c+G, ...), then the steps [t0, t1) of
// the shared tail, step = (unit - W*G) * nkt + key tile.
struct Sched {
  int nfull, nsteps;
  long long t0;
};

__host__ __device__ __forceinline__ long long tail_bound(long long c, const AttnArgs& a) {
  return c * a.tailT / a.G;
}

// The CTA whose tail run contains step s (runs may be empty when tailT < G), from the
// CTA's table tb[c] = tail_bound(c) (no 64-bit divisions on the merge path): the largest
// c < G with tb[c] <= s.
__device__ __forceinline__ int tail_cta_tb(const int* tb, long long s, int G) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb[mid] <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Sched make_sched(const AttnArgs& a) {
  Sched s;
  const int c = blockIdx.x;
  long long t1 = 0;
  s.t0 = 0;
  if (a.split) {
    s.nfull = a.W;
    s.t0 = tail_bound(c, a);
    t1 = tail_bound(c + 1, a);
  } else {
    s.nfull = (a.U - c + a.G - 1) / a.G;
  }
  s.nsteps = s.nfull * a.nkt + (int)(t1 - s.t0);
  return s;
}

// A segment: the run of one unit's key tiles [j0, j0 + len) that this CTA processes
// from step v on.  Divisions happen once per segment, never inside a step.
struct Seg {
  int u, j0, len;
  bool tail;  // a segment of the shared tail (may be a piece of a cut unit)
};

__device__ __forceinline__ Seg seg_at(const Sched& s, int v, const AttnArgs& a) {
  Seg g;
  const int vf = s.nfull * a.nkt;
  if (v < vf) {  // v is a multiple of nkt here
    g.u = (int)blockIdx.x + (v / a.nkt) * a.G;
    g.j0 = 0;
    g.len = a.nkt;
    g.tail = false;
  } else {
    const long long tv = s.t0 + (v - vf);
    const int ut = (int)(tv / a.nkt);
    g.j0 = (int)(tv - (long long)ut * a.nkt);
    g.u = a.W * a.G + ut;
    g.len = min(a.nkt - g.j0, s.nsteps - v);
    g.tail = true;
  }
  return g;
}

struct UnitPos {
  int b, h, patch0, q0;  // q0: first query row of the unit within its patch
};

__host__ __device__ __forceinline__ UnitPos unit_pos(int u, const AttnArgs& a) {
  UnitPos x;
  const int pair = u % a.n_pairs;
  int r = u / a.n_pairs;
  const int p = r % a.P;
  r /= a.P;
  x.h = r % a.heads;
  x.b = r / a.heads;
  x.patch0 = p * a.Lp;
  x.q0 = 2 * pair * QT;
  return x;
}

// The power of two 2^e that brings V of (batch b, head h) into fp16's full-precision
// range: e = 0 when max|V| lies in [2^-6, 2^15); otherwise 14 - floor(log2 max|V|), so
// that the scaled maximum lies in [2^14, 2^15), clamped to [-125, 125] (only |V| below
// 2^-111 then keeps some fp16 subnormals).  An all-zero V gets 0.
// Extents for the index checks: batches, elements of O (and of each of Q/K/V), partial
// records, piece counters.
__device__ __forceinline__ long long n_batch(const AttnArgs& a) {
  return a.U / ((long long)a.heads * a.P * a.n_pairs);
}
__device__ __forceinline__ long long n_elems(const AttnArgs& a) {
  return n_batch(a) * a.L * a.heads * D;
}
__device__ __forceinline__ long long n_records(const AttnArgs& a) {
  return a.split ? (long long)a.G + a.U - (long long)a.W * a.G : 0;
}

__device__ __forceinline__ unsigned vmax_bits(const AttnArgs& a, int b, int h) {
  return DPP_IN(b * a.heads + h, 1, n_batch(a) * a.heads) ? __ldg(a.vmax + b * a.heads + h) : 0u;
}
__device__ __forceinline__ int v_exponent(unsigned bits) {
  const float amax = __uint_as_float(bits);
  if (bits == 0 || (amax >= 0.015625f && amax < 32768.0f)) return 0;
  const int E = (int)(bits >> 23) - 127;  // floor(log2 amax); a subnormal amax gives -127
  return max(-125, min(125, 14 - E));
}

__device__ __forceinline__ float pow2(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const AttnArgs& a,
                                              Bars* bars) {
  if (ptx::mbar_wait(bar, parity, a.wait_limit, &bars->abort_flag)) return true;
  set_status(a.status, DPP_ERR_TIMEOUT);
  bars->abort_flag = 1;
  return false;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16 fp32 values (raw bits, as read from TMEM) scaled by s, as bf16 (two 16-byte stores).
__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const uint32_t (&o)[16],
                                              float s) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    d4[i] = make_uint4(
        pack_bf16x2(__uint_as_float(o[8 * i]) * s, __uint_as_float(o[8 * i + 1]) * s),
        pack_bf16x2(__uint_as_float(o[8 * i + 2]) * s, __uint_as_float(o[8 * i + 3]) * s),
        pack_bf16x2(__uint_as_float(o[8 * i + 4]) * s, __uint_as_float(o[8 * i + 5]) * s),
        pack_bf16x2(__uint_as_float(o[8 * i + 6]) * s, __uint_as_float(o[8 * i + 7]) * s));
}

// The same as fp16 (the partial results of cut units).
__device__ __forceinline__ void store_f16x16(uint4* d4, const uint32_t (&o)[16], float s) {
#pragma unroll
  for (int i = 0; i < 2; ++i)
    d4[i] = make_uint4(
        pack_f16x2(__uint_as_float(o[8 * i]) * s, __uint_as_float(o[8 * i + 1]) * s),
        pack_f16x2(__uint_as_float(o[8 * i + 2]) * s, __uint_as_float(o[8 * i + 3]) * s),
        pack_f16x2(__uint_as_float(o[8 * i + 4]) * s, __uint_as_float(o[8 * i + 5]) * s),
        pack_f16x2(__uint_as_float(o[8 * i + 6]) * s, __uint_as_float(o[8 * i + 7]) * s));
}

// Merges the pieces of tail unit ut for row r of query tile t: records of CTAs
// ca..cb (those with a non-empty run), in that order.  With pieces i = (m_i, l_i,
// O_i/l_i), in one pass with a running maximum M: each piece rescales the sums so far by
// 2^(M_old - M) and adds w_i = l_i 2^(m_i - M); o = sum_i w_i (O_i/l_i) / sum_i w_i,
// times 2^-e (the records hold O in V's scaled units).  The records were written by other
// SMs and are complete when the merge starts; this SM has not read them before, so they
// are prefetched into L1 (all pieces' round trips to L2 overlapped) and read from there.
__device__ __forceinline__ void merge_rows(const AttnArgs& a, const int* tb, int ut, int t,
                                           int r, int ca, int cb, const UnitPos& up, int e) {
  const int row_in_patch = up.q0 + t * QT + r;
  if (row_in_patch >= a.Lp) return;
  const long long s_a = (long long)ut * a.nkt;
  const size_t row = (size_t)(t * QT + r);
  // a CTA's first tail segment, or the last one of the CTA that started before the unit
  auto rec_index = [&](int c) -> int { return (c == ca && tb[c] != s_a) ? a.G + ut : c; };
  auto record = [&](int c) -> const uint8_t* {
    return a.part + (size_t)rec_index(c) * REC_BYTES;
  };
  // every piece's lines of this row into L1 first, so that their round trips to L2 overlap
  // (the records are complete: the pieces' counter has been read)
  for (int c = ca; c <= cb; ++c) {
    if (tb[c] == tb[c + 1] || !DPP_IN(rec_index(c), 1, n_records(a))) continue;
    const uint8_t* base = record(c);
    ptx::prefetch_l1(base + row * D * 2);
    ptx::prefetch_l1(reinterpret_cast<const float*>(base + REC_M) + row);
    ptx::prefetch_l1(reinterpret_cast<const float*>(base + REC_L) + row);
  }
  float M = -INFINITY, wsum = 0.f;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;
  for (int c = ca; c <= cb; ++c) {
    if (tb[c] == tb[c + 1]) continue;  // empty run
    if (!DPP_IN(rec_index(c), 1, n_records(a))) continue;
    const uint8_t* base = record(c);
    const float m = __ldca(reinterpret_cast<const float*>(base + REC_M) + row);
    const float l = __ldca(reinterpret_cast<const float*>(base + REC_L) + row);
    const uint4* src = reinterpret_cast<const uint4*>(base + row * D * 2);
    uint4 u[D / 8];
#pragma unroll
    for (int q = 0; q < D / 8; ++q) u[q] = __ldca(src + q);
    const float mn = fmaxf(M, m);
    const float sc = exp2f(M - mn), w = l * exp2f(m - mn);
    M = mn;
    wsum = fmaf(wsum, sc, w);
#pragma unroll
    for (int q = 0; q < D / 8; ++q) {
      const uint32_t hw[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[k]));
        acc[8 * q + 2 * k] = fmaf(w, f.x, acc[8 * q + 2 * k] * sc);
        acc[8 * q + 2 * k + 1] = fmaf(w, f.y, acc[8 * q + 2 * k + 1] * sc);
      }
    }
  }
  const long long o_off =
      ((long long)up.b * a.L + up.patch0 + row_in_patch) * (long long)(a.heads * D) + up.h * D;
  if (!DPP_IN(o_off, D, n_elems(a))) return;
  __nv_bfloat16* dst = a.o + o_off;
  const float inv = pow2(-e) / wsum;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < D / 8; ++q)
    d4[q] = make_uint4(pack_bf16x2(acc[8 * q] * inv, acc[8 * q + 1] * inv),
                       pack_bf16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                       pack_bf16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv),
                       pack_bf16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
}

// Row maximum of a thread's 128 raw scores (four independent max3 chains).
__device__ __forceinline__ float row_max(const uint32_t (&sv)[128]) {
  float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 128; i += 8) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      mq[u] = ptx::max3(mq[u], __uint_as_float(sv[i + 2 * u]), __uint_as_float(sv[i + 2 * u + 1]));
  }
  return ptx::max3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
}

// p = 2^(s log2(e)/sqrt(64) - m_ref) for the 128 scores, as fp16 pairs (column c holds keys
// 2c in the low half and 2c+1 in the high half); pairs of keys in packed fp32x2 (one FMA
// and one add per two keys).  Returns the fp32 sum of the p.
__device__ __forceinline__ float exp_tile(const uint32_t (&sv)[128], float m_ref,
                                          uint32_t (&pk)[64]) {
  const uint64_t c2 = ptx::pack_f32x2(kScaleLog2, kScaleLog2);
  const uint64_t nm2 = ptx::pack_f32x2(-m_ref, -m_ref);
  uint64_t lq[2] = {ptx::pack_f32x2(0.f, 0.f), ptx::pack_f32x2(0.f, 0.f)};
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const uint64_t s2 = ptx::pack_f32x2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]));
    float a0, a1;
    ptx::unpack_f32x2(ptx::fma_f32x2(s2, c2, nm2), a0, a1);
    const float p0 = ex2(a0), p1 = ex2(a1);
    lq[i & 1] = ptx::add_f32x2(lq[i & 1], ptx::pack_f32x2(p0, p1));
    pk[i] = pack_f16x2(p0, p1);
  }
  float x0, x1, y0, y1;
  ptx::unpack_f32x2(lq[0], x0, x1);
  ptx::unpack_f32x2(lq[1], y0, y1);
  return (x0 + x1) + (y0 + y1);
}

// The row maximum re-read from the scores in TMEM, 32 columns at a time (keys >= nvalid
// excluded).  Warp-collective.
__device__ __forceinline__ float tile_max(uint32_t t_row, int nvalid) {
  float m = -INFINITY;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t x[32];
    ptx::tmem_ld32(t_row + c * 32, x);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c * 32 + i < nvalid) m = fmaxf(m, __uint_as_float(x[i]));
  }
  return m;
}

// exp_tile from the scores in TMEM, written straight to P in TMEM, 32 keys at a time;
// returns the sum.  Warp-collective.
__device__ __forceinline__ float exp_store(uint32_t s_row, uint32_t p_row, int nvalid,
                                           float m_ref) {
  float sum = 0.f;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t x[32], pk[16];
    ptx::tmem_ld32(s_row + c * 32, x);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float s0 = c * 32 + 2 * i < nvalid ? __uint_as_float(x[2 * i]) : -INFINITY;
      const float s1 = c * 32 + 2 * i + 1 < nvalid ? __uint_as_float(x[2 * i + 1]) : -INFINITY;
      const float p0 = ex2(fmaf(s0, kScaleLog2, -m_ref)), p1 = ex2(fmaf(s1, kScaleLog2, -m_ref));
      sum += p0 + p1;
      pk[i] = pack_f16x2(p0, p1);
    }
    ptx::tmem_st16(p_row + c * 16, pk);
  }
  return sum;
}

// max |V| of each (batch, head) over the fresh V and, when P > 1, the stale V (every
// row of both is read by some patch); the result goes to vmax (zero before the launch)
// as fp32 bits through atomicMax, which orders non-negative floats like their bits.
// Grid (chunks, heads, B); a warp reads four 128-byte head rows per load.
__global__ void __launch_bounds__(256) vrange_kernel(const __nv_bfloat16* vf,
                                                     const __nv_bfloat16* vs, int L, int heads,
                                                     int rows_per_block, int use_stale,
                                                     unsigned* vmax) {
  __shared__ unsigned red[8];
  const int b = blockIdx.z, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long C = (long long)heads * D;
  const int r0 = blockIdx.x * rows_per_block;
  const int r1 = min(L, r0 + rows_per_block);
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  unsigned m = 0;
  for (int r = r0 + warp * 4 + (lane >> 3); r < r1; r += 32) {
    const long long off = ((long long)b * L + r) * C + h * D + (lane & 7) * 8;
    if (!DPP_IN(off, 8, (long long)gridDim.z * L * C)) continue;
    uint4 u = __ldg(reinterpret_cast<const uint4*>(vf + off));
    unsigned w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) m = max(m, max(w4[k] & 0x7FFFu, (w4[k] >> 16) & 0x7FFFu));
    if (use_stale) {
      u = __ldg(reinterpret_cast<const uint4*>(vs + off));
      const unsigned s4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) m = max(m, max(s4[k] & 0x7FFFu, (s4[k] >> 16) & 0x7FFFu));
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 1; i < 8; ++i) m = max(m, red[i]);
    if (m && DPP_IN(b * heads + h, 1, (long long)gridDim.z * heads))
      atomicMax(vmax + b * heads + h, m << 16);  // bf16 bits -> fp32 bits
  }
}

__global__ void __launch_bounds__(ATTN_THREADS, 1)
    tc_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKf,
                   const __grid_constant__ CUtensorMap tmKs, const __grid_constant__ CUtensorMap tmVf,
                   const __grid_constant__ CUtensorMap tmVs, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  __shared__ int tb[MAX_G + 1];  // tail_bound(c) < 2^31: the plan limits tiles x key tiles
  for (int c = threadIdx.x; c <= a.G && c <= MAX_G; c += blockDim.x) tb[c] = c * a.tq + c * a.tr / a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int qb = 0; qb < 2; ++qb) {
      ptx::mbar_init(&bars->q_full[qb], 1);
      ptx::mbar_init(&bars->q_empty[qb], 1);  // committed after a unit's last Q K^T
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      ptx::mbar_init(&bars->k_full[s], 1);
      ptx::mbar_init(&bars->v_full[s], 1);
      ptx::mbar_init(&bars->v_conv[s], NUM_CONVERTERS);
      ptx::mbar_init(&bars->kv_empty[s], 4);  // the tile-1 softmax warps, after P_1 V
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(&bars->s_full[t], 1);
      ptx::mbar_init(&bars->p_full[t], 4);  // one arrival per softmax warp
      ptx::mbar_init(&bars->pv_done[t], 1);  // committed after each P V
    }
    ptx::mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmKf);
    ptx::tma_prefetch_desc(&tmKs);
    ptx::tma_prefetch_desc(&tmVf);
    ptx::tma_prefetch_desc(&tmVs);
  }
  if (warp == 9) {
    ptx::tmem_alloc(&bars->tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const Sched sc = make_sched(a);
  // the set-up above overlaps the previous kernel; its outputs are read from here on
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp >= 8) {
    // Register split (launch: 384 threads x 168): this warpgroup drops to 80 per
    // thread, the two softmax warpgroups rise to 208: 128 x 80 + 256 x 208 <= 64512.
    ptx::regs_dec<80>();
    if (warp == 8) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        int issued = 0, q_issued = 0;
        const int nsub = KT / a.g;
        bool ok = true;
        for (int v = 0; v < sc.nsteps && ok;) {
          const Seg sg = seg_at(sc, v, a);
          const UnitPos up = unit_pos(sg.u, a);
          {  // Q of this unit into buffer n & 1, once its last user is done
            const int n = q_issued, qb = n & 1;
            if (!wait_or_abort(&bars->q_empty[qb], ((n >> 1) & 1) ^ 1, a, bars)) break;
            ptx::mbar_arrive_expect_tx(&bars->q_full[qb], 2 * TILE_BYTES);
            for (int t = 0; t < 2; ++t)
              ptx::tma_load_3d(smem + OFF_Q + (2 * qb + t) * TILE_BYTES, &tmQ, &bars->q_full[qb],
                               up.h * D, up.patch0 + up.q0 + t * QT, up.b);
            ++q_issued;
          }
          for (int j = sg.j0; j < sg.j0 + sg.len; ++j, ++v) {
            const int st = v % KV_STAGES;
            if (!wait_or_abort(&bars->kv_empty[st], ((v / KV_STAGES) & 1) ^ 1, a, bars)) {
              ok = false;
              break;
            }
            ++issued;
            if (v == a.skip_load) continue;  // test hook: this step's K and V never land
            uint8_t* kdst = smem + OFF_KV + st * 2 * TILE_BYTES;
            uint8_t* vdst = kdst + TILE_BYTES;
            ptx::mbar_arrive_expect_tx(&bars->k_full[st], TILE_BYTES);
            ptx::mbar_arrive_expect_tx(&bars->v_full[st], TILE_BYTES);
            for (int i = 0; i < nsub; ++i) {
              const int row = j * KT + i * a.g;
              const bool fresh = row >= up.patch0 && row < up.patch0 + a.Lp;
              ptx::tma_load_3d(kdst + i * a.g * 128, fresh ? &tmKf : &tmKs, &bars->k_full[st],
                               up.h * D, row, up.b);
            }
            for (int i = 0; i < nsub; ++i) {
              const int row = j * KT + i * a.g;
              const bool fresh = row >= up.patch0 && row < up.patch0 + a.Lp;
              ptx::tma_load_3d(vdst + i * a.g * 128, fresh ? &tmVf : &tmVs, &bars->v_full[st],
                               up.h * D, row, up.b);
            }
          }
        }
        if (*reinterpret_cast<volatile int*>(&bars->abort_flag)) {
          // wait for own copies in flight before exiting: a Q load is issued only after
          // the MMAs of the unit two before it have completed, so only the last two can
          // still be in flight
          for (int n = q_issued > 2 ? q_issued - 2 : 0; n < q_issued; ++n)
            ptx::mbar_wait(&bars->q_full[n & 1], (n >> 1) & 1, kDrainWaitLimit, nullptr);
          const int first = issued > KV_STAGES ? issued - KV_STAGES : 0;
          for (int j = first; j < issued; ++j) {
            if (j == a.skip_load) continue;
            ptx::mbar_wait(&bars->k_full[j % KV_STAGES], (j / KV_STAGES) & 1, kDrainWaitLimit,
                           nullptr);
            ptx::mbar_wait(&bars->v_full[j % KV_STAGES], (j / KV_STAGES) & 1, kDrainWaitLimit,
                           nullptr);
          }
        }
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && sc.nsteps > 0) {
        constexpr uint32_t idesc_qk = ptx::idesc_f16(QT, KT, 1, 0, 0);
        constexpr uint32_t idesc_pv = ptx::idesc_f16(QT, D, 0, 0, 1);
        // Descriptors are affine in the smem address (address field = bytes >> 4, no
        // carry out for offsets inside shared memory): precompute the bases once.
        const uint64_t q_desc = ptx::sw128_desc(ptx::smem_u32(smem + OFF_Q), 16, 1024);
        const uint64_t k_desc = ptx::sw128_desc(ptx::smem_u32(smem + OFF_KV), 16, 1024);
        const uint64_t v_desc =
            ptx::sw128_desc(ptx::smem_u32(smem + OFF_KV + TILE_BYTES), TILE_BYTES, 1024);
        constexpr uint64_t kStageStep = (2 * TILE_BYTES) >> 4;  // next K/V stage
        constexpr uint64_t kQTile = TILE_BYTES >> 4;            // next query tile
        bool any = false;
        bool ok = wait_or_abort(&bars->q_full[0], 0, a, bars) &&
                  wait_or_abort(&bars->k_full[0], 0, a, bars);
        if (ok) {
          ptx::tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              ptx::mma_ss(tmem + 128u * t, q_desc + t * kQTile + 2 * k, k_desc + 2 * k, idesc_qk,
                          k ? 1u : 0u);
            ptx::mma_commit(&bars->s_full[t]);
          }
          any = true;
        }
        int n = 0;  // segment of step v
        for (int v = 0; v < sc.nsteps && ok; ++n) {
          const Seg sg = seg_at(sc, v, a);
          const int vbeg = v, vend = v + sg.len;
          for (; v < vend; ++v) {
            const bool last = v == vend - 1;
            const bool more = v + 1 < sc.nsteps;
            const bool new_seg = last && more;  // step v+1 starts another unit
            const int qn = new_seg ? n + 1 : n;   // segment of step v+1
            const int st = v % KV_STAGES;
            const uint64_t vd = v_desc + (uint64_t)st * kStageStep;
            const uint64_t kd = k_desc + (uint64_t)((v + 1) % KV_STAGES) * kStageStep;
            const uint64_t qd = q_desc + (uint64_t)(qn & 1) * 2 * kQTile;
            const uint32_t acc0 = v > vbeg ? 1u : 0u;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              // P_t(v); once per step V(v) widened and K(v+1) landed (v_conv)
              if (!wait_or_abort(&bars->p_full[t], v & 1, a, bars) ||
                  (t == 0 && !wait_or_abort(&bars->v_conv[st], (v / KV_STAGES) & 1, a, bars)) ||
                  (t == 0 && new_seg &&
                   !wait_or_abort(&bars->q_full[qn & 1], (qn >> 1) & 1, a, bars))) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              const uint32_t tO = tmem + 256u + 64u * t, tP = tmem + 384u + 64u * t;
              // The next scores first: the softmax of tile t waits for them, while P V
              // is needed only before its next P store.  Two independent accumulator
              // chains in flight also keep the tensor pipe busier than one after the
              // other (measured: 720 vs 865 cycles for one tile's batch).
              if (more) {  // S_t = Q_t K(v+1)^T, Q of the unit of step v+1
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                  ptx::mma_ss(tmem + 128u * t, qd + t * kQTile + 2 * k, kd + 2 * k, idesc_qk,
                              k ? 1u : 0u);
                ptx::mma_commit(&bars->s_full[t]);
              }
#pragma unroll
              for (int k = 0; k < KT / 16; ++k)  // O_t += P_t(v) V(v)
                ptx::mma_ts(tO, tP + k * 8, vd + 128 * k, idesc_pv, k ? 1u : acc0);
              ptx::mma_commit(&bars->pv_done[t]);
            }
            if (!ok) break;
            // after a unit's last step every Q K^T of it has been issued: free its Q buffer
            if (last) ptx::mma_commit(&bars->q_empty[n & 1]);
          }
        }
        if (!ok && any) {  // let issued MMAs finish before TMEM is released
          ptx::mma_commit(&bars->drain);
          ptx::mbar_wait(&bars->drain, 0, kDrainWaitLimit, nullptr);
        }
      }
    } else if (warp >= 10) {
      // ------------------------------------------------ V widening (warps 10, 11)
      // Each landed V tile: this warp's half, 16 KB / 2 / 32 lanes = 16 vectors per lane,
      // in two passes of 8, bf16 -> fp16 times 2^e (exact: a power of two, and fp16 holds
      // every bf16 value of the scaled range).  The MMA thread issues step v's MMAs only
      // after both halves are done and K(v+1) has landed (v_conv).
      const int half = warp - 10;
      bool ok = true;
      for (int v = 0; v < sc.nsteps && ok;) {
        const Seg sg = seg_at(sc, v, a);
        const UnitPos up = unit_pos(sg.u, a);
        const float scale = pow2(v_exponent(vmax_bits(a, up.b, up.h)));
        for (const int vend = v + sg.len; v < vend; ++v) {
          const int st = v % KV_STAGES;
          if (!wait_or_abort(&bars->v_full[st], (v / KV_STAGES) & 1, a, bars)) {
            ok = false;
            break;
          }
          uint4* vt = reinterpret_cast<uint4*>(smem + OFF_KV + st * 2 * TILE_BYTES + TILE_BYTES) +
                      half * (TILE_BYTES / 16 / NUM_CONVERTERS);
#pragma unroll 1
          for (int pass = 0; pass < 2; ++pass) {
            uint4 u[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) u[i] = vt[lane + 32 * (8 * pass + i)];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
              for (int k = 0; k < 4; ++k)
                w[k] = pack_f16x2(__uint_as_float(w[k] << 16) * scale,
                                  __uint_as_float(w[k] & 0xFFFF0000u) * scale);
              vt[lane + 32 * (8 * pass + i)] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          // S(v+1) = Q K(v+1)^T is issued in the same batch as P(v) V(v)
          if (v + 1 < sc.nsteps &&
              !wait_or_abort(&bars->k_full[(v + 1) % KV_STAGES], ((v + 1) / KV_STAGES) & 1, a,
                             bars)) {
            ok = false;
            break;
          }
          if (lane == 0) ptx::mbar_arrive(&bars->v_conv[st]);
        }
      }
    }
  } else {
    ptx::regs_inc<208>();
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int t = warp >> 2;             // query tile of this warpgroup
    const int quarter = warp & 3;        // TMEM lanes [32*quarter, +32)
    const int r = quarter * 32 + lane;   // row within the query tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + 128u * (uint32_t)t;        // S_t: 128 columns
    const uint32_t tO = tmem + 256u + 64u * (uint32_t)t;  // O_t: 64 columns
    const uint32_t tP = tmem + 384u + 64u * (uint32_t)t;  // P_t: 64 columns
    bool ok = true;
    bool tail_seen = false;  // a tail segment of this CTA has ended
    for (int v = 0, n = 0; v < sc.nsteps && ok; ++n) {
      const Seg sg = seg_at(sc, v, a);
      const int vbeg = v, vend = v + sg.len;
      const UnitPos up = unit_pos(sg.u, a);
      const int e_cur = v_exponent(vmax_bits(a, up.b, up.h));
      float m_ref = -INFINITY, l = 0.f;
      for (int j = sg.j0; v < vend; ++v, ++j) {
        // S_t(v) ready (the MMA thread issues it before P_t(v-1) V(v-1), which may still
        // be running: P_t and O_t are touched only after pv_done below)
        if (!wait_or_abort(&bars->s_full[t], v & 1, a, bars)) { ok = false; break; }
        ptx::tc_fence_after();
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          ptx::tmem_ld32(tS + lane_off + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
        ptx::tmem_ld_wait();
        const int nvalid = a.L - j * KT;
        if (nvalid < KT) {  // only the last key tile can be partial: mask keys >= L
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= nvalid) sv[i] = __float_as_uint(-INFINITY);
        }
        // The reference maximum m_ref (log2 units) is the row maximum of the segment's
        // first key tile; later tiles are exponentiated against it directly, and only a
        // row whose tile sum reaches 2^15 (so that some P might come near fp16's 65504, or
        // overflow) takes its true maximum as the new reference: then O and l are
        // rescaled and that warp recomputes its P from the scores still in TMEM.
        if (v == vbeg) {
          m_ref = row_max(sv) * kScaleLog2;
          l = 0.f;
        }
        uint32_t pk[64];
        float s_step = exp_tile(sv, m_ref, pk);
        const bool big = v > vbeg && !(s_step < kRefSum);
        const bool redo = __any_sync(0xffffffffu, big);
        float alpha = 1.f;
        if (redo) {  // rare
          const float m_new = fmaxf(tile_max(tS + lane_off, nvalid) * kScaleLog2, m_ref);
          if (big) {
            alpha = ex2(m_ref - m_new);
            m_ref = m_new;
            l *= alpha;
          }
        }
        // P_t and O_t are free once P_t(v-1) V(v-1) has completed
        if (v > 0 && !wait_or_abort(&bars->pv_done[t], (v - 1) & 1, a, bars)) {
          ok = false;
          break;
        }
        if (t == 1 && v > vbeg) {  // K(v-1), V(v-1) no longer read: free their stage
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bars->kv_empty[(v - 1) % KV_STAGES]);
        }
        ptx::tc_fence_after();
        if (redo) {  // rescale the running O_t, then P from the scores in TMEM
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[16];
            ptx::tmem_ld16(tO + lane_off + c * 16, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st16(tO + lane_off + c * 16, o);
          }
          s_step = exp_store(tS + lane_off, tP + lane_off, nvalid, m_ref);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            ptx::tmem_st16(tP + lane_off + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * c]));
        }
        l += s_step;
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->p_full[t]);
      }
      if (!ok) break;
      // ---- end of the segment: O_t complete once its last P V has finished
      if (!wait_or_abort(&bars->pv_done[t], (vend - 1) & 1, a, bars)) { ok = false; break; }
      if (t == 1) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->kv_empty[(vend - 1) % KV_STAGES]);
      }
      ptx::tc_fence_after();
      if (sg.j0 == 0 && sg.len == a.nkt) {  // whole unit: normalised bf16 output
        const float inv = pow2(-e_cur) / l;
        const int row_in_patch = up.q0 + t * QT + r;
        const long long o_off = ((long long)up.b * a.L + up.patch0 + row_in_patch) *
                                    (long long)(a.heads * D) + up.h * D;
        const bool valid = row_in_patch < a.Lp && DPP_IN(o_off, D, n_elems(a));
        __nv_bfloat16* dst = a.o + o_off;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[16];
          ptx::tmem_ld16(tO + lane_off + c * 16, o);
          ptx::tmem_ld_wait();
          if (valid) store_bf16x16(dst + c * 16, o, inv);
        }
      } else {  // one piece of a cut unit: O/l in fp16 (V's scaled units), m and l in fp32
        const float inv = 1.f / l;
        const int ut = sg.u - a.W * a.G;
        const int rec = tail_seen ? a.G + ut : (int)blockIdx.x;
        const bool rec_in = DPP_IN(rec, 1, n_records(a));  // the same for the whole warp
        uint8_t* base = a.part + (size_t)rec * REC_BYTES;
        uint4* dst = reinterpret_cast<uint4*>(base + ((size_t)(t * QT + r) * D) * 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[16];
          ptx::tmem_ld16(tO + lane_off + c * 16, o);
          ptx::tmem_ld_wait();
          if (rec_in) store_f16x16(dst + 2 * c, o, inv);
        }
        if (rec_in) {
          reinterpret_cast<float*>(base + REC_M)[t * QT + r] = m_ref;
          reinterpret_cast<float*>(base + REC_L)[t * QT + r] = l;
        }
        // The last piece of the unit to finish merges them all, warp by warp: each warp's
        // 32 rows have their own counter, so that no warp waits for another.
        __threadfence();
        __syncwarp();
        const long long s_a = (long long)ut * a.nkt;
        const int ca = tail_cta_tb(tb, s_a, a.G), cb = tail_cta_tb(tb, s_a + a.nkt - 1, a.G);
        int last = 0;
        if (lane == 0) {
          int np = 0;
          for (int c = ca; c <= cb; ++c) np += tb[c] != tb[c + 1];
          int* cnt = a.cnt + (2 * ut + t) * 4 + quarter;
          last = DPP_IN((2 * ut + t) * 4 + quarter, 1, (n_records(a) - a.G) * 8) &&
                 atomicAdd(cnt, 1) == np - 1;
          if (last) atomicExch(cnt, 0);  // all arrived: ready for the next call
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __syncwarp();
          __threadfence();
          merge_rows(a, tb, ut, t, r, ca, cb, up, e_cur);
        }
      }
      if (sg.tail) tail_seen = true;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

bool make_map3(CUtensorMap* m, const void* base, int L, int B, int C, int box_rows) {
  auto fn = tc_encode_fn();
  if (!fn) return false;
  const uint64_t dims[3] = {(uint64_t)C, (uint64_t)L, (uint64_t)B};
  const uint64_t strides[2] = {(uint64_t)C * 2, (uint64_t)L * C * 2};
  const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
  const uint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int set_attn_smem() {
  static std::once_flag once;
  static int rc = DPP_OK;
  std::call_once(once, [] {
    if (cudaFuncSetAttribute(tc_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ATTN_SMEM) != cudaSuccess)
      rc = DPP_ERR_CUDA;
  });
  return rc;
}

// Schedule of one launch; false if the shape is not supported.
bool plan(int B, int L, int heads, int P, bool split, AttnArgs* a) {
  if (B <= 0 || L <= 0 || heads <= 0 || P <= 0 || L % P) return false;
  const int Lp = L / P;
  if (Lp % 8) return false;
  int g = 128;
  while (Lp % g) g >>= 1;
  *a = AttnArgs{};
  a->L = L; a->heads = heads; a->P = P; a->Lp = Lp; a->g = g;
  a->n_pairs = ((Lp + QT - 1) / QT + 1) / 2;
  a->nkt = (L + KT - 1) / KT;
  const long long U = (long long)B * heads * P * a->n_pairs;
  if (U * a->nkt > (1ll << 31) - 1) return false;
  a->U = (int)U;
  const int sms = dpp_host::sm_count();
  if (split) {
    const long long T = U * a->nkt;
    const int gmax = sms < MAX_G ? sms : MAX_G;  // the CTAs' table of tail runs
    a->G = (int)(T < gmax ? T : gmax);
    a->W = a->U / a->G;
    // The last full round joins the leftover units in the shared tail: each CTA's
    // tail run is then longer than a unit, so a cut unit has at most two pieces
    // (one short merge per unit instead of a long chain).
    if (a->U % a->G && a->W > 0) --a->W;
    a->tailT = (long long)(a->U - a->W * a->G) * a->nkt;
    a->split = a->U % a->G != 0;
    if (!a->split) {
      a->W = 0;
      a->tailT = 0;
    }
  } else {
    a->G = (int)(U < sms ? U : sms);
  }
  a->tq = (int)(a->tailT / a->G);
  a->tr = (int)(a->tailT % a->G);
  a->skip_load = -1;
  return true;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// The scratch buffer: the per-(batch, head) maxima of |V|, then (split schedule) the
// per-(tail unit, query tile, warp) counters and the partial records.  The maxima and the
// counters must be zero when a launch starts.
size_t vmax_bytes(int B, int heads) { return align256((size_t)B * heads * sizeof(unsigned)); }
size_t counter_bytes(const AttnArgs& a) {  // per (tail unit, query tile, 32-row warp)
  return a.split ? align256((size_t)8 * (a.U - a.W * a.G) * sizeof(int)) : 0;
}
size_t record_bytes(const AttnArgs& a) {
  return a.split ? (size_t)(a.G + (a.U - a.W * a.G)) * REC_BYTES : 0;
}

}  // namespace

DPP_BOUNDS_READER(bounds_tc_attn)

size_t tc_attention_scratch_bytes(int B, int L, int heads, int P, bool split) {
  AttnArgs a;
  if (!plan(B, L, heads, P, split, &a)) return 0;
  return vmax_bytes(B, heads) + counter_bytes(a) + record_bytes(a);
}

int tc_attention_zero_ints(int B, int L, int heads, int P, bool split) {
  AttnArgs a;
  if (!plan(B, L, heads, P, split, &a)) return 0;
  return (int)((vmax_bytes(B, heads) + counter_bytes(a)) / sizeof(int));
}

int launch_tc_attention(const void* q, const void* kf, const void* vf, const void* ks,
                        const void* vs, void* o, int B, int L, int heads, int P, bool split,
                        void* scratch, size_t scratch_bytes, bool scratch_zeroed,
                        bool vmax_ready, int* status, long long wait_limit, int skip_load,
                        cudaStream_t s) {
  AttnArgs a;
  if (!plan(B, L, heads, P, split, &a)) return DPP_ERR_SHAPE;
  const size_t vb = vmax_bytes(B, heads), cb = counter_bytes(a);
  if (!scratch || scratch_bytes < vb + cb + record_bytes(a)) return DPP_ERR_ARG;
  const int C = heads * D;
  int rc = set_attn_smem();
  if (rc) return rc;
  CUtensorMap mq, mkf, mks, mvf, mvs;
  if (!make_map3(&mq, q, L, B, C, QT) || !make_map3(&mkf, kf, L, B, C, a.g) ||
      !make_map3(&mks, ks, L, B, C, a.g) || !make_map3(&mvf, vf, L, B, C, a.g) ||
      !make_map3(&mvs, vs, L, B, C, a.g))
    return DPP_ERR_CUDA;
  a.o = static_cast<__nv_bfloat16*>(o);
  unsigned* vmax = static_cast<unsigned*>(scratch);
  a.vmax = vmax;
  if (a.split) {
    a.cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(scratch) + vb);
    a.part = static_cast<uint8_t*>(scratch) + vb + cb;
  }
  if (!scratch_zeroed && cudaMemsetAsync(scratch, 0, vb + cb, s) != cudaSuccess)
    return DPP_ERR_CUDA;
  a.status = status;
  a.wait_limit = wait_limit;
  a.skip_load = skip_load;
  // max |V| per (batch, head): about 2.5 blocks of 256 per SM
  const int want = 2 * dpp_host::sm_count() * 5 / 2 / (B * heads);
  const int chunks = want < 1 ? 1 : want;
  int rows = (L + chunks - 1) / chunks;
  rows = (rows + 31) / 32 * 32;
  const dim3 vgrid((unsigned)((L + rows - 1) / rows), (unsigned)heads, (unsigned)B);
  cudaError_t e = cudaSuccess;
  if (!vmax_ready)
    e = dpp_host::launch_pdl(vrange_kernel, vgrid, dim3(256), 0, s,
                             static_cast<const __nv_bfloat16*>(vf),
                             static_cast<const __nv_bfloat16*>(vs), L, heads, rows,
                             P > 1 && vs != vf ? 1 : 0, vmax);
  if (e != cudaSuccess) return DPP_ERR_CUDA;
  e = dpp_host::launch_pdl(tc_attn_kernel, dim3(a.G), dim3(ATTN_THREADS), ATTN_SMEM, s, mq, mkf,
                           mks, mvf, mvs, a);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

}  // namespace dpp
