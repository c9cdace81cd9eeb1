// tcgen05 GEMM engine for the bf16 path: the Q/K/V and output projections, and
// the halo conv3x3 as an implicit GEMM (M = B*H*W pixels, N = Cout, K = 9*Cin).
//
// Persistent: one CTA per SM walks output tiles of 128 x BN (BN = 320, 256, 160
// or 128, chosen per shape by pick_bn).  Warp 0 streams 64-wide K slices of A and
// B into a shared-memory ring with TMA (128-byte swizzle); warp 1 issues
// tcgen05.mma (M=128, K=16; one MMA of N=BN, or two of N=BN/2 for BN=320) and
// releases each stage with tcgen05.commit; warps 2-5 drain the accumulator
// (tcgen05.ld -> bf16 -> global).  With two TMEM accumulators (BN <= 256) a
// tile's epilogue overlaps the next tile's main loop.
//
// Halo conv staging ("Benchmarking DistVAE", Glossary: the halo rows a sharded
// convolution needs; "OTIL for SDXL on 4x L40S", item 3: the conv halo buffers
// are stale): for tap (di, dj) the A slice of an M tile is the tile's pixels
// shifted by (di, dj), fetched as row segments with a 4-D tensor map over the NHWC
// map.  A segment whose source row is inside its own row's band comes from the fresh
// map, one whose source row is the neighbouring band's (the halo) from the stale map,
// and the TMA zero fill of out-of-range rows/columns is the convolution's zero padding.
// Three tilings of the pixels (AMODE): 128 consecutive pixels as whole rows or one
// segment (W a multiple of 128, or 128 a multiple of W); 128 consecutive pixels as
// segments of gcd(W, 128) pixels that wrap across rows; or, when W has a divisor tp in
// [112, 128] (tp = 120 for the SDXL-3840 latent's W = 240), tp pixels of one row per
// tile -- one box per tap, the MMA's last 128 - tp rows never stored.
//
// Two opt-in variants: GNF (the conv's A is raw x; warps 6-9 apply GroupNorm to the
// landed in-band segments before the MMA reads a stage) and RFX (the Q/K/V projection
// whose epilogue, warps 2-9 in two groups taking alternate tiles, also quantises the
// K/V residual against the stale rows and writes the refreshed rows and the message).
#include <cudaTypedefs.h>

#include <mutex>

#include "ptx.cuh"
#include "quant.cuh"
#include "tc.cuh"

namespace dpp {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int GEMM_THREADS = 192;     // producer, MMA, 4 epilogue warps
constexpr int GEMM_GN_THREADS = 320;  // + 4 warps applying GroupNorm to the A operand
constexpr int kBarBytes = 512;        // barriers, flags and per-stage notes

constexpr int kMaxDynSmem = 227 * 1024;

template <int BN>
struct Cfg {
  static constexpr int MMA_N = BN > 256 ? BN / 2 : BN;  // N of one MMA (<= 256)
  static constexpr int NMMA = BN / MMA_N;               // MMAs per K step
  static constexpr int NACC = 2 * BN <= 512 ? 2 : 1;    // TMEM accumulators
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (kMaxDynSmem - 1024 /*align*/ - kBarBytes) / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + kBarBytes;
  static constexpr uint32_t TMEM_COLS = NACC * BN <= 256 ? 256 : 512;
  static_assert(BN % MMA_N == 0 && MMA_N % 16 == 0 && MMA_N <= 256, "MMA shape");
  static_assert(SMEM <= kMaxDynSmem && STAGES >= 2, "shared memory");
};

struct GemmArgs {
  long long M;
  int N, K, nkb;
  int m_tiles, n_tiles;
  void* out[3];
  int ncols;
  int* status;
  long long wait_limit;
  long long skip_load;  // test hook: the producer never loads this K slice (-1: none)
  // implicit conv
  int H, W, Cin, Hp, cin_blocks, boxes, box_px;
  // conv with GroupNorm applied to the in-band rows of A (raw x): [B][P][3][Cin] fp32
  // (mean, rstd * gamma, beta per channel of each batch and patch)
  const float* gn_par;
  int P;
  // linear whose K and V outputs (1, 2) are also refreshed (RFX): against the stale
  // values at rfx_stale[i] into rfx_out[i], codes and block scales at the message
  // offsets of each
  const void* rfx_stale[2];
  void* rfx_out[2];
  int8_t* rfx_codes[2];
  float* rfx_scales[2];
  // linear with a three-way split output: max |out| of the third output (V) per (batch of
  // vmax_L rows, 64-column head) into vmax as fp32 bits by atomicMax, or NULL
  unsigned* vmax;
  int vmax_L, vmax_heads;
  // conv: max |V| per (batch of vmax_L rows, 64-column head) of this [vs_rows, vs_C] bf16
  // tensor (the stale V) into vmax (NULL: none); vs_scan = 1: by the CTAs past the last
  // tile, which do nothing else; 0: by the epilogue warps while the first accumulator fills
  const __nv_bfloat16* vs_src;
  long long vs_rows;
  int vs_C;
  int vs_scan;
};

// What the producer fetched into a stage, for the GroupNorm warps: the boxes' first
// column (c0 + dj) and which boxes hold in-band rows of x (bit per box).
struct StageNote {
  int col0, fresh;
};

// GNF (conv only): tmA maps the raw input x, tmA2 the stale GroupNorm output; warps
// 6-9 turn each landed in-band box of x into y = (x - mean) * scale + beta in place
// (the zero fill of out-of-image positions stays 0) before the MMA reads the stage.
// The epilogue of one 128-column K or V row with its refresh: the accumulator row is
// rounded to bf16 and stored as fresh K/V (as in the plain epilogue), the residual
// against the stale row is quantised (one 128-element block: shared quantiser) and the
// refreshed row, the 128 codes and the block scale are written.  `flat` is the row's
// offset in the flat [B*L*C] tensor, a multiple of 128.  The stale row is loaded at once
// (one memory latency per row); the quantising pass walks the four 32-column chunks in
// a loop that is not unrolled (the unrolled row did not fit the instruction cache),
// re-reading each chunk from TMEM and picking its stale vectors by compares.
__device__ __forceinline__ uint4 pick4(const uint4 (&v)[16], int ch, int i) {
  const uint4 a = v[i], b = v[4 + i], c = v[8 + i], d = v[12 + i];
  return ch == 0 ? a : ch == 1 ? b : ch == 2 ? c : d;
}

__device__ __forceinline__ void pack_row32(const uint32_t (&v)[32], uint4 (&f)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[i].x = pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1]));
    f[i].y = pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3]));
    f[i].z = pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5]));
    f[i].w = pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7]));
  }
}

__device__ __forceinline__ void refresh_row(uint32_t t_row, __nv_bfloat16* dst, bool live,
                                            bool is_k, const GemmArgs& args, long long flat) {
  const __nv_bfloat16* sp =
      static_cast<const __nv_bfloat16*>(is_k ? args.rfx_stale[0] : args.rfx_stale[1]) + flat;
  __nv_bfloat16* op = static_cast<__nv_bfloat16*>(is_k ? args.rfx_out[0] : args.rfx_out[1]) + flat;
  int8_t* cp = (is_k ? args.rfx_codes[0] : args.rfx_codes[1]) + flat;
  float* scp = (is_k ? args.rfx_scales[0] : args.rfx_scales[1]) + flat / 128;
  uint4 sb[16];  // the stale row, 8 values per vector
  if (live) {
#pragma unroll
    for (int i = 0; i < 16; ++i) sb[i] = __ldcs(reinterpret_cast<const uint4*>(sp) + i);
  }
  // pass 1: fresh K/V out, and the block's absolute maximum of fresh - stale
  float amax = 0.0f;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t v[32];
    ptx::tmem_ld32(t_row + ch * 32, v);
    ptx::tmem_ld_wait();
    uint4 f[4];
    pack_row32(v, f);
    if (live) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        reinterpret_cast<uint4*>(dst)[4 * ch + i] = f[i];
        float fv[8], sv[8];
        unpack16(f[i], fv);
        unpack16(pick4(sb, ch, i), sv);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(fv[e] - sv[e]));
      }
    }
  }
  if (!live) return;
  const QuantBlock qb = quant_block(amax);
  *scp = qb.s;
  // pass 2: codes and refreshed values
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t v[32];
    ptx::tmem_ld32(t_row + ch * 32, v);
    ptx::tmem_ld_wait();
    uint4 f[4];
    pack_row32(v, f);
    uint32_t cw[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float fv[8], sv[8], d[8], tm[8], nv[8];
      unpack16(f[i], fv);
      unpack16(pick4(sb, ch, i), sv);
#pragma unroll
      for (int e = 0; e < 8; ++e) d[e] = fv[e] - sv[e];
      quant8(qb, d, sv, tm, nv);
      const uint2 c = pack_codes(tm);
      cw[2 * i] = c.x;
      cw[2 * i + 1] = c.y;
      __stcs(reinterpret_cast<uint4*>(op) + 4 * ch + i, pack16(nv));
    }
    __stcs(reinterpret_cast<uint4*>(cp) + 2 * ch, make_uint4(cw[0], cw[1], cw[2], cw[3]));
    __stcs(reinterpret_cast<uint4*>(cp) + 2 * ch + 1, make_uint4(cw[4], cw[5], cw[6], cw[7]));
  }
}

// max |V| per (batch, head) over rows [vs_rows e / E, vs_rows (e + 1) / E) of the stale V,
// by every thread of the CTA: virtual thread c takes the 16-byte column c mod ncol (eight
// channels of one head) of rows r0 + c / ncol, then every rpp-th row, eight rows' loads in
// flight, and flushes its maximum by atomicMax (fp32 bits of a non-negative value) when
// its rows enter the next batch.
__device__ __noinline__ void scan_vmax(const GemmArgs& a, int e, int E) {
  const int ncol = a.vs_C / 8;
  const int rpp = max(1, (int)blockDim.x / ncol);
  const long long r0 = a.vs_rows * e / E, r1 = a.vs_rows * (e + 1) / E;
  const long long nv = a.vs_rows * a.vs_C, nmax = a.vs_rows / a.vmax_L * a.vmax_heads;
  for (int c = threadIdx.x; c < ncol * rpp; c += blockDim.x) {
    const int cc = c % ncol;
    unsigned* const col_max = a.vmax + (cc * 8) / 64;
    uint32_t m = 0;
    long long row = r0 + c / ncol;
    long long b = row / a.vmax_L, bend = (b + 1) * a.vmax_L;
    for (; row < r1; row += 8ll * rpp) {
      uint4 u[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (row + (long long)k * rpp < r1 &&
            DPP_IN((row + (long long)k * rpp) * a.vs_C + cc * 8, 8, nv))
          u[k] = __ldcs(reinterpret_cast<const uint4*>(a.vs_src + (row + (long long)k * rpp) *
                                                                     a.vs_C) + cc);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const long long rk = row + (long long)k * rpp;
        if (rk >= r1) break;
        while (rk >= bend) {  // next batch: flush this one's maximum
          if (m && DPP_IN(b * a.vmax_heads + (cc * 8) / 64, 1, nmax))
            atomicMax(col_max + b * a.vmax_heads, m << 16);
          m = 0;
          ++b;
          bend += a.vmax_L;
        }
        const uint32_t w4[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) m = max(m, max(w4[i] & 0x7FFFu, (w4[i] >> 16) & 0x7FFFu));
      }
    }
    if (m && DPP_IN(b * a.vmax_heads + (cc * 8) / 64, 1, nmax))
      atomicMax(col_max + b * a.vmax_heads, m << 16);
  }
}

// RFX (linear, 128-wide tiles): a K or V tile row is exactly one 128-element refresh
// block, so the epilogue thread that stores a row of fresh K or V also quantises its
// residual against the stale row and writes the refreshed row, the codes and the scale.
template <bool CONV, int BN, bool GNF, bool RFX = false, int AMODE = 0>
__global__ void __launch_bounds__(GNF || RFX ? GEMM_GN_THREADS : GEMM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  using C = Cfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;   // [NACC] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;    // [NACC] epilogue -> MMA (4 warps)
  uint64_t* drain = acc_empty + 2;
  uint64_t* xform = drain + 1;           // [STAGES] GroupNorm warps -> MMA (GNF)
  StageNote* note = reinterpret_cast<StageNote*>(xform + STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(note + STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((2 * STAGES + 5 + STAGES) * 8 + STAGES * sizeof(StageNote) + 8 <= kBarBytes,
                "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = args.m_tiles * args.n_tiles;
  if constexpr (CONV && !GNF) {
    if (args.vs_scan && (int)blockIdx.x >= ntiles) {  // no tile: the stale V's maxima only
      ptx::grid_dep_wait();  // vmax was zeroed by an earlier kernel of the chain
      scan_vmax(args, blockIdx.x - ntiles, gridDim.x - ntiles);
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
      if (GNF) ptx::mbar_init(&xform[s], 4);  // one arrival per GroupNorm warp
    }
    for (int b = 0; b < C::NACC; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], 4);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    if (CONV) ptx::tma_prefetch_desc(&tmA2);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the set-up above overlaps the previous kernel; its outputs are read from here on
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      long long g = 0;  // global K-slice counter across tiles
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int mt = tile / args.n_tiles, nt = tile - mt * args.n_tiles;
        const long long m0 = (long long)mt * BM;
        const int n0 = nt * BN;
        int b = 0, r = 0, c0 = 0;
        if (CONV && AMODE == 2) {  // a tile is box_px pixels of one row (rows padded)
          const int tpr = args.W / args.box_px, R = mt / tpr;
          b = R / args.H;
          r = R - b * args.H;
          c0 = (mt - R * tpr) * args.box_px;
        } else if (CONV) {
          const long long hw = (long long)args.H * args.W;
          b = (int)(m0 / hw);
          const int rem = (int)(m0 - (long long)b * hw);
          r = rem / args.W;
          c0 = rem - r * args.W;
        }
        // K slices in a rotated order that depends only on the tile, so that CTAs
        // working on the same B tile at the same time fetch different slices (no
        // hot spot on one L2 slice) while a given tile always sums in one order.
        const int rot = (int)(mt % args.nkb);
        // Per tile, once: for each row shift di and A box bx, whether the source row is
        // the neighbouring band's halo (stale map) and, for the GroupNorm warps, whether it
        // is an in-band row of the image (fresh x).  Bit (di + 1) * 16 + bx; the per-slice
        // path then holds no division (the single producer thread's issue time bounds the
        // slice rate: measured, each further box with its divisions cost ~0.2 us a slice).
        uint64_t stale_bits = 0, fresh_bits = 0;
        if (CONV) {
          int rk = r, ck = c0;  // image row and column of box bx's first pixel
          for (int bx = 0; bx < args.boxes; ++bx) {
            for (int d = -1; d <= 1; ++d) {
              const int rr = rk + d;
              const bool in = rr >= 0 && rr < args.H;
              const bool same = in && (rr / args.Hp) == (rk / args.Hp);
              if (in && !same) stale_bits |= 1ull << ((d + 1) * 16 + bx);
              if (same) fresh_bits |= 1ull << ((d + 1) * 16 + bx);
            }
            if (AMODE == 1) {
              ck += args.box_px;
              if (ck == args.W) {
                ck = 0;
                ++rk;
              }
            } else {
              ++rk;
            }
          }
        }
        // the current slice kb and its tap (di, dj) and input-channel block cb, advanced
        // by one slice at a time
        int kb = rot, cb = 0, di = -1, dj = -1;
        if (CONV) {
          const int tap = rot / args.cin_blocks;
          cb = rot - tap * args.cin_blocks;
          di = tap / 3 - 1;
          dj = tap - 3 * (tap / 3) - 1;
        }
        for (int kq = 0; kq < args.nkb; ++kq, ++g) {
          const int s = (int)(g % STAGES);
          const uint32_t ph = (uint32_t)((g / STAGES) & 1);
          if (!ptx::mbar_wait(&empty[s], ph ^ 1, args.wait_limit, abort_flag)) {
            set_status(args.status, DPP_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (g != args.skip_load) {  // test hook: that slice never lands
            uint8_t* a_dst = smem + s * C::STAGE_BYTES;
            uint8_t* b_dst = a_dst + C::A_BYTES;
            const int sh = (di + 1) * 16;
            if (GNF)  // the note first: the arrive below releases it to the waiters
              note[s] = StageNote{c0 + dj, (int)((fresh_bits >> sh) & 0xFFFFu)};
            // padded row tiles: only box_px of the 128 A rows are loaded (the MMA rows past
            // them compute values that the epilogue never stores)
            ptx::mbar_arrive_expect_tx(
                &full[s], AMODE == 2 ? (uint32_t)(args.box_px * 128 + C::B_BYTES) : C::STAGE_BYTES);
            if (CONV) {
              // box bx holds pixels [m0 + bx * box_px, +box_px) of the image: one row
              // segment (box_px divides W).  Whole rows (box_px == W) or one box per tile
              // (W a multiple of 128): box bx is row r + bx from column c0; with WRAP the
              // segments wrap across rows.
              int rk = r, ck = c0;
              for (int bx = 0; bx < args.boxes; ++bx) {
                const bool stale = (stale_bits >> (sh + bx)) & 1u;
                ptx::tma_load_4d(a_dst + bx * args.box_px * 128, stale ? &tmA2 : &tmA,
                                 &full[s], cb * BK, ck + dj, rk + di, b);
                if (AMODE == 1) {
                  ck += args.box_px;
                  if (ck == args.W) {
                    ck = 0;
                    ++rk;
                  }
                } else {
                  ++rk;
                }
              }
            } else {
              ptx::tma_load_2d(a_dst, &tmA, &full[s], kb * BK, (int)m0);
            }
#pragma unroll
            for (int h = 0; h < C::NMMA; ++h)
              ptx::tma_load_2d(b_dst + h * C::MMA_N * 128, &tmB, &full[s], kb * BK,
                               n0 + h * C::MMA_N);
          }
          // the next slice in the rotated order
          if (++kb == args.nkb) {
            kb = 0;
            cb = 0;
            di = -1;
            dj = -1;
          } else if (CONV && ++cb == args.cin_blocks) {
            cb = 0;
            if (++dj == 2) {
              dj = -1;
              ++di;
            }
          }
        }
      }
      if (*abort_flag) {  // wait for own copies still in flight before the CTA may exit
        const long long first = g > STAGES ? g - STAGES : 0;
        for (long long q = first; q < g; ++q)
          if (q != args.skip_load)
            ptx::mbar_wait(&full[q % STAGES], (uint32_t)((q / STAGES) & 1), kDrainWaitLimit,
                           nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_f16(BM, C::MMA_N, 1, 0, 0);
      bool any = false, ok = true;
      long long g = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
        const int ab = it % C::NACC;
        if (!ptx::mbar_wait(&acc_empty[ab], ((it / C::NACC) & 1) ^ 1, args.wait_limit,
                            abort_flag)) {
          set_status(args.status, DPP_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + ab * BN;
        for (int kb = 0; kb < args.nkb; ++kb, ++g) {
          const int s = (int)(g % STAGES);
          const uint32_t ph = (uint32_t)((g / STAGES) & 1);
          if (!ptx::mbar_wait(GNF ? &xform[s] : &full[s], ph, args.wait_limit, abort_flag)) {
            set_status(args.status, DPP_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
#pragma unroll
            for (int h = 0; h < C::NMMA; ++h)
              ptx::mma_ss(d_tmem + h * C::MMA_N, ptx::sw128_desc(a_addr + k * 32, 16, 1024),
                          ptx::sw128_desc(b_addr + h * C::MMA_N * 128 + k * 32, 16, 1024), idesc,
                          (kb | k) ? 1u : 0u);
          any = true;
          ptx::mma_commit(&empty[s]);
        }
        if (ok) ptx::mma_commit(&acc_full[ab]);
      }
      if (*abort_flag && any) {  // let issued MMAs finish before TMEM is released
        ptx::mma_commit(drain);
        ptx::mbar_wait(drain, 0, kDrainWaitLimit, nullptr);
      }
    }
  } else if (GNF && warp >= 6) {
    // ------------------------------------------------ GroupNorm on A (warps 6..9)
    // Per stage: the in-band boxes of raw x become y = (x - mean) * scale + beta, the
    // apply of the separate GroupNorm kernel written out (same operations, same bf16
    // rounding); boxes of stale y and the zero fill outside the image are left as they
    // are.  The 128-byte swizzle puts logical 16-byte chunk (ch ^ (row & 7)) of a
    // 128-byte row at physical chunk ch (box rows start on 1024-byte boundaries).
    // Thread t handles 16-byte chunk (t & 7) of A rows (t >> 3) + 16 i, i = 0..7: every
    // such row has the same (row & 7), so the thread's 8 channels are the same in all
    // eight chunks and their parameters are loaded once per stage.
    const int tid = threadIdx.x - 6 * 32;
    const int ch = tid & 7, row_lo = tid >> 3;
    const int c = (ch ^ (row_lo & 7)) << 3;  // first of the thread's 8 channels
    const int box_lg = __ffs(args.box_px) - 1;  // box_px is a power of two
    long long g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      // the tile's batch and band, and its K-slice rotation, as the producer has them:
      // the parameters of a stage are fetched before its data lands
      const int mt = tile / args.n_tiles;
      const long long m0 = (long long)mt * BM;
      const long long hw = (long long)args.H * args.W;
      const int tb = (int)(m0 / hw);
      const int band = (int)((m0 - (long long)tb * hw) / args.W) / args.Hp;
      const float* par_tile = args.gn_par + ((long long)tb * args.P + band) * 3 * args.Cin + c;
      const int rot = (int)(mt % args.nkb);
      for (int kq = 0; kq < args.nkb; ++kq, ++g) {
        const int s = (int)(g % STAGES);
        const uint32_t ph = (uint32_t)((g / STAGES) & 1);
        const int kb = kq + rot < args.nkb ? kq + rot : kq + rot - args.nkb;
        const float* par = par_tile + (kb % args.cin_blocks) * BK;
        float mu[8], sc[8], be[8];
        const bool par_in = DPP_IN(((long long)tb * args.P + band) * 3 * args.Cin + c +
                                       (kb % args.cin_blocks) * BK,
                                   2 * args.Cin + 8, args.M / hw * args.P * 3 * args.Cin);
#pragma unroll
        for (int h = 0; h < 2 && par_in; ++h) {
          const float4 m = __ldg(reinterpret_cast<const float4*>(par) + h);
          const float4 k = __ldg(reinterpret_cast<const float4*>(par + args.Cin) + h);
          const float4 e = __ldg(reinterpret_cast<const float4*>(par + 2 * args.Cin) + h);
          mu[4 * h] = m.x; mu[4 * h + 1] = m.y; mu[4 * h + 2] = m.z; mu[4 * h + 3] = m.w;
          sc[4 * h] = k.x; sc[4 * h + 1] = k.y; sc[4 * h + 2] = k.z; sc[4 * h + 3] = k.w;
          be[4 * h] = e.x; be[4 * h + 1] = e.y; be[4 * h + 2] = e.z; be[4 * h + 3] = e.w;
        }
        if (!ptx::mbar_wait(&full[s], ph, args.wait_limit, abort_flag)) {
          set_status(args.status, DPP_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const StageNote nt = note[s];
        const uint32_t fresh = (uint32_t)nt.fresh;
        if (fresh) {
          uint8_t* a_st = smem + s * C::STAGE_BYTES + ch * 16;
          uint4 v[8];
          uint32_t take = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = row_lo + 16 * i;  // row of the 128-row A tile
            const int bx = row >> box_lg;
            const int col = nt.col0 + (row & (args.box_px - 1));
            if (((fresh >> bx) & 1) && col >= 0 && col < args.W) {
              take |= 1u << i;
              v[i] = *reinterpret_cast<const uint4*>(a_st + row * 128);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (!((take >> i) & 1)) continue;
            float f[8];
            unpack16(v[i], f);
#pragma unroll
            for (int k = 0; k < 8; ++k) f[k] = fmaf(f[k] - mu[k], sc[k], be[k]);
            *reinterpret_cast<uint4*>(a_st + (row_lo + 16 * i) * 128) = pack16(f);
          }
          ptx::fence_proxy_async_smem();  // generic writes -> the tensor core's reads
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&xform[s]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5; RFX: 2..9)
    // With RFX two groups of four warps take alternate tiles (group g drains
    // accumulator g), so a refreshing epilogue may take two main loops' time.
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int group = RFX ? (warp - 2) >> 2 : 0;
    if (CONV && !GNF && args.vs_src && !args.vs_scan) {
      // This CTA's share of the rows, eight rows' loads in flight per thread; thread t
      // takes the 16-byte columns t, t + 128, ... of each row (eight channels of one head)
      // and keeps its maximum until the rows' batch changes.
      const int et = threadIdx.x - 64, ncol = args.vs_C / 8;
      const long long r0 = args.vs_rows * blockIdx.x / gridDim.x;
      const long long r1 = args.vs_rows * (blockIdx.x + 1) / gridDim.x;
      const long long nv = args.vs_rows * args.vs_C;
      const long long nmax = args.vs_rows / args.vmax_L * args.vmax_heads;
      for (int cc = et; cc < ncol; cc += 128) {
        uint32_t m = 0;
        long long b = r0 / args.vmax_L, bend = (b + 1) * args.vmax_L;
        for (long long row = r0; row < r1; row += 8) {
          uint4 u[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (row + k < r1 && DPP_IN((row + k) * args.vs_C + cc * 8, 8, nv))
              u[k] = __ldcs(reinterpret_cast<const uint4*>(args.vs_src + (row + k) * args.vs_C) + cc);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (row + k >= r1) break;
            if (row + k == bend) {  // next batch: flush this one's maximum
              if (m && DPP_IN(b * args.vmax_heads + (cc * 8) / 64, 1, nmax))
                atomicMax(args.vmax + b * args.vmax_heads + (cc * 8) / 64, m << 16);
              m = 0;
              ++b;
              bend += args.vmax_L;
            }
            const uint32_t w4[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) m = max(m, max(w4[e] & 0x7FFFu, (w4[e] >> 16) & 0x7FFFu));
          }
        }
        if (m && DPP_IN(b * args.vmax_heads + (cc * 8) / 64, 1, nmax))
          atomicMax(args.vmax + b * args.vmax_heads + (cc * 8) / 64, m << 16);
      }
    }
    int it = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
      if (RFX && (it & 1) != group) continue;
      const int ab = it % C::NACC;
      if (!ptx::mbar_wait(&acc_full[ab], (it / C::NACC) & 1, args.wait_limit, abort_flag)) {
        set_status(args.status, DPP_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const int mt = tile / args.n_tiles, nt = tile - mt * args.n_tiles;
      long long row = (long long)mt * BM + quarter * 32 + lane;
      bool row_ok = row < args.M;
      if (CONV && AMODE == 2) {  // pixel c0 + local of image row R
        const int tpr = args.W / args.box_px, R = mt / tpr, local = quarter * 32 + lane;
        row = (long long)R * args.W + (long long)(mt - R * tpr) * args.box_px + local;
        row_ok = local < args.box_px;
      }
      const int n0 = nt * BN;
      const int which = n0 / args.ncols;
      const int col0 = n0 - which * args.ncols;
      // select, not index: a run-time index into the parameter struct would copy it
      // to local memory
      void* const obase = which == 0 ? args.out[0] : which == 1 ? args.out[1] : args.out[2];
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(obase) + row * args.ncols + col0;
      const uint32_t t_base = tmem + ab * BN + ((uint32_t)(quarter * 32) << 16);
      const bool rfx_row = RFX && which > 0;
      const long long nout = args.M * args.ncols;  // elements of each output
      if (rfx_row)
        refresh_row(t_base, dst, row_ok && DPP_IN(row * args.ncols + col0, 128, nout), which == 1,
                    args, row * args.ncols + col0);
#pragma unroll 1
      for (int ch = 0; ch < (rfx_row ? 0 : BN / 32); ++ch) {
        uint32_t v[32];
        ptx::tmem_ld32(t_base + ch * 32, v);
        ptx::tmem_ld_wait();
        uint4 pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pk[i].x = pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1]));
          pk[i].y = pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3]));
          pk[i].z = pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5]));
          pk[i].w = pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7]));
        }
        if (row_ok && DPP_IN(row * args.ncols + col0 + ch * 32, 32, nout)) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = pk[i];
        }
        if (!CONV && which == 2 && args.vmax) {  // max |V| of these 32 columns (one head)
          uint32_t m = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t w4[4] = {pk[i].x, pk[i].y, pk[i].z, pk[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) m = max(m, max(w4[e] & 0x7FFFu, (w4[e] >> 16) & 0x7FFFu));
          }
          m = __reduce_max_sync(0xffffffffu, row_ok ? m : 0u);
          const long long r0 = (long long)mt * BM + quarter * 32;
          if (lane == 0 && m &&  // the warp's 32 rows lie in one batch (L % 128 == 0)
              DPP_IN((r0 / args.vmax_L) * args.vmax_heads + (col0 + ch * 32) / 64, 1,
                     args.M / args.vmax_L * args.vmax_heads)) {
            atomicMax(args.vmax + (r0 / args.vmax_L) * args.vmax_heads + (col0 + ch * 32) / 64,
                      m << 16);
          }
        }
      }
      // accumulator drained: the MMA warp may reuse it
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

DPP_BOUNDS_READER(bounds_tc_gemm)

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

namespace {

// bf16 tensor map with 128-byte swizzle; dims/box innermost first, strides in bytes
// for dims 1..rank-1.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box) {
  auto fn = tc_encode_fn();
  if (!fn) return false;
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool CONV, int BN, bool GNF, bool RFX = false, int AMODE = 0>
int prepare() {
  static std::once_flag once;
  static int rc = DPP_OK;
  std::call_once(once, [] {
    if (cudaFuncSetAttribute(tc_gemm_kernel<CONV, BN, GNF, RFX, AMODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<BN>::SMEM) != cudaSuccess)
      rc = DPP_ERR_CUDA;
  });
  return rc;
}

// Tile width for an M x N x (nkb * 64) GEMM.  Measured on the GB300 at the layer's
// sizes, the time per K slice is nearly the same for 36 KB and 56 KB stages (the
// ring's latency, not its bytes, sets it), so the 128 x 320 tile (two MMAs per K
// step, one accumulator) does twice the work per slice: it halved the SDXL-1024
// conv (K = 5760, 90 slices).  With one accumulator its epilogue (~3 us) is not
// overlapped, which costs more than it saves for the K = 640 projections (10
// slices), so it is taken only for long K loops; otherwise the widest of 256 / 160
// / 128 that divides N, with two accumulators.
int pick_bn(int N, int ncols, int nkb) {
  if (nkb >= 32 && N % 320 == 0 && ncols % 320 == 0) return 320;
  for (int bn : {256, 160, 128})
    if (N % bn == 0 && ncols % bn == 0) return bn;  // no tile straddles two split outputs
  return 0;
}

constexpr int mma_n(int bn) { return bn > 256 ? bn / 2 : bn; }

template <bool CONV, int BN, bool GNF, bool RFX = false, int AMODE = 0>
int launch(const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb, GemmArgs g,
           cudaStream_t s) {
  int rc = prepare<CONV, BN, GNF, RFX, AMODE>();
  if (rc) return rc;
  g.n_tiles = g.N / BN;
  const long long ntiles = (long long)g.m_tiles * g.n_tiles;
  const int sms = dpp_host::sm_count();
  int grid = (int)(ntiles < sms ? ntiles : sms);
  // The stale V's maxima: by CTAs of their own on the SMs the tiles leave idle (at most
  // 1 MB each, a few us beside the tiles' main loops), else by the epilogue warps.
  if (CONV && !GNF && g.vs_src && ntiles < sms &&
      (long long)(sms - ntiles) << 20 >= g.vs_rows * g.vs_C * 2) {
    g.vs_scan = 1;
    grid = sms;
  }
  const cudaError_t e =
      dpp_host::launch_pdl(tc_gemm_kernel<CONV, BN, GNF, RFX, AMODE>, dim3(grid),
                           dim3(GNF || RFX ? GEMM_GN_THREADS : GEMM_THREADS), Cfg<BN>::SMEM, s, ta, ta2,
                           tb, g);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? DPP_OK : DPP_ERR_CUDA;
}

template <bool CONV, bool GNF, int AMODE = 0>
int dispatch(int bn, const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb,
             const GemmArgs& g, cudaStream_t s) {
  switch (bn) {
    case 320: return launch<CONV, 320, GNF, false, AMODE>(ta, ta2, tb, g, s);
    case 256: return launch<CONV, 256, GNF, false, AMODE>(ta, ta2, tb, g, s);
    case 160: return launch<CONV, 160, GNF, false, AMODE>(ta, ta2, tb, g, s);
    case 128: return launch<CONV, 128, GNF, false, AMODE>(ta, ta2, tb, g, s);
    default: return DPP_ERR_SHAPE;
  }
}

}  // namespace

bool tc_linear_supported(long long M, int C) {
  return M % BM == 0 && C % 128 == 0 && C % BK == 0 && M < (1ll << 31);
}

// Tiles of 128 pixels never straddle two images; each is fetched per tap as 128 / box_px
// row segments of box_px = gcd(W, 128) pixels (at least 8: W a multiple of 8).
bool tc_conv_supported(int B, int H, int W, int Cin, int Cout, int P) {
  if (Cin % BK || Cin <= 0 || Cout <= 0 || !pick_bn(Cout, Cout, 9 * Cin / BK)) return false;
  if (W % 8 || ((long long)H * W) % BM) return false;
  (void)B;
  (void)P;
  return true;
}

// The GroupNorm-fused variant assumes one band and one starting column per tile.
bool tc_conv_gn_supported(int H, int W, int P) {
  return (W % 128 == 0 || 128 % W == 0) && ((long long)(H / P) * W) % BM == 0;
}

int launch_tc_linear(const void* a, const void* w, void* o0, void* o1, void* o2, long long M,
                     int N, int K, int* status, long long wait_limit, cudaStream_t s,
                     unsigned* vmax, int vmax_L, int vmax_heads) {
  if (M % BM || N % 128 || K % BK) return DPP_ERR_SHAPE;
  const int ncols = o1 ? N / 3 : N;
  const int bn = pick_bn(N, ncols, K / BK);
  if (!bn) return DPP_ERR_SHAPE;
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)K * 2};
  const uint32_t ba[2] = {BK, BM};
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N}, sb[1] = {(uint64_t)K * 2};
  const uint32_t bb[2] = {BK, (uint32_t)mma_n(bn)};
  if (!make_map(&ta, a, 2, da, sa, ba) || !make_map(&tb, w, 2, db, sb, bb)) return DPP_ERR_CUDA;
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.nkb = K / BK;
  g.m_tiles = (int)(M / BM);
  g.out[0] = o0; g.out[1] = o1; g.out[2] = o2;
  g.ncols = ncols;
  g.status = status;
  g.wait_limit = wait_limit;
  g.skip_load = dpp_host::skip_load_from_env("linear");
  if (vmax && (!o2 || vmax_L % BM || ncols % 64)) return DPP_ERR_SHAPE;
  g.vmax = vmax;
  g.vmax_L = vmax_L;
  g.vmax_heads = vmax_heads;
  return dispatch<false, false>(bn, ta, ta, tb, g, s);
}

int launch_tc_linear_refresh(const void* a, const void* w, void* o0, void* o1, void* o2,
                             long long M, int N, int K, const void* k_stale, const void* v_stale,
                             void* k_out, void* v_out, int8_t* codes, float* scales,
                             int* status, long long wait_limit, cudaStream_t s) {
  if (M % BM || N % 384 || K % BK || !o1 || !o2) return DPP_ERR_SHAPE;
  const int ncols = N / 3;
  if (ncols % 128) return DPP_ERR_SHAPE;
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)K * 2};
  const uint32_t ba[2] = {BK, BM};
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N}, sb[1] = {(uint64_t)K * 2};
  const uint32_t bb[2] = {BK, 128};
  if (!make_map(&ta, a, 2, da, sa, ba) || !make_map(&tb, w, 2, db, sb, bb)) return DPP_ERR_CUDA;
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.nkb = K / BK;
  g.m_tiles = (int)(M / BM);
  g.out[0] = o0; g.out[1] = o1; g.out[2] = o2;
  g.ncols = ncols;
  g.status = status;
  g.wait_limit = wait_limit;
  g.skip_load = dpp_host::skip_load_from_env("linear");
  const long long blc = M * ncols;  // elements of K (and of V): V's codes follow K's
  g.rfx_stale[0] = k_stale; g.rfx_stale[1] = v_stale;
  g.rfx_out[0] = k_out; g.rfx_out[1] = v_out;
  g.rfx_codes[0] = codes; g.rfx_codes[1] = codes + blc;
  g.rfx_scales[0] = scales; g.rfx_scales[1] = scales + blc / 128;
  return launch<false, 128, false, true>(ta, ta, tb, g, s);
}

int launch_tc_conv(const void* yf, const void* ys, const void* w, void* out, int B, int H, int W,
                   int Cin, int Cout, int P, const float* gn_par, int* status,
                   long long wait_limit, cudaStream_t s, const void* vstale, int vs_C,
                   unsigned* vmax, int heads) {
  if (!tc_conv_supported(B, H, W, Cin, Cout, P)) return DPP_ERR_SHAPE;
  const int bn = pick_bn(Cout, Cout, 9 * Cin / BK);
  if (!bn) return DPP_ERR_SHAPE;
  int box_px = 128;  // gcd(W, 128)
  while (W % box_px) box_px >>= 1;
  // When gcd(W, 128) is small (e.g. 16 for the SDXL-3840 latent's W = 240) a 128-pixel
  // tile would need many short row segments per tap; instead a tile is the largest
  // divisor tp <= 128 of W (120 for W = 240) pixels of one row -- one box per tap -- with
  // the MMA's last 128 - tp rows unused, when that wastes at most 1/8 of the rows.
  int amode = box_px == W || box_px == 128 ? 0 : 1;
  if (amode == 1 && !gn_par) {
    int tp = 128;
    while (W % tp) --tp;
    if (tp >= 112) {
      amode = 2;
      box_px = tp;
    }
  }
  if (gn_par && !tc_conv_gn_supported(H, W, P)) return DPP_ERR_SHAPE;
  CUtensorMap tf, ts, tw;
  const uint64_t dy[4] = {(uint64_t)Cin, (uint64_t)W, (uint64_t)H, (uint64_t)B};
  const uint64_t sy[3] = {(uint64_t)Cin * 2, (uint64_t)W * Cin * 2, (uint64_t)H * W * Cin * 2};
  const uint32_t by[4] = {BK, (uint32_t)box_px, 1, 1};
  const int K = 9 * Cin;
  const uint64_t dw[2] = {(uint64_t)K, (uint64_t)Cout}, sw[1] = {(uint64_t)K * 2};
  const uint32_t bw[2] = {BK, (uint32_t)mma_n(bn)};
  if (!make_map(&tf, yf, 4, dy, sy, by) || !make_map(&ts, ys, 4, dy, sy, by) ||
      !make_map(&tw, w, 2, dw, sw, bw))
    return DPP_ERR_CUDA;
  GemmArgs g{};
  g.M = (long long)B * H * W; g.N = Cout; g.K = K; g.nkb = K / BK;
  g.m_tiles = amode == 2 ? B * H * (W / box_px) : (int)(g.M / BM);
  g.out[0] = out; g.ncols = Cout;
  g.status = status;
  g.wait_limit = wait_limit;
  g.skip_load = dpp_host::skip_load_from_env("conv");
  g.H = H; g.W = W; g.Cin = Cin; g.Hp = H / P; g.cin_blocks = Cin / BK;
  g.boxes = amode == 2 ? 1 : BM / box_px;
  g.box_px = box_px;
  g.gn_par = gn_par;
  g.P = P;
  if (vstale && !gn_par) {  // [B, H*W, vs_C] stale V: its maxima (scan CTAs or epilogue)
    if (!vmax || vs_C % 64 || heads * 64 != vs_C) return DPP_ERR_SHAPE;
    g.vs_src = static_cast<const __nv_bfloat16*>(vstale);
    g.vs_rows = (long long)B * H * W;
    g.vs_C = vs_C;
    g.vmax = vmax;
    g.vmax_L = H * W;
    g.vmax_heads = heads;
  }
  if (gn_par) return dispatch<true, true>(bn, tf, ts, tw, g, s);
  // each A staging mode is its own kernel instantiation, so that the common shapes keep
  // the simplest producer (a run-time branch alone cost the SDXL-1024 conv 7%)
  return amode == 0 ? dispatch<true, false>(bn, tf, ts, tw, g, s)
         : amode == 1 ? dispatch<true, false, 1>(bn, tf, ts, tw, g, s)
                      : dispatch<true, false, 2>(bn, tf, ts, tw, g, s);
}

}  // namespace dpp
