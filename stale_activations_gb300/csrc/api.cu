// C ABI of the displaced-patch layer library: argument checks, workspace layout
// and the composition of one layer step ("DistriFusion", How It Works: the
// first step synchronous, later steps on the previous step's activations;
// "OTIL for SDXL on 4x L40S", Periodic layer-context refresh: counter 0 puts
// GroupNorm, the patched conv and the patched attention on their synchronous
// branch).  Every step of the path runs in this library's kernels.
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "groupnorm.cuh"
#include "otil.cuh"
#include "refresh.cuh"
#include "simt.cuh"
#include "tc.cuh"

namespace dpp_host {

long long wait_limit_from_env() {
  const char* s = getenv("DPP_DEBUG_WAIT_LIMIT");
  if (!s || !*s) return dpp::kDefaultWaitLimit;
  long long v = atoll(s);
  return v < 0 ? dpp::kDefaultWaitLimit : v;
}

int skip_load_from_env(const char* kind) {
  const char* s = getenv("DPP_DEBUG_SKIP_LOAD");
  if (!s || !*s) return -1;
  const size_t n = strlen(kind);
  if (strncmp(s, kind, n) != 0 || s[n] != ':') return -1;
  const int v = atoi(s + n + 1);
  return v < 0 ? -1 : v;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return dpp::kNumSMs;
  std::lock_guard<std::mutex> g(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = dpp::kNumSMs;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace dpp_host

namespace {

using dpp_host::aligned16;

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
size_t esize(int dtype) { return dtype == DPP_BF16 ? 2 : 4; }
long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

int check_dtype(int dtype) {
  return (dtype == DPP_F32 || dtype == DPP_BF16) ? DPP_OK : DPP_ERR_DTYPE;
}

int check_conv(int B, int H, int W, int Cin, int Cout, int P, int dtype) {
  if (B <= 0 || H <= 0 || W <= 0 || Cin <= 0 || Cout <= 0 || P <= 0) return DPP_ERR_SHAPE;
  if (H % P) return DPP_ERR_SHAPE;
  if ((long long)B * H * W * (long long)(Cin > Cout ? Cin : Cout) >= (1ll << 40)) return DPP_ERR_SHAPE;
  if (dtype == DPP_BF16 && !dpp::tc_conv_supported(B, H, W, Cin, Cout, P)) return DPP_ERR_SHAPE;
  return DPP_OK;
}

int check_attn(int B, int L, int heads, int head_dim, int P, int dtype) {
  if (B <= 0 || L <= 0 || heads <= 0 || P <= 0) return DPP_ERR_SHAPE;
  if (head_dim != 64) return DPP_ERR_SHAPE;
  if (L % P || (L / P) % 8) return DPP_ERR_SHAPE;
  if ((long long)B * L * heads * 64 >= (1ll << 40)) return DPP_ERR_SHAPE;
  // the tensor-core kernel numbers its (unit, key tile) steps with 32-bit integers
  const long long units = (long long)B * heads * P * (((L / P + 127) / 128 + 1) / 2);
  if (dtype == DPP_BF16 && units * ((L + 127) / 128) >= (1ll << 31)) return DPP_ERR_SHAPE;
  return DPP_OK;
}

int check_layer(const dpp_layer_params* p) {
  if (!p) return DPP_ERR_NULL;
  int rc = check_dtype(p->dtype);
  if (rc) return rc;
  if (p->B <= 0 || p->H <= 0 || p->W <= 0 || p->C <= 0 || p->P <= 0 || p->G <= 0 ||
      p->heads <= 0)
    return DPP_ERR_SHAPE;
  if (p->C % p->G || p->C != p->heads * p->head_dim) return DPP_ERR_SHAPE;
  const int vec = p->dtype == DPP_BF16 ? 8 : 4;
  if (p->C % vec || p->C / vec > 256) return DPP_ERR_SHAPE;
  if (p->refresh != 0 && p->refresh != 1) return DPP_ERR_ARG;
  if (p->gn_mode < DPP_GN_SPLICED || p->gn_mode > DPP_GN_PREVIOUS) return DPP_ERR_ARG;
  if (p->fuse_gn != 0 && !(p->fuse_gn == 1 && p->dtype == DPP_BF16)) return DPP_ERR_ARG;
  if (p->fuse_gn && !dpp::tc_conv_gn_supported(p->H, p->W, p->P)) return DPP_ERR_SHAPE;
  if (p->fuse_refresh != 0 &&
      !(p->fuse_refresh == 1 && p->dtype == DPP_BF16 && p->C % 128 == 0))
    return DPP_ERR_ARG;
  if (!(p->eps >= 0.f)) return DPP_ERR_ARG;
  rc = check_conv(p->B, p->H, p->W, p->C, p->C, p->P, p->dtype);
  if (rc) return rc;
  rc = check_attn(p->B, p->H * p->W, p->heads, p->head_dim, p->P, p->dtype);
  if (rc) return rc;
  if (p->dtype == DPP_BF16 && !dpp::tc_linear_supported((long long)p->B * p->H * p->W, p->C))
    return DPP_ERR_SHAPE;
  return DPP_OK;
}

int layout(const dpp_layer_params* p, dpp_workspace_layout* o) {
  int rc = check_layer(p);
  if (rc) return rc;
  const dpp::GnDims g = dpp::make_gn_dims(p->B, p->H, p->W, p->C, p->P, p->G);
  const size_t act = (size_t)p->B * p->H * p->W * p->C * esize(p->dtype);
  size_t off = 0;
  o->status = off; off = align256(off + 256);
  o->gn_partial = off; off = align256(off + dpp::gn_partial_bytes(g));
  o->gn_fresh = off; off = align256(off + (size_t)p->B * p->P * p->G * 2 * sizeof(float));
  // per-channel GroupNorm parameters the conv applies to its input tiles (fuse_gn)
  o->gn_params = off;
  off = align256(off + (p->fuse_gn ? (size_t)p->B * p->P * 3 * p->C * sizeof(float) : 0));
  o->y = off; off = align256(off + act);
  o->h = off; off = align256(off + act);
  o->q = off; off = align256(off + act);
  o->k = off; off = align256(off + act);
  o->v = off; off = align256(off + act);
  o->o = off; off = align256(off + act);
  // the attention's scratch: the per-(batch, head) range of V and the partial results of
  // the split schedule (a region of its own, so that every stage's output stays
  // readable after the step)
  const size_t part = p->dtype == DPP_BF16 ? dpp::tc_attention_scratch_bytes(
                                                 p->B, p->H * p->W, p->heads, p->P, true)
                                           : 0;
  o->attn_partial = off; off = align256(off + part);
  o->attn_partial_bytes = part;
  o->total = off;
  return DPP_OK;
}

int run_conv(const void* yf, const void* ys, const void* w, void* out, int B, int H, int W,
             int Cin, int Cout, int P, int dtype, const float* gn_par, int* st, cudaStream_t s,
             const void* vstale = nullptr, unsigned* vmax = nullptr, int heads = 0) {
  if (dtype == DPP_BF16)
    return dpp::launch_tc_conv(yf, ys, w, out, B, H, W, Cin, Cout, P, gn_par, st,
                               dpp_host::wait_limit_from_env(), s, vstale, Cout, vmax, heads);
  return dpp::launch_simt_conv(yf, ys, w, out, B, H, W, Cin, Cout, P, dtype, s);
}

int run_linear(const void* a, const void* w, void* o0, void* o1, void* o2, long long M, int N,
               int K, int dtype, int* st, cudaStream_t s, unsigned* vmax = nullptr,
               int vmax_L = 0, int vmax_heads = 0) {
  if (dtype == DPP_BF16)
    return dpp::launch_tc_linear(a, w, o0, o1, o2, M, N, K, st, dpp_host::wait_limit_from_env(),
                                 s, vmax, vmax_L, vmax_heads);
  dpp::SimtOut o{};
  o.ptr[0] = o0; o.ptr[1] = o1; o.ptr[2] = o2;
  o.ncols = o1 ? N / 3 : N;
  return dpp::launch_simt_linear(a, w, o, M, N, K, dtype, s);
}

int run_attention(const void* q, const void* kf, const void* vf, const void* ks, const void* vs,
                  void* o, int B, int L, int heads, int P, int dtype, bool split, void* scratch,
                  size_t scratch_bytes, bool scratch_zeroed, int* st, cudaStream_t s,
                  bool vmax_ready = false) {
  if (dtype == DPP_BF16)
    return dpp::launch_tc_attention(q, kf, vf, ks, vs, o, B, L, heads, P, split, scratch,
                                    scratch_bytes, scratch_zeroed, vmax_ready, st,
                                    dpp_host::wait_limit_from_env(),
                                    dpp_host::skip_load_from_env("attn"), s);
  return dpp::launch_simt_attention(q, kf, vf, ks, vs, o, B, L, heads, P, dtype, s);
}

int refresh_segments(dpp::RefreshSeg* segs, int nseg, int dtype, cudaStream_t s) {
  for (int i0 = 0; i0 < nseg; i0 += dpp::kMaxRefreshSegs) {
    dpp::RefreshTable tab{};
    tab.nseg = nseg - i0 < dpp::kMaxRefreshSegs ? nseg - i0 : dpp::kMaxRefreshSegs;
    tab.blk_start[0] = 0;
    for (int j = 0; j < tab.nseg; ++j) {
      tab.seg[j] = segs[i0 + j];
      tab.blk_start[j + 1] = tab.blk_start[j] + cdiv(tab.seg[j].n, 128);
    }
    int rc = dpp::launch_refresh(tab, dtype, s);
    if (rc) return rc;
  }
  return DPP_OK;
}

}  // namespace

#ifdef DPP_DEBUG_BOUNDS
namespace dpp {  // each kernel file's index-check record (DPP_BOUNDS_READER)
int bounds_groupnorm(long long* rec, int reset);
int bounds_refresh(long long* rec, int reset);
int bounds_tc_gemm(long long* rec, int reset);
int bounds_tc_attn(long long* rec, int reset);
int bounds_simt(long long* rec, int reset);
int bounds_otil(long long* rec, int reset);
}  // namespace dpp
#endif

extern "C" {

const char* dpp_status_string(int status) {
  switch (status) {
    case DPP_OK: return "ok";
    case DPP_ERR_NULL: return "null pointer";
    case DPP_ERR_SHAPE: return "unsupported or invalid shape";
    case DPP_ERR_ALIGN: return "misaligned pointer";
    case DPP_ERR_DTYPE: return "invalid dtype";
    case DPP_ERR_CUDA: return "CUDA error";
    case DPP_ERR_TIMEOUT: return "device wait gave up (timeout)";
    case DPP_ERR_BOUNDS: return "device index check failed";
    case DPP_ERR_UNSUPPORTED: return "unsupported combination";
    case DPP_ERR_ARG: return "invalid argument";
    case DPP_ERR_SCRATCH_LIMIT: return "layer workspace exceeds the fixed no-alloc scratch";
    default: return "unknown status";
  }
}

int dpp_version(void) { return 200; }

int refresh_residual(const void* fresh, void* stale, int8_t* codes, float* scales, int64_t n,
                     int dtype, void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  if (n < 0) return DPP_ERR_SHAPE;
  if (n == 0) return DPP_OK;
  if (!fresh || !stale || !codes || !scales) return DPP_ERR_NULL;
  if (!aligned16(fresh) || !aligned16(stale) || !aligned16(codes) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u))
    return DPP_ERR_ALIGN;
  dpp::RefreshSeg sg{fresh, stale, codes, scales, (long long)n, 1, 0, stale};
  return refresh_segments(&sg, 1, dtype, static_cast<cudaStream_t>(stream));
}

int apply_residual(const int8_t* codes, const float* scales, void* stale, int64_t n, int dtype,
                   void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  if (n < 0) return DPP_ERR_SHAPE;
  if (n == 0) return DPP_OK;
  if (!codes || !scales || !stale) return DPP_ERR_NULL;
  if (!aligned16(codes) || !aligned16(stale) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return DPP_ERR_ALIGN;
  dpp::ApplyTable tab{};
  tab.nseg = 1;
  tab.seg[0] = dpp::ApplySeg{codes, scales, stale, (long long)n, 1, 0};
  tab.blk_start[1] = cdiv(n, 128);
  return dpp::launch_apply(tab, dtype, static_cast<cudaStream_t>(stream));
}

int halo_conv3x3(const void* y_fresh, const void* y_stale, const void* w, void* out, int B, int H,
                 int W, int Cin, int Cout, int P, int dtype, int* dev_status, void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  if (!y_fresh || !y_stale || !w || !out) return DPP_ERR_NULL;
  rc = check_conv(B, H, W, Cin, Cout, P, dtype);
  if (rc) return rc;
  if (!aligned16(y_fresh) || !aligned16(y_stale) || !aligned16(w) || !aligned16(out))
    return DPP_ERR_ALIGN;
  return run_conv(y_fresh, y_stale, w, out, B, H, W, Cin, Cout, P, dtype, nullptr, dev_status,
                  static_cast<cudaStream_t>(stream));
}

size_t dpp_attention_scratch_size(int B, int L, int heads, int head_dim, int P, int dtype,
                                  int split) {
  if (check_dtype(dtype) || check_attn(B, L, heads, head_dim, P, dtype)) return 0;
  return dtype == DPP_BF16 ? dpp::tc_attention_scratch_bytes(B, L, heads, P, split != 0) : 0;
}

static int attention_call(const void* q, const void* k_fresh, const void* v_fresh,
                          const void* k_stale, const void* v_stale, void* o, int B, int L,
                          int heads, int head_dim, int P, int dtype, bool split, void* scratch,
                          size_t scratch_bytes, int* dev_status, void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  if (!q || !k_fresh || !v_fresh || !k_stale || !v_stale || !o) return DPP_ERR_NULL;
  rc = check_attn(B, L, heads, head_dim, P, dtype);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k_fresh) || !aligned16(v_fresh) || !aligned16(k_stale) ||
      !aligned16(v_stale) || !aligned16(o) || (scratch && !aligned16(scratch)))
    return DPP_ERR_ALIGN;
  const size_t need = dpp_attention_scratch_size(B, L, heads, head_dim, P, dtype, split);
  if (need && (!scratch || scratch_bytes < need)) return DPP_ERR_ARG;
  return run_attention(q, k_fresh, v_fresh, k_stale, v_stale, o, B, L, heads, P, dtype, split,
                       scratch, scratch_bytes, false, dev_status,
                       static_cast<cudaStream_t>(stream));
}

int stale_kv_attention(const void* q, const void* k_fresh, const void* v_fresh,
                       const void* k_stale, const void* v_stale, void* o, int B, int L, int heads,
                       int head_dim, int P, int dtype, void* scratch, size_t scratch_bytes,
                       int* dev_status, void* stream) {
  return attention_call(q, k_fresh, v_fresh, k_stale, v_stale, o, B, L, heads, head_dim, P, dtype,
                        false, scratch, scratch_bytes, dev_status, stream);
}

int stale_kv_attention_split(const void* q, const void* k_fresh, const void* v_fresh,
                             const void* k_stale, const void* v_stale, void* o, int B, int L,
                             int heads, int head_dim, int P, int dtype, void* scratch,
                             size_t scratch_bytes, int* dev_status, void* stream) {
  return attention_call(q, k_fresh, v_fresh, k_stale, v_stale, o, B, L, heads, head_dim, P, dtype,
                        true, scratch, scratch_bytes, dev_status, stream);
}

int dpp_workspace_query(const dpp_layer_params* prm, dpp_workspace_layout* out) {
  if (!out) return DPP_ERR_NULL;
  return layout(prm, out);
}

size_t dpp_workspace_size(const dpp_layer_params* prm) {
  dpp_workspace_layout l;
  return layout(prm, &l) == DPP_OK ? l.total : 0;
}

int64_t dpp_message_elems(const dpp_layer_params* p) {
  if (check_layer(p)) return -1;
  const long long blc = (long long)p->B * p->H * p->W * p->C;
  return 2 * blc + (long long)p->B * (p->P - 1) * 2 * p->W * p->C;
}

int64_t dpp_message_blocks(const dpp_layer_params* p) {
  if (check_layer(p)) return -1;
  const long long blc = (long long)p->B * p->H * p->W * p->C;
  return 2 * cdiv(blc, 128) + (long long)p->B * (p->P - 1) * cdiv(2ll * p->W * p->C, 128);
}

int dpp_layer_kernel_count(const dpp_layer_params* p, int mode) {
  if (check_layer(p)) return -1;
  int n = 2 /* gn */ + 1 /* conv */ + 1 /* qkv */ + 1 /* attention */ + 1 /* out proj */;
  // the attention's separate max |V| pass, when the GroupNorm and projection kernels do
  // not take it on the way (fuse_gn; fuse_refresh with a second state set)
  if (p->dtype == DPP_BF16 && (p->fuse_gn || p->fuse_refresh)) n += 1;
  if (mode == DPP_STALE && p->refresh) {
    // a launch per full table of segments, and always a last one (it also copies
    // the GroupNorm sums)
    const long long nseg = 2 + (long long)p->B * (p->P - 1);
    n += (int)(nseg / dpp::kMaxRefreshSegs) + 1;
  }
  return n;
}

int patch_layer_step(const dpp_layer_params* prm, const dpp_layer_weights* wts,
                     const dpp_layer_state* st, const void* x, void* out, int mode,
                     void* workspace, void* stream) {
  return patch_layer_step_timed(prm, wts, st, x, out, mode, workspace, stream, nullptr);
}

int patch_layer_step_timed(const dpp_layer_params* prm, const dpp_layer_weights* wts,
                           const dpp_layer_state* st, const void* x, void* out, int mode,
                           void* workspace, void* stream, void* const* stage_events) {
  if (!prm || !wts || !st || !x || !out || !workspace) return DPP_ERR_NULL;
  if (mode != DPP_SYNC && mode != DPP_STALE) return DPP_ERR_ARG;
  dpp_workspace_layout lo;
  int rc = layout(prm, &lo);
  if (rc) return rc;
  const dpp_layer_params& p = *prm;
  if (!wts->gamma || !wts->beta || !wts->w_conv || !wts->w_qkv || !wts->w_o) return DPP_ERR_NULL;
  if (!st->gn_stats || !st->y_stale || !st->k_stale || !st->v_stale) return DPP_ERR_NULL;
  const bool refresh = mode == DPP_STALE && p.refresh;
  if (refresh && (!st->codes || !st->scales)) return DPP_ERR_NULL;
  // the second state set: all four buffers or none, none equal to its counterpart
  const int nnext = (st->gn_next != nullptr) + (st->y_next != nullptr) +
                    (st->k_next != nullptr) + (st->v_next != nullptr);
  if (nnext != 0 && nnext != 4) return DPP_ERR_NULL;
  const bool dbuf = nnext == 4;
  if (dbuf && (st->gn_next == st->gn_stats || st->y_next == st->y_stale ||
               st->k_next == st->k_stale || st->v_next == st->v_stale))
    return DPP_ERR_ARG;
  if (dbuf && (!aligned16(st->y_next) || !aligned16(st->k_next) || !aligned16(st->v_next) ||
               (reinterpret_cast<uintptr_t>(st->gn_next) & 3u)))
    return DPP_ERR_ALIGN;
  // where the new state goes
  float* const gn_dst = dbuf ? st->gn_next : st->gn_stats;
  void* const y_dst = dbuf ? st->y_next : st->y_stale;
  void* const k_dst = dbuf ? st->k_next : st->k_stale;
  void* const v_dst = dbuf ? st->v_next : st->v_stale;
  // with a second set and fuse_refresh (bf16, whole 128-element blocks per K/V row), the
  // K/V refresh runs in the projection's epilogue
  const bool fuse_rfx = refresh && dbuf && p.fuse_refresh;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return DPP_ERR_ALIGN;
  if (!aligned16(x) || !aligned16(out) || !aligned16(wts->w_conv) || !aligned16(wts->w_qkv) ||
      !aligned16(wts->w_o) || !aligned16(st->y_stale) || !aligned16(st->k_stale) ||
      !aligned16(st->v_stale) || (refresh && !aligned16(st->codes)) ||
      (reinterpret_cast<uintptr_t>(wts->gamma) & 3u) ||
      (reinterpret_cast<uintptr_t>(wts->beta) & 3u) ||
      (reinterpret_cast<uintptr_t>(st->gn_stats) & 3u) ||
      (refresh && (reinterpret_cast<uintptr_t>(st->scales) & 3u)))
    return DPP_ERR_ALIGN;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + lo.status);
  float* gn_partial = reinterpret_cast<float*>(ws + lo.gn_partial);
  float* gn_fresh = reinterpret_cast<float*>(ws + lo.gn_fresh);
  void* y = ws + lo.y;
  void* h = ws + lo.h;
  void* q = ws + lo.q;
  void* k = ws + lo.k;
  void* v = ws + lo.v;
  void* o = ws + lo.o;
  const bool sync = mode == DPP_SYNC;
  const int L = p.H * p.W;
  const long long M = (long long)p.B * L;

  auto mark = [&](int i) -> int {
    if (!stage_events || !stage_events[i]) return DPP_OK;
    return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s) == cudaSuccess
               ? DPP_OK
               : DPP_ERR_CUDA;
  };
  // state geometry and the compressed refresh (a7/a8) of the segments in message order:
  // K, V (with_kv), then each batch's P-1 halo ranges of y, packed into fixed-size
  // tables and launched whenever a table fills up; the last launch also copies the fresh
  // GroupNorm sums.  Every launch runs alongside the kernel before it, which must touch
  // none of its buffers (the table's `early`).
  const size_t es = esize(p.dtype);
  const size_t act = (size_t)M * p.C * es;
  const size_t gn_bytes = (size_t)p.B * p.P * p.G * 2 * sizeof(float);
  const size_t halo_bytes = 2ull * p.W * p.C * es;            // rows r-1 and r
  const size_t band_bytes = (size_t)(p.H / p.P) * p.W * p.C * es;
  const size_t img_bytes = (size_t)p.H * p.W * p.C * es;
  const long long blc = M * p.C;
  auto refresh_state = [&](bool with_kv) -> int {
    dpp::RefreshTable tab{};
    tab.early = 1;
    long long coff = with_kv ? 0 : 2 * blc, soff = with_kv ? 0 : 2 * cdiv(blc, 128);
    auto add = [&](const void* fr, void* stl, void* outp, long long n) -> int {
      const bool ok = aligned16(fr) && aligned16(stl) && aligned16(outp) &&
                      aligned16(st->codes + coff);
      tab.seg[tab.nseg] = dpp::RefreshSeg{fr, stl, st->codes + coff, st->scales + soff, n,
                                          ok ? 1 : 0, 0, outp};
      tab.blk_start[tab.nseg + 1] = tab.blk_start[tab.nseg] + cdiv(n, 128);
      ++tab.nseg;
      coff += n;
      soff += cdiv(n, 128);
      if (tab.nseg == dpp::kMaxRefreshSegs) {
        const int r = dpp::launch_refresh(tab, p.dtype, s);
        tab.nseg = 0;
        tab.blk_start[0] = 0;
        return r;
      }
      return DPP_OK;
    };
    int r = DPP_OK;
    if (with_kv &&
        ((r = add(k, st->k_stale, k_dst, blc)) || (r = add(v, st->v_stale, v_dst, blc))))
      return r;
    for (int b = 0; b < p.B; ++b)
      for (int pp = 1; pp < p.P; ++pp) {
        const size_t off = b * img_bytes + pp * band_bytes - halo_bytes / 2;
        r = add(static_cast<char*>(y) + off, static_cast<char*>(st->y_stale) + off,
                static_cast<char*>(y_dst) + off, 2ll * p.W * p.C);
        if (r) return r;
      }
    tab.copy_n = (int)(gn_bytes / sizeof(float));
    tab.copy_src = gn_fresh;
    tab.copy_dst = gn_dst;
    return dpp::launch_refresh(tab, p.dtype, s);
  };

  if ((rc = mark(0))) return rc;
  // a1 + a2: fresh sums of every patch, spliced GroupNorm
  const dpp::GnDims g = dpp::make_gn_dims(p.B, p.H, p.W, p.C, p.P, p.G);
  // the first kernel also zeroes the status word and the start of the attention's scratch
  // (its V maxima and piece counters)
  const int ncnt = p.dtype == DPP_BF16 ? dpp::tc_attention_zero_ints(p.B, L, p.heads, p.P, true)
                                        : 0;
  // fuse_gn: the apply writes only the rows other bands read as halos (and the state
  // update reads), plus the per-channel parameters; the conv normalises its own band's
  // rows of x as its tiles land in shared memory
  const bool fused = p.fuse_gn != 0;
  float* gn_params = fused ? reinterpret_cast<float*>(ws + lo.gn_params) : nullptr;
  // The attention's V scaling needs max |V| per (batch, head) of the V it reads: on the
  // plain bf16 path the Q/K/V projection's epilogue takes it over the fresh V, and over
  // the stale V (a stale step with P > 1) the conv when each CTA's share is at most 256
  // rows (CTAs of their own on the SMs its tiles leave idle, else its epilogue warps while
  // the first accumulator fills), or else the GroupNorm apply -- not a separate pass.
  const bool vmax_fold = p.dtype == DPP_BF16 && !fused && !fuse_rfx;
  const bool vs_need = vmax_fold && !sync && p.P > 1;
  const bool vs_in_conv = vs_need && M <= 256ll * dpp_host::sm_count();
  unsigned* vmax = reinterpret_cast<unsigned*>(ws + lo.attn_partial);
  rc = dpp::launch_gn(x, y, gn_partial, sync ? nullptr : st->gn_stats, gn_fresh, wts->gamma,
                      wts->beta, g, p.eps, sync ? DPP_GN_SYNC : p.gn_mode, p.dtype, status,
                      reinterpret_cast<int*>(ws + lo.attn_partial), ncnt, gn_params,
                      fused ? 1 : 0, vs_need && !vs_in_conv ? st->v_stale : nullptr, vmax,
                      p.heads, s);
  if (rc || (rc = mark(1))) return rc;
  // a3: halo conv, halo rows from the stale conv input (fresh at the synchronous step)
  rc = run_conv(fused ? x : y, sync ? y : st->y_stale, wts->w_conv, h, p.B, p.H, p.W, p.C, p.C,
                p.P, p.dtype, gn_params, status, s,
                vs_in_conv ? st->v_stale : nullptr, vmax, p.heads);
  if (rc || (rc = mark(2))) return rc;
  // a7 for the halo rows of y and a8, when the projection refreshes K and V: it runs
  // alongside the conv's end (it writes only the second state set and the message's
  // halo part; the conv reads the stale y, which it leaves unchanged)
  if (fuse_rfx && (rc = refresh_state(false))) return rc;
  // a4: Q, K, V projections (one GEMM over the packed [3C, C] weight); with fuse_rfx its
  // epilogue also refreshes K and V into the second state set (a7)
  if (fuse_rfx)
    rc = dpp::launch_tc_linear_refresh(h, wts->w_qkv, q, k, v, M, 3 * p.C, p.C, st->k_stale,
                                       st->v_stale, k_dst, v_dst, st->codes, st->scales, status,
                                       dpp_host::wait_limit_from_env(), s);
  else
    rc = run_linear(h, wts->w_qkv, q, k, v, M, 3 * p.C, p.C, p.dtype, status, s,
                    vmax_fold ? vmax : nullptr, L, p.heads);
  if (rc || (rc = mark(3))) return rc;
  // a5: stale-KV attention
  rc = run_attention(q, k, v, sync ? k : st->k_stale, sync ? v : st->v_stale, o, p.B, L, p.heads,
                     p.P, p.dtype, true, ws + lo.attn_partial, lo.attn_partial_bytes,
                     true /* zeroed by gn_stats */, status, s, vmax_fold);
  if (rc || (rc = mark(4))) return rc;
  // a6: output projection
  rc = run_linear(o, wts->w_o, out, nullptr, nullptr, M, p.C, p.C, p.dtype, status, s);
  if (rc || (rc = mark(5))) return rc;

  // a7/a8: state update, after every virtual rank has read the old state
  if (sync) {
    DPP_CUDA_CHECK(cudaMemcpyAsync(k_dst, k, act, cudaMemcpyDeviceToDevice, s));
    DPP_CUDA_CHECK(cudaMemcpyAsync(v_dst, v, act, cudaMemcpyDeviceToDevice, s));
    DPP_CUDA_CHECK(cudaMemcpyAsync(gn_dst, gn_fresh, gn_bytes, cudaMemcpyDeviceToDevice, s));
    if (p.P > 1) {
      for (int b = 0; b < p.B; ++b) {
        const size_t off = b * img_bytes + band_bytes - halo_bytes / 2;  // row Hp-1 of batch b
        DPP_CUDA_CHECK(cudaMemcpy2DAsync(static_cast<char*>(y_dst) + off, band_bytes,
                                         static_cast<char*>(y) + off, band_bytes, halo_bytes,
                                         p.P - 1, cudaMemcpyDeviceToDevice, s));
      }
    }
    return mark(6);
  }
  if (!refresh || fuse_rfx) return mark(6);
  // The refresh runs alongside the output projection, which touches none of its
  // buffers; the kernels that read the old state (conv, attention) and wrote the fresh
  // K, V, y had all completed before the projection passed its own dependency wait.
  if ((rc = refresh_state(true))) return rc;
  return mark(6);
}

int dpp_apply_layer_message(const dpp_layer_params* prm, const int8_t* codes,
                            const float* scales, const float* gn_sums,
                            const dpp_layer_state* copy, void* stream) {
  int rc = check_layer(prm);
  if (rc) return rc;
  if (!codes || !scales || !gn_sums || !copy || !copy->gn_stats || !copy->y_stale ||
      !copy->k_stale || !copy->v_stale)
    return DPP_ERR_NULL;
  const dpp_layer_params& p = *prm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = esize(p.dtype);
  const long long blc = (long long)p.B * p.H * p.W * p.C;
  const size_t halo_bytes = 2ull * p.W * p.C * es;
  const size_t band_bytes = (size_t)(p.H / p.P) * p.W * p.C * es;
  const size_t img_bytes = (size_t)p.H * p.W * p.C * es;
  dpp::ApplyTable tab{};
  long long coff = 0, soff = 0;
  auto add = [&](void* stl, long long n) -> int {
    const bool ok = aligned16(stl) && aligned16(codes + coff);
    tab.seg[tab.nseg] = dpp::ApplySeg{codes + coff, scales + soff, stl, n, ok ? 1 : 0, 0};
    tab.blk_start[tab.nseg + 1] = tab.blk_start[tab.nseg] + cdiv(n, 128);
    ++tab.nseg;
    coff += n;
    soff += cdiv(n, 128);
    if (tab.nseg == dpp::kMaxRefreshSegs) {
      const int r = dpp::launch_apply(tab, p.dtype, s);
      tab.nseg = 0;
      return r;
    }
    return DPP_OK;
  };
  if ((rc = add(copy->k_stale, blc)) || (rc = add(copy->v_stale, blc))) return rc;
  for (int b = 0; b < p.B; ++b)
    for (int pp = 1; pp < p.P; ++pp) {
      const size_t off = b * img_bytes + pp * band_bytes - halo_bytes / 2;
      if ((rc = add(static_cast<char*>(copy->y_stale) + off, 2ll * p.W * p.C))) return rc;
    }
  // the last launch also copies the GroupNorm sums
  tab.copy_n = p.B * p.P * p.G * 2;
  tab.copy_src = gn_sums;
  tab.copy_dst = copy->gn_stats;
  return dpp::launch_apply(tab, p.dtype, s);
}

int dpp_otil_blocks(const dpp_otil_params* prm) { return dpp::otil_blocks(prm); }

int dpp_otil_step(const dpp_otil_params* prm, const void* fresh, void* views, uint8_t* visited,
                  int32_t* sel, void* msg, void* stream) {
  const int rc = dpp::otil_check(prm);
  if (rc) return rc;
  if (!fresh || !views || !visited || !sel || !msg) return DPP_ERR_NULL;
  const size_t es = esize(prm->dtype);
  if (reinterpret_cast<uintptr_t>(fresh) % es || reinterpret_cast<uintptr_t>(views) % es ||
      reinterpret_cast<uintptr_t>(msg) % es || reinterpret_cast<uintptr_t>(sel) % 4)
    return DPP_ERR_ALIGN;
  return dpp::launch_otil_step(*prm, fresh, views, visited, sel, msg,
                               static_cast<cudaStream_t>(stream));
}

int dpp_otil_finalize(const dpp_otil_params* prm, const void* fresh, void* views,
                      uint8_t* visited, int reset, void* stream) {
  const int rc = dpp::otil_check(prm);
  if (rc) return rc;
  if (!fresh || !views || !visited) return DPP_ERR_NULL;
  const size_t es = esize(prm->dtype);
  if (reinterpret_cast<uintptr_t>(fresh) % es || reinterpret_cast<uintptr_t>(views) % es)
    return DPP_ERR_ALIGN;
  return dpp::launch_otil_finalize(*prm, fresh, views, visited, reset ? 1 : 0,
                                   static_cast<cudaStream_t>(stream));
}

int dpp_read_device_status(const void* workspace, void* stream) {
  if (!workspace) return DPP_ERR_NULL;
  int v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DPP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DPP_ERR_CUDA;
  return v;
}

int dpp_debug_bounds(long long* rec, int reset) {
  if (!rec) return DPP_ERR_NULL;
  for (int i = 0; i < 4; ++i) rec[i] = 0;
#ifdef DPP_DEBUG_BOUNDS
  if (cudaDeviceSynchronize() != cudaSuccess) return DPP_ERR_CUDA;
  // the record of each translation unit that holds kernels, in the order the header lists
  int (*const readers[])(long long*, int) = {dpp::bounds_groupnorm, dpp::bounds_refresh,
                                             dpp::bounds_tc_gemm,   dpp::bounds_tc_attn,
                                             dpp::bounds_simt,      dpp::bounds_otil};
  int rc = DPP_OK;
  for (int f = 0; f < 6; ++f) {
    long long r[3];
    const int e = readers[f](r, reset);
    if (e) return e;
    if (r[0] && rc == DPP_OK) {
      rec[0] = f + 1;
      rec[1] = r[0];
      rec[2] = r[1];
      rec[3] = r[2];
      rc = DPP_ERR_BOUNDS;
    }
  }
  return rc;
#else
  (void)reset;
  return DPP_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
