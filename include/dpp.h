/*
 * dpp.h -- C ABI of the displaced-patch-parallel layer library for GB300 (sm_103a).
 *
 * One denoising-step layer pass of DistriFusion-style displaced patch
 * parallelism, with the P "ranks" emulated on one GPU: the feature map is cut
 * into P row patches; each patch computes on its fresh activations spliced into
 * stale full-size buffers left by the previous step, and a refresh kernel writes
 * the fresh activations back as a compressed residual.
 *   - "DistriFusion" project summary, How It Works: synchronous first step,
 *     then asynchronous reuse of the previous step's activations.
 *   - "OTIL for SDXL on 4x L40S", What is implemented where (Periodic layer-
 *     context refresh; GroupNorm sync without the rest) and "Read this before
 *     interpreting the numbers", item 3: the stale state is the conv halo rows,
 *     the cross-slice attention K/V and the two GroupNorm scalars per group.
 *   - "A way to reduce bandwidth requirement for xDiT" (raylight issue): send
 *     only the compressed residual, the real change.
 *   - "Benchmarking DistVAE", Glossary: halo rows, row bands (patchify).
 *
 * Conventions for every call
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise; the
 *     library allocates nothing, frees nothing and keeps no global state.
 *   - Layout: NHWC == [B, L = H*W, C], row-major, contiguous.  Head h owns
 *     channels [h*head_dim, (h+1)*head_dim).  Row patch p owns image rows
 *     [p*H/P, (p+1)*H/P), i.e. the contiguous tokens [p*L/P, (p+1)*L/P).
 *   - dtype: DPP_F32 (fp32 storage, fp32 SIMT arithmetic) or DPP_BF16 (bf16
 *     storage, tcgen05 tensor cores with fp32 accumulation).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; they return before it finishes.
 *   - Return value: DPP_OK or an error code.  Argument errors are found on the
 *     host before anything is launched.  Pointers must be 16-byte aligned
 *     (128-bit accesses and TMA need it) unless stated otherwise.
 *   - Device-side give-ups: every wait inside a kernel is bounded; a kernel
 *     that gives up stores DPP_ERR_TIMEOUT into the device status word (if the
 *     word is already 0) and returns early, leaving its output incomplete.
 *     The environment variable DPP_DEBUG_WAIT_LIMIT (read at each call)
 *     overrides the wait bound; 0 makes every such wait give up at once.
 *   - DPP_DEBUG_SKIP_LOAD=<kind>:<i> (read at each call; kind attn, conv or linear):
 *     every CTA of the attention kernel, of the conv's GEMM or of the projections'
 *     GEMM leaves its i-th K/V tile or K slice unloaded, so its bounded waits give up
 *     and the device status becomes DPP_ERR_TIMEOUT.  For tests of that path; unset in
 *     normal use.
 */
#ifndef DPP_H_
#define DPP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define DPP_OK 0
#define DPP_ERR_NULL 1        /* a required pointer is NULL */
#define DPP_ERR_SHAPE 2       /* a size is out of range or not a supported multiple */
#define DPP_ERR_ALIGN 3       /* a pointer is not aligned as required */
#define DPP_ERR_DTYPE 4       /* dtype is neither DPP_F32 nor DPP_BF16 */
#define DPP_ERR_CUDA 5        /* a CUDA runtime/driver call failed */
#define DPP_ERR_TIMEOUT 6     /* device status: a bounded wait gave up */
#define DPP_ERR_BOUNDS 7      /* dpp_debug_bounds: a kernel of the index-checking build
                                 computed a global index outside its tensor's extent */
#define DPP_ERR_UNSUPPORTED 8 /* the combination is not implemented */
#define DPP_ERR_ARG 9         /* an enum/flag argument is invalid */
#define DPP_ERR_SCRATCH_LIMIT 10 /* the layer needs more workspace than the fixed
                                    scratch of patch_layer_step_noalloc */

#define DPP_F32 0
#define DPP_BF16 1

#define DPP_SYNC 0  /* warm-up / periodic refresh step: stale := fresh before use */
#define DPP_STALE 1 /* steady step: use the stale state as given */

/* Human-readable name of a status code (static string, never NULL). */
const char* dpp_status_string(int status);

/* Library ABI version (major*100 + minor). */
int dpp_version(void);

/*
 * refresh_residual -- compressed-residual refresh of a flat stale buffer, in place.
 * ("A way to reduce bandwidth requirement for xDiT": send the compressed
 * residual; the quantiser is block int8 with one fp32 scale per 128 elements.)
 *
 * For each block of 128 consecutive elements [128*j, min(128*j+128, n)):
 *   d_i = f32(fresh_i) - f32(stale_i);  a = max |d_i|;  s = a / 127 (IEEE);
 *   q_i = s == 0 ? 0 : clamp(rint(d_i / s), -127, 127)   (ties to even);
 *   stale_i = store(fmaf(q_i, s, f32(stale_i)))  with store = bf16 RNE or fp32;
 *   codes[i] = q_i;  scales[j] = s.
 * fresh, stale: [n] elements of `dtype`.  codes: [n] int8.  scales: [ceil(n/128)]
 * fp32 (4-byte alignment suffices).  n == 0 is a no-op.  Values must be finite.
 * The codes/scales pair is the message a rank would send; stale holds what every
 * receiver reconstructs.  Bit-exact across runs and against an IEEE CPU evaluation.
 */
int refresh_residual(const void* fresh, void* stale, int8_t* codes, float* scales,
                     int64_t n, int dtype, void* stream);

/*
 * apply_residual -- the receiver's half of refresh_residual: applies a message to a
 * copy of the stale buffer, in place.  ("A way to reduce bandwidth requirement for
 * xDiT": each receiver adds the dequantised residual to its own stale copy.)
 * For each element i of block j: stale_i = store(fmaf(codes[i], scales[j], f32(stale_i))),
 * the sender's last step exactly, so a copy that equalled the sender's stale buffer
 * before refresh_residual equals it bit for bit afterwards.  Layout, alignment and
 * n == 0 as in refresh_residual; codes/scales are read only.
 */
int apply_residual(const int8_t* codes, const float* scales, void* stale, int64_t n, int dtype,
                   void* stream);

/*
 * halo_conv3x3 -- 3x3 "same" convolution of each row band with stale halo rows.
 * ("Benchmarking DistVAE", Glossary: halo; "OTIL for SDXL on 4x L40S", item 3.)
 *
 * out[b,r,c,o] = sum_{i,j in {-1,0,1}} sum_k w[o,i+1,j+1,k] * yhat[b,r+i,c+j,k]
 * where, for r in band p = [r0, r1): yhat = y_fresh inside [r0, r1), y_stale
 * for rows r0-1 and r1, and 0 outside the image (rows < 0, >= H; cols < 0, >= W).
 * y_fresh, y_stale: [B,H,W,Cin]; w: [Cout,3,3,Cin]; out: [B,H,W,Cout]; all `dtype`.
 * With y_stale == y_fresh the result is the unbanded convolution.
 * Requires H % P == 0.  DPP_BF16 also requires Cin % 64 == 0, Cout a multiple of
 * 128 or of 160, W % 8 == 0 and H*W % 128 == 0.
 * dev_status: device int (may be NULL) that receives a give-up code.
 */
int halo_conv3x3(const void* y_fresh, const void* y_stale, const void* w, void* out,
                 int B, int H, int W, int Cin, int Cout, int P, int dtype,
                 int* dev_status, void* stream);

/*
 * stale_kv_attention -- per-patch attention of fresh queries over spliced K/V.
 * ("OTIL for SDXL on 4x L40S", item 3 and Periodic layer-context refresh: the
 * cross-slice attention K/V are stale; Self-tests: own slice fresh, never a blend.)
 *
 * For token t in patch p (tokens [p*L/P, (p+1)*L/P)) and head h:
 *   o[t,h] = sum_s softmax_s(q[t,h] . Khat_p[s,h] / sqrt(head_dim)) Vhat_p[s,h]
 * Khat_p[s] = k_fresh[s] for s in patch p, else k_stale[s]; same for Vhat.  All L
 * keys, no mask.  q, k_*, v_*, o: [B, L, heads*head_dim] of `dtype`.
 * Requires head_dim == 64, L % P == 0 and (L/P) % 8 == 0; for DPP_BF16 also
 * B*heads*P*ceil(L/P/256) * ceil(L/128) < 2^31 (the kernel's step counter).
 * Values must be finite.  DPP_BF16 numerics: fp32 scores and softmax, the
 * probabilities rounded to fp16 for the P.V product, V widened to fp16 after an exact
 * scaling by a power of two per (batch, head) chosen from max|V| over the fresh and
 * stale V (no scaling when max|V| lies in [2^-6, 2^15); otherwise the scaled maximum
 * lies in [2^14, 2^15)), so that any finite bf16 V keeps fp16's full precision
 * relative to its largest value (down to max|V| of about 2^-111).
 * scratch: caller-owned device buffer, 16-byte aligned, of at least
 * dpp_attention_scratch_size(..., split = 0) bytes for DPP_BF16 (it receives the
 * per-(batch, head) maxima of |V|; its contents are not used after the call); may be
 * NULL for DPP_F32, whose size is 0.  Returns DPP_ERR_ARG if it is missing or short.
 * dev_status: device int (may be NULL) that receives a give-up code.
 */
size_t dpp_attention_scratch_size(int B, int L, int heads, int head_dim, int P, int dtype,
                                  int split);
int stale_kv_attention(const void* q, const void* k_fresh, const void* v_fresh,
                       const void* k_stale, const void* v_stale, void* o,
                       int B, int L, int heads, int head_dim, int P, int dtype,
                       void* scratch, size_t scratch_bytes, int* dev_status, void* stream);

/*
 * stale_kv_attention_split -- the same operation and result (up to rounding) with
 * the load spread evenly over the SMs.  (The pages have no counterpart of this
 * call: it is a schedule of stale_kv_attention for this GPU, used by
 * patch_layer_step.)
 * The bf16 kernel works on units of 256 queries (two 128-row tiles of one batch,
 * head and patch) against all L keys, one CTA per SM.  stale_kv_attention gives
 * each CTA whole units, so when their number is not a multiple of the SM count
 * the last round leaves SMs idle.  Here those last units are cut into runs of
 * 128-key tiles shared evenly by all CTAs; each piece leaves a partial result
 * (O/l rounded to fp16, the running maximum m and sum l in fp32) in the scratch,
 * and whichever piece of a unit finishes last merges them all in a fixed order
 * (deterministic; the call zeroes the counters it uses for this at the start of the
 * buffer).  The merge reads O/l in fp16, whose rounding (2^-11 relative) stays well
 * below that of the bf16 output.
 * scratch: as for stale_kv_attention, of at least
 * dpp_attention_scratch_size(..., split = 1) bytes; that size depends on the current
 * device's SM count, so query it on the device that runs the call.
 */
int stale_kv_attention_split(const void* q, const void* k_fresh, const void* v_fresh,
                             const void* k_stale, const void* v_stale, void* o,
                             int B, int L, int heads, int head_dim, int P, int dtype,
                             void* scratch, size_t scratch_bytes,
                             int* dev_status, void* stream);

/* ---------------------------------------------------------------- layer step */

/* Where patch p's GroupNorm statistics come from at a DPP_STALE step (a DPP_SYNC step
 * always uses every patch's fresh sums):
 *   DPP_GN_SPLICED   its own fresh sums + the other patches' sums of the previous step
 *                    (the stale global statistics; "OTIL for SDXL on 4x L40S", Periodic
 *                    layer-context refresh);
 *   DPP_GN_SYNC      every patch's fresh sums while the conv and the attention stay
 *                    stale (same page, "GroupNorm sync without the rest");
 *   DPP_GN_PREVIOUS  every patch's sums of the previous step, its own included. */
#define DPP_GN_SPLICED 0
#define DPP_GN_SYNC 1
#define DPP_GN_PREVIOUS 2

typedef struct dpp_layer_params {
  int B, H, W, C;  /* feature map [B,H,W,C] */
  int P;           /* row patches (virtual ranks); H % P == 0 */
  int G;           /* GroupNorm groups; C % G == 0 */
  int heads;       /* attention heads; C == heads * head_dim */
  int head_dim;    /* must be 64 */
  int dtype;       /* DPP_F32 or DPP_BF16 */
  int refresh;     /* DPP_STALE only: 1 = refresh the state, 0 = leave it (no_sync) */
  float eps;       /* GroupNorm epsilon */
  int gn_mode;     /* DPP_GN_SPLICED (0), DPP_GN_SYNC or DPP_GN_PREVIOUS */
  int fuse_gn;     /* DPP_BF16 only (0 for DPP_F32), and W % 128 == 0 or 128 % W == 0,
                      (H/P)*W % 128 == 0: 1 = the conv applies GroupNorm to its
                      own band's rows of x as its input tiles land in shared memory, and
                      the workspace's y holds only each band's first and last row (the
                      rows the neighbours read as halos); 0 = a separate apply pass
                      writes all of y (the faster choice on the SDXL-1024 layer) */
  int fuse_refresh; /* DPP_BF16 with C a multiple of 128 only (0 otherwise); used only
                      when the step gets the second state set: 1 = the K/V refresh runs
                      in the Q/K/V projection's epilogue instead of a separate pass
                      after the output projection (same message and values; the
                      separate pass is the faster choice on the SDXL-1024 layer) */
} dpp_layer_params;

typedef struct dpp_layer_weights {
  const float* gamma; /* [C] fp32 GroupNorm scale */
  const float* beta;  /* [C] fp32 GroupNorm shift */
  const void* w_conv; /* [C,3,3,C] `dtype` conv weight (no bias) */
  const void* w_qkv;  /* [3C,C] `dtype`: rows [0,C) = Wq, [C,2C) = Wk, [2C,3C) = Wv */
  const void* w_o;    /* [C,C] `dtype` output projection */
} dpp_layer_weights;

typedef struct dpp_layer_state {
  float* gn_stats; /* [B,P,G,2] fp32: (sum x, sum x^2) of each patch, previous step */
  void* y_stale;   /* [B,H,W,C] `dtype`: previous conv input; only the 2(P-1) halo
                      rows per batch (rows r-1, r at each boundary r) are read/written */
  void* k_stale;   /* [B,L,C] `dtype` previous keys */
  void* v_stale;   /* [B,L,C] `dtype` previous values */
  int8_t* codes;   /* [dpp_message_elems] int8 residual codes (message order: K, V,
                      then for each batch the P-1 halo ranges of 2*W*C elements) */
  float* scales;   /* [dpp_message_blocks] fp32 block scales, same order */
  /* Optional second state (all four or none; none of them may overlap its counterpart
     above).  When given, a step reads the state above and leaves it unchanged, and
     writes the new state here (same layouts): a synchronous step the exact copies, a
     stale step with refresh the refreshed values, a stale step without refresh nothing
     (the caller then keeps the state above).  The caller swaps the two sets after a step
     that wrote them.  The message (codes, scales) is the same as with the in-place
     state; see fuse_refresh for where the K/V refresh then runs. */
  float* gn_next;
  void* y_next;
  void* k_next;
  void* v_next;
} dpp_layer_state;

/* Byte offsets of the pieces of the caller-allocated workspace (all 256-aligned). */
typedef struct dpp_workspace_layout {
  size_t status;     /* int device status word (zeroed by each patch_layer_step) */
  size_t gn_partial; /* fp32 per-chunk GroupNorm partial sums */
  size_t gn_fresh;   /* [B,P,G,2] fp32 fresh sums of this step */
  size_t gn_params;  /* fuse_gn: [B,P,3,C] fp32 mean, rstd*gamma, beta of each band (the
                        conv applies them to its band's rows of x); else an empty piece */
  size_t y;          /* [B,H,W,C] GroupNorm output (conv input); with fuse_gn only the
                        first and last row of each band */
  size_t h;          /* [B,H,W,C] conv output */
  size_t q, k, v;    /* [B,L,C] fresh projections */
  size_t o;          /* [B,L,C] attention output */
  size_t attn_partial;       /* the attention's scratch: per-(batch, head) range of V and
                                the split schedule's partial results
                                (dpp_attention_scratch_size(..., split = 1) bytes) */
  size_t attn_partial_bytes; /* its size (a size, not an offset; 0 for DPP_F32) */
  size_t total;      /* bytes to allocate */
} dpp_workspace_layout;

/* Fills *out for these params; returns a status (argument checks as below). */
int dpp_workspace_query(const dpp_layer_params* prm, dpp_workspace_layout* out);
/* Workspace bytes for these params, or 0 if the params are invalid. */
size_t dpp_workspace_size(const dpp_layer_params* prm);
/* Number of int8 codes / fp32 scales in one refresh message of this layer. */
int64_t dpp_message_elems(const dpp_layer_params* prm);
int64_t dpp_message_blocks(const dpp_layer_params* prm);

/*
 * patch_layer_step -- one layer pass of all P virtual ranks, then the state update.
 *   a1  fresh GroupNorm sums of every patch;
 *   a2  GroupNorm of patch p with its fresh sums + the other patches' stale sums;
 *   a3  halo conv3x3 (halo rows from state->y_stale);
 *   a4  Q, K, V = h . Wq^T, h . Wk^T, h . Wv^T;
 *   a5  stale-KV attention (own rows of K/V fresh, others from the state);
 *   a6  out = O . Wo^T;
 *   a7/a8 state update (after all patches have read the old state):
 *     DPP_SYNC: stale := fresh is used in a1-a6, then the state is written
 *       exactly (GN sums, halo rows of y, K, V); codes/scales are not touched.
 *     DPP_STALE, refresh = 1: refresh_residual of K, V and the halo rows of y
 *       (message in codes/scales), GN sums copied exactly.
 *     DPP_STALE, refresh = 0 (no_sync): the state is left untouched.
 *   The new state is written in place, or into the second state set when the state
 *   carries one (dpp_layer_state: gn_next, y_next, k_next, v_next), leaving the old one
 *   as it was.
 * x, out: [B,H,W,C] `dtype`.  workspace: dpp_workspace_size() bytes, 256-aligned.
 * Requirements: those of halo_conv3x3 (Cin = Cout = C) and stale_kv_attention
 * (L = H*W), C % G == 0, C == heads*64, and for DPP_BF16 C % 128 == 0.
 * The device status word is zeroed at the start of each call.
 */
int patch_layer_step(const dpp_layer_params* prm, const dpp_layer_weights* wts,
                     const dpp_layer_state* st, const void* x, void* out, int mode,
                     void* workspace, void* stream);

/* Same as patch_layer_step, and records stage_events[i] (cudaEvent_t, created by the
 * caller) on `stream` at each stage boundary: [0] start, [1] after GroupNorm (a1+a2),
 * [2] after the halo conv, [3] after the QKV projection, [4] after the attention,
 * [5] after the output projection, [6] after the state update.  stage_events may be
 * NULL (then no event is recorded). */
#define DPP_NUM_STAGE_EVENTS 7
int patch_layer_step_timed(const dpp_layer_params* prm, const dpp_layer_weights* wts,
                           const dpp_layer_state* st, const void* x, void* out, int mode,
                           void* workspace, void* stream, void* const* stage_events);

/* Synchronizes `stream` and returns the workspace's device status word
 * (DPP_OK, DPP_ERR_TIMEOUT, ...), or DPP_ERR_CUDA if the copy fails. */
int dpp_read_device_status(const void* workspace, void* stream);

/*
 * dpp_debug_bounds -- the index check of a library built with -DDPP_DEBUG_BOUNDS (a
 * self-checking build that stands in for a memory checker).  In that build every kernel
 * checks each global-memory index it computes (TMA copies excepted: the copy engine
 * clips them to their tensor maps) against the extent that the call's shapes give the
 * tensor it addresses; an index outside skips that access, traps nothing, and the first
 * one is recorded.  rec (host, 4 values): {source file (1 groupnorm.cu, 2 refresh.cu,
 * 3 tc_gemm.cu, 4 tc_attn.cu, 5 simt.cu, 6 otil.cu), source line, index, extent} of the
 * first recorded index since the last reset, all 0 if none; reset != 0 clears the
 * records.  Synchronizes the device.  Returns DPP_OK (checked build, nothing recorded),
 * DPP_ERR_BOUNDS (checked build, rec holds the first violation), DPP_ERR_UNSUPPORTED
 * (a normal build: no checks compiled, rec zeroed), DPP_ERR_NULL or DPP_ERR_CUDA.
 */
int dpp_debug_bounds(long long* rec, int reset);

/*
 * dpp_apply_layer_message -- brings another rank's copy of the layer state up to date
 * from the message of one DPP_STALE patch_layer_step with refresh (no counterpart
 * on the pages as a call: it is the receiving end of the exchange that "A way to
 * reduce bandwidth requirement for xDiT" describes, emulated on one device).
 * codes, scales: the message in message order (dpp_message_elems / _blocks: K, V,
 * then for each batch the P-1 halo ranges of y); gn_sums: the sender's fresh GroupNorm
 * sums [B,P,G,2] fp32 (its state's gn_stats after the step), copied exactly.
 * copy: the rank's gn_stats, y_stale, k_stale, v_stale (its codes/scales are not
 * used).  A copy equal to the sender's state before the step equals it after.
 */
int dpp_apply_layer_message(const dpp_layer_params* prm, const int8_t* codes,
                            const float* scales, const float* gn_sums,
                            const dpp_layer_state* copy, void* stream);

/*
 * patch_layer_step_noalloc -- patch_layer_step without a caller workspace.
 * (The pages have no counterpart of this call; it exists for callers that cannot
 * allocate device memory when they run a layer: a plugin in a host framework
 * whose own allocator and budget own all device memory, or a latency-critical
 * loop where cudaMalloc's implicit synchronisation is not allowed.)
 *
 * Same arguments, semantics and results as patch_layer_step, except that the
 * workspace is one fixed 80 MiB array of device memory inside the library; no
 * cudaMalloc, cudaFree or other allocating routine is called.  Every GPU that
 * loads this part of the library holds the 80 MiB until the process exits.
 *   - Layers whose dpp_workspace_size() exceeds 80 MiB return
 *     DPP_ERR_SCRATCH_LIMIT before anything is launched (the SDXL-1024
 *     mid-level layer, B=2 x 64x64 x 640 bf16, needs about 71 MiB).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture on that device.
 *   - All calls share the one array and it keeps the last call's contents:
 *     calls whose work overlaps on the GPU (different streams, or another
 *     thread) race on it and must be serialised by the caller.
 *   - The device status word lives at the start of the array; a kernel that gives
 *     up stores DPP_ERR_TIMEOUT there and returns early, as with patch_layer_step.
 *     dpp_noalloc_read_status reads it.
 */
int patch_layer_step_noalloc(const dpp_layer_params* prm, const dpp_layer_weights* wts,
                             const dpp_layer_state* st, const void* x, void* out, int mode,
                             void* stream);

/* Synchronizes `stream` and returns the device status word of the last
 * patch_layer_step_noalloc on the current device (DPP_OK, DPP_ERR_TIMEOUT, ...), or
 * DPP_ERR_CUDA if the read fails.  Allocates nothing.  (No counterpart on the pages.) */
int dpp_noalloc_read_status(void* stream);

/* ---------------------------------------------------------------- OTIL exchange */

/*
 * OTIL selective latent transmit ("OTIL for SDXL on 4x L40S", What is implemented
 * where / Self-tests), P virtual ranks on one device.  The latent (the noise prediction,
 * "Read this before interpreting the numbers", item 3) is [B, C, H, W]; rank p owns
 * rows [p*H/P, (p+1)*H/P) and views[p] is its copy of the whole latent.  A sub-block is
 * a bh x bw tile of a band over all B and C, numbered row-major over the band
 * (K = (H/P/bh) * (W/bw) per band).
 *
 * dpp_otil_step: every rank p scores its K sub-blocks -- d = 1 - cos(fresh block, the
 * peers' copy of it), cos = 0 if a norm is 0, plus 10 if the block was not sent since
 * the last reset -- sends the k highest (ties to the lower index): sel[p][0..k) in
 * index order, msg[p][j] = the fresh block sel[p][j] ([B, C, bh, bw] each), flags set;
 * every other rank copies the blocks into its view, rank p's own band of views[p]
 * becomes fresh.  Copies only (never a blend).  The scores are fp32 sums over the block.
 * dpp_otil_finalize: every view := fresh (the exact gather); reset != 0 also clears the
 * flags (the synchronous step).
 * fresh: [B,C,H,W] `dtype` holding every rank's fresh band; views: [P][B,C,H,W];
 * visited: [P][K] uint8 (zero before the first step); sel: [P][k] int32; msg:
 * [P][k][B][C][bh][bw] `dtype`.  Requires P >= 2, H % P == 0, (H/P) % bh == 0,
 * W % bw == 0, K <= 4096, 1 <= k <= min(K, 256).
 */
typedef struct dpp_otil_params {
  int B, C, H, W;  /* latent [B,C,H,W] */
  int P;           /* ranks (row bands) */
  int bh, bw;      /* sub-block rows and columns */
  int k;           /* sub-blocks each rank sends per step */
  int dtype;       /* DPP_BF16 or DPP_F32 */
} dpp_otil_params;

/* K (sub-blocks per band) for these params, or -1 if they are invalid. */
int dpp_otil_blocks(const dpp_otil_params* prm);
int dpp_otil_step(const dpp_otil_params* prm, const void* fresh, void* views, uint8_t* visited,
                  int32_t* sel, void* msg, void* stream);
int dpp_otil_finalize(const dpp_otil_params* prm, const void* fresh, void* views,
                      uint8_t* visited, int reset, void* stream);

/* Number of kernels one patch_layer_step launches for these params and mode (with
 * fuse_refresh counted as in effect, i.e. for a state with the second set). */
int dpp_layer_kernel_count(const dpp_layer_params* prm, int mode);

#ifdef __cplusplus
}
#endif

#endif /* DPP_H_ */
