"""CPU oracle for one displaced-patch layer step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may use this package.  It shares no code with the CUDA path: plain numpy in
fp64, one function per step, each citing the passage it follows.

Sources (page title, section):
  * "DistriFusion" project summary, "How It Works": the image is cut into
    patches across devices; the first step communicates synchronously, later
    steps reuse the activations of the previous step (stale) asynchronously.
  * "OTIL for SDXL on 4x L40S", "What is implemented where" / "Periodic
    layer-context refresh": three layer kinds carry stale context -- the
    patched conv (halo rows), the patched self-attention (cross-slice K/V) and
    GroupNorm; step counter 0 runs all of them on their synchronous branch.
    Same page, "GroupNorm sync without the rest": GroupNorm reduces two
    scalars per group.  Same page, "Read this before interpreting the numbers",
    item 3: the stale traffic is the attention KV and conv halo buffers.
    Same page, "Self-tests": a rank's own slice is fresh, a remote position is
    received or stale, never a blend.
  * "Benchmarking DistVAE", "Glossary": a halo is the neighbouring rows a
    sharded convolution needs; patchify splits an activation into rank-local
    row bands.

Readings where the pages are silent (each is listed with its reason in the
design notes): own patch fresh + other patches' stale partial sums for the
GroupNorm statistics; biased variance clamped at 0; zero padding at the image
edges; conv halo taken from the previous step's conv input; the layer is
out = Wo . Attn(QKV(conv3x3(GN(x)))) with no bias, activation or residual add;
attention scale 1/sqrt(head_dim), non-causal; H % P == 0.

Layout: NHWC == [B, L = H*W, C] row-major; head h owns channels
[h*head_dim, (h+1)*head_dim).  Storage dtypes are 'bf16' and 'f32'; every
tensor the layer stores (y, h, Q, K, V, O, out) is rounded to the storage dtype
at the point where it is stored, exactly once, with round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np

SYNC = 0
STALE = 1

# Where a patch's GroupNorm statistics come from at a stale step.
GN_SPLICED = 0   # own patch fresh, other patches from the previous step (the default)
GN_SYNC = 1      # every patch fresh: "GroupNorm sync without the rest" ("OTIL for SDXL
                 # on 4x L40S", What is implemented where), conv and attention stay stale
GN_PREVIOUS = 2  # every patch from the previous step (the whole previous-step statistics)


# ---------------------------------------------------------------- storage rounding
def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 has an 8-bit significand and fp32's exponent range: for |x| in
    [2^e, 2^(e+1)) the spacing is 2^(e-7), and below 2^-126 it is 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, E = np.frexp(x)                      # |x| in [2^(E-1), 2^E)
    e = np.maximum(E - 1, -126)
    q = np.ldexp(np.ones_like(x), e - 7)    # spacing of bf16 values near x
    r = np.rint(x / q) * q                  # x / q is exact (power-of-two scaling)
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, r), r)
    return np.where(x == 0, x, r)


def to_storage(x, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "f64":                       # no storage rounding (used by the pins)
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


def patch_rows(H: int, P: int, p: int):
    """Rows [r0, r1) of row patch p ("Benchmarking DistVAE", Glossary: patchify)."""
    if H % P:
        raise ValueError("H must be a multiple of P")
    Hp = H // P
    return p * Hp, (p + 1) * Hp


# ---------------------------------------------------------------- GroupNorm
def gn_partial_stats(x: np.ndarray, P: int, G: int) -> np.ndarray:
    """Per (batch, patch, group): the two sums that decide a group's statistics.

    "OTIL for SDXL on 4x L40S", GroupNorm sync without the rest: two scalars per
    group.  Returns [B, P, G, 2] = (sum x, sum x^2) over the patch's rows, all
    columns and the group's C/G channels.
    """
    B, H, W, C = x.shape
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros((B, P, G, 2))
    for p in range(P):
        r0, r1 = patch_rows(H, P, p)
        xs = x[:, r0:r1].reshape(B, (r1 - r0) * W, G, C // G)
        out[:, p, :, 0] = xs.sum(axis=(1, 3))
        out[:, p, :, 1] = (xs * xs).sum(axis=(1, 3))
    return out


def gn_apply_spliced(x: np.ndarray, fresh: np.ndarray, stale: np.ndarray, gamma, beta,
                     G: int, eps: float, dtype: str, gn_mode: int = GN_SPLICED) -> np.ndarray:
    """GroupNorm of each patch with statistics spliced from fresh and stale sums.

    GN_SPLICED: patch p uses its own fresh sums plus every other patch's stale sums
    (the stale global statistics of DistriFusion's GroupNorm; "OTIL for SDXL on 4x
    L40S", Periodic layer-context refresh).  GN_SYNC: every patch's fresh sums
    (same page, GroupNorm sync without the rest).  GN_PREVIOUS: every patch's
    stale sums.  Own patch first, then the others in order.
    mu = S1/N, var = max(S2/N - mu^2, 0), y = (x - mu) / sqrt(var + eps) * gamma_c
    + beta_c, N = H*W*C/G.
    """
    B, H, W, C = x.shape
    P = fresh.shape[1]
    N = H * W * (C // G)
    x = np.asarray(x, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    y = np.empty_like(x)
    other = fresh if gn_mode == GN_SYNC else stale
    own = stale if gn_mode == GN_PREVIOUS else fresh
    for p in range(P):
        tot = own[:, p].copy()                                # [B, G, 2]
        for q in range(P):
            if q != p:
                tot += other[:, q]
        mu = tot[..., 0] / N
        var = np.maximum(tot[..., 1] / N - mu * mu, 0.0)
        rstd = 1.0 / np.sqrt(var + eps)
        r0, r1 = patch_rows(H, P, p)
        xs = x[:, r0:r1].reshape(B, r1 - r0, W, G, C // G)
        ys = (xs - mu[:, None, None, :, None]) * rstd[:, None, None, :, None]
        ys = ys.reshape(B, r1 - r0, W, C) * gamma + beta
        y[:, r0:r1] = ys
    return to_storage(y, dtype)


# ---------------------------------------------------------------- halo conv
def halo_conv3x3(y_fresh: np.ndarray, y_stale: np.ndarray, w: np.ndarray, P: int,
                 dtype: str, rows=None) -> np.ndarray:
    """3x3 "same" convolution of each row band, its halo rows taken from the stale map.

    "Benchmarking DistVAE", Glossary (halo: the neighbouring rows a sharded
    convolution needs); "OTIL for SDXL on 4x L40S", item 3 and Periodic
    layer-context refresh (the conv halo buffers are stale).  For output row r of
    band p = [r0, r1):
      h[b,r,c,o] = sum_{i,j in -1..1} sum_k w[o, i+1, j+1, k] * yhat[b, r+i, c+j, k]
    yhat = fresh y inside the band, stale y for rows r0-1 and r1, zero outside
    the image (rows and columns).  w is [Cout, 3, 3, Cin].

    ``rows``: optional sorted output rows to evaluate (each output row depends
    only on its own three source rows); the result is then [B, len(rows), W, Cout].
    """
    B, H, W, Cin = y_fresh.shape
    Cout = w.shape[0]
    yf = np.asarray(y_fresh, dtype=np.float64)
    ys = np.asarray(y_stale, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    sel = np.arange(H) if rows is None else np.asarray(rows)
    h = np.empty((B, len(sel), W, Cout))
    for p in range(P):
        r0, r1 = patch_rows(H, P, p)
        Hp = r1 - r0
        mine = np.nonzero((sel >= r0) & (sel < r1))[0]
        if mine.size == 0:
            continue
        yhat = np.zeros((B, Hp + 2, W + 2, Cin))
        yhat[:, 1:Hp + 1, 1:W + 1] = yf[:, r0:r1]
        if r0 > 0:
            yhat[:, 0, 1:W + 1] = ys[:, r0 - 1]
        if r1 < H:
            yhat[:, Hp + 1, 1:W + 1] = ys[:, r1]
        loc = sel[mine] - r0                      # output rows within the band
        acc = np.zeros((B, len(loc), W, Cout))
        for i in range(3):
            for j in range(3):
                acc += yhat[:, loc + i, j:j + W, :] @ w[:, i, j, :].T
        h[:, mine] = acc
    return to_storage(h, dtype)


# ---------------------------------------------------------------- projections
def linear(x: np.ndarray, w: np.ndarray, dtype: str) -> np.ndarray:
    """x [..., K] times w[N, K] transposed, no bias (the QKV and output projections)."""
    return to_storage(np.asarray(x, np.float64) @ np.asarray(w, np.float64).T, dtype)


# ---------------------------------------------------------------- stale-KV attention
def stale_kv_attention(q, k_fresh, v_fresh, k_stale, v_stale, heads: int, P: int,
                       dtype: str, rows=None) -> np.ndarray:
    """Self-attention of each patch's fresh queries over spliced full-sequence K/V.

    "OTIL for SDXL on 4x L40S", item 3 and Periodic layer-context refresh: the
    cross-slice attention K/V are stale; "Self-tests": a rank's own slice is
    fresh and any other position is stale, never a blend.  For token t in patch
    p (tokens [p*L/P, (p+1)*L/P)) and head h:
      O[t,h] = sum_s softmax_s(Q[t,h] . Khat_p[s,h] / sqrt(d)) Vhat_p[s,h]
    with Khat_p[s] = K_fresh[s] if s is in patch p else K_stale[s] (same for V),
    over all L keys, no mask.  Softmax subtracts the row maximum, in fp64.

    ``rows``: optional sorted array of token indices (shared by all batches) to
    evaluate; the result then has shape [B, len(rows), C].
    """
    B, L, C = q.shape
    d = C // heads
    if L % P:
        raise ValueError("L must be a multiple of P")
    Lp = L // P
    scale = 1.0 / np.sqrt(d)
    tok = np.arange(L) if rows is None else np.asarray(rows)
    out = np.empty((B, len(tok), C))
    for b in range(B):
        for p in range(P):
            sel = np.nonzero((tok >= p * Lp) & (tok < (p + 1) * Lp))[0]
            if sel.size == 0:
                continue
            kh = np.array(k_stale[b], dtype=np.float64)
            vh = np.array(v_stale[b], dtype=np.float64)
            kh[p * Lp:(p + 1) * Lp] = k_fresh[b, p * Lp:(p + 1) * Lp]
            vh[p * Lp:(p + 1) * Lp] = v_fresh[b, p * Lp:(p + 1) * Lp]
            for c0 in range(0, sel.size, 256):          # independent query rows
                idx = sel[c0:c0 + 256]
                qs = np.asarray(q[b, tok[idx]], dtype=np.float64)
                for hh in range(heads):
                    cs = slice(hh * d, (hh + 1) * d)
                    s = (qs[:, cs] @ kh[:, cs].T) * scale
                    s -= s.max(axis=1, keepdims=True)
                    e = np.exp(s)
                    out[b, idx, cs] = (e @ vh[:, cs]) / e.sum(axis=1, keepdims=True)
    return to_storage(out, dtype)


# ---------------------------------------------------------------- refresh
def refresh_residual(fresh: np.ndarray, stale: np.ndarray, dtype: str):
    """Compressed-residual refresh of a flat buffer; returns (new_stale, codes, scales).

    The arithmetic is in ``refresh.c`` (exact fp32 operation sequence); see there.
    """
    from . import refresh as _r
    return _r.refresh_residual(fresh, stale, dtype)


def apply_residual(stale: np.ndarray, codes, scales, dtype: str) -> np.ndarray:
    """What a receiving rank does with a message: stale += dequant(codes, scales)."""
    from . import refresh as _r
    return _r.apply_residual(stale, codes, scales, dtype)


def halo_segments(H: int, W: int, C: int, P: int):
    """Flat (row-major [H, W, C]) element ranges of the 2(P-1) halo rows of one batch.

    The rows any band reads from another band are r-1 and r at each interior
    boundary r = p*H/P, p = 1..P-1: two adjacent rows, one contiguous range.
    """
    Hp = H // P
    return [((p * Hp - 1) * W * C, (p * Hp + 1) * W * C) for p in range(1, P)]


# ---------------------------------------------------------------- whole layer
def layer_forward(x, state, wts, P: int, G: int, heads: int, eps: float, dtype: str,
                  mode: int, rows=None, gn_mode: int = GN_SPLICED):
    """Steps a1-a6 for all P virtual ranks; returns a dict of every stored tensor.

    SYNC (the warm-up / refresh step, "DistriFusion", How It Works; "OTIL for
    SDXL on 4x L40S", Periodic layer-context refresh): every stale input is
    replaced by its fresh counterpart before use.  STALE: the state given is used.
    """
    B, H, W, C = x.shape
    L = H * W
    x = np.asarray(x, np.float64)
    fresh_stats = gn_partial_stats(x, P, G)
    stale_stats = fresh_stats if mode == SYNC else np.asarray(state["gn_stats"], np.float64)
    y = gn_apply_spliced(x, fresh_stats, stale_stats, wts["gamma"], wts["beta"], G, eps, dtype,
                         gn_mode)
    y_st = y if mode == SYNC else state["y_stale"]
    h = halo_conv3x3(y, y_st, wts["w_conv"], P, dtype)
    hf = h.reshape(B, L, C)
    wqkv = np.asarray(wts["w_qkv"], np.float64)
    Q = linear(hf, wqkv[:C], dtype)
    K = linear(hf, wqkv[C:2 * C], dtype)
    V = linear(hf, wqkv[2 * C:], dtype)
    Ks = K if mode == SYNC else np.asarray(state["k_stale"], np.float64).reshape(B, L, C)
    Vs = V if mode == SYNC else np.asarray(state["v_stale"], np.float64).reshape(B, L, C)
    O = stale_kv_attention(Q, K, V, Ks, Vs, heads, P, dtype, rows=rows)
    out = linear(O, wts["w_o"], dtype)
    return dict(gn_fresh=fresh_stats, y=y, h=h, q=Q, k=K, v=V, o=O, out=out)


def layer_state_update(fwd: dict, state: dict, P: int, dtype: str, mode: int, refresh: bool):
    """Step a7-a8: the state the next step reads.  Returns a new state dict.

    SYNC writes the state exactly (GN sums, the halo rows of y, K, V).  STALE
    with refresh sends the compressed residual of K, V and the halo rows of y
    and copies the GN sums exactly ("OTIL for SDXL on 4x L40S", GroupNorm sync
    without the rest: two scalars per group); without refresh (no_sync, item 3)
    the state is left as it was.  codes/scales are returned in message order:
    K, V, then the halo ranges of each batch.
    """
    y = fwd["y"]
    B, H, W, C = y.shape
    new = {k: np.array(v, copy=True) for k, v in state.items()}
    segs = halo_segments(H, W, C, P)
    if mode == SYNC:
        new["gn_stats"] = fwd["gn_fresh"].copy()
        new["k_stale"] = fwd["k"].reshape(new["k_stale"].shape).copy()
        new["v_stale"] = fwd["v"].reshape(new["v_stale"].shape).copy()
        ys = new["y_stale"].reshape(B, -1)
        yf = y.reshape(B, -1)
        for (a, b_) in segs:
            ys[:, a:b_] = yf[:, a:b_]
        new["y_stale"] = ys.reshape(y.shape)
        return new, None, None
    if not refresh:
        return new, None, None
    codes, scales = [], []
    for name, src in (("k_stale", fwd["k"]), ("v_stale", fwd["v"])):
        ns, c, s = refresh_residual(src.reshape(-1), new[name].reshape(-1), dtype)
        new[name] = ns.reshape(new[name].shape)
        codes.append(c)
        scales.append(s)
    ys = new["y_stale"].reshape(B, -1)
    yf = y.reshape(B, -1)
    for b in range(B):
        for (a, b_) in segs:
            ns, c, s = refresh_residual(yf[b, a:b_], ys[b, a:b_], dtype)
            ys[b, a:b_] = ns
            codes.append(c)
            scales.append(s)
    new["y_stale"] = ys.reshape(y.shape)
    new["gn_stats"] = fwd["gn_fresh"].copy()
    return new, np.concatenate(codes), np.concatenate(scales)


def patch_layer_step(x, state, wts, P: int, G: int, heads: int, eps: float, dtype: str,
                     mode: int, refresh: bool = True, gn_mode: int = GN_SPLICED):
    """One layer pass of all P virtual ranks followed by the state update."""
    fwd = layer_forward(x, state, wts, P, G, heads, eps, dtype, mode, gn_mode=gn_mode)
    new_state, codes, scales = layer_state_update(fwd, state, P, dtype, mode, refresh)
    return fwd, new_state, codes, scales


def empty_state(B: int, H: int, W: int, C: int, P: int, G: int) -> dict:
    L = H * W
    return dict(gn_stats=np.zeros((B, P, G, 2)), y_stale=np.zeros((B, H, W, C)),
                k_stale=np.zeros((B, L, C)), v_stale=np.zeros((B, L, C)))
