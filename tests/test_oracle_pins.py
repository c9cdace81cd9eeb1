"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties an oracle function to a closed form, a library routine that
computes the same textbook operation, a brute-force evaluation on tiny inputs,
or a hand-worked golden case under tests/golden/.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ bf16 rounding
def test_round_bf16_hand_cases():
    # spacing near 1 is 2^-7: 1 + 2^-8 is a tie -> even (1); 1 + 3*2^-8 -> 1 + 2^-6
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3.0, 1e-45, -1e-40, 0.0])
    exp = np.array([1.0, 1 + 2 ** -6, -1.0, 3.0, 0.0, -(2.0 ** -133), 0.0])
    np.testing.assert_array_equal(oracle.round_bf16(x), exp)


def test_round_bf16_matches_torch_on_fp32_values():
    f = np.concatenate([RNG.standard_normal(20000), RNG.standard_normal(2000) * 1e-39,
                        RNG.standard_normal(2000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(f.astype(np.float64)), ref)


# ------------------------------------------------------------------ GroupNorm
def test_gn_golden_two_patch(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "gn_two_patch.json")))
    x = np.array(g["x"])
    fresh = oracle.gn_partial_stats(x, g["P"], g["G"])
    np.testing.assert_array_equal(fresh, np.array(g["fresh_sums"]))
    stale = np.array(g["stale_sums"])
    gamma, beta = np.ones(2), np.zeros(2)
    ev = lambda e: eval(e, {"sqrt": math.sqrt})  # noqa: E731
    y = oracle.gn_apply_spliced(x, fresh, stale, gamma, beta, g["G"], g["eps"], "f64")
    exp = np.array([[ev(e) for e in row] for row in g["y_stale_expr"]])
    np.testing.assert_allclose(y[0, :, 0, :], exp, rtol=1e-14, atol=1e-14)
    y = oracle.gn_apply_spliced(x, fresh, fresh, gamma, beta, g["G"], g["eps"], "f64")
    exp = np.array([[ev(e) for e in row] for row in g["y_sync_expr"]])
    np.testing.assert_allclose(y[0, :, 0, :], exp, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_gn_sync_equals_torch_group_norm(P):
    B, H, W, C, G = 2, 16, 8, 24, 4
    x = RNG.standard_normal((B, H, W, C)) * 2 + 0.5
    gamma, beta = RNG.standard_normal(C), RNG.standard_normal(C)
    s = oracle.gn_partial_stats(x, P, G)
    y = oracle.gn_apply_spliced(x, s, s, gamma, beta, G, 1e-5, "f64")
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    ref = torch.nn.functional.group_norm(xt, G, torch.from_numpy(gamma), torch.from_numpy(beta),
                                         eps=1e-5).permute(0, 2, 3, 1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_gn_constant_input_gives_beta():
    B, H, W, C, G, P = 1, 8, 4, 8, 2, 2
    x = np.full((B, H, W, C), 3.25)
    beta = RNG.standard_normal(C)
    s = oracle.gn_partial_stats(x, P, G)
    y = oracle.gn_apply_spliced(x, s, s, np.ones(C), beta, G, 1e-5, "f64")
    np.testing.assert_allclose(y, np.broadcast_to(beta, y.shape), atol=1e-12)


def test_gn_stale_uses_only_other_patches():
    # Changing patch p's own stale sums must not change patch p's output.
    B, H, W, C, G, P = 1, 8, 4, 8, 2, 4
    x = RNG.standard_normal((B, H, W, C))
    f = oracle.gn_partial_stats(x, P, G)
    st = f + RNG.standard_normal(f.shape) * 0.1
    st[..., 1] = np.abs(st[..., 1])
    y1 = oracle.gn_apply_spliced(x, f, st, np.ones(C), np.zeros(C), G, 1e-5, "f64")
    st2 = st.copy()
    st2[:, 1] += 5.0
    y2 = oracle.gn_apply_spliced(x, f, st2, np.ones(C), np.zeros(C), G, 1e-5, "f64")
    np.testing.assert_array_equal(y1[:, 2:4], y2[:, 2:4])          # patch 1 unchanged
    assert np.abs(y1[:, :2] - y2[:, :2]).max() > 1e-3               # others changed


@pytest.mark.parametrize("P", [2, 4])
def test_gn_sync_mode_ignores_stale_and_equals_torch(P):
    """GN_SYNC (GroupNorm sync without the rest): every patch uses every patch's fresh
    sums, so any stale state gives textbook GroupNorm of the whole map."""
    B, H, W, C, G = 2, 16, 8, 24, 4
    x = RNG.standard_normal((B, H, W, C)) * 2 + 0.5
    gamma, beta = RNG.standard_normal(C), RNG.standard_normal(C)
    s = oracle.gn_partial_stats(x, P, G)
    junk = RNG.standard_normal(s.shape) * 100.0
    y = oracle.gn_apply_spliced(x, s, junk, gamma, beta, G, 1e-5, "f64", oracle.GN_SYNC)
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    ref = torch.nn.functional.group_norm(xt, G, torch.from_numpy(gamma), torch.from_numpy(beta),
                                         eps=1e-5).permute(0, 2, 3, 1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_gn_previous_mode_uses_only_the_stale_statistics():
    """GN_PREVIOUS: every patch is normalised with the previous step's statistics alone.
    With the stale sums of another map x2 the output is (x - mean(x2)) / sqrt(var(x2) +
    eps) per group, the biased mean and variance of x2 taken directly (numpy)."""
    B, H, W, C, G, P = 2, 8, 4, 12, 3, 4
    x = RNG.standard_normal((B, H, W, C))
    x2 = RNG.standard_normal((B, H, W, C)) * 1.5 - 0.25
    f = oracle.gn_partial_stats(x, P, G)
    st = oracle.gn_partial_stats(x2, P, G)
    y = oracle.gn_apply_spliced(x, f, st, np.ones(C), np.zeros(C), G, 1e-5, "f64",
                                oracle.GN_PREVIOUS)
    g2 = x2.reshape(B, H, W, G, C // G)
    mu = g2.mean(axis=(1, 2, 4))
    var = g2.var(axis=(1, 2, 4))
    ref = ((x.reshape(B, H, W, G, C // G) - mu[:, None, None, :, None]) /
           np.sqrt(var[:, None, None, :, None] + 1e-5)).reshape(B, H, W, C)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)
    # the fresh sums do not enter at all
    y2 = oracle.gn_apply_spliced(x, f * 3.0 + 1.0, st, np.ones(C), np.zeros(C), G, 1e-5, "f64",
                                 oracle.GN_PREVIOUS)
    np.testing.assert_array_equal(y, y2)


# ------------------------------------------------------------------ halo conv
@pytest.mark.parametrize("P", [1, 2, 4])
def test_conv_unbanded_matches_torch_conv2d(P):
    B, H, W, Ci, Co = 2, 8, 5, 6, 7
    y = RNG.standard_normal((B, H, W, Ci))
    w = RNG.standard_normal((Co, 3, 3, Ci))
    h = oracle.halo_conv3x3(y, y, w, P, "f64")
    ref = torch.nn.functional.conv2d(torch.from_numpy(y).permute(0, 3, 1, 2),
                                     torch.from_numpy(w).permute(0, 3, 1, 2), padding=1)
    np.testing.assert_allclose(h, ref.permute(0, 2, 3, 1).numpy(), rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("ti,tj", [(0, 0), (0, 1), (1, 1), (2, 1), (2, 2)])
def test_conv_sentinel_halo_source(ti, tj):
    """fresh = +1, stale = -1, one-hot tap weight: each output equals the source
    of the input pixel that tap reads, derived here from the band rule alone."""
    B, H, W, C, P = 1, 12, 4, 2, 3
    yf = np.ones((B, H, W, C))
    ys = -np.ones((B, H, W, C))
    w = np.zeros((1, 3, 3, C))
    w[0, ti, tj, 1] = 1.0
    h = oracle.halo_conv3x3(yf, ys, w, P, "f64")[0, :, :, 0]
    Hp = H // P
    for r in range(H):
        band = r // Hp
        for c in range(W):
            rr, cc = r + ti - 1, c + tj - 1
            if rr < 0 or rr >= H or cc < 0 or cc >= W:
                exp = 0.0
            elif rr // Hp == band:
                exp = 1.0
            else:
                exp = -1.0
            assert h[r, c] == exp, (r, c)


# ------------------------------------------------------------------ projections
def test_linear_identity_and_torch():
    x = RNG.standard_normal((5, 8))
    np.testing.assert_array_equal(oracle.linear(x, np.eye(8), "f64"), x)
    w = RNG.standard_normal((3, 8))
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    np.testing.assert_allclose(oracle.linear(x, w, "f64"), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ attention
def _attention_bruteforce(q, kf, vf, ks, vs, heads, P):
    B, L, C = q.shape
    d = C // heads
    Lp = L // P
    out = np.zeros_like(q)
    for b in range(B):
        for t in range(L):
            p = t // Lp
            for h in range(heads):
                sc = []
                for s in range(L):
                    src_k = kf if p * Lp <= s < (p + 1) * Lp else ks
                    sc.append(sum(q[b, t, h * d + e] * src_k[b, s, h * d + e] for e in range(d))
                              / math.sqrt(d))
                m = max(sc)
                ex = [math.exp(v - m) for v in sc]
                z = sum(ex)
                for e in range(d):
                    acc = 0.0
                    for s in range(L):
                        src_v = vf if p * Lp <= s < (p + 1) * Lp else vs
                        acc += ex[s] * src_v[b, s, h * d + e]
                    out[b, t, h * d + e] = acc / z
    return out


def test_attention_bruteforce_tiny():
    B, L, heads, d, P = 2, 8, 2, 4, 2
    C = heads * d
    q, kf, vf, ks, vs = (RNG.standard_normal((B, L, C)) for _ in range(5))
    o = oracle.stale_kv_attention(q, kf, vf, ks, vs, heads, P, "f64")
    np.testing.assert_allclose(o, _attention_bruteforce(q, kf, vf, ks, vs, heads, P),
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_attention_q0_closed_form(P):
    """Q = 0: the softmax is uniform, so with V_fresh = +1 and V_stale = -1 the
    output is (Lp - (L - Lp)) / L for every query: pins the splice range."""
    B, L, heads, d = 1, 64, 1, 4
    q = np.zeros((B, L, d))
    k = RNG.standard_normal((B, L, d))
    o = oracle.stale_kv_attention(q, k, np.ones((B, L, d)), k, -np.ones((B, L, d)), heads, P, "f64")
    Lp = L // P
    np.testing.assert_allclose(o, (2 * Lp - L) / L, atol=1e-14)


def test_attention_stale_equals_fresh_is_sdpa():
    B, L, heads, d, P = 2, 32, 3, 8, 4
    C = heads * d
    q, k, v = (RNG.standard_normal((B, L, C)) for _ in range(3))
    o = oracle.stale_kv_attention(q, k, v, k, v, heads, P, "f64")
    tq, tk, tv = (torch.from_numpy(t).view(B, L, heads, d).transpose(1, 2) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)
    np.testing.assert_allclose(o, ref.transpose(1, 2).reshape(B, L, C).numpy(), rtol=1e-11,
                               atol=1e-11)


def test_attention_rows_subset_matches_full():
    B, L, heads, d, P = 1, 40, 2, 4, 4
    C = heads * d
    q, kf, vf, ks, vs = (RNG.standard_normal((B, L, C)) for _ in range(5))
    full = oracle.stale_kv_attention(q, kf, vf, ks, vs, heads, P, "f64")
    rows = np.array([0, 9, 10, 23, 39])
    sub = oracle.stale_kv_attention(q, kf, vf, ks, vs, heads, P, "f64", rows=rows)
    np.testing.assert_allclose(sub, full[:, rows], rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------ refresh
def test_refresh_golden_block(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "refresh_block.json")))
    n = g["n"]
    fresh = np.zeros(n)
    stale = np.zeros(n)
    fresh[:5] = g["fresh_head"]
    fresh[128:] = stale[128:] = g["block1_value"]
    new, codes, scales = oracle.refresh_residual(fresh, stale, "bf16")
    np.testing.assert_array_equal(codes[:5], g["codes_head"])
    assert not codes[5:].any()
    np.testing.assert_array_equal(scales, np.array(g["scales"], dtype=np.float32))
    np.testing.assert_array_equal(new[:5], g["new_stale_head"])
    np.testing.assert_array_equal(new[5:128], 0.0)
    np.testing.assert_array_equal(new[128:], g["block1_value"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_zero_delta_is_identity(dtype):
    s = oracle.to_storage(RNG.standard_normal(1000), dtype)
    new, codes, scales = oracle.refresh_residual(s, s, dtype)
    np.testing.assert_array_equal(new, s)
    assert not codes.any() and not scales.any()


def _round_fraction(x: Fraction, p: int) -> Fraction:
    """Exact round-to-nearest-even of a rational to a binary float with a p-bit
    significand and fp32's exponent range (p = 24: fp32, p = 8: bf16)."""
    if x == 0:
        return Fraction(0)
    sgn = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - (p - 1))
    m = a / ulp
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * fl * ulp


def _rint_even(x: Fraction) -> int:
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def _refresh_exact(fresh, stale, p_store):
    """The refresh rule evaluated with exact rationals and one explicit rounding per
    IEEE fp32 operation (sub, div, div, fma), then the storage rounding."""
    n = len(fresh)
    new, codes, scales = [], [], []
    for b0 in range(0, n, 128):
        fs = [Fraction(float(v)) for v in fresh[b0:b0 + 128]]
        ss = [Fraction(float(v)) for v in stale[b0:b0 + 128]]
        d = [_round_fraction(f - s, 24) for f, s in zip(fs, ss)]
        a = max(abs(v) for v in d)
        sc = _round_fraction(a / 127, 24)
        scales.append(float(sc))
        for dv, sv in zip(d, ss):
            q = 0 if sc == 0 else max(-127, min(127, _rint_even(_round_fraction(dv / sc, 24))))
            codes.append(q)
            new.append(float(_round_fraction(_round_fraction(q * sc + sv, 24), p_store)))
    return np.array(new), np.array(codes, dtype=np.int8), np.array(scales, dtype=np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_matches_exact_rational_evaluation(dtype):
    n = 300
    stale = oracle.to_storage(RNG.standard_normal(n), dtype)
    delta = RNG.standard_normal(n) * np.repeat([0.05, 1.0, 0.001], 128)[:n]
    fresh = oracle.to_storage(stale + delta, dtype)
    new, codes, scales = oracle.refresh_residual(fresh, stale, dtype)
    en, ec, es = _refresh_exact(fresh, stale, 8 if dtype == "bf16" else 24)
    np.testing.assert_array_equal(codes, ec)
    np.testing.assert_array_equal(scales, es)
    np.testing.assert_array_equal(new, en)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_error_bound_and_no_accumulation(dtype):
    n = 128 * 40
    stale = oracle.to_storage(RNG.standard_normal(n), dtype)
    fresh = oracle.to_storage(stale + RNG.standard_normal(n) * 0.05, dtype)
    new, codes, scales = oracle.refresh_residual(fresh, stale, dtype)
    s_e = np.repeat(scales.astype(np.float64), 128)
    ulp = np.abs(new) * (2.0 ** -7 if dtype == "bf16" else 2.0 ** -23)
    err = np.abs(new - fresh)
    assert np.all(err <= s_e / 2 + ulp + 1e-30)
    # the element with the largest |delta| in each block carries code +-127
    d = (fresh - stale).reshape(-1, 128)
    imax = np.abs(d).argmax(axis=1)
    np.testing.assert_array_equal(np.abs(codes.reshape(-1, 128)[np.arange(len(imax)), imax]), 127)
    # refreshing again against the same fresh values never increases the error
    new2, _, _ = oracle.refresh_residual(fresh, new, dtype)
    assert np.abs(new2 - fresh).max() <= err.max()
    assert np.linalg.norm(new2 - fresh) <= np.linalg.norm(err) + 1e-12


def test_apply_residual_reproduces_refresh():
    n = 128 * 3 + 17
    stale = oracle.round_bf16(RNG.standard_normal(n))
    fresh = oracle.round_bf16(stale + RNG.standard_normal(n) * 0.05)
    new, codes, scales = oracle.refresh_residual(fresh, stale, "bf16")
    np.testing.assert_array_equal(oracle.apply_residual(stale, codes, scales, "bf16"), new)


# ------------------------------------------------------------------ whole layer
def _layer_case(B=1, H=16, W=4, C=16, G=4, heads=2, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, H, W, C))
    wts = dict(gamma=1 + 0.1 * rng.standard_normal(C), beta=0.1 * rng.standard_normal(C),
               w_conv=rng.standard_normal((C, 3, 3, C)) * 0.1,
               w_qkv=rng.standard_normal((3 * C, C)) * 0.2, w_o=rng.standard_normal((C, C)) * 0.2)
    return x, wts


def _garbage_state(B, H, W, C, P, G, seed=5):
    rng = np.random.default_rng(seed)
    st = oracle.empty_state(B, H, W, C, P, G)
    return {k: rng.standard_normal(v.shape) + (5.0 if k == "gn_stats" else 0.0)
            for k, v in st.items()}


@pytest.mark.parametrize("P", [2, 4, 8])
def test_layer_sync_equals_unpartitioned(P):
    """At the synchronous step the patched layer equals the full layer for any P
    ("DistriFusion", How It Works: the first step is synchronous)."""
    B, H, W, C, G, heads = 1, 16, 4, 16, 4, 2
    x, wts = _layer_case(B, H, W, C, G, heads)
    ref = oracle.layer_forward(x, None, wts, 1, G, heads, 1e-5, "f64", oracle.SYNC)
    got = oracle.layer_forward(x, _garbage_state(B, H, W, C, P, G), wts, P, G, heads, 1e-5,
                               "f64", oracle.SYNC)
    np.testing.assert_allclose(got["out"], ref["out"], rtol=1e-10, atol=1e-12)


def test_layer_stale_P1_equals_sync():
    B, H, W, C, G, heads = 1, 8, 4, 16, 4, 2
    x, wts = _layer_case(B, H, W, C, G, heads)
    st = _garbage_state(B, H, W, C, 1, G)
    st["gn_stats"] = np.abs(st["gn_stats"])
    a = oracle.layer_forward(x, st, wts, 1, G, heads, 1e-5, "f64", oracle.STALE)
    b = oracle.layer_forward(x, None, wts, 1, G, heads, 1e-5, "f64", oracle.SYNC)
    np.testing.assert_array_equal(a["out"], b["out"])


@pytest.mark.parametrize("gn_mode", [0, 1, 2])
def test_layer_stale_with_synced_state_equals_sync(gn_mode):
    B, H, W, C, G, heads, P = 2, 16, 4, 16, 4, 2, 4
    x, wts = _layer_case(B, H, W, C, G, heads)
    st0 = oracle.empty_state(B, H, W, C, P, G)
    fwd, st, _, _ = oracle.patch_layer_step(x, st0, wts, P, G, heads, 1e-5, "f32", oracle.SYNC)
    again = oracle.layer_forward(x, st, wts, P, G, heads, 1e-5, "f32", oracle.STALE,
                                 gn_mode=gn_mode)
    np.testing.assert_allclose(again["out"], fwd["out"], rtol=1e-6, atol=1e-7)


def test_layer_gn_sync_mode_keeps_conv_and_attention_stale():
    """GN_SYNC changes only the GroupNorm: its y equals the SYNC step's y on the same x
    while the attention still reads the stale K/V (so out differs from SYNC's)."""
    B, H, W, C, G, heads, P = 1, 8, 4, 16, 4, 2, 2
    x, wts = _layer_case(B, H, W, C, G, heads)
    st0 = oracle.empty_state(B, H, W, C, P, G)
    x_prev = x + 0.5 * RNG.standard_normal(x.shape)
    _, st, _, _ = oracle.patch_layer_step(x_prev, st0, wts, P, G, heads, 1e-5, "f32", oracle.SYNC)
    sync = oracle.layer_forward(x, st, wts, P, G, heads, 1e-5, "f32", oracle.SYNC)
    gs = oracle.layer_forward(x, st, wts, P, G, heads, 1e-5, "f32", oracle.STALE,
                              gn_mode=oracle.GN_SYNC)
    np.testing.assert_array_equal(gs["y"], sync["y"])
    # the conv still takes its halo rows from the old state, the attention its K/V
    assert np.linalg.norm(gs["h"] - sync["h"]) > 1e-3 * np.linalg.norm(sync["h"])
    assert not np.array_equal(gs["out"], sync["out"])


def test_layer_stale_state_changes_only_remote_dependence():
    """Own slice fresh: with K/V state perturbed only inside patch p's own rows,
    patch p's attention output is unchanged ("OTIL for SDXL on 4x L40S", Self-tests)."""
    B, H, W, C, G, heads, P = 1, 16, 4, 16, 4, 2, 4
    x, wts = _layer_case(B, H, W, C, G, heads)
    st0 = oracle.empty_state(B, H, W, C, P, G)
    _, st, _, _ = oracle.patch_layer_step(x * 1.1, st0, wts, P, G, heads, 1e-5, "f64",
                                          oracle.SYNC)
    a = oracle.layer_forward(x, st, wts, P, G, heads, 1e-5, "f64", oracle.STALE)
    st2 = {k: v.copy() for k, v in st.items()}
    Lp = H * W // P
    st2["k_stale"][:, Lp:2 * Lp] += 3.0
    st2["v_stale"][:, Lp:2 * Lp] -= 3.0
    b = oracle.layer_forward(x, st2, wts, P, G, heads, 1e-5, "f64", oracle.STALE)
    np.testing.assert_array_equal(a["o"][:, Lp:2 * Lp], b["o"][:, Lp:2 * Lp])
    assert np.abs(a["o"][:, :Lp] - b["o"][:, :Lp]).max() > 1e-3


def test_multirank_copies_stay_identical():
    """P ranks with their own stale copies, each sending only the residual of its
    own rows: all copies stay identical to the one shared buffer the GPU path
    keeps, over several steps."""
    B, H, W, C, G, heads, P = 1, 16, 4, 128, 4, 2, 4
    rng = np.random.default_rng(3)
    x0, wts = _layer_case(B, H, W, C, G, heads, seed=3)
    dt = "bf16"
    wts = {k: (oracle.round_bf16(v) if k.startswith("w_") else v) for k, v in wts.items()}
    shared = oracle.empty_state(B, H, W, C, P, G)
    fwd, shared, _, _ = oracle.patch_layer_step(oracle.round_bf16(x0), shared, wts, P, G, heads,
                                                1e-5, dt, oracle.SYNC)
    copies = [{k: v.copy() for k, v in shared.items()} for _ in range(P)]
    L, Lp = H * W, H * W // P
    for step in range(3):
        x = oracle.round_bf16(x0 + 0.05 * (step + 1) * rng.standard_normal(x0.shape))
        fwd, shared_new, _, _ = oracle.patch_layer_step(x, shared, wts, P, G, heads, 1e-5, dt,
                                                        oracle.STALE)
        for name in ("k", "v"):
            fresh = fwd[name].reshape(B, L * C)
            for p in range(P):
                seg = slice(p * Lp * C, (p + 1) * Lp * C)
                own = copies[p][name + "_stale"].reshape(B, L * C)
                _, codes, scales = oracle.refresh_residual(fresh[0, seg], own[0, seg], dt)
                for r in range(P):
                    cr = copies[r][name + "_stale"].reshape(B, L * C)
                    cr[0, seg] = oracle.apply_residual(cr[0, seg], codes, scales, dt)
        for r in range(P):
            for name in ("k_stale", "v_stale"):
                np.testing.assert_array_equal(copies[r][name].reshape(-1),
                                              shared_new[name].reshape(-1))
        # own rows of the reconstruction are the quantised fresh rows; never a blend
        # of two steps: every element is either the old value or old + code*scale
        shared = shared_new


def test_conv_rows_subset_matches_full():
    B, H, W, Ci, Co, P = 1, 12, 5, 4, 3, 3
    yf = RNG.standard_normal((B, H, W, Ci))
    ys = RNG.standard_normal((B, H, W, Ci))
    w = RNG.standard_normal((Co, 3, 3, Ci))
    full = oracle.halo_conv3x3(yf, ys, w, P, "f64")
    rows = np.array([0, 3, 4, 7, 11])
    np.testing.assert_allclose(oracle.halo_conv3x3(yf, ys, w, P, "f64", rows=rows), full[:, rows],
                               rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("P", [2, 4])
def test_state_update_stale_refreshes_exactly_the_halo_rows_of_y(P):
    """The STALE branch of the state update ("OTIL for SDXL on 4x L40S", item 3: the
    stale state is the conv halo rows, the attention K/V and the two GroupNorm scalars
    per group), pinned with sentinels.  Fresh y = +1 and stale y = -1 everywhere, so
    each refreshed block has delta 2, scale 2/127 and codes 127, and its refreshed bf16
    value rounds to exactly +1; h carries a third value (+5) that a refresh of the
    wrong tensor would show.  Exactly rows r-1 and r at each interior boundary r become
    +1, every other row stays -1; the message holds K, V, then 2*W*C codes of 127 per
    (batch, boundary); the GroupNorm sums are copied exactly, not quantised."""
    B, H, W, C, G = 2, 4 * P, 4, 8, 2
    L = H * W
    rng = np.random.default_rng(11)
    y_f = np.ones((B, H, W, C))
    fwd = dict(y=y_f, h=np.full((B, H, W, C), 5.0),
               k=oracle.round_bf16(rng.standard_normal((B, L, C))),
               v=oracle.round_bf16(rng.standard_normal((B, L, C))),
               gn_fresh=rng.standard_normal((B, P, G, 2)) * 10.0 + 0.123456789)
    state = dict(gn_stats=rng.standard_normal((B, P, G, 2)),
                 y_stale=-np.ones((B, H, W, C)),
                 k_stale=oracle.round_bf16(rng.standard_normal((B, L, C))),
                 v_stale=oracle.round_bf16(rng.standard_normal((B, L, C))))
    new, codes, scales = oracle.layer_state_update(fwd, state, P, "bf16", oracle.STALE, True)
    Hp = H // P
    halo = sorted({r for p in range(1, P) for r in (p * Hp - 1, p * Hp)})
    assert len(halo) == 2 * (P - 1)
    want = -np.ones((B, H, W, C))
    want[:, halo] = 1.0
    np.testing.assert_array_equal(new["y_stale"], want)
    # GroupNorm sums: a bit-exact copy of this step's fresh sums
    np.testing.assert_array_equal(new["gn_stats"], fwd["gn_fresh"])
    # K and V refreshed towards the fresh values (not copied, not left alone)
    for name in ("k", "v"):
        got, fresh, old = new[name + "_stale"], fwd[name], state[name + "_stale"]
        assert not np.array_equal(got, fresh) and not np.array_equal(got, old)
        assert np.abs(got - fresh).max() < 0.05 * np.abs(fresh - old).max() + 2 ** -7
    # message order and content: K (B*L*C), V (B*L*C), then per batch and boundary 2*W*C
    n_kv = B * L * C
    assert codes.size == 2 * n_kv + B * (P - 1) * 2 * W * C
    np.testing.assert_array_equal(codes[2 * n_kv:], 127)
    halo_scales = scales[2 * ((n_kv + 127) // 128):]
    np.testing.assert_array_equal(halo_scales, np.float32(2.0) / np.float32(127.0))
    # no refresh (no_sync) leaves every part of the state as it was
    same, c0, s0 = oracle.layer_state_update(fwd, state, P, "bf16", oracle.STALE, False)
    assert c0 is None and s0 is None
    for k in state:
        np.testing.assert_array_equal(same[k], state[k])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_edge_blocks_match_exact_rational_evaluation(dtype):
    """Hand-built blocks at the quantiser's edges: fp32 quotients d/s exactly on a
    half-integer with scales that are not powers of two (and their fp32 neighbours),
    maxima whose rounded scale puts |a/s| just above or below 127, and subnormal scales.
    The oracle's codes, scales and refreshed values equal the rule evaluated with exact
    rationals and one rounding per IEEE operation; a ragged copy of the first blocks
    checks a partial last block too."""
    from tests.refresh_edges import edge_blocks
    fresh, stale, _ = edge_blocks(dtype)
    fresh = np.concatenate([fresh, fresh[:200]])
    stale = np.concatenate([stale, stale[:200]])
    new, codes, scales = oracle.refresh_residual(fresh, stale, dtype)
    en, ec, es = _refresh_exact(fresh, stale, 8 if dtype == "bf16" else 24)
    np.testing.assert_array_equal(codes, ec)
    np.testing.assert_array_equal(scales, es)
    np.testing.assert_array_equal(new, en)
    # the blocks do reach the edges they were built for
    q = (fresh - stale).astype(np.float32)
    blk = q[:(q.size // 128) * 128].reshape(-1, 128)
    s = (np.abs(blk).max(axis=1) / np.float32(127)).astype(np.float32)
    t = (blk / s[:, None]).astype(np.float32)
    assert np.sum(t - np.floor(t) == 0.5) >= 15
    assert np.any(s < np.finfo(np.float32).tiny) and np.all(s > 0)
    assert np.any(np.abs(codes) == 127)
