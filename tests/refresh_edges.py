"""Hand-built refresh blocks at the quantiser's edges (test inputs only; no expected
values here -- those come from the oracle and, on the CPU, from an exact rational
evaluation of the rule).

The rule of each 128-element block is s = a/127 with a = max|d|, q = rint(d/s) with
ties to even, clamped to +-127.  Inputs that a random draw almost never produces:

  * ties: elements whose fp32 quotient d/s is exactly k + 1/2, with a scale s that is
    not a power of two (so 1/s is not exact), and the fp32 neighbours of such d,
    whose quotients sit within an ulp of the half-integer;
  * clamp edge: several elements at +-a, where the rounded scale makes |a/s| a hair
    above or below 127;
  * scales just above and just below 2^-96, with ties (a kernel may form the quotient
    differently on the two sides of such a threshold);
  * subnormal scales: a block maximum so small that a/127 is an fp32 subnormal, with
    ties constructed there too.

For bf16 storage the deltas are formed as f32(fresh) - f32(stale) from two bf16 values
of different magnitude, which gives deltas with more than bf16's 8 significant bits.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def _bf16_grid(lo: float, hi: float) -> np.ndarray:
    """Every positive bf16 value in [lo, hi] (as float32)."""
    u0 = np.array([lo], dtype=np.float32).view(np.uint32)[0] >> 16
    u1 = np.array([hi], dtype=np.float32).view(np.uint32)[0] >> 16
    u = np.arange(u0, u1 + 1, dtype=np.uint32) << 16
    return u.view(np.float32)


def _bf16_round(x) -> np.ndarray:
    """Round-to-nearest-even to bf16 (float32 in, float32 out)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def _tie_pairs_f32(s: np.float32, ks, rng):
    """fp32 deltas d with fl(d / s) == k + 1/2 exactly, plus each one's two fp32
    neighbours; returns (fresh, stale) with stale = 0."""
    out = []
    for k in ks:
        target = F32(k + 0.5)
        d0 = F32(target * s)
        cands = [d0]
        for direction in (np.inf, -np.inf):
            d = d0
            for _ in range(64):
                d = np.nextafter(d, F32(direction), dtype=np.float32)
                cands.append(d)
        hit = [d for d in cands if F32(d / s) == target]
        if not hit:
            continue
        d = hit[0]
        out += [d, np.nextafter(d, F32(np.inf), dtype=np.float32),
                np.nextafter(d, F32(-np.inf), dtype=np.float32)]
    out = np.array(out, dtype=np.float32)
    return out, np.zeros_like(out)


def _tie_pairs_bf16(s: np.float32, ks, rng):
    """bf16 pairs (f, st) with fl(fl(f - st) / s) == k + 1/2 exactly: f runs over the
    bf16 values next to (k + 1/2) s and st over small bf16 values of both signs."""
    fr, st = [], []
    for k in ks:
        target = F32(k + 0.5)
        mag = abs(float(target * s))
        f0 = _bf16_round(F32(target * s))[()]
        u0 = np.array([f0], dtype=np.float32).view(np.uint32)[0]
        fs = (np.arange(-2, 3, dtype=np.int64) * 0x10000 + int(u0)).astype(np.uint32)
        small = _bf16_grid(mag * 2.0 ** -24, mag * 2.0 ** -5)
        small = np.concatenate([small, -small]).astype(np.float32)
        for f in fs.view(np.float32):
            d = (F32(f) - small).astype(np.float32)
            qq = (d / s).astype(np.float32)
            ok = np.nonzero(qq == target)[0]
            if ok.size:
                j = ok[rng.integers(ok.size)]
                fr.append(f)
                st.append(small[j])
                # and the candidates whose quotients lie closest above and below it
                for side in (qq > target, qq < target):
                    idx = np.nonzero(side)[0]
                    if idx.size:
                        jj = idx[np.argmin(np.abs(qq[idx] - target))]
                        fr.append(f)
                        st.append(small[jj])
                break
    return np.array(fr, dtype=np.float32), np.array(st, dtype=np.float32)


def _block(maxval: float, fr_extra, st_extra, rng, dtype, neg_max=False, n_max=1):
    """One block: n_max elements at +-maxval (fresh = +-maxval, stale = 0), the given
    pairs, the rest random deltas strictly inside (-maxval, maxval)."""
    fr = np.zeros(128, dtype=np.float32)
    st = np.zeros(128, dtype=np.float32)
    m = F32(maxval)
    for i in range(n_max):
        fr[i] = -m if (i % 2 == 0) == neg_max else m
    k = min(len(fr_extra), 128 - n_max)
    fr[n_max:n_max + k] = fr_extra[:k]
    st[n_max:n_max + k] = st_extra[:k]
    rest = 128 - n_max - k
    r = (rng.uniform(-0.9, 0.9, rest) * float(m)).astype(np.float32)
    if dtype == "bf16":
        r = _bf16_round(r)
    fr[n_max + k:] = r
    return fr, st


def edge_blocks(dtype: str, seed: int = 0):
    """(fresh, stale) as float64 arrays of whole 128-element blocks (values exactly
    representable in ``dtype``), and a short description of each block."""
    rng = np.random.default_rng(seed)
    blocks, what = [], []
    ks = [-127, -100, -64, -3, -1, 0, 1, 2, 5, 33, 63, 64, 100, 125, 126]
    # ties with scales that are not powers of two; block maxima exactly representable
    for amax in (3.0, 5.0, 0.75, 100.0, 1.0 / 3.0 if dtype == "f32" else 0.3359375, 7.0e-3):
        a = F32(amax) if dtype == "f32" else _bf16_round(F32(amax))[()]
        s = F32(a / F32(127.0))
        assert s != 0 and (s.view(np.uint32) & 0x7FFFFF) != 0, "scale is a power of two"
        pick = _tie_pairs_f32 if dtype == "f32" else _tie_pairs_bf16
        fr, st = pick(s, ks, rng)
        assert fr.size > 0, f"no tie found for a={a}"
        blocks.append(_block(a, fr, st, rng, dtype))
        what.append(f"ties, a={float(a):.6g}")
    # clamp edge: |a/s| just above and just below 127 (several elements at +-a)
    found = {True: 0, False: 0}
    for a in _bf16_grid(1.0, 4.0)[::3]:
        s = F32(a / F32(127.0))
        above = F32(a / s) > F32(127.0)
        if found[bool(above)] < 2:
            found[bool(above)] += 1
            blocks.append(_block(a, [], [], rng, dtype, neg_max=bool(found[bool(above)] % 2),
                                 n_max=6))
            what.append(f"clamp edge, a/s {'>' if above else '<='} 127, a={float(a):.6g}")
        if min(found.values()) >= 2:
            break
    assert min(found.values()) >= 1
    # scales just above and just below 2^-96 (not powers of two), with ties
    t96 = F32(2.0 ** -96)
    side = {True: None, False: None}
    for a in _bf16_grid(float(F32(120.0) * t96), float(F32(134.0) * t96)):
        s = F32(a / F32(127.0))
        if (s.view(np.uint32) & 0x7FFFFF) == 0:
            continue
        key = bool(s >= t96)
        if side[key] is None or abs(float(s) - float(t96)) < abs(float(side[key][1]) - float(t96)):
            side[key] = (a, s)
    for key in (True, False):
        a, s = side[key]
        fr, st = _tie_pairs_f32(s, ks, rng) if dtype == "f32" else _tie_pairs_bf16(s, ks, rng)
        assert fr.size > 0
        blocks.append(_block(a, fr, st, rng, dtype))
        what.append(f"scale {'>=' if key else '<'} 2^-96, a={float(a):.6g}, {fr.size} tie elements")
    # subnormal scales (a / 127 below FLT_MIN), with ties constructed there too
    for amax in (1.0e-37, 3.0e-38, 1.0e-36):
        a = F32(amax) if dtype == "f32" else _bf16_round(F32(amax))[()]
        s = F32(a / F32(127.0))
        assert 0 < s < np.finfo(np.float32).tiny
        fr, st = _tie_pairs_f32(s, ks, rng) if dtype == "f32" else _tie_pairs_bf16(s, ks, rng)
        blocks.append(_block(a, fr, st, rng, dtype))
        what.append(f"subnormal scale, a={float(a):.3g}, {fr.size} tie elements")
    fresh = np.concatenate([b[0] for b in blocks]).astype(np.float64)
    stale = np.concatenate([b[1] for b in blocks]).astype(np.float64)
    if dtype == "bf16":
        assert np.array_equal(_bf16_round(fresh.astype(np.float32)), fresh.astype(np.float32))
        assert np.array_equal(_bf16_round(stale.astype(np.float32)), stale.astype(np.float32))
    return fresh, stale, what
