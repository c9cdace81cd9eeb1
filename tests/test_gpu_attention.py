"""GPU parity: stale_kv_attention against the CPU oracle; the fresh/stale splice
range pinned bit-exactly with a uniform-softmax sentinel."""
import numpy as np
import pytest
import torch

import oracle
import stale_activations_gb300 as dpp
import synth
from tests.util import TOL_BF16, TOL_F32, np64, rel_err

pytestmark = pytest.mark.gpu


def _attn_gpu(q, kf, vf, ks, vs, heads, P, split=False):
    """split=False: stale_kv_attention (whole units per CTA); split=True:
    stale_kv_attention_split (the last units cut into key-tile runs and merged)."""
    o = torch.empty_like(q, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (q.cuda(), kf.cuda(), vf.cuda(), ks.cuda(), vs.cuda(), o, heads, P)
    if split:
        dpp.stale_kv_attention_split(*args, dev_status=st)
    else:
        dpp.stale_kv_attention(*args, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return o


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("dtype,B,L,heads,P", [
    ("bf16", 1, 1024, 2, 4),    # 8 units of 8 key tiles: split, every unit in 8 pieces
    ("bf16", 2, 960, 1, 8),     # 120-token patches: ragged query tiles, straddling key tiles
    ("bf16", 1, 4096, 10, 4),   # the SDXL-1024 mid-level attention (160 units)
    ("bf16", 3, 1984, 3, 8),    # 248-token patches, partial last key tile; 72 units, all cut
    ("f32", 1, 1024, 1, 2),
    ("f32", 1, 96, 2, 3),
])
def test_attention_matches_oracle(dtype, B, L, heads, P, split):
    q, kf, vf, ks, vs = synth.attention_inputs(B, L, heads, 64, dtype, seed=L + heads)
    o = _attn_gpu(q, kf, vf, ks, vs, heads, P, split)
    ref = oracle.stale_kv_attention(*(np64(t) for t in (q, kf, vf, ks, vs)), heads, P, dtype)
    assert rel_err(np64(o), ref) < (TOL_BF16 if dtype == "bf16" else TOL_F32)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("L,P", [(1024, 4), (960, 8), (14400, 8)])
def test_attention_splice_sentinel_bitexact(L, P, split):
    """Q = 0 gives a uniform softmax; V_fresh = +1 and V_stale = -1 then give
    (2*Lp - L)/L in every output (exact in bf16 for these sizes).  L/P = 1800 makes
    the splice granularity 8 rows (sub-boxes of 8 keys).  With the split schedule a
    piece's mean of V is rounded to fp16 (error < 2^-11), far below half a bf16 step
    of these exactly representable results, so they stay exact."""
    heads = 2
    C = heads * 64
    q = torch.zeros(1, L, C, dtype=torch.bfloat16)
    k = synth.attention_inputs(1, L, heads, 64, "bf16", seed=3)[1]
    vf = torch.ones(1, L, C, dtype=torch.bfloat16)
    vs = -torch.ones(1, L, C, dtype=torch.bfloat16)
    o = _attn_gpu(q, k, vf, k, vs, heads, P, split).float().cpu()
    Lp = L // P
    exp = (2 * Lp - L) / L
    np.testing.assert_array_equal(o.numpy(), float(torch.tensor(exp).to(torch.bfloat16)))


@pytest.mark.parametrize("split", [False, True])
def test_attention_sdxl3840_sampled_rows(split):
    """The SDXL-3840 attention level: B=2, L=57600, 10 heads, P=8 (7200-token
    patches).  Sampled query rows (patch edges, tile edges, interiors) vs the oracle;
    with the split schedule the last 80 units (batch 1, head 9, patches 5-7) are the
    cut ones, so rows of patches 5-7 are sampled too."""
    B, L, heads, P = 2, 57600, 10, 8
    q, kf, vf, ks, vs = synth.attention_inputs(B, L, heads, 64, "bf16", seed=0)
    o = _attn_gpu(q, kf, vf, ks, vs, heads, P, split)
    rows = np.array([0, 127, 128, 7199, 7200, 7327, 7328, 14399, 30000, 37800, 43455, 50399,
                     50400, 57599])
    ref = oracle.stale_kv_attention(*(np64(t) for t in (q, kf, vf, ks, vs)), heads, P, "bf16",
                                    rows=rows)
    assert rel_err(np64(o)[:, rows], ref) < TOL_BF16


@pytest.mark.parametrize("rows", ["all", "alternating"])
@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("P", [1, 2])
def test_attention_late_large_scores_rescale(P, split, rows):
    """Scores in a late key tile far above those of the first tiles: the running
    reference maximum must move (O and the row sum rescaled, P recomputed) and the
    result still matches the oracle.  rows="alternating": the jump happens only for
    every other query row (the others see the same keys as very low scores), so rows of
    one warp take different paths."""
    B, L, heads = 1, 1024, 1
    g = torch.Generator().manual_seed(11)
    q = (0.5 + 0.05 * torch.randn(B, L, 64, generator=g))
    if rows == "alternating":
        q[:, 1::2] *= -1.0
    q = q.to(torch.bfloat16)
    k = (0.1 * torch.randn(B, L, 64, generator=g))
    k[:, 640:768] += 3.0          # tile 5: scores ~ 0.5*3*64/8 = 12 above the rest
    k[:, 900:910] += 6.0          # a few even larger keys later on
    k = k.to(torch.bfloat16)
    v = torch.randn(B, L, 64, generator=g).to(torch.bfloat16)
    vs = (v.float() + 0.05 * torch.randn(B, L, 64, generator=g)).to(torch.bfloat16)
    o = _attn_gpu(q, k, v, k, vs, heads, P, split)
    ref = oracle.stale_kv_attention(*(np64(t) for t in (q, k, v, k, vs)), heads, P, "bf16")
    assert rel_err(np64(o), ref) < TOL_BF16


def test_attention_split_deterministic_and_close_to_whole_units():
    """The split schedule merges the pieces of a unit in a fixed order: two runs give
    identical bytes.  Against the whole-unit schedule the fp32 results differ only by
    the fp16 rounding of the pieces (2^-11 of |V|) and the order of the sums; after
    the bf16 rounding many outputs sit one step apart, so the two are compared
    normwise at the bf16 tolerance (each is also checked against the oracle above)."""
    B, L, heads, P = 1, 4096, 10, 4
    q, kf, vf, ks, vs = synth.attention_inputs(B, L, heads, 64, "bf16", seed=5)
    o1 = _attn_gpu(q, kf, vf, ks, vs, heads, P, True)
    o2 = _attn_gpu(q, kf, vf, ks, vs, heads, P, True)
    o0 = _attn_gpu(q, kf, vf, ks, vs, heads, P, False)
    assert torch.equal(o1, o2)
    assert rel_err(np64(o1), np64(o0)) < TOL_BF16


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("vscale", [1e4, 1e-5, 1e6, 1e-30, "mixed"])
def test_attention_v_outside_fp16_range(vscale, split):
    """P.V runs in fp16, whose full-precision range is [2^-14, 65504].  V at scale 1e4
    (max near 4.5e4), 1e6 (beyond fp16), 1e-5 and 1e-30 (fp16 subnormal or zero without
    scaling), and per-head mixtures of those, all within the bf16 bound: the kernel
    scales V by a power of two per (batch, head) and removes it from O."""
    B, L, heads, P = 2, 1024, 4, 4
    q, kf, vf, ks, vs = synth.attention_inputs(B, L, heads, 64, "bf16", seed=77)
    if vscale == "mixed":
        f = torch.tensor([1e4, 1e-5, 1.0, 3e5], dtype=torch.float32).repeat_interleave(64)
    else:
        f = torch.full((heads * 64,), float(vscale))
    vf = (vf.float() * f).to(torch.bfloat16)
    vs = (vs.float() * f).to(torch.bfloat16)
    assert torch.isfinite(vf.float()).all() and vf.float().abs().max() > 0
    o = _attn_gpu(q, kf, vf, ks, vs, heads, P, split)
    ref = oracle.stale_kv_attention(*(np64(t) for t in (q, kf, vf, ks, vs)), heads, P, "bf16")
    for h in range(heads):  # each head on its own scale
        cs = slice(h * 64, (h + 1) * 64)
        err = rel_err(np64(o)[..., cs], ref[..., cs])
        assert err < TOL_BF16, (h, err)
