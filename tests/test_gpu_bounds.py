"""The index-checking build (-DDPP_DEBUG_BOUNDS, the stand-in for a memory checker): every
kernel checks each global-memory index it computes against the extent that the call's
shapes give its tensor, skips an access outside it and records the first such index.
Each entry point runs through both libraries on shapes that reach every code path (the
layer step plain, with the fused GroupNorm, with the second state set and the fused
refresh, on maps whose stale-V maxima come from the conv's spare CTAs, its epilogue warps
or the GroupNorm apply, and in fp32; the standalone attention with whole and cut units and
ragged patches; the conv's three pixel tilings; ragged refresh segments; the OTIL
exchange).  The checked build must record nothing and produce the same bytes as
the normal one: the checks change no arithmetic."""
import pytest
import torch

import stale_activations_gb300 as dpp
import synth
from stale_activations_gb300 import build as _build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    rel = dpp.load()
    bnd = dpp.open_library(_build.build_library(bounds=True))
    assert dpp.debug_bounds()[0] == 8  # DPP_ERR_UNSUPPORTED: no checks in the normal build
    with dpp.using(bnd):
        rc, rec = dpp.debug_bounds(reset=True)
        assert (rc, rec) == (0, (0, 0, 0, 0))
    return rel, bnd


def _both(libs, run):
    """run() -> dict of result tensors, once with each library; returns both results and
    the checked build's record."""
    rel, bnd = libs
    with dpp.using(rel):
        a = {k: v.detach().cpu().clone() for k, v in run().items()}
    with dpp.using(bnd):
        dpp.debug_bounds(reset=True)
        b = {k: v.detach().cpu().clone() for k, v in run().items()}
        torch.cuda.synchronize()
        rc, rec = dpp.debug_bounds(reset=True)
    return a, b, rc, rec


def _check(libs, run):
    a, b, rc, rec = _both(libs, run)
    assert (rc, rec) == (0, (0, 0, 0, 0)), f"index outside its tensor: {rec}"
    for k in a:
        assert torch.equal(a[k], b[k]), k


def _layer_run(cfg, fuse_gn=False, dbuf=False, frx=False, steps=2):
    wts = synth.layer_weights(cfg, seed=3, affine=True)
    x, x_prev = synth.layer_inputs(cfg, seed=3)

    def run():
        prm = dpp.make_params(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G, cfg.heads,
                              dpp.BF16 if cfg.dtype == "bf16" else dpp.F32,
                              fuse_gn=fuse_gn, fuse_refresh=frx)
        state, ws = dpp.alloc_layer(prm, double_buffer=dbuf)
        wd = {k: v.cuda() for k, v in wts.items()}
        out = torch.empty(cfg.B, cfg.H, cfg.W, cfg.C, dtype=x.dtype, device="cuda")
        res = {}
        for s in range(steps):
            dpp.patch_layer_step(prm, wd, state, (x_prev if s == 0 else x).cuda(), out,
                                 dpp.SYNC if s == 0 else dpp.STALE, ws)
            assert dpp.read_device_status(ws) == 0
            if dbuf:
                dpp.swap_state(state)
            res[f"out{s}"] = out.clone()
        res.update({k: v for k, v in state.items() if not k.endswith("_next")})
        return res
    return run


LAYERS = {
    "bf16": synth.LayerConfig("b", B=1, H=16, W=64, C=128, P=4, G=8, heads=2, head_dim=64,
                              dtype="bf16"),
    "bf16_conv_epilogue_vmax": synth.LayerConfig("e", B=1, H=256, W=128, C=128, P=4, G=8,
                                                 heads=2, head_dim=64, dtype="bf16"),
    "bf16_groupnorm_vmax": synth.LayerConfig("g", B=1, H=320, W=128, C=128, P=4, G=8,
                                             heads=2, head_dim=64, dtype="bf16"),
    "bf16_narrow_b2": synth.LayerConfig("n", B=2, H=32, W=16, C=128, P=4, G=8, heads=2,
                                        head_dim=64, dtype="bf16"),
    "bf16_w240": synth.LayerConfig("w", B=1, H=16, W=240, C=128, P=4, G=8, heads=2,
                                   head_dim=64, dtype="bf16"),
    "f32": synth.LayerConfig("f", B=1, H=32, W=32, C=64, P=2, G=8, heads=1, head_dim=64,
                             dtype="f32"),
}


@pytest.mark.parametrize("name", list(LAYERS))
def test_bounds_layer(libs, name):
    _check(libs, _layer_run(LAYERS[name]))


@pytest.mark.parametrize("fuse_gn,dbuf,frx", [(True, False, False), (False, True, True),
                                              (True, True, True)])
def test_bounds_layer_fused_paths(libs, fuse_gn, dbuf, frx):
    _check(libs, _layer_run(LAYERS["bf16"], fuse_gn=fuse_gn, dbuf=dbuf, frx=frx))


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("B,L,heads,P,scale", [
    (1, 1024, 2, 4, 1.0),      # every unit cut into pieces (split)
    (2, 960, 1, 8, 1.0),       # 120-token patches: ragged query tiles
    (3, 1984, 3, 8, 1.0),      # partial last key tile
    (1, 1024, 2, 4, 3.0e4),    # V beyond fp16's range: scaled by a power of two
])
def test_bounds_attention(libs, split, B, L, heads, P, scale):
    q, kf, vf, ks, vs = synth.attention_inputs(B, L, heads, 64, "bf16", seed=L + heads)
    vf, vs = (vf.float() * scale).to(vf.dtype), (vs.float() * scale).to(vs.dtype)

    def run():
        o = torch.empty_like(q, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        f = dpp.stale_kv_attention_split if split else dpp.stale_kv_attention
        f(q.cuda(), kf.cuda(), vf.cuda(), ks.cuda(), vs.cuda(), o, heads, P, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        return {"o": o}
    _check(libs, run)


@pytest.mark.parametrize("dtype,B,H,W,Cin,Cout,P", [
    ("bf16", 2, 16, 64, 128, 128, 4),    # whole rows per tile
    ("bf16", 2, 16, 240, 64, 128, 4),    # tiles of 120 pixels of one row (padded rows)
    ("bf16", 1, 12, 96, 128, 128, 3),    # row segments that wrap across rows
    ("bf16", 1, 16, 64, 256, 320, 2),    # 128 x 320 tiles
    ("f32", 1, 6, 5, 3, 7, 3),           # SIMT path, ragged sizes
])
def test_bounds_conv(libs, dtype, B, H, W, Cin, Cout, P):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(H * W + Cin)
    yf = torch.randn(B, H, W, Cin, generator=g).to(tdt)
    ys = torch.randn(B, H, W, Cin, generator=g).to(tdt)
    w = (0.05 * torch.randn(Cout, 3, 3, Cin, generator=g)).to(tdt)

    def run():
        out = torch.empty(B, H, W, Cout, dtype=tdt, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        dpp.halo_conv3x3(yf.cuda(), ys.cuda(), w.cuda(), out, P, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        return {"out": out}
    _check(libs, run)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [128 * 50 + 37, 128 * 7 + 5, 3])  # ragged last blocks
def test_bounds_refresh_and_apply(libs, dtype, n):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(n)
    fresh = torch.randn(n, generator=g).to(tdt)
    stale = (fresh.float() + 0.1 * torch.randn(n, generator=g)).to(tdt)

    def run():
        f, s = fresh.cuda(), stale.clone().cuda()
        copy = stale.clone().cuda()
        codes = torch.zeros(n, dtype=torch.int8, device="cuda")
        scales = torch.zeros((n + 127) // 128, device="cuda")
        dpp.refresh_residual(f, s, codes, scales)
        dpp.apply_residual(codes, scales, copy)
        torch.cuda.synchronize()
        return {"stale": s, "codes": codes, "scales": scales, "copy": copy}
    _check(libs, run)


@pytest.mark.parametrize("dtype,B,C,H,W,P,bh,bw,k", [
    ("bf16", 2, 4, 128, 128, 4, 8, 32, 4),
    ("bf16", 1, 2, 48, 24, 3, 2, 8, 7),
    ("f32", 1, 4, 32, 32, 2, 4, 8, 3),
])
def test_bounds_otil(libs, dtype, B, C, H, W, P, bh, bw, k):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(B * H + k)
    xs = [torch.randn(B, C, H, W, generator=g).to(tdt) for _ in range(4)]

    def run():
        prm = dpp.otil_params(B, C, H, W, P, bh, bw, k, dpp.BF16 if dtype == "bf16" else dpp.F32)
        st = dpp.otil_alloc(prm, xs[0])
        res = {}
        for i, x in enumerate(xs[1:]):
            dpp.otil_step(prm, x.cuda(), st)
            res[f"msg{i}"] = st["msg"].clone()
            res[f"sel{i}"] = st["sel"].clone()
        dpp.otil_finalize(prm, xs[-1].cuda(), st, reset=True)
        torch.cuda.synchronize()
        res.update(views=st["views"], visited=st["visited"])
        return res
    _check(libs, run)
