"""Failure detection without a GPU fault: every wait inside the kernels is bounded.

A test hook (DPP_DEBUG_SKIP_LOAD=<kind>:<i>) makes the TMA producer of every CTA of
one kernel kind leave its i-th load unissued, so the consumers' bounded waits must run
out: the kernel has to report exactly DPP_ERR_TIMEOUT in the device status word, drain
what it issued and return, and the next normal call on the same context must again
match the oracle.  DPP_DEBUG_WAIT_LIMIT shortens the bound so that each case takes
milliseconds."""
import numpy as np
import pytest
import torch

import oracle
import stale_activations_gb300 as dpp
import synth
from tests.util import TOL_BF16, np64, rel_err

pytestmark = pytest.mark.gpu
TIMEOUT = 6  # DPP_ERR_TIMEOUT


def _attention_case(split):
    B, L, heads, P = 1, 1024, 2, 4
    q, kf, vf, ks, vs = synth.attention_inputs(B, L, heads, 64, "bf16", seed=41)
    dev = [t.cuda() for t in (q, kf, vf, ks, vs)]
    o = torch.empty_like(dev[0])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = dpp.stale_kv_attention_split if split else dpp.stale_kv_attention
    fn(*dev, o, heads, P, dev_status=st)
    torch.cuda.synchronize()
    ref = oracle.stale_kv_attention(*(np64(t) for t in (q, kf, vf, ks, vs)), heads, P, "bf16")
    return st.item(), rel_err(np64(o), ref)


@pytest.mark.parametrize("split,step", [(False, 3), (False, 0), (True, 0)])
def test_attention_gives_up_on_a_missing_tile(split, step, monkeypatch):
    """Whole units (8 CTAs of 8 key tiles: a tile missing mid-unit, after MMAs were
    issued, or the first one) and the split schedule (64 CTAs of one key tile each)."""
    monkeypatch.setenv("DPP_DEBUG_WAIT_LIMIT", "2000")
    monkeypatch.setenv("DPP_DEBUG_SKIP_LOAD", f"attn:{step}")
    status, _ = _attention_case(split)
    assert status == TIMEOUT
    monkeypatch.delenv("DPP_DEBUG_SKIP_LOAD")
    monkeypatch.delenv("DPP_DEBUG_WAIT_LIMIT")
    status, err = _attention_case(split)
    assert status == 0 and err < TOL_BF16, err


def _conv_case():
    yf, ys, w = synth.conv_inputs(1, 16, 64, 128, 128, "bf16", seed=1)
    out = torch.empty(1, 16, 64, 128, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dpp.halo_conv3x3(yf.cuda(), ys.cuda(), w.cuda(), out, 4, dev_status=st)
    torch.cuda.synchronize()
    ref = oracle.halo_conv3x3(np64(yf), np64(ys), np64(w), 4, "bf16")
    return st.item(), rel_err(np64(out), ref)


def test_conv_gives_up_on_a_missing_slice(monkeypatch):
    monkeypatch.setenv("DPP_DEBUG_WAIT_LIMIT", "2000")
    monkeypatch.setenv("DPP_DEBUG_SKIP_LOAD", "conv:5")
    status, _ = _conv_case()
    assert status == TIMEOUT
    monkeypatch.delenv("DPP_DEBUG_SKIP_LOAD")
    monkeypatch.delenv("DPP_DEBUG_WAIT_LIMIT")
    status, err = _conv_case()
    assert status == 0 and err < TOL_BF16, err


@pytest.mark.parametrize("kind", ["linear:1", "conv:7", "attn:0"])
def test_layer_step_reports_a_give_up_and_recovers(kind, monkeypatch):
    """Through the layer step: the projections' GEMM (after its first K slice), the conv
    (after seven slices) or the attention (its first key tile) gives up; the step's status word says so.  The next step on the same
    workspace and context, with the hook unset, matches the oracle again."""
    cfg = synth.LayerConfig("small", B=1, H=16, W=64, C=128, P=4, G=8, heads=2, head_dim=64,
                            dtype="bf16")
    wts = synth.layer_weights(cfg, seed=3, affine=True)
    x, x_prev = synth.layer_inputs(cfg, seed=3)
    prm = dpp.make_params(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G, cfg.heads, dpp.BF16)
    wd = {k: t.cuda() for k, t in wts.items()}
    out = torch.empty(cfg.B, cfg.H, cfg.W, cfg.C, dtype=torch.bfloat16, device="cuda")
    state, ws = dpp.alloc_layer(prm)
    monkeypatch.setenv("DPP_DEBUG_WAIT_LIMIT", "2000")
    monkeypatch.setenv("DPP_DEBUG_SKIP_LOAD", kind)
    dpp.patch_layer_step(prm, wd, state, x_prev.cuda(), out, dpp.SYNC, ws)
    assert dpp.read_device_status(ws) == TIMEOUT
    monkeypatch.delenv("DPP_DEBUG_SKIP_LOAD")
    monkeypatch.delenv("DPP_DEBUG_WAIT_LIMIT")
    state = dpp.alloc_layer(prm)[0]  # the failed step left the old state incomplete
    dpp.patch_layer_step(prm, wd, state, x_prev.cuda(), out, dpp.SYNC, ws)
    assert dpp.read_device_status(ws) == 0
    wn = {k: np64(v) for k, v in wts.items()}
    st0 = oracle.empty_state(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G)
    fwd, _, _, _ = oracle.patch_layer_step(np64(x_prev), st0, wn, cfg.P, cfg.G, cfg.heads,
                                           cfg.eps, "bf16", oracle.SYNC)
    err = rel_err(np64(out), fwd["out"])
    assert err < 2e-3, err
