"""patch_layer_step_noalloc: the layer step for callers that cannot allocate
device memory when they run a layer (a plugin whose host framework owns every
byte of device memory through its own allocator, a latency-critical loop where
cudaMalloc's implicit synchronisation is not allowed).

It takes its workspace from a fixed 80 MiB device array inside the library, so
its results must match patch_layer_step with a caller-allocated workspace, call
after call.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import stale_activations_gb300 as dpp
import synth
from tests.util import np64, rel_err


def _fresh_state_pair(prm):
    a, ws = dpp.alloc_layer(prm)
    b, _ = dpp.alloc_layer(prm)
    return a, b, ws


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cfg = synth.SDXL1024_MID  # the bench workload: about 71 MiB of workspace
    prm = dpp.make_params(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G, cfg.heads, dpp.BF16,
                          refresh=True, eps=cfg.eps)
    wts = {k: v.cuda() for k, v in synth.layer_weights(cfg, seed=5, affine=True).items()}
    x, x_prev = (t.cuda() for t in synth.layer_inputs(cfg, seed=5))
    st_ref, st_na, ws = _fresh_state_pair(prm)
    out_ref = torch.empty_like(x)
    out_na = torch.full_like(x, float("nan"))
    for mode, inp in ((dpp.SYNC, x_prev), (dpp.STALE, x)):
        dpp.patch_layer_step(prm, wts, st_ref, inp, out_ref, mode, ws)
        dpp.patch_layer_step_noalloc(prm, wts, st_na, inp, out_na, mode)
        torch.cuda.synchronize()
        assert dpp.read_device_status(ws) == 0
        assert dpp.noalloc_read_status() == 0
        # the same deterministic kernels on the same bytes: equal bit for bit (a byte of
        # the shared scratch that a call read before writing would show here)
        assert torch.equal(out_na, out_ref), rel_err(np64(out_na), np64(out_ref))
        for k in ("k_stale", "v_stale", "y_stale", "gn_stats"):
            assert torch.equal(st_na[k], st_ref[k]), k
        if mode == dpp.STALE:
            assert torch.equal(st_na["codes"], st_ref["codes"])
            assert torch.equal(st_na["scales"], st_ref["scales"])


def test_noalloc_rejects_layers_beyond_the_scratch():
    lib = dpp.load(build_if_missing=True)
    prm = dpp.make_params(2, 128, 128, 640, 4, 32, 10, dpp.BF16)  # ~240 MiB of workspace
    assert dpp.workspace_size(prm) > 80 * 1024 * 1024
    rc = lib.patch_layer_step_noalloc(ctypes.byref(prm), ctypes.byref(dpp.LayerWeights()),
                                      ctypes.byref(dpp.LayerState()), ctypes.c_void_p(256),
                                      ctypes.c_void_p(256), dpp.STALE, None)
    assert rc == 10
    assert "no-alloc" in dpp.status_string(rc)
