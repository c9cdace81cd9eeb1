"""GPU parity of the OTIL exchange (dpp_otil_step / dpp_otil_finalize) against the CPU
oracle.  The selection is decided by fp32 block scores on the GPU and fp64 on the CPU:
where the gap between the k-th and (k+1)-th oracle scores exceeds the fp32 error bound
the two selections must be identical, otherwise the GPU's must still be a valid top k.
Given the GPU's selection, views, flags and message are compared bit for bit."""
import math

import numpy as np
import pytest
import torch

import stale_activations_gb300 as dpp
from oracle import otil
from tests.util import np64

pytestmark = pytest.mark.gpu
# fp32 sums over a block of at most a few thousand elements: the cosine is off by far
# less than this, and the +10 unvisited bonus is exact
SCORE_TOL = 1e-4


def _check_selection(sc_row, sel_row, k):
    order = sorted(range(len(sc_row)), key=lambda i: (-sc_row[i], i))
    kth = sc_row[order[k - 1]]
    nxt = sc_row[order[k]] if k < len(order) else -math.inf
    g = set(int(i) for i in sel_row)
    assert len(g) == k and list(sel_row) == sorted(sel_row)
    if kth - nxt > 2 * SCORE_TOL:
        assert g == set(order[:k])
    else:
        assert all(sc_row[i] >= kth - SCORE_TOL for i in g)
        assert all(sc_row[i] <= kth + SCORE_TOL for i in range(len(sc_row)) if i not in g)


@pytest.mark.parametrize("dtype,B,C,H,W,P,bh,bw,k", [
    ("bf16", 2, 4, 128, 128, 4, 8, 32, 4),   # the noise prediction of the pages, K = 16
    ("f32", 1, 4, 32, 32, 2, 4, 8, 3),       # K = 16 per band
    ("bf16", 1, 2, 48, 24, 3, 2, 8, 7),      # K = 24, ragged k
])
def test_otil_exchange_matches_oracle(dtype, B, C, H, W, P, bh, bw, k):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    prm = dpp.otil_params(B, C, H, W, P, bh, bw, k, dpp.BF16 if dtype == "bf16" else dpp.F32)
    K = dpp.otil_blocks(prm)
    assert K == len(otil.sub_blocks(H, W, P, bh, bw))
    g = torch.Generator().manual_seed(H + k)
    x = torch.randn(B, C, H, W, generator=g).to(tdt)
    st = dpp.otil_alloc(prm, x)
    views = np64(st["views"])
    visited = np.zeros((P, K), dtype=np.uint8)
    steps = math.ceil(K / k) + 3
    for s in range(steps):
        noise = torch.randn(B, C, H, W, generator=g) * (0.05 + 0.3 * (s % 2))
        x = (x.float() + noise).to(tdt)
        xd = x.cuda()
        dpp.otil_step(prm, xd, st)
        torch.cuda.synchronize()
        xf = np64(x)
        sc = otil.scores(xf, views, visited, P, bh, bw)
        sel = st["sel"].cpu().numpy().astype(np.int64)
        for p in range(P):
            _check_selection(sc[p], sel[p], k)
        views, visited, msg = otil.apply_selection(xf, views, visited, sel, P, bh, bw)
        np.testing.assert_array_equal(np64(st["views"]), views)
        np.testing.assert_array_equal(st["visited"].cpu().numpy(), visited)
        np.testing.assert_array_equal(np64(st["msg"]), msg)
        if s == math.ceil(K / k) - 1:   # every block sent once within ceil(K/k) steps
            assert visited.all()
    dpp.otil_finalize(prm, xd, st, reset=True)
    torch.cuda.synchronize()
    for r in range(P):
        assert torch.equal(st["views"][r], xd)
    assert not st["visited"].any()
