"""Pins of the OTIL selective-transmit oracle ("OTIL for SDXL on 4x L40S", What is
implemented where / Self-tests): the dissimilarity against an independent cosine, the
polling rule on hand-worked scores, coverage within ceil(K/k) steps, and the
reconstruction invariants (own slice exact, remote positions received or stale, never a
blend, k blocks per peer, exact finalize)."""
import math

import numpy as np
import pytest

from oracle import otil

RNG = np.random.default_rng(7)


def test_dissimilarity_closed_forms_and_scipy():
    scipy_dist = pytest.importorskip("scipy.spatial.distance")
    x = RNG.standard_normal(300)
    assert otil.dissimilarity(x, x) == pytest.approx(0.0, abs=1e-14)
    assert otil.dissimilarity(x, 3.5 * x) == pytest.approx(0.0, abs=1e-14)
    assert otil.dissimilarity(x, -x) == pytest.approx(2.0, abs=1e-14)
    e1, e2 = np.eye(4)[0], np.eye(4)[1]
    assert otil.dissimilarity(e1, e2) == 1.0
    assert otil.dissimilarity(np.zeros(5), np.ones(5)) == 1.0       # cos taken as 0
    for _ in range(20):
        a, b = RNG.standard_normal(64), RNG.standard_normal(64)
        assert otil.dissimilarity(a, b) == pytest.approx(scipy_dist.cosine(a, b), abs=1e-12)


def test_select_top_k_hand_worked():
    # unvisited blocks carry +10; ties go to the lower index; output in index order
    s = np.array([1.0, 11.0, 11.0, 0.5, 12.0, 1.0])
    np.testing.assert_array_equal(otil.select_top_k(s, 2), [1, 4])
    np.testing.assert_array_equal(otil.select_top_k(s, 3), [1, 2, 4])
    np.testing.assert_array_equal(otil.select_top_k(s, 4), [0, 1, 2, 4])   # 1.0 tie -> 0
    np.testing.assert_array_equal(otil.select_top_k(np.zeros(5), 2), [0, 1])


def _setup(B=2, C=4, H=32, W=32, P=4, seed=0):
    rng = np.random.default_rng(seed)
    x0 = rng.standard_normal((B, C, H, W)).astype(np.float32)
    views = np.broadcast_to(x0, (P, B, C, H, W)).copy()
    return rng, x0, views


@pytest.mark.parametrize("bh,bw,k", [(4, 8, 3), (8, 16, 1), (2, 32, 5)])
def test_coverage_within_ceil_K_over_k_steps(bh, bw, k):
    B, C, H, W, P = 2, 4, 32, 32, 4
    rng, x, views = _setup(B, C, H, W, P)
    K = len(otil.sub_blocks(H, W, P, bh, bw))
    visited = np.zeros((P, K), dtype=np.uint8)
    sent = [set() for _ in range(P)]
    for step in range(math.ceil(K / k)):
        x = x + 0.1 * rng.standard_normal(x.shape).astype(np.float32)
        views, visited, sel, _ = otil.exchange_step(x, views, visited, P, bh, bw, k)
        for p in range(P):
            new = set(int(i) for i in sel[p])
            if len(sent[p]) + k <= K:      # unvisited first: no repeat before full coverage
                assert not (new & sent[p])
            sent[p] |= new
    assert all(len(s) == K for s in sent)
    assert visited.all()


def test_reconstruction_invariants_over_steps():
    """Own slice exact; each remote position keeps its old value or takes this step's
    fresh value of a selected sub-block (never a blend); k blocks from each peer."""
    B, C, H, W, P, bh, bw, k = 2, 4, 32, 32, 4, 4, 8, 3
    rng, x, views = _setup(B, C, H, W, P, seed=3)
    K = len(otil.sub_blocks(H, W, P, bh, bw))
    visited = np.zeros((P, K), dtype=np.uint8)
    Hp = H // P
    for step in range(7):
        x = x + 0.2 * rng.standard_normal(x.shape).astype(np.float32)
        old = views.copy()
        views, visited, sel, msg = otil.exchange_step(x, views, visited, P, bh, bw, k)
        assert sel.shape == (P, k) and all(len(set(r)) == k for r in sel)
        for r in range(P):
            np.testing.assert_array_equal(views[r][:, :, r * Hp:(r + 1) * Hp],
                                          x[:, :, r * Hp:(r + 1) * Hp])
            for p in range(P):
                if p == r:
                    continue
                band_new = views[r][:, :, p * Hp:(p + 1) * Hp]
                band_old = old[r][:, :, p * Hp:(p + 1) * Hp]
                band_fr = x[:, :, p * Hp:(p + 1) * Hp]
                assert np.all((band_new == band_old) | (band_new == band_fr))
                for i in range(K):   # exactly the selected blocks took fresh values
                    nb = otil.block_view(views[r], p, i, P, bh, bw)
                    fb = otil.block_view(x, p, i, P, bh, bw)
                    if i in sel[p]:
                        np.testing.assert_array_equal(nb, fb)
                    else:
                        np.testing.assert_array_equal(nb, otil.block_view(old[r], p, i, P, bh,
                                                                          bw))
        for p in range(P):
            for j, i in enumerate(sel[p]):
                np.testing.assert_array_equal(msg[p, j], otil.block_view(x, p, int(i), P, bh, bw))


def test_finalize_is_exact_and_reset_clears_flags():
    B, C, H, W, P, bh, bw, k = 1, 4, 16, 16, 2, 4, 4, 2
    rng, x, views = _setup(B, C, H, W, P, seed=5)
    K = len(otil.sub_blocks(H, W, P, bh, bw))
    visited = np.zeros((P, K), dtype=np.uint8)
    x = x + rng.standard_normal(x.shape).astype(np.float32)
    views, visited, _, _ = otil.exchange_step(x, views, visited, P, bh, bw, k)
    v2, f2 = otil.finalize(x, views, visited, reset=False)
    for r in range(P):
        np.testing.assert_array_equal(v2[r], x)
    np.testing.assert_array_equal(f2, visited)
    _, f3 = otil.finalize(x, views, visited, reset=True)
    assert not f3.any()


def test_most_changed_block_goes_first_once_all_visited():
    """With every block visited, the one that changed most (in angle) is sent."""
    B, C, H, W, P, bh, bw = 1, 2, 16, 8, 2, 4, 4
    rng, x, views = _setup(B, C, H, W, P, seed=9)
    K = len(otil.sub_blocks(H, W, P, bh, bw))
    visited = np.ones((P, K), dtype=np.uint8)
    y = x.copy()
    otil.block_view(y, 0, 2, P, bh, bw)[...] *= -1.0            # block 2 of band 0 flips
    otil.block_view(y, 1, 1, P, bh, bw)[...] += 0.3 * rng.standard_normal((B, C, bh, bw))
    _, _, sel, _ = otil.exchange_step(y.astype(np.float32), views, visited, P, bh, bw, 1)
    assert sel[0, 0] == 2 and sel[1, 0] == 1
