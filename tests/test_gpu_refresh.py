"""GPU parity: refresh_residual against the CPU oracle, bit-exact (codes, scales
and the refreshed buffer), at small sizes with ragged tails and at the full
refresh-sweep size (sampled blocks)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import stale_activations_gb300 as dpp
import synth
from tests.util import np64

pytestmark = pytest.mark.gpu
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _run_gpu(fresh, stale):
    n = fresh.numel()
    f, s = fresh.cuda(), stale.clone().cuda()
    codes = torch.full((max(n, 1),), 99, dtype=torch.int8, device="cuda")[:n]
    scales = torch.full((max((n + 127) // 128, 1),), -1.0, device="cuda")[:(n + 127) // 128]
    dpp.refresh_residual(f, s, codes, scales)
    torch.cuda.synchronize()
    return s, codes, scales


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [1, 5, 127, 128, 129, 1000, 128 * 997 + 77])
def test_refresh_matches_oracle_bitexact(dtype, n):
    fresh, stale = synth.refresh_inputs(n, dtype, seed=n)
    s, codes, scales = _run_gpu(fresh, stale)
    en, ec, es = oracle.refresh_residual(np64(fresh), np64(stale), dtype)
    np.testing.assert_array_equal(codes.cpu().numpy(), ec)
    np.testing.assert_array_equal(scales.cpu().numpy(), es)
    np.testing.assert_array_equal(np64(s), en)


def test_refresh_golden_block(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "refresh_block.json")))
    n = g["n"]
    fresh = torch.zeros(n, dtype=torch.bfloat16)
    stale = torch.zeros(n, dtype=torch.bfloat16)
    fresh[:5] = torch.tensor(g["fresh_head"], dtype=torch.bfloat16)
    fresh[128:] = g["block1_value"]
    stale[128:] = g["block1_value"]
    s, codes, scales = _run_gpu(fresh, stale)
    assert codes[:5].cpu().tolist() == g["codes_head"] and not codes[5:].cpu().any()
    assert scales.cpu().tolist() == g["scales"]
    assert s[:5].float().cpu().tolist() == g["new_stale_head"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_zero_delta_identity(dtype):
    _, stale = synth.refresh_inputs(128 * 50 + 3, dtype, seed=2)
    s, codes, scales = _run_gpu(stale, stale)
    assert torch.equal(s.cpu(), stale)
    assert not codes.cpu().any() and not scales.cpu().any()


def test_refresh_sweep_full_size_sampled():
    """200 MiB of bf16 stale buffers + the 2x4x128x128 noise prediction, in one call;
    4096 sampled blocks (and the ragged-free tail) against the oracle."""
    fresh, stale = synth.refresh_sweep_inputs(seed=0)
    n = fresh.numel()
    assert n == 104_988_672
    s, codes, scales = _run_gpu(fresh, stale)
    nblk = n // 128
    rng = np.random.default_rng(0)
    blocks = np.unique(np.concatenate([rng.integers(0, nblk, 4096), [0, nblk - 1, 819_200]]))
    idx = (blocks[:, None] * 128 + np.arange(128)).reshape(-1)
    en, ec, es = oracle.refresh_residual(np64(fresh[idx]), np64(stale[idx]), "bf16")
    np.testing.assert_array_equal(codes.cpu().numpy()[idx], ec)
    np.testing.assert_array_equal(scales.cpu().numpy()[blocks], es)
    np.testing.assert_array_equal(np64(s[torch.from_numpy(idx).cuda()]), en)


def test_refresh_rejects_misaligned():
    x = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(1024, dtype=torch.int8, device="cuda")
    sc = torch.zeros(8, device="cuda")
    with pytest.raises(dpp.DppError) as e:
        dpp.refresh_residual(x[1:513], x[1:513], c[:512], sc[:4])
    assert e.value.code == 3


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [1, 127, 129, 1000, 128 * 997 + 77])
def test_apply_residual_matches_oracle_bitexact(dtype, n):
    """The receiver's half: the oracle's message (codes, scales) applied on the GPU to a
    copy of the old stale buffer gives the oracle's refreshed buffer, bit for bit."""
    fresh, stale = synth.refresh_inputs(n, dtype, seed=n + 3)
    en, ec, es = oracle.refresh_residual(np64(fresh), np64(stale), dtype)
    copy = stale.clone().cuda()
    dpp.apply_residual(torch.from_numpy(ec).cuda(), torch.from_numpy(es).cuda(), copy)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np64(copy), en)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_refresh_edge_blocks_bitexact(dtype):
    """Blocks at the quantiser's edges (tests/refresh_edges.py): half-integer quotients
    with scales that are not powers of two and their neighbours, |a/s| just above and
    below 127, scales just above and below 2^-96 (where the kernel switches from its
    division-free quotient to the IEEE division) and subnormal scales.  The streaming
    loop, and the scalar pass on a ragged copy of the first blocks, give the oracle's
    codes, scales and refreshed values bit for bit; the receiver's apply of the oracle's
    message gives its refreshed buffer."""
    from tests.refresh_edges import edge_blocks
    f64, s64, _ = edge_blocks(dtype)
    f64 = np.concatenate([f64, f64[:200]])
    s64 = np.concatenate([s64, s64[:200]])
    fresh = torch.from_numpy(f64).to(DT[dtype])
    stale = torch.from_numpy(s64).to(DT[dtype])
    assert np.array_equal(np64(fresh), f64) and np.array_equal(np64(stale), s64)
    s, codes, scales = _run_gpu(fresh, stale)
    en, ec, es = oracle.refresh_residual(f64, s64, dtype)
    np.testing.assert_array_equal(codes.cpu().numpy(), ec)
    np.testing.assert_array_equal(scales.cpu().numpy(), es)
    np.testing.assert_array_equal(np64(s), en)
    copy = stale.clone().cuda()
    dpp.apply_residual(torch.from_numpy(ec).cuda(), torch.from_numpy(es).cuda(), copy)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np64(copy), en)
