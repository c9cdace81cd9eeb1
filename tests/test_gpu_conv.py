"""GPU parity: halo_conv3x3 (tcgen05 implicit GEMM for bf16, SIMT for fp32)
against the CPU oracle; halo-row sourcing pinned bit-exactly with sentinels."""
import numpy as np
import pytest
import torch

import oracle
import stale_activations_gb300 as dpp
import synth
from tests.util import TOL_BF16, TOL_F32, np64, rel_err

pytestmark = pytest.mark.gpu
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _conv_gpu(yf, ys, w, P):
    B, H, W, _ = yf.shape
    out = torch.empty(B, H, W, w.shape[0], dtype=yf.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dpp.halo_conv3x3(yf.cuda(), ys.cuda(), w.cuda(), out, P, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out


@pytest.mark.parametrize("dtype,B,H,W,Cin,Cout,P", [
    ("bf16", 2, 16, 64, 128, 128, 4),     # 2 image rows per 128-pixel tile
    ("bf16", 1, 8, 256, 64, 128, 2),      # half a row per tile
    ("bf16", 1, 16, 32, 64, 256, 4),      # 4 rows per tile
    ("bf16", 1, 16, 128, 192, 128, 8),    # one row per tile, 1-row bands (both halos stale)
    ("bf16", 1, 8, 64, 64, 128, 8),       # 2 rows per tile, 1-row bands: both rows' halos stale
    ("bf16", 1, 16, 64, 256, 320, 2),     # 36 K slices: 128 x 320 tiles (two MMAs per step)
    ("bf16", 1, 160, 128, 256, 320, 4),   # 160 such tiles: some CTAs reuse one accumulator
    # W neither a divisor nor a multiple of 128: tiles of 128 / gcd(W, 128) row segments
    # that wrap across rows, bands whose pixel count is not a multiple of 128
    ("bf16", 2, 16, 240, 64, 128, 4),     # 16-pixel segments (the SDXL-3840 latent width)
    ("bf16", 1, 12, 96, 128, 128, 3),     # 32-pixel segments, 4-row bands
    ("bf16", 1, 16, 40, 64, 160, 8),      # 8-pixel segments, 2-row bands
    ("f32", 1, 32, 32, 64, 64, 2),
    ("f32", 1, 6, 5, 3, 7, 3),            # ragged sizes on the SIMT path
])
def test_conv_matches_oracle(dtype, B, H, W, Cin, Cout, P):
    yf, ys, w = synth.conv_inputs(B, H, W, Cin, Cout, dtype, seed=H * W + Cin)
    out = _conv_gpu(yf, ys, w, P)
    ref = oracle.halo_conv3x3(np64(yf), np64(ys), np64(w), P, dtype)
    assert rel_err(np64(out), ref) < (TOL_BF16 if dtype == "bf16" else TOL_F32)


@pytest.mark.parametrize("W,P", [(32, 4), (64, 4), (256, 4), (240, 4), (40, 4), (64, 16),
                                 (32, 16), (16, 2)])
def test_conv_sentinel_halo_rows_bitexact(W, P):
    """fresh = +1, stale = -1 and one-hot weights (output channel o reads tap o % 9
    of input channel o % Cin): every output is -1, 0 or +1 by the band rule alone.  Whole-row
    tiles (W = 16, 32, 64) with 4-row bands, tiles that are whole bands (W = 16, 8-row bands)
    and 1-row bands (every shifted row from the stale map)."""
    B, H, Cin, Cout = 1, 16, 64, 128
    yf = torch.ones(B, H, W, Cin, dtype=torch.bfloat16)
    ys = -torch.ones(B, H, W, Cin, dtype=torch.bfloat16)
    w = torch.zeros(Cout, 3, 3, Cin, dtype=torch.bfloat16)
    for o in range(Cout):
        w[o, (o % 9) // 3, (o % 9) % 3, o % Cin] = 1.0
    out = _conv_gpu(yf, ys, w, P).float().cpu().numpy()
    Hp = H // P
    exp = np.zeros((H, W, Cout))
    for o in range(Cout):
        ti, tj = (o % 9) // 3, (o % 9) % 3
        for r in range(H):
            rr = r + ti - 1
            for c in range(W):
                cc = c + tj - 1
                if 0 <= rr < H and 0 <= cc < W:
                    exp[r, c, o] = 1.0 if rr // Hp == r // Hp else -1.0
    np.testing.assert_array_equal(out[0], exp)


def test_conv_vae_size_banded_equals_unbanded_and_oracle_rows():
    """The VAE-decoder-like workload: 1x256x256x512 -> 512, P = 8 row bands.
    With stale == fresh the banded conv equals the unbanded one bit for bit; with a
    stale halo, sampled output rows (band edges and interiors) match the oracle."""
    B, H, W, C, P = 1, 256, 256, 512, 8
    yf, ys, w = synth.conv_inputs(B, H, W, C, C, "bf16", seed=0)
    banded = _conv_gpu(yf, yf, w, P)
    unbanded = _conv_gpu(yf, yf, w, 1)
    assert torch.equal(banded, unbanded)
    out = _conv_gpu(yf, ys, w, P)
    rows = np.array([0, 1, 31, 32, 63, 100, 127, 128, 224, 255])
    ref = oracle.halo_conv3x3(np64(yf), np64(ys), np64(w), P, "bf16", rows=rows)
    assert rel_err(np64(out)[:, rows], ref) < TOL_BF16
    ref1 = oracle.halo_conv3x3(np64(yf), np64(yf), np64(w), 1, "bf16", rows=rows)
    assert rel_err(np64(unbanded)[:, rows], ref1) < TOL_BF16
