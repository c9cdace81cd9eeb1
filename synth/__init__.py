"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no arithmetic of the method itself: it only draws seeded
random tensors with the shapes and value distributions of the five workloads
(SDXL-1024 mid level, SDXL-3840 attention level, VAE-decoder halo conv,
residual refresh sweep, tiny fp32 step).  Every tensor is keyed by
(seed, tensor id), so any tensor can be regenerated on its own.

Values are drawn in fp32 on the CPU with torch's seeded generator and are
rounded to the storage dtype once by the caller (``to_storage``); the same
bytes then feed both the GPU path and the oracle.
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch

# Tensor ids: one stream per logical tensor, so adding a tensor never
# shifts the values of another.
TID = {
    "w_conv": 1, "w_qkv": 2, "w_o": 3, "gamma": 4, "beta": 5,
    "x": 10, "x_prev_noise": 11,
    "q": 20, "k": 21, "v": 22, "k_noise": 23, "v_noise": 24,
    "y": 30, "y_noise": 31,
    "stale": 40, "fresh_noise": 41, "spike_pick": 42, "spike": 43,
    "noise_pred": 44, "noise_pred_noise": 45,
}


def _key(seed: int, tid: int) -> int:
    h = hashlib.sha256(f"dpp:{seed}:{tid}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def normal(shape, seed: int, tid: str, std: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std^2) tensor of ``shape`` from stream (seed, tid)."""
    g = torch.Generator(device="cpu").manual_seed(_key(seed, TID[tid]))
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def uniform(shape, seed: int, tid: str) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(_key(seed, TID[tid]))
    return torch.rand(*shape, generator=g, dtype=torch.float32)


def to_storage(t: torch.Tensor, dtype: str) -> torch.Tensor:
    """Round an fp32 tensor to the storage dtype ('bf16' or 'f32') once."""
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "f32":
        return t.to(torch.float32)
    raise ValueError(dtype)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one displaced-patch layer step (NHWC == [B, L=H*W, C])."""
    name: str
    B: int
    H: int
    W: int
    C: int
    P: int
    G: int
    heads: int
    head_dim: int
    dtype: str
    w_std: float = 0.02
    stale_std: float = 0.05
    eps: float = 1e-5

    @property
    def L(self) -> int:
        return self.H * self.W


# The layer workloads: the tiny fp32 step and the SDXL-1024 mid-level block.
TINY_F32 = LayerConfig("tiny_f32_32x32_c64_p2", B=1, H=32, W=32, C=64, P=2, G=8,
                       heads=1, head_dim=64, dtype="f32", stale_std=0.01)
SDXL1024_MID = LayerConfig("sdxl1024_mid_b2_64x64_c640_p4", B=2, H=64, W=64, C=640, P=4,
                           G=32, heads=10, head_dim=64, dtype="bf16", stale_std=0.05)


def layer_weights(cfg: LayerConfig, seed: int = 0, affine: bool = False):
    """Conv [C,3,3,C], packed QKV [3C,C], O [C,C] weights N(0, w_std^2); gamma/beta fp32.

    The workloads use gamma = 1, beta = 0; ``affine=True`` draws them (unit tests).
    """
    C = cfg.C
    w_conv = to_storage(normal((C, 3, 3, C), seed, "w_conv", cfg.w_std), cfg.dtype)
    w_qkv = to_storage(normal((3 * C, C), seed, "w_qkv", cfg.w_std), cfg.dtype)
    w_o = to_storage(normal((C, C), seed, "w_o", cfg.w_std), cfg.dtype)
    if affine:
        gamma = 1.0 + 0.1 * normal((C,), seed, "gamma")
        beta = 0.1 * normal((C,), seed, "beta")
    else:
        gamma = torch.ones(C, dtype=torch.float32)
        beta = torch.zeros(C, dtype=torch.float32)
    return dict(w_conv=w_conv, w_qkv=w_qkv, w_o=w_o, gamma=gamma, beta=beta)


def layer_inputs(cfg: LayerConfig, seed: int = 0):
    """x [B,H,W,C] N(0,1) and the previous step's input x_prev = x + N(0, stale_std^2).

    The stale state of a step is the state a synchronous pass over x_prev leaves.
    """
    shape = (cfg.B, cfg.H, cfg.W, cfg.C)
    x32 = normal(shape, seed, "x")
    xp32 = x32 + normal(shape, seed, "x_prev_noise", cfg.stale_std)
    return to_storage(x32, cfg.dtype), to_storage(xp32, cfg.dtype)


def attention_inputs(B: int, L: int, heads: int, head_dim: int, dtype: str = "bf16",
                     seed: int = 0, stale_std: float = 0.05):
    """Q, K_fresh, V_fresh [B,L,heads*head_dim] N(0,1); K/V_stale = fresh + N(0, stale_std^2)."""
    C = heads * head_dim
    q = normal((B, L, C), seed, "q")
    k = normal((B, L, C), seed, "k")
    v = normal((B, L, C), seed, "v")
    ks = k + normal((B, L, C), seed, "k_noise", stale_std)
    vs = v + normal((B, L, C), seed, "v_noise", stale_std)
    return tuple(to_storage(t, dtype) for t in (q, k, v, ks, vs))


def conv_inputs(B: int, H: int, W: int, Cin: int, Cout: int, dtype: str = "bf16",
                seed: int = 0, stale_std: float | None = 0.05, w_std: float = 0.02):
    """y [B,H,W,Cin] N(0,1); y_stale = y (stale_std None) or y + N(0, stale_std^2); w [Cout,3,3,Cin]."""
    y = normal((B, H, W, Cin), seed, "y")
    ys = y.clone() if stale_std is None else y + normal((B, H, W, Cin), seed, "y_noise", stale_std)
    w = normal((Cout, 3, 3, Cin), seed, "w_conv", w_std)
    return to_storage(y, dtype), to_storage(ys, dtype), to_storage(w, dtype)


def refresh_inputs(n: int, dtype: str = "bf16", seed: int = 0, noise_std: float = 0.05,
                   spike_frac: float = 0.10, block: int = 128):
    """stale [n] N(0,1); fresh = stale + N(0, noise_std^2), except that a seeded
    ``spike_frac`` of the ``block``-element blocks carry N(0,1) deltas instead."""
    stale = normal((n,), seed, "stale")
    nblk = (n + block - 1) // block
    pick = uniform((nblk,), seed, "spike_pick") < spike_frac
    std = torch.full((nblk,), noise_std).masked_fill(pick, 1.0)
    std_e = std.repeat_interleave(block)[:n]
    delta = normal((n,), seed, "fresh_noise") * std_e
    fresh = stale + delta
    return to_storage(fresh, dtype), to_storage(stale, dtype)


def refresh_sweep_inputs(seed: int = 0, kv_bytes: int = 200 * 1024 * 1024,
                         noise_pred_shape=(2, 4, 128, 128)):
    """The refresh sweep: 200 MiB of bf16 stale KV/halo buffers plus the
    2x4x128x128 noise prediction, as one flat bf16 buffer of fresh and stale."""
    n_kv = kv_bytes // 2
    n_np = 1
    for d in noise_pred_shape:
        n_np *= d
    return refresh_inputs(n_kv + n_np, "bf16", seed)
