"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch


def rel_err(a, b) -> float:
    """Normwise relative error ||a - b||_2 / ||b||_2 (fp64)."""
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def tensor(a, dtype, device="cuda"):
    """fp64 array holding values exactly representable in ``dtype`` -> device tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    out = t.to(dtype)
    assert torch.equal(out.to(torch.float64), t), "values not representable in target dtype"
    return out.to(device)


# Tolerances (normwise relative error), stated by the method's accuracy target:
# bf16 outputs 2e-3, fp32 outputs 1e-5.
TOL_BF16 = 2e-3
TOL_F32 = 1e-5
