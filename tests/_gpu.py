"""Helpers for the GPU parity tests (comparison metric and tolerances)."""
import numpy as np
import torch

# Max-norm relative error bounds: fp32 storage 1e-5; bf16 storage with fp32
# arithmetic 2e-2 (each bf16 rounding is <= 2^-9 relative, a few enter).
TOL = {"f32": 1e-5, "bf16": 2e-2}


def rel_err(got, ref) -> float:
    """max_e |got_e - ref_e| / max_e |ref_e| over the whole tensor."""
    g = got.detach().float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if not np.all(np.isfinite(g)):
        return float("inf")
    scale = max(float(np.max(np.abs(r))), 1e-30)
    return float(np.max(np.abs(g - r))) / scale


def dev():
    return torch.device("cuda:0")


def dtype_of(name):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]
