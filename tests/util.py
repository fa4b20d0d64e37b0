"""Comparison helpers shared by the GPU parity tests."""
import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


# Tolerances (rel-L2 per tensor): float32 path 1e-4 everywhere; bf16 storage
# with float32 accumulation 1e-2 on outputs and 2e-2 on gradients; CE loss
# absolute error 1e-3.
TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-2, 2e-2)}
CE_LOSS_ABS = 1e-3
