"""Comparison helpers shared by the tests (no method arithmetic here)."""
import numpy as np
import torch

# Per-tensor relative L2 tolerances: bf16 operands with fp32 accumulation, and
# the all-fp32 path.
TOL = {"bf16": 5e-3, "f32": 1e-4}


def round_like(ref64: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Round an fp64 oracle result to the output dtype (RNE), back to fp64."""
    return torch.from_numpy(np.ascontiguousarray(ref64)).to(dtype).to(torch.float64).numpy()


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    if den == 0.0:
        return 0.0 if np.all(x == 0) else float("inf")
    return float(np.linalg.norm(x - ref) / den)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()
