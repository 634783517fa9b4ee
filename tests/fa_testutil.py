"""Shared helpers of the GPU parity tests (comparison against the oracle)."""
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tolerances():
    vals = {}
    with open(os.path.join(GOLDEN, "tolerances.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


TOL = _tolerances()
ABS_TOL = TOL["abs_tol"]  # 2e-2
REL_TOL = TOL["rel_tol"]  # 1e-2 of max |oracle|


def assert_parity(gpu: torch.Tensor, ora: np.ndarray, what: str = ""):
    """Acceptance bound for bf16 inputs / fp32 accumulation:
    max|gpu - oracle| <= 2e-2 and <= 1e-2 * max|oracle| (elementwise, in fp64)."""
    g = gpu.detach().float().cpu().double().numpy().reshape(ora.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ora).max() if ora.size else 0.0
    scale = np.abs(ora).max() if ora.size else 0.0
    assert err <= ABS_TOL, f"{what}: max abs err {err:.3e} > {ABS_TOL}"
    assert err <= REL_TOL * max(scale, 1e-30) or ora.size == 0, \
        f"{what}: max abs err {err:.3e} > {REL_TOL} * max|out| ({scale:.3e})"
    return err


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(n_total: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    idx = rng.choice(n_total, size=min(k, n_total), replace=False)
    return np.sort(idx)
