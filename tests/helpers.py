"""Comparison helpers shared by the tests (no arithmetic of the mixer)."""

import numpy as np
import torch


def np64(t):
    """A torch tensor (any device, bf16 or fp32) as a float64 NumPy array."""
    if t is None:
        return None
    return t.detach().to('cpu', torch.float64).numpy()


def rel_l2(x, ref):
    """||x - ref||_2 / ||ref||_2 over the whole tensor."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


# Tolerances (rel-L2 over a whole tensor): fp32 paths vs the fp64 oracle, and
# the bf16 tensor-core chunk path.
TOL_F32 = 1e-4
TOL_BF16 = 1e-2
