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

# Per-row bars.  Every row -- every vector along the last axis: one (token, head)
# of an output, one key row of a state -- must also be close on its own, so that
# a wrong row, head or chunk cannot hide inside the tensor-level norm (one wholly
# wrong (token, head) row of a 4096 x 32-head output moves the tensor rel-L2 by
# only ~0.006).  A row's error is taken relative to max(its norm, ROW_FLOOR x the
# RMS row norm): the rounding error of a bf16 tensor-core output is set by the
# scale of the state and of the whole tensor, not by the row, so rows far smaller
# than typical carry the same absolute error as the rest.  The bars are 10x the
# tensor bars; they catch gross errors (a wholly wrong row scores about 1 or
# more), not the rounding tail: with a floor of a quarter of the median row norm,
# the worst of ~10^6 rows reached 0.114 on a GB300 (packed workload).
TOL_ROW_F32 = 1e-3
TOL_ROW_BF16 = 1e-1
ROW_FLOOR = 0.5
# Rows of y = gated_rmsnorm(o, z): the norm divides each row by its own RMS, so a
# row whose core output o is small by cancellation (q nearly orthogonal to the
# state's rows) keeps the state's bf16 rounding error relative to itself, and the
# floor above cannot act (every y row has a typical norm); the o rows themselves
# are checked at TOL_ROW_BF16.  Measured at the full workloads: worst y row 0.11
# of the 131,072 rows of prefill_t4096.  An entirely wrong row scores about sqrt(2).
TOL_ROW_Y_BF16 = 0.25


def row_rel_err(x, ref):
    """max over rows (last axis) of ||x_r - ref_r|| / max(||ref_r||, ROW_FLOOR * RMS row norm)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if x.size == 0:
        return 0.0
    n = ref.shape[-1] if ref.ndim else 1
    x = x.reshape(-1, n)
    ref = ref.reshape(-1, n)
    d = np.linalg.norm(x - ref, axis=1)
    rn = np.linalg.norm(ref, axis=1)
    den = np.maximum(rn, ROW_FLOOR * np.sqrt(np.mean(rn * rn)))
    den = np.where(den > 0, den, 1.0)
    return float((d / den).max())


def assert_close(x, ref, tol, row_tol=None, what=''):
    """Tensor-level rel-L2 <= tol and per-row error <= row_tol (by default the row bar
    that goes with tol)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    e = rel_l2(x, ref)
    assert e <= tol, ('rel-L2', what, e, tol)
    if row_tol is None:
        row_tol = TOL_ROW_F32 if tol <= TOL_F32 else TOL_ROW_BF16
    r = row_rel_err(x, ref)
    assert r <= row_tol, ('row', what, r, row_tol)
