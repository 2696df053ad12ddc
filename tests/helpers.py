"""Shared test helpers: moving seeded inputs between numpy and torch, and the
GEMM error metric.  No quantisation arithmetic lives here."""
import numpy as np

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None

# Maximum error of a GEMM result relative to the largest reference magnitude
# of its own output row.  Rows are the unit because visual and text rows differ
# by ~34x in magnitude, so a tensor-wide normaliser would hide text-row errors.
GEMM_REL_TOL = 1e-3


def row_rel_err(c: np.ndarray, ref: np.ndarray) -> float:
    c = np.asarray(c, dtype=np.float64).reshape(-1, ref.shape[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    den = np.max(np.abs(r), axis=1, keepdims=True)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(c - r) / den)) if c.size else 0.0


def to_dev(a: np.ndarray, dtype=None):
    """numpy -> CUDA tensor with the same bytes (uint16 arrays become bfloat16)."""
    if a.dtype == np.uint16 and dtype is None:
        return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int16:
        return t.numpy().view(np.uint16)
    return t.numpy()
