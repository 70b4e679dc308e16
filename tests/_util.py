"""Helpers shared by the tests (comparison metrics, device availability)."""
import numpy as np


def rel_rmse(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def min_row_cosine(y, ref):
    y = np.asarray(y, dtype=np.float64).reshape(-1, np.shape(y)[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, np.shape(ref)[-1])
    num = np.sum(y * ref, axis=1)
    den = np.linalg.norm(y, axis=1) * np.linalg.norm(ref, axis=1)
    return float(np.min(num / np.maximum(den, 1e-300)))


def cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
