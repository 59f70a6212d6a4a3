"""Helpers shared by the GPU parity tests."""
import numpy as np

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None


def dev(a, device="cuda"):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def rel_err_rows(got, ref):
    """Per token: max_o |got - ref| / max_o |ref| (the tolerance measure)."""
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    ref2 = ref.reshape(-1, ref.shape[-1])
    got2 = got.reshape(-1, ref.shape[-1])
    return np.max(np.abs(got2 - ref2), axis=1) / np.maximum(np.max(np.abs(ref2), axis=1), 1e-30)


TOL = 2e-3  # relative tolerance on GEMV / MoE outputs (max-normalised per token)
