"""Shared helpers for the tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

BF16_TOL = 2e-2   # max|gpu - oracle| / max|oracle| for bf16 inputs (fp32 state and accumulation)
F32_TOL = 1e-4    # the same bound for fp32 inputs


def to_np(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_err(x, ref):
    x, ref = to_np(x), to_np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    denom = max(float(np.max(np.abs(ref))), 1e-30) if ref.size else 1.0
    return float(np.max(np.abs(x - ref))) / denom if ref.size else 0.0


def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch.device("cuda:0")


def to_dev(d, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
