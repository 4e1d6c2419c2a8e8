"""Shared test helpers: device copies of seeded inputs and the error metric."""
import numpy as np

from selective_state_space_160_b300.inputs import bf16_bits


def to_dev(a, bf16=False, device="cuda"):
    """numpy float32 (bf16-representable when bf16) -> torch CUDA tensor."""
    import torch
    if a is None:
        return None
    if bf16:
        t = torch.from_numpy(bf16_bits(a).view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device)


def max_rel_err(gpu, ref):
    """max |gpu - ref| / (1 + |ref|), the parity metric of every test."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if gpu.size == 0:
        return 0.0
    return float(np.max(np.abs(gpu - ref) / (1.0 + np.abs(ref))))
