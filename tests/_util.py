"""Small helpers shared by the tests (no attention arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view of a tensor; bf16 becomes its raw uint16 bit patterns
    (the oracle widens those exactly)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening through torch's own conversion (bf16/fp16 -> fp32 -> fp64)."""
    return t.detach().cpu().to(torch.float32).to(torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a tensor, for bit-exact comparisons."""
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy().copy() if t.element_size() == 1 else \
        t.view({2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()]).numpy().copy()


def tolerance(dtype: torch.dtype):
    """(atol, rtol) of the parity bar: fp32 inputs max-abs 1e-5; bf16/fp16
    inputs |gpu - ref| <= 2e-2 + 1e-2 |ref| with fp32 accumulation."""
    if dtype == torch.float32:
        return 1e-5, 0.0
    return 2e-2, 1e-2


def assert_close_to_ref(gpu: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, what: str = ""):
    atol, rtol = tolerance(dtype)
    g = to_f64(gpu)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance "
            f"(max err {np.nanmax(err):.3e}); first at {idx.tolist()}: "
            f"gpu={g[tuple(idx[0])]:.6f} ref={ref[tuple(idx[0])]:.6f}")
    return float(np.max(err)) if err.size else 0.0
