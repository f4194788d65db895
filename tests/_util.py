"""Shared test helpers: host<->device moves of bf16 bit arrays, tolerances."""
import numpy as np

# Tolerances for bf16 attention outputs against the fp64 oracle: the
# largest and the mean absolute difference over all outputs.
ATOL_MAX = 2e-2
ATOL_MEAN = 2e-3


def to_dev_bf16(bits: np.ndarray, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_dev(arr: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def bf16_dev_to_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_dev_to_f64(t) -> np.ndarray:
    import torch
    return t.float().cpu().numpy().astype(np.float64)


def assert_close_attn(got: np.ndarray, want: np.ndarray, what: str = ""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= ATOL_MAX, f"{what}: max abs err {mx:.3e} > {ATOL_MAX} at {np.unravel_index(err.argmax(), err.shape)}"
    assert mean <= ATOL_MEAN, f"{what}: mean abs err {mean:.3e} > {ATOL_MEAN}"
    return mx, mean
