"""The softmax's polynomial 2^x (poly_exp2x2, on the FMA pipes) against its
stated error bound: relative error below 2.2e-4 of the exact 2^x over the
softmax's input range [-125, 8], and the clamp below -125 (the result for
any smaller x, -inf included, is the value at -125).

The probe kernel in tests/csrc/exp2_probe.cu is compiled here with nvcc for
sm_103a; the reference values are numpy float64 powers of two."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
BOUND = 2.2e-4


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("exp2probe") / "libexp2probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", os.path.join(HERE, "csrc", "exp2_probe.cu"),
                    "-o", out], check=True, capture_output=True, text=True)
    lib = ctypes.CDLL(out)
    lib.poly_exp2_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                    ctypes.c_void_p]
    lib.poly_exp2_probe.restype = ctypes.c_int
    return lib


def _run(probe, x: np.ndarray) -> np.ndarray:
    import torch
    if x.size % 2:
        x = np.append(x, np.float32(0))
    xd = torch.from_numpy(x.astype(np.float32)).cuda()
    yd = torch.empty_like(xd)
    st = probe.poly_exp2_probe(xd.data_ptr(), yd.data_ptr(), x.size // 2,
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return yd.cpu().numpy()[:x.size]


def test_poly_exp2_relative_error_bound(probe):
    dense = np.linspace(-125.0, 8.0, 8_000_001, dtype=np.float64).astype(np.float32)
    # the ends of every reduction interval: half-integers and their float
    # neighbours (f = +-1/2, where the cubic's error is largest)
    half = np.arange(-125, 8, dtype=np.float64) + 0.5
    edges = np.concatenate([half, np.nextafter(half.astype(np.float32), np.float32(-np.inf)),
                            np.nextafter(half.astype(np.float32), np.float32(np.inf)),
                            np.arange(-125, 9, dtype=np.float32)]).astype(np.float32)
    x = np.concatenate([dense, edges])
    y = _run(probe, x).astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y - exact) / exact
    assert np.all(np.isfinite(y)) and np.all(y > 0)
    worst = float(rel.max())
    assert worst < BOUND, f"max relative error {worst:.3e} at x = {x[rel.argmax()]}"
    # the bound is close to tight at f = +1/2 (x = k + 1/2)
    assert worst > 0.5 * BOUND


def test_poly_exp2_clamps_below_minus_125(probe):
    x = np.array([-125.0, -125.5, -126.0, -200.0, -1e30, -np.inf], dtype=np.float32)
    y = _run(probe, x)
    assert np.all(y == y[0]), y
    assert abs(float(y[0]) / 2.0 ** -125 - 1.0) < BOUND
