"""Shared helpers for the GPU parity tests: device gate, tensor transfer, and
the fp16 output tolerance |y - y_ref| <= 2e-3 * max|y_ref| + 1 ulp(y_ref),
where ulp(v) is the fp16 spacing at |v| (2^-24 in the subnormal range)."""
import numpy as np
import pytest
import torch

REL_TOL = 2e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import w4a8_quantized_linear_gb300 as cider
    if not cider.cider_is_available():
        pytest.fail("libcider reports the current device is not a supported sm_103 GPU")
    return cider


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def fp16_ulp(v: np.ndarray) -> np.ndarray:
    return np.spacing(np.abs(v.astype(np.float16))).astype(np.float64)


def assert_fp16_close(y: np.ndarray, y_ref: np.ndarray, what: str = ""):
    y64 = y.astype(np.float64)
    r64 = y_ref.astype(np.float64)
    assert np.all(np.isfinite(r64)), "reference has non-finite values"
    bound = REL_TOL * np.max(np.abs(r64)) + fp16_ulp(y_ref)
    err = np.abs(y64 - r64)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outputs out of tolerance; "
                             f"first at {tuple(i)}: got {y64[tuple(i)]}, want {r64[tuple(i)]}, "
                             f"bound {bound[tuple(i)]}")


def assert_bits_equal(a: np.ndarray, b: np.ndarray, what: str = ""):
    if a.dtype == np.float16:
        a, b = a.view(np.uint16), b.view(np.uint16)
    if not np.array_equal(a, b):
        idx = np.argwhere(a != b)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {a.size} differ; first at {i}: "
                             f"got {a[i]}, want {b[i]}")
