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


# Every fp16 (amax, x) pair, for the exhaustive quantization tests.
def positive_fp16() -> np.ndarray:
    """All positive finite fp16 values in increasing order (31743 values:
    the 1023 subnormals, then every normal up to 65504)."""
    return np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16)


# Row layout of the exhaustive test: element 0 is the row's maximum a_i, then
# J = 1023 pairs (+v, -v) of values v <= a_i, then one zero.  Amax i (the i-th
# positive value) needs ceil((i + 1) / J) rows to hold all i + 1 values <= it.
EXH_W = 2048
EXH_J = (EXH_W - 2) // 2


def exhaustive_rows(pos: np.ndarray, i0: int, i1: int) -> np.ndarray:
    """The rows for amax indices [i0, i1) (zeros where a row has no more values)."""
    idx = np.arange(i0, i1)
    counts = (idx + EXH_J) // EXH_J                   # ceil((i + 1) / J)
    amax_i = np.repeat(idx, counts)
    first = np.repeat(np.cumsum(counts) - counts, counts)
    r = np.arange(len(amax_i)) - first                  # row number within its amax
    j = r[:, None] * EXH_J + np.arange(EXH_J)[None, :]
    valid = j <= amax_i[:, None]
    vals = np.where(valid, pos[np.minimum(j, len(pos) - 1)], np.float16(0))
    x = np.zeros((len(amax_i), EXH_W), np.float16)
    x[:, 0] = pos[amax_i]
    x[:, 1:1 + 2 * EXH_J:2] = vals
    x[:, 2:2 + 2 * EXH_J:2] = -vals
    return x
