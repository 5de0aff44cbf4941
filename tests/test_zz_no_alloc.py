"""Tests of cider_w8a8_linear_noalloc, the W8A8 linear for callers that must
not allocate device memory while they run (an engine that reserved almost all
of HBM up front, or a decode loop that cannot let a memory pool grow).

It runs the same dispatch and kernels as cider_w8a8_linear but takes its
scratch from one fixed array in device memory, which every call reuses and
overwrites.  So its results are checked against the oracle itself (per
channel bit for bit, per group within the fp16 tolerance), on two calls in a
row with different inputs, and against cider_w8a8_linear bit for bit.  This
file is collected last so that a stop-at-first-failure run has already run
every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import assert_bits_equal, assert_fp16_close, require_gpu, to_host
from w4a8_quantized_linear_gb300 import _build, inputs

SCRATCH_BYTES = 32 * 1024 * 1024


def noalloc_entry(lib):
    f = lib.cider_w8a8_linear_noalloc
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [p, i64, i64, i64, p, p, i32, i32, p, p]
    f.restype = i32
    return f


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,gs", [
    (200, 264, 1024, 0),      # tensor-core path, per channel
    (300, 136, 2048, 128),    # tensor-core path, per group
    (3, 136, 2560, 64),       # small M, rows quantized inside the GEMV (M * K <= 8192)
    (2, 264, 10240, 0),       # small M, dp4a form, rows quantized first (M * K > 8192)
    (2, 264, 10240, 128),
    (16, 520, 2560, 0),       # small M, tensor-core form, rows quantized first
    (16, 520, 2560, 64),
    (1, 520, 12288, 128),     # one token, long rows
    (4096, 10240, 2560, 0),   # the benchmark workload (needs 21 MB of the 32 MiB array)
])
def test_noalloc_matches_oracle_on_consecutive_calls(M, N, K, gs):
    cider = require_gpu()
    f = noalloc_entry(cider.library())
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    W = inputs.weights(N, K, seed=N + K)
    qw_h, sw_h = oracle.quantize_weight_int8(W, gs)
    qw, sw = torch.from_numpy(qw_h).to(dev), torch.from_numpy(sw_h).to(dev)
    gran = cider.CIDER_PER_GROUP if gs else cider.CIDER_PER_CHANNEL
    xs_h = [inputs.activations(M, K, seed=40 + i) for i in range(2)]
    xs = [torch.from_numpy(x).to(dev) for x in xs_h]
    ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in range(2)]
    # two calls in a row through the C ABI; the second reuses the same scratch
    for x, y in zip(xs, ys):
        st = f(x.data_ptr(), M, N, K, qw.data_ptr(), sw.data_ptr(), gran, gs, y.data_ptr(), stream)
        assert st == 0, cider.library().cider_status_string(st)
    torch.cuda.synchronize()
    full = M * N * K <= 2 ** 31
    rows = np.arange(M) if full else np.array(sorted({0, 1, M // 2, M - 2, M - 1, 1234, 3001}))
    for i, (xh, x, y) in enumerate(zip(xs_h, xs, ys)):
        got = to_host(y)[rows]
        want = oracle.linear(xh, qw_h, sw_h, gs, rows=rows, threads=8)
        what = f"noalloc call {i} M={M} N={N} K={K} gs={gs}"
        if gs == 0:
            assert_bits_equal(got, want, what)
        else:
            assert_fp16_close(got, want, what)
        # and the same bits as the pooled entry point (same kernels, same dispatch)
        assert_bits_equal(got, to_host(cider.cider_w8a8_linear(x, qw, sw, gs))[rows], what + " vs pooled")
    assert cider.cider_check_device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(monkeypatch):
    """Host-side check, no GPU needed: the size limit is enforced before the
    device is touched (CIDER_FORCE_UNSUPPORTED=1 stops well-formed calls at the
    device check, so nothing is launched)."""
    import w4a8_quantized_linear_gb300 as cider
    _build.build()
    f = noalloc_entry(cider.library())
    monkeypatch.setenv("CIDER_FORCE_UNSUPPORTED", "1")
    P = 0x10000
    K = 2560
    def need(M):  # codes (2*M*K bytes), scales and code sums (4*M each), in 256-byte blocks
        return -(-2 * M * K // 256) * 256 + 2 * (-(-4 * M // 256) * 256)
    m_max = max(M for M in range(6000, 7000) if need(M) <= SCRATCH_BYTES)
    assert m_max == 6543
    assert f(P, m_max + 1, 1024, K, P, P, 0, 0, P, None) == 1   # CIDER_ERR_INVALID_ARGUMENT
    assert f(P, m_max, 1024, K, P, P, 0, 0, P, None) == 3       # passes the size check
    assert f(P, 0, 1024, K, None, None, 0, 0, None, None) == 0  # empty problem
    assert f(P, 16, 1024, K, P, P, 1, 0, P, None) == 1          # per group without a group size
