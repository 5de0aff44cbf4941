"""GPU parity of the quantization kernels against the oracle, bit-exact:
per-token activation quantization (codes and scales) and the INT8 / INT4
weight quantizers (codes, packed bytes and scales)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import assert_bits_equal, require_gpu, to_dev, to_host
from w4a8_quantized_linear_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cider():
    return require_gpu()


def special_rows(K):
    rows = [np.zeros(K, np.float16)]                               # all zero -> s = 1, q = 0
    r = np.zeros(K, np.float16)
    ties = np.array([127, 0.5, 1.5, 2.5, -0.5, -2.5, 63.5, 62.5, -126.5], np.float16)
    r[:len(ties)] = ties                                            # s = 1, ties to even
    rows.append(r)
    r = np.full(K, -65504, np.float16)
    r[1::2] = 65504                                                 # extremes
    rows.append(r)
    r = (np.arange(K) % 7 - 3).astype(np.float16) * np.float16(2 ** -20)  # subnormals
    rows.append(r)
    r = np.zeros(K, np.float16)
    r[K - 1] = -3.0                                                 # amax at the last element
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (37, 2560), (128, 4096), (5, 10240),
                                 (2, 16384), (3, 18432), (300, 2048), (17, 12288)])
def test_quantize_act_bit_exact(cider, M, K):
    x = inputs.activations(M, K, seed=100 + M)
    x = np.concatenate([x, special_rows(K)])
    qa, sa = cider.cider_quantize_act(to_dev(x))
    qref, sref = oracle.quantize_act(x)
    assert_bits_equal(to_host(sa).view(np.uint32), sref.view(np.uint32), "s_a")
    assert_bits_equal(to_host(qa), qref, "q_a")


@pytest.mark.parametrize("gs", [0, 64, 128])
@pytest.mark.parametrize("N,K", [(8, 128), (136, 256), (64, 2560), (16, 12288)])
def test_quantize_weight_int8_bit_exact(cider, N, K, gs):
    W = inputs.weights(N, K, seed=7)
    W[1] = 0.0
    W[2, :64] = 0.0
    W[3, 5] = 1.0
    qw, sw = cider.cider_quantize_weight_int8(to_dev(W), gs)
    qref, sref = oracle.quantize_weight_int8(W, gs)
    assert_bits_equal(to_host(qw), qref, "q_w")
    assert_bits_equal(to_host(sw).view(np.uint32), sref.view(np.uint32), "s_w")


@pytest.mark.parametrize("gs", [0, 64, 128])
@pytest.mark.parametrize("N,K", [(8, 128), (136, 256), (64, 2560), (16, 12288)])
def test_quantize_weight_int4_bit_exact(cider, N, K, gs):
    W = inputs.weights(N, K, seed=8)
    W[1] = 0.0
    W[2, :64] = 0.0
    W[3, 5] = -1.0
    qp, sw = cider.cider_quantize_weight_int4(to_dev(W), gs)
    q4, sref = oracle.quantize_weight_int4(W, gs)
    assert_bits_equal(to_host(qp), oracle.pack_int4(q4), "packed q_w")
    assert_bits_equal(to_host(sw).view(np.uint32), sref.view(np.uint32), "s_w")


def test_no_device_error_left(cider):
    assert cider.cider_check_device_error() == 0


def _exhaustive_amax_values():
    rng = np.random.default_rng(2024)
    fixed = [65504.0, 1.0, 127.0, 3.140625, 0.0009765625, 2.0 ** -24 * 37, 2.0 ** -14, 1000.0,
             0.0016956329345703125, 0.50732421875, 2.0 ** -24, 6.0e-5, 0.3333, 254.0, 8191.0]
    allv = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    pos = allv[np.isfinite(allv) & (allv > 0)]
    return fixed + [float(v) for v in rng.choice(pos, 25, replace=False)]


@pytest.mark.parametrize("amax", _exhaustive_amax_values())
def test_quantize_act_exhaustive_fp16_values(cider, amax):
    """Every finite fp16 value |x| <= amax, in rows whose maximum is amax: codes
    and scales bit-exact against the oracle (exercises the division, rounding
    and clamp for all inputs a scale can see)."""
    allv = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    vals = allv[np.isfinite(allv) & (np.abs(allv.astype(np.float64)) <= amax)]
    W = 2048
    pad = (-len(vals)) % (W - 1)
    vals = np.concatenate([vals, np.zeros(pad, np.float16)]).reshape(-1, W - 1)
    x = np.concatenate([np.full((vals.shape[0], 1), amax, np.float16), vals], axis=1)
    qa, sa = cider.cider_quantize_act(to_dev(x))
    qref, sref = oracle.quantize_act(x)
    assert_bits_equal(to_host(sa).view(np.uint32), sref.view(np.uint32), "s_a")
    assert_bits_equal(to_host(qa), qref, "q_a")
