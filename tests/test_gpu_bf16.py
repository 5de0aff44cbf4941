"""GPU parity of the bf16-activation entry points and of the offset-binary
INT4 import against the oracle: per-token quantization of bf16 rows (codes and
scales bit-exact, every finite bf16 value below several amax values), the
bf16 linears on the small-M and tensor-core paths (per channel bit-exact, per
group within the fp16 tolerance), and the INT4 re-encoding (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import assert_bits_equal, assert_fp16_close, require_gpu, to_dev, to_host
from w4a8_quantized_linear_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cider():
    return require_gpu()


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def special_rows_bf16(K):
    def row(vals):
        r = np.zeros(K, np.uint16)
        r[:len(vals)] = vals
        return r
    rows = [np.zeros(K, np.uint16),                                   # all zero -> s = 1
            row([0x42FE, 0x3F00, 0x3FC0, 0x4020, 0xBF00, 0xC020, 0x427E, 0x427A, 0xC2FD]),  # ties
            row([0x74FE, 0x7220, 0x71C0, 0x7100, 0xF220]),             # beyond the fp16 range
            row([0x007F, 0x0003, 0x8001, 0x0040]),                     # subnormals
            np.where(np.arange(K) % 2 == 0, 0x7F7F, 0xFF7F).astype(np.uint16)]  # +- largest finite
    r = np.zeros(K, np.uint16)
    r[K - 1] = 0xC040                                                  # amax (-3) at the last element
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (37, 2560), (128, 4096), (5, 10240),
                                 (2, 16384), (3, 18432), (300, 2048)])
def test_quantize_act_bf16_bit_exact(cider, M, K):
    x = np.concatenate([inputs.activations_bf16(M, K, seed=200 + M), special_rows_bf16(K)])
    qa, sa = cider.cider_quantize_act_bf16(bf16_dev(x))
    qref, sref = oracle.quantize_act_bf16(x)
    assert_bits_equal(to_host(sa).view(np.uint32), sref.view(np.uint32), "s_a")
    assert_bits_equal(to_host(qa), qref, "q_a")


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x4049, 0x7F7F, 0x0080, 0x3A83])
def test_quantize_act_bf16_exhaustive_values(cider, amax_bits):
    """Every finite bf16 value with |x| <= amax, in rows that contain amax."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    allv = (allb.astype(np.uint32) << 16).view(np.float32)
    amax = (np.uint32(amax_bits) << 16).view(np.float32)
    with np.errstate(invalid="ignore"):
        vals = allb[np.isfinite(allv) & (np.abs(allv) <= amax)]
    W = 1024
    pad = (-len(vals)) % (W - 1)
    vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, W - 1)
    x = np.concatenate([np.full((vals.shape[0], 1), amax_bits, np.uint16), vals], axis=1)
    qa, sa = cider.cider_quantize_act_bf16(bf16_dev(x))
    qref, sref = oracle.quantize_act_bf16(x)
    assert_bits_equal(to_host(sa).view(np.uint32), sref.view(np.uint32), "s_a")
    assert_bits_equal(to_host(qa), qref, "q_a")


def make_weights(N, K, gs, bits, seed):
    W = inputs.weights(N, K, seed=seed)
    if bits == 8:
        qw, sw = oracle.quantize_weight_int8(W, gs)
        return qw, qw, sw
    q4, sw = oracle.quantize_weight_int4(W, gs)
    return oracle.pack_int4(q4), q4, sw


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 128])
@pytest.mark.parametrize("M,N,K", [(1, 264, 2560), (5, 136, 1024), (16, 264, 2048),
                                   (64, 256, 1024), (300, 264, 2560), (600, 520, 4096)])
def test_linear_bf16_matches_oracle(cider, M, N, K, gs, bits):
    x = inputs.activations_bf16(M, K, seed=300 + M)
    qw_dev, qw_vals, sw = make_weights(N, K, gs, bits, seed=301)
    fn = cider.cider_w8a8_linear_bf16 if bits == 8 else cider.cider_w4a8_linear_bf16
    y = to_host(fn(bf16_dev(x), to_dev(qw_dev), to_dev(sw), gs))
    yref = oracle.linear(x, qw_vals, sw, gs, threads=8, bf16=True)
    if gs == 0:
        assert_bits_equal(y, yref, f"bf16 linear M={M} N={N} K={K} bits={bits}")
    else:
        assert_fp16_close(y, yref, f"bf16 linear M={M} N={N} K={K} gs={gs} bits={bits}")


@pytest.mark.parametrize("nbytes", [1, 15, 16, 4096 + 7, 1 << 20])
def test_int4_from_offset_binary_bit_exact(cider, nbytes):
    rng = np.random.default_rng(nbytes)
    src = rng.integers(0, 256, size=nbytes, dtype=np.uint8)
    out = to_host(cider.cider_int4_from_offset_binary(to_dev(src)))
    assert_bits_equal(out, oracle.int4_from_offset_binary(src), "re-encoded bytes")
    t = to_dev(src)
    cider.cider_int4_from_offset_binary(t, out=t)                      # in place
    assert_bits_equal(to_host(t), oracle.int4_from_offset_binary(src), "in place")


def test_offset_binary_weights_give_the_same_linear(cider):
    """INT4 weights stored offset-binary, imported, then used by the W4A8
    linear: the same result as the two's complement weights."""
    M, N, K = 32, 264, 1024
    x = inputs.activations(M, K, seed=310)
    q4, sw = oracle.quantize_weight_int4(inputs.weights(N, K, seed=311), 0)
    offset = (((q4[:, 0::2] + 8) & 0xF) | (((q4[:, 1::2] + 8) & 0xF) << 4)).astype(np.uint8)
    imported = cider.cider_int4_from_offset_binary(to_dev(offset))
    y = to_host(cider.cider_w4a8_linear(to_dev(x), imported, to_dev(sw), 0))
    assert_bits_equal(y, oracle.linear(x, q4, sw, 0, threads=8), "imported weights")


def test_no_device_error_left(cider):
    assert cider.cider_check_device_error() == 0


# ---------------------------------------------------------------- bf16 outputs
def _bf16_as_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_bf16_close(y_bits, ref_bits, what=""):
    """|y - y_ref| <= 2e-3 max|y_ref| + 1 bf16 ulp(y_ref): the output
    tolerance, with the ulp of the output's own format."""
    y, r = _bf16_as_f64(y_bits), _bf16_as_f64(ref_bits)
    assert np.all(np.isfinite(r))
    ulp = np.spacing(np.abs(r).astype(np.float32)).astype(np.float64) * 2.0 ** 16
    bound = 2e-3 * np.max(np.abs(r)) + ulp
    bad = np.abs(y - r) > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance"


@pytest.mark.parametrize("x_bf16", [False, True])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 128, 64])
@pytest.mark.parametrize("M,N,K", [(1, 264, 1024), (3, 136, 2560), (16, 520, 4096), (2, 264, 8192),
                                   (200, 264, 1024), (300, 520, 2048)])
def test_linear_bf16_output_matches_oracle(cider, M, N, K, gs, bits, x_bf16):
    """y in bf16 through the small-M path (with and without K slices) and the
    two tensor-core GEMMs: per channel bit for bit, per group within the
    tolerance, against the oracle's single rounding of the same fp32 value."""
    if bits == 4 and gs == 64:
        pytest.skip("covered by the 8-bit case")
    if x_bf16:
        xb = inputs.activations_bf16(M, K, seed=600 + M)
        xd = bf16_dev(xb)
        x_or = xb
    else:
        x_or = inputs.activations(M, K, seed=600 + M)
        xd = to_dev(x_or)
    W = inputs.weights(N, K, seed=601)
    if bits == 8:
        qw, sw = oracle.quantize_weight_int8(W, gs)
        qv, fn = qw, cider.cider_w8a8_linear_ex
    else:
        q4, sw = oracle.quantize_weight_int4(W, gs)
        qw, qv, fn = oracle.pack_int4(q4), q4, cider.cider_w4a8_linear_ex
    y = fn(xd, to_dev(qw), to_dev(sw), gs, y_dtype=torch.bfloat16)
    assert y.dtype == torch.bfloat16
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.linear(x_or, qv, sw, gs, threads=8, bf16=x_bf16, out_bf16=True)
    what = f"bf16 y M={M} N={N} K={K} gs={gs} bits={bits} x_bf16={x_bf16}"
    if gs == 0:
        assert_bits_equal(yb, ref, what)
    else:
        assert_bf16_close(yb, ref, what)
    # fp16 output through the same entry point is the fp16 linear, bit for bit
    yh = fn(xd, to_dev(qw), to_dev(sw), gs, y_dtype=torch.float16)
    base = (cider.cider_w8a8_linear_bf16 if bits == 8 else cider.cider_w4a8_linear_bf16) if x_bf16 \
        else (cider.cider_w8a8_linear if bits == 8 else cider.cider_w4a8_linear)
    assert_bits_equal(to_host(yh), to_host(base(xd, to_dev(qw), to_dev(sw), gs)), what + " (fp16)")
