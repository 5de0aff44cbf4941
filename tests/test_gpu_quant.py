"""GPU parity of the quantization kernels against the oracle, bit-exact:
per-token activation quantization (codes and scales) and the INT8 / INT4
weight quantizers (codes, packed bytes and scales)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import (EXH_J, EXH_W, assert_bits_equal, exhaustive_rows,
                               positive_fp16, require_gpu, to_dev, to_host)
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


@pytest.mark.timeout(900)
def test_quantize_act_every_fp16_amax_and_value(cider):
    """Every positive finite fp16 amax (31743 values) with every finite fp16
    value |x| <= amax of both signs: about 1e9 (amax, x) pairs, all quantized
    by cider_quantize_act and compared bit for bit (codes and scales) with the
    oracle.  This covers the kernels' reciprocal-and-FMA division for every
    input an fp16 row can give it."""
    import os
    pos = positive_fp16()
    threads = max(1, min(16, os.cpu_count() or 1))
    n = len(pos)
    # chunks of about 24k rows (96 MB of fp16) each
    bounds = [0]
    rows_so_far = 0
    for i in range(n):
        rows_so_far += (i + EXH_J) // EXH_J
        if rows_so_far >= 24576:
            bounds.append(i + 1)
            rows_so_far = 0
    if bounds[-1] != n:
        bounds.append(n)
    pairs = 0
    for i0, i1 in zip(bounds[:-1], bounds[1:]):
        x = exhaustive_rows(pos, i0, i1)
        qa, sa = cider.cider_quantize_act(to_dev(x))
        qref, sref = oracle.quantize_act(x, threads=threads)
        assert_bits_equal(to_host(sa).view(np.uint32), sref.view(np.uint32),
                          f"s_a, amax {float(pos[i0])}..{float(pos[i1 - 1])}")
        assert_bits_equal(to_host(qa), qref, f"q_a, amax {float(pos[i0])}..{float(pos[i1 - 1])}")
        pairs += int(sum(2 * (i + 1) for i in range(i0, i1)))
    assert pairs > 1_000_000_000


def _sampled_amax_indices(count: int) -> np.ndarray:
    """Amax indices for the GEMV checks: the extremes, the subnormal /
    normal boundary, every power of two, and a seeded random sample."""
    pos = positive_fp16()
    fixed = {0, 1, 2, 1022, 1023, 1024, len(pos) - 1}
    fixed |= set(np.nonzero((pos.view(np.uint16) & 0x03FF) == 0)[0].tolist())   # powers of two
    rng = np.random.default_rng(2025)
    rest = rng.choice(len(pos), count - len(fixed), replace=False)
    return np.array(sorted(fixed | set(rest.tolist())))


@pytest.mark.parametrize("M", [1, 4])
def test_fused_gemv_quantization_sampled_fp16_values(cider, M):
    """The small-M GEMV quantizes the rows itself for one token (dp4a form)
    and for M * K <= 8192 (tensor-core form at M = 4).  Its codes are read
    back through selector weights (weight row n holds a single 1 at column n,
    so acc[m, n] = q_a[m, n]) and a power-of-two weight scale that keeps every
    product in the fp16 normal range, where distinct codes give distinct y:
    y must equal the oracle's dequantization of the oracle's codes, bit for
    bit, for every value |x| <= amax of about 600 amax values."""
    K = EXH_W
    pos = positive_fp16()
    idx = _sampled_amax_indices(600)
    rows = np.concatenate([exhaustive_rows(pos, i, i + 1) for i in idx])
    pad = (-len(rows)) % M
    rows = np.concatenate([rows, np.zeros((pad, K), np.float16)])
    sel = torch.eye(K, dtype=torch.int8, device="cuda")
    qref, sref = oracle.quantize_act(rows, threads=8)
    for r0 in range(0, len(rows), M):
        x = rows[r0:r0 + M]
        amax = float(np.abs(x.astype(np.float32)).max())
        # 2^e with amax * 2^e in [512, 1024): every |y| <= 127 s_a 2^e < 1024 and,
        # for nonzero codes, |y| >= s_a 2^e >= 4 (rows of one call share their amax
        # up to a factor 2^10 here, far inside the fp16 normal range)
        e = int(np.floor(np.log2(1024.0 / amax))) if amax > 0 else 0
        sw = np.full((K, 1), np.float32(2.0 ** e), np.float32)
        y = to_host(cider.cider_w8a8_linear(to_dev(x), sel, to_dev(sw), 0))
        acc = qref[r0:r0 + M].astype(np.int32)
        want = oracle.dequant_pc(acc, sref[r0:r0 + M], sw)
        assert_bits_equal(y, want, f"fused GEMV M={M}, rows {r0}..{r0 + M - 1}, amax {amax}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 64, 128])
@pytest.mark.parametrize("p", [99.9, 99.0, 50.0, 100.0, 0.1])
@pytest.mark.parametrize("N,K", [(16, 128), (40, 2560), (8, 12288)])
def test_quantize_weight_clip_bit_exact(cider, N, K, gs, p, bits):
    """Percentile-clipped weight scales and codes (the radix select of whole
    rows, the rank count of 64 / 128-element groups) bit for bit against the
    oracle, with ties, zero blocks and outliers planted."""
    W = inputs.weights(N, K, seed=int(p * 10) + K)
    W[1] = 0.0                                   # an all-zero row
    W[2, :64] = 0.0                              # an all-zero first group
    W[3, ::7] = 0.25                             # many equal values (ties)
    W[4, 5] = 3.0                                # one outlier above the clip
    W[5] = np.float32(0.0125)                    # a constant row
    fn = cider.cider_quantize_weight_int8 if bits == 8 else cider.cider_quantize_weight_int4
    qd, sd = fn(to_dev(W), gs, clip_percentile=p)
    if bits == 8:
        qref, sref = oracle.quantize_weight_int8(W, gs, clip_percentile=p)
    else:
        q4, sref = oracle.quantize_weight_int4(W, gs, clip_percentile=p)
        qref = oracle.pack_int4(q4)
    assert_bits_equal(to_host(sd).view(np.uint32), sref.view(np.uint32), f"clip s_w p={p} gs={gs}")
    assert_bits_equal(to_host(qd), qref, f"clip q_w p={p} gs={gs}")
