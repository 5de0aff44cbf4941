"""Pins for the CPU oracle: checks against facts fixed by the Cider README
(page "cider") and by mathematics, never against the oracle itself.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, round-half-away instead of half-even, a reciprocal
multiply instead of a divide, a transposed operand, a reversed group order)
fails at least one of them; ``test_oracle_mutations.py`` plants such mistakes
in a copy of the oracle and checks that these pins catch them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _blocks(path, keys):
    cur, out = {}, []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            cur[k.strip()] = v.split()
            if all(kk in cur for kk in keys):
                out.append(cur)
                cur = {}
    return out


# ------------------------------------------------------------ fp16 plumbing
def test_f16_decode_all_bit_patterns_match_numpy():
    """fp16 -> fp32 is exact; compare every bit pattern with numpy's decoder."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits[::257]], np.float32)
    np.testing.assert_array_equal(got, ref[::257])


def test_f32_to_f16_rounds_to_nearest_even_like_numpy():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 1000,
                           np.float32([65504, 65519.99, 65520, 1e-8, 2 ** -25, 3 * 2 ** -26,
                                       1 + 2 ** -11, 1 + 3 * 2 ** -11, -0.0])])
    got = np.array([oracle.f32_to_f16(float(v)) for v in vals], np.uint16)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------ a1 activation quant
def test_quantize_act_hand_worked_cases():
    for case in _blocks(os.path.join(GOLDEN, "quant_act_hand.txt"), ("x", "q", "s")):
        x = np.array([float(v) for v in case["x"]], np.float16)[None, :]
        qa, sa = oracle.quantize_act(x)
        assert qa[0].tolist() == [int(v) for v in case["q"]], case
        assert sa[0] == np.float32(float(case["s"][0]))


def _f32_div(a, b):
    """Correctly rounded binary32 a/b, from the exact quotient in binary64
    (53 >= 2*24 + 2, so rounding the double quotient to float is exact RN)."""
    return (np.asarray(a, np.float64) / np.asarray(b, np.float64)).astype(np.float32)


def _independent_quant_row(x16, qmax=127):
    xf = x16.astype(np.float64)
    amax = np.max(np.abs(xf))
    s = np.float32(1.0) if amax == 0 else _f32_div(amax, qmax)
    q = np.rint(_f32_div(xf, s).astype(np.float64))
    return np.clip(q, -qmax, qmax).astype(np.int8), np.float32(s)


# 0.0016956329345703125 and 0.50732421875 are amax values for which an IEEE
# divide and a reciprocal multiply give different codes for some fp16 x.
@pytest.mark.parametrize("amax", [65504.0, 1.0, 127.0, 3.140625, 0.0009765625,
                                  2.0 ** -24 * 37, 2.0 ** -14, 1000.0,
                                  0.0016956329345703125, 0.50732421875])
def test_quantize_act_brute_force_all_fp16_below_amax(amax):
    """Every fp16 value with |x| <= amax, quantized in rows that contain amax,
    against an independent binary64 computation of the same fp32 steps."""
    allv = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    ok = np.isfinite(allv) & (np.abs(allv.astype(np.float64)) <= amax)
    vals = allv[ok]
    W = 1024
    pad = (-len(vals)) % (W - 1)
    vals = np.concatenate([vals, np.zeros(pad, np.float16)]).reshape(-1, W - 1)
    x = np.concatenate([np.full((vals.shape[0], 1), amax, np.float16), vals], axis=1)
    qa, sa = oracle.quantize_act(x)
    for r in range(x.shape[0]):
        qref, sref = _independent_quant_row(x[r])
        assert sa[r] == sref
        np.testing.assert_array_equal(qa[r], qref)
    assert np.all(qa[:, 0] == 127)


def test_quantize_act_zero_row_and_signs():
    x = np.zeros((3, 64), np.float16)
    x[1, 5] = -3.0
    x[2] = np.linspace(-2, 2, 64).astype(np.float16)
    qa, sa = oracle.quantize_act(x)
    assert sa[0] == 1.0 and not qa[0].any()
    assert qa[1, 5] == -127 and np.count_nonzero(qa[1]) == 1
    assert qa[2, 0] == -127 and qa[2, -1] == 127
    # symmetric: negating x negates q and keeps s
    qn, sn = oracle.quantize_act(-x)
    np.testing.assert_array_equal(qn, -qa)
    np.testing.assert_array_equal(sn, sa)


def test_quantize_act_random_rows_match_independent():
    from w4a8_quantized_linear_gb300 import inputs
    x = inputs.activations(37, 320, seed=11)
    qa, sa = oracle.quantize_act(x)
    for r in range(x.shape[0]):
        qref, sref = _independent_quant_row(x[r])
        assert sa[r] == sref
        np.testing.assert_array_equal(qa[r], qref)


# ------------------------------------------------------------ a2 weight quant
def test_weight_quant_hand_worked_cases():
    path = os.path.join(GOLDEN, "weight_quant_hand.txt")
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, rest = line.split(None, 1)
            key, vals = rest.split(":", 1)
            rows.append((int(bits), key.strip(), vals.split()))
    for i in range(0, len(rows), 3):
        bits = rows[i][0]
        w = np.array([float(v) for v in rows[i][2]], np.float32)[None, :]
        fn = oracle.quantize_weight_int8 if bits == 8 else oracle.quantize_weight_int4
        q, s = fn(w, 0)
        assert q[0].tolist() == [int(v) for v in rows[i + 1][2]]
        assert s[0, 0] == np.float32(float(rows[i + 2][2][0]))


@pytest.mark.parametrize("gs", [0, 64, 128])
@pytest.mark.parametrize("bits", [8, 4])
def test_weight_quant_matches_independent_blockwise(gs, bits):
    from w4a8_quantized_linear_gb300 import inputs
    W = inputs.weights(9, 256, seed=3)
    W[2, :] = 0.0                      # zero row
    W[3, 64:128] = 0.0                 # zero block
    W[4, 7] = 0.5                      # dominant element
    qmax, qmin = (127, -127) if bits == 8 else (7, -8)
    fn = oracle.quantize_weight_int8 if bits == 8 else oracle.quantize_weight_int4
    q, s = fn(W, gs)
    g = gs or 256
    G = 256 // g
    assert s.shape == (9, G)
    for n in range(9):
        for j in range(G):
            blk = W[n, j * g:(j + 1) * g].astype(np.float64)
            amax = np.max(np.abs(blk))
            sref = np.float32(1.0) if amax == 0 else _f32_div(amax, qmax)
            qref = np.clip(np.rint(_f32_div(blk, sref).astype(np.float64)), qmin, qmax)
            assert s[n, j] == sref
            np.testing.assert_array_equal(q[n, j * g:(j + 1) * g], qref.astype(np.int8))
    assert np.abs(q).max() <= qmax and q.min() >= qmin
    # the element holding the block maximum maps to +-qmax
    assert q[4, 7] == qmax


# ------------------------------------------------------------ a4 int4 packing
def test_int4_nibbles_hand_worked():
    with open(os.path.join(GOLDEN, "int4_nibbles.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    packed = np.array([[int(r[0], 16) for r in rows]], np.uint8)
    q = oracle.unpack_int4(packed)[0]
    for i, r in enumerate(rows):
        assert (q[2 * i], q[2 * i + 1]) == (int(r[1]), int(r[2])), r


def test_int4_unpack_exhaustive_and_pack_roundtrip():
    allb = np.arange(256, dtype=np.uint8)[None, :]
    q = oracle.unpack_int4(allb)[0]
    for b in range(256):
        lo, hi = b & 15, b >> 4
        assert q[2 * b] == (lo - 16 if lo >= 8 else lo)
        assert q[2 * b + 1] == (hi - 16 if hi >= 8 else hi)
    np.testing.assert_array_equal(oracle.pack_int4(q[None, :]), allb)
    vals = np.array([(a, b) for a in range(-8, 8) for b in range(-8, 8)], np.int8).reshape(1, -1)
    np.testing.assert_array_equal(oracle.unpack_int4(oracle.pack_int4(vals)), vals)


# ------------------------------------------------------------ a3 integer GEMM
def test_gemm_closed_forms():
    K = 640
    a = np.full((2, K), 127, np.int8)
    w = np.full((3, K), 127, np.int8)
    assert np.all(oracle.gemm_acc(a, w) == 16129 * K)
    alt = np.tile(np.array([127, -127], np.int8), K // 2)[None, :]
    assert np.all(oracle.gemm_acc(alt, w) == 0)
    assert np.all(oracle.gemm_acc(a, -w) == -16129 * K)
    # selector weights pick activation columns: acc[m,n] = qa[m, sel[n]] * 1
    rng = np.random.default_rng(2)
    qa = rng.integers(-127, 128, (5, K), dtype=np.int8)
    sel = np.array([0, 3, K - 1, 200])
    qw = np.zeros((4, K), np.int8)
    qw[np.arange(4), sel] = 1
    np.testing.assert_array_equal(oracle.gemm_acc(qa, qw)[:, :, 0], qa[:, sel])
    # a weight row that is a basis vector times -7 at column 5
    qw2 = np.zeros((1, K), np.int8)
    qw2[0, 5] = -7
    np.testing.assert_array_equal(oracle.gemm_acc(qa, qw2)[:, 0, 0], -7 * qa[:, 5].astype(np.int32))


def test_gemm_brute_force_python_ints_and_group_sums():
    rng = np.random.default_rng(4)
    M, N, K = 3, 4, 256
    qa = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    for gs in (0, 64, 128):
        acc = oracle.gemm_acc(qa, qw, gs)
        g = gs or K
        for m in range(M):
            for n in range(N):
                for j in range(K // g):
                    ref = sum(int(qa[m, k]) * int(qw[n, k]) for k in range(j * g, (j + 1) * g))
                    assert acc[m, n, j] == ref
        # invariant: group accumulators sum to the per-channel one
        np.testing.assert_array_equal(acc.sum(axis=2), oracle.gemm_acc(qa, qw, 0)[:, :, 0])


def test_gemm_is_not_transposed():
    """Non-square case where acc[m,n] = <qa[m], qw[n]> differs from any
    transposed reading."""
    qa = np.array([[1, 2, 0, 0], [0, 0, 3, 0]], np.int8)
    qw = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 0, 1]], np.int8)
    acc = oracle.gemm_acc(qa, qw)[:, :, 0]
    np.testing.assert_array_equal(acc, [[1, 2, 0], [0, 0, 0]])


def test_gemm_overflow_is_reported():
    K = 133184                       # 16129 * K > 2^31 - 1
    a = np.full((1, K), 127, np.int8)
    with pytest.raises(OverflowError):
        oracle.gemm_acc(a, a)


# ------------------------------------------------------------ a5 dequant
def _r32(v):
    """Round an exact rational / double to binary32 (RN)."""
    return np.float32(float(v))


def test_dequant_pc_special_cases():
    acc = np.arange(-2048, 2049, dtype=np.int32)[None, :]
    N = acc.shape[1]
    y = oracle.dequant_pc(acc, np.float32([1.0]), np.ones(N, np.float32))
    np.testing.assert_array_equal(y.astype(np.float64), acc.astype(np.float64))
    # scaling s_w by 2 doubles y exactly (no overflow at these magnitudes)
    rng = np.random.default_rng(7)
    acc = rng.integers(-10 ** 6, 10 ** 6, (4, 50)).astype(np.int32)
    sa = rng.uniform(1e-3, 1e-1, 4).astype(np.float32)
    sw = rng.uniform(1e-5, 1e-3, 50).astype(np.float32)
    y1 = oracle.dequant_pc(acc, sa, sw)
    y2 = oracle.dequant_pc(acc, sa, sw * 2)
    np.testing.assert_array_equal(y2.astype(np.float32), y1.astype(np.float32) * 2)
    # overflow saturates to inf
    yo = oracle.dequant_pc(np.int32([[10 ** 9]]), np.float32([1.0]), np.float32([1.0]))
    assert np.isinf(yo[0, 0])


def test_dequant_pc_exact_emulation():
    """((float(acc) * s_a) * s_w) in binary32, emulated with exact rationals and
    one rounding per operation, then rounded to fp16."""
    rng = np.random.default_rng(8)
    acc = rng.integers(-(2 ** 27), 2 ** 27, (6, 40)).astype(np.int32)
    sa = rng.uniform(1e-4, 1.0, 6).astype(np.float32)
    sw = rng.uniform(1e-6, 1e-4, 40).astype(np.float32)
    y = oracle.dequant_pc(acc, sa, sw)
    for m in range(6):
        for n in range(40):
            a = _r32(int(acc[m, n]))                   # int32 -> fp32 RN
            t = _r32(Fraction(float(a)) * Fraction(float(sa[m])))
            t = _r32(Fraction(float(t)) * Fraction(float(sw[n])))
            assert y[m, n] == np.float16(t)


def test_dequant_pg_order_hand_worked():
    with open(os.path.join(GOLDEN, "dequant_order.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for r in rows:
        acc = np.array([[[int(r[0]), int(r[1]), int(r[2])]]], np.int32)
        y = oracle.dequant_pg(acc, np.float32([1.0]), np.ones((1, 3), np.float32))
        assert float(y[0, 0]) == float(r[3]), r


def test_dequant_pg_exact_emulation():
    rng = np.random.default_rng(9)
    M, N, G = 5, 7, 20
    acc = rng.integers(-(2 ** 21), 2 ** 21, (M, N, G)).astype(np.int32)
    sa = rng.uniform(1e-3, 1.0, M).astype(np.float32)
    sw = rng.uniform(1e-5, 1e-2, (N, G)).astype(np.float32)
    y = oracle.dequant_pg(acc, sa, sw)
    for m in range(M):
        for n in range(N):
            s = np.float32(0)
            for g in range(G):
                sc = _r32(Fraction(float(sa[m])) * Fraction(float(sw[n, g])))
                term = _r32(Fraction(float(sc)) * int(acc[m, n, g]))
                s = _r32(Fraction(float(s)) + Fraction(float(term)))
            assert y[m, n] == np.float16(s)


# ------------------------------------------------------------ whole layer
def test_linear_is_composition_and_rows_are_independent():
    from w4a8_quantized_linear_gb300 import inputs
    x, W = inputs.layer(19, 48, 256)
    for gs in (0, 64, 128):
        qw, sw = oracle.quantize_weight_int8(W, gs)
        qa, sa = oracle.quantize_act(x)
        acc = oracle.gemm_acc(qa, qw, gs)
        yref = oracle.dequant_pg(acc, sa, sw) if gs else oracle.dequant_pc(acc, sa, sw)
        y = oracle.linear(x, qw, sw, gs)
        np.testing.assert_array_equal(y.view(np.uint16), yref.view(np.uint16))
        rows = [18, 3, 7]
        np.testing.assert_array_equal(oracle.linear(x, qw, sw, gs, rows=rows).view(np.uint16),
                                      yref[rows].view(np.uint16))
        np.testing.assert_array_equal(oracle.linear(x, qw, sw, gs, threads=4).view(np.uint16),
                                      yref.view(np.uint16))


def test_linear_close_to_unquantized_product():
    """Sanity (not a parity pin): the quantized layer approximates x W^T."""
    from w4a8_quantized_linear_gb300 import inputs
    x, W = inputs.layer(32, 64, 512)
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    for bits, gs in ((8, 0), (8, 128), (4, 128)):
        if bits == 8:
            qw, sw = oracle.quantize_weight_int8(W, gs)
        else:
            qw, sw = oracle.quantize_weight_int4(W, gs)
        y = oracle.linear(x, qw, sw, gs).astype(np.float64)
        cos = (y * ref).sum() / np.sqrt((y * y).sum() * (ref * ref).sum())
        assert cos > (0.99 if bits == 8 else 0.95), (bits, gs, cos)


# ------------------------------------------------------------ a1 with bf16 activations
def _bf16_to_f32(bits):
    """bf16 bit patterns -> fp32 values, by definition (the upper half of an
    IEEE binary32)."""
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_bf16_widening_matches_torch_for_every_pattern():
    """The oracle's bf16 reading of every bit pattern equals PyTorch's own
    bf16 -> fp32 conversion (a library routine independent of the oracle):
    a row holding one pattern at a time quantizes against amax = |x|."""
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(_bf16_to_f32(bits)[np.isfinite(ref)], ref[np.isfinite(ref)])
    finite = bits[np.isfinite(ref) & (np.abs(ref) > 0)]
    qa, sa = oracle.quantize_act_bf16(finite[:, None])
    np.testing.assert_array_equal(sa, _f32_div(np.abs(ref[np.isfinite(ref) & (np.abs(ref) > 0)]), 127))
    assert np.all(np.abs(qa[:, 0]) == 127)


def test_quantize_act_bf16_hand_worked_cases():
    for case in _blocks(os.path.join(GOLDEN, "quant_act_bf16_hand.txt"), ("x", "q", "s")):
        x = np.array([int(v, 16) for v in case["x"]], np.uint16)[None, :]
        qa, sa = oracle.quantize_act_bf16(x)
        assert qa[0].tolist() == [int(v) for v in case["q"]], case
        assert sa[0] == np.float32(float.fromhex(case["s"][0])), case


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x42FE, 0x4049, 0x7F7F, 0x0080, 0x007F, 0x3A83])
def test_quantize_act_bf16_brute_force_all_bf16_below_amax(amax_bits):
    """Every finite bf16 value with |x| <= amax (1, 127, 3.140625, the largest
    finite, the smallest normal, a subnormal, ~0.001), in rows that contain
    amax, against an independent binary64 computation of the same steps."""
    amax = float(_bf16_to_f32([amax_bits])[0])
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    allv = _bf16_to_f32(allb)
    with np.errstate(invalid="ignore"):
        ok = np.isfinite(allv) & (np.abs(allv.astype(np.float64)) <= amax)
    vals = allb[ok]
    W = 1024
    pad = (-len(vals)) % (W - 1)
    vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, W - 1)
    x = np.concatenate([np.full((vals.shape[0], 1), amax_bits, np.uint16), vals], axis=1)
    qa, sa = oracle.quantize_act_bf16(x)
    for r in range(x.shape[0]):
        xf = _bf16_to_f32(x[r]).astype(np.float64)
        s = _f32_div(np.max(np.abs(xf)), 127)
        q = np.clip(np.rint(_f32_div(xf, s).astype(np.float64)), -127, 127).astype(np.int8)
        assert sa[r] == s
        np.testing.assert_array_equal(qa[r], q)


def test_quantize_act_bf16_agrees_with_fp16_on_shared_values():
    """Values exact in both formats quantize identically from either."""
    rng = np.random.default_rng(21)
    ints = rng.integers(-255, 256, size=(9, 200))
    x = (ints * np.float32(2.0) ** rng.integers(-8, 3, size=(9, 1))).astype(np.float32)
    x16 = x.astype(np.float16)
    assert np.array_equal(x16.astype(np.float32), x)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_bf16_to_f32(xb), x)
    q1, s1 = oracle.quantize_act(x16)
    q2, s2 = oracle.quantize_act_bf16(xb)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)


def test_linear_bf16_is_composition():
    rng = np.random.default_rng(22)
    xb = (rng.standard_normal((5, 256)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qw = rng.integers(-127, 128, size=(24, 256)).astype(np.int8)
    sw = rng.random(24).astype(np.float32) * 0.01
    y = oracle.linear(xb, qw, sw, 0, bf16=True)
    qa, sa = oracle.quantize_act_bf16(xb)
    np.testing.assert_array_equal(y.view(np.uint16),
                                  oracle.dequant_pc(oracle.gemm_acc(qa, qw, 0)[:, :, 0], sa, sw).view(np.uint16))


# ------------------------------------------------------------ offset-binary INT4 import
def test_int4_offset_binary_hand_worked():
    """"Symmetric INT4 (zp=8)" ("Quantization" table): nibble u holds u - 8.
    0x00 -> (-8, -8) -> 0x88; 0x88 -> (0, 0) -> 0x00; 0xFF -> (7, 7) -> 0x77;
    0x80 -> (-8, 0) -> 0x08; 0x08 -> (0, -8) -> 0x80; 0x9A -> (2, 1) -> 0x12."""
    src = np.array([0x00, 0x88, 0xFF, 0x80, 0x08, 0x9A], np.uint8)
    assert oracle.int4_from_offset_binary(src).tolist() == [0x88, 0x00, 0x77, 0x08, 0x80, 0x12]


def test_int4_offset_binary_exhaustive():
    """All 256 bytes: the re-encoded nibbles decode (two's complement, low
    nibble first) to the offset values u - 8."""
    src = np.arange(256, dtype=np.uint8)
    dst = oracle.int4_from_offset_binary(src)
    vals = oracle.unpack_int4(dst[None, :])[0].astype(np.int16)
    np.testing.assert_array_equal(vals[0::2], (src & 0xF).astype(np.int16) - 8)
    np.testing.assert_array_equal(vals[1::2], (src >> 4).astype(np.int16) - 8)


# ---------------------------------------------------------------- bf16 outputs
def _torch_bf16_bits(v: np.ndarray) -> np.ndarray:
    """PyTorch's fp32 -> bf16 conversion (round to nearest even), as uint16."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_bf16_output_rounding_matches_pytorch():
    """The oracle's fp32 -> bf16 rounding against PyTorch's conversion: every
    tie pattern around 1.0 and 2^-126, values past the bf16 range, bf16 and
    fp32 subnormals, signs, and random values."""
    ties = []
    for base in (0x3F800000, 0x3F810000, 0x00800000, 0x7F7F0000, 0x00010000):
        for low in (0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
            ties.append(base | low)
    rng = np.random.default_rng(5)
    bits = np.concatenate([np.array(ties, np.uint32), rng.integers(0, 0x7F800000, 20000, dtype=np.uint32)])
    bits = np.concatenate([bits, bits | 0x80000000])
    vals = bits.view(np.float32)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, _torch_bf16_bits(vals))
    # one hand case per rule: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 (even: 1),
    # 1 + 3 * 2^-8 halfway between 1 + 2^-7 and 1 + 2^-6 (even: the latter); the
    # largest fp32 rounds past the bf16 range to +inf
    assert oracle.f32_to_bf16(1.00390625) == 0x3F80
    assert oracle.f32_to_bf16(1.01171875) == 0x3F82
    assert oracle.f32_to_bf16(float(np.finfo(np.float32).max)) == 0x7F80


def test_dequant_bf16_special_cases():
    """s_a = s_w = 1 and |acc| <= 256: y is acc exactly (integers up to 2^8
    are bf16 values); per group with one group equals per channel; doubling
    every s_w doubles y; and where the fp32 result is exact in both formats
    (small integers) the bf16 and fp16 outputs hold the same value."""
    acc = np.arange(-256, 257, dtype=np.int32).reshape(1, -1)
    ones_a = np.ones(1, np.float32)
    ones_w = np.ones(acc.shape[1], np.float32)
    y = oracle.dequant_pc(acc, ones_a, ones_w, bf16=True)
    assert np.array_equal(y, _torch_bf16_bits(acc.astype(np.float32)))
    assert np.array_equal((y.astype(np.uint32) << 16).view(np.float32), acc.astype(np.float32))
    yh = oracle.dequant_pc(acc, ones_a, ones_w)
    assert np.array_equal((y.astype(np.uint32) << 16).view(np.float32), yh.astype(np.float32))
    rng = np.random.default_rng(6)
    acc = rng.integers(-2 ** 20, 2 ** 20, (4, 40)).astype(np.int32)
    sa = (rng.random(4) * 1e-2 + 1e-3).astype(np.float32)
    sw = (rng.random(40) * 1e-3 + 1e-4).astype(np.float32)
    ypc = oracle.dequant_pc(acc, sa, sw, bf16=True)
    assert np.array_equal(oracle.dequant_pg(acc[:, :, None], sa, sw[:, None], bf16=True), ypc)
    y2 = oracle.dequant_pc(acc, sa, 2 * sw, bf16=True)
    assert np.array_equal((y2.astype(np.uint32) << 16).view(np.float32),
                          2 * (ypc.astype(np.uint32) << 16).view(np.float32))


def test_linear_bf16_output_is_the_fp16_paths_fp32_value_rounded_otherwise():
    """The whole layer with bf16 y and with fp16 y differ only in the last
    rounding: both are within half an ulp (of their own format) of one fp32
    value, so the two outputs lie within half a bf16 ulp plus half an fp16 ulp
    of each other, and they agree exactly wherever that fp32 value is exact in
    both formats (checked via all-zero rows)."""
    from w4a8_quantized_linear_gb300 import inputs
    x = inputs.activations(6, 256, seed=3)
    x[2] = 0
    W = inputs.weights(40, 256, seed=4)
    for gs in (0, 64):
        qw, sw = oracle.quantize_weight_int8(W, gs)
        yb = oracle.linear(x, qw, sw, gs, out_bf16=True)
        yh = oracle.linear(x, qw, sw, gs)
        fb = (yb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        fh = yh.astype(np.float64)
        ulp_b = np.spacing(np.abs(fb).astype(np.float32)).astype(np.float64) * 2.0 ** 16
        ulp_h = np.spacing(np.abs(yh)).astype(np.float64)
        assert np.all(np.abs(fb - fh) <= 0.5 * ulp_b + 0.5 * ulp_h)
        assert np.all(fb[2] == 0) and np.all(fh[2] == 0)


# ---------------------------------------------------------------- clipped scales
def _read_clip_golden():
    here = os.path.dirname(os.path.abspath(__file__))
    blocks = {"arange1_100": np.arange(1, 101, dtype=np.float32),
              "m3_1_2_4": np.array([-3, 1, 2, 4], np.float32),
              "z0_0_0_5": np.array([0, 0, 0, 5], np.float32)}
    rows = []
    with open(os.path.join(here, "golden", "clip_percentile_hand.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, p, qmax, s_hex, codes = [t.strip() for t in line.split("|")]
            rows.append((blocks[name], float(p), int(qmax), int(s_hex, 16),
                         np.array(codes.split(), np.int64)))
    return rows


def test_clip_percentile_hand_worked_cases():
    for blk, p, qmax, s_bits, codes in _read_clip_golden():
        W = blk.reshape(1, -1)
        if qmax == 127:
            q, s = oracle.quantize_weight_int8(W, 0, clip_percentile=p)
        else:
            q, s = oracle.quantize_weight_int4(W, 0, clip_percentile=p)
        assert int(s.view(np.uint32)[0, 0]) == s_bits, (blk, p, hex(int(s.view(np.uint32)[0, 0])))
        assert np.array_equal(q[0, -len(codes):].astype(np.int64), codes), (blk, p, q)


@pytest.mark.parametrize("gs", [0, 64, 128])
def test_clip_percentile_100_is_min_max(gs):
    from w4a8_quantized_linear_gb300 import inputs
    W = inputs.weights(24, 512, seed=9)
    W[3] = 0
    for f in (oracle.quantize_weight_int8, oracle.quantize_weight_int4):
        q1, s1 = f(W, gs, clip_percentile=100.0)
        q0, s0 = f(W, gs)
        assert np.array_equal(q1, q0) and np.array_equal(s1.view(np.uint32), s0.view(np.uint32))


@pytest.mark.parametrize("n", [4, 64, 128, 2560])
@pytest.mark.parametrize("p", [99.9, 99.0, 95.0, 50.0, 0.1])
def test_clip_percentile_matches_numpy_linear_percentile(n, p):
    """The clip value behind each scale against numpy.percentile (linear
    interpolation between closest ranks, computed in float64): equal to a few
    fp32 roundings (the oracle's interpolation is in fp32)."""
    rng = np.random.default_rng(n + int(p * 10))
    W = (rng.standard_normal((8, n)) * 0.02).astype(np.float32)
    q, s = oracle.quantize_weight_int8(W, 0, clip_percentile=p)
    want = np.percentile(np.abs(W).astype(np.float64), p, axis=1, method="linear") / 127.0
    assert np.allclose(s[:, 0].astype(np.float64), want, rtol=4e-7, atol=0)
