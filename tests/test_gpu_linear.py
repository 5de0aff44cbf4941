"""GPU parity of the integer GEMM paths (small-M GEMV and tensor-core GEMM)
against the oracle.

* int32 accumulators (per channel and per group): bit-exact, including
  adversarial inputs whose sums exceed 2^24 (the fp32 significand) and mixes
  of large and small products;
* fp16 outputs: per channel bit-exact (same operation order as the oracle),
  per group within |y - y_ref| <= 2e-3 max|y_ref| + 1 ulp;
* the pre-quantized entry points give the same bits as the fused ones;
* at the benchmark's full sizes, sampled rows against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.parity_util import (assert_bits_equal, assert_fp16_close, require_gpu, to_dev,
                               to_host)
from w4a8_quantized_linear_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cider():
    return require_gpu()


def make_weights(N, K, gs, bits, seed):
    W = inputs.weights(N, K, seed=seed)
    if bits == 8:
        qw, sw = oracle.quantize_weight_int8(W, gs)
        return qw, qw, sw
    q4, sw = oracle.quantize_weight_int4(W, gs)
    return oracle.pack_int4(q4), q4, sw


def run_acc(cider, qa, qw_dev_arr, gs, bits):
    fn = cider.cider_w8a8_accumulators if bits == 8 else cider.cider_w4a8_accumulators
    return to_host(fn(to_dev(qa), to_dev(qw_dev_arr), gs))


def run_linear(cider, x, qw_dev_arr, sw, gs, bits):
    fn = cider.cider_w8a8_linear if bits == 8 else cider.cider_w4a8_linear
    return to_host(fn(to_dev(x), to_dev(qw_dev_arr), to_dev(sw), gs))


SHAPES = [  # (M, N, K): GEMV bucket (M <= 16) and GEMM tiles with ragged edges
    (1, 8, 128), (1, 136, 2560), (3, 64, 544), (5, 256, 1024), (16, 200, 2048),
    (17, 136, 128), (64, 256, 576), (128, 128, 2560), (130, 264, 1088), (300, 200, 2048),
    (257, 384, 4096), (300, 136, 4608), (40, 264, 6144),
]


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 64, 128])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_accumulators_bit_exact(cider, M, N, K, gs, bits):
    if gs and K % gs:
        pytest.skip("K not a multiple of the group size")
    x = inputs.activations(M, K, seed=M + 3)
    qa, _ = oracle.quantize_act(x)
    qw_dev, qw_vals, _ = make_weights(N, K, gs, bits, seed=N + K)
    acc = run_acc(cider, qa, qw_dev, gs, bits)
    assert_bits_equal(acc, oracle.gemm_acc(qa, qw_vals, gs), f"acc M={M} N={N} K={K} gs={gs}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("M", [4, 160])
def test_accumulators_exact_beyond_fp32_significand(cider, M, bits):
    """All codes at the extreme: |acc| = 16129 K (8-bit) reaches 8.3e7 > 2^24
    at K = 5120; plus rows mixing large products with +-1 products."""
    N, K = 136, (2560 if M == 4 else 5120)
    qa = np.full((M, K), 127, np.int8)
    qa[1::2] = -127
    qa[2, :] = 1
    qa[3, 511::512] = 1                      # small terms right after a full chunk of big ones
    if bits == 8:
        qw_vals = np.full((N, K), 127, np.int8)
        qw_vals[5, ::3] = -1
        qw_vals[6, 1::2] = 1
        qw_dev = qw_vals
    else:
        qw_vals = np.full((N, K), -8, np.int8)
        qw_vals[5, ::3] = 7
        qw_vals[6, 1::2] = 1
        qw_dev = oracle.pack_int4(qw_vals)
    for gs in (0, 64, 128):
        acc = run_acc(cider, qa, qw_dev, gs, bits)
        assert_bits_equal(acc, oracle.gemm_acc(qa, qw_vals, gs), f"extreme acc gs={gs}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 64, 128])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_matches_oracle(cider, M, N, K, gs, bits):
    if gs and K % gs:
        pytest.skip("K not a multiple of the group size")
    x = inputs.activations(M, K, seed=M + 5)
    qw_dev, qw_vals, sw = make_weights(N, K, gs, bits, seed=N + K + 1)
    y = run_linear(cider, x, qw_dev, sw, gs, bits)
    yref = oracle.linear(x, qw_vals, sw, gs)
    if gs == 0:
        assert_bits_equal(y, yref, f"y per-channel M={M} N={N} K={K}")
    else:
        assert_fp16_close(y, yref, f"y per-group M={M} N={N} K={K} gs={gs}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 128])
@pytest.mark.parametrize("M", [7, 200])
def test_prequant_equals_fused(cider, M, gs, bits):
    N, K = 264, 1024
    x = inputs.activations(M, K, seed=21)
    qw_dev, _, sw = make_weights(N, K, gs, bits, seed=22)
    xd = to_dev(x)
    qa, sa = cider.cider_quantize_act(xd)
    fn_pre = cider.cider_w8a8_linear_prequant if bits == 8 else cider.cider_w4a8_linear_prequant
    y_pre = to_host(fn_pre(qa, sa, to_dev(qw_dev), to_dev(sw), gs))
    y = run_linear(cider, x, qw_dev, sw, gs, bits)
    assert_bits_equal(y_pre, y, "prequant vs fused")


def test_zero_activation_rows_give_zero(cider):
    M, N, K = 130, 136, 512
    x = inputs.activations(M, K, seed=30)
    x[::3] = 0
    qw_dev, qw_vals, sw = make_weights(N, K, 0, 8, seed=31)
    y = run_linear(cider, x, qw_dev, sw, 0, 8)
    assert not np.any(y[::3].astype(np.float32))
    assert_bits_equal(y, oracle.linear(x, qw_vals, sw, 0), "zero rows")


# Full-size workloads: sampled rows against the oracle (rows are independent,
# so a row subset of the oracle is exact).
FULL = [
    # (M, N, K, gs, bits)
    (4096, 10240, 2560, 0, 8),      # benchmark headline
    (8192, 2560, 10240, 0, 8),
    (4096, 10240, 2560, 128, 8),
    (4096, 10240, 2560, 64, 8),
    (4096, 10240, 2560, 128, 4),
    (3455, 6144, 2048, 0, 8),       # Qwen3-2B-shaped gate/up at the longest prefill
    (4096, 12288, 4096, 128, 4),    # Qwen3-8B-shaped gate/up
    (1, 10240, 2560, 0, 8),
    (16, 2560, 10240, 128, 4),
    (1, 4096, 12288, 128, 8),       # Qwen3-8B-shaped down projection, decode
]


@pytest.mark.parametrize("M,N,K,gs,bits", FULL)
def test_full_size_sampled_rows(cider, M, N, K, gs, bits):
    x = inputs.activations(M, K, seed=0)
    qw_dev, qw_vals, sw = make_weights(N, K, gs, bits, seed=1)
    y = run_linear(cider, x, qw_dev, sw, gs, bits)
    rng = np.random.default_rng(M + N)
    rows = sorted(set([0, M - 1, M // 2] + list(rng.integers(0, M, 5))))
    yref = oracle.linear(x, qw_vals, sw, gs, rows=rows, threads=8)
    if gs == 0:
        assert_bits_equal(y[rows], yref, f"full-size rows M={M} N={N} K={K}")
    else:
        assert_fp16_close(y[rows], yref, f"full-size rows M={M} N={N} K={K} gs={gs}")


def test_single_layer_workload_all_rows(cider):
    """The single W8A8 per-channel layer workload (x fp16 [128, 2560], W [2560,
    2560], seed 0): every output against the oracle, bit for bit."""
    M, N, K = 128, 2560, 2560
    x, W = inputs.layer(M, N, K, base_seed=0, index=0)
    qw, sw = oracle.quantize_weight_int8(W, 0)
    y = run_linear(cider, x, qw, sw, 0, 8)
    assert_bits_equal(y, oracle.linear(x, qw, sw, 0, threads=8), "single layer, all rows")


@pytest.mark.parametrize("bits", [8, 4])
def test_whole_rounds_then_cut_tiles_all_outputs(cider, bits):
    """A shape whose per-channel GEMM runs a whole round of 256 x 256 tiles and
    then cuts the remaining tiles along K into pieces that add up each
    other's partial sums: every output and every accumulator, bit for bit."""
    M, N, K = 2560, 2048, 4096
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    info, _ = cider.cider_debug_pair_schedule(M, N, K, pairs)
    if not (info["whole_tiles"] > 0 and info["cut_tiles"] > 0):
        pytest.skip(f"no cut on this device: {info}")
    x = inputs.activations(M, K, seed=123)
    qw_dev, qw_vals, sw = make_weights(N, K, 0, bits, seed=124)
    y = run_linear(cider, x, qw_dev, sw, 0, bits)
    assert_bits_equal(y, oracle.linear(x, qw_vals, sw, 0, threads=8), f"cut tiles y bits={bits}")
    qa, _ = oracle.quantize_act(x)
    acc = run_acc(cider, qa, qw_dev, 0, bits)
    assert_bits_equal(acc, oracle.gemm_acc(qa, qw_vals, 0), f"cut tiles acc bits={bits}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("gs", [0, 128])
@pytest.mark.parametrize("M,N,K", [(2, 264, 8192), (5, 136, 6144), (16, 264, 8192),
                                   (1, 520, 12288)])
def test_small_m_split_k_all_outputs(cider, M, N, K, gs, bits):
    """Few weight-row blocks with long rows: the small-M path cuts K into
    slices on separate CTAs and adds their partial sums in a second kernel.
    Every output against the oracle (per channel bit for bit), through both
    the fused and the pre-quantized entry points."""
    x = inputs.activations(M, K, seed=400 + M)
    qw_dev, qw_vals, sw = make_weights(N, K, gs, bits, seed=401)
    yref = oracle.linear(x, qw_vals, sw, gs, threads=8)
    y = run_linear(cider, x, qw_dev, sw, gs, bits)
    qa, sa = cider.cider_quantize_act(to_dev(x))
    pre = cider.cider_w8a8_linear_prequant if bits == 8 else cider.cider_w4a8_linear_prequant
    y2 = to_host(pre(qa, sa, to_dev(qw_dev), to_dev(sw), gs))
    if gs == 0:
        assert_bits_equal(y, yref, f"split-K small M={M} N={N} K={K} bits={bits}")
        assert_bits_equal(y2, yref, f"split-K small prequant M={M} bits={bits}")
    else:
        assert_fp16_close(y, yref, f"split-K small M={M} N={N} K={K} gs={gs} bits={bits}")
        assert_fp16_close(y2, yref, f"split-K small prequant M={M} gs={gs} bits={bits}")


@pytest.mark.parametrize("M,N,K,gs,bits", [(16, 264, 8192, 0, 8), (16, 264, 8192, 128, 4),
                                           (8, 1024, 2048, 0, 4), (300, 264, 1024, 0, 8),
                                           (200, 136, 1024, 128, 8)])
def test_back_to_back_calls_on_one_stream(cider, M, N, K, gs, bits):
    """Several calls with different rows, enqueued one after another on one
    stream with no synchronization between them.  Inside a call the later
    launches (GEMV or GEMM, K-slice combine) start before the earlier ones
    end and wait for their results; the calls reuse the same scratch for the
    codes.  Every call's result against the oracle (per channel bit for bit)."""
    qw_dev, qw_vals, sw = make_weights(N, K, gs, bits, seed=501)
    qw_d, sw_d = to_dev(qw_dev), to_dev(sw)
    lin = cider.cider_w8a8_linear if bits == 8 else cider.cider_w4a8_linear
    xs = [inputs.activations(M, K, seed=510 + i) for i in range(6)]
    xd = [to_dev(x) for x in xs]
    torch.cuda.synchronize()
    ys = [lin(x, qw_d, sw_d, gs) for x in xd]
    torch.cuda.synchronize()
    for i, (x, y) in enumerate(zip(xs, ys)):
        yref = oracle.linear(x, qw_vals, sw, gs, threads=8)
        if gs == 0:
            assert_bits_equal(to_host(y), yref, f"back-to-back call {i} M={M} N={N} K={K}")
        else:
            assert_fp16_close(to_host(y), yref, f"back-to-back call {i} M={M} N={N} K={K} gs={gs}")


def test_no_device_error_left(cider):
    assert cider.cider_check_device_error() == 0


def test_bounded_wait_reports_timeout(cider):
    """A kernel waiting on a barrier nothing completes gives up after the poll
    limit, sets the device error word, and the context stays usable."""
    assert cider.cider_debug_wait_timeout(1000) == 0
    assert cider.cider_check_device_error() == 5
    assert cider.cider_check_device_error() == 0
    x = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
    qa, sa = cider.cider_quantize_act(x)
    torch.cuda.synchronize()
    assert float(sa.sum()) == 2.0


def test_kernel_timing_facility(cider):
    M, N, K = 256, 512, 1024
    x = torch.from_numpy(inputs.activations(M, K, seed=3)).cuda()
    qw, sw = cider.cider_quantize_weight_int8(torch.from_numpy(inputs.weights(N, K)).cuda(), 0)
    cider.cider_timing_begin(2)
    for _ in range(3):                     # the third call is beyond the capacity: untimed
        cider.cider_w8a8_linear(x, qw, sw, 0)
    n, ms = cider.cider_timing_end()
    assert n == 2 and ms > 0.0
    n, ms = cider.cider_timing_end()       # timing is off again
    assert n == 0 and ms == 0.0


@pytest.mark.parametrize("bits,K", [(8, 2560), (4, 10240), (8, 6144)])
def test_mixed_fast_and_slow_token_tiles(cider, bits, K):
    """The per-channel kernel decides per 256-token tile whether one fp32
    accumulation over all of K is provably exact; tiles with extreme
    activations take the chunked exact path.  Mix both kinds in one call."""
    M, N = 700, 264
    x = inputs.activations(M, K, seed=77)
    rng = np.random.default_rng(78)
    # rows of the second token tile: every code at +-127 (sum |q| = 127 K)
    x[256:512] = (rng.choice([-1.0, 1.0], size=(256, K)) * 3.0).astype(np.float16)
    qw_dev, qw_vals, sw = make_weights(N, K, 0, bits, seed=79)
    qa, _ = oracle.quantize_act(x)
    assert np.abs(qa[300].astype(np.int64)).sum() == 127 * K
    acc = run_acc(cider, qa, qw_dev, 0, bits)
    assert_bits_equal(acc, oracle.gemm_acc(qa, qw_vals, 0), f"mixed-tile acc bits={bits}")
    y = run_linear(cider, x, qw_dev, sw, 0, bits)
    assert_bits_equal(y, oracle.linear(x, qw_vals, sw, 0, threads=8), f"mixed-tile y bits={bits}")


@pytest.mark.parametrize("M,N,K,gs,bits", [(1, 264, 1024, 0, 8), (16, 136, 2048, 128, 4),
                                           (16, 2560, 10240, 0, 8), (16, 2560, 10240, 128, 4),
                                           (300, 264, 1024, 0, 8), (200, 136, 1024, 64, 8)])
def test_linear_replays_from_cuda_graph(cider, M, N, K, gs, bits):
    """The entry points enqueue only stream-ordered work (kernels, pool
    allocations), so a captured call replays to the same bits as an eager one.
    The small-M shapes include the quantization -> GEMV -> K-slice combine
    chain, whose later launches may start before the earlier ones end."""
    x = to_dev(inputs.activations(M, K, seed=90))
    qw_dev, _, sw = make_weights(N, K, gs, bits, seed=91)
    qw_d, sw_d = to_dev(qw_dev), to_dev(sw)
    lin = cider.cider_w8a8_linear if bits == 8 else cider.cider_w4a8_linear
    want = lin(x, qw_d, sw_d, gs)
    y = torch.zeros_like(want)
    lin(x, qw_d, sw_d, gs, out=y)              # warm-up outside capture
    torch.cuda.synchronize()
    y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lin(x, qw_d, sw_d, gs, out=y)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(to_host(y), to_host(want), "graph replay")


def test_kernel_timing_inside_cuda_graph(cider):
    M, N, K = 1, 1024, 2048
    x = torch.from_numpy(inputs.activations(M, K, seed=3)).cuda()
    qw, sw = cider.cider_quantize_weight_int8(torch.from_numpy(inputs.weights(N, K)).cuda(), 0)
    y = cider.cider_w8a8_linear(x, qw, sw, 0)
    torch.cuda.synchronize()
    cider.cider_timing_begin(2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cider.cider_w8a8_linear(x, qw, sw, 0, out=y)
        cider.cider_w8a8_linear(x, qw, sw, 0, out=y)
    g.replay()
    n, ms = cider.cider_timing_end()
    assert n == 2 and 0.0 < ms < 100.0


def _rows_with_l1(targets, K, rng):
    """fp16 activation rows whose codes are exactly chosen: each row holds
    127 (so s_a = 127 / 127 = 1 and q = x, integers exact in fp16) and has
    sum_k |q| = target, all codes >= 0: floor(target / 127) codes of 127 and
    one code of target % 127, at random positions."""
    x = np.zeros((len(targets), K), np.float16)
    for r, t in enumerate(targets):
        n127, rem = divmod(int(t), 127)
        assert n127 >= 1 and n127 + (rem > 0) <= K
        cols = rng.permutation(K)[:n127 + 1]
        x[r, cols[:n127]] = 127
        if rem:
            x[r, cols[n127]] = rem
    return x


@pytest.mark.parametrize("bits", [8, 4])
def test_fast_tile_bound_at_its_limit(cider, bits):
    """The per-channel kernel runs a 256-token tile as one fp32 accumulation
    over all of K when every token satisfies qmax_w * sum_k |q_a| <= 2^23
    (qmax_w = 127 for INT8, 8 for INT4), else as exact chunked passes.

    Token tile 0: every row exactly at the limit sum |q_a| = floor(2^23 /
    qmax_w) (fast tile), with a weight row of constant sign so the partial
    sums climb to ~8.39e6.  Tile 1: the same plus one row at limit + 1 (the
    whole tile must take the chunked path).  Tile 2 (ragged): rows whose
    weight-row-0 sum is odd and above 2^24, which one fp32 accumulation cannot
    represent, so only the chunked path gets them right.  Accumulators and y
    bit for bit against the oracle."""
    qmax = 127 if bits == 8 else 8
    limit = (1 << 23) // qmax
    # INT4 needs longer rows to reach its limit (2^20 / 127 codes of 127) and an odd
    # weight (7) whose product sum passes 2^24
    K = 2560 if bits == 8 else 20480
    wbig = 127 if bits == 8 else 7
    over = (1 << 24) // wbig + 1
    over += 1 - over % 2                      # odd sum, odd weight: odd product sum > 2^24
    assert wbig * over > (1 << 24) and (wbig * over) % 2 == 1
    rng = np.random.default_rng(321)
    t0 = [limit] * 256
    t1 = [limit] * 255 + [limit + 1]
    t2 = [over] * 60 + [limit] * 20
    x = _rows_with_l1(t0 + t1 + t2, K, rng)
    M, N = x.shape[0], 136
    qa, sa = oracle.quantize_act(x)
    assert np.all(sa == 1.0)
    l1 = np.abs(qa.astype(np.int64)).sum(axis=1)
    assert l1[:256].max() == limit and l1[256:512].max() == limit + 1 and l1[512] == over
    lo, hi = (-127, 127) if bits == 8 else (-8, 7)
    qw = rng.integers(lo, hi + 1, size=(N, K)).astype(np.int8)
    qw[0] = wbig                              # sign-matched: partial sums climb monotonically
    qw[1] = -wbig
    qw[2] = lo
    qw_dev = qw if bits == 8 else oracle.pack_int4(qw)
    acc_ref = oracle.gemm_acc(qa, qw, 0)
    assert acc_ref[0, 0, 0] == wbig * limit and acc_ref[512, 0, 0] == wbig * over
    acc = run_acc(cider, qa, qw_dev, 0, bits)
    assert_bits_equal(acc, acc_ref, f"bound acc bits={bits}")
    sw = (rng.random((N, 1)) * 1e-4 + 1e-5).astype(np.float32)
    y = run_linear(cider, x, qw_dev, sw, 0, bits)
    assert_bits_equal(y, oracle.linear(x, qw, sw, 0, threads=8), f"bound y bits={bits}")


def test_full_size_shared_activation_projection_set(cider):
    """The Qwen3-2B-shaped Q / K / V projections at prefill M = 1334: one
    activation quantization (cider_quantize_act) shared by the three
    projections through cider_w8a8_linear_prequant, per channel; sampled rows
    bit for bit against the oracle."""
    M, hidden = 1334, 2048
    x = inputs.activations(M, hidden, seed=0)
    qa, sa = cider.cider_quantize_act(to_dev(x))
    rng = np.random.default_rng(1334)
    rows = sorted(set([0, M - 1, M // 2] + list(rng.integers(0, M, 6))))
    for i, name in enumerate(("q", "k", "v")):
        N, K = inputs.QWEN3_2B[name]
        qw, sw = oracle.quantize_weight_int8(inputs.weights(N, K, seed=1 + 2 * i), 0)
        y = to_host(cider.cider_w8a8_linear_prequant(qa, sa, to_dev(qw), to_dev(sw), 0))
        assert y.shape == (M, N)
        yref = oracle.linear(x, qw, sw, 0, rows=rows, threads=8)
        assert_bits_equal(y[rows], yref, f"Qwen3-2B {name} projection rows")


def test_trim_scratch_pool_keeps_results(cider):
    """Trimming the pooled scratch after a large call releases it and the
    next calls allocate again and compute the same bits."""
    M, N, K = 2048, 1024, 4096
    x = to_dev(inputs.activations(M, K, seed=5))
    qw_dev, _, sw = make_weights(N, K, 0, 8, seed=6)
    qw_d, sw_d = to_dev(qw_dev), to_dev(sw)
    y0 = cider.cider_w8a8_linear(x, qw_d, sw_d, 0)
    cider.cider_trim_scratch_pool(0)
    y1 = cider.cider_w8a8_linear(x, qw_d, sw_d, 0)
    cider.cider_trim_scratch_pool(1 << 20)
    assert_bits_equal(to_host(y1), to_host(y0), "after trimming the pool")
    assert cider.cider_check_device_error() == 0


@pytest.mark.parametrize("gs,bits", [(0, 8), (0, 4), (128, 8), (64, 4)])
@pytest.mark.parametrize("y_dtype", ["f16", "bf16"])
def test_output_views_at_16_byte_offsets(cider, gs, bits, y_dtype):
    """y written into a view that starts 16 bytes (not 32) into its buffer,
    with N % 16 == 0: the per-channel epilogue then takes its 16-byte-store
    path and the per-group kernel's TMA stores start at a 16-byte boundary.
    The outputs equal the oracle's (per channel bit for bit, per group within
    the tolerance); the bytes around the view stay untouched."""
    M, N, K = 300, 1024, 1024
    x = inputs.activations(M, K, seed=21)
    qw_dev, qv, sw = make_weights(N, K, gs, bits, seed=22)
    dt = torch.float16 if y_dtype == "f16" else torch.bfloat16
    big = torch.full((M * N + 16,), 7.0, dtype=dt, device="cuda")
    y = big[8:8 + M * N].view(M, N)
    assert y.data_ptr() % 32 == 16
    fn = cider.cider_w8a8_linear_ex if bits == 8 else cider.cider_w4a8_linear_ex
    fn(to_dev(x), to_dev(qw_dev), to_dev(sw), gs, y_dtype=dt, out=y)
    ref = oracle.linear(x, qv, sw, gs, out_bf16=(y_dtype == "bf16"))
    got = y.cpu().view(torch.int16).numpy().view(np.uint16) if y_dtype == "bf16" else to_host(y)
    want = ref.view(np.uint16) if y_dtype == "bf16" else ref
    if gs == 0:
        assert_bits_equal(got, want, f"16-byte offset view, bits {bits}, {y_dtype}")
    elif y_dtype == "f16":
        assert_fp16_close(got, want, f"16-byte offset view, bits {bits} gs {gs}")
    else:
        from tests.test_gpu_bf16 import assert_bf16_close
        assert_bf16_close(got, want, f"16-byte offset view, bits {bits} gs {gs}")
    edge = big.cpu().float().numpy()
    assert np.all(edge[:8] == 7.0) and np.all(edge[8 + M * N:] == 7.0)
