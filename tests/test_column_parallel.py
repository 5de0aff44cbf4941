"""Output-channel split of one linear across ranks (Cider pages, "How It
Works" and SplitLinear's 64-aligned output-channel split).

Host logic on the CPU: the partition covers every output column once with
64-aligned boundaries, and the all-gather of the ranks' parts reproduces the
whole layer bit for bit (world sizes 2 and 3, gloo, each rank computing its
slice with the oracle).  On the GPU: every rank's slice through the library
kernels, concatenated, equals the one-call result bit for bit (the ranks are
run one after another on one GPU; their gather is the CPU-tested part)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from w4a8_quantized_linear_gb300 import column_parallel as cp
from w4a8_quantized_linear_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("N", [8, 64, 136, 264, 1000, 2048, 10240, 12296])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_column_slices_cover_every_column_once(N, world):
    sl = cp.column_slices(N, world)
    assert len(sl) == world and sl[0][0] == 0 and sl[-1][1] == N
    for (a, b), (c, _) in zip(sl, sl[1:]):
        assert a <= b == c                      # contiguous, in order, no overlap
    for a, b in sl[1:]:
        assert a % cp.SPLIT_ALIGN == 0          # every share starts 64-aligned
    cover = np.zeros(N, np.int64)
    for a, b in sl:
        cover[a:b] += 1
    assert np.all(cover == 1)
    if N >= cp.SPLIT_ALIGN * world:
        sizes = [b - a for a, b in sl]
        assert max(sizes) - min(sizes) <= 2 * cp.SPLIT_ALIGN


def test_two_device_split_matches_the_pages_rule():
    """With two ranks the first share is floor(N / 2) rounded down to a
    multiple of 64 and the second takes the rest, as SplitLinear does with a
    fraction of one half."""
    for N in (2048, 6144, 1000, 136):
        (a0, b0), (a1, b1) = cp.column_slices(N, 2)
        assert (a0, b0) == (0, (N // 2) // 64 * 64) and (a1, b1) == (b0, N)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, cases, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from w4a8_quantized_linear_gb300 import column_parallel as cpar
    from w4a8_quantized_linear_gb300 import inputs as inp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = []
        for M, N, K, gs, bits in cases:
            x, W = inp.layer(M, N, K, base_seed=7, index=0)        # replicated on every rank
            if bits == 8:
                qv, sw = oracle.quantize_weight_int8(W, gs)
            else:
                qv, sw = oracle.quantize_weight_int4(W, gs)
            sl = cpar.column_slices(N, world)
            n0, n1 = sl[rank]
            y_local = oracle.linear(x, qv[n0:n1], sw[n0:n1], gs)   # this rank's output channels
            y = cpar.gather_columns(torch.from_numpy(np.ascontiguousarray(y_local)), sl)
            whole = oracle.linear(x, qv, sw, gs)
            res.append(bool(np.array_equal(y.numpy().view(np.uint16), whole.view(np.uint16))))
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_gather_the_whole_layer_bit_for_bit(world):
    cases = [(5, 264, 256, 0, 8), (7, 1000, 128, 64, 8), (3, 136, 256, 128, 4), (4, 64, 128, 0, 8)]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), cases, out), nprocs=world, join=True)
        res = dict(out)
    assert all(all(r) for r in res.values()), res


@pytest.mark.gpu
@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("M,N,K,gs,bits", [(300, 2048, 1024, 0, 8), (17, 1000, 512, 128, 8),
                                           (4, 6144, 2048, 0, 8), (260, 1032, 1024, 128, 4)])
def test_rank_slices_through_the_kernels_concatenate_to_the_whole_layer(world, M, N, K, gs, bits):
    from tests.parity_util import assert_bits_equal, require_gpu
    cider = require_gpu()
    x, W = inputs.layer(M, N, K, base_seed=11, index=0)
    xd = torch.from_numpy(x).cuda()
    Wd = torch.from_numpy(W).cuda()
    if bits == 8:
        qw, sw = cider.cider_quantize_weight_int8(Wd, gs)
        fn = cider.cider_w8a8_linear
    else:
        qw, sw = cider.cider_quantize_weight_int4(Wd, gs)
        fn = cider.cider_w4a8_linear
    whole = fn(xd, qw, sw, gs)
    parts = []
    for rank in range(world):
        q_r, s_r = cp.shard_weights(qw, sw, rank, world)
        parts.append(fn(xd, q_r, s_r, gs) if q_r.shape[0] else
                     torch.empty((M, 0), dtype=torch.float16, device="cuda"))
    y = torch.cat(parts, dim=1)
    assert_bits_equal(y.cpu().numpy(), whole.cpu().numpy(), f"{world} ranks M={M} N={N}")
