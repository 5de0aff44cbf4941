"""Output-channel (N) split of one quantized linear across ranks, one GPU each.

The Cider pages split a linear along its output channels between two
devices and concatenate the parts ("mininglamp-ai--cider/experimental",
section "How It Works"; "…/experimental/split_linear.py", class SplitLinear:
the first device's share of the output channels is rounded down to a
multiple of SPLIT_ALIGN = 64, the other device takes the rest).  Every
output column n depends only on weight row n and its scales, so a rank
holding rows [n0, n1) of q_w and s_w computes exactly y[:, n0:n1] of the
whole layer: the same bits as one GPU computing all of y.  Each rank
quantizes the (replicated) activations itself, which is deterministic, so no
collective is needed before the multiply; the parts are gathered along N
afterwards (an all-gather over torch.distributed: NCCL between GPUs).

Here the split generalises to P ranks: boundary r (0 < r < P) is
floor(floor(N r / P) / 64) * 64, so every rank's share starts at a multiple
of 64 and the last rank takes the remainder.

Every step of the multiply runs in the library's CUDA kernels
(``cider_w8a8_linear`` / ``cider_w4a8_linear`` on the rank's GPU); this module
only partitions, slices and gathers.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

SPLIT_ALIGN = 64


def column_slices(N: int, world: int, align: int = SPLIT_ALIGN) -> List[Tuple[int, int]]:
    """[(n0, n1)] per rank: contiguous output-channel ranges covering [0, N)
    once, each starting at a multiple of ``align`` (a rank's range may be
    empty when N < align * world)."""
    if N < 0 or world < 1 or align < 1:
        raise ValueError("need N >= 0, world >= 1, align >= 1")
    bounds = [0]
    for r in range(1, world):
        bounds.append(max(bounds[-1], (N * r // world) // align * align))
    bounds.append(N)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def shard_weights(qw: torch.Tensor, sw: torch.Tensor, rank: int, world: int,
                  align: int = SPLIT_ALIGN):
    """This rank's rows of the quantized weights [N, ...] and scales [N, G]
    (contiguous copies, ready for the library's row-major entry points)."""
    n0, n1 = column_slices(qw.shape[0], world, align)[rank]
    return qw[n0:n1].contiguous(), sw.reshape(qw.shape[0], -1)[n0:n1].contiguous()


def gather_columns(y_local: torch.Tensor, slices: Sequence[Tuple[int, int]],
                   group: Optional["torch.distributed.ProcessGroup"] = None) -> torch.Tensor:
    """All-gather every rank's y[:, n0:n1] into the whole y [M, N] on every
    rank.  The parts are padded to the widest share (all-gather wants equal
    sizes) and their bytes are moved, so the result holds exactly the bits
    each rank computed."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    if len(slices) != world:
        raise ValueError("one slice per rank")
    rank = dist.get_rank(group)
    M = y_local.shape[0]
    width = max(n1 - n0 for n0, n1 in slices)
    n0, n1 = slices[rank]
    if y_local.shape != (M, n1 - n0):
        raise ValueError(f"local part has shape {tuple(y_local.shape)}, expected {(M, n1 - n0)}")
    esz = y_local.element_size()
    raw = (y_local.contiguous().view(torch.uint8).reshape(M, (n1 - n0) * esz) if n1 > n0 else
           torch.empty((M, 0), dtype=torch.uint8, device=y_local.device))
    padded = torch.zeros((M, width * esz), dtype=torch.uint8, device=y_local.device)
    padded[:, :raw.shape[1]] = raw
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    y = torch.cat([p[:, :(b - a) * esz] for p, (a, b) in zip(parts, slices)], dim=1)
    return y.contiguous().view(y_local.dtype)


def linear_column_parallel(x: torch.Tensor, qw_local: torch.Tensor, sw_local: torch.Tensor,
                           N: int, group_size: int = 0, bits: int = 8,
                           group: Optional["torch.distributed.ProcessGroup"] = None,
                           align: int = SPLIT_ALIGN) -> torch.Tensor:
    """y fp16 [M, N] of the whole layer on every rank: this rank's output
    channels (``qw_local``, ``sw_local`` from :func:`shard_weights`) through the
    library on its GPU, then :func:`gather_columns`."""
    import torch.distributed as dist
    from . import cider_w4a8_linear, cider_w8a8_linear
    slices = column_slices(N, dist.get_world_size(group), align)
    n0, n1 = slices[dist.get_rank(group)]
    if qw_local.shape[0] != n1 - n0:
        raise ValueError("local weight rows do not match this rank's slice")
    fn = cider_w8a8_linear if bits == 8 else cider_w4a8_linear
    if n1 > n0:
        y_local = fn(x, qw_local, sw_local, group_size)
    else:
        y_local = torch.empty((x.shape[0], 0), dtype=torch.float16, device=x.device)
    return gather_columns(y_local, slices, group)
