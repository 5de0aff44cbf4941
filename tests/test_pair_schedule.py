"""The per-channel GEMM's work split between CTA pairs (host arithmetic of the
library, no GPU): whole 256 x 256 tiles for whole rounds, then, when cheaper,
each remaining tile cut along K into equal pieces on several pairs that
exchange partial sums.  Checked on many shapes and pair counts:

* every (tile, 128-K block) is computed exactly once;
* every weight row of every tile is dequantized and stored by exactly one
  unit: a whole tile by its unit, a cut tile by the piece whose share of the
  tile's weight rows holds it (the shares of a tile's pieces partition it);
* a pair takes at most one piece, after all its whole tiles, and the pieces
  of a tile run on distinct launched pairs (they wait for each other);
* the cut is only used when it leaves fewer blocks per pair than a last
  partial round of whole tiles would.
"""
import itertools

import pytest

from w4a8_quantized_linear_gb300 import cider_debug_pair_schedule, library

WHOLE, PIECE = 0, 1


@pytest.fixture(scope="module", autouse=True)
def lib():
    try:
        library()
    except Exception as e:  # the library is built by __graft_entry__.build()
        pytest.skip(f"libcider.so not built: {e}")


def check_schedule(M, N, K, pairs):
    info, units = cider_debug_pair_schedule(M, N, K, pairs)
    tiles = ((M + 255) // 256) * ((N + 255) // 256)
    nkb = (K + 127) // 128
    assert info["tiles"] == tiles and info["blocks_per_tile"] == nkb
    assert 1 <= info["pairs"] <= pairs

    covered = {}
    stored = {}
    pieces_of = {}
    by_pair = {}
    for (p, t, kb0, kb1, kind, r0, r1) in units:
        assert 0 <= p < info["pairs"] and 0 <= t < tiles
        assert 0 <= kb0 < kb1 <= nkb and 0 <= r0 <= r1 <= 256
        for kb in range(kb0, kb1):
            assert (t, kb) not in covered, f"block {(t, kb)} computed twice"
            covered[(t, kb)] = p
        for r in range(r0, r1):
            assert (t, r) not in stored, f"row {r} of tile {t} stored twice"
            stored[(t, r)] = p
        by_pair.setdefault(p, []).append((t, kb0, kb1, kind))
        if kind == WHOLE:
            assert (kb0, kb1, r0, r1) == (0, nkb, 0, 256)
        else:
            assert r0 % 8 == 0 and r1 % 8 == 0   # whole groups of eight outputs
            pieces_of.setdefault(t, []).append(p)
    assert len(covered) == tiles * nkb, "every block computed"
    assert len(stored) == tiles * 256, "every weight row of every tile stored"

    for t, ps in pieces_of.items():
        assert len(ps) == len(set(ps)) == info["pieces"] >= 2
    for p, us in by_pair.items():
        kinds = [u[3] for u in us]
        assert kinds.count(PIECE) <= 1 and (PIECE not in kinds or kinds[-1] == PIECE)
        for i, u in enumerate(us):
            if u[3] == WHOLE:
                assert u[0] == p + i * info["pairs"], "whole tiles dealt round-robin"

    if info["cut_tiles"]:
        s = info["pieces"]
        assert info["whole_tiles"] % pairs == 0 and info["cut_tiles"] == tiles % pairs
        assert info["cut_tiles"] * s <= pairs and s * 4 <= nkb
        assert s <= 16, "the pieces' slices of the partials must fit the pipeline stages"
        rounds = tiles // pairs
        assert rounds * nkb + -(-nkb // s) < (rounds + 1) * nkb
        lens = [u[2] - u[1] for us in by_pair.values() for u in us if u[3] == PIECE]
        assert max(lens) - min(lens) <= 1
    else:
        assert info["whole_tiles"] == tiles
    return info, units


SHAPES = [(128, 2560, 2560), (4096, 10240, 2560), (3455, 6144, 2048), (1024, 10240, 2560),
          (4096, 2560, 10240), (8192, 10240, 2560), (128, 10240, 2560), (1334, 2048, 2048),
          (700, 264, 2560), (700, 264, 10240), (257, 384, 4096), (40, 264, 6144), (17, 136, 128),
          (300, 200, 2048), (4096, 12288, 4096), (2393, 6144, 2048), (1, 8, 128),
          (256, 256, 10240)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("pairs", [76, 74, 7, 1])
def test_schedule_computes_and_stores_everything_once(M, N, K, pairs):
    check_schedule(M, N, K, pairs)


def test_schedule_exhaustive_small():
    cut = 0
    for M, N, K, pairs in itertools.product([1, 256, 257, 600], [256, 520, 1300],
                                            [128, 384, 1000, 4096], [1, 2, 3, 5, 9, 16]):
        info, _ = check_schedule(M, N, K, pairs)
        cut += info["cut_tiles"] > 0
    assert cut > 20


def test_long_k_shape_cuts_the_last_tiles_into_nine_pieces():
    """4096 x 2560 x 10240: 160 tiles of 80 blocks on 76 pairs, i.e. 2 whole
    rounds and 8 more tiles; those are cut into 9 pieces of 8-9 blocks on 72
    pairs instead of a third round of 80 blocks."""
    info, units = check_schedule(4096, 2560, 10240, 76)
    assert info == {"pairs": 76, "whole_tiles": 152, "cut_tiles": 8, "pieces": 9,
                    "blocks_per_tile": 80, "tiles": 160}
    pieces = [u for u in units if u[4] == PIECE]
    assert len(pieces) == 72 and {u[3] - u[2] for u in pieces} == {8, 9}


def test_short_k_keeps_the_last_partial_round_whole():
    """4096 x 10240 x 2560: a ninth round of 32 whole tiles (measured faster
    than halves on 64 pairs after eight full rounds)."""
    info, units = check_schedule(4096, 10240, 2560, 76)
    assert info["cut_tiles"] == 0 and info["whole_tiles"] == 640


def test_small_problem_is_cut_across_idle_pairs():
    info, units = check_schedule(128, 2560, 2560, 76)   # 10 tiles of 20 blocks
    assert (info["cut_tiles"], info["pieces"], info["pairs"]) == (10, 5, 50)


def test_no_cut_when_tiles_fill_the_rounds():
    info, units = check_schedule(4096, 256 * 19, 2560, 76)    # 16 x 19 = 304 = 4 x 76 tiles
    assert info["cut_tiles"] == 0 and all(u[4] == WHOLE for u in units)


def test_rejects_bad_arguments():
    from w4a8_quantized_linear_gb300 import CiderError
    with pytest.raises(CiderError):
        cider_debug_pair_schedule(0, 256, 256, 76)
    with pytest.raises(CiderError):
        cider_debug_pair_schedule(256, 256, 256, 0)


def test_small_m_path_cuts_k_only_for_long_rows_and_few_row_blocks():
    from w4a8_quantized_linear_gb300 import CiderError, cider_debug_small_m_slices as slices
    # many row blocks or short rows: one slice, as before
    assert slices(1, 10240, 2560, 8, 0, 152) == 1
    assert slices(16, 10240, 2560, 8, 0, 152) == 1
    assert slices(16, 200, 2048, 8, 0, 152) == 1
    # 160 row blocks of 40 (int8) or 20 (int4) weight tiles on 152 SMs: several slices
    assert slices(16, 2560, 10240, 8, 0, 152) > 1
    assert slices(16, 2560, 10240, 4, 128, 152) > 1
    assert slices(1, 4096, 12288, 8, 128, 152) > 1
    for M, N, K in [(1, 520, 12288), (2, 264, 8192), (5, 136, 6144), (16, 264, 8192)]:
        ks = slices(M, N, K, 8, 0, 152)
        assert 2 <= ks <= 16
    with pytest.raises(CiderError):
        slices(17, 256, 256, 8, 0, 152)
