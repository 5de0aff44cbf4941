"""Shared-memory bounds of the small-M (weight-streaming) path, checked on the
host over a sweep of shapes: the launch sizes come from the library's own
host code (cider_debug_small_m_launch), no GPU is involved.

The tensor-core form (4..16 tokens) copies each token row's codes of its K
slice into shared memory with one bulk copy of min(staged codes, K - first
code) bytes, into rows padded to a pitch of 64 mod 128 bytes (so that the two
token rows a quarter-warp reads fall in different banks).  These tests check
that every such copy is a whole number of 16-byte units, fits its row, that
a slice's copies stay below the transaction count an mbarrier can track, that
the slices cover K exactly once, and that the ring and the staged rows fit the
kernel's shared memory."""
import pytest

import w4a8_quantized_linear_gb300 as cider

MBAR_TX_LIMIT = 1 << 20      # an mbarrier's pending transaction count is below 2^20 bytes
RING_MIN, RING_MAX = 4, 12

K_VALUES = list(range(32, 4097, 32)) + list(range(4096 + 512, 16385, 512))


def launch_or_none(M, N, K, bits, gs, split, sms):
    try:
        return cider.cider_debug_small_m_launch(M, N, K, bits, gs, split, sms)
    except Exception:
        return None        # the problem does not take the weight-streaming path


def check_sizes(M, N, K, bits, gs, split, sms, z):
    what = f"M={M} N={N} K={K} bits={bits} gs={gs} split={split} sms={sms}: {z}"
    mb, ks, tps, ka, pitch = z["mb"], z["slices"], z["tiles_per_slice"], z["staged_codes"], z["pitch"]
    assert mb >= M and mb & (mb - 1) == 0, what
    assert RING_MIN <= z["ring_slots"] <= RING_MAX, what
    assert z["smem"] <= z["smem_cap"], what
    if z["mma"]:
        assert mb >= 4 and pitch % 128 == 64 and pitch >= ka, what
    else:
        assert pitch == ka, what
    if ks == 1:
        assert ka == K, what
    else:
        assert split and ka == tps * z["codes_per_tile"] and ka < K, what
    covered = 0
    for s in range(ks):
        kbase = s * tps * z["codes_per_tile"]
        assert kbase < K, f"empty slice {s}: {what}"
        assert kbase % 16 == 0, what
        nbytes = min(ka, K - kbase)
        assert nbytes > 0 and nbytes % 32 == 0, what            # whole 16-byte units
        assert (mb - 1) * pitch + nbytes <= mb * pitch, what      # the last row's copy fits
        assert M * nbytes < MBAR_TX_LIMIT, what
        covered += nbytes
    assert covered == K, what


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16])
def test_small_m_launch_sizes_stay_in_bounds(M, bits):
    cases = 0
    for N in (8, 136, 2560, 10240):
        for K in K_VALUES:
            for gs in (0, 64, 128):
                if gs and K % gs:
                    continue
                for split in (False, True):
                    for sms in (152, 148):
                        z = launch_or_none(M, N, K, bits, gs, split, sms)
                        if z is None:
                            continue
                        check_sizes(M, N, K, bits, gs, split, sms, z)
                        cases += 1
    assert cases > 1000


def test_known_workloads():
    # 16 tokens, W4A8 per group, N 2560, K 10240: K in 5 slices of 4 tiles
    z = cider.cider_debug_small_m_launch(16, 2560, 10240, 4, 128, True, 152)
    assert (z["mma"], z["slices"], z["tiles_per_slice"], z["staged_codes"]) == (1, 5, 4, 2048)
    assert z["pitch"] == 2112 and z["ring_slots"] == 4
    # the same rows quantized inside the kernel: no split, the whole row staged
    z = cider.cider_debug_small_m_launch(16, 2560, 10240, 4, 128, False, 152)
    assert z["slices"] == 1 and z["staged_codes"] == 10240
    # one token: the dp4a form, unpadded rows, one ring slot per tile of a row block
    z = cider.cider_debug_small_m_launch(1, 10240, 2560, 8, 0, False, 152)
    assert (z["mma"], z["pitch"], z["ring_slots"]) == (0, 2560, 10)


def test_rejects_problems_off_the_path():
    for args in [(17, 256, 1024, 8, 0, False, 152), (16, 256, 16384, 8, 0, False, 152),
                 (4, 0, 1024, 8, 0, False, 152), (4, 256, 1024, 8, 0, False, 0)]:
        with pytest.raises(Exception):
            cider.cider_debug_small_m_launch(*args)
