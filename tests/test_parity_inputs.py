"""Host-side checks of the input layouts that the GPU parity tests build
(no GPU needed)."""
import numpy as np

from tests.parity_util import exhaustive_rows, positive_fp16


def test_exhaustive_rows_cover_every_pair():
    """The layout above: every amax a gets every value |x| <= a of both signs,
    and every row's maximum is its a (checked on the host, small range)."""
    pos = positive_fp16()
    x = exhaustive_rows(pos, 1020, 1030)
    amax = np.abs(x.astype(np.float32)).max(axis=1)
    assert np.array_equal(amax, x[:, 0].astype(np.float32))
    for i in (1020, 1022, 1023, 1029):
        rows = x[x[:, 0] == pos[i]]
        got = set(rows[:, 1:].ravel().view(np.uint16).tolist())
        want = set(pos[:i + 1].view(np.uint16).tolist()) | set((-pos[:i + 1]).view(np.uint16).tolist())
        assert want <= got and got - want <= {0, 0x8000}
