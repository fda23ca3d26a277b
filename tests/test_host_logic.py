"""Host-side logic of the binding that needs no GPU."""
import numpy as np

from adaptive_gradient_summation_gb300 import segment_groups


def test_segment_groups_cover_every_segment_in_order():
    rs = np.random.default_rng(4)
    for trial in range(50):
        lengths = rs.integers(0, 5000, size=int(rs.integers(1, 60)))
        offs = np.concatenate([[0], np.cumsum(lengths)])
        bpp = int(rs.integers(1, 64))
        chunk = int(rs.integers(1, 200_000))
        groups = segment_groups(offs, bpp, chunk)
        flat = [s for a, b in groups for s in range(a, b)]
        assert flat == list(range(len(lengths)))
        for a, b in groups[:-1]:
            size = (offs[b] - offs[a]) * bpp
            assert size >= chunk                       # closed only once full
            assert (offs[b - 1] - offs[a]) * bpp < chunk  # ... and not later than that


def test_segment_groups_long_segment_alone():
    offs = np.array([0, 10, 20, 10_020, 10_030])
    assert segment_groups(offs, 2, 1000) == [(0, 3), (3, 4)]
    assert segment_groups(offs, 2, 10) == [(0, 1), (1, 2), (2, 3), (3, 4)]
    assert segment_groups(np.array([0, 5]), 4, 1 << 30) == [(0, 1)]
