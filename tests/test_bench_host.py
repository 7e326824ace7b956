"""Host-side arithmetic of bench.py (CPU only)."""
import bench


def test_spread_is_nearest_rank_p10_median_p90():
    ms = [5, 1, 3, 2, 4, 6, 7, 8, 9, 10]
    assert bench.spread(ms) == {"p10": 2, "median": 5.5, "p90": 9}
    assert bench.spread([2.0]) == {"p10": 2.0, "median": 2.0, "p90": 2.0}
    assert bench.spread([]) is None
    # order of the samples does not matter
    assert bench.spread(list(reversed(ms))) == bench.spread(ms)
