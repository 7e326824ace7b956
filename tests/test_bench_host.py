"""Host-side arithmetic of bench.py (CPU only)."""
import bench


def test_spread_is_nearest_rank_p10_median_p90():
    ms = [5, 1, 3, 2, 4, 6, 7, 8, 9, 10]
    assert bench.spread(ms) == {"p10": 2, "median": 5.5, "p90": 9}
    assert bench.spread([2.0]) == {"p10": 2.0, "median": 2.0, "p90": 2.0}
    assert bench.spread([]) is None
    # order of the samples does not matter
    assert bench.spread(list(reversed(ms))) == bench.spread(ms)


def test_packed_layout_aligns_and_views_round_trip():
    """The end-to-end loop moves a step's tensors packed in one buffer: every
    start is 256-byte aligned (the kernels' tensor maps want 16), the views
    cover disjoint byte ranges, and values written through a view land in
    the bytes of that view only."""
    import torch
    specs = [((3, 5), torch.bfloat16), ((7,), torch.float32), ((2, 2, 2), torch.bfloat16), ((1,), torch.int32)]
    offs, n = bench._layout(specs)
    assert all(o % 256 == 0 for o in offs) and n % 256 == 0
    sizes = [15 * 2, 7 * 4, 8 * 2, 4]
    ends = [o + b for o, b in zip(offs, sizes)]
    assert all(e <= o2 for e, o2 in zip(ends, offs[1:])) and ends[-1] <= n
    buf = torch.zeros(n, dtype=torch.uint8)
    views = bench._views(buf, specs, offs)
    assert [tuple(v.shape) for v in views] == [s for s, _ in specs]
    assert [v.dtype for v in views] == [d for _, d in specs]
    for i, v in enumerate(views):
        v.fill_(i + 1)
    for i, (v, (o, b)) in enumerate(zip(views, zip(offs, sizes))):
        assert torch.equal(buf[o:o + b].view(v.dtype), torch.full((v.numel(),), i + 1, dtype=v.dtype))
    covered = torch.zeros(n, dtype=torch.bool)
    for o, b in zip(offs, sizes):
        covered[o:o + b] = True
    assert int(buf[~covered].sum()) == 0
