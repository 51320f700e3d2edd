"""Host logic of the multi-fragment driver (no GPU): fragment planning against brute
force membership, and the packed amax layout."""
import numpy as np
import pytest

from mxfp8_master_weight_gb300 import api, driver
from mxfp8_master_weight_gb300 import workloads as wl


def _brute_plan(specs, bounds):
    owner = np.empty(sum(s.numel for s in specs), np.int64)
    for s in range(len(bounds) - 1):
        owner[bounds[s]:bounds[s + 1]] = s
    plan = [[] for _ in range(len(bounds) - 1)]
    off = 0
    for w, spec in enumerate(specs):
        seg = owner[off:off + spec.numel]
        for s in np.unique(seg):
            idx = np.flatnonzero(seg == s)
            plan[s].append((w, int(idx[0]), int(idx.size), off + int(idx[0]) - bounds[s]))
        off += spec.numel
    return plan


@pytest.mark.parametrize("bounds_fn", [
    lambda t: [0, t],
    lambda t: [0, 17, 17, t],
    lambda t: [0, 1, t // 3 + 5, t // 3 + 5, t - 1, t],
])
def test_plan_matches_brute_force(bounds_fn):
    specs = [driver.WeightSpec(64, 96, True), driver.WeightSpec(33, 65, False),
             driver.WeightSpec(32, 32, True)]
    total = sum(s.numel for s in specs)
    bounds = bounds_fn(total)
    plan = driver.plan_fragments(specs, bounds)
    brute = _brute_plan(specs, bounds)
    got = [[(c.weight, c.start, c.length, c.shard_offset) for c in cuts] for cuts in plan]
    assert got == brute
    # every element is covered exactly once
    assert sum(c.length for cuts in plan for c in cuts) == total


def test_plan_rejects_bad_bounds():
    specs = [driver.WeightSpec(32, 32, True)]
    with pytest.raises(ValueError):
        driver.plan_fragments(specs, [0, 10, 5, 1024])
    with pytest.raises(ValueError):
        driver.plan_fragments(specs, [0, 1000])


def test_cfg5_plan_shape():
    b = wl.cfg5_sharded_batch(seed=0, scale=8)
    specs = [driver.WeightSpec(w.rows, w.cols, w.colwise) for w in b.weights]
    plan = driver.plan_fragments(specs, b.bounds)
    assert len(plan) == 4 and plan[2] == []           # the empty shard
    assert b.bounds[1] % 32 != 0                       # boundary inside a 32-value block of W0
    assert plan[0][-1].weight == 0 and plan[1][0].weight == 0
    assert [c.weight for c in plan[0]] == [0]


def test_packed_layout():
    import torch
    specs = [driver.WeightSpec(64, 96, True), driver.WeightSpec(40, 70, False),
             driver.WeightSpec(32, 32, True)]
    lay = driver.PackedLayout(specs)
    spans = []
    for w, spec in enumerate(specs):
        o, shp = lay.rowwise[w]
        assert shp == (spec.rows, (spec.cols + 31) // 32) and o % 16 == 0
        spans.append((o, o + shp[0] * shp[1]))
        if spec.colwise:
            o, shp = lay.colwise[w]
            assert shp == ((spec.rows + 31) // 32, spec.cols) and o % 16 == 0
            spans.append((o, o + shp[0] * shp[1]))
        else:
            assert lay.colwise[w] is None
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans[:-1], spans[1:]))  # no overlap
    assert spans[-1][1] <= lay.total
    buf = torch.arange(lay.total, dtype=torch.float32)
    vr, vc = lay.views(buf, 1)
    assert vc is None and vr.shape == (40, 3) and vr.is_contiguous()


def _written_entries(rows, cols, colwise, start, length):
    """Linear grid indices the oracle's partial amax writes for a fragment: grids filled
    with a NaN sentinel, every written entry holds a finite maximum afterwards."""
    import oracle
    rng = np.random.default_rng(start * 31 + length)
    frag = (rng.standard_normal(length) * 0.02).astype(np.float32)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    ar = np.full((rr, rc), np.nan, np.float32)
    ac = np.full((cr, cc), np.nan, np.float32) if colwise else None
    oracle.partial_amax(frag, rows, cols, start, ar, ac)
    row = set(np.flatnonzero(~np.isnan(ar.reshape(-1))).tolist())
    col = set(np.flatnonzero(~np.isnan(ac.reshape(-1))).tolist()) if colwise else set()
    return row, col


def _expand(ranges):
    return {e for a, b in ranges for e in range(a, b)}


@pytest.mark.parametrize("rows,cols", [(70, 50), (64, 96), (33, 65), (96, 7)])
def test_fragment_block_ranges_are_the_written_entries(oracle_mod, rows, cols):
    """The ranges the driver gives the ranged reduction are exactly the entries the
    partial amax writes, for fragments of every shape: inside a row, across two rows of
    one band (the gap case), across bands, whole weights."""
    n = rows * cols
    rng = np.random.default_rng(rows * cols)
    cases = [(0, n), (0, 1), (n - 1, 1), (cols - 3, 5), (cols * 31 + 7, 2 * cols - 10),
             (cols * 30 + 40 % cols, cols + 3), (5, cols * 40)]
    cases += [(int(s), int(rng.integers(1, n - s + 1))) for s in rng.integers(0, n, 40)]
    for start, length in cases:
        if start + length > n or length <= 0:
            continue
        for colwise in (True, False):
            spec = driver.WeightSpec(rows, cols, colwise)
            row, col = driver.fragment_block_ranges(spec, start, length)
            w_row, w_col = _written_entries(rows, cols, colwise, start, length)
            assert _expand(row) == w_row, (rows, cols, start, length)
            assert _expand(col) == w_col, (rows, cols, start, length, colwise)
            assert all(a < b for a, b in row + col)


def test_slot_ranges_cover_each_grid_and_count_runs():
    """Every entry of every grid is held by at least one slot; entries of blocks cut by a
    shard boundary by exactly two; the run count matches a brute-force cut."""
    specs = [driver.WeightSpec(96, 64, True), driver.WeightSpec(64, 96, False),
             driver.WeightSpec(32, 128, True)]
    total = sum(s.numel for s in specs)
    bounds = [0, 1000, 1000, 96 * 64 + 17, total]
    plan = driver.plan_fragments(specs, bounds)
    layout = driver.PackedLayout(specs)
    ranges = layout.slot_ranges(plan)
    holders = {}
    for s, a, b in ranges:
        for e in range(a, b):
            holders.setdefault(e, set()).add(s)
    grids = [g for w in range(3) for g in (layout.rowwise[w], layout.colwise[w]) if g is not None]
    for off, (nr, nc) in grids:
        for e in range(off, off + nr * nc):
            assert 1 <= len(holders.get(e, ())) <= 2
    # brute-force runs: consecutive grid entries with the same holder set
    want = []
    for off, (nr, nc) in grids:
        prev = None
        for e in range(off, off + nr * nc):
            h = frozenset(holders[e])
            if h != prev:
                want.append([off, e - off, e - off + 1])
            else:
                want[-1][2] += 1
            prev = h
    assert [list(r) for r in driver.reduce_runs(layout, ranges)] == want
    assert len(driver.reduce_runs(layout, None)) == len(grids)
    # pieces: each run's entries from the first multiple of 4 to the last in one piece,
    # each ragged end in its own
    pieces = 0
    for _, lo, hi in want:
        quads = [e for e in range(lo, hi) if e % 4 == 0 and e + 4 <= hi]
        pieces += 1 if not quads else 1 + (lo < quads[0]) + (quads[-1] + 4 < hi)
    assert driver.reduce_pieces(layout, ranges) == pieces


def test_launch_count_groups_by_dtype_and_output_alignment():
    """Aligned and realigning fragments of one dtype share the amax and cast launches; a
    cast launch is split only by dtype and by whether the outputs allow word stores
    (full-size outputs: their own address), at most 64 jobs per launch."""
    import torch
    specs = [driver.WeightSpec(64, 64, True), driver.WeightSpec(32, 128, False)]
    master = torch.zeros(64 * 64 + 32 * 128 + 8)
    outs = [torch.zeros(64 * 64 + 16, dtype=torch.uint8), torch.zeros(32 * 128 + 16, dtype=torch.uint8)]

    def jobs(frag_shift, out_shift):
        amax, cast = [], []
        for w, (spec, start, n) in enumerate(((specs[0], 3, 1000), (specs[1], 0, 512))):
            frag = master[frag_shift + start:frag_shift + start + n]
            q = outs[w][out_shift:out_shift + spec.numel]
            amax.append((frag, None, None, spec.rows, spec.cols, start))
            cast.append((frag, None, None, q, None, spec.rows, spec.cols, start))
        return amax, cast

    a0, c0 = jobs(0, 0)
    a1, c1 = jobs(1, 0)        # other fragment offsets: realigning, same launches
    a2, c2 = jobs(0, 1)        # outputs one byte off a word boundary
    base = driver._count_launches(a0, c0, 1, specs, fused_reduce=True)
    assert base == 1 + 1 + 1   # amax, reduction + scales, cast
    assert driver._count_launches(a0 + a1, c0 + c1, 1, specs, fused_reduce=True) == 3
    assert driver._count_launches(a0 + a2, c0 + c2, 1, specs, fused_reduce=True) == 4
    many_a, many_c = a0 * 33, c0 * 33  # 66 jobs: two launches per phase (64 per launch)
    assert driver._count_launches(many_a, many_c, 1, specs, fused_reduce=True) == 2 + 1 + 2
    bf = [(f.to(torch.bfloat16),) + j[1:] for f, j in ((j[0], j) for j in a0)]
    bfc = [(f.to(torch.bfloat16),) + j[1:] for f, j in ((j[0], j) for j in c0)]
    assert driver._count_launches(a0 + bf, c0 + bfc, 1, specs, fused_reduce=True) == 2 + 1 + 2
