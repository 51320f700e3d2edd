"""Host logic of the multi-fragment driver (no GPU): fragment planning against brute
force membership, and the packed amax layout."""
import numpy as np
import pytest

from mxfp8_master_weight_gb300 import driver
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
