"""Batched entry points: many fragments of several weights (FP32 and BF16, row-only and
bidirectional, aligned and shifted fragment buffers, fragment-sized outputs) in one
call each, bit-identical to the oracle; a bad job rejects the whole call before any
launch."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import _capi, api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, to_device, to_host

pytestmark = pytest.mark.gpu


def _weights():
    rng = np.random.default_rng(31)
    specs = [(256, 1024, "f32", True), (96, 2048, "bf16", False), (33, 96, "f32", False),
             (128, 512, "bf16", True)]
    out = []
    for rows, cols, dt, col in specs:
        x = wl.normal_f32(rng, rows * cols) * np.float32(4.0) ** rng.integers(-6, 6, rows * cols).astype(np.float32)
        if dt == "bf16":
            x = wl.truncate_to_bf16_bits(x)
        out.append((rows, cols, x, col))
    return out


def _fragments(rows, cols, n_cuts, rng):
    n = rows * cols
    cuts = sorted(set(int(c) for c in rng.integers(1, n, n_cuts)))
    return list(zip([0] + cuts, cuts + [n]))


@pytest.mark.parametrize("n_cuts", [3, 40])
def test_batched_amax_scales_cast_match_oracle(n_cuts):
    """4 weights cut into n_cuts + 1 fragments each: 16 jobs per call, or 164 (more than one
    64-job launch and more than one 64-job host window per call)."""
    rng = np.random.default_rng(32 + n_cuts)
    amax_jobs, cast_jobs, checks = [], [], []
    keep = []
    for w, (rows, cols, x, col) in enumerate(_weights()):
        (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
        frags = _fragments(rows, cols, n_cuts, rng)
        dt = torch.float32 if x.dtype == np.float32 else torch.bfloat16
        slots_r = torch.zeros((len(frags), rr, rc), dtype=dt, device="cuda")
        slots_c = torch.zeros((len(frags), cr, cc), dtype=dt, device="cuda") if col else None
        qr = torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device="cuda")
        qc = torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device="cuda") if col else None
        devs = []
        for f, (a, b) in enumerate(frags):
            d = to_device(np.ascontiguousarray(x[a:b]), shift=(w + f) % 4)  # mixed alignments
            devs.append(d)
            amax_jobs.append((d, slots_r[f], slots_c[f] if col else None, rows, cols, a))
        checks.append((rows, cols, x, col, frags, devs, slots_r, slots_c, qr, qc))
        keep.append(devs)
    api.mxfp8_partial_amax_batched(amax_jobs)
    scale_jobs, reduced = [], []
    for rows, cols, x, col, frags, devs, slots_r, slots_c, qr, qc in checks:
        red_r = torch.empty(slots_r.shape[1:], dtype=slots_r.dtype, device="cuda")
        api.mxfp8_amax_max_reduce(slots_r.view(len(frags), -1), red_r)
        red_c = None
        if col:
            red_c = torch.empty(slots_c.shape[1:], dtype=slots_c.dtype, device="cuda")
            api.mxfp8_amax_max_reduce(slots_c.view(len(frags), -1), red_c)
        sr = torch.empty(red_r.shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(red_c.shape, dtype=torch.uint8, device="cuda") if col else None
        scale_jobs.append((red_r, red_c, sr, sc, rows, cols))
        reduced.append((red_r, red_c, sr, sc))
        for d, (a, b) in zip(devs, frags):
            cast_jobs.append((d, sr, sc, qr, qc, rows, cols, a))
    api.mxfp8_update_scales_batched(scale_jobs)
    api.mxfp8_partial_cast_batched(cast_jobs)
    torch.cuda.synchronize()
    for (rows, cols, x, col, frags, devs, slots_r, slots_c, qr, qc), (rr_, rc_, sr, sc) in zip(checks, reduced):
        want = oracle.full_cast(x, rows, cols, col)
        got = (to_host(rr_), None if rc_ is None else to_host(rc_), to_host(sr),
               None if sc is None else to_host(sc), to_host(qr), None if qc is None else to_host(qc))
        assert_bitwise(got, want, f"{rows}x{cols} colwise={col}")


def test_batched_equals_single_calls_with_fragment_outputs():
    rng = np.random.default_rng(33)
    rows, cols, x, col = _weights()[0]
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    sr = torch.randint(110, 130, (rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.randint(110, 130, (cr, cc), dtype=torch.uint8, device="cuda")
    jobs, singles = [], []
    for f, (a, b) in enumerate(_fragments(rows, cols, 5, rng)):
        d = to_device(np.ascontiguousarray(x[a:b]), shift=f % 4)
        q1 = [torch.zeros(b - a, dtype=torch.uint8, device="cuda") for _ in range(2)]
        q2 = [torch.zeros(b - a, dtype=torch.uint8, device="cuda") for _ in range(2)]
        jobs.append((d, sr, sc, q1[0], q1[1], rows, cols, a, 0))
        api.mxfp8_partial_cast(d, sr, sc, q2[0], q2[1], rows, cols, a, 0)
        singles.append((q1, q2))
    api.mxfp8_partial_cast_batched(jobs)
    torch.cuda.synchronize()
    for q1, q2 in singles:
        assert torch.equal(q1[0], q2[0]) and torch.equal(q1[1], q2[1])


def test_batched_rejects_a_bad_job_before_launching():
    rows, cols = 64, 64
    x = torch.ones(rows * cols, device="cuda")
    ar = [torch.full((rows, 2), 7.0, device="cuda") for _ in range(3)]
    bad = torch.full((rows, 1), 7.0, device="cuda")  # too few row blocks
    jobs = [(x, ar[0], None, rows, cols, 0), (x[:100], bad, None, rows, cols, 0),
            (x, ar[2], None, rows, cols, 0)]
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_partial_amax_batched(jobs)
    assert e.value.status == 2 and "job 1" in str(e.value)
    torch.cuda.synchronize()
    assert all(torch.all(a == 7.0) for a in ar)


def test_batched_empty_and_zero_jobs():
    api.mxfp8_partial_amax_batched([])
    api.mxfp8_partial_cast_batched([])
    rows, cols = 32, 64
    x = torch.ones(rows * cols, device="cuda")
    ar = torch.full((rows, 2), 7.0, device="cuda")
    api.mxfp8_partial_amax_batched([(x[:0], ar, None, rows, cols, 5), (x[:0], ar, None, rows, cols, 9)])
    torch.cuda.synchronize()
    assert torch.all(ar == 7.0)
