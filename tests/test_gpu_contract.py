"""API contract on the GPU: omission by empty handles, ignored columnwise scales,
required-argument errors, the caller's stream, and that the product path is the
in-tree CUDA library (no fallback)."""
import numpy as np
import pytest
import torch

from mxfp8_master_weight_gb300 import _capi, api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, gpu_fragment, oracle_fragment, to_device, to_host

pytestmark = pytest.mark.gpu


def _setup(rows=128, cols=256, seed=0):
    rng = np.random.default_rng(seed)
    x = to_device(wl.normal_f32(rng, rows * cols))
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    ar = torch.zeros((rr, rc), device="cuda")
    ac = torch.zeros((cr, cc), device="cuda")
    api.mxfp8_partial_amax(x, ar, ac, rows, cols, 0)
    sr = torch.empty((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.empty((cr, cc), dtype=torch.uint8, device="cuda")
    api.mxfp8_update_scales(ar, ac, sr, sc, rows, cols)
    return x, sr, sc, rows, cols


def test_unused_colwise_scales_are_ignored():
    x, sr, sc, rows, cols = _setup()
    q1 = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    q2 = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(x, sr, None, q1, None, rows, cols, 0)
    api.mxfp8_partial_cast(x, sr, sc, q2, None, rows, cols, 0)           # present but unused
    garbage = torch.zeros(3, dtype=torch.float32, device="cuda")
    q3 = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(x, sr, garbage, q3, None, rows, cols, 0)      # not even validated
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(q1, q3)


def test_zero_element_views_are_omitted_directions():
    x, sr, sc, rows, cols = _setup()
    q_ref = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(x, sr, None, q_ref, None, rows, cols, 0)
    backing = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    empty_view = backing[5:5]  # zero elements, non-null storage pointer
    q = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(x, sr, sc[:0], q, empty_view, rows, cols, 0)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref) and torch.all(backing == 0)


def test_missing_required_rejected():
    x, sr, sc, rows, cols = _setup()
    q = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_partial_cast(x, sr, None, q, q.clone(), rows, cols, 0)
    assert e.value.status == 4
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_partial_cast(x, None, sc, q, None, rows, cols, 0)
    assert e.value.status == 4
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_partial_amax(x, None, None, rows, cols, 0)
    assert e.value.status == 4
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_partial_cast(x.view(rows, cols).t(), sr, None, q, None, rows, cols, 0)
    assert e.value.status == 5


def test_runs_on_caller_stream():
    rows, cols = 1024, 1024
    rng = np.random.default_rng(3)
    xh = wl.normal_f32(rng, rows * cols)
    x = to_device(xh)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    s = torch.cuda.Stream()
    ar = torch.zeros((rr, rc), device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        api.mxfp8_partial_amax(x, ar, None, rows, cols, 0)
    s.synchronize()
    want = np.abs(xh.reshape(rows, rc, 32)).max(axis=2)
    assert np.array_equal(to_host(ar), want)


def test_library_is_the_in_tree_build():
    import os
    lib = _capi.load()
    assert os.path.dirname(os.path.abspath(_capi.LIB_PATH)).endswith("mxfp8_master_weight_gb300")
    maps = open("/proc/self/maps").read()
    assert "libmxfp8_gb300.so" in maps
    assert lib.mxfp8_version() >= 100


# NaN patterns a block may hold: signalling, quiet, with payload, negative
NAN_F32_PATTERNS = (0x7F800001, 0x7FBFFFFF, 0x7FC00000, 0x7FFFFFFF, 0xFFC00000, 0xFF800001)


def test_special_values_follow_stated_conventions():
    """NaN / Inf in a block: amax NaN or Inf -> scale 0xFF -> block bytes 0x7F."""
    x = np.zeros(64, np.float32)
    x[3] = np.nan
    x[40] = np.inf
    got = gpu_fragment(x, 1, 64, 0, False)
    assert np.isnan(got[0][0, 0]) and np.isinf(got[0][0, 1])
    assert got[2][0, 0] == 0xFF and got[2][0, 1] == 0xFF
    assert np.all(got[4] == 0x7F)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nan_amax_bits_match_the_oracle(dtype):
    """Every NaN pattern in a block gives the same amax bits as the oracle (the canonical
    quiet NaN), in both directions, through the split and the one-pass paths."""
    rows, cols = 64, 256
    rng = np.random.default_rng(31)
    x = wl.normal_f32(rng, rows * cols)
    bits = x.view(np.uint32)
    for k, pat in enumerate(NAN_F32_PATTERNS):  # one NaN per row block, spread over rows
        bits[(7 * k) * cols + 32 * k + 3] = pat
    if dtype == "bf16":
        hb = (bits >> 16).astype(np.uint16)
        for k, pat in enumerate(NAN_F32_PATTERNS):
            i = (7 * k) * cols + 32 * k + 3
            hb[i] = (pat >> 16) | (0 if (pat >> 16) & 0x7F else 0x40)  # stays a NaN
        x = hb
    got = gpu_fragment(x, rows, cols, 0, True)
    want = oracle_fragment(x, rows, cols, 0, True)
    assert_bitwise(got, want, f"{dtype} NaN patterns")
    # the one-pass path writes the same amaxes
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    xd = to_device(x)
    ar = torch.zeros((rr, rc), dtype=dt, device="cuda")
    ac = torch.zeros((cr, cc), dtype=dt, device="cuda")
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda")
    qr = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_quantize_whole_blocks(xd, ar, ac, sr, sc, qr, qc, rows, cols, 0)
    torch.cuda.synchronize()
    assert_bitwise([to_host(t) for t in (ar, ac, sr, sc, qr, qc)], want, f"{dtype} one-pass")


def test_kernels_see_the_writes_of_the_kernel_before_them():
    """Every library kernel is launched as a programmatic dependent of the kernel before
    it in the stream and waits for it before touching memory: a torch kernel that
    rewrites the master weight right before the amax, our own amax -> scales -> cast
    chain, and a torch kernel that consumes the cast output right after it all see
    each other's writes, step after step, with no synchronisation in between."""
    rows, cols = 1024, 2048
    rng = np.random.default_rng(9)
    x = to_device(wl.normal_f32(rng, rows * cols))
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    ar = torch.zeros((rr, rc), device="cuda")
    ac = torch.zeros((cr, cc), device="cuda")
    sr = torch.empty((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.empty((cr, cc), dtype=torch.uint8, device="cuda")
    qr = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.empty(rows * cols, dtype=torch.uint8, device="cuda")
    first = None
    seen = []
    for step in range(6):
        x.mul_(2.0)                                   # producer: a torch kernel
        api.mxfp8_partial_amax(x, ar, ac, rows, cols, 0)
        api.mxfp8_update_scales(ar, ac, sr, sc, rows, cols)
        api.mxfp8_partial_cast(x, sr, sc, qr, qc, rows, cols, 0)
        seen.append((sr.to(torch.int32).sum(), qr.to(torch.int64).sum()))  # consumer kernels
        if first is None:
            first = (ar.clone(), sr.clone(), qr.clone(), qc.clone())
    torch.cuda.synchronize()
    # doubling x doubles every amax and adds one to every scale byte; the data are unchanged
    assert torch.equal(ar, first[0] * 32.0)
    assert torch.equal(sr.to(torch.int32), first[1].to(torch.int32) + 5)
    assert torch.equal(qr, first[2]) and torch.equal(qc, first[3])
    sums = [(int(a), int(b)) for a, b in seen]
    assert all(sums[k + 1][0] - sums[k][0] == rr * rc for k in range(5))
    assert len({b for _, b in sums}) == 1
