"""The allocation-free sharded update, called through the C ABI.

Some callers cannot allocate device memory when they need a master-weight update (a
memory-pool allocator doing its own maintenance, a framework that reserved all device
memory up front, code where cudaMalloc would synchronise the device).  For them the
library runs the update with its own fixed 64 MiB device array as working memory.
These checks compare that entry point with the ordinary entry points and with the CPU
oracle's whole-weight cast on two calls in a row (the second call must clear what the
first one left in the shared array), check that an oversized request is refused, and
that a call refused by validation writes nothing.  The file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import _capi, api
from mxfp8_master_weight_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _reference(frags, starts, rows, cols, colwise, dtype):
    """The same update through the ordinary entry points (driver-style own buffers)."""
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    slots_r = torch.zeros((len(frags), rr, rc), dtype=dtype, device="cuda")
    slots_c = torch.zeros((len(frags), cr, cc), dtype=dtype, device="cuda") if colwise else None
    for f, (x, s) in enumerate(zip(frags, starts)):
        api.mxfp8_partial_amax(x, slots_r[f], slots_c[f] if colwise else None, rows, cols, s)
    red_r = torch.empty((rr, rc), dtype=dtype, device="cuda")
    api.mxfp8_amax_max_reduce(slots_r.view(len(frags), -1), red_r)
    red_c = None
    if colwise:
        red_c = torch.empty((cr, cc), dtype=dtype, device="cuda")
        api.mxfp8_amax_max_reduce(slots_c.view(len(frags), -1), red_c)
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda") if colwise else None
    api.mxfp8_update_scales(red_r, red_c, sr, sc, rows, cols)
    qr = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda") if colwise else None
    for x, s in zip(frags, starts):
        api.mxfp8_partial_cast(x, sr, sc, qr, qc, rows, cols, s)
    return sr, sc, qr, qc


def _no_alloc(frags, starts, rows, cols, colwise):
    """Direct C ABI call of mxfp8_sharded_update_noalloc."""
    lib = _capi.load()
    fn = lib.mxfp8_sharded_update_noalloc
    T = ctypes.POINTER(_capi.Tensor)
    fn.argtypes = [T, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32, T, T, T, T,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    sr = torch.full((rr, rc), 0x55, dtype=torch.uint8, device="cuda")
    sc = torch.full((cr, cc), 0x55, dtype=torch.uint8, device="cuda") if colwise else None
    qr = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda") if colwise else None
    frs = (_capi.Tensor * len(frags))(*[api.handle(x, "fragment") for x in frags])
    st = (ctypes.c_int64 * len(frags))(*starts)
    hs = [api.handle(t, n) for t, n in ((sr, "sr"), (sc, "sc"), (qr, "qr"), (qc, "qc"))]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(frs, st, len(frags), *[ctypes.byref(h) for h in hs], rows, cols, stream)
    assert rc == 0, lib.mxfp8_last_error()
    return sr, sc, qr, qc


@pytest.mark.parametrize("dtype,rows,cols,colwise,cuts", [
    (torch.float32, 1024, 1024, True, [0, 37 * 1024 + 17, 600 * 1024 + 3, 1024 * 1024]),
    (torch.bfloat16, 256, 2048, False, [0, 5, 5, 300000, 256 * 2048]),
])
def test_no_alloc_matches_entry_points_twice(dtype, rows, cols, colwise, cuts):
    n = rows * cols
    for call in range(2):  # two calls in a row: the shared working memory is reused
        rng = np.random.default_rng(100 + call)
        x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
        full = torch.from_numpy(x).cuda().to(dtype)
        # every fragment in its own buffer, as a rank's shard would be
        frags = [full[a:b].clone() for a, b in zip(cuts[:-1], cuts[1:])]
        starts = cuts[:-1]
        got = _no_alloc(frags, starts, rows, cols, colwise)
        want = _reference(frags, starts, rows, cols, colwise, dtype)
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert (g is None and w is None) or torch.equal(g, w), f"call {call}"
        # and against the oracle's cast of the whole weight (the union of the fragments)
        host = full.cpu()
        hx = (host.view(torch.int16).numpy().view(np.uint16) if dtype == torch.bfloat16
              else host.numpy())
        o = oracle.full_cast(hx, rows, cols, colwise)
        names = ("scale_rowwise", "scale_colwise", "data_rowwise", "data_colwise")
        for name, g, w in zip(names, got, (o[2], o[3], o[4], o[5])):
            if w is None:
                assert g is None
                continue
            assert np.array_equal(g.cpu().numpy(), w), f"call {call} {name} differs from the oracle"


def test_no_alloc_refuses_requests_beyond_its_array():
    lib = _capi.load()
    rows, cols = 16384, 6144  # 25 MB per bidirectional FP32 amax slot: 3 slots do not fit
    x = torch.zeros(64, device="cuda")
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda")
    q = torch.zeros(64, dtype=torch.uint8, device="cuda")  # room for both tiny fragments
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_sharded_update_noalloc([x[:32], x[32:]], [0, 32], sr, sc, q, q, rows, cols)
    assert e.value.status == 2 and "static scratch" in str(e.value)
    assert lib.mxfp8_last_error().startswith(b"needs")


def test_no_alloc_refused_call_writes_nothing():
    """A call that fails validation (here: a columnwise output without columnwise
    scales, and overlapping fragments) returns its status before anything is launched:
    the caller's scale grids and outputs keep their sentinel bytes."""
    rows, cols = 256, 512
    x = torch.randn(rows * cols, device="cuda") * 0.02
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    sr = torch.full((rr, rc), 0x5A, dtype=torch.uint8, device="cuda")
    qr = torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device="cuda")
    qc = torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device="cuda")
    frags, starts = [x[:40000], x[40000:]], [0, 40000]
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_sharded_update_noalloc(frags, starts, sr, None, qr, qc, rows, cols)
    assert e.value.status == 4
    with pytest.raises(_capi.MXFP8Error) as e:
        api.mxfp8_sharded_update_noalloc([x[:40000], x[39999:]], [0, 39999], sr, None, qr, None,
                                         rows, cols)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert bool((sr == 0x5A).all()) and bool((qr == 0xA5).all()) and bool((qc == 0xA5).all())
