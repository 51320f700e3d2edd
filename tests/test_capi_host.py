"""C ABI checks that need no GPU: the library builds, loads and exports every entry
point declared in include/*.h, and argument validation rejects bad calls with the
documented status before any CUDA work is attempted."""
import ctypes
import glob
import os
import re

import pytest

from mxfp8_master_weight_gb300 import _capi
from mxfp8_master_weight_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _capi.load()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^\s*(?:MXFP8_API\s+)?(?:const\s+)?\w+\s*\*?\s*((?:mxfp8|nvfp4)_\w+)\s*\(",
                                text, flags=re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = _declared_symbols()
    for n in ("mxfp8_partial_amax", "mxfp8_amax_max_reduce", "mxfp8_update_scales",
              "mxfp8_partial_cast", "mxfp8_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert lib.mxfp8_version() >= 100


def test_only_the_c_abi_is_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _capi.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    text_syms = [l.split()[-1] for l in out.stdout.splitlines() if " T " in l]
    assert set(text_syms) == set(_declared_symbols())


def T(ptr, dtype, *shape):
    sh = list(shape) + [0] * (2 - len(shape))
    return _capi.Tensor(ctypes.c_void_p(ptr), dtype, len(shape), (ctypes.c_int64 * 2)(*sh))


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


F32, BF16, U8 = _capi.DTYPE_F32, _capi.DTYPE_BF16, _capi.DTYPE_U8
P = 0x10000  # fake, never dereferenced: every call below fails validation first
E = _capi.empty_tensor


def amax(lib, inp, ar, ac, rows, cols, start):
    return lib.mxfp8_partial_amax(ctypes.byref(inp), ctypes.byref(ar), ctypes.byref(ac),
                                  rows, cols, start, None)


def cast(lib, inp, sr, sc, qr, qc, rows, cols, start, out_off):
    return lib.mxfp8_partial_cast(*[ctypes.byref(t) for t in (inp, sr, sc, qr, qc)],
                                  rows, cols, start, out_off, None)


def test_amax_validation(lib):
    inp = T(P, F32, 100)
    ar = T(P, F32, 64, 2)
    ac = T(P, F32, 2, 64)
    assert amax(lib, inp, ar, ac, 0, 64, 0) == 1                 # rows must be positive
    assert amax(lib, inp, ar, ac, 1, 2 ** 37 + 1, 0) == 1        # one row past the column limit
    assert b"2^37" in lib.mxfp8_last_error()
    assert amax(lib, inp, ar, ac, 2 ** 21, 2 ** 19 + 32, 0) == 1  # past 2^40 elements
    assert b"2^40" in lib.mxfp8_last_error()
    assert amax(lib, inp, ar, ac, 2 ** 62, 2 ** 3, 0) == 1       # rows*cols would overflow int64
    assert amax(lib, inp, ar, ac, 64, 64, -1) == 1               # negative start
    assert amax(lib, inp, ar, ac, 64, 64, 64 * 64 - 99) == 1     # fragment past the end
    assert b"exceeds" in lib.mxfp8_last_error()
    assert amax(lib, inp, E(), ac, 64, 64, 0) == 4               # rowwise amax required
    assert amax(lib, inp, T(P, F32, 64, 1), ac, 64, 64, 0) == 2  # too few row blocks
    assert amax(lib, inp, ar, T(P, F32, 2, 63), 64, 64, 0) == 2  # colwise shape[1] < cols
    assert amax(lib, inp, ar, T(P, F32, 1, 64), 64, 64, 0) == 2  # too few column bands
    assert amax(lib, inp, T(P, BF16, 64, 2), ac, 64, 64, 0) == 3  # amax dtype != input dtype
    assert amax(lib, inp, ar, T(P, BF16, 2, 64), 64, 64, 0) == 3
    assert amax(lib, T(P, U8, 100), ar, ac, 64, 64, 0) == 3      # input must be F32/BF16
    assert amax(lib, T(P + 2, F32, 100), ar, ac, 64, 64, 0) == 1  # misaligned element pointer
    assert amax(lib, T(P, F32, 100), T(P, F32, 2), ac, 64, 64, 0) == 2  # amax must be 2-D


def test_empty_fragment_is_a_noop(lib):
    # zero-length fragment: validated, nothing launched, status 0 (even without a GPU)
    assert amax(lib, E(), E(), E(), 64, 64, 17) == 0
    assert amax(lib, T(P, F32, 0), T(P, F32, 64, 2), E(), 64, 64, 64 * 64) == 0
    assert cast(lib, E(), E(), E(), E(), E(), 64, 64, 5, 5) == 0


def test_cast_validation(lib):
    inp = T(P, F32, 100)
    sr = T(P, U8, 64, 2)
    sc = T(P, U8, 2, 64)
    q = T(P, U8, 64 * 64)
    assert cast(lib, inp, E(), sc, q, q, 64, 64, 0, 0) == 4         # rowwise scales required
    assert cast(lib, inp, sr, sc, E(), q, 64, 64, 0, 0) == 4        # rowwise output required
    assert cast(lib, inp, sr, E(), q, q, 64, 64, 0, 0) == 4         # colwise output needs scales
    assert b"scale_inv_colwise" in lib.mxfp8_last_error()
    assert cast(lib, inp, sr, sc, T(P, U8, 99), E(), 64, 64, 0, 0) == 2  # output too small
    assert cast(lib, inp, sr, sc, q, q, 64, 64, 0, 64 * 64 - 99) == 2   # out_offset + len too big
    assert cast(lib, inp, sr, sc, q, q, 64, 64, 0, -1) == 1
    assert cast(lib, inp, T(P, F32, 64, 2), sc, q, q, 64, 64, 0, 0) == 3  # scales must be U8
    assert cast(lib, inp, sr, sc, T(P, F32, 4096), E(), 64, 64, 0, 0) == 3
    assert cast(lib, inp, sr, T(P, U8, 2, 10), q, q, 64, 64, 0, 0) == 2  # colwise scales too small


@pytest.mark.skipif(_has_gpu(), reason="would launch on fake pointers; the GPU contract tests cover it")
def test_cast_ignores_colwise_scales_without_colwise_output(lib):
    # a malformed colwise scale handle is not inspected when the colwise output is
    # absent: validation passes and the call reaches the device lookup, which fails
    # here because this host has no CUDA device
    inp = T(P, F32, 100)
    bad_sc = T(P, F32, 1, 1)
    rc = cast(lib, inp, T(P, U8, 64, 2), bad_sc, T(P, U8, 64 * 64), E(), 64, 64, 0, 0)
    assert rc == 6
    assert b"cuda" in lib.mxfp8_last_error().lower()


def test_scales_and_reduce_validation(lib):
    ar = T(P, F32, 64, 2)
    ac = T(P, F32, 2, 64)
    sr = T(P, U8, 64, 2)
    sc = T(P, U8, 2, 64)
    up = lib.mxfp8_update_scales
    assert up(ctypes.byref(ar), ctypes.byref(ac), ctypes.byref(sr), ctypes.byref(sc), 2 ** 40, 2, None) == 1
    assert up(ctypes.byref(ar), ctypes.byref(ac), ctypes.byref(sr), ctypes.byref(E()), 64, 64, None) == 4
    assert up(ctypes.byref(E()), ctypes.byref(ac), ctypes.byref(sr), ctypes.byref(sc), 64, 64, None) == 4
    assert up(ctypes.byref(ar), ctypes.byref(ac), ctypes.byref(T(P, U8, 64, 1)), ctypes.byref(sc), 64, 64, None) == 2
    assert up(ctypes.byref(ar), ctypes.byref(T(P, BF16, 2, 64)), ctypes.byref(sr), ctypes.byref(sc), 64, 64, None) == 3
    red = lib.mxfp8_amax_max_reduce
    slots = T(P, F32, 4, 100)
    assert red(ctypes.byref(slots), ctypes.byref(T(P + 4096, F32, 99)), None) == 2
    assert red(ctypes.byref(slots), ctypes.byref(T(P + 4096, BF16, 100)), None) == 3
    assert red(ctypes.byref(slots), ctypes.byref(E()), None) == 4
    assert red(ctypes.byref(slots), ctypes.byref(T(P + 400, F32, 100)), None) == 1  # overlap


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        saved = _capi._lib
        try:
            _capi._lib = None
            _capi.load(str(tmp_path / "nope.so"))
        finally:
            _capi._lib = saved


def fused(lib, inp, ar, ac, sr, sc, qr, qc, rows, cols, start, out_off):
    return lib.mxfp8_quantize_whole_blocks(*[ctypes.byref(t) for t in (inp, ar, ac, sr, sc, qr, qc)],
                                           rows, cols, start, out_off, None)


def test_fused_rejects_fragments_that_cut_blocks(lib):
    rows, cols = 64, 256
    sr, sc = T(P, U8, rows, 8), T(P, U8, 2, cols)
    q = T(P, U8, rows * cols)
    # row-only: the fragment must start and end on 1x32 block boundaries
    assert fused(lib, T(P, F32, 100), E(), E(), sr, E(), q, E(), rows, cols, 0, 0) == 1
    assert b"cuts a 1x32 block" in lib.mxfp8_last_error()
    assert fused(lib, T(P, F32, 64), E(), E(), sr, E(), q, E(), rows, cols, 17, 17) == 1
    # bidirectional: whole 32-row bands
    assert fused(lib, T(P, F32, 256), E(), E(), sr, sc, q, q, rows, cols, 256, 256) == 1
    assert b"cuts a 32x1 block" in lib.mxfp8_last_error()
    # missing columnwise scales for a columnwise output, wrong amax dtype
    assert fused(lib, T(P, F32, 32 * cols), E(), E(), sr, E(), q, q, rows, cols, 0, 0) == 4
    assert fused(lib, T(P, F32, 32 * cols), T(P, BF16, rows, 8), E(), sr, sc, q, q, rows, cols, 0, 0) == 3


def test_swizzle_size_and_validation(lib):
    assert lib.mxfp8_swizzled_scales_size(16384, 192, 0) == 16384 * 192
    assert lib.mxfp8_swizzled_scales_size(130, 6, 0) == 256 * 8
    assert lib.mxfp8_swizzled_scales_size(130, 6, 1) == 128 * 132
    sw = lib.mxfp8_swizzle_scales
    s = T(P, U8, 130, 6)
    assert sw(ctypes.byref(s), ctypes.byref(T(P + 8192, U8, 2047)), 130, 6, 0, None) == 2
    assert sw(ctypes.byref(s), ctypes.byref(T(P + 8192, U8, 2048)), 130, 6, 2, None) == 1
    assert sw(ctypes.byref(T(P, F32, 130, 6)), ctypes.byref(T(P + 8192, U8, 2048)), 130, 6, 0, None) == 3
    assert sw(ctypes.byref(s), ctypes.byref(E()), 130, 6, 0, None) == 4
    assert sw(ctypes.byref(T(P, U8, 129, 6)), ctypes.byref(T(P + 8192, U8, 2048)), 130, 6, 0, None) == 2


def test_code_digest_ignores_comments_only():
    from mxfp8_master_weight_gb300 import build
    a = "int f(int x) {  // doubles x\n  return 2 * x; /* fast */ }\n"
    b = "/* a header */\nint f(int x) {\n  return 2 * x;\n}  // changed comment\n"
    c = "int f(int x) { return 3 * x; }"
    assert build.code_text(a) == build.code_text(b)
    assert build.code_text(a) != build.code_text(c)
    assert len(build.source_digest()) == 64


def test_python_binding_has_every_entry_point():
    """The binding exposes a function of the same name for every C entry point."""
    from mxfp8_master_weight_gb300 import api
    missing = [n for n in _declared_symbols() if not callable(getattr(api, n, None))]
    assert not missing, missing
    assert api.mxfp8_version() >= 100 and isinstance(api.mxfp8_last_error(), str)


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "mxfp8_partial.h"

int main(void) {
  float dummy[64];
  mxfp8_tensor in = {dummy, MXFP8_DTYPE_F32, 1, {64, 0}};
  mxfp8_tensor ar = {dummy, MXFP8_DTYPE_F32, 2, {2, 1}};
  /* rows <= 0 is rejected during validation, before any device work */
  int rc = mxfp8_partial_amax(&in, &ar, NULL, -1, 32, 0, NULL);
  printf("version=%d status=%d error=%s\n", mxfp8_version(), rc, mxfp8_last_error());
  return rc == MXFP8_ERR_INVALID && strlen(mxfp8_last_error()) > 0 ? 0 : 1;
}
"""


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """A plain C11 client compiles against include/mxfp8_partial.h, links the library,
    and gets a validation status and message back without a GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(_capi.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(_capi.LIB_PATH),
                    "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "status=1" in out.stdout and "rows and cols must be positive" in out.stdout


def test_noalloc_refuses_bad_arguments_before_any_device_work(lib):
    """The allocation-free sharded update checks every argument on the host before it
    touches a device: overlapping fragments, a missing or too small output, columnwise
    output without columnwise scales -- all refused here, on a host without a GPU (a
    call that got as far as the device would fail with status 6 instead)."""
    fn = lib.mxfp8_sharded_update_noalloc
    TP = ctypes.POINTER(_capi.Tensor)
    fn.argtypes = [TP, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32, TP, TP, TP, TP,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    rows, cols = 64, 64
    sr, sc = T(P, U8, 64, 2), T(P, U8, 2, 64)
    q = T(P, U8, 64 * 64)

    def call(frags, starts, sr_, sc_, qr_, qc_):
        arr = (_capi.Tensor * len(frags))(*frags)
        st = (ctypes.c_int64 * len(starts))(*starts)
        return fn(arr, st, len(frags), *[ctypes.byref(t) for t in (sr_, sc_, qr_, qc_)],
                  rows, cols, None)

    two = [T(P, F32, 2048), T(P + 8192, F32, 2048)]
    assert call([T(P, F32, 2048), T(P + 8192, F32, 2049)], [0, 2047], sr, sc, q, q) == 1
    assert b"overlap" in lib.mxfp8_last_error()
    assert call([T(P, F32, 100), E(), T(P + 8192, F32, 10)], [200, 0, 250], sr, sc, q, q) == 1
    assert b"fragments 0 and 2 overlap" in lib.mxfp8_last_error()
    assert call(two, [0, 2048], sr, sc, E(), q) == 4                 # rowwise output required
    assert call(two, [0, 2048], sr, E(), q, q) == 4                  # colwise output needs scales
    assert b"scale_inv_colwise" in lib.mxfp8_last_error()
    assert call(two, [0, 2048], E(), sc, q, q) == 4                  # rowwise scales required
    assert call(two, [0, 2048], sr, sc, T(P, U8, 100), q) == 2       # output too small
    assert call(two, [0, 3000], sr, sc, q, q) == 1                   # fragment past the end
    assert call([T(P, F32, 2048), T(P + 8192, BF16, 2048)], [0, 2048], sr, sc, q, q) == 3
    assert call([E(), E()], [0, 0], sr, sc, q, q) == 0              # nothing to do


def test_ranged_reduction_validation(lib):
    fn = lib.mxfp8_amax_max_reduce_update_scales_ranged
    slots = T(P, F32, 4, 100)
    red = T(P + 4096, F32, 100)
    job = _capi.ScaleJob(T(P + 4096, F32, 2, 50), E(), T(P + 8192, U8, 2, 50), E(), 2, 1600)

    def call(triples, slots_=slots):
        flat = [v for t in triples for v in t]
        arr = (ctypes.c_int64 * max(1, len(flat)))(*flat)
        return fn(ctypes.byref(slots_), ctypes.byref(red), ctypes.byref(job), 1, arr,
                  len(triples), None)

    assert call([(4, 0, 10)]) == 1              # no slot 4
    assert call([(0, 20, 10)]) == 1             # begin > end
    assert call([(0, 0, 101)]) == 1             # past the slot
    assert call([(-1, 0, 1)]) == 1
    assert b"slot range" in lib.mxfp8_last_error()
    assert call([(0, 0, 10)], T(P, F32, 65, 100)) == 1  # ranges need at most 64 slots
    assert b"64" in lib.mxfp8_last_error()
    assert fn(ctypes.byref(slots), ctypes.byref(red), ctypes.byref(job), 1, None, 1, None) == 1


def test_nvfp4_validation(lib):
    F = F32
    inp = T(P, F, 100)
    ar, ac, at = T(P, F, 64, 4), T(P, F, 4, 64), T(P, F, 1)
    sr, sc = T(P, U8, 64, 4), T(P, U8, 4, 64)
    q = T(P, U8, 64 * 32)
    amax = lambda *a: lib.nvfp4_partial_amax(*[ctypes.byref(t) for t in a[:4]], *a[4:], None)
    cast = lambda *a: lib.nvfp4_partial_cast(*[ctypes.byref(t) for t in a[:6]], *a[6:], None)
    up = lambda *a: lib.nvfp4_update_scales(*[ctypes.byref(t) for t in a[:5]], *a[5:], None)
    assert amax(inp, ar, ac, E(), 64, 64, 0) == 4            # tensor amax required
    assert amax(inp, ar, ac, T(P, BF16, 1), 64, 64, 0) == 3  # tensor amax must be F32
    assert amax(inp, T(P, F, 64, 3), ac, at, 64, 64, 0) == 2  # 4 row blocks of 16 needed
    assert amax(inp, T(P, BF16, 64, 4), ac, at, 64, 64, 0) == 3  # NVFP4 amax grids are F32
    assert amax(E(), E(), E(), E(), 64, 64, 3) == 0           # empty fragment: nothing to do
    assert cast(inp, sr, sc, at, q, q, 64, 64, 1, 1) == 1       # odd start
    assert b"even" in lib.mxfp8_last_error()
    assert cast(T(P, F, 99), sr, sc, at, q, q, 64, 64, 0, 0) == 1  # odd length
    assert cast(inp, sr, sc, at, q, q, 64, 63, 0, 0) == 1      # odd cols
    assert cast(inp, sr, sc, at, q, q, 64, 64, 0, 3) == 1      # odd out_offset
    assert cast(inp, sr, E(), at, q, q, 64, 64, 0, 0) == 4     # colwise output needs scales
    assert cast(inp, sr, sc, E(), q, q, 64, 64, 0, 0) == 4     # tensor amax required
    assert cast(inp, sr, sc, at, T(P, U8, 49), E(), 64, 64, 0, 0) == 2  # 100 codes need 50 bytes
    assert cast(inp, T(P, U8, 64, 3), sc, at, q, q, 64, 64, 0, 0) == 2
    assert up(ar, ac, at, sr, E(), 64, 64) == 4
    assert up(ar, ac, at, T(P, U8, 4, 63), sc, 64, 64) == 2
