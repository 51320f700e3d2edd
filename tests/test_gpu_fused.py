"""One-pass quantisation of fragments made of whole blocks: bit-identical to the oracle's
whole-weight cast (and so to the split amax -> scales -> cast path) on the seeded
workloads, ragged shapes, band-aligned and row-aligned fragments, misaligned fragment
buffers and fragment-sized outputs."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, to_device, to_host

pytestmark = pytest.mark.gpu


def _fused(frag, rows, cols, start, colwise, *, shift=0, with_amax=True, out_offset=None):
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    dt = torch.float32 if frag.dtype == np.float32 else torch.bfloat16
    x = to_device(frag, shift)
    ar = torch.zeros((rr, rc), dtype=dt, device="cuda") if with_amax else None
    ac = torch.zeros((cr, cc), dtype=dt, device="cuda") if (with_amax and colwise) else None
    sr = torch.full((rr, rc), 0xEE, dtype=torch.uint8, device="cuda")
    sc = torch.full((cr, cc), 0xEE, dtype=torch.uint8, device="cuda") if colwise else None
    if out_offset is None:
        out_offset, size = start, rows * cols
    else:
        size = frag.size + out_offset
    qr = torch.full((size,), 0xA5, dtype=torch.uint8, device="cuda")
    qc = torch.full((size,), 0xA5, dtype=torch.uint8, device="cuda") if colwise else None
    api.mxfp8_quantize_whole_blocks(x, ar, ac, sr, sc, qr, qc, rows, cols, start, out_offset)
    torch.cuda.synchronize()
    h = lambda t: None if t is None else to_host(t)
    return h(ar), h(ac), h(sr), h(sc), h(qr), h(qc)


def _oracle_fragment(frag, rows, cols, start, colwise, out_offset=None):
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    ar = np.zeros((rr, rc), frag.dtype)
    ac = np.zeros((cr, cc), frag.dtype) if colwise else None
    oracle.partial_amax(frag, rows, cols, start, ar, ac)
    sr = np.full((rr, rc), 0xEE, np.uint8)
    sc = np.full((cr, cc), 0xEE, np.uint8) if colwise else None
    # only blocks the fragment touches get a scale (untouched entries keep 0xEE)
    touched_r = np.zeros((rr, rc), bool)
    touched_c = np.zeros((cr, cc), bool)
    k = np.arange(start, start + frag.size)
    touched_r[k // cols, (k % cols) // 32] = True
    touched_c[(k // cols) // 32, k % cols] = True
    full_sr = np.zeros((rr, rc), np.uint8)
    oracle.update_scales(ar, rr, rc, full_sr)
    sr[touched_r] = full_sr[touched_r]
    if colwise:
        full_sc = np.zeros((cr, cc), np.uint8)
        oracle.update_scales(ac, cr, cc, full_sc)
        sc[touched_c] = full_sc[touched_c]
    if out_offset is None:
        out_offset, size = start, rows * cols
    else:
        size = frag.size + out_offset
    qr = np.full(size, 0xA5, np.uint8)
    qc = np.full(size, 0xA5, np.uint8) if colwise else None
    oracle.partial_cast(frag, rows, cols, start, sr, sc, qr, qc, out_offset)
    return ar, ac, sr, sc, qr, qc


@pytest.mark.parametrize("colwise", [True, False])
def test_fused_cfg4_headline(colwise):
    w = wl.cfg4_headline()
    got = _fused(w.data, w.rows, w.cols, 0, colwise)
    want = oracle.full_cast(w.data, w.rows, w.cols, colwise)
    assert_bitwise(got, want, f"fused cfg4 colwise={colwise}")


@pytest.mark.parametrize("cfg", ["cfg1", "cfg3"])
def test_fused_full_weights(cfg):
    w = wl.cfg_by_name(cfg)
    got = _fused(w.data, w.rows, w.cols, 0, True, with_amax=False)
    want = oracle.full_cast(w.data, w.rows, w.cols, True)
    assert_bitwise(got[2:], want[2:], f"fused {cfg}")
    assert got[0] is None and got[1] is None


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_every_misalignment(dtype):
    """A whole weight in a buffer that starts at every element offset inside a 16-byte
    chunk, so each offset's specialisation of the realigning loads runs on interior
    tiles, for both direction sets."""
    rows, cols = 96, 1024
    rng = np.random.default_rng(78)
    x = wl.normal_f32(rng, rows * cols) * np.float32(4.0) ** rng.integers(-6, 6, rows * cols).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    per_word = 4 if dtype == "f32" else 8
    for shift in range(per_word):
        for colwise in (True, False):
            got = _fused(x, rows, cols, 0, colwise, shift=shift)
            want = oracle.full_cast(x, rows, cols, colwise)
            assert_bitwise(got, want, f"fused {dtype} shift {shift} colwise {colwise}")
            # fragment-sized outputs at every byte offset inside an output word
            out_offset = (5 * shift + 1) % per_word
            got = _fused(x, rows, cols, 0, colwise, shift=shift, out_offset=out_offset)
            want = _oracle_fragment(x, rows, cols, 0, colwise, out_offset=out_offset)
            assert_bitwise(got, want, f"fused {dtype} shift {shift} out_offset {out_offset}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(33, 65), (100, 70), (64, 4096 + 40), (97, 256), (1, 1)])
def test_fused_ragged_full_weights(dtype, rows, cols):
    rng = np.random.default_rng(rows + 1000 * cols)
    x = wl.normal_f32(rng, rows * cols) * np.float32(10.0) ** rng.uniform(-3, 3, rows * cols).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    for shift in (0, 1, 3):
        got = _fused(x, rows, cols, 0, True, shift=shift)
        want = oracle.full_cast(x, rows, cols, True)
        assert_bitwise(got, want, f"fused {dtype} {rows}x{cols} shift {shift}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift", [0, 1, 2, 5])
def test_fused_band_and_row_aligned_fragments(dtype, shift):
    rows, cols = 256, 1024
    rng = np.random.default_rng(40 + shift)
    x = wl.normal_f32(rng, rows * cols)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    # bidirectional: whole 32-row bands
    start, end = 32 * cols * 2, 32 * cols * 7
    frag = np.ascontiguousarray(x[start:end])
    assert_bitwise(_fused(frag, rows, cols, start, True, shift=shift),
                   _oracle_fragment(frag, rows, cols, start, True), f"bands {dtype} {shift}")
    # row-only: start and end on 1x32 block boundaries inside rows and bands
    start, end = 5 * cols + 64, 77 * cols + 992
    frag = np.ascontiguousarray(x[start:end])
    assert_bitwise(_fused(frag, rows, cols, start, False, shift=shift),
                   _oracle_fragment(frag, rows, cols, start, False), f"rows {dtype} {shift}")
    # fragment-sized output
    assert_bitwise(_fused(frag, rows, cols, start, False, shift=shift, out_offset=0),
                   _oracle_fragment(frag, rows, cols, start, False, out_offset=0),
                   f"fragment output {dtype} {shift}")


def test_fused_batched_equals_single():
    rng = np.random.default_rng(44)
    jobs, singles = [], []
    for rows, cols, col in ((64, 512, True), (96, 256, False), (128, 1024, True)):
        x = to_device(wl.normal_f32(rng, rows * cols))
        (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
        outs = []
        for _ in range(2):
            outs.append([torch.zeros((rr, rc), dtype=torch.uint8, device="cuda"),
                         torch.zeros((cr, cc), dtype=torch.uint8, device="cuda") if col else None,
                         torch.zeros(rows * cols, dtype=torch.uint8, device="cuda"),
                         torch.zeros(rows * cols, dtype=torch.uint8, device="cuda") if col else None])
        a, b = outs
        jobs.append((x, None, None, a[0], a[1], a[2], a[3], rows, cols, 0))
        api.mxfp8_quantize_whole_blocks(x, None, None, b[0], b[1], b[2], b[3], rows, cols, 0)
        singles.append((a, b))
    api.mxfp8_quantize_whole_blocks_batched(jobs)
    torch.cuda.synchronize()
    for a, b in singles:
        for u, v in zip(a, b):
            assert (u is None and v is None) or torch.equal(u, v)


@pytest.mark.parametrize("colwise", [True, False])
def test_fused_f16_model(colwise):
    rows, cols = 512, 2048
    rng = np.random.default_rng(45)
    x = wl.normal_f32(rng, rows * cols) * np.float32(2.0) ** rng.integers(-20, 20, rows * cols).astype(np.float32)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    xd = to_device(x)
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda") if colwise else None
    qr = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda") if colwise else None
    api.mxfp8_quantize_whole_blocks(xd, None, None, sr, sc, qr, qc, rows, cols, 0, model_dtype="f16")
    torch.cuda.synchronize()
    want = oracle.full_cast(x, rows, cols, colwise, model="f16")
    got = (None, None, to_host(sr), None if sc is None else to_host(sc), to_host(qr),
           None if qc is None else to_host(qc))
    assert_bitwise(got[2:], want[2:], f"fused f16 colwise={colwise}")


def test_batched_cast_mixed_model_dtypes():
    rows, cols = 64, 512
    rng = np.random.default_rng(46)
    x = wl.normal_f32(rng, rows * cols) * np.float32(1e3)
    xd = to_device(x)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    sr = torch.full((rr, rc), 120, dtype=torch.uint8, device="cuda")
    outs = {m: torch.zeros(rows * cols, dtype=torch.uint8, device="cuda") for m in ("bf16", "f16")}
    api.mxfp8_partial_cast_batched([(xd, sr, None, outs["bf16"], None, rows, cols, 0, None, "bf16"),
                                    (xd, sr, None, outs["f16"], None, rows, cols, 0, None, "f16")])
    torch.cuda.synchronize()
    hs = to_host(sr)
    for m, q in outs.items():
        want = np.zeros(rows * cols, np.uint8)
        oracle.partial_cast(x, rows, cols, 0, hs, None, want, None, 0, model=m)
        assert np.array_equal(to_host(q), want), m


@pytest.mark.parametrize("colwise", [True, False])
@pytest.mark.parametrize("shift", [0, 1, 2, 3])
def test_fused_without_amax_outputs(colwise, shift):
    """No amax output requested (FP32 input, word-aligned outputs): the one-pass kernel
    takes block maxima on exponents only (packed high halves); scales and data stay
    bit-identical to the oracle, on the headline-like value spread, whole weights,
    band-aligned fragments and fragment buffers at every element offset, and blocks whose
    maximum sits on an exponent boundary, a subnormal, zero, infinity or NaN."""
    rows, cols = 192, 640
    rng = np.random.default_rng(60 + shift)
    n = rows * cols
    x = (wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-6, 6, n).astype(np.float32))
    specials = np.array([2.0, np.nextafter(np.float32(2.0), np.float32(0)), 1e-40, 0.0, -0.0,
                         np.inf, -np.inf, np.nan, 448.0 * 2 ** 100, 2.0 ** -126], np.float32)
    for k, v in enumerate(specials):  # one special per row block, in the first rows
        x[k * cols + 7 * k] = v
    x[5 * cols:6 * cols] = 0.0        # a whole zero row
    for start, length in ((0, n), (32 * cols, 64 * cols), (cols * 96, n - cols * 96)):
        frag = np.ascontiguousarray(x[start:start + length])
        got = _fused(frag, rows, cols, start, colwise, shift=shift, with_amax=False)
        want = _oracle_fragment(frag, rows, cols, start, colwise)
        assert_bitwise(got[2:], want[2:], f"no amax out, shift {shift} [{start},+{length})")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_amax", [True, False])
@pytest.mark.parametrize("colwise", [True, False])
def test_fused_staged_path(dtype, with_amax, colwise):
    """Fragments of whole 32-row bands of a weight whose columns are a multiple of the
    tile width, aligned buffers and outputs: the one-pass kernel that stages tiles in
    shared memory.  Whole weight, interior band ranges and a single band; bit-identical
    to the oracle (values spread over 12 decades, special values in the first rows)."""
    rows, cols = 32 * 13, 1024
    rng = np.random.default_rng(70 + with_amax + 2 * colwise)
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-6, 6, n).astype(np.float32)
    x[:8] = np.array([0.0, -0.0, 1e-40, 2.0, np.nextafter(np.float32(2.0), np.float32(0)),
                      448.0, -3.0e38, 1.5], np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    for a, b in ((0, rows), (32, 32 * 9), (32 * 12, rows), (64, 96)):
        start, length = a * cols, (b - a) * cols
        frag = np.ascontiguousarray(x[start:start + length])
        got = _fused(frag, rows, cols, start, colwise, with_amax=with_amax)
        want = _oracle_fragment(frag, rows, cols, start, colwise)
        if with_amax:
            assert_bitwise(got, want, f"{dtype} staged rows [{a},{b})")
        else:
            assert_bitwise(got[2:], want[2:], f"{dtype} staged rows [{a},{b}) no amax")
