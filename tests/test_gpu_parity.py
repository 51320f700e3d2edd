"""Bit-exact parity of the CUDA path with the CPU oracle on the seeded workloads and
on edge cases: ragged shapes, fragment boundaries anywhere, misaligned fragment
pointers, fragment-sized outputs, padded block grids, empty fragments, and 64-bit
flat indices."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, gpu_fragment, oracle_fragment, to_device, to_host

pytestmark = pytest.mark.gpu


def _frag(w, f):
    return np.ascontiguousarray(w.data[f.start:f.end])


def test_cfg1_tiny_full():
    w = wl.cfg1_tiny()
    f = w.fragments[0]
    got = gpu_fragment(_frag(w, f), w.rows, w.cols, f.start, True)
    want = oracle_fragment(_frag(w, f), w.rows, w.cols, f.start, True)
    assert_bitwise(got, want, "cfg1")


@pytest.mark.parametrize("colwise", [True, False])
def test_cfg2_bf16_partial(colwise):
    w = wl.cfg2_bf16_outliers()
    f = w.fragments[0]
    got = gpu_fragment(_frag(w, f), w.rows, w.cols, f.start, colwise)
    want = oracle_fragment(_frag(w, f), w.rows, w.cols, f.start, colwise)
    assert_bitwise(got, want, f"cfg2 colwise={colwise}")
    # the all-zero 32x32 tile (rows 32..63, cols 64..95): scale byte 0, data 0
    sr, qr = got[2], got[4].reshape(w.rows, w.cols)
    assert np.all(sr[32:64, 2] == 0) and np.all(qr[32:64, 64:96] == 0)
    if colwise:
        assert np.all(got[3][1, 64:96] == 0)


def test_cfg2_row_only_equals_rowwise_half():
    w = wl.cfg2_bf16_outliers()
    f = w.fragments[0]
    bi = gpu_fragment(_frag(w, f), w.rows, w.cols, f.start, True)
    ro = gpu_fragment(_frag(w, f), w.rows, w.cols, f.start, False)
    for k in (0, 2, 4):
        assert np.array_equal(bi[k], ro[k])


def test_cfg3_full_and_partial():
    w = wl.cfg3_square()
    n = w.numel
    full = gpu_fragment(w.data, w.rows, w.cols, 0, True)
    assert_bitwise(full, oracle_fragment(w.data, w.rows, w.cols, 0, True), "cfg3 full")
    f = w.fragments[1]  # start 17, a quarter of the elements
    got = gpu_fragment(_frag(w, f), w.rows, w.cols, f.start, True)
    assert_bitwise(got, oracle_fragment(_frag(w, f), w.rows, w.cols, f.start, True), "cfg3 partial")
    assert f.start == 17 and f.length == n // 4


@pytest.fixture(scope="module")
def cfg4():
    w = wl.cfg4_headline()
    want = oracle_fragment(w.data, w.rows, w.cols, 0, True)
    return w, want


def test_cfg4_headline_bidirectional(cfg4):
    w, want = cfg4
    got = gpu_fragment(w.data, w.rows, w.cols, 0, True)
    assert_bitwise(got, want, "cfg4 bidirectional")


def test_cfg4_headline_row_only(cfg4):
    w, want = cfg4
    got = gpu_fragment(w.data, w.rows, w.cols, 0, False)
    rowwise_half = (want[0], None, want[2], None, want[4], None)
    assert_bitwise(got, rowwise_half, "cfg4 row-only")


RAGGED = [(33, 65), (100, 70), (1, 1), (31, 33), (64, 4096 + 40), (97, 256), (40, 7), (2, 1000)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", RAGGED)
def test_ragged_shapes_random_fragments(dtype, rows, cols):
    rng = np.random.default_rng(rows * 7919 + cols)
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    cases = [(0, n), (0, 1), (n - 1, 1), (min(17, n - 1), max(1, n // 4))]
    cases += [(int(s), int(rng.integers(1, n - s + 1))) for s in rng.integers(0, n, 4)]
    for k, (start, length) in enumerate(cases):
        frag = np.ascontiguousarray(x[start:start + length])
        shift = k % 4  # also exercises fragment pointers that are not 16-byte aligned
        colwise = k % 3 != 2
        got = gpu_fragment(frag, rows, cols, start, colwise, shift=shift, pad=k % 2,
                           amax_fill=0.125)
        want = oracle_fragment(frag, rows, cols, start, colwise, pad=k % 2, amax_fill=0.125)
        assert_bitwise(got, want, f"{dtype} {rows}x{cols} [{start},{start + length}) shift={shift}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pad,pad_s", [(3, 0), (0, 5), (2, 7), (8, 1)])
def test_amax_and_scale_grids_padded_differently(dtype, pad, pad_s):
    """The amax grids and the scale grids carry different row strides: every scale entry
    still comes from its own amax entry, and padding columns keep their sentinels."""
    rows, cols = 96, 160
    rng = np.random.default_rng(pad * 13 + pad_s)
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    for start, length in ((0, n), (17, n // 3), (5 * cols + 40, 2 * cols + 3)):
        frag = np.ascontiguousarray(x[start:start + length])
        for colwise in (True, False):
            got = gpu_fragment(frag, rows, cols, start, colwise, pad=pad, pad_s=pad_s,
                               amax_fill=0.5)
            want = oracle_fragment(frag, rows, cols, start, colwise, pad=pad, pad_s=pad_s,
                                   amax_fill=0.5)
            assert_bitwise(got, want, f"{dtype} pad={pad} pad_s={pad_s} [{start},+{length})")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift", [0, 1, 2, 3, 5])
def test_fragment_output_interface(dtype, shift):
    """out_offset = 0: the output holds only the fragment (fragment-output interface)."""
    rows, cols = 256, 1024
    rng = np.random.default_rng(shift)
    x = wl.normal_f32(rng, rows * cols)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    start, length = 17 + 32 * 1024 * 2, rows * cols // 3
    frag = np.ascontiguousarray(x[start:start + length])
    got = gpu_fragment(frag, rows, cols, start, True, out_offset=0, shift=shift)
    want = oracle_fragment(frag, rows, cols, start, True, out_offset=0)
    assert_bitwise(got, want, f"fragment output {dtype} shift={shift}")
    full = oracle_fragment(frag, rows, cols, start, True)
    assert np.array_equal(got[4], full[4][start:start + length])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("colwise", [True, False])
def test_every_output_misalignment(dtype, colwise):
    """Fragment-sized outputs whose virtual base sits at every byte offset inside an
    output word (4 bytes for FP32 input, 8 for BF16), combined with input buffers at
    every element offset inside a 16-byte chunk: interior tiles store aligned pieces
    (the specialisations for an aligned input and for the input offset that matches
    the output offset) or bytes; bytes before out_offset stay untouched."""
    rows, cols = 128, 1024
    rng = np.random.default_rng(33)
    x = wl.normal_f32(rng, rows * cols) * np.float32(2.0) ** rng.integers(-12, 12, rows * cols).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    start = 3 * cols + 5
    length = rows * cols - start - 11
    frag = np.ascontiguousarray(x[start:start + length])
    per_word = 4 if dtype == "f32" else 8
    for out_offset in range(per_word):
        want = oracle_fragment(frag, rows, cols, start, colwise, out_offset=out_offset)
        for shift in range(per_word):
            got = gpu_fragment(frag, rows, cols, start, colwise, out_offset=out_offset, shift=shift)
            assert_bitwise(got, want, f"{dtype} out_offset {out_offset} input shift {shift}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_output_misalignment_f16_model(dtype):
    """The aligned-piece stores of fragment-sized outputs with FP16 as the model dtype,
    for an aligned input buffer and for the input offset that matches each output offset."""
    rows, cols = 64, 1024
    rng = np.random.default_rng(34)
    x = wl.normal_f32(rng, rows * cols) * np.float32(2.0) ** rng.integers(-20, 8, rows * cols).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    start = cols + 3
    frag = np.ascontiguousarray(x[start:rows * cols - 5])
    per_word = 4 if dtype == "f32" else 8
    for out_offset in range(per_word):
        want = oracle_fragment(frag, rows, cols, start, True, out_offset=out_offset, model="f16")
        # input virtual base aligned (shift = start mod per_word), or offset like the output
        for shift in sorted({start % per_word, out_offset}):
            got = gpu_fragment(frag, rows, cols, start, True, out_offset=out_offset, shift=shift, model="f16")
            assert_bitwise(got, want, f"{dtype} f16 model out_offset {out_offset} shift {shift}")


def test_empty_fragment_writes_nothing():
    rows, cols = 128, 256
    ar = torch.full((rows, 8), 3.0, device="cuda")
    ac = torch.full((4, cols), 3.0, device="cuda")
    empty_view = torch.zeros(64, device="cuda")[10:10]  # zero elements, backing storage
    api.mxfp8_partial_amax(empty_view, ar, ac, rows, cols, 100)
    sr = torch.zeros((rows, 8), dtype=torch.uint8, device="cuda")
    q = torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(empty_view, sr, sr, q, q, rows, cols, 100)
    torch.cuda.synchronize()
    assert torch.all(ar == 3.0) and torch.all(ac == 3.0) and torch.all(q == 0xA5)


def test_boundary_inside_block_gives_whole_block_scale():
    rows, cols = 64, 256
    rng = np.random.default_rng(12)
    x = wl.normal_f32(rng, rows * cols)
    x[40 * cols + 70] = 5.0  # max of row block (40, 2) and column block (1, 70)
    cut = 40 * cols + 75    # inside both of those blocks
    dev = to_device(x)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    slots_r = torch.zeros((2, rr, rc), device="cuda")
    slots_c = torch.zeros((2, cr, cc), device="cuda")
    api.mxfp8_partial_amax(dev[:cut], slots_r[0], slots_c[0], rows, cols, 0)
    api.mxfp8_partial_amax(dev[cut:], slots_r[1], slots_c[1], rows, cols, cut)
    red_r = torch.empty((rr, rc), device="cuda")
    red_c = torch.empty((cr, cc), device="cuda")
    api.mxfp8_amax_max_reduce(slots_r.view(2, -1), red_r)
    api.mxfp8_amax_max_reduce(slots_c.view(2, -1), red_c)
    sr = torch.empty((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.empty((cr, cc), dtype=torch.uint8, device="cuda")
    api.mxfp8_update_scales(red_r, red_c, sr, sc, rows, cols)
    want = oracle.full_cast(x, rows, cols)
    assert np.array_equal(to_host(sr), want[2]) and np.array_equal(to_host(sc), want[3])
    assert to_host(sr)[40, 2] == oracle.e8m0_from_amax(np.array([5.0]))[0]


@pytest.mark.parametrize("start", [2 ** 32 - 5000, None])
def test_flat_indices_beyond_32_bits(start):
    """A weight with more than 2^32 elements and a small fragment far into it."""
    rows, cols = 131072, 32800
    n = rows * cols
    assert n > 2 ** 32
    if start is None:
        start = n - 3 * 32 * cols - 17
    length = 2 * 32 * cols + 1000
    rng = np.random.default_rng(13)
    frag = wl.normal_f32(rng, length)
    (rr, rc), (cr, cc) = api.block_shapes(rows, cols)
    s_r = torch.randint(100, 140, (rr, rc), dtype=torch.uint8, device="cuda")
    s_c = torch.randint(100, 140, (cr, cc), dtype=torch.uint8, device="cuda")
    x = to_device(frag)
    ar = torch.zeros((rr, rc), device="cuda")
    ac = torch.zeros((cr, cc), device="cuda")
    api.mxfp8_partial_amax(x, ar, ac, rows, cols, start)
    qr = torch.zeros(length, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(length, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(x, s_r, s_c, qr, qc, rows, cols, start, 0)
    torch.cuda.synchronize()
    r0, r1 = start // cols, (start + length - 1) // cols
    c0, c1 = r0 // 32, r1 // 32
    want_ar = np.zeros((rr, rc), np.float32)   # untouched pages stay virtual
    want_ac = np.zeros((cr, cc), np.float32)
    oracle.partial_amax(frag, rows, cols, start, want_ar, want_ac)
    assert np.array_equal(to_host(ar[r0:r1 + 1]), want_ar[r0:r1 + 1])
    assert np.array_equal(to_host(ac[c0:c1 + 1]), want_ac[c0:c1 + 1])
    assert float(ar[:r0].abs().sum()) == 0.0 and float(ac[:c0].abs().sum()) == 0.0
    hs_r, hs_c = to_host(s_r), to_host(s_c)
    want_qr = np.zeros(length, np.uint8)
    want_qc = np.zeros(length, np.uint8)
    oracle.partial_cast(frag, rows, cols, start, hs_r, hs_c, want_qr, want_qc, 0)
    assert np.array_equal(to_host(qr), want_qr) and np.array_equal(to_host(qc), want_qc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("colwise", [True, False])
def test_every_fragment_misalignment(dtype, colwise):
    """Fragments whose virtual base sits at every possible offset inside a 16-byte
    chunk (own buffers, as a rank's shard would be): the realigning vector path for
    interior tiles and the masked path for the tiles at the fragment's two ends."""
    rows, cols = 96, 2048
    rng = np.random.default_rng(21)
    x = wl.normal_f32(rng, rows * cols) * np.float32(3.0) ** rng.integers(-8, 8, rows * cols).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    per_chunk = 4 if dtype == "f32" else 8
    for k in range(per_chunk):
        start = 5 * cols + 3 + k
        length = rows * cols - start - 37
        frag = np.ascontiguousarray(x[start:start + length])
        got = gpu_fragment(frag, rows, cols, start, colwise, shift=k)
        want = oracle_fragment(frag, rows, cols, start, colwise)
        assert_bitwise(got, want, f"{dtype} misalignment {k}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(160, 96), (64, 100), (96, 132), (64, 200), (32, 8), (96, 1064)])
def test_tiles_cut_by_the_right_edge(dtype, rows, cols):
    """Weights narrower than, or not a multiple of, a tile's width: tiles whose rows the
    fragment covers whole take the fast path with the lanes past the right edge idle
    (whole weights, whole bands, and fragments that cut a band), bidirectional and
    row-only, against the oracle."""
    rng = np.random.default_rng(rows * 31 + cols)
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    cases = [(0, n), (min(32, rows - 1) * cols, max(1, min(32, rows // 2)) * cols), (cols + 4, n - cols - 4)]
    for start, length in cases:
        for colwise in (True, False):
            frag = np.ascontiguousarray(x[start:start + length])
            got = gpu_fragment(frag, rows, cols, start, colwise, amax_fill=0.125)
            want = oracle_fragment(frag, rows, cols, start, colwise, amax_fill=0.125)
            assert_bitwise(got, want, f"{dtype} {rows}x{cols} [{start},{start + length}) colwise={colwise}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(64, 256), (96, 200), (40, 96), (128, 512)])
def test_small_launches_every_path(dtype, rows, cols):
    """Launches of few tiles run the split kernels (four warps per tile; with right-edge
    tiles when the width is not a multiple of the tile's): whole and partial fragments,
    bidirectional and row-only, full-size and fragment-sized outputs (word-aligned or not),
    fragment buffers aligned and realigning (the realigning ones take the whole-tile kernels),
    BF16 and FP16 model dtypes -- every combination against the oracle."""
    rng = np.random.default_rng(rows * 101 + cols + (dtype == "bf16"))
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    frags = [(0, n), (cols * 33 + 5, n - cols * 33 - 40), (3 * cols, 2 * cols)]
    for start, length in frags:
        frag = np.ascontiguousarray(x[start:start + length])
        for colwise in (True, False):
            for out_offset in (start, 0, 3):
                for shift in (0, 1):
                    for model in ("bf16", "f16"):
                        kw = dict(out_offset=out_offset, amax_fill=0.25, model=model)
                        got = gpu_fragment(frag, rows, cols, start, colwise, shift=shift, **kw)
                        want = oracle_fragment(frag, rows, cols, start, colwise, **kw)
                        assert_bitwise(got, want, f"{dtype} {rows}x{cols} [{start},+{length}) col={colwise} "
                                                  f"out={out_offset} shift={shift} model={model}")
