"""NVFP4 partial amax -> scale update -> partial cast through the C ABI, bit-exact against
the CPU oracle: the configuration workloads (even fragment offsets: two codes share a
byte), ragged shapes with random fragments and misaligned fragment pointers,
fragment-sized outputs, padded grids, every BF16 value through the E2M1 rounding, and
the sharded flow (per-fragment slots, one MAX reduction, scales, casts)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import to_device, to_host

pytestmark = pytest.mark.gpu

NAMES = ("amax_rowwise", "amax_colwise", "amax_tensor", "scale_rowwise", "scale_colwise",
         "data_rowwise", "data_colwise")


def gpu_nvfp4(frag, rows, cols, start, colwise, *, out_offset=None, out_bytes=None, shift=0,
              pad=0, amax_fill=0.0, sentinel=0xA5):
    (rr, rc), (cr, cc) = api.nvfp4_block_shapes(rows, cols)
    x = to_device(frag, shift)
    ar = torch.full((rr, rc + pad), amax_fill, dtype=torch.float32, device="cuda")
    ac = torch.full((cr, cc + pad), amax_fill, dtype=torch.float32, device="cuda") if colwise else None
    at = torch.zeros(1, dtype=torch.float32, device="cuda")
    api.nvfp4_partial_amax(x, ar, ac, at, rows, cols, start)
    sr = torch.full((rr, rc + pad), 0xEE, dtype=torch.uint8, device="cuda")
    sc = torch.full((cr, cc + pad), 0xEE, dtype=torch.uint8, device="cuda") if colwise else None
    api.nvfp4_update_scales(ar, ac, at, sr, sc, rows, cols)
    if out_offset is None:
        out_offset = start
    if out_bytes is None:
        out_bytes = (rows * cols + 1) // 2 if out_offset == start else (frag.size + out_offset + 1) // 2
    qr = torch.full((out_bytes,), sentinel, dtype=torch.uint8, device="cuda")
    qc = torch.full((out_bytes,), sentinel, dtype=torch.uint8, device="cuda") if colwise else None
    api.nvfp4_partial_cast(x, sr, sc, at, qr, qc, rows, cols, start, out_offset)
    torch.cuda.synchronize()
    h = lambda t: None if t is None else to_host(t)
    return h(ar), h(ac), h(at), h(sr), h(sc), h(qr), h(qc)


def oracle_nvfp4(frag, rows, cols, start, colwise, *, out_offset=None, out_bytes=None, pad=0,
                 amax_fill=0.0, sentinel=0xA5):
    (rr, rc), (cr, cc) = api.nvfp4_block_shapes(rows, cols)
    ar = np.full((rr, rc + pad), amax_fill, np.float32)
    ac = np.full((cr, cc + pad), amax_fill, np.float32) if colwise else None
    at = np.zeros(1, np.float32)
    oracle.nvfp4_partial_amax(frag, rows, cols, start, ar, ac, at)
    sr = np.full((rr, rc + pad), 0xEE, np.uint8)
    oracle.nvfp4_update_scales(ar, rr, rc, at[0], sr)
    sc = None
    if colwise:
        sc = np.full((cr, cc + pad), 0xEE, np.uint8)
        oracle.nvfp4_update_scales(ac, cr, cc, at[0], sc)
    if out_offset is None:
        out_offset = start
    if out_bytes is None:
        out_bytes = (rows * cols + 1) // 2 if out_offset == start else (frag.size + out_offset + 1) // 2
    qr = np.full(out_bytes, sentinel, np.uint8)
    qc = np.full(out_bytes, sentinel, np.uint8) if colwise else None
    oracle.nvfp4_partial_cast(frag, rows, cols, start, sr, sc, at[0], qr, qc, out_offset)
    return ar, ac, at, sr, sc, qr, qc


def assert_same(got, want, ctx=""):
    for name, g, w in zip(NAMES, got, want):
        if w is None:
            assert g is None, f"{ctx} {name}: expected absent"
            continue
        gb = g.view(np.uint32) if g.dtype == np.float32 else g
        wb = w.view(np.uint32) if w.dtype == np.float32 else w
        if not np.array_equal(gb, wb):
            bad = np.flatnonzero(gb.reshape(-1) != wb.reshape(-1))
            k = bad[0]
            raise AssertionError(f"{ctx} {name}: {bad.size} mismatches, first at flat {k}: "
                                 f"gpu {gb.reshape(-1)[k]:#x} oracle {wb.reshape(-1)[k]:#x}")


def _frag(w, a, b):
    return np.ascontiguousarray(w.data[a:b])


def test_cfg1_tiny_full():
    w = wl.cfg1_tiny()
    n = w.numel
    assert_same(gpu_nvfp4(_frag(w, 0, n), w.rows, w.cols, 0, True),
                oracle_nvfp4(_frag(w, 0, n), w.rows, w.cols, 0, True), "cfg1")


@pytest.mark.parametrize("colwise", [True, False])
def test_cfg2_bf16_partial(colwise):
    """The 1024x1024 BF16 weight with outliers and an all-zero block; the fragment starts at
    18 (the nearest even offset to the configuration's 17) and covers a quarter."""
    w = wl.cfg2_bf16_outliers()
    a, b = 18, 18 + w.numel // 4
    assert_same(gpu_nvfp4(_frag(w, a, b), w.rows, w.cols, a, colwise),
                oracle_nvfp4(_frag(w, a, b), w.rows, w.cols, a, colwise), f"cfg2 colwise={colwise}")


def test_cfg3_full_and_partial_union():
    """Full weight, and the union of three fragments (own slots, one MAX reduction) equals it."""
    w = wl.cfg3_square()
    n = w.numel
    full = oracle_nvfp4(_frag(w, 0, n), w.rows, w.cols, 0, True)
    assert_same(gpu_nvfp4(_frag(w, 0, n), w.rows, w.cols, 0, True), full, "cfg3 full")
    got = sharded_nvfp4(w.data, w.rows, w.cols, True, [0, 18, 18 + n // 4, n])
    want = (full[0], full[1], full[2], full[3], full[4], full[5], full[6])
    assert_same(got, want, "cfg3 union")


@pytest.mark.parametrize("colwise", [True, False])
def test_cfg4_headline(colwise):
    w = wl.cfg4_headline()
    n = w.numel
    assert_same(gpu_nvfp4(w.data, w.rows, w.cols, 0, colwise),
                oracle_nvfp4(w.data, w.rows, w.cols, 0, colwise), f"cfg4 colwise={colwise}")


def sharded_nvfp4(x, rows, cols, colwise, cuts):
    """Fragments in their own buffers, each with its own FP32 amax slot (tensor amax,
    rowwise grid, columnwise grid packed), one MAX reduction, scales, casts."""
    (rr, rc), (cr, cc) = api.nvfp4_block_shapes(rows, cols)
    P = 4 + rr * rc + (cr * cc if colwise else 0)
    S = len(cuts) - 1
    slots = torch.zeros((S, P), dtype=torch.float32, device="cuda")
    dt = torch.float32 if x.dtype == np.float32 else torch.bfloat16
    frags = [to_device(np.ascontiguousarray(x[a:b]), shift=s % 3) for s, (a, b) in enumerate(zip(cuts[:-1], cuts[1:]))]
    for s, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        v_t = slots[s, 0:1]
        v_r = slots[s, 4:4 + rr * rc].view(rr, rc)
        v_c = slots[s, 4 + rr * rc:].view(cr, cc) if colwise else None
        api.nvfp4_partial_amax(frags[s], v_r, v_c, v_t, rows, cols, a)
    red = torch.empty(P, dtype=torch.float32, device="cuda")
    api.mxfp8_amax_max_reduce(slots, red)
    r_t, r_r = red[0:1], red[4:4 + rr * rc].view(rr, rc)
    r_c = red[4 + rr * rc:].view(cr, cc) if colwise else None
    sr = torch.zeros((rr, rc), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((cr, cc), dtype=torch.uint8, device="cuda") if colwise else None
    api.nvfp4_update_scales(r_r, r_c, r_t, sr, sc, rows, cols)
    nb = (rows * cols + 1) // 2
    qr = torch.full((nb,), 0xA5, dtype=torch.uint8, device="cuda")
    qc = torch.full((nb,), 0xA5, dtype=torch.uint8, device="cuda") if colwise else None
    for s, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        api.nvfp4_partial_cast(frags[s], sr, sc, r_t, qr, qc, rows, cols, a)
    torch.cuda.synchronize()
    h = lambda t: None if t is None else to_host(t)
    return h(r_r), h(r_c), h(r_t), h(sr), h(sc), h(qr), h(qc)


RAGGED = [(1, 16), (7, 40), (33, 66), (64, 96), (50, 130), (17, 256)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", RAGGED)
def test_ragged_shapes_random_fragments(dtype, rows, cols):
    rng = np.random.default_rng(rows * 131 + cols)
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    cases = [(0, n), (0, 2), (n - 2, 2), (min(18, n - 2), max(2, n // 4 // 2 * 2))]
    for s in rng.integers(0, n // 2, 4):
        s = int(s) * 2
        cases.append((s, int(rng.integers(1, (n - s) // 2 + 1)) * 2))
    for k, (start, length) in enumerate(cases):
        frag = np.ascontiguousarray(x[start:start + length])
        colwise = k % 3 != 2
        got = gpu_nvfp4(frag, rows, cols, start, colwise, shift=k % 4, pad=k % 2, amax_fill=0.125)
        want = oracle_nvfp4(frag, rows, cols, start, colwise, pad=k % 2, amax_fill=0.125)
        assert_same(got, want, f"{dtype} {rows}x{cols} [{start},{start + length}) shift={k % 4}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift", [0, 1, 2, 3, 5, 7])
def test_every_fragment_misalignment_and_fragment_output(dtype, shift):
    """Fragments whose buffers start at every element offset (the realigning loads) and
    fragment-sized outputs (out_offset 0) at every even placement."""
    rows, cols = 96, 512
    rng = np.random.default_rng(shift)
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    for start, length in ((0, n), (2 * shift + 32, n // 2), (cols * 33 + 2 * shift, cols * 40 + 6)):
        frag = np.ascontiguousarray(x[start:start + length])
        for colwise in (True, False):
            got = gpu_nvfp4(frag, rows, cols, start, colwise, shift=shift)
            want = oracle_nvfp4(frag, rows, cols, start, colwise)
            assert_same(got, want, f"{dtype} shift={shift} [{start},+{length})")
            got = gpu_nvfp4(frag, rows, cols, start, colwise, shift=shift, out_offset=2 * shift)
            want = oracle_nvfp4(frag, rows, cols, start, colwise, out_offset=2 * shift)
            assert_same(got, want, f"{dtype} shift={shift} fragment output at {2 * shift}")


def test_every_bf16_value_through_e2m1():
    """With tensor amax 6 the tensor scale is 448, every block holding a 6 gets scale
    448 and multiplier 1, so the codes are the E2M1 rounding of the BF16 values
    themselves: every finite BF16 value of magnitude at most 6, 15 per block."""
    bits = np.arange(0, 0x10000, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 6.0)
    v = vals[keep]
    nb = (v.size + 14) // 15
    x = np.zeros((nb, 16), np.float32)
    x[:, 0] = 6.0
    x.reshape(-1)[np.arange(v.size) // 15 * 16 + 1 + np.arange(v.size) % 15] = v
    xb = wl.truncate_to_bf16_bits(x.reshape(-1))
    rows, cols = nb, 16
    got = gpu_nvfp4(xb, rows, cols, 0, True)
    want = oracle_nvfp4(xb, rows, cols, 0, True)
    assert_same(got, want, "every BF16 value")
    assert (want[3] == 0x7E).all()


def test_empty_fragment_and_odd_offsets_refused():
    x = torch.zeros(64, device="cuda")
    (rr, rc), (cr, cc) = api.nvfp4_block_shapes(8, 8)
    sr = torch.full((rr, rc), 7, dtype=torch.uint8, device="cuda")
    at = torch.ones(1, device="cuda")
    q = torch.full((32,), 0xA5, dtype=torch.uint8, device="cuda")
    api.nvfp4_partial_cast(x[:0], sr, None, at, q, None, 8, 8, 10)  # empty: writes nothing
    from mxfp8_master_weight_gb300 import _capi
    with pytest.raises(_capi.MXFP8Error) as e:
        api.nvfp4_partial_cast(x[:4], sr, None, at, q, None, 8, 8, 3)  # odd start
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert bool((q == 0xA5).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_amax_with_odd_fragment_boundaries(dtype):
    """The amax takes any fragment (only the cast needs even boundaries)."""
    rows, cols = 40, 70
    rng = np.random.default_rng(3)
    n = rows * cols
    x = wl.normal_f32(rng, n)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    for start, length in ((17, 1001), (1, n - 1), (cols * 16 - 1, 3)):
        frag = np.ascontiguousarray(x[start:start + length])
        (rr, rc), (cr, cc) = api.nvfp4_block_shapes(rows, cols)
        ar = torch.full((rr, rc), -2.0, device="cuda")
        ac = torch.full((cr, cc), -2.0, device="cuda")
        at = torch.zeros(1, device="cuda")
        api.nvfp4_partial_amax(to_device(frag, 1), ar, ac, at, rows, cols, start)
        war = np.full((rr, rc), -2.0, np.float32)
        wac = np.full((cr, cc), -2.0, np.float32)
        wat = np.zeros(1, np.float32)
        oracle.nvfp4_partial_amax(frag, rows, cols, start, war, wac, wat)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(ar), war) and np.array_equal(to_host(ac), wac)
        assert to_host(at)[0] == wat[0]


def _gpu_scales(a: np.ndarray, g: float) -> np.ndarray:
    """Rowwise NVFP4 scale update of an FP32 amax grid of 64 columns (a weight of 1024
    columns), tensor amax g, on the GPU."""
    rows = a.shape[0]
    (rr, rc), _ = api.nvfp4_block_shapes(rows, 1024)
    assert (rr, rc) == a.shape
    ad = to_device(a).view(a.shape)
    at = torch.tensor([g], dtype=torch.float32, device="cuda")
    sr = torch.full((rr, rc), 0xEE, dtype=torch.uint8, device="cuda")
    api.nvfp4_update_scales(ad, None, at, sr, None, rows, 1024)
    torch.cuda.synchronize()
    return to_host(sr)


def _oracle_scales(a: np.ndarray, g: float) -> np.ndarray:
    s = np.full(a.shape, 0xEE, np.uint8)
    oracle.nvfp4_update_scales(a, a.shape[0], a.shape[1], g, s)
    return s


def _grid64(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, np.float32).reshape(-1)
    pad = (-v.size) % 64
    return np.concatenate([v, np.zeros(pad, np.float32)]).reshape(-1, 64)


@pytest.mark.parametrize("j", [0, 3, -5, 20])
def test_scale_update_rounds_the_quotient_at_e4m3_ties(j):
    """fp32(A / 6) decides the E4M3 block scale where A / 6 * S falls on or next to a tie
    between two E4M3 codes.  With S = 2^j (tensor amax 2688 / 2^j) the product is exact, so
    amaxes 6 t +- k ulps around every E4M3 code value and midpoint t expose any error of
    one unit in the quotient's last place."""
    g = float(np.float32(2688.0) / np.float32(2.0 ** j))
    codes = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
    points = np.unique(np.concatenate([codes, (codes[:-1] + codes[1:]) / 2]))
    base = (points * 6.0 / 2.0 ** j).astype(np.float32)
    base = base[np.isfinite(base) & (base > 0)]
    k = np.arange(-48, 49, dtype=np.int64)
    bits = base.view(np.int32).astype(np.int64)[:, None] + k[None, :]
    bits = bits[(bits > 0) & (bits < 0x7F800000)]
    a = _grid64(bits.astype(np.int32).view(np.float32))
    assert np.array_equal(_gpu_scales(a, g), _oracle_scales(a, g))


def test_scale_update_every_mantissa_and_edge_values():
    """Every FP32 mantissa in binades around the quotient's exactness boundary (2^-126 to
    2^-122), at 1 and near the top of the range, plus zeros, subnormals, infinities, NaNs
    and negative amaxes, under several tensor amaxes (including 0 and a subnormal)."""
    m = np.arange(1 << 23, dtype=np.uint32)
    parts = [((np.uint32(e + 127) << np.uint32(23)) | m).view(np.float32)
             for e in (-126, -125, -124, -123, -122, 0, 127)]
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -1.0, -448.0, 1e-45, 1e-40,
                        1.1754942e-38, np.finfo(np.float32).max], np.float32)
    sub = (np.arange(1, 1 << 16, dtype=np.uint32) * np.uint32(127)).view(np.float32)
    a = _grid64(np.concatenate(parts + [special, sub]))
    for g in (2688.0, 1.0, 6.0, 3.0e-39, 0.0, 3.0e38):
        got, want = _gpu_scales(a, g), _oracle_scales(a, g)
        if not np.array_equal(got, want):
            bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
            v = a.reshape(-1)[bad[0]]
            raise AssertionError(f"g={g}: {bad.size} mismatches, first amax {v!r} "
                                 f"({np.float32(v).view(np.uint32):#x}): gpu {got.reshape(-1)[bad[0]]:#x} "
                                 f"oracle {want.reshape(-1)[bad[0]]:#x}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(64, 256), (96, 200), (40, 96), (160, 96)])
def test_small_launches_split_kernels(dtype, rows, cols):
    """Launches of few tiles run the split NVFP4 kernels (four warps per tile; the amax
    combines each 16-row half's column maxima across two warps): whole and partial (even)
    fragments, both direction sets, aligned and realigning buffers, against the oracle."""
    rng = np.random.default_rng(rows * 7 + cols + (dtype == "bf16"))
    n = rows * cols
    x = wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-3, 3, n).astype(np.float32)
    if dtype == "bf16":
        x = wl.truncate_to_bf16_bits(x)
    for start, length in [(0, n), (2 * cols + 6, n - 2 * cols - 40), (16 * cols, 8 * cols)]:
        frag = np.ascontiguousarray(x[start:start + length])
        for colwise in (True, False):
            for shift in (0, 2):
                got = gpu_nvfp4(frag, rows, cols, start, colwise, shift=shift)
                want = oracle_nvfp4(frag, rows, cols, start, colwise)
                assert_same(got, want, f"{dtype} {rows}x{cols} [{start},+{length}) col={colwise} shift={shift}")
