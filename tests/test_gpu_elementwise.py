"""Element-wise parity through the C ABI: every BF16 bit pattern and a million random
FP32 bit patterns through the cast, under many scale bytes; every BF16 amax pattern
and random FP32 amaxes through the scale update; the packed MAX reduction.
Bit-exact against the oracle (the special-value conventions are stated in the
oracle's header)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, to_device, to_host

pytestmark = pytest.mark.gpu

ROW_SCALES = np.array([0, 1, 8, 60, 100, 119, 127, 135, 160, 200, 240, 246, 250, 253, 254, 255],
                      np.uint8)


def _cast_with_scales(x: np.ndarray, rows: int, cols: int, s_r: np.ndarray, s_c: np.ndarray):
    xd = to_device(x)
    qr = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(xd, torch.from_numpy(s_r).cuda(), torch.from_numpy(s_c).cuda(), qr, qc,
                           rows, cols, 0)
    got_r, got_c = to_host(qr), to_host(qc)
    want_r = np.zeros(rows * cols, np.uint8)
    want_c = np.zeros(rows * cols, np.uint8)
    oracle.partial_cast(x, rows, cols, 0, s_r, s_c, want_r, want_c, 0)
    return got_r, got_c, want_r, want_c


def _scale_grids(rows, cols, seed):
    rng = np.random.default_rng(seed)
    s_r = np.repeat(ROW_SCALES[:rows, None], (cols + 31) // 32, axis=1).copy()
    s_c = rng.integers(0, 256, size=((rows + 31) // 32, cols), dtype=np.uint8)
    return s_r, s_c


def test_cast_every_bf16_pattern():
    rows, cols = 16, 65536
    x = np.tile(np.arange(65536, dtype=np.uint16), rows)
    s_r, s_c = _scale_grids(rows, cols, 1)
    gr, gc, wr, wc = _cast_with_scales(x, rows, cols, s_r, s_c)
    assert_bitwise((gr, gc), (wr, wc), "bf16 patterns")


def test_cast_random_f32_patterns():
    rows, cols = 16, 65536
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 2 ** 32, rows * cols, dtype=np.uint64).astype(np.uint32)
    # make a quarter of them moderate values so most scale bytes produce non-trivial codes
    mod = rng.standard_normal(rows * cols // 4).astype(np.float32) * 2.0 ** rng.integers(-20, 20, rows * cols // 4)
    bits[: mod.size] = mod.astype(np.float32).view(np.uint32)
    # BF16 rounding ties and carries into the exponent
    bits[mod.size:mod.size + 8] = [0x3F808000, 0x3F818000, 0x7F7F8000, 0x7F7FFFFF, 0x00008000,
                                   0x80018000, 0x3FFF8000, 0x437F8000]
    x = rng.permutation(bits).view(np.float32)
    s_r, s_c = _scale_grids(rows, cols, 3)
    gr, gc, wr, wc = _cast_with_scales(x, rows, cols, s_r, s_c)
    assert_bitwise((gr, gc), (wr, wc), "f32 patterns")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scale_update_patterns(dtype):
    rng = np.random.default_rng(4)
    if dtype == "bf16":
        a = np.arange(65536, dtype=np.uint16).reshape(256, 256)
        af = (a.astype(np.uint32) << 16).view(np.float32)
    else:
        a = rng.integers(0, 2 ** 32, 512 * 1024, dtype=np.uint64).astype(np.uint32).view(np.float32)
        a = a.reshape(512, 1024)
        af = a
    rows, cols = a.shape[0], a.shape[1] * 32  # so that the rowwise grid is exactly `a`
    ad = to_device(a).view(a.shape)
    s = torch.zeros(a.shape, dtype=torch.uint8, device="cuda")
    api.mxfp8_update_scales(ad, None, s, None, rows, cols)
    with np.errstate(invalid="ignore"):  # the patterns include signalling NaNs
        want = oracle.e8m0_from_amax(np.abs(af.astype(np.float64)))
    assert np.array_equal(to_host(s), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("nslots,elems", [(1, 1000), (4, 8_912_896), (3, 1001), (7, 64)])
def test_max_reduce(dtype, nslots, elems):
    rng = np.random.default_rng(nslots * 7 + elems)
    x = np.abs(rng.standard_normal((nslots, elems)).astype(np.float32))
    x[rng.random(x.shape) < 0.3] = 0.0
    if dtype == "bf16":
        x = (x.view(np.uint32) >> 16).astype(np.uint16)
    d = to_device(x).view(nslots, elems)
    out = torch.empty(elems, dtype=d.dtype, device="cuda")
    api.mxfp8_amax_max_reduce(d, out)
    assert np.array_equal(to_host(out), oracle.max_reduce(x))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_max_reduce_nan_bits_match_the_oracle(dtype):
    """NaN patterns of every kind in the slots reduce to the oracle's bits (the canonical
    quiet NaN), through the plain reduction and the reduction fused with the scales."""
    pats = (0x7F800001, 0x7FBFFFFF, 0x7FC00000, 0x7FFFFFFF, 0xFFC00000, 0xFF800001)
    rng = np.random.default_rng(12)
    x = wl.normal_f32(rng, (3, 256))
    for k, p in enumerate(pats):
        x.view(np.uint32)[k % 3, 8 * k + 1] = p
    if dtype == "bf16":
        hb = (x.view(np.uint32) >> 16).astype(np.uint16)
        for k, p in enumerate(pats):
            hb[k % 3, 8 * k + 1] = (p >> 16) | (0 if (p >> 16) & 0x7F else 0x40)
        x = hb
    want = oracle.max_reduce(x)
    bits = (lambda a: a.view(np.uint32)) if dtype == "f32" else (lambda a: a)
    d = to_device(x).view(3, 256)
    out = torch.empty(256, dtype=d.dtype, device="cuda")
    api.mxfp8_amax_max_reduce(d, out)
    assert np.array_equal(bits(to_host(out)), bits(want))
    # fused with the scale update: the reduced buffer viewed as an 8x32 amax grid
    red = torch.empty(256, dtype=d.dtype, device="cuda")
    sr = torch.empty((8, 32), dtype=torch.uint8, device="cuda")
    api.mxfp8_amax_max_reduce_update_scales(d, red, [(red.view(8, 32), None, sr, None, 8, 1024)])
    torch.cuda.synchronize()
    assert np.array_equal(bits(to_host(red)), bits(want))
    wf = want.astype(np.float32) if dtype == "f32" else wl.bf16_bits_to_f32(want)
    assert np.array_equal(sr.cpu().numpy().reshape(-1), oracle.e8m0_from_amax(wf.astype(np.float64)))


def test_max_reduce_nan_propagates():
    x = np.zeros((3, 64), np.float32)
    x[1, 5] = np.nan
    x[2, 5] = 1.0
    x[0, 6] = np.inf
    d = to_device(x).view(3, 64)
    out = torch.empty(64, dtype=torch.float32, device="cuda")
    api.mxfp8_amax_max_reduce(d, out)
    h = to_host(out)
    assert np.isnan(h[5]) and np.isinf(h[6]) and h[0] == 0.0


def _cast_with_scales_model(x, rows, cols, s_r, s_c, model):
    xd = to_device(x)
    qr = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    qc = torch.zeros(rows * cols, dtype=torch.uint8, device="cuda")
    api.mxfp8_partial_cast(xd, torch.from_numpy(s_r).cuda(), torch.from_numpy(s_c).cuda(), qr, qc,
                           rows, cols, 0, model_dtype=model)
    want_r = np.zeros(rows * cols, np.uint8)
    want_c = np.zeros(rows * cols, np.uint8)
    oracle.partial_cast(x, rows, cols, 0, s_r, s_c, want_r, want_c, 0, model=model)
    return to_host(qr), to_host(qc), want_r, want_c


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cast_f16_model_dtype(dtype):
    """Rounding through an FP16 model dtype: every BF16 pattern / random FP32 patterns."""
    rows, cols = 16, 65536
    rng = np.random.default_rng(5)
    if dtype == "bf16":
        x = np.tile(np.arange(65536, dtype=np.uint16), rows)
    else:
        bits = rng.integers(0, 2 ** 32, rows * cols, dtype=np.uint64).astype(np.uint32)
        mod = rng.standard_normal(rows * cols // 2).astype(np.float32) * 2.0 ** rng.integers(-30, 20, rows * cols // 2)
        bits[: mod.size] = mod.astype(np.float32).view(np.uint32)
        x = rng.permutation(bits).view(np.float32)
    s_r, s_c = _scale_grids(rows, cols, 6)
    gr, gc, wr, wc = _cast_with_scales_model(x, rows, cols, s_r, s_c, "f16")
    assert_bitwise((gr, gc), (wr, wc), f"f16 model {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("nslots", [1, 3])
def test_fused_reduce_scales_every_pattern(dtype, nslots):
    """The reduction fused with the scale update, against the oracle's MAX over the slots
    and E8M0 of the result: every BF16 bit pattern, or 512K random FP32 patterns plus
    every exponent field with edge mantissas, spread over 1 or 3 slots (the other slots
    holding smaller magnitudes or zeros)."""
    rng = np.random.default_rng(40 + nslots)
    if dtype == "bf16":
        pats = np.arange(65536, dtype=np.uint32)
        width = 16
    else:
        edge = (np.arange(256, dtype=np.uint32)[:, None] << 23) | np.array([0, 1, 0x400000, 0x7FFFFF], np.uint32)
        pats = np.concatenate([rng.integers(0, 2 ** 32, 512 * 1024, dtype=np.uint64).astype(np.uint32),
                               edge.reshape(-1), edge.reshape(-1) | 0x80000000])
        width = 32
    n = pats.size + (-pats.size) % 1024
    pats = np.concatenate([pats, np.zeros(n - pats.size, np.uint32)])
    slots = np.zeros((nslots, n), np.uint32)
    owner = rng.integers(0, nslots, n)
    slots[owner, np.arange(n)] = pats
    for k in range(nslots):  # the other slots: the pattern with a lower exponent, or 0
        other = owner != k
        lower = np.where((pats >> (width - 9)) & 0xFF > 2, pats - (np.uint32(2) << (width - 9)), 0)
        slots[k, other] = np.where(rng.random(other.sum()) < 0.5, lower[other], 0)
    if dtype == "bf16":
        x = slots.astype(np.uint16)
    else:
        x = slots.view(np.float32)
    d = to_device(x).view(nslots, n)
    red = torch.empty(n, dtype=d.dtype, device="cuda")
    cols = 1024 * 32
    sr = torch.empty((n // 1024, 1024), dtype=torch.uint8, device="cuda")
    api.mxfp8_amax_max_reduce_update_scales(d, red, [(red.view(n // 1024, 1024), None, sr, None, n // 1024, cols)])
    torch.cuda.synchronize()
    want = oracle.max_reduce(x)
    bits = (lambda a: a.view(np.uint32)) if dtype == "f32" else (lambda a: a)
    assert np.array_equal(bits(to_host(red)), bits(want))
    wf = want.astype(np.float32) if dtype == "f32" else wl.bf16_bits_to_f32(want)
    with np.errstate(invalid="ignore"):
        ws = oracle.e8m0_from_amax(np.abs(wf.astype(np.float64)))
    assert np.array_equal(sr.cpu().numpy().reshape(-1), ws.reshape(-1))
