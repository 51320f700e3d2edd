"""Flat indices beyond 2^31: 64-bit indexing in every kernel.

A 65600 x 32768 FP32 weight (2,149,580,800 elements, 8.6 GB) goes through the split path
(amax, scale update, cast) and the one-pass path.  The 64-row bands at both ends -- the
last one entirely above flat index 2^31 -- hold seeded data from the input generators and
are checked bit for bit against the oracle run on those bands alone (a band of whole
32-row blocks does not depend on other rows); the rest of the weight is seeded device-side
filler.  A fragment straddling index 2^31 is checked the same way on the rows it touches,
and guard bytes after every output must stay untouched."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_master_weight_gb300 import api
from mxfp8_master_weight_gb300 import workloads as wl

from flows import assert_bitwise, to_host

pytestmark = pytest.mark.gpu

ROWS, COLS = 65600, 32768
N = ROWS * COLS
BANDS = ((0, 64), (ROWS - 64, ROWS))
GUARD = 4096
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def big():
    if torch.cuda.mem_get_info()[0] < 20e9:
        pytest.skip("needs 20 GB of free device memory")
    assert N > 2 ** 31
    x = torch.empty(N, dtype=torch.float32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    x.normal_(0.0, 0.02, generator=g)
    rng = np.random.default_rng(12)
    bands = {}
    for r0, r1 in BANDS:
        h = wl.normal_f32(rng, (r1 - r0) * COLS)
        h *= np.float32(10.0) ** rng.uniform(-3, 3, h.size).astype(np.float32)
        x[r0 * COLS:r1 * COLS].copy_(torch.from_numpy(h))
        bands[(r0, r1)] = h
    (rr, rc), (cr, cc) = api.block_shapes(ROWS, COLS)
    bufs = dict(
        ar=torch.zeros((rr, rc), device="cuda"), ac=torch.zeros((cr, cc), device="cuda"),
        sr=torch.empty((rr, rc), dtype=torch.uint8, device="cuda"),
        sc=torch.empty((cr, cc), dtype=torch.uint8, device="cuda"),
        qr=torch.full((N + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda"),
        qc=torch.full((N + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda"))
    yield x, bands, bufs
    del x, bufs
    torch.cuda.empty_cache()


def _band_results(bufs, r0, r1):
    b0, b1 = r0 // 32, (r1 + 31) // 32
    return (to_host(bufs["ar"][r0:r1]), to_host(bufs["ac"][b0:b1]), to_host(bufs["sr"][r0:r1]),
            to_host(bufs["sc"][b0:b1]), to_host(bufs["qr"][r0 * COLS:r1 * COLS]),
            to_host(bufs["qc"][r0 * COLS:r1 * COLS]))


def _check_bands_and_guards(bands, bufs, what):
    torch.cuda.synchronize()
    for (r0, r1), h in bands.items():
        want = oracle.full_cast(h, r1 - r0, COLS, True)
        assert_bitwise(_band_results(bufs, r0, r1), want, f"{what} rows [{r0}, {r1})")
    for k in ("qr", "qc"):
        assert bool((bufs[k][N:] == SENTINEL).all()), f"{what}: {k} written past its end"


def test_split_path_beyond_2_31(big):
    x, bands, bufs = big
    out_r, out_c = bufs["qr"][:N], bufs["qc"][:N]
    api.mxfp8_partial_amax(x, bufs["ar"], bufs["ac"], ROWS, COLS, 0)
    api.mxfp8_update_scales(bufs["ar"], bufs["ac"], bufs["sr"], bufs["sc"], ROWS, COLS)
    api.mxfp8_partial_cast(x, bufs["sr"], bufs["sc"], out_r, out_c, ROWS, COLS, 0)
    _check_bands_and_guards(bands, bufs, "split")


def test_one_pass_beyond_2_31(big):
    x, bands, bufs = big
    for k in ("qr", "qc"):
        bufs[k].fill_(SENTINEL)
    bufs["ar"].zero_()
    bufs["ac"].zero_()
    api.mxfp8_quantize_whole_blocks(x, bufs["ar"], bufs["ac"], bufs["sr"], bufs["sc"],
                                    bufs["qr"][:N], bufs["qc"][:N], ROWS, COLS, 0)
    _check_bands_and_guards(bands, bufs, "one-pass")


def test_fragment_straddling_2_31(big):
    """Partial amax and cast of [2^31 - 1000, 2^31 + 5000): the oracle runs the same
    fragment as a fragment of the 33 rows it touches (from the start of their band)."""
    x, _, bufs = big
    start, end = 2 ** 31 - 1000, 2 ** 31 + 5000
    frag = x[start:end]
    bufs["ar"].zero_()
    bufs["ac"].zero_()
    api.mxfp8_partial_amax(frag, bufs["ar"], bufs["ac"], ROWS, COLS, start)
    api.mxfp8_update_scales(bufs["ar"], bufs["ac"], bufs["sr"], bufs["sc"], ROWS, COLS)
    bufs["qr"].fill_(SENTINEL)
    bufs["qc"].fill_(SENTINEL)
    api.mxfp8_partial_cast(frag, bufs["sr"], bufs["sc"], bufs["qr"][:N], bufs["qc"][:N], ROWS, COLS, start)
    torch.cuda.synchronize()
    h = to_host(frag)
    ra = (start // COLS) // 32 * 32                  # first row of the touched band
    sub_rows = (end - 1) // COLS - ra + 1
    sub_start = start - ra * COLS
    (rr, rc), (cr, cc) = api.block_shapes(sub_rows, COLS)
    want_ar, want_ac = np.zeros((rr, rc), np.float32), np.zeros((cr, cc), np.float32)
    oracle.partial_amax(h, sub_rows, COLS, sub_start, want_ar, want_ac)
    want_sr, want_sc = np.zeros((rr, rc), np.uint8), np.zeros((cr, cc), np.uint8)
    oracle.update_scales(want_ar, rr, rc, want_sr)
    oracle.update_scales(want_ac, cr, cc, want_sc)
    want_qr = np.full(sub_rows * COLS, SENTINEL, np.uint8)
    want_qc = np.full(sub_rows * COLS, SENTINEL, np.uint8)
    oracle.partial_cast(h, sub_rows, COLS, sub_start, want_sr, want_sc, want_qr, want_qc, sub_start)
    b0 = ra // 32
    got = (to_host(bufs["ar"][ra:ra + sub_rows]), to_host(bufs["ac"][b0:b0 + cr]),
           to_host(bufs["sr"][ra:ra + sub_rows]), to_host(bufs["sc"][b0:b0 + cr]),
           to_host(bufs["qr"][ra * COLS:(ra + sub_rows) * COLS]),
           to_host(bufs["qc"][ra * COLS:(ra + sub_rows) * COLS]))
    assert_bitwise(got, (want_ar, want_ac, want_sr, want_sc, want_qr, want_qc), "straddling 2^31")
    assert bool((bufs["qr"][:start] == SENTINEL).all()) and bool((bufs["qr"][end:] == SENTINEL).all())
