"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each group targets one plausible mistake: a wrong rounding direction or tie rule,
an off-by-one exponent, a transposed block index, a dropped fragment element, a
write outside the fragment, a lost sign.
"""
import os

import numpy as np
import pytest
import torch

from mxfp8_master_weight_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line and not line.startswith("scale"):
                rows.append(line.split()[:2])
    return rows


# ------------------------------------------------------------------ E4M3

def _e4m3_table():
    """The 127 finite non-negative E4M3 values, built from the format definition."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def _e4m3_brute(v):
    """Nearest table entry by exhaustive search; ties to the even code; saturate."""
    table = _e4m3_table()
    out = np.empty(v.shape, np.uint8)
    for k, x in enumerate(v):
        if np.isnan(x):
            out[k] = 0x7F
            continue
        a = min(abs(x), 448.0)
        d = np.abs(table - a)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out[k] = code | (0x80 if np.signbit(x) else 0)
    return out


def test_e4m3_golden(oracle_mod):
    for val, code in _golden_rows("e4m3_points.txt"):
        got = int(oracle_mod.e4m3_encode(np.array([float(val)]))[0])
        assert got == int(code, 16), (val, hex(got), code)


def test_e4m3_vs_brute_force(oracle_mod):
    table = _e4m3_table()
    mids = (table[1:] + table[:-1]) / 2
    rng = np.random.default_rng(1)
    pts = np.concatenate([
        table, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
        2.0 ** rng.uniform(-14, 10, 4000), [0.0, 448.0, 447.99, 464.0, 465.0, 1e6, np.inf],
    ])
    pts = np.concatenate([pts, -pts, [np.nan]])
    assert np.array_equal(oracle_mod.e4m3_encode(pts), _e4m3_brute(pts))


def test_e4m3_vs_torch_float8(oracle_mod):
    """Library cross-check: torch's CPU float8_e4m3fn conversion after clamping to +-448."""
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(200000) * 2.0 ** rng.uniform(-12, 10, 200000)).astype(np.float32)
    v[:5] = [0.0, -0.0, 448.0, -460.0, 1e-30]
    ref = torch.from_numpy(v).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_decode_roundtrip(oracle_mod):
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle_mod.e4m3_decode(codes)
    assert np.array_equal(oracle_mod.e4m3_encode(vals), codes)


# ------------------------------------------------------------------ BF16

def _bf16_neighbour_search(x):
    """Nearest of the two BF16 values bracketing x (truncation and its successor), ties to even."""
    b = x.view(np.uint32)
    lo = b & np.uint32(0xFFFF0000)
    hi = lo + np.uint32(0x10000)  # next magnitude up (same sign)
    vlo = lo.view(np.float32).astype(np.float64)
    vhi = hi.view(np.float32).astype(np.float64)
    vx = x.astype(np.float64)
    dlo, dhi = np.abs(vx - vlo), np.abs(vhi - vx)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (((lo >> 16) & 1) == 1))
    return np.where(pick_hi, hi >> 16, lo >> 16).astype(np.uint16)


def test_bf16_vs_torch_and_neighbours(oracle_mod):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x007FFFFF, 0x00800000, 0x3F808000,
                        0x3F818000, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0xFF7FFFFF, 0x7F800000,
                        0xFF800000, 0x00008000, 0x00018000], np.uint32)
    bits = np.concatenate([bits, special])
    x = bits.view(np.float32)
    finite = np.isfinite(x)
    got = oracle_mod.bf16_rne_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)
    fin_no_overflow = finite & (np.abs(x) < np.float32(3.3e38))
    assert np.array_equal(got[fin_no_overflow], _bf16_neighbour_search(x[fin_no_overflow]))


# ------------------------------------------------------------------ E8M0

def _e8m0_brute(a):
    """Largest p with 2^p <= a by scanning powers of two; then clamp(p - 8) + 127."""
    powers = 2.0 ** np.arange(-160, 130, dtype=np.float64)
    out = np.empty(a.shape, np.uint8)
    for k, x in enumerate(a):
        if not np.isfinite(x):
            out[k] = 0xFF
        elif x == 0:
            out[k] = 0
        else:
            p = int(np.arange(-160, 130)[np.flatnonzero(powers <= x)[-1]])
            out[k] = min(max(p - 8, -127), 127) + 127
    return out


def test_e8m0_golden(oracle_mod):
    for val, byte in _golden_rows("e8m0_points.txt"):
        assert int(oracle_mod.e8m0_from_amax(np.array([float(val)]))[0]) == int(byte), val


def test_e8m0_all_bf16_patterns(oracle_mod):
    bits = np.arange(0, 0x8000, dtype=np.uint32) << 16
    with np.errstate(invalid="ignore"):  # the range holds signalling-NaN patterns
        a = bits.view(np.float32).astype(np.float64)
    assert np.array_equal(oracle_mod.e8m0_from_amax(a), _e8m0_brute(a))


def test_e8m0_random_f32_and_range_invariant(oracle_mod):
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 0x7F800000, 20000, dtype=np.uint32)
    a = bits.view(np.float32).astype(np.float64)
    got = oracle_mod.e8m0_from_amax(a)
    assert np.array_equal(got, _e8m0_brute(a))
    # unclamped range: the scaled block maximum lands in [256, 512)
    inner = (got > 0) & (got < 254)
    scaled = a[inner] * 2.0 ** (127 - got[inner].astype(np.float64))
    assert np.all((scaled >= 256) & (scaled < 512))


# ------------------------------------------------------------------ worked block

def test_worked_block(oracle_mod):
    rows = _golden_rows("worked_block.txt")
    vals = np.zeros(32, np.float32)
    codes = np.zeros(32, np.uint8)
    for k, (v, c) in enumerate(rows):
        vals[k] = np.float32(float(v))
        codes[k] = int(c, 16)
    amax_r, _, scale_r, _, q_r, _ = oracle_mod.full_cast(vals, 1, 32, colwise=False)
    assert amax_r[0, 0] == np.float32(3.0)
    assert scale_r[0, 0] == 120
    assert np.array_equal(q_r, codes)


# ------------------------------------------------------------------ amax geometry

def _amax_brute(x, rows, cols, start, length):
    """Block maxima by enumerating members of each block explicitly (dicts, no index algebra)."""
    r, c = {}, {}
    for k in range(start, start + length):
        i, j = divmod(k, cols)
        a = abs(float(x[k]))
        r[(i, j // 32)] = max(r.get((i, j // 32), 0.0), a)
        c[(i // 32, j)] = max(c.get((i // 32, j), 0.0), a)
    return r, c


@pytest.mark.parametrize("rows,cols", [(40, 7), (33, 65), (64, 96), (5, 100)])
def test_partial_amax_brute_force(oracle_mod, rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    n = rows * cols
    x = wl.normal_f32(rng, n)
    pairs = [(0, n), (0, 0), (n, 0), (n - 1, 1), (0, 1), (17, n // 4)]
    pairs += [(int(s), int(rng.integers(0, n - s + 1))) for s in rng.integers(0, n, 60)]
    nbr, nbc = (cols + 31) // 32, (rows + 31) // 32
    for start, length in pairs:
        sentinel = np.float32(-7.0)
        ar = np.full((rows, nbr + 2), sentinel, np.float32)  # padded leading dimension
        ac = np.full((nbc, cols + 3), sentinel, np.float32)
        oracle_mod.partial_amax(x[start:start + length], rows, cols, start, ar, ac)
        er, ec = _amax_brute(x, rows, cols, start, length)
        exp_r = np.full_like(ar, sentinel)
        exp_c = np.full_like(ac, sentinel)
        for (i, b), v in er.items():
            exp_r[i, b] = v
        for (cb, j), v in ec.items():
            exp_c[cb, j] = v
        assert np.array_equal(ar, exp_r), (start, length)
        assert np.array_equal(ac, exp_c), (start, length)


def test_amax_permutation_invariance(oracle_mod):
    rng = np.random.default_rng(5)
    x = wl.normal_f32(rng, 64 * 64).reshape(64, 64)
    y = x.copy()
    for i in range(64):  # permute inside each 1x32 row block
        y[i, :32] = y[i, rng.permutation(32)]
        y[i, 32:] = y[i, 32 + rng.permutation(32)]
    a = oracle_mod.full_cast(x.reshape(-1), 64, 64)
    b = oracle_mod.full_cast(y.reshape(-1), 64, 64)
    assert np.array_equal(a[0], b[0])


def test_amax_bf16_input_and_nan(oracle_mod):
    x = np.array([1.0, -3.5, 0.25, np.nan] + [0.0] * 28, np.float32)
    xb = wl.truncate_to_bf16_bits(x)
    ar = np.zeros((1, 1), np.uint16)
    oracle_mod.partial_amax(xb[:3], 1, 32, 0, ar, None)
    assert ar[0, 0] == wl.truncate_to_bf16_bits(np.array([3.5], np.float32))[0]
    oracle_mod.partial_amax(xb, 1, 32, 0, ar, None)
    assert np.isnan(wl.bf16_bits_to_f32(ar)[0, 0])


# ------------------------------------------------------------------ reduce

def test_max_reduce(oracle_mod):
    rng = np.random.default_rng(6)
    s = np.abs(wl.normal_f32(rng, (4, 1000)))
    s[1, 10] = 0.0
    assert np.array_equal(oracle_mod.max_reduce(s), s.max(axis=0))
    sb = wl.truncate_to_bf16_bits(s)
    assert np.array_equal(oracle_mod.max_reduce(sb),
                          wl.truncate_to_bf16_bits(s).view(np.uint16).max(axis=0))


def test_max_reduce_nan_propagates(oracle_mod):
    """A NaN in any slot makes the reduced entry NaN (so its E8M0 byte is 0xFF), in
    whichever slot it sits and whatever the other slots hold."""
    s = np.array([[np.nan, 1.0, 3.0, 0.0], [2.0, np.nan, 1.0, 0.5], [1.0, 5.0, np.nan, 0.25]],
                 np.float32)
    r = oracle_mod.max_reduce(s)
    assert np.isnan(r[:3]).all() and r[3] == 0.5
    assert (oracle_mod.e8m0_from_amax(r[:3].astype(np.float64)) == 0xFF).all()


# ------------------------------------------------------------------ cast

def _cast_brute(x_bf16_vals, scale_bytes):
    v = x_bf16_vals.astype(np.float64) * 2.0 ** (127 - scale_bytes.astype(np.float64))
    return _e4m3_brute(v)


def test_cast_vs_brute_force_and_error_bound(oracle_mod):
    rows, cols = 64, 96
    rng = np.random.default_rng(7)
    x = wl.normal_f32(rng, rows * cols)
    x[::97] *= 100.0
    amax_r, amax_c, s_r, s_c, q_r, q_c = oracle_mod.full_cast(x, rows, cols)
    y = wl.bf16_bits_to_f32(oracle_mod.bf16_rne_bits(x)).reshape(rows, cols)
    ii, jj = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    sr = s_r[ii, jj // 32]
    sc = s_c[ii // 32, jj]
    assert np.array_equal(q_r.reshape(rows, cols).ravel(), _cast_brute(y.ravel(), sr.ravel()))
    assert np.array_equal(q_c.reshape(rows, cols).ravel(), _cast_brute(y.ravel(), sc.ravel()))
    # error bound: |decode(q) * 2^e - y| <= half an E4M3 spacing at |v| (unsaturated)
    e = sr.astype(np.float64) - 127
    v = y.astype(np.float64) * 2.0 ** -e
    dec = oracle_mod.e4m3_decode(q_r.reshape(rows, cols))
    spacing = np.where(np.abs(v) < 2.0 ** -6, 2.0 ** -9,
                       2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 1e-300))) - 3))
    unsat = np.abs(v) < 448
    assert np.all(np.abs(dec - v)[unsat] <= spacing[unsat] / 2)


def test_row_only_equals_rowwise_half(oracle_mod):
    rng = np.random.default_rng(8)
    x = wl.normal_f32(rng, 96 * 64)
    bi = oracle_mod.full_cast(x, 96, 64, colwise=True)
    ro = oracle_mod.full_cast(x, 96, 64, colwise=False)
    for k in (0, 2, 4):
        assert np.array_equal(bi[k], ro[k])
    assert ro[1] is None and ro[3] is None and ro[5] is None


def _sharded_flow(oracle_mod, x, rows, cols, cuts, colwise=True, out_fragment=False):
    """Per-shard amax into separate zeroed slots, one max-reduce, scales, per-shard casts."""
    rdim, cdim = oracle_mod.block_dims(rows, cols)
    bounds = list(zip(cuts[:-1], cuts[1:]))
    slots_r = np.zeros((len(bounds),) + rdim, x.dtype)
    slots_c = np.zeros((len(bounds),) + cdim, x.dtype)
    for s, (a, b) in enumerate(bounds):
        oracle_mod.partial_amax(x[a:b], rows, cols, a, slots_r[s], slots_c[s] if colwise else None)
    ar = oracle_mod.max_reduce(slots_r)
    ac = oracle_mod.max_reduce(slots_c) if colwise else None
    sr = np.zeros(rdim, np.uint8)
    oracle_mod.update_scales(ar, *rdim, sr)
    sc = None
    if colwise:
        sc = np.zeros(cdim, np.uint8)
        oracle_mod.update_scales(ac, *cdim, sc)
    qr = np.full(rows * cols, 0xA5, np.uint8)
    qc = np.full(rows * cols, 0xA5, np.uint8) if colwise else None
    for a, b in bounds:
        if out_fragment:
            fr = np.full(b - a, 0xA5, np.uint8)
            fc = np.full(b - a, 0xA5, np.uint8) if colwise else None
            oracle_mod.partial_cast(x[a:b], rows, cols, a, sr, sc, fr, fc, 0)
            qr[a:b] = fr
            if colwise:
                qc[a:b] = fc
        else:
            oracle_mod.partial_cast(x[a:b], rows, cols, a, sr, sc, qr, qc, a)
    return ar, ac, sr, sc, qr, qc


@pytest.mark.parametrize("out_fragment", [False, True])
def test_union_of_fragments_equals_full(oracle_mod, out_fragment):
    rows, cols = 128, 96
    rng = np.random.default_rng(9)
    x = wl.normal_f32(rng, rows * cols)
    n = rows * cols
    full = oracle_mod.full_cast(x, rows, cols)
    for cuts in ([0, 17, 17 + n // 4, n], [0, 50 * 96 + 13, 50 * 96 + 13, n], [0, 33, 65, 99, n]):
        got = _sharded_flow(oracle_mod, x, rows, cols, cuts, out_fragment=out_fragment)
        for k in range(6):
            assert np.array_equal(got[k], full[k]), (cuts, k)


def test_boundary_inside_block_same_scale(oracle_mod):
    rows, cols = 32, 64
    rng = np.random.default_rng(10)
    x = wl.normal_f32(rng, rows * cols)
    x[5] = 0.9  # the block maximum sits on one side of the cut
    full = oracle_mod.full_cast(x, rows, cols)
    got = _sharded_flow(oracle_mod, x, rows, cols, [0, 13, rows * cols])
    assert got[2][0, 0] == full[2][0, 0] == oracle_mod.e8m0_from_amax(np.array([0.9]))[0]


def test_empty_fragment_writes_nothing(oracle_mod):
    rows, cols = 64, 64
    x = np.ones(rows * cols, np.float32)
    ar = np.full((rows, 2), 5.0, np.float32)
    ac = np.full((2, cols), 5.0, np.float32)
    oracle_mod.partial_amax(x[:0], rows, cols, 100, ar, ac)
    assert np.all(ar == 5.0) and np.all(ac == 5.0)
    q = np.full(rows * cols, 0xA5, np.uint8)
    sr = np.zeros((rows, 2), np.uint8)
    oracle_mod.partial_cast(x[:0], rows, cols, 100, sr, sr, q, q, 100)
    assert np.all(q == 0xA5)


def test_cast_bf16_input_no_second_rounding(oracle_mod):
    """BF16 input is already in the model dtype: the oracle must not alter it."""
    rng = np.random.default_rng(11)
    x = wl.truncate_to_bf16_bits(wl.normal_f32(rng, 32 * 64))
    xf = wl.bf16_bits_to_f32(x)
    a = oracle_mod.full_cast(x, 32, 64)
    b = oracle_mod.full_cast(xf, 32, 64)  # FP32 values that are exact BF16 values
    assert np.array_equal(a[4], b[4]) and np.array_equal(a[5], b[5])
    assert np.array_equal(a[2], b[2])


def test_scale_ff_and_nan_conventions(oracle_mod):
    assert oracle_mod.quantize(1.0, 0xFF) == 0x7F
    assert oracle_mod.quantize(float("nan"), 119) == 0x7F
    assert oracle_mod.quantize(float("inf"), 119) == 0x7E
    assert oracle_mod.quantize(float("-inf"), 119) == 0xFE
    assert oracle_mod.quantize(-1e-30, 119) == 0x80


# ------------------------------------------------------------------ FP16 model dtype

def test_f16_golden_points(oracle_mod):
    # hand-derived from the IEEE half-precision definition
    pts = {1.0: 0x3C00, 65504.0: 0x7BFF, 65519.99: 0x7BFF, 65520.0: 0x7C00, 2.0 ** -24: 0x0001,
           2.0 ** -25: 0x0000, 3 * 2.0 ** -26: 0x0001, -0.0: 0x8000, 0.1: 0x2E66, 2.0 ** -14: 0x0400,
           1.0 + 2.0 ** -11: 0x3C00, 1.0 + 3 * 2.0 ** -11: 0x3C02, -2.5: 0xC100}
    got = oracle_mod.f16_bits(np.array(list(pts.keys())))
    assert [int(g) for g in got] == list(pts.values())


def test_f16_vs_torch_and_neighbours(oracle_mod):
    rng = np.random.default_rng(12)
    bits = rng.integers(0, 2 ** 32, 1_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    mod = (rng.standard_normal(500_000) * 2.0 ** rng.uniform(-30, 18, 500_000)).astype(np.float32)
    x = np.concatenate([x, mod])
    got = oracle_mod.f16_bits(x.astype(np.float64))
    ref = torch.from_numpy(x.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    # independent: nearest of the two FP16 values bracketing x (np.float16 grid), ties to even
    small = mod[np.abs(mod) < 60000].astype(np.float64)
    lo = np.abs(small).astype(np.float16)  # some neighbour; refine by stepping
    cand = np.stack([np.nextafter(lo, np.float16(0)), lo, np.nextafter(lo, np.float16(np.inf))]).astype(np.float64)
    d = np.abs(cand - np.abs(small))
    best = d.min(axis=0)
    assert np.all(np.abs(oracle_mod.f16_bits(np.abs(small)).view(np.float16).astype(np.float64)
                         - np.abs(small)) == best)


def test_cast_with_f16_model(oracle_mod):
    rng = np.random.default_rng(13)
    rows, cols = 64, 96
    x = wl.normal_f32(rng, rows * cols) * np.float32(2.0) ** rng.integers(-20, 20, rows * cols).astype(np.float32)
    a = oracle_mod.full_cast(x, rows, cols, True, model="f16")
    yh = oracle_mod.f16_bits(x.astype(np.float64)).view(np.float16).astype(np.float64).reshape(rows, cols)
    ii, jj = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    v = yh * 2.0 ** (127 - a[2][ii, jj // 32].astype(np.float64))
    assert np.array_equal(a[4], oracle_mod.e4m3_encode(v.ravel()))
    # the amax and scales do not depend on the model dtype
    b = oracle_mod.full_cast(x, rows, cols, True, model="bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


# ------------------------------------------------------------------ GEMM scale layout

def test_swizzle_hand_points_and_bijection(oracle_mod):
    # 130 x 6 grid -> padded 256 x 8: two row tiles x two column tiles of 512 bytes
    nr, nc = 130, 6
    S = ((np.arange(nr)[:, None] * 7 + np.arange(nc)[None, :] * 3) % 251 + 1).astype(np.uint8)
    out = oracle_mod.swizzle_scales(S, nr, nc)
    assert out.size == 256 * 8
    # hand-derived offsets: tile (r//128, c//4) in row-major tile order (2 tiles per tile row),
    # inside the tile (r%32)*16 + ((r%128)//32)*4 + c%4
    assert out[0] == S[0, 0]
    assert out[1 * 16 + 0 * 4 + 1] == S[1, 1]
    assert out[0 * 16 + 1 * 4 + 2] == S[32, 2]
    assert out[31 * 16 + 3 * 4 + 3] == S[127, 3]
    assert out[1 * 512 + 5 * 16 + 2 * 4 + 1] == S[69, 5]
    assert out[2 * 512 + 1 * 16 + 0 * 4 + 0] == S[129, 0]
    # padding is zero and every entry of S appears exactly once
    assert np.count_nonzero(out) == nr * nc
    assert sorted(out[out != 0].tolist()) == sorted(S.ravel().tolist())


def test_swizzle_matches_reshape_formulation(oracle_mod):
    """Independent formulation: pad, split into 128x4 tiles, within a tile view rows as
    (4 groups of 32) and order bytes as (row%32, group, col)."""
    rng = np.random.default_rng(14)
    for nr, nc, tr in ((300, 10, False), (64, 512, True), (1, 1, False), (513, 257, True)):
        S = rng.integers(1, 255, (nr, nc + 3), dtype=np.uint8)  # padded leading dimension
        L = S[:nr, :nc].T if tr else S[:nr, :nc]
        pr, pc = -(-L.shape[0] // 128) * 128, -(-L.shape[1] // 4) * 4
        P = np.zeros((pr, pc), np.uint8)
        P[:L.shape[0], :L.shape[1]] = L
        tiles = P.reshape(pr // 128, 128, pc // 4, 4).transpose(0, 2, 1, 3)  # (tr, tc, 128, 4)
        want = tiles.reshape(pr // 128, pc // 4, 4, 32, 4).transpose(0, 1, 3, 2, 4).ravel()
        assert np.array_equal(oracle_mod.swizzle_scales(np.ascontiguousarray(S), nr, nc, tr), want)


# ------------------------------------------------------------------ leading dimensions, NaN bits

def test_update_scales_with_different_leading_dimensions(oracle_mod):
    """Amax grid and scale grid padded by different amounts: entry (r, c) of the scale
    grid comes from entry (r, c) of the amax grid, whatever either row stride is, and
    the padding columns keep their sentinel.  (Both grids carry spare rows so that a
    mistake with the strides still reads and writes inside the buffers.)"""
    rng = np.random.default_rng(21)
    nr, nc = 5, 6
    for ld_a, ld_s in ((9, 13), (13, 9)):
        amax = np.abs(wl.normal_f32(rng, (nr + 6, ld_a))) * np.float32(4.0)
        scale = np.full((nr + 6, ld_s), 0xA5, np.uint8)
        oracle_mod.update_scales(amax, nr, nc, scale)
        want = oracle_mod.e8m0_from_amax(amax[:nr, :nc].astype(np.float64))
        assert np.array_equal(scale[:nr, :nc], want), (ld_a, ld_s)
        assert (scale[:nr, nc:] == 0xA5).all() and (scale[nr:] == 0xA5).all()


NAN_F32_PATTERNS = (0x7F800001, 0x7FBFFFFF, 0x7FC00000, 0x7FFFFFFF, 0xFFC00000, 0xFF800001)


def test_nan_amax_is_the_canonical_quiet_nan(oracle_mod):
    """Whatever NaN pattern (signalling, quiet, negative, with payload) a block holds,
    its amax -- from the partial amax and from the MAX reduction -- is stored as
    0x7FC00000 (FP32) / 0x7FC0 (BF16), the stated convention."""
    for pat in NAN_F32_PATTERNS:
        x = np.zeros(64, np.float32)
        x[5] = np.float32(3.0)
        x.view(np.uint32)[7] = pat
        ar = np.zeros((1, 2), np.float32)
        oracle_mod.partial_amax(x, 1, 64, 0, ar, None)
        assert ar.view(np.uint32)[0, 0] == 0x7FC00000 and ar[0, 1] == 0.0, hex(pat)
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        xb[7] = pat >> 16 if (pat >> 16) & 0x7F else (pat >> 16) | 0x40  # keep it a NaN
        arb = np.zeros((1, 2), np.uint16)
        oracle_mod.partial_amax(xb, 1, 64, 0, arb, None)
        assert arb[0, 0] == 0x7FC0, hex(pat)
        slots = np.zeros((3, 4), np.float32)
        slots.view(np.uint32)[1, 2] = pat
        slots[2, 2] = 7.0
        red = oracle_mod.max_reduce(slots)
        assert red.view(np.uint32)[2] == 0x7FC00000 and red[0] == 0.0, hex(pat)


# ------------------------------------------------------------------ NVFP4 (stated convention)

def _e2m1_table():
    """The 8 non-negative E2M1 values, from the format definition (bias 1, 1 mantissa bit)."""
    vals = []
    for c in range(8):
        e, m = c >> 1, c & 1
        vals.append(0.5 * m if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    return np.array(vals)


def _e2m1_brute(v):
    table = _e2m1_table()
    out = np.empty(v.shape, np.uint8)
    for k, x in enumerate(v):
        a = min(abs(x), 6.0)
        d = np.abs(table - a)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out[k] = code | (0x8 if np.signbit(x) else 0)
    return out


def test_e2m1_golden(oracle_mod):
    for val, code in _golden_rows("e2m1_points.txt"):
        got = int(oracle_mod.e2m1_encode(np.array([float(val)]))[0])
        assert got == int(code, 16), (val, hex(got), code)


def test_e2m1_vs_brute_force(oracle_mod):
    table = _e2m1_table()
    mids = (table[1:] + table[:-1]) / 2
    rng = np.random.default_rng(41)
    v = np.concatenate([table, mids, np.nextafter(mids, 0), np.nextafter(mids, 10), -table, -mids,
                        rng.uniform(-8, 8, 20000), rng.uniform(-0.6, 0.6, 5000),
                        [6.5, 7.0, 7.5, 8.0, 1e30, -1e30, -0.0]])
    assert np.array_equal(oracle_mod.e2m1_encode(v), _e2m1_brute(v))
    for c in range(16):  # every code decodes to its value and encodes back
        d = float(oracle_mod.e2m1_decode(c))
        assert d == (-1 if c & 8 else 1) * table[c & 7]
        assert int(oracle_mod.e2m1_encode(np.array([d]))[0]) == c


def test_nvfp4_tensor_scale_special_cases(oracle_mod):
    """S = 2688 / G: exact for G = 2688 * 2^k and for divisors of 2688; 1 for G = 0;
    the largest float when the quotient overflows."""
    for k in range(-20, 21):
        assert oracle_mod.nvfp4_tensor_scale(2688.0 * 2.0 ** k) == 2.0 ** -k
    assert oracle_mod.nvfp4_tensor_scale(448.0) == 6.0
    assert oracle_mod.nvfp4_tensor_scale(12.0) == 224.0
    assert oracle_mod.nvfp4_tensor_scale(0.0) == 1.0
    assert oracle_mod.nvfp4_tensor_scale(1e-40) == float(np.finfo(np.float32).max)


def test_nvfp4_block_scale_points_and_bound(oracle_mod):
    s224 = np.float32(224.0)
    got = oracle_mod.nvfp4_block_scales(np.array([6.0, 3.0, 12.0, 0.0, 1e-3], np.float32), s224)
    # 224 = 1.75*2^7, 112 = 1.75*2^6, 448 = 1.75*2^8; 1e-3/6*224 = 0.03733 -> 1.25*2^-5
    assert list(got) == [0x76, 0x6E, 0x7E, 0x00, 0x12]
    # the block holding the tensor maximum always gets the largest E4M3 scale, 448
    rng = np.random.default_rng(42)
    g = np.float32(np.abs(rng.standard_normal(200)) * 10.0 ** rng.uniform(-30, 30, 200)).astype(np.float32)
    for gv in g:
        s = oracle_mod.nvfp4_tensor_scale(gv)
        assert int(oracle_mod.nvfp4_block_scales(np.array([gv], np.float32), s)[0]) == 0x7E, gv
    # every block scale is the E4M3 value nearest A*S/6 (within half a unit of E4M3)
    a = np.float32(rng.uniform(0, 1, 5000)) * np.float32(12.0)
    sc = oracle_mod.nvfp4_block_scales(a.astype(np.float32), s224)
    dec = oracle_mod.e4m3_decode(sc)
    u = a.astype(np.float64) / 6 * 224
    table = np.array(sorted(set(oracle_mod.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).tolist())))
    nearest = table[np.abs(table[None, :] - u[:, None]).argmin(axis=1)]
    assert np.all(np.abs(dec - u) <= np.abs(nearest - u) + 1e-9 * u)


def test_nvfp4_worked_block(oracle_mod):
    rows = _golden_rows("nvfp4_worked_block.txt")
    vals = np.array([float(v) for v, _ in rows], np.float32)
    codes = np.array([int(c, 16) for _, c in rows], np.uint8)
    with open(os.path.join(GOLDEN, "nvfp4_worked_block.txt")) as f:
        scales = [int(t, 16) for t in next(l for l in f if l.startswith("scale")).split()[1:]]
    ar, ac, at, sr, sc, qr, qc = oracle_mod.nvfp4_full_cast(vals, 1, 48, False)
    assert at[0] == 12.0 and list(ar[0]) == [6.0, 3.0, 12.0]
    assert list(sr[0]) == scales
    nib = np.stack([qr & 0xF, qr >> 4], axis=1).reshape(-1)
    assert np.array_equal(nib, codes)


def _nvfp4_inputs(rng, rows, cols, spread=2.0):
    n = rows * cols
    return (wl.normal_f32(rng, n) * np.float32(10.0) ** rng.uniform(-spread, spread, n).astype(np.float32))


def _nibbles(q, n):
    return np.stack([q & 0xF, q >> 4], axis=1).reshape(-1)[:n]


def test_nvfp4_partial_amax_brute_force(oracle_mod):
    """Block membership by dicts of members (no index algebra), 1x16 and 16x1 blocks,
    and the tensor amax as the maximum over every fragment element."""
    rng = np.random.default_rng(43)
    for rows, cols in ((40, 38), (33, 16), (17, 70)):
        n = rows * cols
        x = np.abs(_nvfp4_inputs(rng, rows, cols))
        for start, length in [(0, n), (3, n // 2), (n - 7, 7), (cols + 5, 2 * cols)]:
            frag = x[start:start + length]
            (rr, rc), (cr, cc) = oracle_mod.nvfp4_block_dims(rows, cols)
            ar = np.full((rr, rc), -1.0, np.float32)
            ac = np.full((cr, cc), -1.0, np.float32)
            at = np.array([0.5], np.float32)
            oracle_mod.nvfp4_partial_amax(frag, rows, cols, start, ar, ac, at)
            rb, cb = {}, {}
            for k in range(start, start + length):
                i, j = k // cols, k % cols
                rb.setdefault((i, j // 16), []).append(x[k])
                cb.setdefault((i // 16, j), []).append(x[k])
            want_r = np.full((rr, rc), -1.0, np.float32)
            want_c = np.full((cr, cc), -1.0, np.float32)
            for (i, b), m in rb.items():
                want_r[i, b] = max(m)
            for (c, j), m in cb.items():
                want_c[c, j] = max(m)
            assert np.array_equal(ar, want_r) and np.array_equal(ac, want_c)
            assert at[0] == max(0.5, frag.max())


def test_nvfp4_cast_invariants_and_error_bound(oracle_mod):
    """On a whole weight: every block whose scale is a normal E4M3 value has its largest
    element at E2M1 6 (the scale maps the block maximum near 6); every code is the
    E2M1 value nearest y*M (within the FP32 rounding of the product); the dequantised
    value decode(q) * decode(s) / S lies within half an E2M1 spacing (scaled) of y."""
    rng = np.random.default_rng(44)
    rows, cols = 48, 80
    x = _nvfp4_inputs(rng, rows, cols)
    ar, ac, at, sr, sc, qr, qc = oracle_mod.nvfp4_full_cast(x, rows, cols, True)
    s_enc = oracle_mod.nvfp4_tensor_scale(at[0])
    y = wl.bf16_bits_to_f32(oracle_mod.bf16_rne_bits(x)).astype(np.float64).reshape(rows, cols)
    table = _e2m1_table()
    for name, q, sgrid, blk in (("row", qr, sr, lambda i, j: (i, j // 16)),
                                ("col", qc, sc, lambda i, j: (i // 16, j))):
        codes = _nibbles(q, rows * cols).reshape(rows, cols)
        vals = oracle_mod.e2m1_decode(codes)
        groups = {}
        for i in range(rows):
            for j in range(cols):
                groups.setdefault(blk(i, j), []).append((i, j))
        for b, members in groups.items():
            s = int(sgrid[b])
            d = float(oracle_mod.e4m3_decode(np.array([s], np.uint8))[0])
            m = oracle_mod.nvfp4_multiplier(s, s_enc)
            if d >= 2.0 ** -6:
                assert max(abs(vals[i, j]) for i, j in members) == 6.0, (name, b)
            for i, j in members:
                p = y[i, j] * m
                spacing = 0.5 if abs(p) < 2 else (1.0 if abs(p) < 4 else 2.0)
                if abs(p) <= 6.0:
                    assert abs(abs(vals[i, j]) - abs(p)) <= spacing / 2 * (1 + 1e-6), (name, i, j)
                    assert abs(vals[i, j] * d / s_enc - y[i, j]) <= spacing / 2 * d / s_enc * (1 + 1e-5) + 1e-30
                assert np.signbit(vals[i, j]) == np.signbit(y[i, j]) or vals[i, j] == 0 and codes[i, j] in (0, 8)


def test_nvfp4_union_row_only_and_empty_fragment(oracle_mod):
    """Fragments with their own amax slots, MAX-reduced, give the whole-weight result bit
    for bit (full-size and fragment-size outputs); the row-only result is the rowwise
    half; an empty fragment writes nothing; a boundary inside a 16-value block gives the
    whole-block scale after the reduction."""
    rng = np.random.default_rng(45)
    rows, cols = 40, 48
    n = rows * cols
    x = _nvfp4_inputs(rng, rows, cols)
    full = oracle_mod.nvfp4_full_cast(x, rows, cols, True)
    cuts = [0, 6, 6, 16 * cols + 10, n - 2, n]   # an empty fragment; boundaries inside blocks
    (rr, rc), (cr, cc) = oracle_mod.nvfp4_block_dims(rows, cols)
    slots_r = np.zeros((len(cuts) - 1, rr, rc), np.float32)
    slots_c = np.zeros((len(cuts) - 1, cr, cc), np.float32)
    slots_t = np.zeros((len(cuts) - 1, 1), np.float32)
    for s, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        oracle_mod.nvfp4_partial_amax(x[a:b], rows, cols, a, slots_r[s], slots_c[s], slots_t[s])
    red_r = oracle_mod.max_reduce(slots_r.reshape(len(cuts) - 1, -1)).reshape(rr, rc)
    red_c = oracle_mod.max_reduce(slots_c.reshape(len(cuts) - 1, -1)).reshape(cr, cc)
    g = oracle_mod.max_reduce(slots_t)[0]
    assert g == full[2][0] and np.array_equal(red_r, full[0]) and np.array_equal(red_c, full[1])
    sr = np.zeros((rr, rc), np.uint8)
    sc = np.zeros((cr, cc), np.uint8)
    oracle_mod.nvfp4_update_scales(red_r, rr, rc, g, sr)
    oracle_mod.nvfp4_update_scales(red_c, cr, cc, g, sc)
    assert np.array_equal(sr, full[3]) and np.array_equal(sc, full[4])
    qr = np.full(n // 2, 0xA5, np.uint8)
    qc = np.full(n // 2, 0xA5, np.uint8)
    for a, b in zip(cuts[:-1], cuts[1:]):
        before = (qr.copy(), qc.copy())
        oracle_mod.nvfp4_partial_cast(x[a:b], rows, cols, a, sr, sc, g, qr, qc, a)
        if a == b:
            assert np.array_equal(before[0], qr) and np.array_equal(before[1], qc)
        # fragment-size output: the same codes, packed from nibble 0
        fr = np.full((b - a + 1) // 2, 0x5A, np.uint8)
        oracle_mod.nvfp4_partial_cast(x[a:b], rows, cols, a, sr, None, g, fr, None, 0)
        assert np.array_equal(_nibbles(fr, b - a), _nibbles(full[5], n)[a:b])
    assert np.array_equal(qr, full[5]) and np.array_equal(qc, full[6])
    ro = oracle_mod.nvfp4_full_cast(x, rows, cols, False)
    assert np.array_equal(ro[5], full[5]) and np.array_equal(ro[3], full[3]) and ro[6] is None


def test_nvfp4_bf16_input_is_not_rounded_again(oracle_mod):
    rng = np.random.default_rng(46)
    x = _nvfp4_inputs(rng, 32, 64)
    xb = oracle_mod.bf16_rne_bits(x)
    xf = wl.bf16_bits_to_f32(xb)
    a = oracle_mod.nvfp4_full_cast(xb, 32, 64, True)
    b = oracle_mod.nvfp4_full_cast(xf, 32, 64, True)
    for k in (0, 1, 2, 3, 4, 5, 6):
        assert np.array_equal(a[k], b[k]), k


def test_nvfp4_rounds_through_bf16_first(oracle_mod):
    """FP32 values just below an E2M1 midpoint whose BF16 rounding lands on it: the code
    follows the BF16 value (ties to even), not the FP32 one.  G = 6 gives S = 448 and a
    block scale of 448, so the multiplier is 1."""
    x = np.zeros(16, np.float32)
    x[:4] = [6.0, 0.7499, 1.7499, -4.9999]  # BF16: 0.75, 1.75, -5.0
    ar, ac, at, sr, sc, qr, qc = oracle_mod.nvfp4_full_cast(x, 1, 16, False)
    assert at[0] == 6.0 and sr[0, 0] == 0x7E
    assert oracle_mod.nvfp4_multiplier(0x7E, oracle_mod.nvfp4_tensor_scale(6.0)) == 1.0
    # 0.75 -> 1.0 (code 2), 1.75 -> 2.0 (code 4), -5.0 -> -4 (code 0xE)
    assert list(_nibbles(qr, 4)) == [0x7, 0x2, 0x4, 0xE]
