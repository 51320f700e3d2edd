"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU, in a
temporary directory), builds it as a separate library, and runs the pins of
test_oracle_pins.py against it: at least one pin must fail.  The mistakes are the
kinds a restatement of the pages' steps could make -- a rounding tie rule, an
exponent or threshold off by one, a lost sign of zero, a dropped fragment element,
the wrong direction's scale, a write outside the touched blocks, NaN not
propagated, a swapped index in the GEMM layout.  Every mutant stays inside its
buffers, so a mutant can only compute wrong values, never touch foreign memory.
"""
import importlib.util
import inspect
import os

import pytest

import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_INIT = os.path.join(ROOT, "oracle", "__init__.py")
ORACLE_SRC = os.path.join(ROOT, "oracle", "mxfp8_oracle.c")

MUTATIONS = {
    "e4m3 ties away from zero": (
        "double r = nearbyint(a / quantum);            /* ties to even (default mode) */",
        "double r = round(a / quantum);"),
    "bf16 ties away from zero": (
        "double r = nearbyint(a / quantum) * quantum;  /* a/quantum is exact in double */",
        "double r = round(a / quantum) * quantum;"),
    "e8m0 exponent off by one": (
        "e = floor_log2(a) - 8;", "e = floor_log2(a) - 7;"),
    "e4m3 sign of zero lost": (
        "uint8_t sign = signbit(v) ? 0x80 : 0x00;", "uint8_t sign = v < 0 ? 0x80 : 0x00;"),
    "bf16 subnormal threshold off by one": (
        "if (p < -126) p = -126;", "if (p < -125) p = -125;"),
    "e4m3 saturates only past 480": (
        "if (a >= 448.0) return sign | 0x7E;", "if (a > 480.0) return sign | 0x7E;"),
    "scale exponent off by one": (
        "return ldexp(y, 127 - (int)s);", "return ldexp(y, 126 - (int)s);"),
    "first fragment element dropped from the amax": (
        "    for (int64_t k = start; k < start + len; ++k) {\n        int64_t i = k / cols, j = k % cols;\n        double a = fabs(load_value(frag, dtype, k - start));\n        int64_t br = (i - r0) * nbr + j / 32;",
        "    for (int64_t k = start + 1; k < start + len; ++k) {\n        int64_t i = k / cols, j = k % cols;\n        double a = fabs(load_value(frag, dtype, k - start));\n        int64_t br = (i - r0) * nbr + j / 32;"),
    "rowwise data scaled by the columnwise scale": (
        "out_r[o] = oracle_quantize(y, scale_r[i * ld_sr + j / 32]);",
        "out_r[o] = oracle_quantize(y, scale_c ? scale_c[(i / 32) * ld_sc + j] : scale_r[i * ld_sr + j / 32]);"),
    "untouched row blocks overwritten": (
        "            if (hit_r[(i - r0) * nbr + b])\n                store_value(amax_r, dtype,",
        "            if (1)\n                store_value(amax_r, dtype,"),
    "nvfp4 untouched row blocks overwritten": (
        "            if (hit_r[(i - r0) * nbr + b])\n                store_value(amax_r, ORACLE_F32,",
        "            if (1)\n                store_value(amax_r, ORACLE_F32,"),
    "NaN not propagated by the reduction": (
        "            if (isnan(a) || isnan(m)) m = NAN;", "            if (isnan(m)) m = NAN;"),
    "GEMM layout with row fields swapped": (
        "(rr % 32) * 16 + (rr / 32) * 4 + cc", "(rr / 32) * 16 + (rr % 32) * 4 + cc"),
    "fp16 overflow threshold off by one unit": (
        "if (r > 65504.0) r = INFINITY;", "if (r >= 65504.0) r = INFINITY;"),
    "fp16 ties away from zero": (
        "    double r = nearbyint(a / quantum) * quantum;\n    if (r > 65504.0)",
        "    double r = round(a / quantum) * quantum;\n    if (r > 65504.0)"),
    "fp16 subnormal threshold off by one": (
        "if (p < -14) p = -14;", "if (p < -15) p = -15;"),
    "e4m3 subnormal spacing off by one": (
        "int p = (a < ldexp(1.0, -6)) ? -6 : floor_log2(a);",
        "int p = (a < ldexp(1.0, -7)) ? -7 : floor_log2(a);"),
    "e4m3 decode exponent bias off by one": (
        "else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    "infinite amax not mapped to the NaN scale": (
        "if (isnan(amax) || isinf(amax)) return 0xFF;", "if (isnan(amax)) return 0xFF;"),
    "NaN scale byte not special-cased in the cast": (
        "if (s == 0xFF) return 0x7F;", "if (s == 0xFF) return 0x00;"),
    "out_offset ignored by the cast": (
        "int64_t o = out_offset + (k - start);", "int64_t o = (k - start);"),
    "columnwise data scaled by the column's row-block scale index": (
        "scale_c[(i / 32) * ld_sc + j]);", "scale_c[(i / 32) * ld_sc + j / 32 * 32]);"),
    "NaN amax stored as the all-ones pattern": (
        "        bits = 0x7FC00000u;", "        bits = 0x7FFFFFFFu;"),
    "scale update with the leading dimensions swapped": (
        "scale[r * ld_s + c] = oracle_e8m0_from_amax(load_value(amax, dtype, r * ld_a + c));",
        "scale[r * ld_a + c] = oracle_e8m0_from_amax(load_value(amax, dtype, r * ld_s + c));"),
    "e2m1 ties away from zero": (
        "    double r = nearbyint(a / quantum) * quantum;\n    if (r > 6.0)",
        "    double r = round(a / quantum) * quantum;\n    if (r > 6.0)"),
    "e2m1 saturates to the wrong code": (
        "    if (r > 6.0) r = 6.0;", "    if (r > 6.0) r = 4.0;"),
    "nvfp4 tensor scale with 448 * 8": (
        "float s = 2688.0f / g;", "float s = 3584.0f / g;"),
    "nvfp4 zero tensor amax gives scale 0": (
        "if (g == 0.0f) return 1.0f;", "if (g == 0.0f) return 0.0f;"),
    "nvfp4 block scale divides by 4": (
        "float t = amax / 6.0f;", "float t = amax / 4.0f;"),
    "nvfp4 multiplier inverted": (
        "return s_enc / d;", "return d / s_enc;"),
    "nvfp4 row blocks of 32": (
        "int64_t br = (i - r0) * nbr + j / 16;", "int64_t br = (i - r0) * nbr + j / 32;"),
    "nvfp4 column blocks of 32 rows": (
        "int64_t bc = (i / 16 - c0) * cols + j;", "int64_t bc = (i / 32 - c0 / 2) * cols + j;"),
    "nvfp4 nibbles swapped": (
        "if (p % 2 == 0) *b", "if (p % 2 != 0) *b"),
    "nvfp4 cast skips the BF16 rounding": (
        "float y = (float)((dtype == ORACLE_F32) ? oracle_bf16_round((float)x) : x);",
        "float y = (float)x;"),
    "nvfp4 tensor amax misses the first element": (
        "        if (isnan(a) || isnan(tmax)) tmax = NAN;\n        else if (a > tmax) tmax = a;",
        "        if (k > start) { if (isnan(a) || isnan(tmax)) tmax = NAN;\n        else if (a > tmax) tmax = a; }"),
    "amax column index shifted by one": (
        "        int64_t i = k / cols, j = k % cols;\n        double a = fabs(load_value(frag, dtype, k - start));\n        int64_t br = (i - r0) * nbr + j / 32;",
        "        int64_t i = k / cols, j = (k + 1) % cols;\n        double a = fabs(load_value(frag, dtype, k - start));\n        int64_t br = (i - r0) * nbr + j / 32;"),
}


def _pin_calls():
    """(name, function, kwargs) for every pin that takes the oracle module, once per
    parameter set of parametrized pins."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        params = list(inspect.signature(fn).parameters)
        if not name.startswith("test_") or not params or params[0] != "oracle_mod":
            continue
        sets = [{}]
        for mark in getattr(fn, "pytestmark", []):
            if mark.name == "parametrize":
                argnames, argvalues = mark.args[0], mark.args[1]
                names = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
                values = [v if len(names) > 1 else (v,) for v in argvalues]
                sets = [dict(kw, **dict(zip(names, v))) for kw in sets for v in values]
        calls += [(name, fn, kw) for kw in sets]
    return calls


def _mutant(tmp_path, label, find, replace):
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(find) == 1, f"mutation site for {label!r} must occur exactly once"
    d = tmp_path / label.replace(" ", "_")
    d.mkdir()
    (d / "mxfp8_oracle.c").write_text(src.replace(find, replace))
    spec = importlib.util.spec_from_file_location("oracle_mutant_" + d.name, ORACLE_INIT)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "mxfp8_oracle.c")
    mod._LIB_PATH = str(d / "liboracle.so")
    mod._lib = None
    mod.build(force=True)
    return mod


@pytest.mark.parametrize("label", sorted(MUTATIONS))
def test_pins_kill_mutant(tmp_path, label):
    find, replace = MUTATIONS[label]
    mod = _mutant(tmp_path, label, find, replace)
    for name, fn, kwargs in _pin_calls():
        try:
            fn(mod, **kwargs)
        except AssertionError:
            return  # killed
    pytest.fail(f"no pin fails for the mutant: {label}")
