"""The NVFP4 scale update divides each block amax by 6 with Markstein's method (a product
with RN(1/6), an exact FMA remainder, one corrective FMA) instead of a full IEEE division,
and claims the two agree for every float from 2^-124 up to the largest float.  This test
checks that claim on the host, input by input, against the correctly rounded quotient:
the quotient is computed in double and rounded to float, which gives the correctly rounded
float quotient because 53 >= 2 * 24 + 2 (double rounding is innocuous for division;
S. A. Figueroa, "When is double rounding innocuous?", SIGNUM Newsletter 30(3), 1995).

For normal inputs whose remainder stays normal, scaling a by 2 scales q0, the remainder
and q by 2 exactly, so the result depends on the mantissa alone; the default run covers
every mantissa of the binades above the boundary (2^-125 .. 2^-122), of 2^0 and of the top
binade.  MXFP8_DIV6_FULL=1 runs every float from 2^-125 to the largest (minutes).
"""
import os
import subprocess

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
static float f(uint32_t b) { float x; memcpy(&x, &b, 4); return x; }
static uint32_t bits(float x) { uint32_t b; memcpy(&b, &x, 4); return b; }
int main(int argc, char** argv) {
  const float inv6 = 0x1.555556p-3f;  /* RN(1/6) */
  uint64_t fails = 0, n = 0;
  for (int k = 1; k + 1 < argc; k += 2) {
    const uint32_t lo = (uint32_t)strtoul(argv[k], 0, 0), hi = (uint32_t)strtoul(argv[k + 1], 0, 0);
    for (uint32_t b = lo; b < hi; ++b, ++n) {
      const float a = f(b);
      const float q0 = a * inv6;
      const float r = fmaf(-6.0f, q0, a);
      const float q = fmaf(r, inv6, q0);
      if (bits(q) != bits((float)((double)a / 6.0))) ++fails;
    }
  }
  printf("%llu %llu\n", (unsigned long long)n, (unsigned long long)fails);
  return 0;
}
"""


def _run(tmp_path, ranges):
    src = tmp_path / "div6.c"
    exe = tmp_path / "div6"
    src.write_text(SRC)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-o", str(exe), str(src), "-lm"], check=True)
    args = [str(exe)] + [hex(v) for r in ranges for v in r]
    n, fails = map(int, subprocess.run(args, check=True, capture_output=True, text=True).stdout.split())
    return n, fails


def _binade(e):
    return ((e + 127) << 23, (e + 128) << 23)


def test_markstein_div6_equals_the_correctly_rounded_quotient(tmp_path):
    if os.environ.get("MXFP8_DIV6_FULL") == "1":
        ranges = [(0x01000000, 0x7F800000)]
    else:
        ranges = [_binade(e) for e in (-125, -124, -123, -122, 0, 127)]
    n, fails = _run(tmp_path, ranges)
    assert n == sum(b - a for a, b in ranges)
    assert fails == 0


def test_markstein_div6_fails_below_the_boundary(tmp_path):
    """Why the kernel falls back to the IEEE division under 2^-124: in the lowest binades
    the remainder is subnormal and the corrected quotient can be off."""
    _, fails = _run(tmp_path, [(1, 0x00800000)])
    assert fails > 0
