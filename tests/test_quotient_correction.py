"""The quantiser's division-free quotient, checked exhaustively on the host.

quantize_codes_kernel forms w / s for FP16 w and s as y = RN(1/s), q0 = RN(w y),
r = fma(-q0, s, w), q1 = fma(r, y, q0) (Markstein's one-step correction) and relies on q1 being
the correctly rounded float32 quotient, so that rint(q1) matches the IEEE division the quantiser
is defined by (deep-dive article, "可复现的调用链": q = clamp(rint(w / s) + 8, 0, 15)).  The
quotient's rounding depends only on the two significands while no intermediate under- or
overflows, which holds for FP16 operands, so every pair of FP16 significands (1..2047 each) is
checked at several exponent offsets, in C with IEEE float32 arithmetic and fmaf."""
import shutil
import subprocess

import pytest

SOURCE = r"""
#include <math.h>
#include <stdio.h>
int main(void) {
  const int shifts[] = {0, -30, 25, -14, 7};
  long long bad = 0, n = 0;
  for (int si = 0; si < 5; ++si)
    for (int A = 1; A < 2048; ++A)
      for (int B = 1; B < 2048; ++B) {
        const float w = ldexpf((float)A, -10 + shifts[si]);
        const float s = ldexpf((float)B, -10);
        const float y = 1.0f / s;
        const float q0 = w * y;
        const float q1 = fmaf(fmaf(-q0, s, w), y, q0);
        ++n;
        if (q1 != w / s || -q1 != (-w) / s) ++bad;
      }
  printf("%lld %lld\n", n, bad);
  return 0;
}
"""


def test_corrected_quotient_is_correctly_rounded_for_all_fp16_significands(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "quot.c"
    src.write_text(SOURCE)
    exe = tmp_path / "quot"
    # no contraction: every product and sum above is one IEEE float32 operation
    subprocess.run([gcc, "-O2", "-ffp-contract=off", "-o", str(exe), str(src), "-lm"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    n, bad = int(out[0]), int(out[1])
    assert n == 5 * 2047 * 2047
    assert bad == 0
