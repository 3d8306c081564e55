"""The forward kernel's division by launch constants (csrc/fast_div.h).

The unit decode of the persistent forward kernel divides unit indices by
launch constants (key ranges, m-blocks, heads, GQA group) with a
multiply-high and a shift (Granlund and Montgomery, "Division by invariant
integers using multiplication", 1994).  The header's host form is the same
arithmetic as its device form (``__umulhi`` is the high word of the 64-bit
product); this test compiles it with the host compiler and compares every
quotient with exact integer division over the whole range the kernel uses
(0 <= x < 2^31), densely near zero and at multiples of the divisor, and at
random points.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "attention_attn_fwd_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "fast_div.h"
int main() {
  using attn::FastDiv;
  long long bad = 0, n = 0;
  unsigned long long st = 88172645463325252ull;
  auto rnd = [&]() {
    st ^= st << 13; st ^= st >> 7; st ^= st << 17;
    return static_cast<int>(st & 0x7fffffff);
  };
  auto check = [&](int x, const FastDiv& f) {
    ++n;
    if (attn::fast_div(x, f) != x / f.d) {
      if (bad < 5) std::printf("x=%d d=%d got %d\n", x, f.d, attn::fast_div(x, f));
      ++bad;
    }
  };
  const int big[] = {65535, 65536, 65537, 1 << 20, (1 << 20) + 1, 123456789,
                     (1 << 30) - 1, 1 << 30, (1 << 30) + 1, 0x7fffffff};
  for (int d = 1; d <= 3000; ++d) {
    const FastDiv f = attn::make_fast_div(d);
    for (int x = 0; x < 5000; ++x) check(x, f);
    for (int i = 0; i < 500; ++i) check(rnd(), f);
    for (long long k = 1; k * d <= 0x7fffffffLL && k < 2000; ++k) {
      check(static_cast<int>(k * d), f);
      check(static_cast<int>(k * d - 1), f);
    }
    check(0x7fffffff, f);
    check(0x7fffffff - 0x7fffffff % d, f);
  }
  for (int d : big) {
    const FastDiv f = attn::make_fast_div(d);
    for (int i = 0; i < 200000; ++i) check(rnd(), f);
    for (long long k = 0; k * d <= 0x7fffffffLL && k < 5000; ++k) {
      check(static_cast<int>(k * d), f);
      if (k > 0) check(static_cast<int>(k * d - 1), f);
    }
    check(0x7fffffff, f);
  }
  std::printf("%lld checked, %lld wrong\n", n, bad);
  return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_fast_div_matches_integer_division(tmp_path):
    src = tmp_path / "fast_div_check.cpp"
    exe = tmp_path / "fast_div_check"
    src.write_text(DRIVER)
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert " 0 wrong" in out.stdout
