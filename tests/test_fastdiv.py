"""CPU check of the launch-time divider (FastDiv in qmv_layout.h) that the
matvec kernel uses instead of integer division: compiled with the host
compiler, its quotient and remainder equal integer division for every
dividend and divisor range the kernel uses (dividends below 2^23, divisors
below 2^17), exhaustively over the divisors 1..4096 and sampled above."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r'''
#include <cstdio>
#include <cstdint>
#include "qmv_layout.h"
using namespace qmv;
static int check(uint32_t d, uint32_t n) {
  const FastDiv f = make_fastdiv(d);
  return fast_div(n, f) != n / d || fast_mod(n, f) != n % d;
}
int main() {
  long bad = 0;
  for (uint32_t d = 1; d <= 4096; ++d) {
    for (uint32_t n = 0; n < 70000; ++n) bad += check(d, n);
    for (uint32_t n = (1u << 23) - 70000; n < (1u << 23); ++n) bad += check(d, n);
    for (uint32_t k = 1; k < 2048 && k * d < (1u << 23); ++k) { bad += check(d, k * d - 1); bad += check(d, k * d); }
  }
  uint64_t s = 88172645463325252ull;
  for (long i = 0; i < 20000000; ++i) {
    s ^= s << 13; s ^= s >> 7; s ^= s << 17;
    const uint32_t d = 1 + (uint32_t)(s % ((1u << 17) - 1));
    const uint32_t n = (uint32_t)((s >> 20) % (1u << 23));
    bad += check(d, n);
  }
  printf("%ld\n", bad);
  return 0;
}
'''


def test_fastdiv_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "fd.cpp"
    src.write_text(SRC)
    exe = tmp_path / "fd"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "bit_quantized_moe_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.strip()
    assert out == "0"
