"""The kernels' fixed-divisor quotient (FastDiv, Granlund and Montgomery's
division by invariant integers) against true division, on the CPU.

A host program built with nvcc includes the library's header, takes the
magic numbers from its make_fastdiv, and evaluates the device formula
(umulhi(n, m) + n) >> l with the same 32-bit wrap-around.  It checks:
- every divisor 1..4096;
- 20000 random divisors below 2^31;
- numerators at 0, near each multiple boundary, at 2^31 - 1, and at random.
The claim under test is floor(n / d) exactly for n, d < 2^31.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_48_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <random>
#include "sv_pass_common.cuh"

static unsigned umulhi_host(unsigned a, unsigned b) {
  return (unsigned)(((unsigned long long)a * b) >> 32);
}

int main() {
  std::mt19937_64 rng(7);
  long long checks = 0, bad = 0;
  auto check = [&](unsigned n, unsigned d) {
    const sv::FastDiv f = sv::make_fastdiv(d);
    const unsigned sum = umulhi_host(n, f.m) + n;  // 32-bit, as on the device
    const unsigned q = sum >> f.l;
    ++checks;
    if (q != n / d) {
      if (bad < 5) std::printf("bad n=%u d=%u got %u want %u\n", n, d, q, n / d);
      ++bad;
    }
  };
  const unsigned top = 0x7fffffffu;
  auto numerators = [&](unsigned d) {
    check(0, d);
    check(top, d);
    for (unsigned k : {1u, 2u, 3u, 1000u, top / d - 1, top / d}) {
      const unsigned long long base = (unsigned long long)k * d;
      for (long long o = -2; o <= 2; ++o) {
        const long long n = (long long)base + o;
        if (n >= 0 && n <= (long long)top) check((unsigned)n, d);
      }
    }
    for (int i = 0; i < 64; ++i) check((unsigned)(rng() % (top + 1ull)), d);
  };
  for (unsigned d = 1; d <= 4096; ++d) numerators(d);
  for (int i = 0; i < 20000; ++i) numerators((unsigned)(rng() % top) + 1u);
  std::printf("checks %lld bad %lld\n", checks, bad);
  return bad != 0;
}
"""


def test_fastdiv_is_exact_below_2_31(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is not available")
    src = tmp_path / "fastdiv_check.cu"
    exe = tmp_path / "fastdiv_check"
    src.write_text(PROGRAM)
    r = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"),
                        "-I", CSRC, str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout
    assert "bad 0" in out.stdout
