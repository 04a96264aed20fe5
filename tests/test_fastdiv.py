"""The row geometry divides by q_len and by heads with a multiply-high (Granlund and
Montgomery, "Division by invariant integers using multiplication", Figure 4.1).  The host code
that forms the constants and the quotient function are compiled here with the host compiler and
checked against C's own unsigned division: every divisor up to 4096, the divisors next to
powers of two, the largest 31-bit one and random ones, each at edge and random dividends.  No GPU
is needed; the kernels call the same function."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "deterministic_attention_softmax_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdint>
#include <cstdio>
#include <vector>
#include "fos_internal.h"
static uint64_t state = 0x9e3779b97f4a7c15ull;
static uint32_t next() {  // splitmix64
  uint64_t z = (state += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return (uint32_t)(z ^ (z >> 31));
}
int main() {
  std::vector<uint32_t> ds;
  for (uint32_t d = 1; d <= 4096; ++d) ds.push_back(d);
  for (int k = 1; k < 31; ++k) {
    ds.push_back((1u << k) - 1); ds.push_back(1u << k); ds.push_back((1u << k) + 1);
  }
  ds.push_back(2147483647u);
  for (int i = 0; i < 4000; ++i) ds.push_back(next() % 2147483647u + 1);
  long bad = 0, n = 0;
  for (uint32_t d : ds) {
    const fos::FastDiv f = fos::make_fastdiv(d);
    const uint32_t edge[] = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 2 * d, 2147483647u, 4294967295u};
    for (uint32_t x : edge) { ++n; if (fos::fast_div(x, f) != x / d) ++bad; }
    for (int j = 0; j < 64; ++j) { const uint32_t x = next(); ++n; if (fos::fast_div(x, f) != x / d) ++bad; }
  }
  printf("%ld %ld\n", n, bad);
  return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                    reason="needs g++ and the CUDA headers")
def test_multiply_high_division_is_exact(tmp_path):
    src = tmp_path / "fastdiv.cpp"
    exe = tmp_path / "fastdiv"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, "-I", CUDA_INC, str(src), "-o",
                    str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    checks, bad = map(int, out.stdout.split())
    assert out.returncode == 0 and bad == 0 and checks > 500_000
