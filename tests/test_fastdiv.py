"""The multiply-shift division that maps work items to (batch, head, rows)
in the kernels (csrc/fastdiv.h), checked against integer division on the host.
The header compiles as plain C++ and runs the host branch of the same
arithmetic (a 64-bit product instead of __umulhi)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "tiled_attention_forward_fwd_gb300", "csrc")

CHECKER = r"""
#include <stdio.h>
#include <stdint.h>
#include "fastdiv.h"
using namespace attn;
static uint64_t rng = 0x9e3779b97f4a7c15ull;
static uint32_t next31() { rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17; return (uint32_t)(rng >> 33); }
static int check(uint32_t d, uint32_t n) {
  const FastDiv f = fastdiv_make(d);
  int q, r;
  fastdiv_divmod(f, (int)n, q, r);
  if ((uint32_t)q != n / d || (uint32_t)r != n % d || fastdiv_div(f, n) != n / d) {
    printf("FAIL d=%u n=%u got %d %d want %u %u\n", d, n, q, r, n / d, n % d);
    return 1;
  }
  return 0;
}
int main() {
  const uint32_t nmax = 0x7fffffffu;
  uint32_t big[] = {65521u, 65536u, 65537u, 1000003u, 1u << 20, (1u << 20) + 1, 16777213u,
                    (1u << 30) - 1, 1u << 30, (1u << 30) + 3, 2147483629u, nmax - 1, nmax};
  long fails = 0, n_checked = 0;
  for (uint32_t d = 1; d <= 4096 + 13; ++d) {
    const uint32_t dd = d <= 4096 ? d : big[d - 4097];
    for (uint32_t n = 0; n < 3000; ++n, ++n_checked) fails += check(dd, n);
    for (uint32_t k = 1; k < 200; ++k) {  // around multiples of d, up to the top of the range
      const uint64_t m = (uint64_t)dd * (uint64_t)(nmax / dd / k);
      for (int e = -1; e <= 1; ++e) {
        const int64_t n = (int64_t)m + e;
        if (n >= 0 && n <= nmax) { fails += check(dd, (uint32_t)n); ++n_checked; }
      }
    }
    for (int i = 0; i < 2000; ++i, ++n_checked) fails += check(dd, next31());
    fails += check(dd, nmax);
    if (fails > 20) break;
  }
  printf("checked %ld, failures %ld\n", n_checked, fails);
  return fails != 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "fastdiv_check.cpp"
    src.write_text(CHECKER)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures 0" in r.stdout
