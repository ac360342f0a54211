"""The conv's multiply-shift division (conv_parts.cuh, FastDiv), compiled from
the library's own header for the host with nvcc and checked against integer
division: every divisor 1..4096 and a set of large ones, each against the
dividends that straddle its multiples (q*d - 1, q*d, q*d + d - 1) over the
whole domain n < 2^31 (quotients sampled densely at both ends) plus the
domain's ends."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "hashed_gram_embedding_engram_gb300", "csrc")

PROGRAM = r'''
#include <cstdio>
#include <cstdint>
#include "conv_parts.cuh"
using engram::cv::FastDiv;
using engram::cv::make_fastdiv;
static int check(uint32_t d, uint32_t n, const FastDiv& f) {
  if (n > 0x7FFFFFFFu) return 0;
  if (f.div(n) != n / d) { std::printf("FAIL d=%u n=%u got %u\n", d, n, f.div(n)); return 1; }
  return 0;
}
int main() {
  const uint32_t big[] = {4097u, 65535u, 65536u, 65537u, 1000003u, 16777216u, 16777217u, 0x40000000u,
                          0x7FFFFFFFu};
  uint32_t ds[4096 + sizeof(big) / 4];
  int nd = 0;
  for (uint32_t d = 1; d <= 4096; ++d) ds[nd++] = d;
  for (uint32_t b : big) ds[nd++] = b;
  long long checked = 0;
  int bad = 0;
  for (int i = 0; i < nd; ++i) {
    const uint32_t d = ds[i];
    const FastDiv f = make_fastdiv(d);
    const uint64_t qmax = 0x7FFFFFFFull / d;
    for (uint64_t q = 0; q <= qmax + 1; ) {
      const uint64_t n0 = q * d;
      const uint64_t cand[3] = {n0 ? n0 - 1 : 0, n0, n0 + d - 1};
      for (uint64_t n : cand) if (n <= 0x7FFFFFFFull) { bad += check(d, static_cast<uint32_t>(n), f); ++checked; }
      // every quotient near both ends, geometric steps in between
      q = (q < 4096 || q + 4096 > qmax) ? q + 1 : q + 1 + q / 64;
    }
    bad += check(d, 0x7FFFFFFFu, f);
    bad += check(d, 0x7FFFFFFEu, f);
    if (bad) break;
  }
  std::printf("checked %lld bad %d\n", checked, bad);
  return bad != 0;
}
'''


@pytest.mark.timeout(600)
def test_multiply_shift_division_is_exact(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "fastdiv_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    "-gencode", "arch=compute_103a,code=sm_103a", str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
