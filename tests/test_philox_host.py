"""The library's dropout generator compiled as host code and checked against the oracle's.

`csrc/fa_philox.cuh` holds Philox4x32-10 twice over: the plain ten rounds, and the form the
forward kernel uses, in which the products of rounds 1-2 that depend only on the words fixed
for a thread (counter words x1-x3 and the key) are formed once (`prefix_x0`) and each call
runs the rest (`run_x0`).  Both must give exactly the generator of Salmon et al. (SC 2011)
that `oracle/dropout.py` writes out independently.  The header's functions are host-callable;
this test builds a small host program around them with nvcc (no GPU needed) and compares its
output word for word with the oracle on seeded inputs and on edge values.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import dropout as odrop

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_28_gb300", "csrc")
INC = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <cstdio>
#include "fa_philox.cuh"
int main() {
  unsigned v[6];
  while (std::scanf("%u %u %u %u %u %u", &v[0], &v[1], &v[2], &v[3], &v[4], &v[5]) == 6) {
    const fa::philox::Words a = fa::philox::philox4x32_10(v[0], v[1], v[2], v[3], v[4], v[5]);
    const fa::philox::PrefixX0 s = fa::philox::prefix_x0(v[1], v[2], v[3], v[4], v[5]);
    const fa::philox::Words b = fa::philox::run_x0(s, v[0]);
    std::printf("%u %u %u %u %u %u %u %u\n", a.w[0], a.w[1], a.w[2], a.w[3], b.w[0], b.w[1],
                b.w[2], b.w[3]);
  }
  return 0;
}
"""


def _inputs():
    rng = np.random.default_rng(20261203)
    rows = [[0] * 6, [0xFFFFFFFF] * 6, [1, 2, 3, 4, 5, 6]]
    rows += rng.integers(0, 2**32, size=(200, 6), dtype=np.uint64).tolist()
    # the kernels' shapes: small key-chunk and row-pair words, head index, zero offset
    for t in range(40):
        rows.append([4 * t + (t % 4), 8 * (t // 2) + t % 8, t % 32, 0, 0x1234ABCD, 0x9F00])
    return rows


def test_generator_and_prefix_form_match_the_oracle(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "philox_host.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "philox_host"
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                    "-I", INC, str(src), "-o", str(exe)], check=True, capture_output=True)
    rows = _inputs()
    stdin = "\n".join(" ".join(str(int(x)) for x in r) for r in rows) + "\n"
    out = subprocess.run([str(exe)], input=stdin, capture_output=True, text=True, check=True)
    got = np.array([[int(x) for x in line.split()] for line in out.stdout.splitlines()],
                   dtype=np.uint64)
    assert got.shape == (len(rows), 8)
    ref = np.stack([np.stack(odrop.philox4x32(tuple(np.uint64(x) for x in r[:4]), (r[4], r[5])))
                    for r in rows]).reshape(len(rows), 4)
    np.testing.assert_array_equal(got[:, :4], ref)   # plain rounds
    np.testing.assert_array_equal(got[:, 4:], ref)   # prefix form
