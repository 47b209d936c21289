"""The CTA order of the forward, dQ and dK/dV launches (work_unit in
csrc/kernels.h), checked on the host: a small program compiled with nvcc
calls the same inline function for every CTA of a launch.

For each (levels, heads, tail) the map must be a bijection onto the (head,
level) units; the CTAs before the tail run head by head with level 0 (the
heaviest causal unit) first; the tail runs its heads level by level, so the
launch's last CTAs are the highest levels (the lightest units) of the last
heads.  No GPU is needed."""
import itertools
import os
import shutil
import subprocess

import pytest

from scaled_dot_product_08_gb300.build import CSRC, nvcc

CASES = [(nlev, nheads, tail)
         for nlev, nheads in itertools.product([1, 2, 8, 16, 32], [1, 3, 16, 128])
         for tail in sorted({1, 2, 15, 16, 29, nheads}) if tail <= nheads]

PROGRAM = r"""
#include <cstdio>
#include "kernels.h"
int main() {
  int nlev, nheads, tail;
  while (std::scanf("%d %d %d", &nlev, &nheads, &tail) == 3) {
    for (int cta = 0; cta < nlev * nheads; ++cta) {
      int h = -1, l = -1;
      sdpa::work_unit(cta, nlev, nheads, tail, h, l);
      std::printf("%d %d\n", h, l);
    }
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def order_bin(tmp_path_factory):
    cc = nvcc()
    if not shutil.which(cc) and not os.path.exists(cc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("order")
    src, exe = d / "order.cu", d / "order"
    src.write_text(PROGRAM)
    r = subprocess.run([cc, "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_work_unit_order(order_bin):
    inp = "".join(f"{a} {b} {c}\n" for a, b, c in CASES)
    out = subprocess.run([str(order_bin)], input=inp, capture_output=True, text=True, check=True).stdout.split("\n")
    pos = 0
    for nlev, nheads, tail in CASES:
        units = [tuple(map(int, out[pos + c].split())) for c in range(nlev * nheads)]
        pos += nlev * nheads
        case = f"levels {nlev}, heads {nheads}, tail {tail}"
        assert sorted(units) == [(h, l) for h in range(nheads) for l in range(nlev)], case
        lead = (nheads - tail) * nlev
        assert units[:lead] == [(h, l) for h in range(nheads - tail) for l in range(nlev)], case
        assert units[lead:] == [(h, l) for l in range(nlev) for h in range(nheads - tail, nheads)], case
