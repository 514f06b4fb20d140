"""Draw-unit placement of the verify grid (csrc/schedule.h), compiled on the host with g++.

The verify kernel's correctness needs every sequence's draw units placed exactly once per
launch; the order only matters for speed.  These checks run the library's own header.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_34_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "schedule.h"
using namespace specverify;
int main(int argc, char** argv) {
  if (argc == 5) {   // print the mapping of one launch: z -> sequence
    const int nb = atoi(argv[1]), delta = atoi(argv[2]), ndefer = atoi(argv[3]);
    (void)argv[4];
    const int G = draw_groups(nb, delta, ndefer);
    for (int z = 0; z < G; ++z) printf("%d\n", draw_group_seq(z, nb, delta, ndefer));
    return 0;
  }
  long checked = 0;
  for (int nb = 1; nb <= 300; nb += (nb < 80 ? 1 : 7))
    for (int delta = 0; delta <= nb + 3; delta += (delta < 40 ? 1 : 9))
      for (int ndefer = 0; ndefer <= nb + 5; ndefer += (ndefer < 40 ? 1 : 11)) {
        const int G = draw_groups(nb, delta, ndefer);
        std::vector<int> seen(nb, 0);
        for (int z = 0; z < G; ++z) {
          const int b = draw_group_seq(z, nb, delta, ndefer);
          if (b < -1 || b >= nb) { printf("FAIL range nb=%d delta=%d ndefer=%d z=%d b=%d\n", nb, delta, ndefer, z, b); return 1; }
          if (b >= 0 && z < nb && b > z) { printf("FAIL ahead nb=%d delta=%d ndefer=%d z=%d b=%d\n", nb, delta, ndefer, z, b); return 1; }
          if (b >= 0) ++seen[b];
        }
        for (int z = G; z < G + 3; ++z)
          if (draw_group_seq(z, nb, delta, ndefer) != -1) { printf("FAIL past end nb=%d\n", nb); return 1; }
        for (int b = 0; b < nb; ++b)
          if (seen[b] != 1) { printf("FAIL count nb=%d delta=%d ndefer=%d b=%d seen=%d\n", nb, delta, ndefer, b, seen[b]); return 1; }
        ++checked;
      }
  printf("ok %ld\n", checked);
  return 0;
}
"""


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("sched")
    src, exe = d / "sched.cpp", d / "sched"
    src.write_text(HARNESS)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return str(exe)


def test_every_sequence_drawn_exactly_once(harness):
    out = subprocess.run([harness], capture_output=True, text=True, check=True).stdout
    assert out.startswith("ok"), out




@pytest.mark.parametrize("nb,delta,ndefer", [(128, 36, 94), (1024, 36, 94), (5, 36, 94), (256, 20, 0)])
def test_launch_layout(harness, nb, delta, ndefer):
    out = subprocess.run([harness, str(nb), str(delta), str(ndefer), "x"], capture_output=True, text=True, check=True).stdout
    z2b = [int(x) for x in out.split()]
    nl = min(delta, nb)
    nd = min(ndefer, nb - nl)
    assert len(z2b) == nb + nl + nd
    # row groups: sequence z - delta draws there when it is not deferred
    for z in range(nb):
        bl = z - delta
        assert z2b[z] == (bl if bl >= ndefer else -1)
    # the tail: the first nd sequences in order, then the last nl in order
    assert z2b[nb:] == list(range(nd)) + list(range(nb - nl, nb))
