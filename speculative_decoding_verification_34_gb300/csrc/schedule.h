// Placement of the draw units in the verify grid (host and device; plain C++ otherwise, so that
// a host-only test can compile it).  Internal to the library, not part of the ABI.
#pragma once

#if defined(__CUDACC__)
#define SPEC_HD __host__ __device__
#else
#define SPEC_HD
#endif

namespace specverify {

// The sequence whose B units sit in group z of a launch of nb sequences (-1: none).  Groups
// 0..nb-1 hold the row units of sequence z and, delta groups behind them, the B units of the
// sequences from ndefer on.  After the last row unit come the B units of the first ndefer
// sequences, whose plans are long out: their draws keep HBM busy while the last sequences are
// decided.  Then those of the last delta sequences, which cannot sit delta groups behind (their
// plans come out only after their row units end); placed last, they find their plans out
// instead of holding block slots while they wait.
SPEC_HD inline int draw_group_seq(int z, int nb, int delta, int ndefer) {
  const int nl = delta < nb ? delta : nb;   // the last sequences
  if (z < nb) {
    const int bl = z - delta;
    return bl >= ndefer ? bl : -1;
  }
  const int j = z - nb;
  const int nd = ndefer < nb - nl ? ndefer : nb - nl;
  if (j < nd) return j;
  const int jl = j - nd;
  return jl < nl ? nb - nl + jl : -1;
}

// Groups in a launch of nb sequences: one per sequence, then the tail of draw-only groups.
SPEC_HD inline int draw_groups(int nb, int delta, int ndefer) {
  const int nl = delta < nb ? delta : nb;
  const int nd = ndefer < nb - nl ? ndefer : nb - nl;
  return nb + nl + nd;
}

}  // namespace specverify
