// Host check of the kernels' grid order (grid_pos, l2_group in kernels.cuh):
// every (tile, split, problem) is visited exactly once for any group size,
// and group == B*H gives the plain (tile, split, problem) order.  Built with
// nvcc as host code and run by tests/test_grid_order.py; exits non-zero on a
// mismatch.
#include <cstdio>
#include <vector>
#include "kernels.cuh"

using exattn::GridPos;
using exattn::grid_pos;
using exattn::l2_group;

int main() {
  long long cases = 0, bad = 0;
  for (int BH = 1; BH <= 37; ++BH)
    for (int T = 1; T <= 9; ++T)
      for (int S = 1; S <= 4; ++S)
        for (int G = 1; G <= BH; ++G) {
          std::vector<int> seen(static_cast<size_t>(BH) * T * S, 0);
          for (int b = 0; b < BH * T * S; ++b) {
            const GridPos p = grid_pos(b, BH, T, S, G);
            if (p.tile < 0 || p.tile >= T || p.sub < 0 || p.sub >= S || p.bh < 0 || p.bh >= BH) {
              ++bad;
              continue;
            }
            // Problems of one group only: bh // G is the group index.
            if (p.bh / G != b / (G * T * S) && b < (BH / G) * G * T * S) ++bad;
            ++seen[(static_cast<size_t>(p.bh) * T + p.tile) * S + p.sub];
            if (G == BH && (p.tile != b / (BH * S) || p.sub != b % (BH * S) / BH || p.bh != b % BH)) ++bad;
          }
          for (int x : seen) bad += (x != 1);
          ++cases;
        }
  // Group sizes: 64 MB of re-read operand per group, at least one problem, at most B*H.
  if (l2_group(4ll << 20, 16) != 16 || l2_group(1ll << 20, 128) != 64 || l2_group(64ll << 20, 1) != 1 ||
      l2_group(1ll << 30, 8) != 1 || l2_group(0, 5) != 5 || l2_group(1ll << 20, 128, 32ll << 20) != 32)
    ++bad;
  std::printf("%lld cases, %lld mismatches\n", cases, bad);
  return bad != 0;
}
