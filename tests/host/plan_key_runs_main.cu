// Host-only harness: prints the key runs that plan_key_runs (shared by the
// host planner and the graph-mode kernels) produces for a grid of streaming
// calls, one line per call: c W R Lc has_sink use_sink kcur nseg total then
// (src row0 nrows tile0) per segment.  No device code runs.
#include <cstdio>

#include "../../streaming_attention_block_gb300/csrc/sab_internal.h"

int main() {
  const int lcs[] = {64, 100, 128, 405};
  for (int Lc : lcs)
    for (int R = 1; R <= 6; ++R)
      for (int has_sink = 0; has_sink <= 1; ++has_sink)
        for (int use_sink = 0; use_sink <= has_sink; ++use_sink)
          for (int kcur = 0; kcur <= 1; ++kcur)
            for (int W = 0; W <= (kcur ? R : R - 1); ++W)
              for (long long c = 0; c <= 3 * R + 2; ++c) {
                sab::KeyPlan kp;
                sab::plan_key_runs(c, W, R, Lc, has_sink, use_sink, kcur, kp);
                std::printf("%lld %d %d %d %d %d %d %d %d", c, W, R, Lc, has_sink, use_sink, kcur, kp.nseg,
                            kp.total_tiles);
                for (int i = 0; i < kp.nseg; ++i)
                  std::printf(" %d %d %d %d", kp.seg[i].src, kp.seg[i].row0, kp.seg[i].nrows, kp.seg[i].tile0);
                std::printf("\n");
              }
  return 0;
}
