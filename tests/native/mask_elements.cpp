// Host dump of the element-wise key mask as the library's mask arithmetic
// (csrc/mask.h) states it, for comparison with the oracle's mask:
// reads lines "Sq Sk window_left window_right num_sink bottom_right" from
// stdin and, for each, writes three Sq x Sk planes of 0 / 1 bytes to stdout:
//   1. mask_live(i, j);
//   2. the row form the CUDA-core kernels use: j < sink, or j inside
//      mask_row_range(i);
//   3. the column form: j < sink (every row), or i inside mask_col_range(j).
// The descriptor is converted as the C ABI does it: a negative bound is
// unbounded, and bottom-right alignment shifts the window by Sk - Sq.
#include <cstdio>
#include <vector>

#include "mask.h"

int main() {
  int sq, sk, wl, wr, ns, br;
  while (std::scanf("%d %d %d %d %d %d", &sq, &sk, &wl, &wr, &ns, &br) == 6) {
    attn::MaskSpec m;
    m.wl = wl < 0 ? attn::kMaskUnbounded : wl;
    m.wr = wr < 0 ? attn::kMaskUnbounded : wr;
    m.sink = ns;
    m = attn::mask_aligned(m, br ? sk - sq : 0);
    std::vector<unsigned char> a((size_t)sq * sk), b((size_t)sq * sk), c((size_t)sq * sk, 0);
    for (int i = 0; i < sq; ++i) {
      int lo, hi;
      attn::mask_row_range(m, i, sk, &lo, &hi);
      for (int j = 0; j < sk; ++j) {
        a[(size_t)i * sk + j] = attn::mask_live(m, i, j) ? 1 : 0;
        b[(size_t)i * sk + j] = (j < m.sink || (j >= lo && j <= hi)) ? 1 : 0;
      }
    }
    for (int j = 0; j < sk; ++j) {
      int lo = 0, hi = sq - 1;
      if (j >= m.sink) attn::mask_col_range(m, j, sq, &lo, &hi);
      for (int i = lo; i <= hi; ++i) c[(size_t)i * sk + j] = 1;
    }
    std::fwrite(a.data(), 1, a.size(), stdout);
    std::fwrite(b.data(), 1, b.size(), stdout);
    std::fwrite(c.data(), 1, c.size(), stdout);
    std::fflush(stdout);
  }
  return 0;
}
