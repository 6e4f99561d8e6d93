// Host check of the tile walk the dense tensor-core kernel uses: the live
// query-tile range of every key tile (live_query_tiles) and the live key
// tiles of every query tile (live_key_tiles) must be exactly the tiles that
// tile_any marks live, over many masks, lengths and tile sizes.
// Prints "ok <cases>" and exits 0, or prints the first mismatch and exits 1.
#include <cstdio>
#include <vector>

#include "mask.h"

using attn::MaskSpec;

static MaskSpec spec(int wl, int wr, int sink) {
  MaskSpec m;
  m.wl = wl;
  m.wr = wr;
  m.sink = sink;
  return m;
}

int main() {
  const int U = attn::kMaskUnbounded;
  std::vector<MaskSpec> masks = {spec(U, U, 0),   spec(U, 0, 0),    spec(U, 0, 4),
                                 spec(127, 0, 4), spec(40, 25, 3),  spec(10, 0, 0),
                                 spec(0, 0, 0),   spec(3, 200, 0),  spec(U, -256, 0),
                                 spec(-100, U, 2), spec(31, -5, 70), spec(U, 130, 300),
                                 spec(-300, 100, 0), spec(5, 5, 1000)};
  const int lens[] = {1, 5, 64, 100, 128, 129, 200, 256, 300, 384, 700};
  const int tiles[][2] = {{128, 128}, {64, 32}, {16, 8}};
  long cases = 0;
  for (const MaskSpec& m : masks)
    for (int sq : lens)
      for (int sk : lens)
        for (const auto& t : tiles) {
          const int tq = t[0], tk = t[1];
          const int nmt = (sq + tq - 1) / tq, nnt = (sk + tk - 1) / tk;
          for (int nt = 0; nt < nnt; ++nt) {
            int lo, hi;
            attn::live_query_tiles(m, sq, sk, tq, tk, nt * tk, &lo, &hi);
            for (int mt = 0; mt < nmt; ++mt) {
              const int m0 = mt * tq, n0 = nt * tk;
              const bool want = attn::tile_any(m, m0, m0 + tq < sq ? m0 + tq : sq, n0,
                                               n0 + tk < sk ? n0 + tk : sk);
              const bool got = lo <= mt && mt <= hi;
              ++cases;
              if (want != got) {
                std::printf("query tiles: wl=%d wr=%d sink=%d sq=%d sk=%d tile=%dx%d nt=%d mt=%d"
                            " want=%d got=%d\n", m.wl, m.wr, m.sink, sq, sk, tq, tk, nt, mt,
                            want, got);
                return 1;
              }
            }
          }
          for (int mt = 0; mt < nmt; ++mt) {
            int s_end, w_lo, w_hi;
            attn::live_key_tiles(m, sq, sk, tq, tk, mt * tq, &s_end, &w_lo, &w_hi);
            for (int nt = 0; nt < nnt; ++nt) {
              const int m0 = mt * tq, n0 = nt * tk;
              const bool want = attn::tile_any(m, m0, m0 + tq < sq ? m0 + tq : sq, n0,
                                               n0 + tk < sk ? n0 + tk : sk);
              const bool got = nt < s_end || (w_lo <= nt && nt <= w_hi);
              ++cases;
              if (want != got) {
                std::printf("key tiles: wl=%d wr=%d sink=%d sq=%d sk=%d tile=%dx%d mt=%d nt=%d"
                            " want=%d got=%d\n", m.wl, m.wr, m.sink, sq, sk, tq, tk, mt, nt,
                            want, got);
                return 1;
              }
            }
          }
        }
  std::printf("ok %ld\n", cases);
  return 0;
}
