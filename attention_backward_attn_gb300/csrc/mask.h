// Key-mask arithmetic shared by the host (validation, tile classes) and the
// kernels. Plain C++ apart from the __host__ __device__ qualifiers, so that
// host-only code (and host tests) can include it without the CUDA compiler.
#pragma once

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

// live(i, j) = j < sink || (i - wl <= j <= i + wr); negative bound = unbounded
// ("22_sink_tokens_fmha.py" mask builders, top-left aligned).
// Key mask over (query i, key j): live when j < sink or -wl <= j - i <= wr.
// The bounds are relative to the diagonal j = i; kMaskUnbounded leaves that
// side open. They may be negative: a bottom-right aligned mask is a top-left
// one with both bounds shifted by Sk - Sq. Bounds are clamped to
// [-kMaskMaxBound, kMaskMaxBound] and lengths to kMaxMaskedLen, so i +- bound
// stays inside int.
constexpr int kMaskUnbounded = 1 << 29;
constexpr int kMaskMaxBound = 1 << 28;
constexpr int kMaxMaskedLen = 1 << 28;
struct MaskSpec {
  int wl;
  int wr;
  int sink;
};

// The bounds of a mask whose diagonal is moved by off keys (bottom-right
// alignment of a top-left mask: off = Sk - Sq); open sides stay open.
ATTN_HD MaskSpec mask_aligned(MaskSpec m, int off) {
  if (m.wl != kMaskUnbounded) m.wl -= off;
  if (m.wr != kMaskUnbounded) m.wr += off;
  return m;
}

ATTN_HD bool mask_live(const MaskSpec& m, int i, int j) {
  if (j < m.sink) return true;
  return j >= i - m.wl && j <= i + m.wr;
}

// Non-sink key range [lo, hi] (inclusive, clipped to [0, n); empty when
// lo > hi) live for row i.
ATTN_HD void mask_row_range(const MaskSpec& m, int i, int n, int* lo, int* hi) {
  const int a = i - m.wl, b = i + m.wr;
  *lo = a < 0 ? 0 : a;
  *hi = b > n - 1 ? n - 1 : b;
}

// Non-sink query range [lo, hi] live for key j (j >= sink), clipped to [0, n).
ATTN_HD void mask_col_range(const MaskSpec& m, int j, int n, int* lo, int* hi) {
  const int a = j - m.wr, b = j + m.wl;
  *lo = a < 0 ? 0 : a;
  *hi = b > n - 1 ? n - 1 : b;
}

// Tile classification over rows [m0, m1) x keys [n0, n1) for the same mask:
// tile_any = at least one live entry, tile_full = every entry live.
ATTN_HD bool tile_any(const MaskSpec& m, int m0, int m1, int n0, int n1) {
  if (m0 >= m1 || n0 >= n1) return false;
  if (n0 < m.sink) return true;
  const int dmax = (n1 - 1) - m0;  // largest j - i in the tile
  const int dmin = n0 - (m1 - 1);  // smallest j - i in the tile
  return dmax >= -m.wl && dmin <= m.wr;
}

ATTN_HD bool tile_full(const MaskSpec& m, int m0, int m1, int n0, int n1) {
  const int a = n0 > m.sink ? n0 : m.sink;  // first column not covered by the sinks
  if (a >= n1) return true;
  const int dmax = (n1 - 1) - m0;
  const int dmin = a - (m1 - 1);
  return dmin >= -m.wl && dmax <= m.wr;
}

// Live tiles without a scan (the same sets tile_any gives, on tiles clipped
// to the lengths sq x sk; tile sizes tq x tk).
// Query tiles of the key tile at n0: [*lo, *hi] (empty when *lo > *hi). The
// rows live for some key of [n0, n1) form one interval: all rows when the
// tile holds a sink key, else [n0 - wr, n1 - 1 + wl].
ATTN_HD void live_query_tiles(const MaskSpec& m, int sq, int sk, int tq, int tk, int n0, int* lo,
                              int* hi) {
  const int n1 = n0 + tk < sk ? n0 + tk : sk;
  if (sq <= 0 || n0 >= n1) {
    *lo = 1;
    *hi = 0;
    return;
  }
  int a = 0, b = sq - 1;
  if (n0 >= m.sink) {
    a = n0 - m.wr;
    b = n1 - 1 + m.wl;
    a = a < 0 ? 0 : a;
    b = b > sq - 1 ? sq - 1 : b;
  }
  if (a > b) {
    *lo = 1;
    *hi = 0;
  } else {
    *lo = a / tq;
    *hi = b / tq;
  }
}

// Key tiles of the query tile at m0: the tiles holding a sink key,
// [0, *s_end), then the window tiles [*w_lo, *w_hi] (the keys live for some
// row of [m0, m1) form [m0 - wl, m1 - 1 + wr]); the two may overlap.
ATTN_HD void live_key_tiles(const MaskSpec& m, int sq, int sk, int tq, int tk, int m0, int* s_end,
                            int* w_lo, int* w_hi) {
  const int m1 = m0 + tq < sq ? m0 + tq : sq;
  const int ns = m.sink < sk ? m.sink : sk;
  *s_end = ns > 0 ? (ns + tk - 1) / tk : 0;
  int a = m0 - m.wl, b = m1 - 1 + m.wr;
  a = a < 0 ? 0 : a;
  b = b > sk - 1 ? sk - 1 : b;
  if (m0 >= m1 || a > b) {
    *w_lo = 1;
    *w_hi = 0;
    if (m0 >= m1) *s_end = 0;
  } else {
    *w_lo = a / tk;
    *w_hi = b / tk;
  }
}

}  // namespace attn
