// Host-side check of a two-level mask (STOF, 手法 / 2 段階ストレージ形式) held in host memory:
// everything the kernels rely on when they read an encoded mask, so that a mask assembled
// outside sta_encode_mask (or damaged on its way) can be rejected before any launch.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "sta.h"

namespace {

constexpr int kOT = 64;

inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Bits of the inner-tile words of outer tile (a, c) that lie inside the Lq x Lk mask:
// word 8p + q, bit 8r + cc is element (64a + 8p + r, 64c + 8q + cc).
void in_range_words(int64_t a, int64_t c, int Lq, int Lk, uint64_t* w) {
  for (int p = 0; p < 8; ++p)
    for (int q = 0; q < 8; ++q) {
      uint64_t m = 0;
      for (int r = 0; r < 8; ++r)
        for (int cc = 0; cc < 8; ++cc)
          if (64 * a + 8 * p + r < Lq && 64 * c + 8 * q + cc < Lk) m |= 1ull << (8 * r + cc);
      w[8 * p + q] = m;
    }
}

int popcount64(uint64_t x) {
  int n = 0;
  while (x) {
    x &= x - 1;
    ++n;
  }
  return n;
}

}  // namespace

extern "C" sta_status sta_validate_mask(const sta_bsr_mask* m, int* failed_check) {
  int dummy = 0;
  int& fail = failed_check ? *failed_check : dummy;
  fail = 0;
  auto bad = [&](int code) {
    fail = code;
    return STA_ERR_INVALID_ARG;
  };
  if (!m) return bad(1);
  const int Hm = m->n_mask_heads, Lq = m->Lq, Lk = m->Lk;
  if (Hm < 1 || Lq < 1 || Lk < 1) return bad(1);
  const int64_t R = cdiv64(Lq, kOT), C = cdiv64(Lk, kOT);
  if (m->ot_rows != R || m->ot_cols != C) return bad(2);
  if (m->n_full < 0 || m->n_part < 0 || (int64_t)Hm * R * C > INT32_MAX) return bad(3);
  if (!m->full_row_ptr || !m->part_row_ptr || (m->n_full > 0 && !m->full_col_idx) ||
      (m->n_part > 0 && (!m->part_col_idx || !m->part_bitmap)))
    return bad(4);
  const int64_t rows = (int64_t)Hm * R;
  // row pointers: start at 0, never decrease, end at the tile counts
  const int32_t* frp = m->full_row_ptr;
  const int32_t* prp = m->part_row_ptr;
  if (frp[0] != 0 || prp[0] != 0) return bad(5);
  for (int64_t i = 0; i < rows; ++i)
    if (frp[i + 1] < frp[i] || prp[i + 1] < prp[i]) return bad(6);
  if (frp[rows] != m->n_full || prp[rows] != m->n_part) return bad(7);
  std::vector<uint8_t> kind((size_t)C);
  uint64_t inr[64];
  int64_t valid = 0;
  for (int64_t row = 0; row < rows; ++row) {
    const int64_t a = row % R;
    std::memset(kind.data(), 0, kind.size());
    // columns ascending and inside the mask, within each structure
    for (int s = 0; s < 2; ++s) {
      const int32_t* rp = s ? prp : frp;
      const int32_t* ci = s ? m->part_col_idx : m->full_col_idx;
      for (int64_t t = rp[row]; t < rp[row + 1]; ++t) {
        const int32_t c = ci[t];
        if (c < 0 || c >= C) return bad(8);
        if (t > rp[row] && ci[t - 1] >= c) return bad(9);
        if (kind[c]) return bad(10);  // listed as full and as part
        kind[c] = (uint8_t)(1 + s);
      }
    }
    // full tiles lie wholly inside the mask (an edge tile is never full)
    for (int64_t t = frp[row]; t < frp[row + 1]; ++t) {
      const int32_t c = m->full_col_idx[t];
      if (64 * (a + 1) > Lq || 64 * ((int64_t)c + 1) > Lk) return bad(11);
      valid += 64 * 64;
    }
    // part tiles: no bit outside the mask, at least one bit, not every in-range bit
    for (int64_t t = prp[row]; t < prp[row + 1]; ++t) {
      const int32_t c = m->part_col_idx[t];
      in_range_words(a, c, Lq, Lk, inr);
      const uint64_t* w = m->part_bitmap + t * 64;
      bool any = false, all = true;
      for (int k = 0; k < 64; ++k) {
        if (w[k] & ~inr[k]) return bad(12);
        any = any || w[k] != 0;
        all = all && w[k] == inr[k];
        valid += popcount64(w[k]);
      }
      if (!any) return bad(13);
      if (all && 64 * (a + 1) <= Lq && 64 * ((int64_t)c + 1) <= Lk) return bad(14);  // that is a full tile
    }
  }
  if (m->n_valid >= 0 && m->n_valid != valid) return bad(15);
  // optional column lists of the block-wise kernel (host copy): each slot the union of the
  // non-empty columns of its two outer-tile rows, ascending, with both rows' kinds
  if (m->tile_lists) {
    if (C > 1024) return bad(16);
    const int64_t Cp = (C + 7) / 8 * 8, T = (R + 1) / 2, slot = 16 + 10 * Cp;
    const uint8_t* base = static_cast<const uint8_t*>(m->tile_lists);
    std::vector<int32_t> ka((size_t)C), kb((size_t)C);
    for (int64_t hm = 0; hm < Hm; ++hm)
      for (int64_t qt = 0; qt < T; ++qt) {
        for (int half = 0; half < 2; ++half) {
          std::vector<int32_t>& k = half ? kb : ka;
          std::fill(k.begin(), k.end(), -1);
          const int64_t a = 2 * qt + half;
          if (a >= R) continue;
          const int64_t row = hm * R + a;
          for (int64_t t = frp[row]; t < frp[row + 1]; ++t) k[m->full_col_idx[t]] = -2;
          for (int64_t t = prp[row]; t < prp[row + 1]; ++t) k[m->part_col_idx[t]] = (int32_t)t;
        }
        const uint8_t* sl = base + (hm * T + qt) * slot;
        int32_t n;
        std::memcpy(&n, sl, 4);
        const uint16_t* cols = reinterpret_cast<const uint16_t*>(sl + 16);
        const int32_t* la = reinterpret_cast<const int32_t*>(sl + 16 + 2 * Cp);
        const int32_t* lb = la + Cp;
        int64_t e = 0;
        for (int64_t c = 0; c < C; ++c) {
          if (ka[c] == -1 && kb[c] == -1) continue;
          if (e >= n || cols[e] != c || la[e] != ka[c] || lb[e] != kb[c]) return bad(17);
          ++e;
        }
        if (e != n) return bad(17);
      }
  }
  return STA_OK;
}
