// Two-level mask encoder (STOF, 手法 / 統合 MHA モジュール / 2 段階ストレージ形式):
// 64x64 outer tiles classified empty / full / part, full and part tiles listed in
// two CSR structures, one uint64 bitmap per 8x8 inner tile of each part tile.
//
// Kernels per call: classify (64 outer tiles of one OT row per block; every source is read
// as 64-bit row words -- bit-packed masks as stored, dense bytes compressed, patterns as
// intervals -- with popcounts and all-ones tests per tile; the last block to finish scans
// the per-row counts into row_ptr), fill (column lists by ballot prefixes over a pair of
// OT rows, and, when the caller asks for them, the block-wise kernel's column lists: the
// union of the non-empty columns of the pair), and bitmap (one part tile per 64-thread
// group: its 64 row words transposed into inner-tile words with warp shuffles).
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kMaxSrcPerLaunch = 32;

struct SrcDev {
  int32_t kind, causal;
  int64_t win_lo, win_hi, n_global;
  const void* data;
};

struct SrcBatch {
  SrcDev s[kMaxSrcPerLaunch];
  int32_t hm[kMaxSrcPerLaunch];  // mask head of entry t (classify)
  int32_t h0;                    // first mask head of this batch (bitmap: entries h0 .. h0 + n - 1)
};

// Bits lo..hi (clamped to 0..63) of a 64-bit word; 0 when the range is empty.
__device__ __forceinline__ uint64_t span_bits(int64_t lo, int64_t hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > 63 ? 63 : hi;
  if (lo > hi) return 0ull;
  return (~0ull << lo) & (~0ull >> (63 - hi));
}

// 16 mask bytes -> 16 bits (bit k: byte k nonzero). Per 32-bit lane __vsetne4 leaves 0 or 1
// in each byte; the multiply moves byte k's bit to bit 28 + k with no carries (the other
// partial products land on distinct bits below 28).
__device__ __forceinline__ uint32_t u8x16_bits(uint4 v) {
  const uint32_t x[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) out |= ((__vsetne4(x[k], 0u) * 0x10204080u) >> 28) << (4 * k);
  return out;
}

// Row i of the mask over OT column c: bit u = element (i, 64c + u). Rows past Lq give 0,
// columns past Lk are cleared. Bit-packed masks hold this word as is (one load); dense
// bytes take four 16-byte loads when rows are 16-byte aligned; patterns are intervals.
__device__ __forceinline__ uint64_t row_word(const SrcDev& s, int Lq, int Lk, int i, int c) {
  if (i >= Lq) return 0ull;
  const int64_t J0 = (int64_t)c * STA_OT;
  const int valid = Lk - (int)J0;  // columns of this word inside the mask (> 0)
  uint64_t w;
  if (s.kind == STA_MASK_DENSE_BITS) {
    const int64_t W = (Lk + 63) >> 6;
    w = __ldg(static_cast<const uint64_t*>(s.data) + (int64_t)i * W + c);
  } else if (s.kind == STA_MASK_DENSE_U8) {
    const uint8_t* row = static_cast<const uint8_t*>(s.data) + (int64_t)i * Lk + J0;
    if (valid >= 64 && ((reinterpret_cast<uintptr_t>(row) & 15) == 0)) {
      const uint4* v = reinterpret_cast<const uint4*>(row);
      w = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) w |= (uint64_t)u8x16_bits(__ldg(v + k)) << (16 * k);
    } else {
      w = 0;
      const int n = valid < 64 ? valid : 64;
      for (int u = 0; u < n; ++u) w |= (uint64_t)(row[u] != 0) << u;
    }
  } else {  // pattern: window [i + win_lo, i + win_hi], global columns [0, n_global), causal j <= i
    w = span_bits(i + s.win_lo - J0, i + s.win_hi - J0) | span_bits(-J0, s.n_global - 1 - J0);
    if (s.causal) w &= span_bits(0, i - J0);
  }
  if (valid < 64) w &= (1ull << valid) - 1ull;
  return w;
}

// The inner-tile word w (= 8p + q) of a 64-thread group whose thread w holds tile row w:
// word (p, q) is byte q of rows 8p..8p+7, gathered from the 8 lanes of the same warp.
__device__ __forceinline__ uint64_t transpose_tile_rows(uint64_t row, int w) {
  const int lane = w & 31, q = w & 7, rbase = lane & ~7;
  const uint32_t lo = (uint32_t)row, hi = (uint32_t)(row >> 32);
  uint64_t out = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint32_t xl = __shfl_sync(0xffffffffu, lo, rbase + r), xh = __shfl_sync(0xffffffffu, hi, rbase + r);
    const uint32_t byte = q < 4 ? (xl >> (8 * q)) & 0xFFu : (xh >> (8 * (q - 4))) & 0xFFu;
    out |= (uint64_t)byte << (8 * r);
  }
  return out;
}

constexpr int kClassifyCols = 64;  // outer-tile columns per classify block
constexpr int kClassifyThreads = 256;
constexpr int kRowGroups = kClassifyThreads / kClassifyCols;  // threads sharing one outer tile
constexpr int kRowsPerThread = STA_OT / kRowGroups;

// Exclusive scans of the per-row counts into row_ptr, totals[0..2] = n_full, n_part,
// n_valid; run by one whole block of kClassifyThreads threads, kScanPerThread consecutive
// rows per thread and pass (every count of a pass loaded at once).
constexpr int kScanPerThread = 8;

__device__ void scan_row_counts(const int32_t* full_cnt, const int32_t* part_cnt, const unsigned long long* valid_cnt,
                                int n, int32_t* full_row_ptr, int32_t* part_row_ptr, long long* totals) {
  constexpr int kWarps = kClassifyThreads / 32;
  __shared__ int s_wf[kWarps], s_wp[kWarps];
  __shared__ unsigned long long s_wv[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long carry_f = 0, carry_p = 0;
  unsigned long long vsum = 0;
  for (int base = 0; base < n; base += kClassifyThreads * kScanPerThread) {
    const int i0 = base + tid * kScanPerThread;
    int f[kScanPerThread], p[kScanPerThread];
    unsigned long long v = 0;
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {  // written by other blocks' atomics: read through L2
      const int i = i0 + e;
      f[e] = i < n ? __ldcg(full_cnt + i) : 0;
      p[e] = i < n ? __ldcg(part_cnt + i) : 0;
      v += i < n ? __ldcg(valid_cnt + i) : 0ull;
    }
    int sf = 0, sp = 0;
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) { sf += f[e]; sp += p[e]; }
    int xf = sf, xp = sp;  // inclusive over the warp's threads
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yf = __shfl_up_sync(0xffffffffu, xf, o), yp = __shfl_up_sync(0xffffffffu, xp, o);
      if (lane >= o) { xf += yf; xp += yp; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 31) { s_wf[warp] = xf; s_wp[warp] = xp; }
    if (lane == 0) s_wv[warp] = v;
    __syncthreads();
    int off_f = 0, off_p = 0, tot_f = 0, tot_p = 0;
    unsigned long long tot_v = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) { off_f += s_wf[w]; off_p += s_wp[w]; }
      tot_f += s_wf[w];
      tot_p += s_wp[w];
      tot_v += s_wv[w];
    }
    long long rf = carry_f + off_f + xf - sf, rp = carry_p + off_p + xp - sp;
#pragma unroll
    for (int e = 0; e < kScanPerThread; ++e) {
      const int i = i0 + e;
      if (i < n) {
        full_row_ptr[i] = (int32_t)rf;
        part_row_ptr[i] = (int32_t)rp;
      }
      rf += f[e];
      rp += p[e];
    }
    carry_f += tot_f;
    carry_p += tot_p;
    vsum += tot_v;
    __syncthreads();
  }
  if (tid == 0) {
    full_row_ptr[n] = (int32_t)carry_f;
    part_row_ptr[n] = (int32_t)carry_p;
    totals[0] = carry_f;
    totals[1] = carry_p;
    totals[2] = (long long)vsum;
  }
}

struct ScanOut {
  unsigned int* done;  // blocks finished, over every classify launch of the call (zeroed before)
  unsigned int n_blocks;
  int n_rows;  // Hm * R
  int32_t* full_row_ptr;
  int32_t* part_row_ptr;
  long long* totals;
};

// grid (R * ceil(C / 64), heads in batch), 256 threads: 64 outer tiles of one OT row per
// block. Thread (g, u) takes rows g, g + 4, ... of tile column u and keeps the popcount and
// the all-ones flag; the four row groups are combined in shared memory. The row counts add
// up across blocks (the counters are zeroed before the first launch) and the last block to
// finish scans them.
//
// kBulk (bit-packed sources whose rows start on 16 bytes and hold an even number of words):
// the block's rows arrive in shared memory by one bulk copy each (no registers hold loads in
// flight, so the whole tile row of 32 KB is requested at once) and the threads read them
// from there. Otherwise every thread requests its row words itself (bit-packed: 16 at once).
template <bool kBulk>
__global__ void __launch_bounds__(kClassifyThreads, kBulk ? 6 : 4) encode_classify_kernel(SrcBatch batch, int Lq, int Lk, int R,
                                                                          int C, uint8_t* __restrict__ cls,
                                                                          int32_t* __restrict__ full_cnt,
                                                                          int32_t* __restrict__ part_cnt,
                                                                          unsigned long long* __restrict__ valid_cnt,
                                                                          ScanOut so, int* err) {
  const SrcDev& src = batch.s[blockIdx.y];
  const int CB = (C + kClassifyCols - 1) / kClassifyCols;
  const int hm = batch.hm[blockIdx.y], a = blockIdx.x / CB, cb = blockIdx.x % CB;
  const int tid = threadIdx.x, lane = tid & 31, g = tid / kClassifyCols, u = tid % kClassifyCols;
  __shared__ int s_pop[kRowGroups][kClassifyCols];
  __shared__ int s_all[kRowGroups][kClassifyCols];
  __shared__ bool s_last;
  const int c_beg = cb * kClassifyCols;
  const int c = c_beg + u;
  const int i0 = a * STA_OT + g;
  int pop = 0;
  bool all = true;
  if constexpr (kBulk) {
    __shared__ __align__(128) uint64_t s_rows[STA_OT * kClassifyCols];
    __shared__ __align__(8) uint64_t s_bar;
    const int n_c = min(C, c_beg + kClassifyCols) - c_beg;  // even (C is even on this path)
    const int rows = min(STA_OT, Lq - a * STA_OT);          // rows of this OT row inside the mask
    const int64_t W = (Lk + 63) >> 6;
    if (tid == 0) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) mbar_arrive_expect_tx(&s_bar, (uint32_t)(rows * n_c * 8));
    if (tid < rows)
      bulk_g2s(s_rows + tid * kClassifyCols,
               static_cast<const uint64_t*>(src.data) + (int64_t)(a * STA_OT + tid) * W + c_beg, (uint32_t)(n_c * 8),
               &s_bar);
    const bool ok = mbar_wait(&s_bar, 0, err, 0x301);  // bounded; on timeout the counts are void
    if (u < n_c) {
      const int valid = Lk - c * STA_OT;  // columns of this word inside the mask
      const uint64_t keep = valid < 64 ? (1ull << valid) - 1ull : ~0ull;
#pragma unroll
      for (int k = 0; k < kRowsPerThread; ++k) {
        const int r = g + kRowGroups * k;
        const uint64_t w = ok && r < rows ? s_rows[r * kClassifyCols + u] & keep : 0ull;
        pop += __popcll(w);
        all = all && w == ~0ull;
      }
    }
  } else if (c < C) {
    if (src.kind == STA_MASK_DENSE_BITS) {  // every load of the thread in flight at once
      uint64_t rw[kRowsPerThread];
#pragma unroll
      for (int k = 0; k < kRowsPerThread; ++k) rw[k] = row_word(src, Lq, Lk, i0 + kRowGroups * k, c);
#pragma unroll
      for (int k = 0; k < kRowsPerThread; ++k) {
        pop += __popcll(rw[k]);
        all = all && rw[k] == ~0ull;
      }
    } else {
#pragma unroll 4
      for (int k = 0; k < kRowsPerThread; ++k) {
        const uint64_t w = row_word(src, Lq, Lk, i0 + kRowGroups * k, c);
        pop += __popcll(w);
        all = all && w == ~0ull;
      }
    }
  }
  s_pop[g][u] = pop;
  s_all[g][u] = all;
  __syncthreads();
  const int64_t row = (int64_t)hm * R + a;
  if (tid < kClassifyCols) {  // warps 0 and 1: one tile each
    int tot = 0, full = 1;
#pragma unroll
    for (int x = 0; x < kRowGroups; ++x) {
      tot += s_pop[x][tid];
      full &= s_all[x][tid];
    }
    const int k = c < C ? (tot == 0 ? 0 : (full ? 1 : 2)) : 0;
    if (c < C) cls[row * C + c] = (uint8_t)k;
    const int nf = __popc(__ballot_sync(0xffffffffu, k == 1)), np = __popc(__ballot_sync(0xffffffffu, k == 2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) {
      if (nf) atomicAdd(&full_cnt[row], nf);
      if (np) atomicAdd(&part_cnt[row], np);
      if (tot) atomicAdd(&valid_cnt[row], (unsigned long long)tot);
      __threadfence();  // the counts are visible before this block counts as done
    }
  }
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(so.done, 1u) == so.n_blocks - 1u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  scan_row_counts(full_cnt, part_cnt, valid_cnt, so.n_rows, so.full_row_ptr, so.part_row_ptr, so.totals);
}

// The block-wise kernel's column list of one (mask head, 128-row query tile) slot from the
// kinds of the tile's two OT rows (kinds[0..C) row 2t, kinds[C..2C) row 2t+1; -1 empty,
// -2 full, else the part-tile index): the columns non-empty in either row, ascending, each
// with both kinds. Slot layout: int32 n (16 bytes), uint16 cols[Cp], int32 ka[Cp], kb[Cp].
// Run by a whole block (a multiple of 32 threads, C <= 1024).
__device__ void write_tile_list(const int32_t* kinds, int C, int Cp, uint8_t* slot) {
  __shared__ uint32_t colbits[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int nwords = (C + 31) >> 5;
  for (int wd = warp; wd < nwords; wd += nwarps) {
    const int c = wd * 32 + lane;
    const unsigned b = __ballot_sync(0xffffffffu, c < C && (kinds[c] != -1 || kinds[C + c] != -1));
    if (lane == 0) colbits[wd] = b;
  }
  __syncthreads();
  uint16_t* cols = reinterpret_cast<uint16_t*>(slot + 16);
  int32_t* ka = reinterpret_cast<int32_t*>(slot + 16 + 2 * Cp);
  int32_t* kb = ka + Cp;
  const unsigned wl = lane < nwords ? colbits[lane] : 0u;
  int incl = __popc(wl);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - __popc(wl);
  for (int wd = warp; wd < nwords; wd += nwarps) {
    const unsigned b = __shfl_sync(0xffffffffu, wl, wd);
    const int base = __shfl_sync(0xffffffffu, excl, wd);
    const int c = wd * 32 + lane;
    if ((b >> lane) & 1u) {
      const int pos = base + __popc(b & ((1u << lane) - 1u));
      cols[pos] = (uint16_t)c;
      ka[pos] = kinds[c];
      kb[pos] = kinds[C + c];
    }
  }
  const int n = __shfl_sync(0xffffffffu, incl, 31);
  if (threadIdx.x == 0) reinterpret_cast<int4*>(slot)[0] = make_int4(n, 0, 0, 0);
}

// grid (ceil(R / 2), Hm), 256 threads: the column lists of the full and part tiles of OT
// rows 2t and 2t+1 (positions from ballot prefixes over the tile classes, 256 columns per
// pass), a marker in the first bitmap word of each part tile (its CSR row, read by the
// bitmap kernel) and, when lists is set, the block-wise kernel's column-list slot of the
// pair (dynamic shared memory: int32 kinds[2][C], C <= 1024).
__global__ void __launch_bounds__(256) encode_fill_kernel(int R, int C, int Cp, const uint8_t* __restrict__ cls,
                                                          const int32_t* __restrict__ full_row_ptr,
                                                          const int32_t* __restrict__ part_row_ptr,
                                                          int32_t* __restrict__ full_col_idx,
                                                          int32_t* __restrict__ part_col_idx,
                                                          uint64_t* __restrict__ part_bitmap, int64_t cap_full,
                                                          int64_t cap_part, uint8_t* __restrict__ lists) {
  extern __shared__ int32_t kinds[];  // [2][C] when lists != nullptr
  const int hm = blockIdx.y, t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ int s_wf[8], s_wp[8];
  for (int half = 0; half < 2; ++half) {
    const int a = 2 * t + half;
    if (a >= R) {
      if (lists)
        for (int c = tid; c < C; c += blockDim.x) kinds[half * C + c] = -1;
      continue;
    }
    const int64_t row = (int64_t)hm * R + a;
    const int64_t fbase = full_row_ptr[row], pbase = part_row_ptr[row];
    int64_t run_f = 0, run_p = 0;
    for (int c0 = 0; c0 < C; c0 += 256) {
      const int c = c0 + tid;
      const int k = c < C ? cls[row * C + c] : 0;
      const unsigned bf = __ballot_sync(0xffffffffu, k == 1), bp = __ballot_sync(0xffffffffu, k == 2);
      const unsigned below = (1u << lane) - 1u;
      if (lane == 0) { s_wf[warp] = __popc(bf); s_wp[warp] = __popc(bp); }
      __syncthreads();
      int off_f = 0, off_p = 0, tot_f = 0, tot_p = 0;
      for (int x = 0; x < 8; ++x) {
        if (x < warp) { off_f += s_wf[x]; off_p += s_wp[x]; }
        tot_f += s_wf[x];
        tot_p += s_wp[x];
      }
      int32_t kind = -1;
      if (k == 1) {
        const int64_t pos = fbase + run_f + off_f + __popc(bf & below);
        if (pos < cap_full) full_col_idx[pos] = c;
        kind = -2;
      }
      if (k == 2) {
        const int64_t pos = pbase + run_p + off_p + __popc(bp & below);
        if (pos < cap_part) {
          part_col_idx[pos] = c;
          part_bitmap[pos * 64] = (uint64_t)row;  // read (then overwritten) by the bitmap kernel
        }
        kind = (int32_t)pos;
      }
      if (lists && c < C) kinds[half * C + c] = kind;
      run_f += tot_f;
      run_p += tot_p;
      __syncthreads();
    }
  }
  if (!lists) return;
  __syncthreads();
  const int T = (R + 1) / 2;
  write_tile_list(kinds, C, Cp, lists + ((int64_t)hm * T + t) * (16 + 10 * (int64_t)Cp));
}

// Bitmaps of the part tiles: grid ceil(n_part / 4), 256 threads, one part tile per group of
// 64 threads (one inner-tile word each). The tile's OT row (mask head * R + OT row) is the
// first word of its bitmap slot, left there by the fill kernel, when one launch covers every
// mask head (up to 32); with more heads each launch searches part_row_ptr instead, and
// leaves the tiles of heads outside its batch to their batch.
__global__ void __launch_bounds__(256) encode_bitmap_kernel(SrcBatch batch, int nb, int Hm, int Lq, int Lk, int R,
                                                            const int32_t* __restrict__ part_row_ptr,
                                                            const int32_t* __restrict__ part_col_idx,
                                                            uint64_t* __restrict__ part_bitmap, int64_t n_part) {
  const int g = threadIdx.x >> 6, w = threadIdx.x & 63;
  const int64_t t = (int64_t)blockIdx.x * 4 + g;
  int hm = -1, a = 0, c = -1;
  if (t < n_part) {
    int64_t row;
    if (nb == Hm) {  // one launch for all heads: the row is in the slot, left there by the fill kernel
      row = (int64_t)part_bitmap[t * 64];
    } else {  // several launches: earlier ones have overwritten slots, search part_row_ptr
      int lo = 0, hi = Hm * R;  // part_row_ptr[lo] <= t < part_row_ptr[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(part_row_ptr + mid) <= t) lo = mid;
        else hi = mid;
      }
      row = lo;
    }
    hm = (int)(row / R);
    a = (int)(row - (int64_t)hm * R);
    c = __ldg(part_col_idx + t);
  }
  __syncthreads();  // every group has read its slot's first word before any group writes
  const int bh = hm - batch.h0;
  const bool mine = t < n_part && bh >= 0 && bh < nb;
  // every thread of the group takes part in the word (warp shuffles); the source is uniform
  // over the group
  const SrcDev& src = batch.s[mine ? bh : 0];
  const uint64_t word = transpose_tile_rows(mine ? row_word(src, Lq, Lk, a * STA_OT + w, c) : 0ull, w);
  if (mine) part_bitmap[t * 64 + w] = word;
}

inline int64_t clamp40(int64_t x) {
  constexpr int64_t kLim = (int64_t)1 << 40;
  return x < -kLim ? -kLim : (x > kLim ? kLim : x);
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct EncodeWs {
  size_t cls, full_cnt, part_cnt, valid_cnt, totals, done, total;
};

EncodeWs encode_ws_layout(int64_t Hm, int64_t R, int64_t C) {
  EncodeWs w;
  size_t off = 0;
  w.cls = off; off += align256((size_t)(Hm * R * C));
  w.full_cnt = off; off += align256(sizeof(int32_t) * Hm * R);
  w.part_cnt = off; off += align256(sizeof(int32_t) * Hm * R);
  w.valid_cnt = off; off += align256(sizeof(unsigned long long) * Hm * R);
  w.totals = off; off += align256(sizeof(long long) * 4);
  w.done = off; off += align256(sizeof(unsigned int));
  w.total = off;
  return w;
}

}  // namespace

size_t tile_lists_bytes(int Hm, int Lq, int Lk) {
  if (Hm < 1 || Lq < 1 || Lk < 1) return 0;
  const int64_t R = cdiv(Lq, STA_OT), C = cdiv(Lk, STA_OT);
  if (C > kMaxTileListCols) return 0;
  const int64_t Cp = (C + 7) / 8 * 8;
  return (size_t)Hm * (size_t)((R + 1) / 2) * (size_t)(16 + 10 * Cp);
}

}  // namespace sta

using namespace sta;

extern "C" size_t sta_tile_lists_bytes(int Hm, int Lq, int Lk) { return tile_lists_bytes(Hm, Lq, Lk); }

extern "C" sta_status sta_encode_mask(const sta_mask_src* srcs, int Hm, int Lq, int Lk, sta_bsr_mask* out,
                                      void* workspace, size_t* workspace_bytes, sta_stream stream) {
  if (!srcs || !out || !workspace_bytes || Hm < 1 || Lq < 1 || Lk < 1 || Lq >= (1 << 30) || Lk >= (1 << 30))
    return STA_ERR_INVALID_ARG;
  const int64_t R = cdiv(Lq, STA_OT), C = cdiv(Lk, STA_OT);
  if ((int64_t)Hm * R * C > INT32_MAX || (int64_t)Hm * R >= (1 << 24)) return STA_ERR_INVALID_ARG;
  for (int h = 0; h < Hm; ++h) {
    const sta_mask_src& s = srcs[h];
    if (s.kind == STA_MASK_PATTERN) {
      if (s.win_lo > s.win_hi && s.n_global_cols <= 0) { /* all-empty pattern: allowed */ }
    } else if (s.kind == STA_MASK_DENSE_U8 || s.kind == STA_MASK_DENSE_BITS) {
      if (!s.data) return STA_ERR_INVALID_ARG;
      if (s.kind == STA_MASK_DENSE_BITS && ((uintptr_t)s.data & 7)) return STA_ERR_UNSUPPORTED;
    } else {
      return STA_ERR_INVALID_ARG;
    }
  }
  const EncodeWs L = encode_ws_layout(Hm, R, C);
  if (!workspace) {
    *workspace_bytes = L.total;
    return STA_OK;
  }
  if (*workspace_bytes < L.total) return STA_ERR_WORKSPACE;
  if ((uintptr_t)workspace & 255) return STA_ERR_INVALID_ARG;
  if (!out->full_row_ptr || !out->part_row_ptr) return STA_ERR_INVALID_ARG;
  const bool query = !out->full_col_idx && !out->part_col_idx && !out->part_bitmap;
  if (!query) {
    if (out->n_full < 0 || out->n_part < 0) return STA_ERR_INVALID_ARG;
    if ((out->n_full > 0 && !out->full_col_idx) || (out->n_part > 0 && (!out->part_col_idx || !out->part_bitmap)))
      return STA_ERR_INVALID_ARG;
    if (out->tile_lists && (C > kMaxTileListCols || ((uintptr_t)out->tile_lists & 15))) return STA_ERR_INVALID_ARG;
  }
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  uint8_t* cls = (uint8_t*)(ws + L.cls);
  int32_t* fcnt = (int32_t*)(ws + L.full_cnt);
  int32_t* pcnt = (int32_t*)(ws + L.part_cnt);
  unsigned long long* vcnt = (unsigned long long*)(ws + L.valid_cnt);
  long long* totals = (long long*)(ws + L.totals);

  // entries t = 0 .. n-1 take mask heads heads[t] (or h0 + t)
  auto make_batch = [&](int h0, int n, const int* heads = nullptr) {
    SrcBatch b;
    memset(&b, 0, sizeof(b));
    b.h0 = h0;
    for (int t = 0; t < n; ++t) {
      const int hm = heads ? heads[t] : h0 + t;
      b.hm[t] = hm;
      const sta_mask_src& s = srcs[hm];
      b.s[t].kind = s.kind;
      b.s[t].causal = s.causal;
      // |j - i| and j stay below 2^30: clamping to +-2^40 keeps every predicate and keeps the
      // kernels' interval arithmetic clear of int64 overflow
      b.s[t].win_lo = clamp40(s.win_lo);
      b.s[t].win_hi = clamp40(s.win_hi);
      b.s[t].n_global = clamp40(s.n_global_cols);
      b.s[t].data = s.data;
    }
    return b;
  };
  STA_CUDA_TRY(cudaMemsetAsync(ws + L.full_cnt, 0, L.total - L.full_cnt, st));  // row counters, done count
  const int64_t CB = cdiv(C, kClassifyCols);
  ScanOut so;
  so.done = (unsigned int*)(ws + L.done);
  so.n_blocks = (unsigned int)(R * CB * Hm);
  so.n_rows = (int)(Hm * R);
  so.full_row_ptr = out->full_row_ptr;
  so.part_row_ptr = out->part_row_ptr;
  so.totals = totals;
  // classify: bit-packed heads whose rows can be bulk-copied (16-byte aligned rows of an even
  // number of words) in one set of launches, every other head in another
  int* err = device_error_word();
  std::vector<int> bulk, other;
  for (int h = 0; h < Hm; ++h) {
    const sta_mask_src& s = srcs[h];
    const bool b = s.kind == STA_MASK_DENSE_BITS && ((uintptr_t)s.data & 15) == 0 && (C & 1) == 0;
    (b ? bulk : other).push_back(h);
  }
  for (int pass = 0; pass < 2; ++pass) {
    const std::vector<int>& hs = pass == 0 ? bulk : other;
    for (size_t t0 = 0; t0 < hs.size(); t0 += kMaxSrcPerLaunch) {
      const int n = (int)std::min(hs.size() - t0, (size_t)kMaxSrcPerLaunch);
      const dim3 grid((unsigned)(R * CB), (unsigned)n);
      const SrcBatch b = make_batch(0, n, hs.data() + t0);
      if (pass == 0)
        encode_classify_kernel<true><<<grid, kClassifyThreads, 0, st>>>(b, Lq, Lk, (int)R, (int)C, cls, fcnt, pcnt,
                                                                        vcnt, so, err);
      else
        encode_classify_kernel<false><<<grid, kClassifyThreads, 0, st>>>(b, Lq, Lk, (int)R, (int)C, cls, fcnt, pcnt,
                                                                         vcnt, so, err);
      STA_LAUNCH_CHECK();
    }
  }
  out->n_mask_heads = Hm;
  out->Lq = Lq;
  out->Lk = Lk;
  out->ot_rows = (int32_t)R;
  out->ot_cols = (int32_t)C;
  if (query) {
    long long h_tot[3] = {0, 0, 0};
    STA_CUDA_TRY(cudaMemcpyAsync(h_tot, totals, sizeof(h_tot), cudaMemcpyDeviceToHost, st));
    std::vector<int32_t> rows;
    std::vector<unsigned long long> vrows;
    if (out->head_valid) {  // per-head valid counts from the per-row counts of the classify pass
      vrows.resize((size_t)Hm * R);
      STA_CUDA_TRY(cudaMemcpyAsync(vrows.data(), vcnt, sizeof(unsigned long long) * Hm * R, cudaMemcpyDeviceToHost,
                                   st));
    }
    if (out->head_tiles) {  // per-head tile counts from the two row_ptr arrays
      rows.resize(2 * ((size_t)Hm * R + 1));
      STA_CUDA_TRY(cudaMemcpyAsync(rows.data(), out->full_row_ptr, sizeof(int32_t) * (Hm * R + 1),
                                   cudaMemcpyDeviceToHost, st));
      STA_CUDA_TRY(cudaMemcpyAsync(rows.data() + Hm * R + 1, out->part_row_ptr, sizeof(int32_t) * (Hm * R + 1),
                                   cudaMemcpyDeviceToHost, st));
    }
    STA_CUDA_TRY(cudaStreamSynchronize(st));
    out->n_full = h_tot[0];
    out->n_part = h_tot[1];
    out->n_valid = h_tot[2];
    if (out->head_tiles) {
      const int32_t* f = rows.data();
      const int32_t* p = rows.data() + Hm * R + 1;
      for (int h = 0; h < Hm; ++h)
        out->head_tiles[h] = (int64_t)(f[(h + 1) * R] - f[h * R]) + (int64_t)(p[(h + 1) * R] - p[h * R]);
    }
    if (out->head_valid) {
      for (int h = 0; h < Hm; ++h) {
        unsigned long long v = 0;
        for (int64_t a = 0; a < R; ++a) v += vrows[(size_t)h * R + a];
        out->head_valid[h] = (int64_t)v;
      }
    }
    return STA_OK;
  }
  const int Cp = (int)((C + 7) / 8 * 8);
  uint8_t* lists = static_cast<uint8_t*>(out->tile_lists);
  encode_fill_kernel<<<dim3((unsigned)((R + 1) / 2), (unsigned)Hm), 256,
                       lists ? 2 * C * sizeof(int32_t) : 0, st>>>((int)R, (int)C, Cp, cls, out->full_row_ptr,
                                                                  out->part_row_ptr, out->full_col_idx,
                                                                  out->part_col_idx, out->part_bitmap, out->n_full,
                                                                  out->n_part, lists);
  STA_LAUNCH_CHECK();
  if (out->n_part > 0) {
    for (int h0 = 0; h0 < Hm; h0 += kMaxSrcPerLaunch) {
      const int n = Hm - h0 < kMaxSrcPerLaunch ? Hm - h0 : kMaxSrcPerLaunch;
      encode_bitmap_kernel<<<(unsigned)cdiv(out->n_part, 4), 256, 0, st>>>(
          make_batch(h0, n), n, Hm, Lq, Lk, (int)R, out->part_row_ptr, out->part_col_idx, out->part_bitmap,
          out->n_part);
      STA_LAUNCH_CHECK();
    }
  }
  return STA_OK;
}
