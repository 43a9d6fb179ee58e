// Two-level mask encoder (STOF, 手法 / 統合 MHA モジュール / 2 段階ストレージ形式):
// 64x64 outer tiles classified empty / full / part, full and part tiles listed in
// two CSR structures, one uint64 bitmap per 8x8 inner tile of each part tile.
//
// Three kernels per call: classify (one CTA per (mask head, OT row), warp-level
// popcounts of the inner-tile words), a single-CTA scan of the per-row counts into
// row_ptr, and fill (ballot-prefix positions, then the bitmaps of part tiles). When
// the caller asks for them, a fourth kernel derives the block-wise kernel's column
// lists (the union of the non-empty columns of each pair of OT rows) from the CSR.
#include <vector>

#include "common.cuh"

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
  int32_t h0;  // first mask head of this batch
};

// Bits of row i, columns j0..j0+7 (j0 % 8 == 0): bit c = column j0 + c.
// Out-of-range rows/columns give 0.
__device__ __forceinline__ uint32_t row_byte(const SrcDev& s, int Lq, int Lk, int i, int j0) {
  if (i >= Lq || j0 >= Lk) return 0u;
  const uint32_t colmask = (Lk - j0 >= 8) ? 0xFFu : ((1u << (Lk - j0)) - 1u);
  uint32_t b = 0;
  if (s.kind == STA_MASK_DENSE_BITS) {
    const int64_t W = (Lk + 63) >> 6;
    const uint64_t w = static_cast<const uint64_t*>(s.data)[(int64_t)i * W + (j0 >> 6)];
    b = (uint32_t)((w >> (j0 & 63)) & 0xFFull);
  } else if (s.kind == STA_MASK_DENSE_U8) {
    const uint8_t* row = static_cast<const uint8_t*>(s.data) + (int64_t)i * Lk;
    const int n = min(8, Lk - j0);
    for (int c = 0; c < n; ++c) b |= (row[j0 + c] != 0 ? 1u : 0u) << c;
  } else {  // pattern
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int64_t j = j0 + c;
      const int64_t dd = j - i;
      bool v = (dd >= s.win_lo && dd <= s.win_hi) || (j < s.n_global);
      if (s.causal && j > i) v = false;
      b |= (v ? 1u : 0u) << c;
    }
  }
  return b & colmask;
}

// Inner-tile word (p, q) of outer tile (a, c): bit 8r + cc = element (64a+8p+r, 64c+8q+cc).
__device__ __forceinline__ uint64_t it_word(const SrcDev& s, int Lq, int Lk, int a, int c, int p, int q) {
  uint64_t w = 0;
  const int i0 = a * STA_OT + p * STA_IT, j0 = c * STA_OT + q * STA_IT;
#pragma unroll
  for (int r = 0; r < 8; ++r) w |= (uint64_t)row_byte(s, Lq, Lk, i0 + r, j0) << (8 * r);
  return w;
}

// grid (R, heads in batch), 256 threads: four outer tiles per pass, 64 threads per tile.
__global__ void __launch_bounds__(256) encode_classify_kernel(SrcBatch batch, int Lq, int Lk, int R, int C,
                                                              uint8_t* __restrict__ cls, int32_t* __restrict__ full_cnt,
                                                              int32_t* __restrict__ part_cnt,
                                                              unsigned long long* __restrict__ valid_cnt) {
  const SrcDev& src = batch.s[blockIdx.y];
  const int hm = batch.h0 + blockIdx.y, a = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = tid >> 6, w = tid & 63, p = w >> 3, q = w & 7;
  __shared__ int s_pop[8], s_all[8];
  __shared__ int s_nf, s_np;
  __shared__ unsigned long long s_nv;
  if (tid == 0) { s_nf = 0; s_np = 0; s_nv = 0; }
  __syncthreads();
  const int64_t row = (int64_t)hm * R + a;
  for (int c0 = 0; c0 < C; c0 += 4) {
    const int c = c0 + g;
    const uint64_t word = (c < C) ? it_word(src, Lq, Lk, a, c, p, q) : 0ull;
    int pop = __popcll(word);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pop += __shfl_xor_sync(0xffffffffu, pop, o);
    const int all = __all_sync(0xffffffffu, word == ~0ull);
    if (lane == 0) { s_pop[warp] = pop; s_all[warp] = all; }
    __syncthreads();
    if (tid < 4 && c0 + tid < C) {
      const int tot = s_pop[2 * tid] + s_pop[2 * tid + 1];
      const int full = s_all[2 * tid] && s_all[2 * tid + 1];
      const uint8_t k = tot == 0 ? 0 : (full ? 1 : 2);
      cls[row * C + c0 + tid] = k;
      if (k == 1) atomicAdd(&s_nf, 1);
      if (k == 2) atomicAdd(&s_np, 1);
      atomicAdd(&s_nv, (unsigned long long)tot);
    }
    __syncthreads();
  }
  if (tid == 0) {
    full_cnt[row] = s_nf;
    part_cnt[row] = s_np;
    valid_cnt[row] = s_nv;
  }
}

// One CTA of 1024 threads: exclusive scans of the per-row counts into row_ptr,
// totals[0..2] = n_full, n_part, n_valid.
__global__ void __launch_bounds__(1024) encode_scan_kernel(const int32_t* __restrict__ full_cnt,
                                                           const int32_t* __restrict__ part_cnt,
                                                           const unsigned long long* __restrict__ valid_cnt, int n,
                                                           int32_t* __restrict__ full_row_ptr,
                                                           int32_t* __restrict__ part_row_ptr,
                                                           long long* __restrict__ totals) {
  __shared__ int s_wf[32], s_wp[32];
  __shared__ unsigned long long s_wv[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long carry_f = 0, carry_p = 0;
  unsigned long long vsum = 0;
  for (int base = 0; base < n; base += 1024) {
    const int i = base + tid;
    const int f = i < n ? full_cnt[i] : 0;
    const int p = i < n ? part_cnt[i] : 0;
    unsigned long long v = i < n ? valid_cnt[i] : 0ull;
    int xf = f, xp = p;
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
    for (int w = 0; w < 32; ++w) {
      if (w < warp) { off_f += s_wf[w]; off_p += s_wp[w]; }
      tot_f += s_wf[w];
      tot_p += s_wp[w];
      tot_v += s_wv[w];
    }
    if (i < n) {
      full_row_ptr[i] = (int32_t)(carry_f + off_f + xf - f);
      part_row_ptr[i] = (int32_t)(carry_p + off_p + xp - p);
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

// grid (R, heads in batch), 256 threads. Positions come from ballot prefixes over
// the tile classes in chunks of 256 columns; part-tile bitmaps are recomputed.
__global__ void __launch_bounds__(256) encode_fill_kernel(SrcBatch batch, int Lq, int Lk, int R, int C,
                                                          const uint8_t* __restrict__ cls,
                                                          const int32_t* __restrict__ full_row_ptr,
                                                          const int32_t* __restrict__ part_row_ptr,
                                                          int32_t* __restrict__ full_col_idx,
                                                          int32_t* __restrict__ part_col_idx,
                                                          uint64_t* __restrict__ part_bitmap, int64_t cap_full,
                                                          int64_t cap_part) {
  const SrcDev& src = batch.s[blockIdx.y];
  const int hm = batch.h0 + blockIdx.y, a = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = tid >> 6, w = tid & 63, p = w >> 3, q = w & 7;
  __shared__ int s_wf[8], s_wp[8];
  __shared__ int s_cols[256];
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
    if (k == 1) {
      const int64_t pos = fbase + run_f + off_f + __popc(bf & below);
      if (pos < cap_full) full_col_idx[pos] = c;
    }
    if (k == 2) {
      const int lp = off_p + __popc(bp & below);
      s_cols[lp] = c;
      const int64_t pos = pbase + run_p + lp;
      if (pos < cap_part) part_col_idx[pos] = c;
    }
    __syncthreads();
    for (int t0 = 0; t0 < tot_p; t0 += 4) {
      const int t = t0 + g;
      if (t < tot_p) {
        const int64_t pos = pbase + run_p + t;
        const uint64_t word = it_word(src, Lq, Lk, a, s_cols[t], p, q);
        if (pos < cap_part) part_bitmap[pos * 64 + w] = word;
      }
    }
    run_f += tot_f;
    run_p += tot_p;
    __syncthreads();
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct EncodeWs {
  size_t cls, full_cnt, part_cnt, valid_cnt, totals, total;
};

EncodeWs encode_ws_layout(int64_t Hm, int64_t R, int64_t C) {
  EncodeWs w;
  size_t off = 0;
  w.cls = off; off += align256((size_t)(Hm * R * C));
  w.full_cnt = off; off += align256(sizeof(int32_t) * Hm * R);
  w.part_cnt = off; off += align256(sizeof(int32_t) * Hm * R);
  w.valid_cnt = off; off += align256(sizeof(unsigned long long) * Hm * R);
  w.totals = off; off += align256(sizeof(long long) * 4);
  w.total = off;
  return w;
}

// Column lists of the block-wise kernel, one CTA per (query tile t, mask head):
// the OT columns non-empty in row 2t or 2t+1, ascending, each with the kinds of
// both rows (-1 empty, -2 full, part-tile index). Dynamic shared memory: two
// int32 arrays of C (kind of each column per row). C <= 1024.
__global__ void __launch_bounds__(256) encode_tile_lists_kernel(const int32_t* __restrict__ full_row_ptr,
                                                                const int32_t* __restrict__ full_col_idx,
                                                                const int32_t* __restrict__ part_row_ptr,
                                                                const int32_t* __restrict__ part_col_idx, int R,
                                                                int C, int Cp, uint8_t* __restrict__ lists) {
  extern __shared__ int32_t kinds[];  // [2][C]
  __shared__ uint32_t colbits[32];
  const int t = blockIdx.x, hm = blockIdx.y, T = (R + 1) / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int c = threadIdx.x; c < 2 * C; c += blockDim.x) kinds[c] = -1;
  __syncthreads();
  for (int half = 0; half < 2; ++half) {
    const int a = 2 * t + half;
    if (a >= R) continue;
    const int64_t row = (int64_t)hm * R + a;
    int32_t* k = kinds + half * C;
    for (int i = full_row_ptr[row] + threadIdx.x; i < full_row_ptr[row + 1]; i += blockDim.x) k[full_col_idx[i]] = -2;
    for (int i = part_row_ptr[row] + threadIdx.x; i < part_row_ptr[row + 1]; i += blockDim.x) k[part_col_idx[i]] = i;
  }
  __syncthreads();
  const int nwords = (C + 31) >> 5;
  for (int wd = warp; wd < nwords; wd += blockDim.x / 32) {
    const int c = wd * 32 + lane;
    const unsigned b = __ballot_sync(0xffffffffu, c < C && (kinds[c] != -1 || kinds[C + c] != -1));
    if (lane == 0) colbits[wd] = b;
  }
  __syncthreads();
  uint8_t* slot = lists + ((int64_t)hm * T + t) * (16 + 10 * (int64_t)Cp);
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
  for (int wd = warp; wd < nwords; wd += blockDim.x / 32) {
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

  auto make_batch = [&](int h0, int n) {
    SrcBatch b;
    memset(&b, 0, sizeof(b));
    b.h0 = h0;
    for (int t = 0; t < n; ++t) {
      const sta_mask_src& s = srcs[h0 + t];
      b.s[t].kind = s.kind;
      b.s[t].causal = s.causal;
      b.s[t].win_lo = s.win_lo;
      b.s[t].win_hi = s.win_hi;
      b.s[t].n_global = s.n_global_cols;
      b.s[t].data = s.data;
    }
    return b;
  };
  for (int h0 = 0; h0 < Hm; h0 += kMaxSrcPerLaunch) {
    const int n = Hm - h0 < kMaxSrcPerLaunch ? Hm - h0 : kMaxSrcPerLaunch;
    encode_classify_kernel<<<dim3((unsigned)R, (unsigned)n), 256, 0, st>>>(make_batch(h0, n), Lq, Lk, (int)R,
                                                                          (int)C, cls, fcnt, pcnt, vcnt);
    STA_LAUNCH_CHECK();
  }
  encode_scan_kernel<<<1, 1024, 0, st>>>(fcnt, pcnt, vcnt, (int)(Hm * R), out->full_row_ptr, out->part_row_ptr,
                                         totals);
  STA_LAUNCH_CHECK();
  out->n_mask_heads = Hm;
  out->Lq = Lq;
  out->Lk = Lk;
  out->ot_rows = (int32_t)R;
  out->ot_cols = (int32_t)C;
  if (query) {
    long long h_tot[3] = {0, 0, 0};
    STA_CUDA_TRY(cudaMemcpyAsync(h_tot, totals, sizeof(h_tot), cudaMemcpyDeviceToHost, st));
    std::vector<int32_t> rows;
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
    return STA_OK;
  }
  for (int h0 = 0; h0 < Hm; h0 += kMaxSrcPerLaunch) {
    const int n = Hm - h0 < kMaxSrcPerLaunch ? Hm - h0 : kMaxSrcPerLaunch;
    encode_fill_kernel<<<dim3((unsigned)R, (unsigned)n), 256, 0, st>>>(
        make_batch(h0, n), Lq, Lk, (int)R, (int)C, cls, out->full_row_ptr, out->part_row_ptr, out->full_col_idx,
        out->part_col_idx, out->part_bitmap, out->n_full, out->n_part);
    STA_LAUNCH_CHECK();
  }
  if (out->tile_lists) {
    const int Cp = (int)((C + 7) / 8 * 8);
    encode_tile_lists_kernel<<<dim3((unsigned)((R + 1) / 2), (unsigned)Hm), 256, 2 * C * sizeof(int32_t), st>>>(
        out->full_row_ptr, out->full_col_idx, out->part_row_ptr, out->part_col_idx, (int)R, (int)C, Cp,
        static_cast<uint8_t*>(out->tile_lists));
    STA_LAUNCH_CHECK();
  }
  return STA_OK;
}
