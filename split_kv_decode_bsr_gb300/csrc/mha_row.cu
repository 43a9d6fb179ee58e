// Row-wise masked MHA kernel (STOF, デュアルカーネル戦略 / 行方向カーネル):
// Q sliced by rows, one warp per query row, warp shuffles for the softmax
// reductions. The warp walks only the non-empty outer tiles of its row: full
// tiles 32 keys at a time (one key per lane), part tiles through the row's bytes
// of their inner-tile words, skipping empty inner tiles and scoring each valid
// key with the head dimensions spread over the lanes. Scores fold into an fp32
// online softmax (running max m, running sum l, output rescaled by
// exp2(m_old - m_new)). Handles bf16 and fp32 inputs, head dims 64 and 128.
// Unlike the pages' kernel, the warps of a block are not independent: its 8 rows
// need the same inner-tile words, which the block stages once per round of 32
// part tiles (one block barrier per round) instead of every warp loading them.
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kRowWarps = 8;

template <int D, bool BF16>
struct RowIO;

template <int D>
struct RowIO<D, true> {
  // dot(q, k_row) with q (pre-scaled) in shared memory as float
  static __device__ __forceinline__ float dot(const float* sq, const void* kbase, int64_t j) {
    const uint4* kr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(kbase) + j * D);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 w = __ldg(kr + c);
      const float4 qa = *reinterpret_cast<const float4*>(sq + 8 * c);
      const float4 qb = *reinterpret_cast<const float4*>(sq + 8 * c + 4);
      acc = fmaf(qa.x, bf16lo(w.x), acc);
      acc = fmaf(qa.y, bf16hi(w.x), acc);
      acc = fmaf(qa.z, bf16lo(w.y), acc);
      acc = fmaf(qa.w, bf16hi(w.y), acc);
      acc = fmaf(qb.x, bf16lo(w.z), acc);
      acc = fmaf(qb.y, bf16hi(w.z), acc);
      acc = fmaf(qb.z, bf16lo(w.w), acc);
      acc = fmaf(qb.w, bf16hi(w.w), acc);
    }
    return acc;
  }
  // this lane's D/32 elements of a row
  static __device__ __forceinline__ void load_lane(const void* base, int64_t row, int lane, float* x) {
    const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + row * D + lane * (D / 32);
    if constexpr (D == 64) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p));
      x[0] = bf16lo(w);
      x[1] = bf16hi(w);
    } else {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
      x[0] = bf16lo(w.x);
      x[1] = bf16hi(w.x);
      x[2] = bf16lo(w.y);
      x[3] = bf16hi(w.y);
    }
  }
  static __device__ __forceinline__ void store_lane(void* base, int64_t row, int lane, const float* x) {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + row * D + lane * (D / 32);
#pragma unroll
    for (int e = 0; e < D / 32; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(p + e) = __floats2bfloat162_rn(x[e], x[e + 1]);
  }
};

template <int D>
struct RowIO<D, false> {
  static __device__ __forceinline__ float dot(const float* sq, const void* kbase, int64_t j) {
    const float4* kr = reinterpret_cast<const float4*>(static_cast<const float*>(kbase) + j * D);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D / 4; ++c) {
      const float4 w = __ldg(kr + c);
      const float4 qa = *reinterpret_cast<const float4*>(sq + 4 * c);
      acc = fmaf(qa.x, w.x, acc);
      acc = fmaf(qa.y, w.y, acc);
      acc = fmaf(qa.z, w.z, acc);
      acc = fmaf(qa.w, w.w, acc);
    }
    return acc;
  }
  static __device__ __forceinline__ void load_lane(const void* base, int64_t row, int lane, float* x) {
    const float* p = static_cast<const float*>(base) + row * D + lane * (D / 32);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) x[e] = __ldg(p + e);
  }
  static __device__ __forceinline__ void store_lane(void* base, int64_t row, int lane, const float* x) {
    float* p = static_cast<float*>(base) + row * D + lane * (D / 32);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) p[e] = x[e];
  }
};

// grid (ceil(Lq / 8), B * H), 8 warps: warp w handles query row blockIdx.x * 8 + w.
// Full tiles are scored 32 keys at a time, one key per lane against q in shared memory.
// Part tiles are scanned four at a time (lane 8u + w reads inner-tile word w of the row's
// group in tile u), and each valid key is then scored with the dimensions spread over the
// lanes (lane owns d/32 of them) and a warp sum, so a sparse row costs work in proportion
// to its valid keys rather than to the 32 keys of each chunk it touches.
template <int D, bool BF16>
__global__ void __launch_bounds__(kRowWarps * 32) mha_row_kernel(const MhaArgs A) {
  using IO = RowIO<D, BF16>;
  constexpr int E = D / 32;
  __shared__ __align__(16) float s_q[kRowWarps][D];
  __shared__ int s_keys[kRowWarps][72];  // valid keys waiting for a batch: fewer than 8, plus one tile's 64
  // a scan round's 32 part tiles, staged once for the CTA's 8 rows (two buffers): row w's
  // 64-bit key mask of each tile, and the tiles' columns
  __shared__ __align__(16) uint64_t s_mask[2][kRowWarps][32];
  __shared__ int s_col[2][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kRowWarps + warp;
  // rows past Lq (only in the last block) skip the work but take part in staging the scan
  // rounds and in the block's barriers
  const bool active = i < A.Lq;
  // grid.y = (batch, launch rank): the launch covers heads hmap.order[0 .. n_ranks-1]
  const int bi = blockIdx.y / A.n_ranks;
  const int h = A.hmap.order[blockIdx.y - bi * A.n_ranks];
  const int64_t bh = (int64_t)bi * A.H + h;
  const int hm = A.hmap.m[h];
  const int64_t qrow = bh * A.Lq + i;
  const int64_t kv0 = bh * A.Lk;  // first K/V row of this (b, h)
  float qd[E];                     // this lane's dimensions of q, pre-scaled
  if (active) IO::load_lane(A.q, qrow, lane, qd);
  else
#pragma unroll
    for (int e = 0; e < E; ++e) qd[e] = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qd[e] *= A.scale_log2;
    s_q[warp][lane * E + e] = qd[e];
  }
  __syncwarp();
  const float* sq = s_q[warp];
  // the block's 8 rows lie in one 64-row outer-tile row (8-aligned): same CSR ranges for all
  const int a = (blockIdx.x * kRowWarps) >> 6, r = i & 63;
  const int64_t mrow = (int64_t)hm * A.mask.ot_rows + a;
  // CSR ranges clamped to the arrays (a damaged mask cannot send the loops past them)
  const int fb = max(A.mask.full_row_ptr[mrow], 0), fe = (int)min((int64_t)A.mask.full_row_ptr[mrow + 1], A.mask.n_full);
  const int pb = max(A.mask.part_row_ptr[mrow], 0), pe = (int)min((int64_t)A.mask.part_row_ptr[mrow + 1], A.mask.n_part);

  float m = -INFINITY, l = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  // Staging of a round (tiles t0 .. t0 + 31): thread 4t + u (t < 32, u < 4) loads words 2u and
  // 2u + 1 of the block's row group of tile t0 + t (16 contiguous bytes; four threads cover
  // the tile's 64) and writes, for every row w of the block, byte w % 4 of the words' low
  // (w < 4) or high halves, as bits 16u .. 16u + 15 of row w's mask of that tile; warp 4 loads
  // the 32 columns. The next round's loads are issued before the current round is scored.
  const int wrow = 8 * (r >> 3);  // the row group of the inner-tile words (row w of the block: byte w % 8)
  const int tid = threadIdx.x;
  uint4 stw = make_uint4(0u, 0u, 0u, 0u);
  int stc = 0;
  auto stage_load = [&](int t0) {
    if (tid < 128) {
      const int tt = t0 + (tid >> 2);
      stw = tt < pe ? __ldg(reinterpret_cast<const uint4*>(A.mask.part_bitmap + (int64_t)tt * 64 + wrow) + (tid & 3))
                    : make_uint4(0u, 0u, 0u, 0u);
    } else if (warp == 4) {
      const int tt = t0 + lane;
      stc = tt < pe ? __ldg(A.mask.part_col_idx + tt) : 0;
    }
  };
  auto stage_store = [&](int buf) {
    if (tid < 128) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(s_mask[buf]) + tid;  // row w: + w * 128
      const uint32_t p01 = __byte_perm(stw.x, stw.z, 0x5140), p23 = __byte_perm(stw.x, stw.z, 0x7362);
      const uint32_t p45 = __byte_perm(stw.y, stw.w, 0x5140), p67 = __byte_perm(stw.y, stw.w, 0x7362);
      dst[0 * 128] = (uint16_t)p01;
      dst[1 * 128] = (uint16_t)(p01 >> 16);
      dst[2 * 128] = (uint16_t)p23;
      dst[3 * 128] = (uint16_t)(p23 >> 16);
      dst[4 * 128] = (uint16_t)p45;
      dst[5 * 128] = (uint16_t)(p45 >> 16);
      dst[6 * 128] = (uint16_t)p67;
      dst[7 * 128] = (uint16_t)(p67 >> 16);
    } else if (warp == 4) {
      s_col[buf][lane] = stc;
    }
  };
  // the first round's loads are in flight while the full tiles are scored
  if (pb < pe) stage_load(pb);

  // ---- full tiles: every key in range is valid
  for (int t = fb; active && t < fe; ++t) {
    // clamped into the mask like the part tiles' columns below
    const int col = (int)min((unsigned)A.mask.full_col_idx[t], (unsigned)A.mask.ot_cols - 1u);
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int64_t j0 = (int64_t)col * 64 + half * 32;
      if (j0 >= A.Lk) break;
      const int nk = (int)min((int64_t)32, A.Lk - j0);
      const bool valid = lane < nk;
      const float s = valid ? IO::dot(sq, A.k, kv0 + j0 + lane) : -INFINITY;
      const float m_new = fmaxf(m, warp_max(s));
      const float alpha = exp2f(m - m_new);  // m = -inf -> 0
      const float p = valid ? exp2f(s - m_new) : 0.f;
      l = l * alpha + warp_sum(p);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= alpha;
      if (nk == 32) {
#pragma unroll 8
        for (int src = 0; src < 32; ++src) {
          const float pj = __shfl_sync(0xffffffffu, p, src);
          float x[E];
          IO::load_lane(A.v, kv0 + j0 + src, lane, x);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, x[e], acc[e]);
        }
      } else {
        for (int src = 0; src < nk; ++src) {
          const float pj = __shfl_sync(0xffffffffu, p, src);
          float x[E];
          IO::load_lane(A.v, kv0 + j0 + src, lane, x);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, x[e], acc[e]);
        }
      }
      m = m_new;
    }
  }

  // ---- part tiles, 32 per round: lane l takes part tile t0 + l, whose 64-bit key mask for
  // this row (byte r % 8 of the row group's eight inner-tile words) the block has staged in
  // shared memory. The valid keys of the round are appended to the warp's list in shared
  // memory, and the list is scored NB keys at a time: every lane loads its dimensions of all
  // NB K and V rows at once, the NB dot products are reduced together (a transpose-reduce
  // that leaves key (lane >> (5 - LB)) of the batch on its lanes), and the running max, sum
  // and output take one update per batch.
  constexpr int LB = E == 2 ? 3 : 2;  // batch of NB = 2^LB keys: 8 at d = 64, 4 at d = 128
  constexpr int NB = 1 << LB;
  int* keys = s_keys[warp];
  const int kid = (lane >> (5 - LB)) & (NB - 1);  // key of a batch whose score this lane ends with
  auto batch = [&](int b0, int nb) {
    float kd[NB][E], vd[NB][E];
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      const int64_t j = kv0 + keys[b0 + (jj < nb ? jj : 0)];
      IO::load_lane(A.k, j, lane, kd[jj]);
      IO::load_lane(A.v, j, lane, vd[jj]);
    }
    float x[NB];
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) part = fmaf(qd[e], kd[jj][e], part);
      x[jj] = part;
    }
    // LB halving steps at offsets 16, 8, ...: a lane keeps the half of its keys selected by
    // its offset bit and adds the partner's copy of that half
#pragma unroll
    for (int st = 0; st < LB; ++st) {
      const int off = 16 >> st, half = NB >> (st + 1);
      const bool hi = lane & off;
#pragma unroll
      for (int k = 0; k < half; ++k) {
        const float send = hi ? x[k] : x[k + half];
        x[k] = (hi ? x[k + half] : x[k]) + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    float sc = x[0];
#pragma unroll
    for (int off = 16 >> LB; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
    if (kid >= nb) sc = -INFINITY;
    float mb = sc;
#pragma unroll
    for (int off = 32 >> LB; off < 32; off <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    const float m_new = fmaxf(m, mb);
    const float alpha = exp2f(m - m_new);  // m = -inf -> 0
    const float p = kid < nb ? exp2f(sc - m_new) : 0.f;
    float ps = p;
#pragma unroll
    for (int off = 32 >> LB; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= alpha;
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj << (5 - LB));
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, vd[jj][e], acc[e]);
    }
    m = m_new;
  };
  int nk = 0;  // keys waiting in the list (fewer than NB after every flush)
  if (pb < pe) stage_store(0);
  __syncthreads();
  int buf = 0;
  for (int t0 = pb; t0 < pe; t0 += 32) {  // the same rounds in every warp of the block
    const bool more = t0 + 32 < pe;
    if (more) stage_load(t0 + 32);
    if (active) {
      const uint64_t bits = s_mask[buf][warp][lane];  // 0 past the row's last part tile
      // column and key clamped into the mask: a damaged mask (sta_validate_mask finds it)
      // gives wrong values but no read outside K and V
      const int64_t base = (int64_t)min((unsigned)s_col[buf][lane], (unsigned)A.mask.ot_cols - 1u) * 64;
      // all keys of the round at once when they fit the list: each lane writes its tile's keys
      // at the prefix of the lanes below it (the same ascending order as one tile at a time)
      const int cnt = __popcll(bits);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (nk + total <= 72) {
        int pos = nk + incl - cnt;
        for (uint64_t bm = bits; bm; bm &= bm - 1) keys[pos++] = (int)min(base + (__ffsll(bm) - 1), (int64_t)A.Lk - 1);
        nk += total;
        __syncwarp();
        if (nk >= NB) {
          int b0 = 0;
          for (; nk - b0 >= NB; b0 += NB) batch(b0, NB);
          const int left = nk - b0;
          const int kl = lane < left ? keys[b0 + lane] : 0;
          __syncwarp();
          if (lane < left) keys[lane] = kl;
          nk = left;
          __syncwarp();
        }
      } else {
        for (unsigned nz = __ballot_sync(0xffffffffu, bits != 0ull); nz; nz &= nz - 1) {
          const int src = __ffs(nz) - 1;
          const uint64_t mb64 = __shfl_sync(0xffffffffu, bits, src);
          const int64_t bs = __shfl_sync(0xffffffffu, base, src);
          // lane c appends keys c and c + 32 of this tile when valid, in ascending order
          const uint32_t lo = (uint32_t)mb64, hi = (uint32_t)(mb64 >> 32);
          const uint32_t below = (1u << lane) - 1u;
          if ((lo >> lane) & 1u) keys[nk + __popc(lo & below)] = (int)min(bs + lane, (int64_t)A.Lk - 1);
          if ((hi >> lane) & 1u) keys[nk + __popc(lo) + __popc(hi & below)] = (int)min(bs + 32 + lane, (int64_t)A.Lk - 1);
          nk += __popc(lo) + __popc(hi);
          __syncwarp();
          if (nk < NB) continue;
          int b0 = 0;
          for (; nk - b0 >= NB; b0 += NB) batch(b0, NB);
          // the (fewer than NB) keys left over move to the front of the list
          const int left = nk - b0;
          const int kl = lane < left ? keys[b0 + lane] : 0;
          __syncwarp();
          if (lane < left) keys[lane] = kl;
          nk = left;
          __syncwarp();
        }
      }
    }
    // the other buffer was last read in the previous round, before that round's barrier
    if (more) stage_store(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
  if (!active) return;
  if (nk > 0) batch(0, nk);

  float out[E];
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = acc[e] * inv;
  IO::store_lane(A.o, o_row(A, bi, h, i), lane, out);
  if (A.lse && lane == 0) A.lse[qrow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace

sta_status launch_mha_row(const MhaArgs& a, cudaStream_t st) {
  const dim3 grid((unsigned)cdiv(a.Lq, kRowWarps), (unsigned)(a.B * a.n_ranks));
  const dim3 block(kRowWarps * 32);
  if (a.dtype == STA_BF16) {
    if (a.d == 64) mha_row_kernel<64, true><<<grid, block, 0, st>>>(a);
    else mha_row_kernel<128, true><<<grid, block, 0, st>>>(a);
  } else {
    if (a.d == 64) mha_row_kernel<64, false><<<grid, block, 0, st>>>(a);
    else mha_row_kernel<128, false><<<grid, block, 0, st>>>(a);
  }
  STA_LAUNCH_CHECK();
  return STA_OK;
}

}  // namespace sta
