// Block-wise masked MHA kernel for sm_103a (STOF, デュアルカーネル戦略 / ブロック方向カーネル:
// Q, K, V split into sub-blocks, shared memory plus asynchronous copies overlapping
// transfer and compute), rebuilt on Blackwell's TMA + tcgen05/TMEM:
//
//  * one CTA per (128-row query tile, batch x head[, chunk of the key-tile list]). The tile
//    spans outer-tile rows 2t and 2t+1; its key loop runs over the union of their non-empty
//    outer-tile columns (copied from the encoded mask's tile lists, or merged here from the
//    CSR arrays), each half masked by its own class (empty / full / part);
//  * warp 0 loads K tiles of 64 keys by TMA (128-byte swizzle) into a ring of stages, warp 6
//    the V tiles and the part-tile bitmaps; Q is loaded once;
//  * warp 1 owns TMEM (256 columns: two S buffers of 64 columns, P buffers, the O
//    accumulator) and issues S = Q K^T (M=128, N=64, K=d, both operands from shared memory);
//    warp 7 issues O += P V (M=128, N=d, K=64, P read from TMEM). A tcgen05.mma costs its
//    issuing thread about 60 cycles, so the two products have their own issuing threads;
//    completion goes to mbarriers through tcgen05.commit;
//  * warps 2..5 run the softmax, one query row per thread: load the S row from TMEM, apply
//    the part-tile bitmap (byte r%8 of the 8 inner-tile words of the row, staged in shared
//    memory), online max with lazy rescaling (O in TMEM is rescaled only when the running
//    max grows by more than 2^8, keeping every exponential below 256), exponentials in base
//    2 on the MUFU unit, score scaling and sums on packed fp32 pairs, and P rounded to bf16
//    into TMEM, where the PV MMA reads it; at the end O / l goes out as bf16 through the idle
//    Q buffer and a TMA store (or as an fp32 partial when the key list is split), LSE as fp32;
//  * two CTAs share an SM (256 TMEM columns and < 114 KB of shared memory each), so one
//    CTA's softmax overlaps the other's MMAs and loads.
// Empty outer tiles are skipped entirely ("skip, don't reset": 問題定義), full tiles are
// never masked, iterative tiling over key blocks and one fused loop for max, sum and PV
// follow Cleave's 複数リダクションのスケジューリング; the split of the key loop with a
// log-sum-exp merge is Cleave's Split演算子によるSplit-Kの対応.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kBM = 128;       // query rows per CTA
constexpr int kBN = 64;        // keys per tile (one outer tile)
constexpr int kThreads = 256;  // warp 0 K loads, warp 1 QK MMAs, warps 2..5 softmax, warp 6 V loads, warp 7 PV MMAs
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum : int { kEmpty = -1, kFull = -2 };

template <int D>
struct BlkCfg {
  static constexpr int KH = D / 64;                 // 128-byte column blocks of a row
  static constexpr int STAGES = D == 64 ? 5 : 2;
  // With two stages the K and V rings move in step with the S/P buffers: stage j & 1 is
  // free again exactly when QK(j) (K) or PV(j) (V) has completed, so the loaders wait on
  // s_full / pv_done and the MMA issuers commit once per tile instead of two or three times.
  static constexpr bool PAIR_RING = STAGES == 2;
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int KV_BYTES = kBN * D * 2;      // one K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BM = OFF_V + STAGES * KV_BYTES;  // per stage: part bitmaps of both halves (2 x 512 B)
  // column list of this CTA's query tile, laid out like a tile-list slot of the encoded
  // mask: 16-byte header (count), uint16 col[Cp], int32 kind_a[Cp], int32 kind_b[Cp]
  static constexpr int OFF_LIST = OFF_BM + STAGES * 1024;
  static constexpr int TMEM_COLS = 256;
  // TMEM columns: S buffers at 0 and 64. With d = 64 there is room for P buffers of their
  // own (columns 128 and 160) and O at 192, so that an S buffer is free again as soon as
  // the softmax has read it; with d = 128, O takes columns 128..255 and P(j) is written
  // over the first 32 columns of S(j), which then stays busy until PV(j) has completed.
  static constexpr bool SEP_P = D == 64;
  static constexpr int S_COL = 0;
  static constexpr int P_COL = SEP_P ? 128 : 0;
  static constexpr int O_COL = SEP_P ? 192 : 128;
  static constexpr uint32_t IDESC_QK = umma_idesc_bf16(kBM, kBN, 0, 0);
  static constexpr uint32_t IDESC_PV = umma_idesc_bf16(kBM, D, 0, 1);
};

__host__ __device__ inline int list_cols_padded(int C) { return (C + 7) / 8 * 8; }
__host__ __device__ inline int list_slot_bytes(int C) { return 16 + 10 * list_cols_padded(C); }

template <int D>
size_t blk_smem_bytes(int C) {
  using Cfg = BlkCfg<D>;
  return 1024 + Cfg::OFF_LIST + (size_t)list_slot_bytes(C);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    mha_block_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const MhaArgs A, const MhaSplit P) {
  using Cfg = BlkCfg<D>;
  constexpr int ST = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // Per buffer b (tile j uses b = j & 1): s_full[b] S(j) is in TMEM; p_full[b] P(j) is in TMEM
  // (all 128 softmax threads); pv_done[b] PV(j) has completed (committed by the MMA warp);
  // s_free[b] the S buffer may be overwritten: read by all 128 softmax threads (separate P
  // buffers) or PV(j) completed (P over S).
  // K stage s is released as soon as its QK has completed (k_empty), V stage s (with the
  // part-tile bitmaps, which the softmax reads) once its PV has completed (v_empty).
  __shared__ __align__(8) uint64_t q_full, list_full, k_full[ST], v_full[ST], k_empty[ST], v_empty[ST], s_full[2],
      s_free[2], p_full[2], pv_done[2];
  __shared__ int s_ncols;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_rowptr[8];         // full/part row_ptr pairs of outer-tile rows 2qt and 2qt+1
  __shared__ uint32_t s_colbits[32];  // bit c: column c is non-empty in either row (C <= 1024)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Query tiles in reverse order: the hardware starts blocks x-fastest, and in the common
  // long-sequence masks (causal, causal windows with global columns) later query tiles
  // carry more key tiles, so the longest items start first.
  const int qt = gridDim.x - 1 - blockIdx.x;
  // blockIdx.y enumerates (head rank, batch, chunk): the heaviest heads' tiles are dispatched first
  const int y = blockIdx.y;
  int rank, n_split, off;
  if (P.uniform_s > 0) {
    n_split = P.uniform_s;
    rank = y / (A.B * n_split);
    off = y - rank * A.B * n_split;
  } else {
    int lo = 0, hi = A.n_ranks;  // P.ybase[lo] <= y < P.ybase[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (P.ybase[mid] <= y) lo = mid;
      else hi = mid;
    }
    rank = lo;
    n_split = P.s[lo];
    off = y - P.ybase[lo];
  }
  const int bi = off / n_split, chunk = off - bi * n_split;
  const int h = A.hmap.order[rank];
  const int64_t bh = (int64_t)bi * A.H + h;
  const int hm = A.hmap.m[h];
  const int R = A.mask.ot_rows, C = A.mask.ot_cols;

  // 1024-byte aligned dynamic shared memory (128-byte swizzle atoms).
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int Cp = list_cols_padded(C);
  uint8_t* lbase = smem + Cfg::OFF_LIST;
  uint16_t* cols = reinterpret_cast<uint16_t*>(lbase + 16);
  int32_t* kind_a = reinterpret_cast<int32_t*>(lbase + 16 + 2 * Cp);
  int32_t* kind_b = kind_a + Cp;
  const bool have_lists = A.mask.tile_lists != nullptr;

  // ---- setup: barriers, TMEM, and the column list: the union of the two outer-tile rows'
  // non-empty columns, copied from the encoded mask's tile lists when present (one bulk
  // copy), else built here from the CSR arrays. The row pointers / the list copy are
  // issued first so that their latency overlaps the barrier and TMEM setup.
  int rp = 0;
  if (!have_lists && threadIdx.x < 8) {
    const int a = 2 * qt + (threadIdx.x >> 2);  // threads 0..3: row 2qt, 4..7: row 2qt+1
    if (a < R) {
      const int64_t r = (int64_t)hm * R + a + (threadIdx.x & 1);
      rp = (threadIdx.x & 2) ? A.mask.part_row_ptr[r] : A.mask.full_row_ptr[r];
    }
  }
  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&list_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], Cfg::SEP_P ? 128 : 1);
      mbar_init(&p_full[s], 128);
      mbar_init(&pv_done[s], 1);
    }
    fence_mbar_init();
    if (have_lists) {
      const int sb = list_slot_bytes(C);
      mbar_arrive_expect_tx(&list_full, (uint32_t)sb);
      bulk_g2s(lbase, A.mask.tile_lists + ((int64_t)hm * ((R + 1) / 2) + qt) * sb, (uint32_t)sb, &list_full);
    }
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  // column-indexed kinds of both rows while the list is built here: scratch in the V stages,
  // which no load has touched yet
  int32_t* infoA = reinterpret_cast<int32_t*>(smem + Cfg::OFF_V);
  int32_t* infoB = infoA + C;
  if (!have_lists) {
    for (int c = threadIdx.x; c < C; c += kThreads) {
      infoA[c] = kEmpty;
      infoB[c] = kEmpty;
    }
    if (threadIdx.x < 8) s_rowptr[threadIdx.x] = rp;
  }
  __syncthreads();
  // Q does not depend on the column list: start its load now, under the list's latency.
  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    mbar_arrive_expect_tx(&q_full, Cfg::Q_BYTES);
#pragma unroll
    for (int kh = 0; kh < Cfg::KH; ++kh)
      tma_load_3d(smem + Cfg::OFF_Q + kh * (kBM * 128), &tm_q, kh * 64, qt * kBM, (int)bh, &q_full);
  }
  int n_cols;  // size of the union
  if (have_lists) {
    if (threadIdx.x == 0) {
      const int n = mbar_wait(&list_full, 0, A.err, 0x20f) ? *reinterpret_cast<const int*>(lbase) : 0;
      s_ncols = n < 0 ? 0 : (n > C ? C : n);  // a damaged list cannot index past the buffers
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    n_cols = s_ncols;
  } else {
    {
      // CSR ranges clamped to the arrays and columns checked against C: a damaged mask
      // reports 0x213 instead of reaching past the buffers
      const int64_t nf = A.mask.n_full, np = A.mask.n_part;
      auto lo = [](int v) { return v < 0 ? 0 : v; };
      const int fA0 = lo(s_rowptr[0]), fA1 = (int)min((int64_t)s_rowptr[1], nf);
      const int pA0 = lo(s_rowptr[2]), pA1 = (int)min((int64_t)s_rowptr[3], np);
      const int fB0 = lo(s_rowptr[4]), fB1 = (int)min((int64_t)s_rowptr[5], nf);
      const int pB0 = lo(s_rowptr[6]), pB1 = (int)min((int64_t)s_rowptr[7], np);
      auto put = [&](int32_t* info, int col, int32_t kind) {
        if ((unsigned)col < (unsigned)C) info[col] = kind;
        else record_error(A.err, 0x213);
      };
      for (int t = fA0 + threadIdx.x; t < fA1; t += kThreads) put(infoA, A.mask.full_col_idx[t], kFull);
      for (int t = pA0 + threadIdx.x; t < pA1; t += kThreads) put(infoA, A.mask.part_col_idx[t], t);
      for (int t = fB0 + threadIdx.x; t < fB1; t += kThreads) put(infoB, A.mask.full_col_idx[t], kFull);
      for (int t = pB0 + threadIdx.x; t < pB1; t += kThreads) put(infoB, A.mask.part_col_idx[t], t);
    }
    __syncthreads();
    // Ascending list of the non-empty columns, built by all warps: one ballot per 32 columns,
    // a prefix over the (at most 32) words, then every set bit written at its rank.
    const int nwords = (C + 31) >> 5;
    for (int wd = warp; wd < nwords; wd += kThreads / 32) {
      const int c = wd * 32 + lane;
      const unsigned b = __ballot_sync(0xffffffffu, c < C && (infoA[c] != kEmpty || infoB[c] != kEmpty));
      if (lane == 0) s_colbits[wd] = b;
    }
    __syncthreads();
    const unsigned wl = lane < nwords ? s_colbits[lane] : 0u;
    int incl = __popc(wl);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - __popc(wl);
    for (int wd = warp; wd < nwords; wd += kThreads / 32) {
      const unsigned b = __shfl_sync(0xffffffffu, wl, wd);
      const int base = __shfl_sync(0xffffffffu, excl, wd);
      const int c = wd * 32 + lane;
      if ((b >> lane) & 1u) {
        const int pos = base + __popc(b & ((1u << lane) - 1u));
        cols[pos] = (uint16_t)c;
        kind_a[pos] = infoA[c];
        kind_b[pos] = infoB[c];
      }
    }
    n_cols = __shfl_sync(0xffffffffu, incl, 31);
    tc_fence_before();
    __syncthreads();  // the list is complete and the scratch in the V stages is dead
    tc_fence_after();
  }
  // this CTA's chunk of the column list (n_cols <= 1024, n_split <= 1024: no overflow)
  const int jb = chunk * n_cols / n_split;
  const int ntiles = (chunk + 1) * n_cols / n_split - jb;
  const uint16_t* lst = cols + jb;
  const int32_t* ka = kind_a + jb;
  const int32_t* kb = kind_b + jb;
  const uint32_t tmem = s_tmem_base;
  const uint32_t sQ = smem_u32(smem + Cfg::OFF_Q);
  const uint32_t sK = smem_u32(smem + Cfg::OFF_K);
  const uint32_t sV = smem_u32(smem + Cfg::OFF_V);

  if (warp == 0) {
    // ------------------------------------------------------------ K loads
    if (lane == 0 && ntiles == 0) mbar_wait(&q_full, 0, A.err, 0x20b);  // drain the Q load before exiting
    if (lane == 0 && ntiles > 0) {
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % ST;
        if (!mbar_wait(Cfg::PAIR_RING ? &s_full[s] : &k_empty[s], ((j / ST) & 1u) ^ 1u, A.err, 0x201)) break;
        mbar_arrive_expect_tx(&k_full[s], Cfg::KV_BYTES);
#pragma unroll
        for (int kh = 0; kh < Cfg::KH; ++kh)
          tma_load_3d(smem + Cfg::OFF_K + s * Cfg::KV_BYTES + kh * (kBN * 128), &tm_k, kh * 64, lst[j] * kBN,
                      (int)bh, &k_full[s]);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ V loads (+ part-tile bitmaps)
    if (lane == 0 && ntiles > 0) {
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % ST;
        if (!mbar_wait(Cfg::PAIR_RING ? &pv_done[s] : &v_empty[s], ((j / ST) & 1u) ^ 1u, A.err, 0x20c)) break;
        const int col = lst[j];
        // (a part index past the mask's part tiles, only possible in a damaged list, fetches nothing)
        const int ia = ka[j] < A.mask.n_part ? ka[j] : kEmpty, ib = kb[j] < A.mask.n_part ? kb[j] : kEmpty;
        mbar_arrive_expect_tx(&v_full[s], Cfg::KV_BYTES + (ia >= 0 ? 512 : 0) + (ib >= 0 ? 512 : 0));
#pragma unroll
        for (int kh = 0; kh < Cfg::KH; ++kh)
          tma_load_3d(smem + Cfg::OFF_V + s * Cfg::KV_BYTES + kh * (kBN * 128), &tm_v, kh * 64, col * kBN, (int)bh,
                      &v_full[s]);
        // the 64 inner-tile words of each half's part tile, for the softmax threads
        if (ia >= 0) bulk_g2s(smem + Cfg::OFF_BM + s * 1024, A.mask.part_bitmap + (int64_t)ia * 64, 512, &v_full[s]);
        if (ib >= 0)
          bulk_g2s(smem + Cfg::OFF_BM + s * 1024 + 512, A.mask.part_bitmap + (int64_t)ib * 64, 512, &v_full[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK MMA issuer
    // (a tcgen05.mma costs its issuing thread ~60 cycles: QK and PV are issued by two
    // threads so that their issue latencies overlap)
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(&q_full, 0, A.err, 0x202);
      // descriptors of Q and of K stage 0; every other operand is a fixed offset from them
      const uint64_t a0 = umma_sdesc_sw128(sQ, 16, 1024), b0 = umma_sdesc_sw128(sK, 16, 1024);
      uint64_t* s_reuse = Cfg::SEP_P ? s_free : (Cfg::PAIR_RING ? pv_done : s_free);
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j % ST, sb = j & 1;
        if (!mbar_wait(&k_full[s], (j / ST) & 1, A.err, 0x205)) break;
        if (j >= 2 && !mbar_wait(&s_reuse[sb], ((j - 2) >> 1) & 1, A.err, 0x206)) break;
        tc_fence_after();
        const uint64_t bs = b0 + (uint64_t)((s * Cfg::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int kh = kk >> 2, ko = (kk & 3) * 32;
          umma_bf16(tmem + Cfg::S_COL + sb * kBN, a0 + (uint64_t)((kh * (kBM * 128) + ko) >> 4),
                    bs + (uint64_t)((kh * (kBN * 128) + ko) >> 4), Cfg::IDESC_QK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[sb]);
        if (!Cfg::PAIR_RING) umma_commit(&k_empty[s]);
      }
    }
  } else if (warp == 7) {
    // ------------------------------------------------------------ PV MMA issuer
    if (lane == 0) {
      const uint64_t v0 = umma_sdesc_sw128(sV, kBN * 128, 1024);
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % ST, sb = j & 1;
        if (!mbar_wait(&p_full[sb], (j >> 1) & 1, A.err, 0x203)) break;
        if (!mbar_wait(&v_full[s], (j / ST) & 1, A.err, 0x204)) break;
        tc_fence_after();
        const uint64_t vs = v0 + (uint64_t)((s * Cfg::KV_BYTES) >> 4);
        const uint32_t p_tmem = Cfg::SEP_P ? tmem + Cfg::P_COL + sb * 32 : tmem + Cfg::S_COL + sb * kBN;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_bf16_ts(tmem + Cfg::O_COL, p_tmem + kk * 8, vs + (uint64_t)((kk * 2048) >> 4), Cfg::IDESC_PV,
                       (j > 0 || kk > 0) ? 1u : 0u);
        if (!Cfg::PAIR_RING) umma_commit(&v_empty[s]);
        umma_commit(&pv_done[sb]);
        if (!Cfg::SEP_P && !Cfg::PAIR_RING) umma_commit(&s_free[sb]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;             // TMEM lane quadrant of this warp
    const int m = qd * 32 + lane;        // row within the tile
    const int half = m >> 6, r = m & 63;
    const int32_t* info = half ? kb : ka;
    const uint32_t t_row = tmem + ((uint32_t)(qd * 32) << 16);
    const float c = A.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1, st = j % ST;
      const int inf = info[j];  // the same for every row of this warp (one half per warp)
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, A.err, 0x207)) { ok = false; break; }
      tc_fence_after();
      float s[64];
      tmem_ld64_sync(t_row + Cfg::S_COL + sb * kBN, s);
      if (Cfg::SEP_P) {  // S(j) is in registers: its buffer may take S(j+2)
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
      }
      uint32_t pk[32];
      float alpha = 1.f;
      bool need = false;
      if (inf == kEmpty) {
        // no valid key of this tile for these rows: their P row is zero, m and l unchanged
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = 0u;
      } else {
        if (inf >= 0) {  // part tile: apply this row's 64-bit mask from the inner-tile words
          if (!mbar_wait(&v_full[st], (j / ST) & 1, A.err, 0x20a)) { ok = false; break; }
          const uint64_t* words = reinterpret_cast<const uint64_t*>(smem + Cfg::OFF_BM + st * 1024 + half * 512);
          const uint64_t bits = part_row_bits(words, r);
          const uint32_t lo = (uint32_t)bits, hi = (uint32_t)(bits >> 32);
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            s[x] = (lo & (1u << x)) ? s[x] : -INFINITY;
            s[x + 32] = (hi & (1u << x)) ? s[x + 32] : -INFINITY;
          }
        }
        float m8[8];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          m8[y] = fmax3(s[y], s[y + 8], s[y + 16]);
          m8[y] = fmax3(m8[y], s[y + 24], s[y + 32]);
          m8[y] = fmax3(m8[y], s[y + 40], s[y + 48]);
          m8[y] = fmaxf(m8[y], s[y + 56]);
        }
        const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * c;
        if (mx > m_ref + kRescaleThreshold) {
          if (m_ref != -INFINITY) {
            alpha = ex2(m_ref - mx);
            need = true;
          }
          m_ref = mx;
        }
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        // exponent arguments and the row sum on packed fp32 pairs (one instruction per pair)
        const uint64_t c2 = f32x2_pack(c, c), nm2 = f32x2_pack(neg_m, neg_m);
        uint64_t l2[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) l2[x] = 0ull;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          float a0, a1;
          f32x2_unpack(f32x2_fma(f32x2_pack(s[2 * x], s[2 * x + 1]), c2, nm2), a0, a1);
          const float p0 = ex2(a0), p1 = ex2(a1);
          l2[x & 3] = f32x2_add(l2[x & 3], f32x2_pack(p0, p1));
          pk[x] = pack_bf16x2(p0, p1);
        }
        float lp[8];
#pragma unroll
        for (int x = 0; x < 4; ++x) f32x2_unpack(l2[x], lp[2 * x], lp[2 * x + 1]);
        l = l * alpha + (((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7])));
      }
      if (__any_sync(0xffffffffu, need)) {
        // O may only be rescaled once PV(j-1) has completed
        if (j >= 1 && !mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, A.err, 0x208)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32_sync(t_row + Cfg::O_COL + c0, o);
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] *= alpha;
          tmem_st32_sync(t_row + Cfg::O_COL + c0, reinterpret_cast<const uint32_t*>(o));
        }
      }
      if (Cfg::SEP_P) {
        // P(j), bf16 pairs, into P buffer j & 1 once PV(j-2) has read it
        if (j >= 2 && !mbar_wait(&pv_done[sb], ((j - 2) >> 1) & 1, A.err, 0x20e)) { ok = false; break; }
        tc_fence_after();
        tmem_st32_sync(t_row + Cfg::P_COL + sb * 32, pk);
      } else {
        // P(j), bf16 pairs, over the first 32 columns of S(j) (already in registers)
        tmem_st32_sync(t_row + Cfg::S_COL + sb * kBN, pk);
      }
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // ---- epilogue: O / l (bf16) and LSE
    const int row = qt * kBM + m;
    if (ok && ntiles > 0) ok = mbar_wait(&pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, A.err, 0x209);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float row_lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    if (n_split == 1) {
      // O / l as bf16 into the Q buffer (idle once the last QK has completed), in the
      // 128-byte-swizzled layout of the O tensor map, then one TMA store per 64 columns;
      // rows past Lq fall outside the tensor map and are not written.
      uint8_t* so = smem + Cfg::OFF_Q;
      // with no tile the Q load may still be landing in that buffer
      if (ntiles == 0 && !mbar_wait(&q_full, 0, A.err, 0x20d)) ok = false;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        if (ntiles > 0) {
          tmem_ld32_sync(t_row + Cfg::O_COL + c0, o);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0.f;
        }
#pragma unroll
        for (int x = 0; x < 32; x += 8) {
          const uint4 w = make_uint4(pack_bf16x2(o[x] * inv, o[x + 1] * inv), pack_bf16x2(o[x + 2] * inv, o[x + 3] * inv),
                                     pack_bf16x2(o[x + 4] * inv, o[x + 5] * inv), pack_bf16x2(o[x + 6] * inv, o[x + 7] * inv));
          const int kh = c0 >> 6, q16 = ((c0 & 63) + x) >> 3;  // 16-byte chunk within the 128-byte row
          *reinterpret_cast<uint4*>(so + kh * (kBM * 128) + m * 128 + ((q16 ^ (m & 7)) << 4)) = w;
        }
      }
      if (row < A.Lq && A.lse) A.lse[bh * A.Lq + row] = row_lse;
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (m == 0) {
#pragma unroll
        for (int kh = 0; kh < Cfg::KH; ++kh) {
          if (A.o_tokens)  // map (d, H, Lq, B): one head's 128 rows, rows H*d apart
            tma_store_4d(&tm_o, so + kh * (kBM * 128), kh * 64, (int)(bh % A.H), qt * kBM, (int)(bh / A.H));
          else
            tma_store_3d(&tm_o, so + kh * (kBM * 128), kh * 64, qt * kBM, (int)bh);
        }
        bulk_commit_group();
        bulk_wait_group_read0();  // shared memory is released when the CTA exits
      }
    } else {
      // normalised fp32 partial of this chunk and its LSE (an empty chunk gives 0 and -inf)
      const int64_t prow = (int64_t)y * A.Lq + row;
      float* po = P.part_o + prow * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        if (ntiles > 0) {
          tmem_ld32_sync(t_row + Cfg::O_COL + c0, o);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0.f;
        }
        if (row < A.Lq) {
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(po + c0 + x) = make_float4(o[x] * inv, o[x + 1] * inv, o[x + 2] * inv, o[x + 3] * inv);
        }
      }
      if (row < A.Lq) P.part_lse[prow] = row_lse;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// Log-sum-exp merge of the chunks of split heads: one warp per (rank, batch, query
// row); O (bf16) and LSE go to the caller's arrays.
template <int D>
__global__ void __launch_bounds__(256) mha_split_merge_kernel(const MhaArgs A, const MhaSplit P) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= A.Lq) return;
  const int rank = blockIdx.y / A.B, bi = blockIdx.y - rank * A.B;
  const int ns = P.uniform_s > 0 ? P.uniform_s : P.s[rank];
  const int y0 = (P.uniform_s > 0 ? rank * A.B * ns : P.ybase[rank]) + bi * ns;
  const int64_t pr = (int64_t)y0 * A.Lq + row;
  float out[E];
  const float L = merge_row<E>(P.part_o + pr * D, (size_t)A.Lq * D, P.part_lse + pr, (size_t)A.Lq, ns, lane, out);
  const int h = A.hmap.order[rank];
  __nv_bfloat16* op = static_cast<__nv_bfloat16*>(A.o) + o_row(A, bi, h, row) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) *reinterpret_cast<uint32_t*>(op + e) = pack_bf16x2(out[e], out[e + 1]);
  if (A.lse && lane == 0) A.lse[((int64_t)bi * A.H + h) * A.Lq + row] = L;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [B*H, L, d] bf16 viewed as a 3-D tensor (d, L, B*H); box (64, rows, 1), 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, int d, int L, int BH, int rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// O as [B, Lq, H, d] bf16 viewed as a 4-D tensor (d, H, Lq, B); box (64, 1, rows, 1), whose
// shared-memory image is that of the 3-D box (64, rows, 1) above.
bool make_tmap_tokens(CUtensorMap* m, const void* base, int d, int H, int L, int B, int rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)L * H * d * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
sta_status launch_t(const MhaArgs& a, const MhaSplit& p, cudaStream_t st) {
  CUtensorMap tq, tk, tv, to;
  const int BH = a.B * a.H;
  const bool o_ok = a.o_tokens ? make_tmap_tokens(&to, a.o, D, a.H, a.Lq, a.B, kBM) : make_tmap(&to, a.o, D, a.Lq, BH, kBM);
  if (!make_tmap(&tq, a.q, D, a.Lq, BH, kBM) || !make_tmap(&tk, a.k, D, a.Lk, BH, kBN) ||
      !make_tmap(&tv, a.v, D, a.Lk, BH, kBN) || !o_ok) {
    note_cuda_error(cudaErrorInvalidValue);  // tensor-map encoding refused
    return STA_ERR_CUDA;
  }
  const size_t smem = blk_smem_bytes<D>(a.mask.ot_cols);
  auto kern = mha_block_kernel<D>;
  STA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const dim3 grid((unsigned)cdiv(a.Lq, kBM), (unsigned)p.n_y);
  kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, to, a, p);
  STA_LAUNCH_CHECK();
  if (p.n_split_ranks > 0) {
    const dim3 mgrid((unsigned)cdiv(a.Lq, 8), (unsigned)(p.n_split_ranks * a.B));
    mha_split_merge_kernel<D><<<mgrid, 256, 0, st>>>(a, p);
    STA_LAUNCH_CHECK();
  }
  return STA_OK;
}

}  // namespace

bool block_kernel_supports(int d, int Lk, int dtype) {
  return dtype == STA_BF16 && (d == 64 || d == 128) && cdiv(Lk, 64) <= kMaxTileListCols;
}

sta_status launch_mha_block(const MhaArgs& a, const MhaSplit& p, cudaStream_t st) {
  if (!block_kernel_supports(a.d, a.Lk, a.dtype)) return STA_ERR_UNSUPPORTED;
  if (p.n_split_ranks > 0 && (!p.part_o || !p.part_lse)) return STA_ERR_WORKSPACE;
  return a.d == 64 ? launch_t<64>(a, p, st) : launch_t<128>(a, p, st);
}

// Split planner. Without an explicit count, the work of an item is its key
// tiles plus kSetupTiles for the prologue (union build, first loads) and
// epilogue; an item longer than the average work of a resident CTA slot (two
// per SM) by more than a factor of two would outlast the rest of the grid, so it
// is cut into chunks of about that length (at least kMinChunk tiles). Shorter
// items stay whole: a chunk costs another prologue and a merged partial.
sta_status plan_mha_split(const MhaArgs& a, const int64_t* mask_head_tiles, int num_splits, int device, MhaSplit& p) {
  constexpr int kMinChunk = 16;
  constexpr int kMaxAutoSplit = 32;
  constexpr double kSetupTiles = 4.0;
  const int H = a.n_ranks, B = a.B;  // the ranks of this launch
  p.part_o = nullptr;
  p.part_lse = nullptr;
  if (num_splits > 0) {
    for (int r = 0; r < H; ++r) p.s[r] = (uint16_t)num_splits;
  } else if (!mask_head_tiles) {
    for (int r = 0; r < H; ++r) p.s[r] = 1;
  } else {
    int sms = 0;
    if (device < 0) STA_CUDA_TRY(cudaGetDevice(&device));
    STA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
    const int64_t nqt = cdiv(a.Lq, kBM);
    const int R = a.mask.ot_rows;
    double w[kMaxHeads], W = 0.0;
    for (int r = 0; r < H; ++r) {
      // key tiles of one 128-row item ~ the mask head's non-empty tiles per outer-tile row
      w[r] = (double)cdiv(mask_head_tiles[a.hmap.m[a.hmap.order[r]]], R);
      W += (double)B * (double)nqt * (w[r] + kSetupTiles);
    }
    const double target = fmax((double)kMinChunk, W / (2.0 * (double)(sms > 0 ? sms : 1)));
    for (int r = 0; r < H; ++r) {
      // an item within twice the target still ends in time: only longer ones are cut
      int sr = w[r] > 2.0 * target ? (int)ceil(w[r] / target) : 1;
      sr = sr < 1 ? 1 : (sr > kMaxAutoSplit ? kMaxAutoSplit : sr);
      if (r > 0 && sr > p.s[r - 1]) sr = p.s[r - 1];  // split ranks stay a prefix of the launch order
      p.s[r] = (uint16_t)sr;
    }
  }
  int64_t y = 0;
  p.n_split_ranks = 0;
  bool uniform = true;
  for (int r = 0; r < H; ++r) {
    p.ybase[r] = (int32_t)y;
    y += (int64_t)B * p.s[r];
    if (y > 65535) return STA_ERR_UNSUPPORTED;  // grid.y limit
    if (p.s[r] > 1) p.n_split_ranks = r + 1;
    uniform = uniform && p.s[r] == p.s[0];
  }
  p.ybase[H] = (int32_t)y;
  p.n_y = (int)y;
  p.uniform_s = uniform ? p.s[0] : 0;
  return STA_OK;
}

size_t mha_split_workspace_bytes(const MhaArgs& a, const MhaSplit& p) {
  if (p.n_split_ranks == 0) return 0;
  const size_t rows = (size_t)p.ybase[p.n_split_ranks] * (size_t)a.Lq;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(rows * (size_t)a.d * sizeof(float)) + al(rows * sizeof(float));
}

}  // namespace sta
