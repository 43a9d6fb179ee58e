// Split-KV GQA decode and log-sum-exp merge (Cleave, the Split operator: a split count s
// parallelises the reduction over the KV tokens; each chunk is attended on its own and the
// partial softmax results are merged by their log-sum-exp).
//
// Decode kernel: persistent-style CTAs, each owning a list of KV segments (request r, token
// range [a, b)) and a block of HB kv heads. One producer warp streams K/V tiles (16 tokens x HB
// heads x d, bf16) from HBM into a ring of shared-memory stages with 1-D bulk copies, one per
// token row, completing on mbarriers; packed and paged K/V differ only in where a row is read
// from. HB consumer warps (one per kv head) compute on the tensor cores with
// mma.sync.m16n8k16 (bf16 operands, fp32 accumulators): the warp's G <= 16 query heads are the
// M of the MMA (rows G..15 are zero), S[16 x 16 tokens] = Q K^T takes d / 16 k-steps over K rows
// read by ldmatrix, the fp32 online softmax runs on the accumulator fragments (a quad of
// lanes holds a row), P passes from the S fragments straight into the A fragments of P V, and
// O[16 x d] accumulates in registers over V rows read by ldmatrix .trans. Token rows are
// padded by 16 bytes in shared memory so that the eight rows one ldmatrix reads fall in
// distinct banks. A segment that covers its whole request writes O (bf16) and LSE directly;
// otherwise it writes a normalised fp32 partial and its LSE, merged afterwards.
//
// Split plans: mode 0 cuts the concatenated token stream [0, T) into equal ranges, one per
// CTA (balanced work whatever the length mix; partial slot of (CTA x, request r) = x + r,
// unique because both grow along the stream); mode 1 cuts every request into s chunks of
// ceil(len / s) keys (slot r*s + c).
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

enum : int { kFirst = 1, kLast = 2, kFinal = 4, kDone = 8 };

struct StageInfo {
  int r, tok0, n, flags, slot;
};

constexpr int kNT = 16;  // tokens per tile

template <int G, int D, int HB>
struct DecCfg {
  static constexpr int ROW = HB * D * 2 + 16;  // padded bytes of one token's HB heads
  static constexpr int TILE = kNT * ROW;       // K or V part of one stage
  static constexpr int STAGES = 3;
  static constexpr int SMEM = STAGES * 2 * TILE;
  static constexpr int THREADS = (HB + 1) * 32;
  static_assert(SMEM <= 110 * 1024, "two CTAs per SM");
};

// Largest r with indptr[r] <= t (indptr non-decreasing, indptr[0] = 0 <= t).
__device__ __forceinline__ int find_request(const int32_t* indptr, int n_req, int t) {
  int lo = 0, hi = n_req;  // answer in [0, n_req]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Request r's token range from the device copy of kv_indptr, kept non-decreasing and inside
// [0, T] (the host copy's total): a device copy that disagrees with the host's reports 0x111
// and cannot send a read past K / V.
__device__ __forceinline__ void request_range(const DecodeArgs& A, int r, int& rb, int& re) {
  rb = __ldg(A.kv_indptr + r);
  re = __ldg(A.kv_indptr + r + 1);
  if (rb < 0 || re < rb || re > A.T) {
    record_error(A.err, 0x111);
    rb = min(max(rb, 0), A.T);
    re = min(max(re, rb), A.T);
  }
}

// Page table lookups of the paged layout, made by the producer warp: lane l holds the page
// number of ordinal base + l of request r (warp-uniform bookkeeping; reloaded when a lookup
// leaves the window of 32 ordinals).
struct PageCache {
  int r = -1, base = 0, page = 0, rb = 0, pb = 0, pe = 0;

  __device__ void load(const DecodeArgs& A, int req, int b, int lane) {
    if (req != r) {
      r = req;
      int re_unused;
      request_range(A, req, rb, re_unused);  // the same clamped start the token ranges use
      pb = __ldg(A.page_indptr + req);
      pe = __ldg(A.page_indptr + req + 1);
    }
    base = b;
    const int o = pb + b + lane;
    page = o < pe ? __ldg(A.page_indices + o) : 0;
  }
  // first token of request req
  __device__ int start(const DecodeArgs& A, int req, int lane) {
    if (req != r) load(A, req, 0, lane);
    return rb;
  }
  // page of this lane's ordinal `mine` in the warp-uniform range [lo, hi] (hi - lo < 32); a
  // page number outside the cache reads page 0 and reports 0x110
  __device__ int lookup(const DecodeArgs& A, int req, int lo, int hi, int mine, int lane) {
    if (req != r || lo < base || hi >= base + 32) load(A, req, lo, lane);
    int pg = __shfl_sync(0xffffffffu, page, mine - base);
    if (pg < 0 || pg >= A.n_pages) {
      record_error(A.err, 0x110);
      pg = 0;
    }
    return pg;
  }
};

template <int G, int D, int HB>
__global__ void __launch_bounds__(DecCfg<G, D, HB>::THREADS, 2) decode_kernel(const DecodeArgs A) {
  using Cfg = DecCfg<G, D, HB>;
  constexpr int STAGES = Cfg::STAGES, KS = D / 16, NB = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ StageInfo info[STAGES];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g0 = blockIdx.y * HB;  // first kv head of this CTA
  const int Hkv = A.Hkv;
  // rows past a tile's tokens are never copied and must hold finite values (weights 0)
  for (int i = threadIdx.x; i < Cfg::SMEM / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], HB);
    }
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zero stores come before any bulk copy into those rows
  __syncthreads();

  if (warp == HB) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    PageCache pc;
    auto emit = [&](int r, int a, int n, int flags, int slot) -> bool {
      if (lane == 0) ok = mbar_wait(&empty_bar[stage], (round & 1u) ^ 1u, A.err, 0x101);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return false;
      if (lane == 0) {
        info[stage] = StageInfo{r, a, n, flags, slot};
        if (n > 0) mbar_arrive_expect_tx(&full_bar[stage], (uint32_t)(2 * n * HB * D * 2));
        else mbar_arrive(&full_bar[stage]);
      }
      __syncwarp();
      // lane l < 16 copies token a + l's K row, lane 16 + l its V row
      const int tok = lane & 15;
      size_t row;  // token row (HB heads from g0) in K / V, in elements
      if (A.page_size == 0) {
        row = ((size_t)(a + tok) * Hkv + g0) * D;
      } else {
        // token a + tok of request r sits at slot rel % P of the request's page rel / P; every
        // lane takes part in the lookup (lanes past n look up the tile's last token)
        const int P = A.page_size;
        const int rel0 = n > 0 ? a - pc.start(A, r, lane) : 0;
        const int rel = rel0 + min(tok, max(n - 1, 0));
        const int pg = n > 0 ? pc.lookup(A, r, rel0 / P, (rel0 + n - 1) / P, rel / P, lane) : 0;
        row = (((size_t)pg * P + rel % P) * Hkv + g0) * D;
      }
      if (tok < n) {
        uint8_t* dst = smem + (size_t)stage * 2 * Cfg::TILE + (lane >> 4) * Cfg::TILE + tok * Cfg::ROW;
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(lane < 16 ? A.k : A.v);
        bulk_g2s(dst, src + row, HB * D * 2, &full_bar[stage]);
      }
      if (++stage == STAGES) { stage = 0; ++round; }
      return true;
    };
    auto emit_segment = [&](int r, int a, int b, bool final, int slot) -> bool {
      if (a >= b) return emit(r, a, 0, kFirst | kLast | (final ? kFinal : 0), slot);
      for (int t = a; t < b; t += kNT) {
        const int n = min(kNT, b - t);
        const int flags = (t == a ? kFirst : 0) | (t + kNT >= b ? kLast : 0) | (final ? kFinal : 0);
        if (!emit(r, t, n, flags, slot)) return false;
      }
      return true;
    };
    if (A.mode == 0) {
      const int T = min(__ldg(A.kv_indptr + A.n_req), A.T);
      const int start = blockIdx.x * A.range_len;
      const int end = min(T, start + A.range_len);
      if (start < end) {
        int r = find_request(A.kv_indptr, A.n_req, start);
        int a = start;
        while (a < end && r < A.n_req) {
          int rb, re;
          request_range(A, r, rb, re);
          if (re <= a) { ++r; continue; }
          const int b = min(end, re);
          if (!emit_segment(r, a, b, a == rb && b == re, blockIdx.x + r)) break;
          a = b;
          ++r;
        }
      }
    } else {
      const int s = A.splits;
      for (int it = blockIdx.x; it < A.n_req * s; it += gridDim.x) {
        const int r = it / s, c = it % s;
        int rb, re;
        request_range(A, r, rb, re);
        const int len = re - rb;
        const int cl = (len + s - 1) / s;
        const int a = rb + min(len, c * cl), b = rb + min(len, (c + 1) * cl);
        if (!emit_segment(r, a, b, s == 1, it)) break;
      }
    }
    emit(0, 0, 0, kDone, 0);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates: rows g, g + 8; columns 2t, 2t + 1
  const int kvh = g0 + warp;              // kv head of this warp
  const int Hq = A.Hq;
  const uint32_t sbase = smem_u32(smem);
  // fragment rows of this lane that hold query heads: g, and g + 8 when G = 16
  constexpr int NR = G > 8 ? 2 : 1;
  uint32_t qa[KS][4];
  float oacc[NB][4];
  float m_r[NR], l_r[NR];  // running max of each row, this lane's share of its sum
  int stage = 0;
  uint32_t round = 0;
  for (;;) {
    if (!mbar_wait(&full_bar[stage], round & 1u, A.err, 0x102)) break;
    const StageInfo inf = info[stage];
    if (inf.flags & kDone) break;
    if (inf.flags & kFirst) {
      // query rows of this warp's G heads as mma A fragments (row x: head x; rows >= G zero)
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(A.q) + ((size_t)inf.r * Hq + (size_t)kvh * G) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(qg + g * D + 16 * ks + 2 * t)) : 0u;
        qa[ks][2] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(qg + g * D + 16 * ks + 8 + 2 * t)) : 0u;
        if constexpr (NR == 2) {
          qa[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qg + (g + 8) * D + 16 * ks + 2 * t));
          qa[ks][3] = __ldg(reinterpret_cast<const uint32_t*>(qg + (g + 8) * D + 16 * ks + 8 + 2 * t));
        } else {
          qa[ks][1] = qa[ks][3] = 0u;
        }
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        m_r[rr] = -INFINITY;
        l_r[rr] = 0.f;
      }
    }
    if (inf.n > 0) {
      const uint32_t ks_base = sbase + stage * 2 * Cfg::TILE + warp * D * 2;  // this head's K rows
      const uint32_t vs_base = ks_base + Cfg::TILE;
      // ---- S[16 x 16 tokens] = Q K^T: n-blocks of tokens 0..7 and 8..15
      float sacc[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // matrices: (tokens 0..7, dims 16ks..), (0..7, 16ks + 8..), (8..15, 16ks..), (8..15, 16ks + 8..)
        uint32_t b[4];
        const int row = (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(ks_base + row * Cfg::ROW + (16 * ks + ((lane >> 3) & 1) * 8) * 2, b);
        mma_bf16_16816(sacc[0], qa[ks], b[0], b[1]);
        mma_bf16_16816(sacc[1], qa[ks], b[2], b[3]);
      }
      // ---- online softmax of row g (and of row g + 8 when it holds a query head; else its P
      // stays zero)
      float p[NR][4], al[NR];
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        float sv[4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const int j = 8 * nb + 2 * t;
          sv[2 * nb] = j < inf.n ? sacc[nb][2 * rr] * A.scale_log2 : -INFINITY;
          sv[2 * nb + 1] = j + 1 < inf.n ? sacc[nb][2 * rr + 1] * A.scale_log2 : -INFINITY;
        }
        float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // every tile holds at least one valid token, so the new maximum is finite
        const float mn = fmaxf(m_r[rr], mx);
        al[rr] = exp2f(m_r[rr] - mn);  // m = -inf -> 0
        m_r[rr] = mn;
#pragma unroll
        for (int i = 0; i < 4; ++i) p[rr][i] = exp2f(sv[i] - mn);
        l_r[rr] = l_r[rr] * al[rr] + ((p[rr][0] + p[rr][1]) + (p[rr][2] + p[rr][3]));
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        oacc[i][0] *= al[0];
        oacc[i][1] *= al[0];
        if constexpr (NR == 2) {
          oacc[i][2] *= al[NR - 1];
          oacc[i][3] *= al[NR - 1];
        }
      }
      // P as the A operand of one k-step over the 16 tokens (the accumulator layout of two
      // adjacent n-blocks is the A fragment layout); rows g + 8 are zero unless they hold heads
      uint32_t pa[4];
      pa[0] = pack_bf16x2(p[0][0], p[0][1]);
      pa[2] = pack_bf16x2(p[0][2], p[0][3]);
      if constexpr (NR == 2) {
        pa[1] = pack_bf16x2(p[NR - 1][0], p[NR - 1][1]);
        pa[3] = pack_bf16x2(p[NR - 1][2], p[NR - 1][3]);
      } else {
        pa[1] = pa[3] = 0u;
      }
      // ---- O[16 x D] += P V
#pragma unroll
      for (int nbd = 0; nbd < NB; nbd += 2) {
        // matrices (transposed): (tokens 0..7, dims 8nbd..), (8..15, 8nbd..), (0..7, 8nbd + 8..), (8..15, 8nbd + 8..)
        uint32_t b[4];
        const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
        ldsm_x4_t(vs_base + row * Cfg::ROW + (8 * nbd + ((lane >> 4) << 3)) * 2, b);
        mma_bf16_16816(oacc[nbd], pa, b[0], b[1]);
        mma_bf16_16816(oacc[nbd + 1], pa, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[stage]);
    if (++stage == STAGES) { stage = 0; ++round; }

    if (inf.flags & kLast) {
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        float lr = l_r[rr];  // the quad's shares
        lr += __shfl_xor_sync(0xffffffffu, lr, 1);
        lr += __shfl_xor_sync(0xffffffffu, lr, 2);
        const int x = g + 8 * rr;  // query head of this fragment row within the group
        if (x < G) {
          const float inv = lr > 0.f ? 1.f / lr : 0.f;
          const float lse_h = lr > 0.f ? (m_r[rr] + log2f(lr)) * kLn2 : -INFINITY;
          const size_t row = (size_t)kvh * G + x;
          if (inf.flags & kFinal) {
            __nv_bfloat16* op = static_cast<__nv_bfloat16*>(A.o) + ((size_t)inf.r * Hq + row) * D + 2 * t;
#pragma unroll
            for (int i = 0; i < NB; ++i)
              *reinterpret_cast<uint32_t*>(op + 8 * i) = pack_bf16x2(oacc[i][2 * rr] * inv, oacc[i][2 * rr + 1] * inv);
            if (A.lse && t == 0) A.lse[(size_t)inf.r * Hq + row] = lse_h;
          } else {
            float* op = A.part_o + ((size_t)inf.slot * Hq + row) * D + 2 * t;
#pragma unroll
            for (int i = 0; i < NB; ++i)
              *reinterpret_cast<float2*>(op + 8 * i) = make_float2(oacc[i][2 * rr] * inv, oacc[i][2 * rr + 1] * inv);
            if (t == 0) A.part_lse[(size_t)inf.slot * Hq + row] = lse_h;
          }
        }
      }
    }
  }
}

// Merge after the decode kernel: one warp per (request, query head) row.
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeArgs A) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= (int64_t)A.n_req * A.Hq) return;
  const int r = (int)(row / A.Hq), h = (int)(row % A.Hq);
  int beg, end;
  request_range(A, r, beg, end);
  int slot0, s;
  if (end > beg) {
    if (A.mode == 0) {
      const int k0 = beg / A.range_len, k1 = (end - 1) / A.range_len;
      if (k0 == k1) return;  // written by the decode kernel
      slot0 = k0 + r;
      s = k1 - k0 + 1;
    } else {
      if (A.splits == 1) return;
      slot0 = r * A.splits;
      s = A.splits;
    }
  } else {
    if (A.mode == 1 && A.splits == 1) return;  // the decode kernel wrote the empty result
    slot0 = 0;
    s = 0;
  }
  float out[E];
  float lse = -INFINITY;
  if (s > 0)
    lse = merge_row<E>(A.part_o + ((size_t)slot0 * A.Hq + h) * D, (size_t)A.Hq * D, A.part_lse + (size_t)slot0 * A.Hq + h,
                       (size_t)A.Hq, s, lane, out);
  else
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = 0.f;
  __nv_bfloat16* op = static_cast<__nv_bfloat16*>(A.o) + (size_t)row * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) *reinterpret_cast<__nv_bfloat162*>(op + e) = __floats2bfloat162_rn(out[e], out[e + 1]);
  if (A.lse && lane == 0) A.lse[row] = lse;
}

template <int E>
__global__ void __launch_bounds__(256) merge_public_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse, int n_rows, int s,
                                                           void* o, int o_dtype, float* lse) {
  constexpr int D = 32 * E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= n_rows) return;
  float out[E];
  const float L = merge_row<E>(part_o + (size_t)row * s * D, D, part_lse + (size_t)row * s, 1, s, lane, out);
  if (o_dtype == STA_BF16) {
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(o) + (size_t)row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) op[e] = __float2bfloat16_rn(out[e]);
  } else {
    float* op = static_cast<float*>(o) + (size_t)row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) op[e] = out[e];
  }
  if (lse && lane == 0) lse[row] = L;
}

template <int G, int D, int HB>
sta_status plan_t(DecodeArgs& a, int64_t T, int device) {
  using Cfg = DecCfg<G, D, HB>;
  auto kern = decode_kernel<G, D, HB>;
  STA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM));
  int occ = 0, sms = 0;
  STA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Cfg::THREADS, Cfg::SMEM));
  STA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
  if (occ < 1) return STA_ERR_UNSUPPORTED;
  const int64_t ctas = (int64_t)sms * occ;
  const int64_t per_x = ctas / (a.Hkv / HB) > 0 ? ctas / (a.Hkv / HB) : 1;  // CTAs along the token axis
  if (a.mode == 0) {
    int64_t rl = T > 0 ? cdiv(T, per_x) : 1;
    if (rl < kNT) rl = kNT;
    a.range_len = (int)rl;
    a.n_ranges = (int)(T > 0 ? cdiv(T, rl) : 0);
  } else {
    const int64_t items = (int64_t)a.n_req * a.splits;
    a.n_ranges = (int)(items < per_x ? items : per_x);
    a.range_len = 0;
  }
  return STA_OK;
}

template <int G, int D, int HB>
sta_status launch_t(const DecodeArgs& a, cudaStream_t st) {
  using Cfg = DecCfg<G, D, HB>;
  if (a.n_ranges > 0) {
    decode_kernel<G, D, HB><<<dim3(a.n_ranges, a.Hkv / HB), Cfg::THREADS, Cfg::SMEM, st>>>(a);
    STA_LAUNCH_CHECK();
  }
  const int64_t rows = (int64_t)a.n_req * a.Hq;
  decode_merge_kernel<D><<<(unsigned)cdiv(rows, 8), 256, 0, st>>>(a);
  STA_LAUNCH_CHECK();
  return STA_OK;
}

int pick_hb(int Hkv) {
  for (int hb = 8; hb > 1; hb >>= 1)
    if (Hkv % hb == 0) return hb;
  return 1;
}

template <int G, int D>
sta_status dispatch_hb(DecodeArgs& a, int64_t T, int device, cudaStream_t st, bool plan) {
  int hb = pick_hb(a.Hkv);
  if (D == 128 && hb > 4) hb = 4;  // at d = 128 a CTA serves at most 4 heads (two CTAs per SM)
  switch (hb) {
    case 8:
      if constexpr (D == 64) return plan ? plan_t<G, D, 8>(a, T, device) : launch_t<G, D, 8>(a, st);
      return STA_ERR_UNSUPPORTED;
    case 4: return plan ? plan_t<G, D, 4>(a, T, device) : launch_t<G, D, 4>(a, st);
    case 2: return plan ? plan_t<G, D, 2>(a, T, device) : launch_t<G, D, 2>(a, st);
    default: return plan ? plan_t<G, D, 1>(a, T, device) : launch_t<G, D, 1>(a, st);
  }
}

template <int D>
sta_status dispatch_g(DecodeArgs& a, int64_t T, int device, cudaStream_t st, bool plan) {
  switch (a.Hq / a.Hkv) {
    case 1: return dispatch_hb<1, D>(a, T, device, st, plan);
    case 2: return dispatch_hb<2, D>(a, T, device, st, plan);
    case 4: return dispatch_hb<4, D>(a, T, device, st, plan);
    case 8: return dispatch_hb<8, D>(a, T, device, st, plan);
    case 16: return dispatch_hb<16, D>(a, T, device, st, plan);
    default: return STA_ERR_UNSUPPORTED;
  }
}

sta_status dispatch(DecodeArgs& a, int64_t T, int device, cudaStream_t st, bool plan) {
  if (a.d == 64) return dispatch_g<64>(a, T, device, st, plan);
  if (a.d == 128) return dispatch_g<128>(a, T, device, st, plan);
  return STA_ERR_UNSUPPORTED;
}

}  // namespace

sta_status decode_plan(DecodeArgs& a, int64_t total_tokens, int device) {
  return dispatch(a, total_tokens, device, nullptr, true);
}

size_t decode_slots(const DecodeArgs& a) {
  if (a.mode == 0) return (size_t)a.n_ranges + (size_t)a.n_req;
  return (size_t)a.n_req * (size_t)a.splits;
}

sta_status launch_decode(const DecodeArgs& a, cudaStream_t st) {
  DecodeArgs c = a;
  return dispatch(c, 0, 0, st, false);
}

sta_status launch_merge_public(const float* part_o, const float* part_lse, int n_rows, int s, int d, void* o,
                               int o_dtype, float* lse, cudaStream_t st) {
  const unsigned grid = (unsigned)cdiv(n_rows, 8);
  switch (d) {
    case 32: merge_public_kernel<1><<<grid, 256, 0, st>>>(part_o, part_lse, n_rows, s, o, o_dtype, lse); break;
    case 64: merge_public_kernel<2><<<grid, 256, 0, st>>>(part_o, part_lse, n_rows, s, o, o_dtype, lse); break;
    case 128: merge_public_kernel<4><<<grid, 256, 0, st>>>(part_o, part_lse, n_rows, s, o, o_dtype, lse); break;
    case 256: merge_public_kernel<8><<<grid, 256, 0, st>>>(part_o, part_lse, n_rows, s, o, o_dtype, lse); break;
    default: return STA_ERR_UNSUPPORTED;
  }
  STA_LAUNCH_CHECK();
  return STA_OK;
}

}  // namespace sta
