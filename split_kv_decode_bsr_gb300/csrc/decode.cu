// Split-KV GQA decode and log-sum-exp merge (Cleave, Split演算子によるSplit-Kの対応:
// a Split operator with a split count s parallelises the KV reduction; each
// chunk is attended on its own and the partial softmax results are merged).
//
// Decode kernel: persistent-style CTAs, each owning a list of KV segments
// (request r, token range [a, b)) and a block of HB kv heads. One producer warp
// streams K/V tiles (NT tokens x HB heads x d, bf16) from HBM into a ring of
// shared-memory stages with 1-D bulk copies completing on mbarriers; HB consumer
// warps (one per kv head) score the G query heads of their group against each
// tile on the FMA pipe (lanes own d/32 dimensions; a 32-way reduce-scatter over
// shuffles turns per-lane partial dot products into one full score per lane),
// run an fp32 online softmax per query head, and accumulate P.V. A segment that
// covers its whole request writes O (bf16) and LSE directly; otherwise it writes
// a normalised fp32 partial and its LSE, merged afterwards.
//
// Split plans: mode 0 cuts the concatenated token stream [0, T) into equal
// ranges, one per CTA (balanced work whatever the length mix; partial slot of
// (CTA x, request r) = x + r, unique because both grow along the stream);
// mode 1 cuts every request into s chunks of ceil(len / s) keys (slot r*s + c).
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

enum : int { kFirst = 1, kLast = 2, kFinal = 4, kDone = 8 };

struct StageInfo {
  int r, tok0, n, flags, slot;
};

template <int G, int D, int HB>
struct DecCfg {
  static constexpr int E = D / 32;
  static constexpr int TG = 32 / G;             // tokens per reduce-scatter group
  static constexpr int NT = TG > 8 ? TG : 8;    // tokens per tile
  static constexpr int GROUPS = NT / TG;
  static constexpr int TILE_BYTES = NT * HB * D * 2;  // K or V part of one stage
  // ~96 KiB of stages so that two CTAs (16 consumer warps) share an SM
  static constexpr int STAGES_RAW = 98304 / (2 * TILE_BYTES);
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : (STAGES_RAW < 2 ? 2 : STAGES_RAW);
  static_assert(2 * STAGES * TILE_BYTES <= 200 * 1024, "decode stages exceed shared memory");
  static constexpr int SMEM = STAGES * 2 * TILE_BYTES;
  static constexpr int THREADS = (HB + 1) * 32;
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

template <int G, int D, int HB>
__global__ void __launch_bounds__(DecCfg<G, D, HB>::THREADS) decode_kernel(const DecodeArgs A) {
  using Cfg = DecCfg<G, D, HB>;
  constexpr int E = Cfg::E, TG = Cfg::TG, NT = Cfg::NT, STAGES = Cfg::STAGES;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ StageInfo info[STAGES];
  __shared__ __align__(16) float s_p[HB][TG * G];
  __shared__ float s_alpha[HB][G];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g0 = blockIdx.y * HB;  // first kv head of this CTA
  const int Hkv = A.Hkv;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], HB);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == HB) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    // Page cache of the paged layout: lane l holds the page number of ordinal pc_base + l of
    // request pc_r (warp-uniform bookkeeping; reloaded when a lookup leaves the window).
    int pc_r = -1, pc_base = 0, pc_page = 0, pc_rb = 0, pc_pb = 0, pc_pe = 0;
    auto pc_load = [&](int r, int base) {
      if (r != pc_r) {
        pc_r = r;
        int re_unused;
        request_range(A, r, pc_rb, re_unused);  // the same clamped start the token ranges use
        pc_pb = __ldg(A.page_indptr + r);
        pc_pe = __ldg(A.page_indptr + r + 1);
      }
      pc_base = base;
      const int o = pc_pb + base + lane;
      pc_page = o < pc_pe ? __ldg(A.page_indices + o) : 0;
    };
    auto pc_start = [&](int r) {
      if (r != pc_r) pc_load(r, 0);
      return pc_rb;
    };
    auto checked = [&](int pg) {
      if (pg < 0 || pg >= A.n_pages) {  // a bad page table: read page 0, report
        record_error(A.err, 0x110);
        pg = 0;
      }
      return pg;
    };
    // page number of ordinal `ord` (warp-uniform) of request r
    auto page_of = [&](int r, int ord) {
      if (r != pc_r || ord < pc_base || ord >= pc_base + 32) pc_load(r, ord);
      return checked(__shfl_sync(0xffffffffu, pc_page, ord - pc_base));
    };
    // per-lane ordinal `mine` within the warp-uniform range [lo, hi] (hi - lo < 32)
    auto pages_for_stage = [&](int r, int lo, int hi, int mine) {
      if (r != pc_r || lo < pc_base || hi >= pc_base + 32) pc_load(r, lo);
      return checked(__shfl_sync(0xffffffffu, pc_page, mine - pc_base));
    };
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
      if (n > 0) {
        uint8_t* ks = smem + (size_t)stage * 2 * Cfg::TILE_BYTES;
        uint8_t* vs = ks + Cfg::TILE_BYTES;
        const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(A.k);
        const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(A.v);
        if (A.page_size == 0) {
          if (HB == Hkv) {
            if (lane == 0) {
              const size_t off = (size_t)a * Hkv * D;
              bulk_g2s(ks, kg + off, (uint32_t)(n * HB * D * 2), &full_bar[stage]);
              bulk_g2s(vs, vg + off, (uint32_t)(n * HB * D * 2), &full_bar[stage]);
            }
          } else if (lane < n) {
            const size_t off = ((size_t)(a + lane) * Hkv + g0) * D;
            bulk_g2s(ks + lane * HB * D * 2, kg + off, HB * D * 2, &full_bar[stage]);
            bulk_g2s(vs + lane * HB * D * 2, vg + off, HB * D * 2, &full_bar[stage]);
          }
        } else {
          // paged K/V: tokens a .. a+n-1 of request r, copied page run by page run; the page
          // numbers come from the warp's page cache (all lanes take part in the lookups)
          const int P = A.page_size;
          const int rel0 = a - pc_start(r);  // position of token a within its request
          if (HB == Hkv) {
            for (int t = 0; t < n;) {
              const int rel = rel0 + t;
              const int run = min(n - t, P - rel % P);
              const size_t off = ((size_t)page_of(r, rel / P) * P + rel % P) * Hkv * D;
              if (lane == 0) {
                bulk_g2s(ks + t * HB * D * 2, kg + off, (uint32_t)(run * HB * D * 2), &full_bar[stage]);
                bulk_g2s(vs + t * HB * D * 2, vg + off, (uint32_t)(run * HB * D * 2), &full_bar[stage]);
              }
              t += run;
            }
          } else {
            const int rel = rel0 + min(lane, n - 1);
            const int pg = pages_for_stage(r, rel0 / P, (rel0 + n - 1) / P, rel / P);
            if (lane < n) {
              const size_t off = (((size_t)pg * P + rel % P) * Hkv + g0) * D;
              bulk_g2s(ks + lane * HB * D * 2, kg + off, HB * D * 2, &full_bar[stage]);
              bulk_g2s(vs + lane * HB * D * 2, vg + off, HB * D * 2, &full_bar[stage]);
            }
          }
        }
      }
      if (++stage == STAGES) { stage = 0; ++round; }
      return true;
    };
    auto emit_segment = [&](int r, int a, int b, bool final, int slot) -> bool {
      if (a >= b) return emit(r, a, 0, kFirst | kLast | (final ? kFinal : 0), slot);
      for (int t = a; t < b; t += NT) {
        const int n = min(NT, b - t);
        const int flags = (t == a ? kFirst : 0) | (t + NT >= b ? kLast : 0) | (final ? kFinal : 0);
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
  const int g = g0 + warp;  // kv head of this warp
  const int Hq = A.Hq;
  // q and the output accumulators as packed fp32 pairs (dims 2e, 2e+1 of this lane's E)
  constexpr int E2 = E / 2;
  uint64_t q2[G][E2], acc2[G][E2];
  float m_l = -INFINITY, l_l = 0.f;  // running max / sum of head (lane / TG)
  int stage = 0;
  uint32_t round = 0;
  const int my_h = lane / TG, my_t = lane % TG;
  for (;;) {
    if (!mbar_wait(&full_bar[stage], round & 1u, A.err, 0x102)) break;
    const StageInfo inf = info[stage];
    if (inf.flags & kDone) break;
    if (inf.flags & kFirst) {
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(A.q) + ((size_t)inf.r * Hq + (size_t)g * G) * D;
      const uint64_t sc2 = f32x2_pack(A.scale_log2, A.scale_log2);
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < E2; ++e) {
          const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(qg + h * D + lane * E + 2 * e));
          q2[h][e] = f32x2_mul(bf16x2_to_f32x2(w), sc2);
          acc2[h][e] = 0ull;
        }
      }
      m_l = -INFINITY;
      l_l = 0.f;
    }
    const __nv_bfloat16* ks =
        reinterpret_cast<const __nv_bfloat16*>(smem + (size_t)stage * 2 * Cfg::TILE_BYTES) + warp * D + lane * E;
    const __nv_bfloat16* vs = ks + Cfg::TILE_BYTES / 2;
#pragma unroll 1
    for (int grp = 0; grp < Cfg::GROUPS; ++grp) {
      const int tb = grp * TG;
      if (tb >= inf.n) break;
      float vals[32];
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        uint64_t k2[E2];
        const __nv_bfloat16* kp = ks + (size_t)(tb + t) * HB * D;
        if constexpr (E == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(kp);
          k2[0] = bf16x2_to_f32x2(w.x);
          k2[1] = bf16x2_to_f32x2(w.y);
        } else {
          k2[0] = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(kp));
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          uint64_t x2 = f32x2_mul(q2[h][0], k2[0]);
#pragma unroll
          for (int e = 1; e < E2; ++e) x2 = f32x2_fma(q2[h][e], k2[e], x2);
          float xl, xh;
          f32x2_unpack(x2, xl, xh);
          vals[h * TG + t] = xl + xh;
        }
      }
      // 32-way reduce-scatter: afterwards lane holds the full score of value `lane`.
#pragma unroll
      for (int k = 16; k >= 1; k >>= 1) {
        const bool upper = (lane & k) != 0;
#pragma unroll
        for (int i = 0; i < k; ++i) {
          const float send = upper ? vals[i] : vals[i + k];
          const float keep = upper ? vals[i + k] : vals[i];
          vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
        }
      }
      const bool valid = tb + my_t < inf.n;
      const float s = valid ? vals[0] : -INFINITY;
      float mx = s;
#pragma unroll
      for (int o = TG / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_l, mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_l - m_new);
      const float p = valid ? exp2f(s - m_new) : 0.f;
      float ps = p;
#pragma unroll
      for (int o = TG / 2; o >= 1; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l_l = l_l * alpha + ps;
      m_l = m_new;
      s_p[warp][my_t * G + my_h] = p;
      if (my_t == 0) s_alpha[warp][my_h] = alpha;
      __syncwarp();
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a_h = s_alpha[warp][h];
        const uint64_t a2 = f32x2_pack(a_h, a_h);
#pragma unroll
        for (int e = 0; e < E2; ++e) acc2[h][e] = f32x2_mul(acc2[h][e], a2);
      }
      const int nv = min(TG, inf.n - tb);
#pragma unroll 4
      for (int t = 0; t < nv; ++t) {
        float pv[G];
#pragma unroll
        for (int h = 0; h < G; ++h) pv[h] = s_p[warp][t * G + h];
        uint64_t v2[E2];
        const __nv_bfloat16* vp = vs + (size_t)(tb + t) * HB * D;
        if constexpr (E == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vp);
          v2[0] = bf16x2_to_f32x2(w.x);
          v2[1] = bf16x2_to_f32x2(w.y);
        } else {
          v2[0] = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(vp));
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const uint64_t p2 = f32x2_pack(pv[h], pv[h]);
#pragma unroll
          for (int e = 0; e < E2; ++e) acc2[h][e] = f32x2_fma(p2, v2[e], acc2[h][e]);
        }
      }
      __syncwarp();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[stage]);
    if (++stage == STAGES) { stage = 0; ++round; }

    if (inf.flags & kLast) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float l_h = __shfl_sync(0xffffffffu, l_l, h * TG);
        const float m_h = __shfl_sync(0xffffffffu, m_l, h * TG);
        const float inv = l_h > 0.f ? 1.f / l_h : 0.f;
        const float lse_h = l_h > 0.f ? (m_h + log2f(l_h)) * kLn2 : -INFINITY;
        const size_t row = (size_t)g * G + h;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E2; ++e) f32x2_unpack(acc2[h][e], acc[2 * e], acc[2 * e + 1]);
        if (inf.flags & kFinal) {
          __nv_bfloat16* op = static_cast<__nv_bfloat16*>(A.o) + ((size_t)inf.r * Hq + row) * D + lane * E;
#pragma unroll
          for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__nv_bfloat162*>(op + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
          if (A.lse && lane == 0) A.lse[(size_t)inf.r * Hq + row] = lse_h;
        } else {
          float* op = A.part_o + ((size_t)inf.slot * Hq + row) * D + lane * E;
#pragma unroll
          for (int e = 0; e < E; ++e) op[e] = acc[e] * inv;
          if (lane == 0) A.part_lse[(size_t)inf.slot * Hq + row] = lse_h;
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
    if (rl < Cfg::NT) rl = Cfg::NT;
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
  constexpr bool kWide = (G == 1 && D == 128);  // 32-token tiles: at most 4 heads per CTA fit
  if (kWide && hb > 4) hb = 4;
  switch (hb) {
    case 8:
      if constexpr (!kWide) return plan ? plan_t<G, D, 8>(a, T, device) : launch_t<G, D, 8>(a, st);
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
