// Decode against a shared latent KV cache: multi-head latent attention in the weight-absorbed
// form (Cleave, 評価結果: MLA among the LLM subgraphs measured; the token reduction is cut into
// chunks merged by log-sum-exp as the Split operator does for GQA, Split演算子によるSplit-Kの対応).
//
// Request r's query heads q[r, h] (576 entries: a 512-entry latent and a 64-entry rotary part)
// score every cached row kv[t] (576 entries, shared by all heads); the output is the
// softmax-weighted sum of the rows' latent parts (their first 512 entries). One KV head for all
// query heads, the values inside the keys.
//
// One CTA per (chunk of one request's tokens, group of 16 query heads), warp-specialised: a copy
// warp, two score warps and four P.V warps, handing work on through mbarrier rings (no CTA-wide
// barrier in the token loop). The 16 heads are the M of mma.sync.m16n8k16 (bf16 operands, fp32
// accumulators). Per tile of 16 cached rows the score warps compute S[16 x 16 tokens] = Q K^T,
// each over half of the 576 entries with its half of Q held in registers (rows read by
// ldmatrix); the first adds the second's partial, runs the fp32 online softmax on the
// accumulator fragments and passes P (already in the A-fragment layout of P.V) and the
// rescaling factors to the P.V warps through a ring of slots; P.V warp w accumulates O[16 x
// 128] for latent entries 128w.. in registers over the same rows (ldmatrix .trans). Cached rows
// arrive by one bulk copy per row into shared-memory rows padded to 1168 bytes (so that the
// eight rows an ldmatrix reads fall in distinct banks); a stage is refilled once both score
// warps and every P.V warp have released it, and the rows that brought Q in become a fifth
// stage once the score warps hold Q in registers. The latent part of the rows is the V
// operand, so each cached row is read from HBM once per head group.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int kHeads = 16;                    // query heads per CTA: the M of one mma
constexpr int kChunkAlign = 32;               // chunks are whole multiples of this many tokens
constexpr int kTok = 16;                      // tokens per tile (one k-step of P.V)
constexpr int kPvWarps = 4;                   // warps 0..3: P.V, 128 latent entries each
constexpr int kScoreWarp = kPvWarps;          // warp 4: scores over entries 0..287, softmax
constexpr int kScoreWarp2 = kPvWarps + 1;     // warp 5: scores over entries 288..575
constexpr int kCopyWarp = kPvWarps + 2;       // warp 6: bulk copies
constexpr int kThreads = (kPvWarps + 3) * 32;
constexpr int kRowBytes = kDqk * 2 + 16;      // padded shared-memory row (1168 bytes)
constexpr int kKsteps = kDqk / 16;            // 36 k-steps of the score product
constexpr int kKhalf = kKsteps / 2;           // k-steps per score warp
constexpr int kDvPerWarp = kDv / kPvWarps;    // 128 latent entries of O per P.V warp
constexpr int kNbDv = kDvPerWarp / 8;         // 16 n-blocks of 8 per P.V warp
constexpr int kStages = 5;                    // tiles of cached rows in shared memory; the last
                                              // stage holds Q until the score warps have it
constexpr int kPSlots = 4;                    // P / rescale slots between score and P.V warps
constexpr int kSlotBytes = 32 * 16 + 32 * 8;  // per lane: the 4 registers of P, the 2 factors
constexpr int kOffKV = 0;
constexpr int kOffQ = kOffKV + (kStages - 1) * kTok * kRowBytes;   // 74,752: Q, then the last stage
constexpr int kOffP = kOffKV + kStages * kTok * kRowBytes;         // 93,440
constexpr int kOffX = kOffP + kPSlots * kSlotBytes;                // + 3,072
constexpr int kOffFin = kOffX + 2 * 32 * 32;                       // + 2,048 (partial scores, 2 tiles)
constexpr int kSmemBytes = kOffFin + 32 * 8;                       // + 256 = 98,816

struct MlaArgs {
  const __nv_bfloat16* q;   // [n_req, Hq, 576]
  const __nv_bfloat16* kv;  // [T, 576]
  const int32_t* kv_indptr;
  __nv_bfloat16* o;         // [n_req, Hq, 512]
  float* lse;               // [n_req, Hq] or null
  float* part_o;            // [items, Hq, 512] (requests cut into more than one chunk)
  float* part_lse;          // [items, Hq]
  int n_req, Hq, T, chunk;  // chunk: tokens per item, a multiple of kChunkAlign
  int items;                // grid.x: the chunks of all requests (host count; bounds the partials)
  float scale_log2;
  int* err;
};

// Request r's token range from the device indptr, kept inside [0, T] and non-decreasing.
__device__ __forceinline__ void mla_range(const MlaArgs& A, int r, int& rb, int& re) {
  rb = __ldg(A.kv_indptr + r);
  re = __ldg(A.kv_indptr + r + 1);
  if (rb < 0 || re < rb || re > A.T) {
    record_error(A.err, 0x111);
    rb = min(max(rb, 0), A.T);
    re = min(max(re, rb), A.T);
  }
}
__device__ __forceinline__ int mla_chunks(int len, int chunk) { return len > chunk ? (len + chunk - 1) / chunk : 1; }

// Item `item` -> request r, its chunk c, the request's chunk count and its first item, found
// by a whole warp 32 requests at a time (chunk counts prefix-summed with shuffles); r = n_req
// when the item lies past the last request. Every lane returns the same values.
__device__ __forceinline__ void mla_item(const MlaArgs& A, int item, int& r, int& c, int& nc, int& first) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int r0 = 0; r0 < A.n_req; r0 += 32) {
    const int x = r0 + lane;
    int n = 0;
    if (x < A.n_req) {
      int rb, re;
      mla_range(A, x, rb, re);
      n = mla_chunks(re - rb, A.chunk);
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (item < base + total) {
      const int L = __ffs(__ballot_sync(0xffffffffu, item < base + incl)) - 1;  // first lane past the item
      r = r0 + L;
      nc = __shfl_sync(0xffffffffu, n, L);
      first = base + __shfl_sync(0xffffffffu, incl, L) - nc;
      c = item - first;
      return;
    }
    base += total;
  }
  r = A.n_req;
  c = 0;
  nc = 1;
  first = base;
}

// First item and chunk count of request r (whole warp, 32 requests at a time).
__device__ __forceinline__ void mla_request_items(const MlaArgs& A, int r, int& first, int& nc) {
  const int lane = threadIdx.x & 31;
  first = 0;
  for (int r0 = 0; r0 < r; r0 += 32) {
    const int x = r0 + lane;
    int n = 0;
    if (x < r) {
      int rb, re;
      mla_range(A, x, rb, re);
      n = mla_chunks(re - rb, A.chunk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    first += n;
  }
  int rb, re;
  mla_range(A, r, rb, re);
  nc = mla_chunks(re - rb, A.chunk);
}

// grid (items, Hq / 16), kThreads threads, kSmemBytes of dynamic shared memory.
__global__ void __launch_bounds__(kThreads, 2) mla_decode_kernel(const MlaArgs A) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t kv_full[kStages], kv_empty[kStages], p_full[kPSlots], p_empty[kPSlots];
  __shared__ __align__(8) uint64_t q_full, q_free, fin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates: rows g, g + 8; columns 2t, 2t + 1
  int r, c, nc, first;
  mla_item(A, blockIdx.x, r, c, nc, first);
  if (r >= A.n_req) return;  // (a grid larger than the item count)
  const int hg = blockIdx.y;
  int rb, re;
  mla_range(A, r, rb, re);
  const int t0 = rb + c * A.chunk, t1 = min(re, t0 + A.chunk);
  const int ntok = max(t1 - t0, 0), ntiles = (ntok + kTok - 1) / kTok;
  const uint32_t sbase = smem_u32(smem);

  // zero the cached-row stages: rows past the chunk's end are never copied and must hold
  // finite values (their weights are 0); the Q rows hold data
  for (int i = threadIdx.x; i < (kStages - 1) * kTok * kRowBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + kOffKV)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], kPvWarps + 2);  // both score warps and every P.V warp release a stage
    }
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(&p_full[s], 1);
      mbar_init(&p_empty[s], kPvWarps);
    }
    mbar_init(&q_full, 1);
    mbar_init(&q_free, 2);  // both score warps hold their half of Q in registers
    mbar_init(&fin, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zero stores come before any bulk copy into those rows
  __syncthreads();

  // Every wait is bounded. A warp whose wait ran out (error word set) stops waiting and leaves
  // its loop; the warps that wait on it then run out once themselves and stop as well.
  if (warp == kCopyWarp) {
    // ---------------------------------------------------------------- copies (lane i: row i)
    if (lane == 0) mbar_arrive_expect_tx(&q_full, (uint32_t)(kHeads * kDqk * 2));
    __syncwarp();
    if (lane < kHeads)
      bulk_g2s(smem + kOffQ + lane * kRowBytes, A.q + ((int64_t)r * A.Hq + hg * kHeads + lane) * kDqk,
               (uint32_t)(kDqk * 2), &q_full);
    int issued = 0;
    for (int k = 0; k < ntiles; ++k) {
      const int s = k % kStages, base = t0 + k * kTok, n = min(kTok, t1 - base);
      bool free_ok = true;  // lane 0 waits, the warp follows its answer
      if (lane == 0) {
        free_ok = mbar_wait(&kv_empty[s], ((uint32_t)(k / kStages) & 1u) ^ 1u, A.err, 0x504);
        if (free_ok && k == kStages - 1) free_ok = mbar_wait(&q_free, 0, A.err, 0x508);  // Q's rows, first use
      }
      if (!__shfl_sync(0xffffffffu, free_ok, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[s], (uint32_t)(n * kDqk * 2));
      __syncwarp();
      if (lane < n)
        bulk_g2s(smem + kOffKV + (s * kTok + lane) * kRowBytes, A.kv + (int64_t)(base + lane) * kDqk,
                 (uint32_t)(kDqk * 2), &kv_full[s]);
      issued = k + 1;
    }
    // no copy may land after the CTA has left: wait (bounded) for the last one of each stage
    if (lane == 0) {
      mbar_wait(&q_full, 0, A.err, 0x503);
      for (int k = max(0, issued - kStages); k < issued; ++k)
        mbar_wait(&kv_full[k % kStages], (uint32_t)(k / kStages) & 1u, A.err, 0x503);
    }
    return;
  }

  if (warp == kScoreWarp || warp == kScoreWarp2) {
    // --------------------------------------------- scores (two warps, half the entries each)
    // Warp kScoreWarp2 adds its partial S into a two-tile exchange buffer; warp kScoreWarp sums,
    // runs the online softmax and hands P on. The two meet on named barrier 1 once per tile (B
    // writes tile k's buffer while A still reads tile k - 1's) and both run every tile, so that
    // neither is left alone at the barrier: after a timed-out wait (error word set) a warp
    // computes on whatever the stages hold and stops waiting.
    const bool lead = warp == kScoreWarp;
    const int kk0 = lead ? 0 : kKhalf;
    bool ok = mbar_wait(&q_full, 0, A.err, 0x501);
    // this warp's 18 k-steps of the 16 query rows as A fragments: matrices (heads 0..7, dims
    // 16kk..), (8..15, 16kk..), (0..7, 16kk + 8..), (8..15, 16kk + 8..)
    uint32_t qa[kKhalf][4];
    {
      const uint32_t q_addr = sbase + kOffQ + (lane & 15) * kRowBytes + ((lane >> 4) << 3) * 2;
#pragma unroll
      for (int i = 0; i < kKhalf; ++i) ldsm_x4(q_addr + (kk0 + i) * 32, qa[i]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_free);  // Q's rows may take cached rows now
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g, g + 8 (l: this lane's share)
    for (int k = 0; k < ntiles; ++k) {
      const int s = k % kStages;
      if (ok) ok = mbar_wait(&kv_full[s], (uint32_t)(k / kStages) & 1u, A.err, 0x502);
      const uint32_t kvs = sbase + kOffKV + s * kTok * kRowBytes;
      // partial S[16 heads x 16 tokens]: n-blocks of tokens 0..7 and 8..15, even and odd k-steps apart;
      // rows: (tokens 0..7, dims 16kk..), (0..7, 16kk + 8..), (8..15, 16kk..), (8..15, 16kk + 8..)
      float sacc[2][2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) sacc[i][nb][0] = sacc[i][nb][1] = sacc[i][nb][2] = sacc[i][nb][3] = 0.f;
      const uint32_t k_addr =
          kvs + ((lane & 7) + ((lane >> 4) << 3)) * kRowBytes + (kk0 * 16 + (((lane >> 3) & 1) << 3)) * 2;
#pragma unroll
      for (int i = 0; i < kKhalf; ++i) {
        uint32_t b[4];
        ldsm_x4(k_addr + i * 32, b);
        mma_bf16_16816(sacc[i & 1][0], qa[i], b[0], b[1]);
        mma_bf16_16816(sacc[i & 1][1], qa[i], b[2], b[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&kv_empty[s]);  // the rows' keys are read
      float4* xb = reinterpret_cast<float4*>(smem + kOffX + (k & 1) * 32 * 32) + lane * 2;
      if (!lead) {
        xb[0] = make_float4(sacc[0][0][0] + sacc[1][0][0], sacc[0][0][1] + sacc[1][0][1], sacc[0][0][2] + sacc[1][0][2],
                            sacc[0][0][3] + sacc[1][0][3]);
        xb[1] = make_float4(sacc[0][1][0] + sacc[1][1][0], sacc[0][1][1] + sacc[1][1][1], sacc[0][1][2] + sacc[1][1][2],
                            sacc[0][1][3] + sacc[1][1][3]);
        named_bar_sync(1, 64);
        continue;
      }
      named_bar_sync(1, 64);
      const float4 x0 = xb[0], x1 = xb[1];
      const float xs[2][4] = {{x0.x, x0.y, x0.z, x0.w}, {x1.x, x1.y, x1.z, x1.w}};
      // online softmax of rows g and g + 8 over the tile's valid tokens
      const int nvalid = min(kTok, ntok - k * kTok);
      float sv[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        const int j = 8 * nb + 2 * t;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = (sacc[0][nb][e] + sacc[1][nb][e] + xs[nb][e]) * A.scale_log2;
          sv[nb][e] = j + (e & 1) < nvalid ? x : -INFINITY;
        }
      }
      float mx0 = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
      float mx1 = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      // every tile holds at least one valid token, so the new maxima are finite
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);  // m = -inf -> 0
      m0 = mn0;
      m1 = mn1;
      float p[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        p[nb][0] = exp2f(sv[nb][0] - mn0);
        p[nb][1] = exp2f(sv[nb][1] - mn0);
        p[nb][2] = exp2f(sv[nb][2] - mn1);
        p[nb][3] = exp2f(sv[nb][3] - mn1);
      }
      l0 = l0 * al0 + ((p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
      l1 = l1 * al1 + ((p[0][2] + p[0][3]) + (p[1][2] + p[1][3]));
      // hand P (as the A fragment of one k-step over the 16 tokens) and the factors on
      const int ps = k % kPSlots;
      if (ok) {
        bool slot_ok = true;
        if (lane == 0) slot_ok = mbar_wait(&p_empty[ps], ((uint32_t)(k / kPSlots) & 1u) ^ 1u, A.err, 0x505);
        ok = __shfl_sync(0xffffffffu, slot_ok, 0);
      }
      if (!ok) continue;
      uint8_t* slot = smem + kOffP + ps * kSlotBytes;
      reinterpret_cast<uint4*>(slot)[lane] = make_uint4(pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(p[0][2], p[0][3]),
                                                        pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(p[1][2], p[1][3]));
      reinterpret_cast<float2*>(slot + 32 * 16)[lane] = make_float2(al0, al1);
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[ps]);
    }
    if (!lead) return;
    // the row sums, then 1 / l for the P.V warps and the LSE (rows without a valid token: 0, -inf)
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (!ok) l0 = l1 = 0.f;
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    reinterpret_cast<float2*>(smem + kOffFin)[lane] = make_float2(inv0, inv1);
    __syncwarp();
    if (lane == 0) mbar_arrive(&fin);
    if (t == 0) {
      const float lse0 = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
      const float lse1 = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
      const int h0 = hg * kHeads + g, h1 = h0 + 8;
      if (nc == 1) {
        if (A.lse) {
          A.lse[(int64_t)r * A.Hq + h0] = lse0;
          A.lse[(int64_t)r * A.Hq + h1] = lse1;
        }
      } else {
        const int64_t item = first + c;
        A.part_lse[item * A.Hq + h0] = lse0;
        A.part_lse[item * A.Hq + h1] = lse1;
      }
    }
    return;
  }

  // -------------------------------------------------------------- P.V warps (warp = 0..3)
  float oacc[kNbDv][4];
#pragma unroll
  for (int i = 0; i < kNbDv; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  bool ok = true;
  // V rows, transposed: matrices (tokens 0..7, entries d0..), (8..15, d0..), (0..7, d0 + 8..), (8..15, d0 + 8..)
  const uint32_t v_off = ((lane & 7) + (((lane >> 3) & 1) << 3)) * kRowBytes +
                         (warp * kDvPerWarp + ((lane >> 4) << 3)) * 2;
  for (int k = 0; k < ntiles; ++k) {
    const int s = k % kStages, ps = k % kPSlots;
    // the stage's rows (this warp observes their copies itself), then P of the tile
    ok = mbar_wait(&kv_full[s], (uint32_t)(k / kStages) & 1u, A.err, 0x502);
    if (ok) ok = mbar_wait(&p_full[ps], (uint32_t)(k / kPSlots) & 1u, A.err, 0x506);
    if (!ok) break;
    const uint8_t* slot = smem + kOffP + ps * kSlotBytes;
    const uint4 pv = reinterpret_cast<const uint4*>(slot)[lane];
    const float2 al = reinterpret_cast<const float2*>(slot + 32 * 16)[lane];
    __syncwarp();
    if (lane == 0) mbar_arrive(&p_empty[ps]);
    const uint32_t pa[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
    for (int i = 0; i < kNbDv; ++i) {
      oacc[i][0] *= al.x;
      oacc[i][1] *= al.x;
      oacc[i][2] *= al.y;
      oacc[i][3] *= al.y;
    }
    const uint32_t vs = sbase + kOffKV + s * kTok * kRowBytes + v_off;
#pragma unroll
    for (int nbd = 0; nbd < kNbDv; nbd += 2) {
      uint32_t b[4];
      ldsm_x4_t(vs + nbd * 16, b);
      mma_bf16_16816(oacc[nbd], pa, b[0], b[1]);
      mma_bf16_16816(oacc[nbd + 1], pa, b[2], b[3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&kv_empty[s]);
  }
  // ---- epilogue: O / l (the score warp's factors)
  float2 inv = make_float2(0.f, 0.f);
  if (mbar_wait(&fin, 0, A.err, 0x507)) inv = reinterpret_cast<const float2*>(smem + kOffFin)[lane];
  const int h0 = hg * kHeads + g, h1 = h0 + 8;
  if (nc == 1) {  // the whole request in this CTA: O (bf16) directly
    __nv_bfloat16* o0 = A.o + ((int64_t)r * A.Hq + h0) * kDv + warp * kDvPerWarp + 2 * t;
    __nv_bfloat16* o1 = A.o + ((int64_t)r * A.Hq + h1) * kDv + warp * kDvPerWarp + 2 * t;
#pragma unroll
    for (int i = 0; i < kNbDv; ++i) {
      *reinterpret_cast<uint32_t*>(o0 + 8 * i) = pack_bf16x2(oacc[i][0] * inv.x, oacc[i][1] * inv.x);
      *reinterpret_cast<uint32_t*>(o1 + 8 * i) = pack_bf16x2(oacc[i][2] * inv.y, oacc[i][3] * inv.y);
    }
  } else {  // a chunk: its normalised fp32 partial, merged afterwards
    const int64_t item = first + c;
    float* o0 = A.part_o + (item * A.Hq + h0) * kDv + warp * kDvPerWarp + 2 * t;
    float* o1 = A.part_o + (item * A.Hq + h1) * kDv + warp * kDvPerWarp + 2 * t;
#pragma unroll
    for (int i = 0; i < kNbDv; ++i) {
      *reinterpret_cast<float2*>(o0 + 8 * i) = make_float2(oacc[i][0] * inv.x, oacc[i][1] * inv.x);
      *reinterpret_cast<float2*>(o1 + 8 * i) = make_float2(oacc[i][2] * inv.y, oacc[i][3] * inv.y);
    }
  }
}

// Log-sum-exp merge of the chunks of requests cut into more than one: one warp per (request,
// head, quarter of the 512 latent entries); lane owns 4 consecutive entries.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaArgs A) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * 8 + warp;
  if (wid >= (int64_t)A.n_req * A.Hq * 4) return;
  const int64_t row = wid >> 2;
  const int quarter = (int)(wid & 3);
  const int r = (int)(row / A.Hq), h = (int)(row % A.Hq);
  int first, nc;
  mla_request_items(A, r, first, nc);
  if (nc == 1) return;  // written by the decode kernel
  if (first + nc > A.items) {  // device and host kv_indptr disagree: no read past the partials
    record_error(A.err, 0x111);
    return;
  }
  float out[4];
  const float L = merge_row<4>(A.part_o + ((int64_t)first * A.Hq + h) * kDv + quarter * (kDv / 4),
                               (size_t)A.Hq * kDv, A.part_lse + (int64_t)first * A.Hq + h, (size_t)A.Hq, nc, lane, out);
  __nv_bfloat16* op = A.o + row * kDv + quarter * (kDv / 4) + lane * 4;
  *reinterpret_cast<uint2*>(op) = make_uint2(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]));
  if (A.lse && lane == 0 && quarter == 0) A.lse[row] = L;
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace sta

using namespace sta;

extern "C" sta_status sta_mla_decode(const void* q, const void* kv, const int32_t* kv_indptr_dev,
                                     const int32_t* kv_indptr_host, int n_req, int Hq, float scale, int chunk_tokens,
                                     void* o, float* lse, void* workspace, size_t* workspace_bytes,
                                     sta_stream stream) {
  if (!workspace_bytes || !kv_indptr_host || n_req < 1 || Hq < kHeads || Hq % kHeads || Hq > 1024 ||
      chunk_tokens < 0 || !(scale > 0.f) || !isfinite(scale))
    return STA_ERR_INVALID_ARG;
  if (kv_indptr_host[0] != 0) return STA_ERR_INVALID_ARG;
  for (int x = 0; x < n_req; ++x)
    if (kv_indptr_host[x + 1] < kv_indptr_host[x]) return STA_ERR_INVALID_ARG;
  const int64_t T = kv_indptr_host[n_req];
  // tokens per chunk: given (rounded up to 32), or about 2 CTAs' share per SM of the whole
  // token stream across all head groups, at least 128
  auto count_items = [&](int ch) {
    int64_t n = 0;
    for (int x = 0; x < n_req; ++x) {
      const int len = kv_indptr_host[x + 1] - kv_indptr_host[x];
      n += len > ch ? (len + ch - 1) / ch : 1;
    }
    return n;
  };
  int chunk = chunk_tokens;
  if (chunk == 0) {
    // the smallest chunk (a multiple of 32 tokens, at least 128) whose items across all head
    // groups fit one wave of resident CTAs (two per SM): a second, partial wave would run a
    // full chunk after the first
    int dev = 0, sms = 0;
    STA_CUDA_TRY(cudaGetDevice(&dev));
    STA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int64_t slots = (int64_t)sms * 2, hg = Hq / kHeads;
    int64_t ch = std::max<int64_t>(4 * kChunkAlign, (T * hg + slots - 1) / slots);
    ch = (ch + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
    while (ch < (1 << 30) && count_items((int)ch) * hg > slots)
      ch += std::max<int64_t>(kChunkAlign, ch / 32 / kChunkAlign * kChunkAlign);
    chunk = (int)std::min<int64_t>(ch, 1 << 30);
  }
  chunk = (chunk + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
  int64_t items = 0, split_items = 0;
  for (int x = 0; x < n_req; ++x) {
    const int len = kv_indptr_host[x + 1] - kv_indptr_host[x];
    const int nc = len > chunk ? (len + chunk - 1) / chunk : 1;
    items += nc;
    if (nc > 1) split_items += nc;
  }
  if (items > INT32_MAX) return STA_ERR_INVALID_ARG;
  const size_t o_bytes = align256((size_t)items * Hq * kDv * sizeof(float));
  const size_t need = split_items ? o_bytes + align256((size_t)items * Hq * sizeof(float)) : 256;
  if (!workspace) {
    *workspace_bytes = need;
    return STA_OK;
  }
  if (*workspace_bytes < need) return STA_ERR_WORKSPACE;
  if (!q || !o || (T > 0 && !kv) || !kv_indptr_dev) return STA_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)o & 15) || ((uintptr_t)workspace & 255))
    return STA_ERR_UNSUPPORTED;
  MlaArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.kv_indptr = kv_indptr_dev;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.part_o = split_items ? static_cast<float*>(workspace) : nullptr;
  a.part_lse = split_items ? reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes) : nullptr;
  a.n_req = n_req;
  a.Hq = Hq;
  a.T = (int)T;
  a.chunk = chunk;
  a.items = (int)items;
  a.scale_log2 = scale * kLog2e;
  a.err = device_error_word();
  cudaStream_t st = (cudaStream_t)stream;
  STA_CUDA_TRY(cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
  mla_decode_kernel<<<dim3((unsigned)items, (unsigned)(Hq / kHeads)), kThreads, kSmemBytes, st>>>(a);
  STA_LAUNCH_CHECK();
  if (split_items) {
    mla_merge_kernel<<<(unsigned)(((int64_t)n_req * Hq * 4 + 7) / 8), 256, 0, st>>>(a);
    STA_LAUNCH_CHECK();
  }
  return STA_OK;
}
