// Decode against a shared latent KV cache: multi-head latent attention in the weight-absorbed
// form (Cleave, 評価結果: MLA among the LLM subgraphs measured; the token reduction is cut into
// chunks merged by log-sum-exp as the Split operator does for GQA, Split演算子によるSplit-Kの対応).
//
// Request r's query heads q[r, h] (576 entries: a 512-entry latent and a 64-entry rotary part)
// score every cached row kv[t] (576 entries, shared by all heads); the output is the
// softmax-weighted sum of the rows' latent parts (their first 512 entries). One KV head for all
// query heads, the values inside the keys.
//
// One CTA per (chunk of one request's tokens, group of 16 query heads): four compute warps and
// a warp that issues the copies. The 16 heads are the M of mma.sync.m16n8k16 (bf16 operands,
// fp32 accumulators): the scores S[16 x 32 tokens] of a tile are split across the compute warps
// by head dimension (a warp keeps its 144 dimensions of the 16 query rows in registers and adds
// its partial S into shared memory), every compute warp then turns the summed S into the
// weights P, and P.V is split by output dimension (128 latent entries per warp, accumulators in
// registers). Cached rows arrive by one bulk copy per row into shared-memory rows padded to 1168
// bytes (so that the eight rows an ldmatrix reads fall in distinct banks), two tiles of 32
// tokens in flight; the copy warp refills a stage once every compute warp has released it. The
// latent part of the same rows is the V operand (ldmatrix .trans), so each cached row is read
// from HBM once per head group.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int kHeads = 16;                    // query heads per CTA: the M of one mma
constexpr int kTile = 32;                     // tokens per tile
constexpr int kWarps = 4;                     // consumer warps; warp kWarps issues the copies
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kRowBytes = kDqk * 2 + 16;      // padded shared-memory row (1168 bytes)
constexpr int kKsteps = kDqk / 16;            // 36 k-steps of the score product
constexpr int kKstepsPerWarp = kKsteps / kWarps;  // 9
constexpr int kDvPerWarp = kDv / kWarps;      // 128 latent entries of O per warp
constexpr int kNbDv = kDvPerWarp / 8;         // 16 n-blocks of 8 per warp
constexpr int kStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kHeads * kRowBytes;                 // 18,688
constexpr int kOffS = kOffKV + kStages * kTile * kRowBytes;        // + 74,752
constexpr int kSRow = kTile + 8;  // partial-score row stride in floats: 8-byte accesses of a
                                   // half-warp (rows g..g+3) fall in distinct banks
constexpr int kSmemBytes = kOffS + kWarps * kHeads * kSRow * 4;    // + 10,240 = 103,680

struct MlaArgs {
  const __nv_bfloat16* q;   // [n_req, Hq, 576]
  const __nv_bfloat16* kv;  // [T, 576]
  const int32_t* kv_indptr;
  __nv_bfloat16* o;         // [n_req, Hq, 512]
  float* lse;               // [n_req, Hq] or null
  float* part_o;            // [items, Hq, 512] (requests cut into more than one chunk)
  float* part_lse;          // [items, Hq]
  int n_req, Hq, T, chunk;  // chunk: tokens per item, a multiple of kTile
  int items;                // grid.x: the chunks of all requests (host count; bounds the partials)
  float scale_log2;
  int* err;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D += A (16 x 16, row) * B (16 x 8, col); bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

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

// grid (items, Hq / 16), 128 threads, kSmemBytes of dynamic shared memory.
__global__ void __launch_bounds__(kThreads, 2) mla_decode_kernel(const MlaArgs A) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], q_full;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates
  int r, c, nc, first;
  mla_item(A, blockIdx.x, r, c, nc, first);
  if (r >= A.n_req) return;  // (a grid larger than the item count)
  const int hg = blockIdx.y;
  int rb, re;
  mla_range(A, r, rb, re);
  const int t0 = rb + c * A.chunk, t1 = min(re, t0 + A.chunk);
  const int ntok = max(t1 - t0, 0), ntiles = (ntok + kTile - 1) / kTile;
  const uint32_t sbase = smem_u32(smem);

  // zero the cached-row stages: rows past the chunk's end are never copied and must hold
  // finite values (their weights are 0)
  for (int i = threadIdx.x; i < kStages * kTile * kRowBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + kOffKV)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);  // one arrival per consumer warp once it has read the stage
    }
    mbar_init(&q_full, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zero stores come before any bulk copy into those rows
  __syncthreads();
  if (warp == kWarps) {
    // ---------------------------------------------------------------- copies (lane i: row i)
    if (lane == 0) mbar_arrive_expect_tx(&q_full, (uint32_t)(kHeads * kDqk * 2));
    __syncwarp();
    if (lane < kHeads)
      bulk_g2s(smem + kOffQ + lane * kRowBytes, A.q + ((int64_t)r * A.Hq + hg * kHeads + lane) * kDqk,
               (uint32_t)(kDqk * 2), &q_full);
    for (int k = 0; k < ntiles; ++k) {
      const int s = k % kStages, base = t0 + k * kTile, n = min(kTile, t1 - base);
      // the stage is free once every consumer warp has finished tile k - kStages
      // lane 0 waits, the warp follows its answer (no lane leaves the loop alone)
      bool free_ok = true;
      if (lane == 0) free_ok = mbar_wait(&empty[s], ((uint32_t)(k / kStages) & 1u) ^ 1u, A.err, 0x504);
      if (!__shfl_sync(0xffffffffu, free_ok, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(n * kDqk * 2));
      __syncwarp();
      if (lane < n)
        bulk_g2s(smem + kOffKV + (s * kTile + lane) * kRowBytes, A.kv + (int64_t)(base + lane) * kDqk,
                 (uint32_t)(kDqk * 2), &full[s]);
    }
    return;
  }
  const bool q_ok = mbar_wait(&q_full, 0, A.err, 0x501);
  bool ok = q_ok;
  int consumed = 0;  // tiles whose copies have landed and been read
  // this warp's 9 k-steps of the 16 query rows, as mma A fragments (matrix j of an x4: rows
  // 8(j & 1).., dimensions +8(j >> 1))
  uint32_t qa[kKstepsPerWarp][4];
#pragma unroll
  for (int ks = 0; ks < kKstepsPerWarp; ++ks) {
    const int kk = warp * kKstepsPerWarp + ks;
    ldsm_x4(sbase + kOffQ + (lane & 15) * kRowBytes + (kk * 16 + (lane >> 4) * 8) * 2, qa[ks]);
  }
  float oacc[kNbDv][4];
#pragma unroll
  for (int i = 0; i < kNbDv; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g and g + 8
  float* s_part = reinterpret_cast<float*>(smem + kOffS);      // [warp][16][kSRow]

  // Every consumer warp runs every tile and reaches every barrier: after a timed-out wait
  // (error word set) the warps stop waiting and compute on whatever the stages hold, so that
  // none is left alone at a named barrier.
  for (int k = 0; k < ntiles; ++k) {
    const int s = k % kStages;
    if (ok) {  // every lane waits (each then sees the copied rows); the warp follows lane 0
      const bool got = mbar_wait(&full[s], (uint32_t)(k / kStages) & 1u, A.err, 0x502);
      ok = __shfl_sync(0xffffffffu, got, 0);
    }
    if (ok) consumed = k + 1;
    const uint32_t kvs = sbase + kOffKV + s * kTile * kRowBytes;
    // ---- partial scores over this warp's dimensions, 4 n-blocks of 8 tokens
    float sacc[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kKstepsPerWarp; ++ks) {
      const int kk = warp * kKstepsPerWarp + ks;
#pragma unroll
      for (int nb = 0; nb < 4; nb += 2) {
        // matrices: (tokens 8nb.., dims 16kk), (8nb.., 16kk + 8), (8nb + 8.., 16kk), (8nb + 8.., 16kk + 8)
        uint32_t b[4];
        const int row = 8 * nb + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(kvs + row * kRowBytes + (kk * 16 + ((lane >> 3) & 1) * 8) * 2, b);
        mma_bf16(sacc[nb], qa[ks], b[0], b[1]);
        mma_bf16(sacc[nb + 1], qa[ks], b[2], b[3]);
      }
    }
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      float* sp = s_part + warp * kHeads * kSRow;
      *reinterpret_cast<float2*>(sp + g * kSRow + 8 * nb + 2 * t) = make_float2(sacc[nb][0], sacc[nb][1]);
      *reinterpret_cast<float2*>(sp + (g + 8) * kSRow + 8 * nb + 2 * t) = make_float2(sacc[nb][2], sacc[nb][3]);
    }
    named_bar_sync(1, kWarps * 32);  // every consumer warp's partial scores are in
    // ---- full scores at this thread's fragment positions (rows g, g + 8; 8 tokens each)
    const int nvalid = min(kTile, ntok - k * kTile);
    float sv[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* sp = s_part + w * kHeads * kSRow;
        const float2 x = *reinterpret_cast<const float2*>(sp + g * kSRow + 8 * nb + 2 * t);
        const float2 y = *reinterpret_cast<const float2*>(sp + (g + 8) * kSRow + 8 * nb + 2 * t);
        a.x += x.x; a.y += x.y; b.x += y.x; b.y += y.y;
      }
      const int j = 8 * nb + 2 * t;
      sv[nb][0] = j < nvalid ? a.x * A.scale_log2 : -INFINITY;
      sv[nb][1] = j + 1 < nvalid ? a.y * A.scale_log2 : -INFINITY;
      sv[nb][2] = j < nvalid ? b.x * A.scale_log2 : -INFINITY;
      sv[nb][3] = j + 1 < nvalid ? b.y * A.scale_log2 : -INFINITY;
    }
    // ---- online softmax of rows g and g + 8 (the four lanes of a quad share a row)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      mx0 = fmaxf(mx0, fmaxf(sv[nb][0], sv[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(sv[nb][2], sv[nb][3]));
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    // every tile holds at least one valid token, so mn is finite here
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);  // m = -inf -> 0
    m0 = mn0;
    m1 = mn1;
    float p[4][4];
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      p[nb][0] = exp2f(sv[nb][0] - mn0);
      p[nb][1] = exp2f(sv[nb][1] - mn0);
      p[nb][2] = exp2f(sv[nb][2] - mn1);
      p[nb][3] = exp2f(sv[nb][3] - mn1);
      ps0 += p[nb][0] + p[nb][1];
      ps1 += p[nb][2] + p[nb][3];
    }
    l0 = l0 * al0 + ps0;  // this lane's share; the quad's shares are added at the end
    l1 = l1 * al1 + ps1;
#pragma unroll
    for (int i = 0; i < kNbDv; ++i) {
      oacc[i][0] *= al0;
      oacc[i][1] *= al0;
      oacc[i][2] *= al1;
      oacc[i][3] *= al1;
    }
    // P as the A operand of two k-steps (tokens 0..15, 16..31): the accumulator layout of two
    // adjacent n-blocks is the A fragment layout
    uint32_t pa[2][4];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      pa[ks][0] = pack_bf16x2(p[2 * ks][0], p[2 * ks][1]);
      pa[ks][1] = pack_bf16x2(p[2 * ks][2], p[2 * ks][3]);
      pa[ks][2] = pack_bf16x2(p[2 * ks + 1][0], p[2 * ks + 1][1]);
      pa[ks][3] = pack_bf16x2(p[2 * ks + 1][2], p[2 * ks + 1][3]);
    }
    // ---- O[16 x this warp's 128 latent entries] += P V, V = the rows' first 512 entries
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int nbd = 0; nbd < kNbDv; nbd += 2) {
        // matrices (transposed): (tokens 16ks.., dims d0), (16ks + 8.., d0), (16ks.., d0 + 8), (16ks + 8.., d0 + 8)
        const int d0 = warp * kDvPerWarp + nbd * 8;
        const int row = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
        uint32_t b[4];
        ldsm_x4_t(kvs + row * kRowBytes + (d0 + ((lane >> 4) << 3)) * 2, b);
        mma_bf16(oacc[nbd], pa[ks], b[0], b[1]);
        mma_bf16(oacc[nbd + 1], pa[ks], b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with stage s
    named_bar_sync(2, kWarps * 32);         // the partial scores may be overwritten
  }
  if (!ok && threadIdx.x == 0) {
    // after a timed-out wait: the last copy of each stage (issued once the consumers released
    // the stage) lands before shared memory is released; every wait is bounded
    if (!q_ok) mbar_wait(&q_full, 0, A.err, 0x503);
    for (int k = max(consumed, ntiles - kStages); k < ntiles; ++k)
      mbar_wait(&full[k % kStages], (uint32_t)(k / kStages) & 1u, A.err, 0x503);
  }
  // ---- epilogue: the row sums, then O / l and the LSE (rows without a valid token: 0, -inf)
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (!ok) l0 = l1 = 0.f;
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const float lse0 = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
  const float lse1 = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
  const int h0 = hg * kHeads + g, h1 = h0 + 8;
  if (nc == 1) {  // the whole request in this CTA: O (bf16) and LSE directly
    __nv_bfloat16* o0 = A.o + ((int64_t)r * A.Hq + h0) * kDv + warp * kDvPerWarp + 2 * t;
    __nv_bfloat16* o1 = A.o + ((int64_t)r * A.Hq + h1) * kDv + warp * kDvPerWarp + 2 * t;
#pragma unroll
    for (int i = 0; i < kNbDv; ++i) {
      *reinterpret_cast<uint32_t*>(o0 + 8 * i) = pack_bf16x2(oacc[i][0] * inv0, oacc[i][1] * inv0);
      *reinterpret_cast<uint32_t*>(o1 + 8 * i) = pack_bf16x2(oacc[i][2] * inv1, oacc[i][3] * inv1);
    }
    if (A.lse && warp == 0 && t == 0) {
      A.lse[(int64_t)r * A.Hq + h0] = lse0;
      A.lse[(int64_t)r * A.Hq + h1] = lse1;
    }
  } else {  // a chunk: its normalised fp32 partial and LSE, merged afterwards
    const int64_t item = first + c;
    float* o0 = A.part_o + (item * A.Hq + h0) * kDv + warp * kDvPerWarp + 2 * t;
    float* o1 = A.part_o + (item * A.Hq + h1) * kDv + warp * kDvPerWarp + 2 * t;
#pragma unroll
    for (int i = 0; i < kNbDv; ++i) {
      *reinterpret_cast<float2*>(o0 + 8 * i) = make_float2(oacc[i][0] * inv0, oacc[i][1] * inv0);
      *reinterpret_cast<float2*>(o1 + 8 * i) = make_float2(oacc[i][2] * inv1, oacc[i][3] * inv1);
    }
    if (warp == 0 && t == 0) {
      A.part_lse[item * A.Hq + h0] = lse0;
      A.part_lse[item * A.Hq + h1] = lse1;
    }
  }
}

// Log-sum-exp merge of the chunks of requests cut into more than one: one warp per (request,
// head); lane owns 16 consecutive latent entries.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaArgs A) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= (int64_t)A.n_req * A.Hq) return;
  const int r = (int)(row / A.Hq), h = (int)(row % A.Hq);
  int first, nc;
  mla_request_items(A, r, first, nc);
  if (nc == 1) return;  // written by the decode kernel
  if (first + nc > A.items) {  // device and host kv_indptr disagree: no read past the partials
    record_error(A.err, 0x111);
    return;
  }
  float out[16];
  const float L = merge_row<16>(A.part_o + ((int64_t)first * A.Hq + h) * kDv, (size_t)A.Hq * kDv,
                                A.part_lse + (int64_t)first * A.Hq + h, (size_t)A.Hq, nc, lane, out);
  __nv_bfloat16* op = A.o + row * kDv + lane * 16;
#pragma unroll
  for (int e = 0; e < 16; e += 2) *reinterpret_cast<uint32_t*>(op + e) = pack_bf16x2(out[e], out[e + 1]);
  if (A.lse && lane == 0) A.lse[row] = L;
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
  // tokens per chunk: given (rounded up to the tile), or about 2 CTAs' share per SM of the
  // whole token stream across all head groups, at least 4 tiles
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
    // the smallest chunk (a multiple of the tile, at least 4 tiles) whose items across all head
    // groups fit one wave of resident CTAs (two per SM): a second, partial wave would run a
    // full chunk after the first
    int dev = 0, sms = 0;
    STA_CUDA_TRY(cudaGetDevice(&dev));
    STA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int64_t slots = (int64_t)sms * 2, hg = Hq / kHeads;
    int64_t ch = std::max<int64_t>(4 * kTile, (T * hg + slots - 1) / slots);
    ch = (ch + kTile - 1) / kTile * kTile;
    while (ch < (1 << 30) && count_items((int)ch) * hg > slots) ch += std::max<int64_t>(kTile, ch / 32 / kTile * kTile);
    chunk = (int)std::min<int64_t>(ch, 1 << 30);
  }
  chunk = (chunk + kTile - 1) / kTile * kTile;
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
    mla_merge_kernel<<<(unsigned)(((int64_t)n_req * Hq + 7) / 8), 256, 0, st>>>(a);
    STA_LAUNCH_CHECK();
  }
  return STA_OK;
}
