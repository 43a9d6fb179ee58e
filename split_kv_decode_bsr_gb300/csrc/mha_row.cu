// Row-wise masked MHA kernel (STOF, デュアルカーネル戦略 / 行方向カーネル):
// Q sliced by rows, one warp per query row, warp shuffles for the softmax
// reductions and no synchronisation between warps. The warp walks only the
// non-empty outer tiles of its row: full tiles 32 keys at a time (one key per
// lane), part tiles through the row's bytes of their inner-tile words, skipping
// empty inner tiles and scoring each valid key with the head dimensions spread
// over the lanes. Scores fold into an fp32 online softmax (running max m,
// running sum l, output rescaled by exp2(m_old - m_new)). Handles bf16 and fp32
// inputs, head dims 64 and 128.
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kRowWarps + warp;
  if (i >= A.Lq) return;
  const int64_t bh = blockIdx.y;
  const int h = (int)(bh % A.H);
  const int hm = A.hmap.m[h];
  const int64_t qrow = bh * A.Lq + i;
  const int64_t kv0 = bh * A.Lk;  // first K/V row of this (b, h)
  float qd[E];                     // this lane's dimensions of q, pre-scaled
  IO::load_lane(A.q, qrow, lane, qd);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qd[e] *= A.scale_log2;
    s_q[warp][lane * E + e] = qd[e];
  }
  __syncwarp();
  const float* sq = s_q[warp];
  const int a = i >> 6, r = i & 63;
  const int64_t mrow = (int64_t)hm * A.mask.ot_rows + a;
  // CSR ranges clamped to the arrays (a damaged mask cannot send the loops past them)
  const int fb = max(A.mask.full_row_ptr[mrow], 0), fe = (int)min((int64_t)A.mask.full_row_ptr[mrow + 1], A.mask.n_full);
  const int pb = max(A.mask.part_row_ptr[mrow], 0), pe = (int)min((int64_t)A.mask.part_row_ptr[mrow + 1], A.mask.n_part);

  float m = -INFINITY, l = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  // ---- full tiles: every key in range is valid
  for (int t = fb; t < fe; ++t) {
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

  // ---- part tiles: the row's byte of each inner-tile word, four tiles per pass (lane
  // 8u + w holds word w of tile u); the words of the next pass are requested before the
  // keys of this one are processed
  const int wrow = 8 * (r >> 3), sh = (r & 7) * 8;
  auto scan = [&](int t0, uint32_t& byte, int& col) {
    const int tt = t0 + (lane >> 3), w = lane & 7;
    byte = 0u;
    col = 0;
    if (tt < pe) {
      byte = (uint32_t)((__ldg(A.mask.part_bitmap + (int64_t)tt * 64 + wrow + w) >> sh) & 0xFFull);
      col = __ldg(A.mask.part_col_idx + tt);
    }
  };
  uint32_t byte_next;
  int col_next;
  scan(pb, byte_next, col_next);
  for (int t0 = pb; t0 < pe; t0 += 4) {
    const uint32_t byte = byte_next;
    const int col = col_next;
    if (t0 + 4 < pe) scan(t0 + 4, byte_next, col_next);
    unsigned nz = __ballot_sync(0xffffffffu, byte != 0u);
    while (nz) {
      const int src = __ffs(nz) - 1;
      nz &= nz - 1;
      uint32_t bits = __shfl_sync(0xffffffffu, byte, src);
      // column and key clamped into the mask: a damaged mask (sta_validate_mask finds it)
      // gives wrong values but no read outside K and V
      const unsigned colv = min((unsigned)__shfl_sync(0xffffffffu, col, src), (unsigned)A.mask.ot_cols - 1u);
      const int64_t base = (int64_t)colv * 64 + 8 * (src & 7);
      while (bits) {
        const int c = __ffs(bits) - 1;
        bits &= bits - 1;
        const int64_t j = kv0 + min(base + c, (int64_t)A.Lk - 1);
        float kd[E], vd[E];
        IO::load_lane(A.k, j, lane, kd);
        IO::load_lane(A.v, j, lane, vd);
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(qd[e], kd[e], part);
        const float sc = warp_sum(part);
        if (sc > m) {  // new running max: rescale what has been accumulated (m = -inf -> 0)
          const float alpha = exp2f(m - sc);
          l *= alpha;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] *= alpha;
          m = sc;
        }
        const float p = exp2f(sc - m);
        l += p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vd[e], acc[e]);
      }
    }
  }

  float out[E];
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = acc[e] * inv;
  IO::store_lane(A.o, o_row(A, bh / A.H, h, i), lane, out);
  if (A.lse && lane == 0) A.lse[qrow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace

sta_status launch_mha_row(const MhaArgs& a, cudaStream_t st) {
  const dim3 grid((unsigned)cdiv(a.Lq, kRowWarps), (unsigned)(a.B * a.H));
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
