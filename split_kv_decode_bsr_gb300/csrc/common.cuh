// Shared device/host helpers of libsta (CUDA path only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sta.h"

#define STA_OT 64  // outer tile edge
#define STA_IT 8   // inner tile edge

namespace sta {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// bf16 <-> f32 without library conversions on the hot path: widening is exact.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kMaxLayerNormCols = 512 * 4 * 8;  // row length of the fused layer norm: 512 threads x 4 vectors of 8
constexpr int kMaxTileListCols = 1024;  // OT columns the block-wise kernel (and its column lists) support

// Size of the block-wise kernel's per-query-tile column lists (0 if not available).
size_t tile_lists_bytes(int Hm, int Lq, int Lk);

// Device copy of the encoded-mask arrays a kernel needs.
struct MaskView {
  const int32_t* full_row_ptr;
  const int32_t* full_col_idx;
  const int32_t* part_row_ptr;
  const int32_t* part_col_idx;
  const uint64_t* part_bitmap;
  const uint8_t* tile_lists;  // optional, see sta_bsr_mask::tile_lists
  int32_t ot_rows, ot_cols;
  int64_t n_part;              // part tiles (bounds the bitmap reads of the block-wise kernel)
  int64_t n_full;              // full tiles (with n_part, bounds the CSR ranges the kernels read)
};

// Row r (0..63) of a part outer tile: 64-bit key mask, bit c = column c of the tile.
// Byte (r % 8) of IT word 8*(r/8) + q holds columns 8q..8q+7 of that row.
__device__ __forceinline__ uint64_t part_row_bits(const uint64_t* words, int r) {
  // the 32-bit half of each word that holds byte r % 8, then byte r % 4 of each gathered
  const uint32_t* w = reinterpret_cast<const uint32_t*>(words + 8 * (r >> 3)) + ((r >> 2) & 1);
  const uint32_t b = (uint32_t)(r & 3), sel = b | ((4u + b) << 4);
  const uint32_t x01 = __byte_perm(w[0], w[2], sel), x23 = __byte_perm(w[4], w[6], sel);
  const uint32_t x45 = __byte_perm(w[8], w[10], sel), x67 = __byte_perm(w[12], w[14], sel);
  return (uint64_t)__byte_perm(x01, x23, 0x5410) | ((uint64_t)__byte_perm(x45, x67, 0x5410) << 32);
}

// Merge s partials of one row; lane owns E consecutive dims. po points at the
// row's first partial, consecutive partials `ostride` floats apart; lse values
// `lstride` apart. Writes out[E] and returns the merged LSE. The partials are
// added in order 0..s-1. The first 32 LSEs (one per lane) and the first U
// partials' values are loaded together, before the maximum is known, and later
// partials U at a time, so that a row costs about one memory round trip per U
// partials instead of one per partial.
template <int E>
__device__ __forceinline__ void load_dims(const float* p, float* v) {
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(p) + q);
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
  } else if constexpr (E % 2 == 0) {
#pragma unroll
    for (int q = 0; q < E / 2; ++q) {
      const float2 x = __ldg(reinterpret_cast<const float2*>(p) + q);
      v[2 * q] = x.x; v[2 * q + 1] = x.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = __ldg(p + e);
  }
}

template <int E>
__device__ __forceinline__ float merge_row(const float* po, size_t ostride, const float* pl, size_t lstride, int s,
                                           int lane, float* out) {
  constexpr int U = E >= 8 ? 2 : 4;  // partials in flight per lane
  const float lse_l = lane < s ? __ldg(pl + (size_t)lane * lstride) : -INFINITY;
  float v[U][E];
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (u < s) load_dims<E>(po + (size_t)u * ostride + lane * E, v[u]);
  float M = lse_l;
  for (int i = lane + 32; i < s; i += 32) M = fmaxf(M, __ldg(pl + (size_t)i * lstride));
  M = warp_max(M);
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = 0.f;
  if (M == -INFINITY) return -INFINITY;
  float wsum = 0.f;
  for (int i0 = 0; i0 < s; i0 += 32) {
    const int nb = min(32, s - i0);
    // lane j: the weight of partial i0 + j
    const float x = i0 == 0 ? lse_l : (lane < nb ? __ldg(pl + (size_t)(i0 + lane) * lstride) : -INFINITY);
    const float wl = lane < nb ? exp2f((x - M) * kLog2e) : 0.f;
    for (int j = 0; j < nb; j += U) {
      if (i0 + j > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (j + u < nb) load_dims<E>(po + (size_t)(i0 + j + u) * ostride + lane * E, v[u]);
      }
      float w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) w[u] = __shfl_sync(0xffffffffu, wl, min(j + u, 31));
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (j + u < nb) {
          wsum += w[u];
#pragma unroll
          for (int e = 0; e < E; ++e) out[e] = fmaf(w[u], v[u][e], out[e]);
        }
      }
    }
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] *= inv;
  return M + logf(wsum);
}

}  // namespace sta

namespace sta {
// Records the CUDA error behind the most recent STA_ERR_CUDA (see sta_last_cuda_error).
void note_cuda_error(cudaError_t e);
}  // namespace sta

#define STA_CUDA_TRY(expr)                          \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) {                        \
      sta::note_cuda_error(e_);                     \
      return STA_ERR_CUDA;                          \
    }                                               \
  } while (0)

#define STA_LAUNCH_CHECK()                          \
  do {                                              \
    cudaError_t e_ = cudaGetLastError();            \
    if (e_ != cudaSuccess) {                        \
      sta::note_cuda_error(e_);                     \
      return STA_ERR_CUDA;                          \
    }                                               \
  } while (0)
