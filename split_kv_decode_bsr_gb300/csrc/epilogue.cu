// Fused epilogue after the attention output projection (STOF, 手法 / 演算子融合モジュール,
// with a fixed rule in place of the search): bias add, residual add and layer
// normalisation of each row in one pass over HBM.
//
// A row of n elements is spread over TPR threads (a warp, four warps or sixteen warps,
// the smallest that leaves each thread at most kMaxVec 16-byte vectors); thread t of the
// row takes vectors t, t + TPR, ... (each load instruction of a warp covers 512
// consecutive bytes). The pre-norm sum stays in registers between the two reductions
// (mean, then the mean square deviation from it), so every input element is read once
// and every output element written once.
#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace sta {
namespace {

constexpr int kMaxVec = 4;  // at most this many 16-byte vectors (8 bf16) per thread and row

__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(u[k] << 16);
    f[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Sum over the TPR threads of a row: warp shuffles, then (TPR > 32) the row's warps
// through shared memory. Every thread of the block calls it (uniform control flow).
template <int TPR>
__device__ __forceinline__ float row_sum(float v, float* s_part) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if constexpr (TPR == 32) {
    return v;
  } else {
    constexpr int W = TPR / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp / W;  // row group of this warp within the block
    __syncthreads();         // s_part free (an earlier call may still be reading it)
    if (lane == 0) s_part[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int x = 0; x < W; ++x) t += s_part[g * W + x];
    return t;
  }
}

// grid ceil(rows / (blockDim / TPR)); blockDim = max(TPR, 256); VEC vectors per thread.
template <int TPR, int VEC>
__global__ void __launch_bounds__(TPR > 256 ? TPR : 256) bias_residual_ln_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ bias,
    const __nv_bfloat16* __restrict__ residual, const float* __restrict__ gamma, const float* __restrict__ beta,
    __nv_bfloat16* __restrict__ y, __nv_bfloat16* __restrict__ h_out, int64_t rows, int n, float eps) {
  __shared__ float s_part[(TPR > 256 ? TPR : 256) / 32];
  const int rows_per_block = blockDim.x / TPR;
  const int t = threadIdx.x % TPR;
  const int64_t row = (int64_t)blockIdx.x * rows_per_block + threadIdx.x / TPR;
  const bool live = row < rows;  // a block's last rows may be past the end: they still join the reductions
  const int nv = n >> 3;         // vectors per row
  const float inv_n = 1.f / (float)n;
  float h[VEC][8];
  const uint4* xr = reinterpret_cast<const uint4*>(x + (live ? row : 0) * (int64_t)n);
  const uint4* rr = residual ? reinterpret_cast<const uint4*>(residual + (live ? row : 0) * (int64_t)n) : nullptr;
  uint4 xw[VEC], rw[VEC];
#pragma unroll
  for (int k = 0; k < VEC; ++k) {  // every load of the thread in flight at once
    const int v = t + k * TPR;
    const bool in = live && v < nv;
    xw[k] = in ? __ldcs(xr + v) : make_uint4(0, 0, 0, 0);
    rw[k] = in && rr ? __ldcs(rr + v) : make_uint4(0, 0, 0, 0);
  }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int v = t + k * TPR;
    float a[8], r[8], b[8];
    unpack8(xw[k], a);
    unpack8(rw[k], r);
    if (bias && v < nv) unpack8(__ldg(reinterpret_cast<const uint4*>(bias) + v), b);
    else {
#pragma unroll
      for (int e = 0; e < 8; ++e) b[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      h[k][e] = (a[e] + b[e]) + r[e];  // zero past the row (all three operands are zero there)
      sum += h[k][e];
    }
  }
  const float mean = row_sum<TPR>(sum, s_part) * inv_n;
  float sq = 0.f;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    if (t + k * TPR < nv) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float dlt = h[k][e] - mean;
        sq = fmaf(dlt, dlt, sq);
      }
    }
  }
  const float var = row_sum<TPR>(sq, s_part) * inv_n;
  const float rstd = 1.f / sqrtf(var + eps);
  if (!live) return;
  uint4* yr = reinterpret_cast<uint4*>(y + row * (int64_t)n);
  uint4* hr = h_out ? reinterpret_cast<uint4*>(h_out + row * (int64_t)n) : nullptr;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int v = t + k * TPR;
    if (v >= nv) continue;
    float g[8], bt[8], o[8];
    if (gamma) {
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v + 1);
      g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w; g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) g[e] = 1.f;
    }
    if (beta) {
      const float4 b0 = __ldg(reinterpret_cast<const float4*>(beta) + 2 * v);
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(beta) + 2 * v + 1);
      bt[0] = b0.x; bt[1] = b0.y; bt[2] = b0.z; bt[3] = b0.w; bt[4] = b1.x; bt[5] = b1.y; bt[6] = b1.z; bt[7] = b1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) bt[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = fmaf((h[k][e] - mean) * rstd, g[e], bt[e]);
    __stcs(yr + v, pack8(o));
    if (hr) __stcs(hr + v, pack8(h[k]));
  }
}

template <int TPR, int VEC>
sta_status launch_ln(const void* x, const void* bias, const void* residual, const float* gamma, const float* beta,
                     void* y, void* h_out, int64_t rows, int n, float eps, cudaStream_t st) {
  constexpr int threads = TPR > 256 ? TPR : 256;
  constexpr int rpb = threads / TPR;
  const int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > INT32_MAX) return STA_ERR_INVALID_ARG;
  bias_residual_ln_kernel<TPR, VEC><<<(unsigned)blocks, threads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(bias),
      static_cast<const __nv_bfloat16*>(residual), gamma, beta, static_cast<__nv_bfloat16*>(y),
      static_cast<__nv_bfloat16*>(h_out), rows, n, eps);
  STA_LAUNCH_CHECK();
  return STA_OK;
}

}  // namespace

// Threads per row for a row of n elements: the smallest of 32, 128, 512 that leaves each
// thread at most kMaxVec vectors of 8 elements.
int ln_threads_per_row(int n) {
  const int nv = n / 8;
  if (nv <= 32 * kMaxVec) return 32;
  if (nv <= 128 * kMaxVec) return 128;
  return 512;
}

}  // namespace sta

using namespace sta;

extern "C" sta_status sta_bias_residual_layernorm(const void* x, const void* bias, const void* residual,
                                                  const float* gamma, const float* beta, void* y, void* h_out,
                                                  int64_t rows, int n, float eps, sta_dtype dtype,
                                                  sta_stream stream) {
  if (rows < 0 || n < 8 || n > kMaxLayerNormCols || (n & 7) || !(eps > 0.f) || !isfinite(eps))
    return STA_ERR_INVALID_ARG;
  if (dtype != STA_BF16) return STA_ERR_UNSUPPORTED;
  if (rows == 0) return STA_OK;
  if (!x || !y) return STA_ERR_INVALID_ARG;
  const void* ptrs[7] = {x, bias, residual, gamma, beta, y, h_out};
  for (const void* p : ptrs)
    if (p && ((uintptr_t)p & 15)) return STA_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  switch (ln_threads_per_row(n)) {
    case 32: return launch_ln<32, kMaxVec>(x, bias, residual, gamma, beta, y, h_out, rows, n, eps, st);
    case 128: return launch_ln<128, kMaxVec>(x, bias, residual, gamma, beta, y, h_out, rows, n, eps, st);
    default: return launch_ln<512, kMaxVec>(x, bias, residual, gamma, beta, y, h_out, rows, n, eps, st);
  }
}
