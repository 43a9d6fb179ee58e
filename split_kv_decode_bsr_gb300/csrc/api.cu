// C-ABI entry points of libsta: host-side validation, the analytic kernel
// selector, the split planner, and the launches (all on the caller's stream).
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"

namespace sta {

// Device error word written by bounded waits that time out (first code wins).
__device__ int g_dev_error = 0;

static std::atomic<int> g_last_cuda_error{0};
void note_cuda_error(cudaError_t e) { g_last_cuda_error.store((int)e); }

int* device_error_word() {
  // one lookup per device, cached; the lock keeps first calls from several host threads apart
  static std::mutex mu;
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

namespace {

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Analytic selector (STOF カーネル選択: mask sparsity and sequence length decide
// between the row-wise and the block-wise kernel), per mask head when the mask carries
// per-head counts. Cost model:
//   block: every non-empty outer tile costs a 128x64 tile pair of MMAs and the softmax of
//          64x64 scores, whatever its fill:      t_b = tiles * 4096
//   row:   every valid (q, k) pair costs two row loads, FMA-pipe work and its share of a
//          batched warp reduction:               t_r = valid * kRowOverBlock(d)
// The ratio is the measured crossover on GB300. Unstructured masks over B=1, H=8, L=4096
// (every outer tile part; time in us, row / block):
//   density   0.1 %      0.2 %      0.4 %      1 %         2 %         5 %
//   d = 64    38 / 82    44 / 83    54 / 82    79 / 83     120 / 82    353 / 82
//   d = 128   44 / 80    50 / 80    62 / 80    99 / 80     158 / 80    444 / 80
// The block kernel's time does not follow the fill of its tiles (part tiles are bound by
// the softmax at both head sizes), the row kernel's follows the valid pairs; the two meet
// near 1.09 % density at d = 64 and 0.70 % at d = 128, i.e. the row kernel spends ~92x
// (d = 64) and ~143x (d = 128) the block kernel's time per computed pair on each valid pair.
double row_over_block(int d) { return d == 64 ? 92.0 : 143.0; }
constexpr int kMaxSplitsPrefill = 1024;

int choose(int64_t tiles, int64_t valid, int d) {
  const double t_block = (double)tiles * 4096.0;
  const double t_row = (double)valid * row_over_block(d);
  return t_row < t_block ? STA_KERNEL_ROW : STA_KERNEL_BLOCK;
}

// The choice for the whole mask (from its total counts).
int select_kernel(const sta_bsr_mask* m, int d, int Lk, sta_dtype dtype) {
  if (dtype != STA_BF16 || !block_kernel_supports(d, Lk, dtype)) return STA_KERNEL_ROW;
  return choose(m->n_full + m->n_part, m->n_valid, d);
}

// The choice for one mask head, when the mask carries per-head counts (else the mask's).
bool per_head_counts(const sta_bsr_mask* m) { return m->head_tiles != nullptr && m->head_valid != nullptr; }
int select_kernel_head(const sta_bsr_mask* m, int hm, int d, int Lk, sta_dtype dtype) {
  if (dtype != STA_BF16 || !block_kernel_supports(d, Lk, dtype)) return STA_KERNEL_ROW;
  if (!per_head_counts(m)) return select_kernel(m, d, Lk, dtype);
  return choose(m->head_tiles[hm], m->head_valid[hm], d);
}

sta_status check_mask(const sta_bsr_mask* mask, int Lq, int Lk) {
  if (!mask) return STA_ERR_INVALID_ARG;
  if (mask->Lq != Lq || mask->Lk != Lk || mask->n_mask_heads < 1) return STA_ERR_INVALID_ARG;
  if (mask->ot_rows != (int)cdiv(Lq, 64) || mask->ot_cols != (int)cdiv(Lk, 64)) return STA_ERR_INVALID_ARG;
  if (!mask->full_row_ptr || !mask->part_row_ptr) return STA_ERR_INVALID_ARG;
  if ((mask->n_full > 0 && !mask->full_col_idx) || (mask->n_part > 0 && (!mask->part_col_idx || !mask->part_bitmap)))
    return STA_ERR_INVALID_ARG;
  return STA_OK;
}

}  // namespace
}  // namespace sta

using namespace sta;

extern "C" const char* sta_status_string(sta_status s) {
  switch (s) {
    case STA_OK: return "ok";
    case STA_ERR_INVALID_ARG: return "invalid argument";
    case STA_ERR_UNSUPPORTED: return "unsupported configuration";
    case STA_ERR_WORKSPACE: return "workspace missing or too small";
    case STA_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

extern "C" int sta_last_cuda_error(void) { return g_last_cuda_error.load(); }

extern "C" const char* sta_last_cuda_error_string(void) {
  return cudaGetErrorString((cudaError_t)g_last_cuda_error.load());
}

extern "C" sta_status sta_device_error(int* code, int reset) {
  if (!code) return STA_ERR_INVALID_ARG;
  int* w = device_error_word();
  if (!w) return STA_ERR_CUDA;
  STA_CUDA_TRY(cudaMemcpy(code, w, sizeof(int), cudaMemcpyDeviceToHost));
  if (reset) STA_CUDA_TRY(cudaMemset(w, 0, sizeof(int)));
  return STA_OK;
}

extern "C" int sta_mha_select_kernel(const sta_bsr_mask* mask, int B, int H, int Lq, int Lk, int d, sta_dtype dtype) {
  if (B < 1 || H < 1 || (d != 64 && d != 128) || (dtype != STA_BF16 && dtype != STA_F32)) return -STA_ERR_INVALID_ARG;
  const sta_status st = check_mask(mask, Lq, Lk);
  if (st != STA_OK) return -st;
  if (!per_head_counts(mask)) return select_kernel(mask, d, Lk, dtype);
  int seen = 0;  // bit k-1: kernel k chosen for some mask head
  for (int hm = 0; hm < mask->n_mask_heads; ++hm) seen |= 1 << (select_kernel_head(mask, hm, d, Lk, dtype) - 1);
  return seen == 3 ? STA_KERNEL_MIXED : (seen == 2 ? STA_KERNEL_ROW : STA_KERNEL_BLOCK);
}

namespace {

// Shared validation of sta_mha_fwd / sta_mha_fwd_splitkv (everything but the
// data pointers): fills the kernel arguments and the kernel to run.
sta_status mha_prepare(const sta_bsr_mask* mask, const int32_t* head_map, int B, int H, int Lq, int Lk, int d,
                       sta_dtype dtype, float scale, int kernel, MhaArgs& a, int& which) {
  if (B < 1 || H < 1 || Lq < 1 || Lk < 1 || H > kMaxHeads || (int64_t)B * H > 65535) return STA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return STA_ERR_INVALID_ARG;
  if (dtype != STA_BF16 && dtype != STA_F32) return STA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return STA_ERR_UNSUPPORTED;
  if (kernel < STA_KERNEL_AUTO || kernel > STA_KERNEL_ROW) return STA_ERR_INVALID_ARG;
  const sta_status st = check_mask(mask, Lq, Lk);
  if (st != STA_OK) return st;
  memset(&a, 0, sizeof(a));
  const int Hm = mask->n_mask_heads;
  for (int h = 0; h < H; ++h) {
    int mh;
    if (head_map) mh = head_map[h];
    else if (Hm == 1) mh = 0;
    else if (Hm == H) mh = h;
    else return STA_ERR_INVALID_ARG;
    if (mh < 0 || mh >= Hm) return STA_ERR_INVALID_ARG;
    a.hmap.m[h] = (uint16_t)mh;
  }
  // launch order of the heads: heaviest mask heads first when their tile counts are known
  for (int h = 0; h < H; ++h) a.hmap.order[h] = (uint16_t)h;
  if (mask->head_tiles) {
    const int64_t* w = mask->head_tiles;
    std::stable_sort(a.hmap.order, a.hmap.order + H,
                     [&](uint16_t x, uint16_t y) { return w[a.hmap.m[x]] > w[a.hmap.m[y]]; });
  }
  a.n_ranks = H;
  if (kernel != STA_KERNEL_AUTO) {
    which = kernel;
  } else {
    int seen = 0;
    for (int h = 0; h < H; ++h) seen |= 1 << (select_kernel_head(mask, a.hmap.m[h], d, Lk, dtype) - 1);
    which = seen == 3 ? STA_KERNEL_MIXED : (seen == 2 ? STA_KERNEL_ROW : STA_KERNEL_BLOCK);
  }
  if (which == STA_KERNEL_BLOCK && !block_kernel_supports(d, Lk, dtype)) return STA_ERR_UNSUPPORTED;
  a.mask = MaskView{mask->full_row_ptr, mask->full_col_idx, mask->part_row_ptr, mask->part_col_idx,
                    mask->part_bitmap, static_cast<const uint8_t*>(mask->tile_lists), mask->ot_rows, mask->ot_cols,
                    mask->n_part, mask->n_full};
  if (mask->tile_lists && (mask->ot_cols > kMaxTileListCols || ((uintptr_t)mask->tile_lists & 15)))
    return STA_ERR_INVALID_ARG;
  a.B = B; a.H = H; a.Lq = Lq; a.Lk = Lk; a.d = d; a.dtype = dtype;
  a.scale_log2 = scale * kLog2e;
  return STA_OK;
}

// Under the per-head choice: the launch order split into the block-wise kernel's heads
// (kept in their heaviest-first order) and the row-wise kernel's.
void split_heads(const MhaArgs& a, const sta_bsr_mask* mask, MhaArgs& blk, MhaArgs& row) {
  blk = a;
  row = a;
  blk.n_ranks = row.n_ranks = 0;
  for (int r = 0; r < a.H; ++r) {
    const int h = a.hmap.order[r];
    if (select_kernel_head(mask, a.hmap.m[h], a.d, a.Lk, (sta_dtype)a.dtype) == STA_KERNEL_ROW)
      row.hmap.order[row.n_ranks++] = (uint16_t)h;
    else
      blk.hmap.order[blk.n_ranks++] = (uint16_t)h;
  }
}

// The library's second stream of a device (non-blocking) and the two events that fork it
// from and join it back into a caller's stream; one set per host thread and device, created
// on first use and kept until exit. Per thread, so that a capture in progress on one thread
// (which holds the side stream until the capture ends) cannot take in another thread's work.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

sta_status side_stream(SideStream*& out) {
  thread_local SideStream cache[64];
  int dev = 0;
  STA_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return STA_ERR_UNSUPPORTED;
  SideStream& c = cache[dev];
  if (!c.s) {  // all three or none: a failed creation leaves nothing half made
    SideStream n;
    cudaError_t e = cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (n.fork) cudaEventDestroy(n.fork);
      if (n.s) cudaStreamDestroy(n.s);
      note_cuda_error(e);
      return STA_ERR_CUDA;
    }
    c = n;
  }
  out = &c;
  return STA_OK;
}

// Both kernels at once: the row-wise kernel on its heads on the side stream (forked from
// and joined back into `st`), the block-wise kernel on the others on `st`.
sta_status launch_mixed(const MhaArgs& blk, const MhaSplit& plan, const MhaArgs& row, cudaStream_t st) {
  SideStream* ss = nullptr;
  sta_status r = side_stream(ss);
  if (r != STA_OK) return r;
  STA_CUDA_TRY(cudaEventRecord(ss->fork, st));
  STA_CUDA_TRY(cudaStreamWaitEvent(ss->s, ss->fork, 0));
  r = launch_mha_row(row, ss->s);
  STA_CUDA_TRY(cudaEventRecord(ss->join, ss->s));  // joined even after a failed launch
  const sta_status b = launch_mha_block(blk, plan, st);
  STA_CUDA_TRY(cudaStreamWaitEvent(st, ss->join, 0));
  return r != STA_OK ? r : b;
}

sta_status mha_set_data(MhaArgs& a, const void* q, const void* k, const void* v, void* o, float* lse) {
  if (!q || !k || !v || !o) return STA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return STA_ERR_UNSUPPORTED;
  if (lse && ((uintptr_t)lse & 3u)) return STA_ERR_UNSUPPORTED;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.err = device_error_word();
  return STA_OK;
}

}  // namespace

extern "C" sta_status sta_mha_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const sta_bsr_mask* mask, const int32_t* head_map, int B, int H, int Lq, int Lk,
                                  int d, sta_dtype dtype, float scale, int kernel, sta_stream stream) {
  if (!q || !k || !v || !o) return STA_ERR_INVALID_ARG;
  MhaArgs a;
  int which = 0;
  sta_status st = mha_prepare(mask, head_map, B, H, Lq, Lk, d, dtype, scale, kernel, a, which);
  if (st != STA_OK) return st;
  if ((st = mha_set_data(a, q, k, v, o, lse)) != STA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (which == STA_KERNEL_ROW) return launch_mha_row(a, s);
  MhaSplit plan;  // no split: one chunk per item
  if (which == STA_KERNEL_MIXED) {
    MhaArgs blk, row;
    split_heads(a, mask, blk, row);
    if ((st = plan_mha_split(blk, nullptr, 1, -1, plan)) != STA_OK) return st;
    return launch_mixed(blk, plan, row, s);
  }
  if ((st = plan_mha_split(a, nullptr, 1, -1, plan)) != STA_OK) return st;
  return launch_mha_block(a, plan, s);
}

extern "C" sta_status sta_mha_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse,
                                         const sta_bsr_mask* mask, const int32_t* head_map, int B, int H, int Lq,
                                         int Lk, int d, sta_dtype dtype, float scale, int kernel, int num_splits,
                                         int o_layout, void* workspace, size_t* workspace_bytes, sta_stream stream) {
  if (!workspace_bytes || num_splits < 0 || num_splits > kMaxSplitsPrefill) return STA_ERR_INVALID_ARG;
  if (o_layout != STA_O_BHLD && o_layout != STA_O_BLHD) return STA_ERR_INVALID_ARG;
  MhaArgs a;
  int which = 0;
  sta_status st = mha_prepare(mask, head_map, B, H, Lq, Lk, d, dtype, scale, kernel, a, which);
  if (st != STA_OK) return st;
  a.o_tokens = o_layout == STA_O_BLHD ? 1 : 0;
  if ((st = mha_set_data(a, q, k, v, o, lse)) != STA_OK && workspace) return st;
  // the block-wise kernel's heads: all of them, or its share under the per-head choice
  MhaArgs blk, row;
  if (which == STA_KERNEL_MIXED) split_heads(a, mask, blk, row);
  MhaArgs& ab = which == STA_KERNEL_MIXED ? blk : a;
  MhaSplit plan;
  size_t need = 256;  // never zero, so that a null workspace always means "query"
  if (which == STA_KERNEL_BLOCK || which == STA_KERNEL_MIXED) {
    if ((st = plan_mha_split(ab, mask->head_tiles, num_splits, -1, plan)) != STA_OK) return st;
    need = std::max(need, mha_split_workspace_bytes(ab, plan));
  }
  if (!workspace) {
    *workspace_bytes = need;
    return STA_OK;
  }
  if (*workspace_bytes < need) return STA_ERR_WORKSPACE;
  if ((uintptr_t)workspace & 255u) return STA_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (which == STA_KERNEL_ROW) return launch_mha_row(a, s);
  if (plan.n_split_ranks > 0) {
    const size_t rows = (size_t)plan.ybase[plan.n_split_ranks] * (size_t)Lq;
    plan.part_o = static_cast<float*>(workspace);
    plan.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             (((rows * (size_t)d * sizeof(float)) + 255) & ~(size_t)255));
  }
  if (which == STA_KERNEL_MIXED) return launch_mixed(blk, plan, row, s);
  return launch_mha_block(a, plan, s);
}

extern "C" sta_status sta_mha_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                                          const sta_bsr_mask* mask, const int32_t* head_map, int B, int H, int Lq,
                                          int Lk, int d, sta_dtype dtype, float scale, int kernel, int num_splits,
                                          void* workspace, size_t* workspace_bytes, sta_stream stream) {
  return sta_mha_fwd_layout(q, k, v, o, lse, mask, head_map, B, H, Lq, Lk, d, dtype, scale, kernel, num_splits,
                            STA_O_BHLD, workspace, workspace_bytes, stream);
}

namespace sta {

sta_status decode_setup(const int32_t* indptr_host, int n_req, int Hq, int Hkv, int d, sta_dtype dtype, int num_splits,
                        DecodeArgs& a, int64_t& T) {
  if (!indptr_host || n_req < 1 || Hq < 1 || Hkv < 1 || num_splits < 0 || num_splits > 4096)
    return STA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return STA_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return STA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return STA_ERR_UNSUPPORTED;
  if (dtype != STA_BF16) return STA_ERR_UNSUPPORTED;
  if (indptr_host[0] != 0) return STA_ERR_INVALID_ARG;
  for (int r = 0; r < n_req; ++r)
    if (indptr_host[r + 1] < indptr_host[r]) return STA_ERR_INVALID_ARG;
  T = indptr_host[n_req];
  if ((int64_t)n_req * Hq > INT32_MAX / 2) return STA_ERR_INVALID_ARG;
  memset(&a, 0, sizeof(a));
  a.n_req = n_req; a.Hq = Hq; a.Hkv = Hkv; a.d = d;
  a.T = (int)T;
  a.mode = num_splits == 0 ? 0 : 1;
  a.splits = num_splits;
  int dev = 0;
  STA_CUDA_TRY(cudaGetDevice(&dev));
  return decode_plan(a, T, dev);
}

}  // namespace sta

namespace {
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

namespace {

// Shared body of the contiguous and the paged decode entry points.
sta_status decode_call(const void* q, const void* k, const void* v, const int32_t* kv_indptr_dev,
                       const int32_t* kv_indptr_host, int n_req, int Hq, int Hkv, int d, sta_dtype dtype, float scale,
                       int num_splits, void* o, float* lse, void* workspace, size_t* workspace_bytes,
                       cudaStream_t stream, int page_size, int n_pages, const int32_t* page_indptr,
                       const int32_t* page_indices) {
  if (!workspace_bytes) return STA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return STA_ERR_INVALID_ARG;
  DecodeArgs a;
  int64_t T = 0;
  sta_status st = decode_setup(kv_indptr_host, n_req, Hq, Hkv, d, dtype, num_splits, a, T);
  if (st != STA_OK) return st;
  const size_t slots = decode_slots(a);
  const size_t o_bytes = align256(slots * (size_t)Hq * d * sizeof(float));
  const size_t need = o_bytes + align256(slots * (size_t)Hq * sizeof(float));
  if (!workspace) {
    *workspace_bytes = need;
    return STA_OK;
  }
  if (*workspace_bytes < need) return STA_ERR_WORKSPACE;
  if (!q || !kv_indptr_dev || !o) return STA_ERR_INVALID_ARG;
  if (T > 0 && (!k || !v)) return STA_ERR_INVALID_ARG;  // K/V may be empty (NULL) only when T == 0
  if (page_size > 0 && T > 0 && (!page_indptr || !page_indices || n_pages < 1)) return STA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || ((uintptr_t)workspace & 255u))
    return STA_ERR_UNSUPPORTED;
  a.q = q; a.k = k; a.v = v; a.kv_indptr = kv_indptr_dev; a.o = o; a.lse = lse;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes);
  a.scale_log2 = scale * kLog2e;
  a.err = device_error_word();
  a.page_size = page_size;
  a.n_pages = n_pages;
  a.page_indptr = page_indptr;
  a.page_indices = page_indices;
  return launch_decode(a, stream);
}

}  // namespace

extern "C" sta_status sta_decode_splitkv(const void* q, const void* k, const void* v, const int32_t* kv_indptr_dev,
                                         const int32_t* kv_indptr_host, int n_req, int Hq, int Hkv, int d,
                                         sta_dtype dtype, float scale, int num_splits, void* o, float* lse,
                                         void* workspace, size_t* workspace_bytes, sta_stream stream) {
  return decode_call(q, k, v, kv_indptr_dev, kv_indptr_host, n_req, Hq, Hkv, d, dtype, scale, num_splits, o, lse,
                     workspace, workspace_bytes, (cudaStream_t)stream, 0, 0, nullptr, nullptr);
}

extern "C" sta_status sta_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages, int page_size,
                                               int n_pages, const int32_t* page_indptr_dev,
                                               const int32_t* page_indices_dev, const int32_t* kv_indptr_dev,
                                               const int32_t* kv_indptr_host, int n_req, int Hq, int Hkv, int d,
                                               sta_dtype dtype, float scale, int num_splits, void* o, float* lse,
                                               void* workspace, size_t* workspace_bytes, sta_stream stream) {
  if (page_size < 1 || n_pages < 0) return STA_ERR_INVALID_ARG;
  return decode_call(q, k_pages, v_pages, kv_indptr_dev, kv_indptr_host, n_req, Hq, Hkv, d, dtype, scale,
                     num_splits, o, lse, workspace, workspace_bytes, (cudaStream_t)stream, page_size, n_pages,
                     page_indptr_dev, page_indices_dev);
}

extern "C" sta_status sta_merge_lse(const float* part_o, const float* part_lse, int n_rows, int s, int d, void* o,
                                    sta_dtype o_dtype, float* lse, sta_stream stream) {
  if (n_rows < 0 || s < 1 || s > 4096) return STA_ERR_INVALID_ARG;
  if (o_dtype != STA_BF16 && o_dtype != STA_F32) return STA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128 && d != 256) return STA_ERR_UNSUPPORTED;
  if (n_rows == 0) return STA_OK;
  if (!part_o || !part_lse || !o) return STA_ERR_INVALID_ARG;
  if ((uintptr_t)part_o & 15u) return STA_ERR_UNSUPPORTED;  // partials are read 16 bytes at a time
  return launch_merge_public(part_o, part_lse, n_rows, s, d, o, o_dtype, lse, (cudaStream_t)stream);
}
