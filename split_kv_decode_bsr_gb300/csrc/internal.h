// Internal launch interfaces between the C-ABI layer and the kernels.
#pragma once
#include "common.cuh"

namespace sta {

constexpr int kMaxHeads = 1024;

struct HeadMap {
  uint16_t m[kMaxHeads];      // attention head -> mask head
  uint16_t order[kMaxHeads];  // launch rank -> attention head (heaviest mask heads first)
};
// A launch covers the attention heads order[0 .. n_ranks-1] of the launch order: all H
// heads, or under the per-head kernel choice the heads of one kernel.

struct MhaArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  MaskView mask;
  HeadMap hmap;
  int B, H, Lq, Lk, d;
  int n_ranks;       // heads of this launch: hmap.order[0 .. n_ranks-1]
  int dtype;
  float scale_log2;  // softmax scale * log2(e)
  int* err;          // device error word
  int o_tokens;      // 0: O is [B, H, Lq, d]; 1: O is [B, Lq, H, d] (heads merged per token)
};

// Row of d elements of O holding (b, h, query row i), in either layout.
__host__ __device__ inline int64_t o_row(const MhaArgs& a, int64_t b, int64_t h, int64_t i) {
  return a.o_tokens ? (b * a.Lq + i) * a.H + h : (b * a.H + h) * a.Lq + i;
}

// Split-KV plan of the block kernel (Cleave, Split演算子によるSplit-Kの対応 applied to
// the key-tile loop). grid.y enumerates (launch rank, batch, chunk): rank r covers
// grid.y indices ybase[r] .. ybase[r+1]-1 as b * s[r] + c. The key-tile list of a
// (query tile, b, h) item with n tiles is cut into s[r] chunks, chunk c taking
// tiles [c*n/s, (c+1)*n/s). Ranks with s > 1 form a prefix of the launch order
// (ranks 0 .. n_split_ranks-1); their chunks write normalised fp32 partials at
// partial row y * Lq + i (y = grid.y index), merged afterwards by log-sum-exp.
struct MhaSplit {
  float* part_o;     // [ybase[n_split_ranks], Lq, d] fp32, or null when nothing is split
  float* part_lse;   // [ybase[n_split_ranks], Lq] fp32 (natural log)
  int n_split_ranks;
  int uniform_s;     // > 0: every rank has s = uniform_s (ybase[r] = r * B * uniform_s)
  int n_y;           // grid.y
  int32_t ybase[kMaxHeads + 1];
  uint16_t s[kMaxHeads];
};

// Fills the plan: s per launch rank from num_splits (> 0: that many chunks for
// every head) or, when num_splits == 0, from the mask heads' tile counts
// (mask_head_tiles, may be null: no split) against the resident CTA slots of
// `device` (-1: the current device; queried only in that last case).
sta_status plan_mha_split(const MhaArgs& a, const int64_t* mask_head_tiles, int num_splits, int device, MhaSplit& p);
size_t mha_split_workspace_bytes(const MhaArgs& a, const MhaSplit& p);

sta_status launch_mha_row(const MhaArgs& a, cudaStream_t st);
sta_status launch_mha_block(const MhaArgs& a, const MhaSplit& p, cudaStream_t st);
bool block_kernel_supports(int d, int Lk, int dtype);

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* kv_indptr;
  void* o;
  float* lse;
  float* part_o;    // [slots, Hq, d]
  float* part_lse;  // [slots, Hq]
  int n_req, Hq, Hkv, d;
  int T;            // tokens (the host copy's kv_indptr[n_req]); device ranges are kept inside it
  float scale_log2;
  int mode;         // 0: balanced token ranges, 1: fixed splits per request
  int splits;       // mode 1: s
  int range_len;    // mode 0: tokens per CTA range
  int n_ranges;     // mode 0: number of ranges (CTAs along x)
  int* err;
  // paged K/V (page_size > 0): k and v are [n_pages, page_size, Hkv, d]; token i of request r
  // (0-based within the request) is slot i % page_size of page page_indices[page_indptr[r] + i / page_size]
  int page_size;
  int n_pages;
  const int32_t* page_indptr;
  const int32_t* page_indices;
};

// Host validation of the decode arguments and the split plan (fills a, T).
sta_status decode_setup(const int32_t* indptr_host, int n_req, int Hq, int Hkv, int d, sta_dtype dtype, int num_splits,
                        DecodeArgs& a, int64_t& T);

// Chooses the launch shape; fills range_len / n_ranges for mode 0.
sta_status decode_plan(DecodeArgs& a, int64_t total_tokens, int device);
size_t decode_slots(const DecodeArgs& a);
sta_status launch_decode(const DecodeArgs& a, cudaStream_t st);

// Generic merge of partial (O, lse) rows.
sta_status launch_merge_public(const float* part_o, const float* part_lse, int n_rows, int s, int d, void* o,
                               int o_dtype, float* lse, cudaStream_t st);

int* device_error_word();  // address of the library's device error word (current device)

}  // namespace sta
