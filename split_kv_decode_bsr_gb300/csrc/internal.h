// Internal launch interfaces between the C-ABI layer and the kernels.
#pragma once
#include "common.cuh"

namespace sta {

constexpr int kMaxHeads = 1024;

struct HeadMap {
  uint16_t m[kMaxHeads];      // attention head -> mask head
  uint16_t order[kMaxHeads];  // launch rank -> attention head (heaviest mask heads first)
};

struct MhaArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  MaskView mask;
  HeadMap hmap;
  int B, H, Lq, Lk, d;
  int dtype;
  float scale_log2;  // softmax scale * log2(e)
  int* err;          // device error word
};

sta_status launch_mha_row(const MhaArgs& a, cudaStream_t st);
sta_status launch_mha_block(const MhaArgs& a, cudaStream_t st);
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
  float scale_log2;
  int mode;         // 0: balanced token ranges, 1: fixed splits per request
  int splits;       // mode 1: s
  int range_len;    // mode 0: tokens per CTA range
  int n_ranges;     // mode 0: number of ranges (CTAs along x)
  int* err;
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
