/*
 * sta.h -- C ABI of libsta: masked multi-head attention over a two-level
 * (BSR + bitmap) mask, split-KV decode (GQA over packed or paged KV, and
 * against a shared latent KV cache) with a log-sum-exp merge, and the fused
 * operators that follow the attention, for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations:
 *  - "Accelerating Sparse Transformer Inference on GPU" (STOF):
 *      問題定義 -- masked MHA with causal, sliding-window and random masks;
 *      手法 / 統合 MHA モジュール / 2 段階ストレージ形式 -- outer tiles that are
 *      empty (skipped), full or part, tracked by pointer arrays, and one uint64
 *      bitmap per 8x8 inner tile of a part tile;
 *      デュアルカーネル戦略 / カーネル選択 -- a row-wise kernel for short, highly
 *      sparse cases, a block-wise kernel for the general case, and an analytic
 *      model that picks between them.
 *      演算子融合モジュール -- fusion of the MHA layer with the operators after
 *      it (here by a fixed rule: sta_mha_fwd_layout, sta_bias_residual_layernorm).
 *  - "Cleave: Scaling Tensor Program Optimization via Decoupled Algebraic
 *    Search and Operator Scheduling": Split演算子によるSplit-Kの対応 and the
 *    abstract -- a Split operator with split count s parallelises a reduction
 *    dimension (FlashDecoding); the partial softmax results are merged;
 *    評価結果 -- MLA among the measured LLM subgraphs (sta_mla_decode).
 *
 * Conventions (the pages leave these open; plainest readings):
 *  - Q, K, V, O are [B, H, L, d] row-major, d innermost (decode: Q/O
 *    [n_req, Hq, d], K/V packed [T, Hkv, d]). LSE is float32, natural log.
 *  - Mask element 1 = key may be attended (additive 0), 0 = masked (-inf).
 *  - Outer tiles (OT) are 64x64; inner tiles (IT) 8x8. A part OT stores 64
 *    uint64 words, ITs row-major (word 8p+q covers OT rows 8p..8p+7, cols
 *    8q..8q+7); bit 8r+c of a word is element (row r, col c) of its IT.
 *    An OT is full only if all 4096 elements are in range and valid; edge
 *    tiles are part with out-of-range bits 0. col_idx is ascending per row.
 *  - A query row with no valid key yields O = 0 and LSE = -inf.
 *
 * Ownership and errors: every pointer to tensor data is a DEVICE pointer
 * owned by the caller unless marked "host". The library allocates no device
 * memory, launches only on the given stream (asynchronously) and synchronises
 * only where a function says so. Arguments are validated on the host before
 * anything is launched; on error nothing is launched and an sta_status other
 * than STA_OK is returned (see sta_status_string). STA_ERR_CUDA reports a
 * launch error from the CUDA runtime.
 */
#ifndef STA_H_
#define STA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int sta_status;
#define STA_OK 0
#define STA_ERR_INVALID_ARG 1  /* null pointer, bad size, inconsistent arguments */
#define STA_ERR_UNSUPPORTED 2  /* dtype / head dim / alignment the library does not handle */
#define STA_ERR_WORKSPACE 3    /* workspace missing or too small */
#define STA_ERR_CUDA 4         /* the CUDA runtime reported an error */

typedef int sta_dtype;
#define STA_BF16 0
#define STA_F32 1

/* cudaStream_t; NULL is the legacy default stream. */
typedef void* sta_stream;

/* ------------------------------------------------------------------------ */
/* Mask sources and the encoded mask                                         */
/* ------------------------------------------------------------------------ */

#define STA_MASK_PATTERN 0    /* predicate below, no data                     */
#define STA_MASK_DENSE_U8 1   /* data: uint8 [Lq][Lk], nonzero = valid        */
#define STA_MASK_DENSE_BITS 2 /* data: uint64 [Lq][ceil(Lk/64)], element (i,j) */
                              /* at word j>>6, bit j&63; bits j >= Lk ignored  */

/* One [Lq, Lk] mask head. For STA_MASK_PATTERN:
 *   valid(i,j) = (!causal || j <= i) &&
 *                ((win_lo <= j-i && j-i <= win_hi) || j < n_global_cols)
 * which covers causal, sliding-window, banded and global-column masks. */
typedef struct {
  int32_t kind;
  int32_t causal;
  int64_t win_lo, win_hi;
  int64_t n_global_cols;
  const void* data; /* device pointer for the DENSE kinds, else NULL */
} sta_mask_src;

/* Two-level mask for Hm mask heads (STOF 2 段階ストレージ形式). Row index
 * of both CSR structures is hm * ot_rows + a (mask head hm, OT row a);
 * col_idx holds OT column numbers. part_bitmap[t*64 + w] is IT word w of the
 * t-th part tile. Device arrays are caller-owned; n_* are host copies. */
typedef struct {
  int32_t n_mask_heads, Lq, Lk, ot_rows, ot_cols;
  int32_t* full_row_ptr; /* [Hm*ot_rows + 1] */
  int32_t* full_col_idx; /* [n_full]         */
  int32_t* part_row_ptr; /* [Hm*ot_rows + 1] */
  int32_t* part_col_idx; /* [n_part]         */
  uint64_t* part_bitmap; /* [n_part * 64]    */
  int64_t n_full, n_part, n_valid;
  /* Optional HOST array [Hm] (caller-owned) or NULL. When set, the size query
   * of sta_encode_mask stores each mask head's number of non-empty outer tiles
   * there, and sta_mha_fwd then starts the query tiles of the heaviest heads
   * first (load balance); results do not depend on it. */
  int64_t* head_tiles;
  /* Optional DEVICE buffer of sta_tile_lists_bytes(Hm, Lq, Lk) bytes (caller-
   * owned, 16-byte aligned) or NULL. When set, the fill call of sta_encode_mask
   * also writes the column lists of the block-wise kernel there, and
   * sta_mha_fwd / sta_mha_fwd_splitkv then read the list of each 128-row query
   * tile with one copy instead of merging its two outer-tile rows themselves;
   * results do not depend on it. Layout: T = ceil(ot_rows / 2) query tiles per
   * mask head, Cp = ot_cols rounded up to a multiple of 8, one slot of
   * 16 + 10 * Cp bytes per (hm, t) at slot index hm * T + t:
   *   int32 n, 12 zero bytes          number of entries
   *   uint16 col[Cp]                  ascending OT columns non-empty in OT row
   *                                   2t or 2t+1 (entries >= n undefined)
   *   int32 kind_a[Cp], kind_b[Cp]    per entry, for OT rows 2t and 2t+1: -1
   *                                   empty, -2 full, >= 0 index of the part
   *                                   tile (row 2t+1 beyond ot_rows is empty)
   * Only for ot_cols <= 1024 (the block-wise kernel's limit). */
  void* tile_lists;
  /* Optional HOST array [Hm] (caller-owned) or NULL. When set, the size query
   * of sta_encode_mask stores each mask head's number of valid elements there.
   * With head_tiles and head_valid both set, STA_KERNEL_AUTO chooses the kernel
   * per mask head (STOF カーネル選択 per head group) instead of once for the
   * whole mask; results do not depend on it beyond rounding. */
  int64_t* head_valid;
} sta_bsr_mask;

/* sta_validate_mask -- check a two-level mask whose arrays are HOST copies
 * (full_row_ptr, full_col_idx, part_row_ptr, part_col_idx, part_bitmap and, when
 * set, tile_lists all point to host memory; head_tiles and head_valid are
 * ignored). Returns
 * STA_OK when the mask is one that sta_encode_mask could have produced, else
 * STA_ERR_INVALID_ARG with *failed_check (may be NULL) set to the first failed
 * check:
 *    1 shape fields < 1     2 ot_rows / ot_cols not ceil(L/64)
 *    3 negative counts or too many tiles    4 a needed array is NULL
 *    5 a row_ptr does not start at 0        6 a row_ptr decreases
 *    7 a row_ptr does not end at n_full / n_part
 *    8 a column outside [0, ot_cols)        9 columns of a row not ascending
 *   10 a tile listed as both full and part 11 a full tile reaching past Lq or Lk
 *   12 a part bitmap bit outside the mask  13 a part tile with no bit set
 *   14 a part tile inside the mask with every bit set (a full tile)
 *   15 n_valid (when >= 0) differs from the count of valid elements
 *   16 tile_lists with ot_cols > 1024      17 a tile-list slot that is not the
 *      union of its two outer-tile rows (columns ascending, kinds -1 / -2 / index)
 * Host only (no CUDA call); cost linear in the mask's tiles and bitmap words.
 * The kernels do not run these checks; given a mask that fails them they stay
 * inside their buffers (CSR ranges clamped to n_full / n_part, columns and keys
 * clamped into the mask, part indices checked against n_part) but compute wrong
 * values, and the block-wise kernel, when it merges a damaged CSR itself, sets
 * 0x213 in the device error word (sta_device_error). Likewise the decode kernels
 * keep every request's token range inside the host copy's kv_indptr[n_req] and
 * set 0x111 when the device copy disagrees. */
sta_status sta_validate_mask(const sta_bsr_mask* mask, int* failed_check);

/* sta_mla_decode -- decode against a shared latent KV cache: multi-head latent
 * attention in the weight-absorbed form (Cleave, 評価結果: MLA among the LLM
 * subgraphs; the token reduction split into chunks and merged by log-sum-exp,
 * Split演算子によるSplit-Kの対応):
 *   O[r, h] = sum_t softmax_t(scale * q[r, h] . kv[t]) * kv[t, 0:512]
 * over the tokens t of request r; LSE the natural-log normaliser.
 *
 *   q              [n_req, Hq, 576] bf16 (device): per query head a 512-entry
 *                  latent part (the query taken into the latent space) then a
 *                  64-entry rotary part
 *   kv             [T, 576] bf16 (device): per cached token its 512-entry latent
 *                  then its 64-entry rotary key, shared by every query head;
 *                  request r owns rows kv_indptr[r] .. kv_indptr[r+1]-1
 *   kv_indptr_dev  int32 [n_req+1] (device); kv_indptr_host: the same values
 *                  (host), non-decreasing from 0 (else STA_ERR_INVALID_ARG); the
 *                  kernels keep each device range inside kv_indptr_host[n_req]
 *                  (0x111 in the device error word when the copies disagree)
 *   Hq             a multiple of 16, at most 1024; scale > 0
 *   chunk_tokens   0: the library picks; else tokens per chunk (rounded up to a
 *                  multiple of 32): a request longer than a chunk is cut into
 *                  chunks attended by their own CTAs, then merged by LSE
 *   o              [n_req, Hq, 512] bf16 (device, written); lse [n_req, Hq] f32
 *                  (device, written; may be NULL). An empty request gives O = 0,
 *                  LSE = -inf.
 *   workspace      device scratch (256-byte aligned) for the chunks' fp32
 *                  partials, or NULL: *workspace_bytes is then set to the size
 *                  needed and nothing is launched
 * q, kv and o 16-byte aligned (else STA_ERR_UNSUPPORTED). One launch, plus a
 * merge launch when some request is cut; asynchronous on `stream`. */
sta_status sta_mla_decode(const void* q, const void* kv, const int32_t* kv_indptr_dev, const int32_t* kv_indptr_host,
                          int n_req, int Hq, float scale, int chunk_tokens, void* o, float* lse, void* workspace,
                          size_t* workspace_bytes, sta_stream stream);

/* Size in bytes of the tile_lists buffer for a mask of Hm heads over Lq x Lk
 * (see sta_bsr_mask), or 0 when Hm, Lq or Lk is < 1 or ceil(Lk/64) > 1024.
 * Host only. */
size_t sta_tile_lists_bytes(int Hm, int Lq, int Lk);

/* sta_encode_mask -- build the two-level mask from Hm sources
 * (STOF, 2 段階ストレージ形式).
 *
 *   srcs            host array [Hm] of mask heads (their data pointers are device)
 *   Hm, Lq, Lk      mask heads and mask shape, all >= 1, Lq, Lk < 2^30
 *   out             host struct; see the three modes below
 *   workspace       device scratch, 256-byte aligned, or NULL
 *   workspace_bytes host in/out
 *
 * Modes:
 *  1. workspace == NULL: *workspace_bytes is set to the scratch size needed;
 *     nothing else happens (no CUDA call).
 *  2. Size query: out->full_row_ptr and out->part_row_ptr set (device,
 *     [Hm*ot_rows+1] each), out->full_col_idx == out->part_col_idx ==
 *     out->part_bitmap == NULL. Classifies every outer tile, writes the two
 *     row_ptr arrays, then SYNCHRONISES the stream and fills out->n_full,
 *     n_part, n_valid and the shape fields. This is the library's only
 *     synchronising call.
 *  3. Fill: all five device arrays set, out->n_full / n_part holding the
 *     capacities from a size query of the same mask. Writes everything,
 *     asynchronously. Entries beyond a capacity are never written.
 *     With out->tile_lists set (ot_cols <= 1024), the per-query-tile column
 *     lists are written as well.
 * Returns STA_ERR_INVALID_ARG for bad sizes, null pointers or kinds (also for
 * tile_lists with ot_cols > 1024 or not 16-byte aligned), and
 * STA_ERR_WORKSPACE if *workspace_bytes is below the requirement. */
sta_status sta_encode_mask(const sta_mask_src* srcs, int Hm, int Lq, int Lk, sta_bsr_mask* out, void* workspace,
                           size_t* workspace_bytes, sta_stream stream);

/* ------------------------------------------------------------------------ */
/* Masked multi-head attention forward                                       */
/* ------------------------------------------------------------------------ */

#define STA_KERNEL_AUTO 0  /* analytic selector (STOF カーネル選択)           */
#define STA_KERNEL_BLOCK 1 /* block-wise: TMA + tcgen05/TMEM, bf16 only        */
#define STA_KERNEL_ROW 2   /* row-wise: one warp per query row, bf16 or f32   */
#define STA_KERNEL_MIXED 3 /* returned by sta_mha_select_kernel only: the     *
                            * per-head choice runs both kernels, each on its  *
                            * own heads, concurrently                         */

/* sta_mha_fwd -- O = softmax(Q K^T * scale + mask) V and its LSE, over the
 * valid elements of an encoded mask (STOF 問題定義, 統合 MHA モジュール).
 * Empty outer tiles are skipped, full ones run unmasked, part ones are masked
 * by their bitmaps.
 *
 *   q        [B, H, Lq, d]  dtype        (device)
 *   k, v     [B, H, Lk, d]  dtype        (device)
 *   o        [B, H, Lq, d]  dtype        (device, written)
 *   lse      [B, H, Lq]     float32      (device, written; may be NULL)
 *   mask     encoded mask with mask->Lq == Lq, mask->Lk == Lk (host struct)
 *   head_map host [H]: attention head h uses mask head head_map[h]; NULL means
 *            mask head 0 for every head if Hm == 1, else head h (then Hm must
 *            equal H)
 *   d        64 or 128; H <= 1024; B*H <= 65535
 *   dtype    STA_BF16 (both kernels) or STA_F32 (row-wise kernel only)
 *   scale    softmax scale, > 0 (e.g. 1/sqrt(d))
 *   kernel   STA_KERNEL_AUTO / BLOCK / ROW; BLOCK needs bf16 and Lk <= 65536
 *            (else STA_ERR_UNSUPPORTED). AUTO applies the analytic selector:
 *            per mask head when mask->head_tiles and mask->head_valid are both
 *            set, else once for the whole mask. When the per-head choice picks
 *            both kernels, the row-wise kernel runs on its heads on a stream of
 *            the library's own (one per host thread and device, created on the
 *            first such call, forked from and joined back into `stream` with
 *            events, so the call stays asynchronous and can be captured in a
 *            CUDA graph) while the block-wise kernel runs on the others on
 *            `stream`.
 * Pointers must be 16-byte aligned. Asynchronous on `stream`. */
sta_status sta_mha_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const sta_bsr_mask* mask,
                       const int32_t* head_map, int B, int H, int Lq, int Lk, int d, sta_dtype dtype, float scale,
                       int kernel, sta_stream stream);

/* sta_mha_fwd_splitkv -- sta_mha_fwd with the key-tile loop of the block-wise
 * kernel split (Cleave, Split演算子によるSplit-Kの対応, applied to masked
 * prefill): the list of non-empty key tiles of each (128-row query tile, b, h)
 * is cut into s chunks, each attended by its own CTA into a normalised fp32
 * partial and its LSE, and the chunks are merged by log-sum-exp as in
 * sta_merge_lse. Long rows (a dense or random head among banded ones, small
 * B*H) then spread over many CTAs instead of one.
 *
 *   q .. kernel  as for sta_mha_fwd; the split applies to the block-wise
 *                kernel only (a row-wise choice runs unsplit)
 *   num_splits   0: the library picks s per head from mask->head_tiles (no
 *                split when it is NULL): heads whose key tiles per query tile
 *                exceed twice the average load of a resident CTA slot (two
 *                per SM; each item counted with a prologue of about 4 tiles)
 *                are cut
 *                into chunks of about that load (at least 16 tiles, at most
 *                32 chunks); other heads run whole;
 *                1..1024: every head is cut into that many chunks (chunks past
 *                a row's tile count are empty and contribute nothing)
 *   workspace    device scratch for the partials, 256-byte aligned;
 *                workspace == NULL sets *workspace_bytes (never 0) and
 *                returns without touching the data pointers
 * Results equal sta_mha_fwd's up to rounding (the merge re-normalises fp32
 * partials). Returns STA_ERR_UNSUPPORTED when B * (sum of the heads' s)
 * exceeds 65535, STA_ERR_WORKSPACE when *workspace_bytes is too small, and
 * otherwise the errors of sta_mha_fwd. Asynchronous on `stream`. */
sta_status sta_mha_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               const sta_bsr_mask* mask, const int32_t* head_map, int B, int H, int Lq, int Lk, int d,
                               sta_dtype dtype, float scale, int kernel, int num_splits, void* workspace,
                               size_t* workspace_bytes, sta_stream stream);

/* Layouts of O for sta_mha_fwd_layout. */
#define STA_O_BHLD 0 /* [B, H, Lq, d]: one block of rows per head (as sta_mha_fwd)      */
#define STA_O_BLHD 1 /* [B, Lq, H, d]: the heads of each query token side by side, i.e. */
                     /* the [B*Lq, H*d] row-major input of the output projection         */

/* sta_mha_fwd_layout -- sta_mha_fwd_splitkv whose epilogue writes O in the
 * layout o_layout. STA_O_BLHD merges the heads per token in the same store that
 * writes O (no separate transpose before the projection GEMM that follows the
 * attention), the fixed-rule form of fusing MHA with its downstream operators
 * (STOF, 演算子融合モジュール). Every other argument, the workspace protocol
 * and the results (element for element, only their places in o differ) are
 * those of sta_mha_fwd_splitkv; lse stays [B, H, Lq]. o_layout outside the two
 * values: STA_ERR_INVALID_ARG. */
sta_status sta_mha_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse,
                              const sta_bsr_mask* mask, const int32_t* head_map, int B, int H, int Lq, int Lk, int d,
                              sta_dtype dtype, float scale, int kernel, int num_splits, int o_layout, void* workspace,
                              size_t* workspace_bytes, sta_stream stream);

/* sta_bias_residual_layernorm -- the elementwise operators that follow the
 * attention output projection, fused into one pass over each row (STOF,
 * 演算子融合モジュール, with a fixed fusion rule in place of its search):
 *   h = (x + bias) + residual
 *   y = (h - mean(h)) / sqrt(var(h) + eps) * gamma + beta
 * mean and var over the n elements of the row, var the population variance
 * (divided by n). Arithmetic in fp32 on the bf16 inputs; y and h_out rounded
 * to bf16 (round to nearest even).
 *
 *   x            [rows, n] bf16 (device), e.g. the projection GEMM's output
 *   bias         [n] bf16 (device) or NULL (0)
 *   residual     [rows, n] bf16 (device) or NULL (0)
 *   gamma, beta  [n] f32 (device) or NULL (1 and 0)
 *   y            [rows, n] bf16 (device, written; may alias neither input)
 *   h_out        [rows, n] bf16 (device, written) or NULL: the pre-norm sum h,
 *                the residual stream of the next sub-layer
 *   rows >= 0 (0: nothing is launched); n % 8 == 0, 8 <= n <= 16384;
 *   eps > 0 and finite; dtype STA_BF16 (else STA_ERR_UNSUPPORTED)
 * Pointers must be 16-byte aligned (else STA_ERR_UNSUPPORTED). One launch,
 * asynchronous on `stream`. */
sta_status sta_bias_residual_layernorm(const void* x, const void* bias, const void* residual, const float* gamma,
                                       const float* beta, void* y, void* h_out, int64_t rows, int n, float eps,
                                       sta_dtype dtype, sta_stream stream);

/* Which kernel sta_mha_fwd would run for these arguments under
 * STA_KERNEL_AUTO: STA_KERNEL_BLOCK or STA_KERNEL_ROW, or STA_KERNEL_MIXED
 * when the per-head choice (mask->head_tiles and mask->head_valid set) picks
 * both kernels among the mask heads; a negative sta_status on invalid
 * arguments. Host only. */
int sta_mha_select_kernel(const sta_bsr_mask* mask, int B, int H, int Lq, int Lk, int d, sta_dtype dtype);

/* ------------------------------------------------------------------------ */
/* Split-KV decode and log-sum-exp merge                                     */
/* ------------------------------------------------------------------------ */

/* sta_decode_splitkv -- one query token per request against its packed KV
 * prefix (every key of the request is valid), with the KV reduction split
 * into chunks that are attended independently and merged by log-sum-exp
 * (Cleave Split operator; FlashDecoding). GQA: query head h reads kv head
 * h / (Hq / Hkv).
 *
 *   q              [n_req, Hq, d] bf16  (device)
 *   k, v           [T, Hkv, d]    bf16  (device), request r owns rows
 *                  kv_indptr[r] .. kv_indptr[r+1]-1; may be NULL when T == 0
 *                  (every request then gets O = 0, LSE = -inf)
 *   kv_indptr_dev  int32 [n_req+1] (device), kv_indptr_host: same values (host)
 *   Hq % Hkv == 0, Hq / Hkv in {1, 2, 4, 8, 16}, d in {64, 128}
 *   num_splits     0: the library picks the split (the whole token stream is
 *                  cut into equal ranges, one per resident CTA); s > 0: every
 *                  request is cut into s chunks of ceil(len/s) keys
 *   o              [n_req, Hq, d] bf16 (device, written); lse [n_req, Hq] f32
 *                  (device, written; may be NULL)
 *   workspace      device scratch for the partial results, 256-byte aligned;
 *                  workspace == NULL sets *workspace_bytes and returns
 * kv_indptr_host must be non-decreasing, start at 0, and match the device copy.
 * Asynchronous on `stream`. */
sta_status sta_decode_splitkv(const void* q, const void* k, const void* v, const int32_t* kv_indptr_dev,
                              const int32_t* kv_indptr_host, int n_req, int Hq, int Hkv, int d, sta_dtype dtype,
                              float scale, int num_splits, void* o, float* lse, void* workspace,
                              size_t* workspace_bytes, sta_stream stream);

/* sta_decode_splitkv_paged -- sta_decode_splitkv over a paged KV cache: the
 * keys and values of all requests live in fixed-size pages, and each request
 * lists its pages in order (the page-table layout of serving systems; a
 * deployment variant of the decode, not a step the pages describe).
 *
 *   k_pages, v_pages  [n_pages, page_size, Hkv, d] bf16 (device); token i of
 *                     request r (0-based within the request) is slot
 *                     i % page_size of page page_indices[page_indptr[r] + i / page_size]
 *   page_size         tokens per page, >= 1
 *   n_pages           pages in k_pages / v_pages (page indices are checked against
 *                     it in the kernel: an index outside [0, n_pages) reads page 0 and
 *                     sets the device error word to 0x110)
 *   page_indptr_dev   int32 [n_req+1] (device): request r owns entries
 *                     page_indptr[r] .. page_indptr[r+1]-1 of page_indices, at least
 *                     ceil(len_r / page_size) of them
 *   page_indices_dev  int32 (device) page numbers
 *   kv_indptr_dev/host token prefix sums [n_req+1] as for sta_decode_splitkv (they give
 *                     each request's length and the token stream the split divides)
 * Everything else -- arguments, split plans, workspace, results, errors -- is that
 * of sta_decode_splitkv; results are identical to it on the same K/V values.
 * Asynchronous on `stream`. */
sta_status sta_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages, int page_size,
                                    int n_pages, const int32_t* page_indptr_dev, const int32_t* page_indices_dev,
                                    const int32_t* kv_indptr_dev, const int32_t* kv_indptr_host, int n_req, int Hq,
                                    int Hkv, int d, sta_dtype dtype, float scale, int num_splits, void* o, float* lse,
                                    void* workspace, size_t* workspace_bytes, sta_stream stream);

/* sta_decode_splitkv_noalloc -- sta_decode_splitkv for callers that cannot
 * allocate device memory: for example code running inside a host framework
 * that owns every device allocation and hands out no allocator, or a serving
 * loop that must not call cudaMalloc (which can synchronise the device) on its
 * hot path. (The pages have no counterpart: this is a deployment variant of the
 * split-KV decode, not part of the method.)
 *
 * Arguments, results and errors are those of sta_decode_splitkv without the
 * workspace: the caller still passes q, k, v, kv_indptr, o and lse. The partial
 * results go to one fixed 16 MiB array in the library's own device memory, which
 * every GPU that loads the library holds until the process exits. The plan must
 * fit it: slots * Hq * (d + 1) * 4 bytes (each part rounded up to 256) <= 16 MiB.
 * With num_splits > 0, slots = n_req * num_splits. With num_splits == 0, slots =
 * ranges + n_req, where ranges (the token ranges the plan cuts the KV stream
 * into, each at least 16 tokens) is at most ceil(T / 16) and at most the
 * resident decode CTAs divided by the KV-head groups a CTA serves; the sum
 * resident CTAs + n_req is therefore an upper bound, not the exact size. Query the exact size with sta_decode_splitkv
 * (workspace == NULL). A larger plan returns STA_ERR_WORKSPACE and launches
 * nothing.
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture. All calls
 * share the array and it keeps the last call's contents (nothing in it needs
 * clearing: every partial that is read is written earlier in the same call), so
 * calls that overlap on the GPU -- on different streams, or on one device from
 * several host threads without ordering -- race and must not be issued. Calls no
 * cudaMalloc, cudaFree or other allocating routine. */
sta_status sta_decode_splitkv_noalloc(const void* q, const void* k, const void* v, const int32_t* kv_indptr_dev,
                                      const int32_t* kv_indptr_host, int n_req, int Hq, int Hkv, int d,
                                      sta_dtype dtype, float scale, int num_splits, void* o, float* lse,
                                      sta_stream stream);

/* sta_merge_lse -- merge s partial attention results per row:
 *   M = max_i lse_i; if M = -inf then O = 0, LSE = -inf; otherwise
 *   w_i = exp(lse_i - M), O = sum_i w_i O_i / sum_i w_i, LSE = M + log sum_i w_i.
 *   part_o   [n_rows, s, d] float32 normalised partial outputs (device, 16-byte
 *            aligned, else STA_ERR_UNSUPPORTED)
 *   part_lse [n_rows, s]    float32 natural-log partial denominators (device)
 *   o        [n_rows, d]    o_dtype (device, written); lse [n_rows] f32 or NULL
 *   1 <= s <= 4096; d in {32, 64, 128, 256}; n_rows == 0 is a no-op.
 *   Asynchronous on `stream`. */
sta_status sta_merge_lse(const float* part_o, const float* part_lse, int n_rows, int s, int d, void* o,
                         sta_dtype o_dtype, float* lse, sta_stream stream);

/* Static string describing a status code. */
const char* sta_status_string(sta_status status);

/* The cudaError_t behind the most recent STA_ERR_CUDA returned by any call of
 * this library (process-wide; 0 if none), and its description. */
int sta_last_cuda_error(void);
const char* sta_last_cuda_error_string(void);

/* Device error word of the current device: kernels whose internal waits
 * (mbarrier phases, bounded to about 2 s) give up record a nonzero code here
 * instead of hanging; 0 means no such event. Copies the word to *code
 * (synchronous) and clears it when reset != 0. */
sta_status sta_device_error(int* code, int reset);

/* sta_check_bounded_wait -- exercises the failure-detection path on the GPU
 * without a fault: one kernel waits, through the bounded mbarrier wait every
 * kernel of this library uses, on a barrier phase that nothing completes. After
 * limit_ns nanoseconds (1e3 <= limit_ns <= 2e9) the wait gives up, records code
 * 0x7f1 in the device error word (read it with sta_device_error) unless an
 * earlier code is there, writes 0 to *outcome_dev (int, device, 4-byte aligned;
 * 1 would mean the wait completed) and the kernel returns: the context stays
 * usable. (The pages have no counterpart: this checks the library's own
 * hang-avoidance, not the method.) Asynchronous on `stream`. */
sta_status sta_check_bounded_wait(int64_t limit_ns, int* outcome_dev, sta_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* STA_H_ */
