/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY. A plain, slow, fp64 CPU restatement of
 * what the masked-attention and split-KV decode path computes. Only the tests,
 * the smoke check and the bench's CPU-baseline / reference legs may load it;
 * the library's own code never does.
 *
 * Sources (the pages this follows):
 *  - "Accelerating Sparse Transformer Inference on GPU" (STOF), sections
 *    "問題定義" (masked MHA; causal, sliding-window and random masks) and
 *    "手法: 統合 MHA モジュール / 2 段階ストレージ形式" (outer tiles that are
 *    empty, full or part; one uint64 bitmap per 8x8 inner tile of a part tile;
 *    the format is an exact encoding of the mask).
 *  - "Cleave: Scaling Tensor Program Optimization via Decoupled Algebraic
 *    Search and Operator Scheduling", section "Split演算子によるSplit-Kの対応"
 *    and the abstract (a Split operator with a symbolic count s partitions a
 *    reduction dimension; FlashDecoding).
 *
 * Everything here is the plain definition, evaluated directly:
 *   O_i = sum_j softmax_j(scale * q_i . k_j + mask_ij) v_j, LSE_i = log sum_j exp(...)
 * with the mask materialised element by element from its description (never
 * from the encoded tiles), a two-pass softmax over the valid keys only (exp of
 * -inf is exactly 0, so skipping masked keys changes nothing), natural-log LSE,
 * and O = 0, LSE = -inf for a row with no valid key.
 *
 * Readings where the pages are silent (bit order inside the uint64, the order of
 * inner tiles, edge tiles, the merge formula) are stated at each function.
 * Compile with -ffp-contract=off so results do not depend on FMA contraction.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* One [Lq, Lk] mask head.
 * kind 0 (pattern): valid(i,j) = (!causal || j <= i) &&
 *                                ((win_lo <= j-i && j-i <= win_hi) || j < n_global_cols)
 * kind 1 (dense u8): u8[i*Lk + j] != 0
 * kind 2 (dense bits): bit (j & 63) of bits[i*W + (j >> 6)], W = ceil(Lk/64) */
typedef struct {
  int32_t kind;
  int32_t causal;
  int64_t win_lo, win_hi;
  int64_t n_global_cols;
  const uint8_t* u8;
  const uint64_t* bits;
} om_mask_head;

static int om_valid(const om_mask_head* m, int64_t Lk, int64_t i, int64_t j) {
  if (m->kind == 0) {
    if (m->causal && j > i) return 0;
    int64_t dd = j - i;
    if (dd >= m->win_lo && dd <= m->win_hi) return 1;
    return j < m->n_global_cols;
  }
  if (m->kind == 1) return m->u8[i * Lk + j] != 0;
  {
    int64_t W = (Lk + 63) / 64;
    return (int)((m->bits[i * W + (j >> 6)] >> (j & 63)) & 1u);
  }
}

/* Materialise mask heads to dense uint8 [Hm, Lq, Lk]. */
void oracle_mask_dense(const om_mask_head* heads, int32_t Hm, int64_t Lq, int64_t Lk, uint8_t* out) {
  for (int32_t h = 0; h < Hm; ++h)
    for (int64_t i = 0; i < Lq; ++i)
      for (int64_t j = 0; j < Lk; ++j) out[(h * Lq + i) * Lk + j] = (uint8_t)om_valid(&heads[h], Lk, i, j);
}

/* Number of valid (i, j) in one mask head. */
int64_t oracle_mask_count(const om_mask_head* m, int64_t Lq, int64_t Lk) {
  int64_t n = 0;
  for (int64_t i = 0; i < Lq; ++i)
    for (int64_t j = 0; j < Lk; ++j) n += om_valid(m, Lk, i, j);
  return n;
}

/* ------------------------------------------------------------------------- */
/* Attention of one query row against a set of keys, two-pass softmax, fp64. */
/* keys: valid key indices, n of them; kv rows are at k + key*kstride.       */
static void om_attend_row(const float* q, const float* k, const float* v, int64_t kstride, int32_t d,
                          const int64_t* keys, int64_t n, double scale, double* s /* scratch [n] */,
                          double* o /* [d] */, double* lse) {
  for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    const float* kr = k + keys[t] * kstride;
    double acc = 0.0;
    for (int32_t c = 0; c < d; ++c) acc += (double)q[c] * (double)kr[c];
    s[t] = scale * acc;
    if (s[t] > m) m = s[t];
  }
  double l = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    double e = exp(s[t] - m);
    l += e;
    const float* vr = v + keys[t] * kstride;
    for (int32_t c = 0; c < d; ++c) o[c] += e * (double)vr[c];
  }
  for (int32_t c = 0; c < d; ++c) o[c] /= l;
  *lse = m + log(l);
}

/* ------------------------------------------------------------------------- */
/* Masked MHA forward, selected rows.                                        */
/* q: [B, H, Lq, d], k/v: [B, H, Lk, d] float32 (exact widenings of the      */
/* inputs). Row r of `rows` is the flat index (b*H + h)*Lq + i; rows == NULL */
/* means every row in order. Outputs o [n_rows, d], lse [n_rows] in fp64.    */
typedef struct {
  const float *q, *k, *v;
  int32_t B, H, d;
  int64_t Lq, Lk;
  double scale;
  const om_mask_head* heads;
  const int32_t* head_map;
  const int64_t* rows;
  int64_t n_rows;
  double *o, *lse;
  int64_t r0, r1;
} om_mha_job;

static void* om_mha_worker(void* arg) {
  om_mha_job* J = (om_mha_job*)arg;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(J->Lk > 0 ? J->Lk : 1));
  double* s = (double*)malloc(sizeof(double) * (size_t)(J->Lk > 0 ? J->Lk : 1));
  for (int64_t r = J->r0; r < J->r1; ++r) {
    int64_t flat = J->rows ? J->rows[r] : r;
    int64_t i = flat % J->Lq;
    int64_t bh = flat / J->Lq;
    int32_t h = (int32_t)(bh % J->H);
    const om_mask_head* m = &J->heads[J->head_map[h]];
    int64_t n = 0;
    for (int64_t j = 0; j < J->Lk; ++j)
      if (om_valid(m, J->Lk, i, j)) keys[n++] = j;
    const float* qr = J->q + flat * J->d;
    const float* kb = J->k + bh * J->Lk * J->d;
    const float* vb = J->v + bh * J->Lk * J->d;
    om_attend_row(qr, kb, vb, J->d, J->d, keys, n, J->scale, s, J->o + r * J->d, J->lse + r);
  }
  free(keys);
  free(s);
  return NULL;
}

static int om_threads(int n_threads) {
  if (n_threads > 0) return n_threads;
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

void oracle_mha_rows(const float* q, const float* k, const float* v, int32_t B, int32_t H, int64_t Lq,
                     int64_t Lk, int32_t d, double scale, const om_mask_head* heads, const int32_t* head_map,
                     const int64_t* rows, int64_t n_rows, double* o, double* lse, int32_t n_threads) {
  int nt = om_threads(n_threads);
  if (nt > n_rows) nt = (int)(n_rows > 0 ? n_rows : 1);
  om_mha_job* jobs = (om_mha_job*)calloc((size_t)nt, sizeof(om_mha_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  for (int t = 0; t < nt; ++t) {
    om_mha_job* J = &jobs[t];
    J->q = q; J->k = k; J->v = v; J->B = B; J->H = H; J->d = d; J->Lq = Lq; J->Lk = Lk;
    J->scale = scale; J->heads = heads; J->head_map = head_map; J->rows = rows; J->n_rows = n_rows;
    J->o = o; J->lse = lse;
    J->r0 = n_rows * t / nt;
    J->r1 = n_rows * (t + 1) / nt;
    if (nt > 1) pthread_create(&th[t], NULL, om_mha_worker, J);
  }
  if (nt == 1) om_mha_worker(&jobs[0]);
  else
    for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
}

/* ------------------------------------------------------------------------- */
/* LSE merge of split partials (Cleave's Split over the softmax reduction).  */
/* The pages do not print the merge; this is the plain identity for          */
/* partials given as (normalised O_i, lse_i = log of partial denominator):   */
/*   M = max_i lse_i; if M = -inf: O = 0, LSE = -inf; else                   */
/*   w_i = exp(lse_i - M), LSE = M + log sum w_i, O = sum w_i O_i / sum w_i.  */
/* part_o [n_rows, s, d], part_lse [n_rows, s] -> o [n_rows, d], lse.        */
void oracle_merge_lse(const double* part_o, const double* part_lse, int64_t n_rows, int32_t s, int32_t d,
                      double* o, double* lse) {
  for (int64_t r = 0; r < n_rows; ++r) {
    const double* pl = part_lse + r * s;
    double M = -INFINITY;
    for (int32_t i = 0; i < s; ++i)
      if (pl[i] > M) M = pl[i];
    double* orow = o + r * d;
    for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int32_t i = 0; i < s; ++i) {
      double w = exp(pl[i] - M);
      wsum += w;
      const double* po = part_o + (r * s + i) * d;
      for (int32_t c = 0; c < d; ++c) orow[c] += w * po[c];
    }
    for (int32_t c = 0; c < d; ++c) orow[c] /= wsum;
    lse[r] = M + log(wsum);
  }
}

/* ------------------------------------------------------------------------- */
/* GQA decode: one query token per request, every key in [0, len_r) valid.   */
/* q [n_req, Hq, d], k/v [T, Hkv, d] packed by kv_indptr; query head h reads */
/* kv head h / (Hq/Hkv). chunk == 0: one pass over all keys (s = 1).         */
/* chunk > 0: keys split into consecutive chunks of `chunk` keys, each chunk */
/* attended on its own (normalised O_c, lse_c), then merged by               */
/* oracle_merge_lse -- the Split form, which must equal s = 1.               */
typedef struct {
  const float *q, *k, *v;
  const int32_t* indptr;
  int32_t n_req, Hq, Hkv, d;
  double scale;
  int64_t chunk;
  double *o, *lse;
  int64_t r0, r1; /* range over n_req*Hq rows */
} om_dec_job;

static void* om_dec_worker(void* arg) {
  om_dec_job* J = (om_dec_job*)arg;
  int32_t group = J->Hq / J->Hkv;
  int64_t maxlen = 0;
  for (int32_t r = 0; r < J->n_req; ++r) {
    int64_t len = J->indptr[r + 1] - J->indptr[r];
    if (len > maxlen) maxlen = len;
  }
  int64_t cap = maxlen > 0 ? maxlen : 1;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
  double* s = (double*)malloc(sizeof(double) * (size_t)cap);
  int64_t max_s = J->chunk > 0 ? (cap + J->chunk - 1) / J->chunk : 1;
  double* po = (double*)malloc(sizeof(double) * (size_t)(max_s * J->d));
  double* pl = (double*)malloc(sizeof(double) * (size_t)max_s);
  for (int64_t row = J->r0; row < J->r1; ++row) {
    int32_t r = (int32_t)(row / J->Hq), h = (int32_t)(row % J->Hq), g = h / group;
    int64_t beg = J->indptr[r], len = J->indptr[r + 1] - beg;
    const float* qr = J->q + row * J->d;
    const float* kb = J->k + (beg * J->Hkv + g) * J->d;
    const float* vb = J->v + (beg * J->Hkv + g) * J->d;
    int64_t kstride = (int64_t)J->Hkv * J->d;
    if (J->chunk <= 0) {
      for (int64_t t = 0; t < len; ++t) keys[t] = t;
      om_attend_row(qr, kb, vb, kstride, J->d, keys, len, J->scale, s, J->o + row * J->d, J->lse + row);
    } else {
      int64_t ns = len > 0 ? (len + J->chunk - 1) / J->chunk : 1;
      for (int64_t c = 0; c < ns; ++c) {
        int64_t a = c * J->chunk, b = a + J->chunk < len ? a + J->chunk : len;
        for (int64_t t = a; t < b; ++t) keys[t - a] = t;
        om_attend_row(qr, kb, vb, kstride, J->d, keys, b - a, J->scale, s, po + c * J->d, pl + c);
      }
      oracle_merge_lse(po, pl, 1, (int32_t)ns, J->d, J->o + row * J->d, J->lse + row);
    }
  }
  free(keys);
  free(s);
  free(po);
  free(pl);
  return NULL;
}

void oracle_decode(const float* q, const float* k, const float* v, const int32_t* kv_indptr, int32_t n_req,
                   int32_t Hq, int32_t Hkv, int32_t d, double scale, int64_t chunk, double* o, double* lse,
                   int32_t n_threads) {
  int64_t n_rows = (int64_t)n_req * Hq;
  int nt = om_threads(n_threads);
  if (nt > n_rows) nt = (int)(n_rows > 0 ? n_rows : 1);
  om_dec_job* jobs = (om_dec_job*)calloc((size_t)nt, sizeof(om_dec_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  for (int t = 0; t < nt; ++t) {
    om_dec_job* J = &jobs[t];
    J->q = q; J->k = k; J->v = v; J->indptr = kv_indptr; J->n_req = n_req; J->Hq = Hq; J->Hkv = Hkv;
    J->d = d; J->scale = scale; J->chunk = chunk; J->o = o; J->lse = lse;
    J->r0 = n_rows * t / nt;
    J->r1 = n_rows * (t + 1) / nt;
    if (nt > 1) pthread_create(&th[t], NULL, om_dec_worker, J);
  }
  if (nt == 1) om_dec_worker(&jobs[0]);
  else
    for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
}

/* ------------------------------------------------------------------------- */
/* Two-level mask encoding (STOF, 2 段階ストレージ形式).                       */
/* Outer tiles (OT) are 64x64, R = ceil(Lq/64) rows by C = ceil(Lk/64) cols.  */
/* An OT is FULL when all 64x64 elements lie inside [0,Lq)x[0,Lk) and are    */
/* valid, EMPTY when no in-range element is valid, and PART otherwise.       */
/* Full and part OTs are listed in two CSR structures (row_ptr over          */
/* (mask head, OT row), ascending col_idx); empty OTs appear in neither.     */
/* A part OT stores 64 uint64 words, one per 8x8 inner tile (IT), ITs in     */
/* row-major order (word 8p + q covers OT rows 8p..8p+7, cols 8q..8q+7);     */
/* inside a word, bit 8r + c is element (row 8p + r, col 8q + c), so byte r  */
/* holds IT row r. Out-of-range elements are 0.                              */
/* Classes: 0 empty, 1 full, 2 part.                                         */
void oracle_encode_classify(const om_mask_head* heads, int32_t Hm, int64_t Lq, int64_t Lk, uint8_t* cls,
                            int64_t* n_full, int64_t* n_part, int64_t* n_valid) {
  int64_t R = (Lq + 63) / 64, C = (Lk + 63) / 64;
  int64_t nf = 0, np = 0, nv = 0;
  for (int32_t h = 0; h < Hm; ++h)
    for (int64_t a = 0; a < R; ++a)
      for (int64_t c = 0; c < C; ++c) {
        int64_t cnt = 0, inrange = 0;
        for (int64_t r = 0; r < 64; ++r)
          for (int64_t cc = 0; cc < 64; ++cc) {
            int64_t i = a * 64 + r, j = c * 64 + cc;
            if (i >= Lq || j >= Lk) continue;
            ++inrange;
            cnt += om_valid(&heads[h], Lk, i, j);
          }
        uint8_t k = 0;
        if (cnt == 0) k = 0;
        else if (cnt == 4096 && inrange == 4096) k = 1;
        else k = 2;
        cls[(h * R + a) * C + c] = k;
        nf += (k == 1);
        np += (k == 2);
        nv += cnt;
      }
  *n_full = nf;
  *n_part = np;
  *n_valid = nv;
}

void oracle_encode_fill(const om_mask_head* heads, int32_t Hm, int64_t Lq, int64_t Lk, const uint8_t* cls,
                        int32_t* full_row_ptr, int32_t* full_col_idx, int32_t* part_row_ptr,
                        int32_t* part_col_idx, uint64_t* part_bitmap) {
  int64_t R = (Lq + 63) / 64, C = (Lk + 63) / 64;
  int64_t nf = 0, np = 0;
  full_row_ptr[0] = 0;
  part_row_ptr[0] = 0;
  for (int32_t h = 0; h < Hm; ++h)
    for (int64_t a = 0; a < R; ++a) {
      for (int64_t c = 0; c < C; ++c) {
        uint8_t k = cls[(h * R + a) * C + c];
        if (k == 1) full_col_idx[nf++] = (int32_t)c;
        if (k == 2) {
          uint64_t* words = part_bitmap + np * 64;
          for (int p = 0; p < 8; ++p)
            for (int qq = 0; qq < 8; ++qq) {
              uint64_t w = 0;
              for (int r = 0; r < 8; ++r)
                for (int cc = 0; cc < 8; ++cc) {
                  int64_t i = a * 64 + p * 8 + r, j = c * 64 + qq * 8 + cc;
                  if (i < Lq && j < Lk && om_valid(&heads[h], Lk, i, j)) w |= (uint64_t)1 << (8 * r + cc);
                }
              words[8 * p + qq] = w;
            }
          part_col_idx[np++] = (int32_t)c;
        }
      }
      full_row_ptr[h * R + a + 1] = (int32_t)nf;
      part_row_ptr[h * R + a + 1] = (int32_t)np;
    }
}

/* Inverse of the encoding: BSR + bitmaps -> dense uint8 [Hm, Lq, Lk]. */
void oracle_decode_mask(int32_t Hm, int64_t Lq, int64_t Lk, const int32_t* full_row_ptr,
                        const int32_t* full_col_idx, const int32_t* part_row_ptr, const int32_t* part_col_idx,
                        const uint64_t* part_bitmap, uint8_t* dense) {
  int64_t R = (Lq + 63) / 64;
  memset(dense, 0, (size_t)(Hm * Lq * Lk));
  for (int32_t h = 0; h < Hm; ++h)
    for (int64_t a = 0; a < R; ++a) {
      for (int32_t t = full_row_ptr[h * R + a]; t < full_row_ptr[h * R + a + 1]; ++t) {
        int64_t c = full_col_idx[t];
        for (int64_t r = 0; r < 64; ++r)
          for (int64_t cc = 0; cc < 64; ++cc) {
            int64_t i = a * 64 + r, j = c * 64 + cc;
            if (i < Lq && j < Lk) dense[(h * Lq + i) * Lk + j] = 1;
          }
      }
      for (int32_t t = part_row_ptr[h * R + a]; t < part_row_ptr[h * R + a + 1]; ++t) {
        int64_t c = part_col_idx[t];
        const uint64_t* words = part_bitmap + (int64_t)t * 64;
        for (int p = 0; p < 8; ++p)
          for (int qq = 0; qq < 8; ++qq)
            for (int r = 0; r < 8; ++r)
              for (int cc = 0; cc < 8; ++cc) {
                int64_t i = a * 64 + p * 8 + r, j = c * 64 + qq * 8 + cc;
                if (i < Lq && j < Lk && ((words[8 * p + qq] >> (8 * r + cc)) & 1u))
                  dense[(h * Lq + i) * Lk + j] = 1;
              }
      }
    }
}
