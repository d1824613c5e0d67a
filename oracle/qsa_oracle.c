/*
 * qsa_oracle.c -- plain, slow CPU oracle for the QSA indexer and its top-k.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *  [QSA]  "SGLang Day-0 support for Qwen3.8-Flash-Next: QSA sparse attention,
 *         IndexShare MTP and HyperConnection kernel optimisations"
 *         (theainews.cc), section "Qwen sparse attention (QSA): coarse
 *         retrieval, fine attention" -- the compressed key, the score
 *         equation, the 512-block budget and the 0-3 pending tokens, the
 *         paged full_slot/4 compressed cache.
 *  [TOPK] SGLang GLM-5.2 blog (aihot.virxact.com), section "Kernel
 *         Optimization / TopK-V2", Figures 2-4 -- exact top-k (k <= 2048)
 *         over FP32 score rows, fused with the page-table transform into
 *         physical KV slots.
 *  [SMLA] "vllm-sparse-mla-blackwell" (shadowgraph.io), section "Design notes
 *         worth knowing" -- the consumer masks on index >= 0, so -1 is the
 *         empty-entry sentinel.
 *  [QSA] also: the compressed keys only index; softmax and value
 *         aggregation read the original K/V at the selected positions.
 *  [QSA] also, section "IndexShare MTP: reusing the QSA selection across
 *         draft steps" -- the selection of the draft-extend row is kept for
 *         the whole MTP iteration and read together with the positions
 *         drafted since; the draft steps run no indexer.
 *
 * Every floating-point step that the pages leave open is done in FP64 and
 * rounded once at the end, except the block mean, which [QSA] fixes as FP32.
 * Readings of points the pages leave open (all listed in the design notes):
 *  - "normalise" is the L2 norm; a zero mean vector stays zero;
 *  - the block's first-token MRoPE position reduces, for text positions, to
 *    plain RoPE with base `rope_base` over all 128 dims, rotate-half pairing
 *    (i, i+64), angle p * base^(-2i/128);
 *  - the query is already position-encoded and is used as given;
 *  - 1/sqrt(128) multiplies the head sum;
 *  - a query row sees L tokens, complete blocks b < floor(L/4) and
 *    L mod 4 pending tokens;
 *  - ties go to the lower index, -0 equals +0, NaN ranks below -inf;
 *  - selected indices are returned ascending, -1 only as tail padding.
 *
 * Parity pins live in tests/ (hand-worked example, closed forms, brute
 * force, invariants).  Functions here are kept obviously correct, not fast.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QSA_D 128      /* index head dim ([QSA]: 128-dim heads)           */
#define QSA_H 4        /* index query heads ([QSA]: 4 query heads)         */
#define QSA_C 4        /* compression ratio c4 ([QSA]: 4 raw keys / block) */

/* ---------- BF16 helpers (bit patterns in uint16_t) ---------------------- */

double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest BF16 value, ties to even, in one step (no
 * intermediate FP32 rounding).  BF16 has 8 significant bits and FP32's
 * exponent range; values below the smallest normal use the fixed subnormal
 * quantum 2^-133.  Inputs here are finite and far from overflow. */
uint16_t oracle_bf16_round(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
  int e;
  frexp(x, &e);                 /* |x| = m * 2^e, m in [0.5, 1) */
  int qexp = e - 8;             /* quantum of an 8-significant-bit value */
  if (qexp < -133) qexp = -133;
  double q = ldexp(1.0, qexp);
  double r = nearbyint(x / q) * q;   /* default rounding mode: to nearest even */
  float f = (float)r;                /* exact: r is a BF16 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

void oracle_bf16_round_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}

/* ---------- paging ([QSA] paged cache; [TOPK] page-table transform) ------ */

/* Physical KV slot of logical token position `pos` of a request whose page
 * table row is `pt_row`: page pt_row[pos / P], offset pos mod P. */
int64_t oracle_slot_of(const int32_t* pt_row, int64_t pos, int64_t page_size) {
  return (int64_t)pt_row[pos / page_size] * page_size + pos % page_size;
}

/* Row of the compressed-key pool that holds block b: [QSA] addresses the
 * compressed cache page-aligned as full_slot/4, where full_slot is the
 * physical slot of the block's first token 4b. */
int64_t oracle_pool_row(const int32_t* pt_row, int64_t b, int64_t page_size) {
  return oracle_slot_of(pt_row, QSA_C * b, page_size) / QSA_C;
}

/* ---------- step 1: compressed index key ([QSA]) ------------------------- */

/* One block: raw[4][128] BF16 keys -> out[128] BF16.
 *   m   = FP32 mean of the four raw keys, summed in index order;
 *   u   = m / ||m||_2  (FP64);
 *   k   = RoPE at position first_pos, rotate-half pairs (i, i+64),
 *         angle first_pos * rope_base^(-2i/128)  (FP64);
 *   out = BF16(k), round to nearest even. */
void oracle_compress_block(const uint16_t* raw, int64_t first_pos, double rope_base,
                           uint16_t* out) {
  float m[QSA_D];
  for (int d = 0; d < QSA_D; ++d) {
    float s = (float)oracle_bf16_to_double(raw[0 * QSA_D + d]);
    s = s + (float)oracle_bf16_to_double(raw[1 * QSA_D + d]);
    s = s + (float)oracle_bf16_to_double(raw[2 * QSA_D + d]);
    s = s + (float)oracle_bf16_to_double(raw[3 * QSA_D + d]);
    m[d] = s * 0.25f;
  }
  double norm2 = 0.0;
  for (int d = 0; d < QSA_D; ++d) norm2 += (double)m[d] * (double)m[d];
  double norm = sqrt(norm2);
  double u[QSA_D];
  for (int d = 0; d < QSA_D; ++d) u[d] = norm > 0.0 ? (double)m[d] / norm : 0.0;

  const int half = QSA_D / 2;
  double k[QSA_D];
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(rope_base, -2.0 * (double)i / (double)QSA_D);
    double theta = (double)first_pos * inv_freq;
    double c = cos(theta), s = sin(theta);
    k[i] = u[i] * c - u[i + half] * s;
    k[i + half] = u[i + half] * c + u[i] * s;
  }
  for (int d = 0; d < QSA_D; ++d) out[d] = oracle_bf16_round(k[d]);
}

/* All blocks: block i belongs to request block_req[i] and is that request's
 * block block_id[i] (first token 4*block_id[i]).  With a page table the key
 * goes to pool row full_slot/4; without one (page_table == NULL) to row i. */
void oracle_compress(const uint16_t* raw, int64_t n_blocks, const int32_t* block_req,
                     const int32_t* block_id, const int32_t* page_table, int64_t ld_pt,
                     int64_t page_size, double rope_base, uint16_t* pool) {
  for (int64_t i = 0; i < n_blocks; ++i) {
    int64_t b = block_id[i];
    int64_t row = i;
    if (page_table) row = oracle_pool_row(page_table + (int64_t)block_req[i] * ld_pt, b, page_size);
    oracle_compress_block(raw + i * QSA_C * QSA_D, QSA_C * b, rope_base, pool + row * QSA_D);
  }
}

/* ---------- key path of a decode step ([QSA]: the raw index keys of the
 * incomplete block wait in a 4-slot ring per request; a completed block is
 * compressed into the pool at full_slot/4) ------------------------------- */

/* Request r appends the raw keys new_keys[req_tok_start[r] + i] at positions
 * req_first_pos[r] + i, i < req_tok_start[r+1] - req_tok_start[r].  Every
 * block b completed by these tokens (4b+3 among the positions) is compressed
 * from its 4 raw keys -- those of this call where present, the ring's
 * (ring[r][q mod 4], written by earlier calls) for the earlier positions --
 * into pool row slot(4b)/4.  Then ring[r][p mod 4] takes the key of every
 * appended position p, in order (later positions overwrite earlier ones).
 * ring is [n_req][4][128] u16, updated in place. */
void oracle_append_keys(const uint16_t* new_keys, const int32_t* req_tok_start,
                        const int32_t* req_first_pos, int64_t n_req, uint16_t* ring,
                        const int32_t* page_table, int64_t ld_pt, int64_t page_size,
                        double rope_base, uint16_t* pool) {
  uint16_t blk[QSA_C * QSA_D];
  for (int64_t r = 0; r < n_req; ++r) {
    int64_t n = req_tok_start[r + 1] - req_tok_start[r];
    int64_t p0 = req_first_pos[r];
    const uint16_t* keys = new_keys + (int64_t)req_tok_start[r] * QSA_D;
    uint16_t* rr = ring + r * QSA_C * QSA_D;
    for (int64_t i = 0; i < n; ++i) {
      int64_t p = p0 + i;
      if (p % QSA_C != QSA_C - 1) continue;
      int64_t b = p / QSA_C;
      for (int c = 0; c < QSA_C; ++c) {
        int64_t q = QSA_C * b + c;
        const uint16_t* src = q >= p0 ? keys + (q - p0) * QSA_D : rr + c * QSA_D;
        memcpy(blk + c * QSA_D, src, QSA_D * sizeof(uint16_t));
      }
      int64_t row = oracle_pool_row(page_table + r * ld_pt, b, page_size);
      oracle_compress_block(blk, QSA_C * b, rope_base, pool + row * QSA_D);
    }
    for (int64_t i = 0; i < n; ++i)
      memcpy(rr + ((p0 + i) % QSA_C) * QSA_D, keys + i * QSA_D, QSA_D * sizeof(uint16_t));
  }
}

/* ---------- step 2: block scores ([QSA] score equation) ------------------ */

/* s = (1/sqrt(128)) * sum_{h<4} ReLU(<q_h, kbar>), in FP64, rounded once to
 * FP32.  q is [4][128] BF16, key is [128] BF16. */
float oracle_score_one(const uint16_t* q, const uint16_t* key) {
  double acc = 0.0;
  for (int h = 0; h < QSA_H; ++h) {
    double dot = 0.0;
    for (int d = 0; d < QSA_D; ++d)
      dot += oracle_bf16_to_double(q[h * QSA_D + d]) * oracle_bf16_to_double(key[d]);
    acc += dot > 0.0 ? dot : 0.0;
  }
  return (float)(acc / sqrt((double)QSA_D));
}

/* Rows are grouped by request: rows req_row_start[r] .. req_row_start[r+1]-1
 * belong to request r.  Row t sees row_len[t] tokens and so scores blocks
 * b < row_len[t]/4, reading block b from pool row full_slot/4.  Writes
 * scores[t][b] for those b only. */
void oracle_index_scores(const uint16_t* q, const uint16_t* pool, int64_t n_req,
                         const int32_t* req_row_start, const int32_t* row_len,
                         const int32_t* page_table, int64_t ld_pt, int64_t page_size,
                         float* scores, int64_t ld_scores) {
  for (int64_t r = 0; r < n_req; ++r) {
    const int32_t* pt_row = page_table + r * ld_pt;
    for (int64_t t = req_row_start[r]; t < req_row_start[r + 1]; ++t) {
      int64_t nb = row_len[t] / QSA_C;
      /* independent blocks: the timing build (-fopenmp) splits them over the
       * host cores; the plain build ignores the pragma */
#pragma omp parallel for schedule(static)
      for (int64_t b = 0; b < nb; ++b) {
        const uint16_t* key = pool + oracle_pool_row(pt_row, b, page_size) * QSA_D;
        scores[t * ld_scores + b] = oracle_score_one(q + t * QSA_H * QSA_D, key);
      }
    }
  }
}

/* ---------- step 3: exact top-k ([TOPK]; ties to the lower index) -------- */

/* Total order used for selection: larger score first; NaN below every
 * number; -0 == +0 (IEEE compare); equal scores by ascending index. */
static int ranks_before(float a, int64_t ia, float b, int64_t ib) {
  int na = isnan(a), nb = isnan(b);
  if (na || nb) {
    if (na && nb) return ia < ib;
    return nb;  /* the non-NaN one ranks first */
  }
  if (a > b) return 1;
  if (a < b) return 0;
  return ia < ib;
}

typedef struct { float s; int64_t i; } scored_t;

static int cmp_rank(const void* pa, const void* pb) {
  const scored_t* a = (const scored_t*)pa;
  const scored_t* b = (const scored_t*)pb;
  if (a->i == b->i) return 0;
  return ranks_before(a->s, a->i, b->s, b->i) ? -1 : 1;
}

static int cmp_index(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* One row: the k best of s[0..n) under the order above, returned as
 * ascending indices; entries past min(k, n) are -1.  Returns min(k, n). */
int64_t oracle_topk_row(const float* s, int64_t n, int64_t k, int32_t* out_idx) {
  scored_t* tmp = (scored_t*)malloc(sizeof(scored_t) * (size_t)(n > 0 ? n : 1));
  for (int64_t i = 0; i < n; ++i) { tmp[i].s = s[i]; tmp[i].i = i; }
  qsort(tmp, (size_t)n, sizeof(scored_t), cmp_rank);
  int64_t m = n < k ? n : k;
  for (int64_t j = 0; j < m; ++j) out_idx[j] = (int32_t)tmp[j].i;
  qsort(out_idx, (size_t)m, sizeof(int32_t), cmp_index);
  for (int64_t j = m; j < k; ++j) out_idx[j] = -1;
  free(tmp);
  return m;
}

/* Many rows.  Row t has n_valid[t] candidates (all ld if n_valid == NULL).
 * With a page table, out_slots[t][j] is the physical slot of index
 * out_idx[t][j] in page-table row row_req[t] (row t if row_req == NULL);
 * -1 stays -1. */
void oracle_topk(const float* scores, int64_t ld, const int32_t* n_valid, int64_t n_rows,
                 int64_t k, const int32_t* page_table, int64_t ld_pt, const int32_t* row_req,
                 int64_t page_size, int32_t* out_idx, int32_t* out_slots) {
  for (int64_t t = 0; t < n_rows; ++t) {
    int64_t n = n_valid ? n_valid[t] : ld;
    oracle_topk_row(scores + t * ld, n, k, out_idx + t * k);
    if (out_slots && page_table) {
      const int32_t* pt_row = page_table + (row_req ? row_req[t] : t) * ld_pt;
      for (int64_t j = 0; j < k; ++j) {
        int32_t i = out_idx[t * k + j];
        out_slots[t * k + j] = i < 0 ? -1 : (int32_t)oracle_slot_of(pt_row, i, page_size);
      }
    }
  }
}

/* ---------- steps 4-5: expansion + slot translation ([QSA], [TOPK]) ------ */

/* One row.  sel[0..k_blk) are selected block ids (ascending, -1 tail).  Each
 * block b expands to token positions 4b..4b+3; then the L mod 4 pending
 * tokens of the incomplete block, positions 4*floor(L/4) .. L-1, follow.
 * The row has 4*k_blk + 3 entries; unused ones are -1.  Slots are the
 * page-table images of the positions; -1 stays -1. */
void oracle_expand_row(const int32_t* sel, int64_t k_blk, int64_t L, const int32_t* pt_row,
                       int64_t page_size, int32_t* out_pos, int32_t* out_slots) {
  int64_t width = QSA_C * k_blk + (QSA_C - 1);
  int64_t w = 0;
  for (int64_t j = 0; j < k_blk; ++j) {
    if (sel[j] < 0) continue;
    for (int c = 0; c < QSA_C; ++c) out_pos[w++] = QSA_C * sel[j] + c;
  }
  for (int64_t p = (L / QSA_C) * QSA_C; p < L; ++p) out_pos[w++] = (int32_t)p;
  for (; w < width; ++w) out_pos[w] = -1;
  for (int64_t j = 0; j < width; ++j)
    out_slots[j] = out_pos[j] < 0 ? -1 : (int32_t)oracle_slot_of(pt_row, out_pos[j], page_size);
}

void oracle_expand(const int32_t* sel, int64_t k_blk, int64_t n_req, const int32_t* req_row_start,
                   const int32_t* row_len, const int32_t* page_table, int64_t ld_pt,
                   int64_t page_size, int32_t* out_pos, int32_t* out_slots) {
  int64_t width = QSA_C * k_blk + (QSA_C - 1);
  for (int64_t r = 0; r < n_req; ++r)
    for (int64_t t = req_row_start[r]; t < req_row_start[r + 1]; ++t)
      oracle_expand_row(sel + t * k_blk, k_blk, row_len[t], page_table + r * ld_pt, page_size,
                        out_pos + t * width, out_slots + t * width);
}

/* ---------- IndexShare reuse ([QSA], section "IndexShare MTP: reusing the
 * QSA selection across draft steps") ------------------------------------- */

/* The selection kept at a request's draft-extend row (the last row the target
 * accepted; it saw cap_len tokens and kept the blocks cap_sel[0..k_blk))
 * serves every later draft row of that request, which runs no scorer and no
 * top-k of its own.  A row that sees L tokens reads, in ascending order:
 *   - the positions 4b..4b+3 of each captured block b, those below L;
 *   - every position from 4*floor(cap_len/4) up to L-1: the capture's own
 *     pending tokens, then every token drafted since;
 * then -1 up to the width 4*k_blk + 3 + n_extra (n_extra: the drafted
 * positions the caller leaves room for).  A captured block that was not
 * complete at the capture (b >= floor(cap_len/4)) is skipped: its positions
 * belong to the second part.  Slots are the page-table images of the
 * positions.  Returns a bit set: 1 = the list did not fit and was cut at the
 * width, 2 = a captured block was skipped. */
int oracle_indexshare_row(const int32_t* cap_sel, int64_t k_blk, int64_t cap_len,
                          int64_t n_extra, int64_t L, const int32_t* pt_row, int64_t page_size,
                          int32_t* out_pos, int32_t* out_slots) {
  int64_t width = QSA_C * k_blk + (QSA_C - 1) + n_extra;
  int64_t nb0 = cap_len / QSA_C;
  int64_t w = 0;
  int flags = 0;
  for (int64_t j = 0; j < k_blk; ++j) {
    int64_t b = cap_sel[j];
    if (b < 0) continue;
    if (b >= nb0) {
      flags |= 2;
      continue;
    }
    for (int c = 0; c < QSA_C; ++c) {
      int64_t p = QSA_C * b + c;
      if (p >= L) continue;
      if (w < width) out_pos[w++] = (int32_t)p;
      else flags |= 1;
    }
  }
  for (int64_t p = QSA_C * nb0; p < L; ++p) {
    if (w < width) out_pos[w++] = (int32_t)p;
    else flags |= 1;
  }
  for (; w < width; ++w) out_pos[w] = -1;
  for (int64_t j = 0; j < width; ++j)
    out_slots[j] = out_pos[j] < 0 ? -1 : (int32_t)oracle_slot_of(pt_row, out_pos[j], page_size);
  return flags;
}

/* Every row t of request r reads the captured row cap_row[r] of cap_sel
 * ([n_cap][k_blk], row lengths cap_len[n_cap]).  A request whose cap_row is
 * outside [0, n_cap) gets a row of -1 and flag 4.  Returns the OR of the
 * rows' flags. */
int oracle_indexshare(const int32_t* cap_sel, const int32_t* cap_len, int64_t n_cap,
                      const int32_t* cap_row, int64_t k_blk, int64_t n_extra, int64_t n_req,
                      const int32_t* req_row_start, const int32_t* row_len,
                      const int32_t* page_table, int64_t ld_pt, int64_t page_size,
                      int32_t* out_pos, int32_t* out_slots) {
  int64_t width = QSA_C * k_blk + (QSA_C - 1) + n_extra;
  int flags = 0;
  for (int64_t r = 0; r < n_req; ++r)
    for (int64_t t = req_row_start[r]; t < req_row_start[r + 1]; ++t) {
      int64_t c = cap_row[r];
      if (c < 0 || c >= n_cap) {
        for (int64_t j = 0; j < width; ++j) out_pos[t * width + j] = out_slots[t * width + j] = -1;
        flags |= 4;
        continue;
      }
      flags |= oracle_indexshare_row(cap_sel + c * k_blk, k_blk, cap_len[c], n_extra, row_len[t],
                                     page_table + r * ld_pt, page_size, out_pos + t * width,
                                     out_slots + t * width);
    }
  return flags;
}

/* ---------- sparse attention over the selected slots ([QSA]; [SMLA]) ----- */

/* [QSA], section "Qwen sparse attention (QSA)": the compressed keys only
 * index; the final softmax and value aggregation read the original,
 * uncompressed K/V at the selected positions (sparse GQA).  [SMLA], "Design
 * notes worth knowing": the only mask is index >= 0, and a token whose whole
 * selection is masked must not come out as NaN.
 * One row: query q [H_q][d], query head h reads KV head h / (H_q / H_kv);
 * slots[0..n_idx) index the caches k, v [n_slots][H_kv][d]; entries < 0 are
 * skipped.  out[h] = sum_j softmax_j(scale <q_h, k_j>) v_j in FP64, rounded
 * to FP32 once; lse[h] = log sum_j exp(scale <q_h, k_j>).  With no valid
 * entry: out = 0, lse = -inf.  Returns 1 if an entry >= n_slots was skipped. */
int oracle_sparse_attn_row(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t n_slots,
                           int64_t h_q, int64_t h_kv, int64_t d, const int32_t* slots,
                           int64_t n_idx, double scale, float* out, float* lse) {
  int64_t group = h_q / h_kv;
  int bad = 0;
  double* logit = (double*)malloc((size_t)(n_idx > 0 ? n_idx : 1) * sizeof(double));
  double* acc = (double*)malloc((size_t)d * sizeof(double));
  for (int64_t h = 0; h < h_q; ++h) {
    int64_t g = h / group;
    double mx = -INFINITY;
    for (int64_t j = 0; j < n_idx; ++j) {
      logit[j] = -INFINITY;
      int64_t s = slots[j];
      if (s < 0) continue;
      if (s >= n_slots) {
        bad = 1;
        continue;
      }
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e)
        dot += oracle_bf16_to_double(q[h * d + e]) * oracle_bf16_to_double(k[(s * h_kv + g) * d + e]);
      logit[j] = scale * dot;
      if (logit[j] > mx) mx = logit[j];
    }
    for (int64_t e = 0; e < d; ++e) acc[e] = 0.0;
    double sum = 0.0;
    if (mx > -INFINITY) {
      for (int64_t j = 0; j < n_idx; ++j) {
        if (logit[j] == -INFINITY) continue;
        double w = exp(logit[j] - mx);
        sum += w;
        int64_t s = slots[j];
        for (int64_t e = 0; e < d; ++e) acc[e] += w * oracle_bf16_to_double(v[(s * h_kv + g) * d + e]);
      }
    }
    for (int64_t e = 0; e < d; ++e) out[h * d + e] = sum > 0.0 ? (float)(acc[e] / sum) : 0.0f;
    if (lse) lse[h] = sum > 0.0 ? (float)(mx + log(sum)) : -INFINITY;
  }
  free(logit);
  free(acc);
  return bad;
}

/* Every row t: q[t], slots[t][0..n_idx) (leading dimension ld_slots),
 * out[t] [H_q][d], lse[t] [H_q] (lse may be NULL).  Returns the OR of the
 * rows' flags. */
int oracle_sparse_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t n_slots,
                       int64_t n_rows, int64_t h_q, int64_t h_kv, int64_t d, const int32_t* slots,
                       int64_t ld_slots, int64_t n_idx, double scale, float* out, float* lse) {
  int bad = 0;
  for (int64_t t = 0; t < n_rows; ++t)
    bad |= oracle_sparse_attn_row(q + t * h_q * d, k, v, n_slots, h_q, h_kv, d, slots + t * ld_slots,
                                  n_idx, scale, out + t * h_q * d, lse ? lse + t * h_q : NULL);
  return bad;
}

/* ---------- the whole decode path: score -> top-k blocks -> slots ------- */

/* Host threads of the timing build (built with -fopenmp); the plain build
 * runs single-threaded and returns 1. */
#ifdef _OPENMP
#include <omp.h>
int oracle_set_threads(int n) {
  omp_set_num_threads(n);
  return n;
}
#else
int oracle_set_threads(int n) {
  (void)n;
  return 1;
}
#endif

/* scores must hold n_rows * ld_scores floats (ld_scores >= max nb).  The
 * selection runs on these FP32 scores, blocks b < row_len/4 only. */
void oracle_indexer_select(const uint16_t* q, const uint16_t* pool, int64_t n_req,
                           const int32_t* req_row_start, const int32_t* row_len,
                           const int32_t* page_table, int64_t ld_pt, int64_t page_size,
                           int64_t k_blk, float* scores, int64_t ld_scores, int32_t* out_blocks,
                           int32_t* out_pos, int32_t* out_slots) {
  oracle_index_scores(q, pool, n_req, req_row_start, row_len, page_table, ld_pt, page_size,
                      scores, ld_scores);
  const int64_t n_rows = req_row_start[n_req];
  /* independent rows (the timing build runs them on the host cores) */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < n_rows; ++t)
    oracle_topk_row(scores + t * ld_scores, row_len[t] / QSA_C, k_blk, out_blocks + t * k_blk);
  oracle_expand(out_blocks, k_blk, n_req, req_row_start, row_len, page_table, ld_pt, page_size,
                out_pos, out_slots);
}

/* ---------- prologue tails: query RoPE and FP8 index keys ----------------
 * SGLang GLM-5.2 blog, section "Indexer Prologue Fusion": the query path is
 * RoPE + FP8 quantisation (+ head gates, which QSA's score does not have),
 * the key path LayerNorm + RoPE + FP8 quantisation + the paged index-cache
 * store.  For QSA's compressed keys the pages give no FP8 layout; the
 * reading taken: e4m3 codes with one FP32 scale per compressed key. */

/* Query RoPE: the 4 heads of row t rotated at the row's own position
 * pos[t] (the newest token it sees), rotate-half pairs (i, i+64), angle
 * pos * rope_base^(-2i/128), in FP64, one round to BF16. */
void oracle_rope_queries(const uint16_t* q, const int32_t* pos, int64_t n_rows, double rope_base,
                         uint16_t* out) {
  const int half = QSA_D / 2;
  for (int64_t t = 0; t < n_rows; ++t)
    for (int h = 0; h < QSA_H; ++h) {
      const uint16_t* x = q + (t * QSA_H + h) * QSA_D;
      uint16_t* y = out + (t * QSA_H + h) * QSA_D;
      for (int i = 0; i < half; ++i) {
        double inv_freq = pow(rope_base, -(2.0 * (double)i) / (double)QSA_D);
        double theta = (double)pos[t] * inv_freq;
        double c = cos(theta), s = sin(theta);
        double u = oracle_bf16_to_double(x[i]), v = oracle_bf16_to_double(x[i + half]);
        y[i] = oracle_bf16_round(u * c - v * s);
        y[i + half] = oracle_bf16_round(v * c + u * s);
      }
    }
}

/* FP8 e4m3 (the "fn" variant): 1 sign bit, 4 exponent bits biased by 7,
 * 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; the
 * largest finite value is 448 (0x7E); 0x7F and 0xFF are NaN; there is no
 * infinity. */
double oracle_e4m3_to_double(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return s ? -v : v;
}

/* Nearest e4m3 value of a float, ties to even, saturating at +-448 (finite
 * results only); NaN gives 0x7F. */
uint8_t oracle_e4m3_round(float xf) {
  double x = (double)xf;
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  int e;
  frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) */
  int qexp = e - 4;                /* quantum of a 4-significant-bit value */
  if (qexp < -9) qexp = -9;        /* subnormal quantum */
  double r = a == 0.0 ? 0.0 : nearbyint(a / ldexp(1.0, qexp)) * ldexp(1.0, qexp);
  if (r > 448.0) r = 448.0;        /* saturate */
  if (r == 0.0) return sign;
  int re;
  frexp(r, &re);                   /* r = g * 2^re, g in [0.5, 1) */
  int ue = re - 1;                 /* r in [2^ue, 2^(ue+1)) */
  uint8_t code;
  if (ue < -6) {                   /* subnormal: r = m * 2^-9 */
    code = (uint8_t)(r / ldexp(1.0, -9));
  } else {
    int m = (int)(r / ldexp(1.0, ue - 3)) - 8;   /* r = (8 + m) * 2^(ue-3) */
    code = (uint8_t)(((ue + 7) << 3) | m);
  }
  return (uint8_t)(sign | code);
}

/* FP8 compressed keys: per key, scale = fp32(max_d |k_d|) / 448 (FP32
 * division) and code_d = e4m3(k_d / scale) (FP32 division, then the nearest
 * e4m3 value, ties to even, saturating); a zero key gets scale 0 and zero
 * codes.  Every step that decides a code is FP32, so both sides of a parity
 * check take the same decisions. */
void oracle_quantize_keys_fp8(const uint16_t* keys, int64_t n, uint8_t* codes, float* scales) {
  for (int64_t r = 0; r < n; ++r) {
    float mx = 0.0f;
    for (int d = 0; d < QSA_D; ++d) {
      float v = fabsf((float)oracle_bf16_to_double(keys[r * QSA_D + d]));
      if (v > mx) mx = v;
    }
    const float scale = mx / 448.0f;
    scales[r] = scale;
    for (int d = 0; d < QSA_D; ++d) {
      float v = (float)oracle_bf16_to_double(keys[r * QSA_D + d]);
      codes[r * QSA_D + d] = scale > 0.0f ? oracle_e4m3_round(v / scale) : 0;
    }
  }
}

/* Nearest IEEE binary16 value (1 sign, 5 exponent bits biased by 15, 10
 * mantissa bits; subnormal quantum 2^-24; largest finite 65504), ties to
 * even, as a double.  Beyond 65520 the nearest value is infinity. */
double oracle_f16_round(double x) {
  if (x == 0.0 || isnan(x)) return x;
  double a = fabs(x);
  int e;
  frexp(a, &e);
  int qexp = e - 11;               /* quantum of an 11-significant-bit value */
  if (qexp < -24) qexp = -24;
  double r = nearbyint(a / ldexp(1.0, qexp)) * ldexp(1.0, qexp);
  if (r > 65504.0) r = INFINITY;
  return signbit(x) ? -r : r;
}

/* Score of one query row against one FP8 key: the FP8 scorer holds the query
 * in FP16 (each BF16 element rounded to the nearest binary16 value), the key
 * is code * scale:
 *   s = (1/sqrt(128)) * sum_h ReLU( sum_d f16(q_hd) * e4m3(c_d) * scale ),
 * in FP64, rounded once to FP32. */
float oracle_score_one_fp8(const uint16_t* q, const uint8_t* codes, float scale) {
  double total = 0.0;
  for (int h = 0; h < QSA_H; ++h) {
    const uint16_t* qh = q + h * QSA_D;   /* head h */
    double hdot = 0.0;
    for (int d = 0; d < QSA_D; ++d)
      hdot += oracle_f16_round(oracle_bf16_to_double(qh[d])) * oracle_e4m3_to_double(codes[d]) * (double)scale;
    total += hdot > 0.0 ? hdot : 0.0;
  }
  return (float)(total / sqrt((double)QSA_D));
}

/* oracle_index_scores with FP8 keys: codes [pool_rows][128], scales
 * [pool_rows], the same pool-row addressing (full_slot/4). */
void oracle_index_scores_fp8(const uint16_t* q, const uint8_t* codes, const float* scales, int64_t n_req,
                             const int32_t* req_row_start, const int32_t* row_len, const int32_t* page_table,
                             int64_t ld_pt, int64_t page_size, float* scores, int64_t ld_scores) {
  for (int64_t r = 0; r < n_req; ++r) {
    const int32_t* pt_row = page_table + r * ld_pt;
    for (int64_t t = req_row_start[r]; t < req_row_start[r + 1]; ++t) {
      const int64_t n_blocks = row_len[t] / QSA_C;   /* complete blocks only */
      for (int64_t b = 0; b < n_blocks; ++b) {
        const int64_t row = oracle_pool_row(pt_row, b, page_size);
        scores[t * ld_scores + b] = oracle_score_one_fp8(q + t * QSA_H * QSA_D, codes + row * QSA_D, scales[row]);
      }
    }
  }
}

/* ---------- head-gated score ([TOPK], "Indexer Prologue Fusion": the query
 * path scales each index head by a gate) ----------------------------------
 * s = (1/sqrt(128)) sum_h g[h] * ReLU(<q_h, kbar>): the gate multiplies the
 * head's rectified dot product; g = 1 for every head is the plain score.
 * FP64, one rounding to FP32. */
float oracle_score_one_gated(const uint16_t* q, const float* g, const uint16_t* key) {
  double sum_w = 0.0;
  for (int hg = 0; hg < QSA_H; ++hg) {
    double hd = 0.0;
    for (int d = 0; d < QSA_D; ++d)
      hd += oracle_bf16_to_double(q[hg * QSA_D + d]) * oracle_bf16_to_double(key[d]);
    const double rect = hd > 0.0 ? hd : 0.0;
    sum_w += (double)g[hg] * rect;
  }
  return (float)(sum_w / sqrt((double)QSA_D));
}

/* Gated block scores: gates [n_rows][4] FP32, one per row and head. */
void oracle_index_scores_gated(const uint16_t* q, const float* gates, const uint16_t* pool, int64_t n_req,
                               const int32_t* req_row_start, const int32_t* row_len, const int32_t* page_table,
                               int64_t ld_pt, int64_t page_size, float* scores, int64_t ld_scores) {
  for (int64_t r = 0; r < n_req; ++r) {
    const int32_t* ptr_r = page_table + r * ld_pt;
    for (int64_t t = req_row_start[r]; t < req_row_start[r + 1]; ++t) {
      const int64_t n_blk = row_len[t] / QSA_C;
      for (int64_t b = 0; b < n_blk; ++b)
        scores[t * ld_scores + b] = oracle_score_one_gated(q + t * QSA_H * QSA_D, gates + t * QSA_H,
                                                           pool + oracle_pool_row(ptr_r, b, page_size) * QSA_D);
    }
  }
}
