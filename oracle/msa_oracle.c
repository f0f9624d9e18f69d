/*
 * msa_oracle.c - TEST INFRASTRUCTURE ONLY.  A plain, slow, fp64 CPU statement
 * of block-sparse, causal, document-local grouped-query attention (MiniMax
 * Sparse Attention, "MSA") and of the k2q plan derived from its selection.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library; the product path never does.  It shares no code with
 * the CUDA path.
 *
 * Sources (web pages on the method):
 *   [PR]  NeMo-Automodel PR "feat(minimax-m3): add SM100 MSA sparse attention
 *         with custom backward" - sections "Changelog" (compact document-local
 *         q2k indices), "Design" (the flat-attention interface
 *         Q[T,64,128], K/V[T,4,128], int32 q2k[4,T,16], -1 for unused slots,
 *         layout = document offsets) and "Supported scope" (64 query / 4 KV /
 *         4 index heads, head dim 128, block 128, top-k 16, causal prefill).
 *   [BWD] API page "msa_backward_sm100" - module description (tiles of 8
 *         queries times the 16 query heads of an index head, grouped by index
 *         head and key block; the delta preprocess), run_backward parameter list (LSE is FP32 [T,64]).
 *
 * Readings taken where the pages are silent:
 *   - query head h uses KV head and index head h/16;
 *   - key block v of a document covers document positions 128v..128v+127 (the
 *     last block may be partial);
 *   - the slots of q2k[g,t,:] form a SET (duplicates count once);
 *   - a selected block after the query's own block contributes no keys;
 *   - a value < -1 or >= the document's block count is an error;
 *   - LSE is the natural-log log-sum-exp of the scaled scores;
 *   - a row with no visible key has O = 0, LSE = -inf and zero gradients;
 *   - delta = rowsum(dO * O) is taken from the oracle's own exact O.
 *
 * Inputs: fp64 arrays.  The Python wrapper widens the bf16 tensors of a
 * problem exactly (bf16 -> fp32 -> fp64), so the oracle sees the same values
 * the GPU path reads; finite-difference tests pass unrounded fp64 values.
 * Built with -DORACLE_BF16_INPUT the same source takes Q, K, V, dO as the
 * bf16 bit patterns themselves and widens each element exactly where it is
 * read, so large problems need no fp64 copy; every arithmetic step is the
 * same, so both builds return bit-identical results on bf16 values.
 * All arithmetic is fp64.  Parallelism is OpenMP over independent
 * rows / buckets only; there is no blocking or fusion beyond the definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NQH 64   /* query heads */
#define NKV 4    /* KV heads = index heads */
#define HPG 16   /* query heads per index head */
#define HD 128   /* head dim */
#define BLK 128  /* key block size */
#define TOPK 16  /* q2k slots */

enum { OR_OK = 0, OR_BAD_ARGS = 1, OR_BAD_Q2K = 2, OR_CAPACITY = 3 };

/* Element type of Q, K, V, dO and its exact widening to fp64. */
#ifdef ORACLE_BF16_INPUT
typedef uint16_t elem_t;
static inline double ld(const elem_t* p, int64_t i) {
  uint32_t u = (uint32_t)p[i] << 16; /* bf16 is the top half of an fp32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}
#else
typedef double elem_t;
static inline double ld(const elem_t* p, int64_t i) { return p[i]; }
#endif

/* Document offsets: offs[0] = 0, strictly increasing, offs[D] = T. */
static int check_offsets(const int32_t* offs, int32_t D, int64_t T) {
  if (D <= 0 || offs[0] != 0 || offs[D] != T) return OR_BAD_ARGS;
  for (int32_t d = 0; d < D; ++d)
    if (offs[d + 1] <= offs[d]) return OR_BAD_ARGS;
  return OR_OK;
}

static int32_t doc_of(const int32_t* offs, int32_t D, int64_t t) {
  int32_t lo = 0, hi = D - 1; /* largest d with offs[d] <= t */
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) / 2;
    if (offs[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static int32_t nblocks(int32_t len) { return (len + BLK - 1) / BLK; }

/* Sel(t,g) as a membership array over the document's blocks; returns
 * OR_BAD_Q2K if a slot holds a value outside [-1, nblk). */
static int selection(const int32_t* q2k, int64_t T, int g, int64_t t, int32_t nblk,
                     unsigned char* sel) {
  memset(sel, 0, (size_t)nblk);
  for (int i = 0; i < TOPK; ++i) {
    int32_t v = q2k[((int64_t)g * T + t) * TOPK + i];
    if (v == -1) continue;
    if (v < -1 || v >= nblk) return OR_BAD_Q2K;
    sel[v] = 1;
  }
  return OR_OK;
}

/* Keys(t,g) = { s_d + j : 0 <= j <= p, floor(j/128) in Sel(t,g) }, ascending. */
static int keys_of(const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D, int g,
                   int64_t t, int64_t* keys, int64_t* nkeys, unsigned char* sel) {
  int32_t d = doc_of(offs, D, t);
  int64_t s = offs[d];
  int32_t len = offs[d + 1] - offs[d];
  int64_t p = t - s;
  int rc = selection(q2k, T, g, t, nblocks(len), sel);
  if (rc) return rc;
  int64_t n = 0;
  for (int64_t j = 0; j <= p; ++j)
    if (sel[j / BLK]) keys[n++] = s + j;
  *nkeys = n;
  return OR_OK;
}

/* Validate q2k in full (every slot of every token and index head). */
static int check_q2k(const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D) {
  for (int64_t t = 0; t < T; ++t) {
    int32_t d = doc_of(offs, D, t);
    int32_t nb = nblocks(offs[d + 1] - offs[d]);
    for (int g = 0; g < NKV; ++g)
      for (int i = 0; i < TOPK; ++i) {
        int32_t v = q2k[((int64_t)g * T + t) * TOPK + i];
        if (v < -1 || v >= nb) return OR_BAD_Q2K;
      }
  }
  return OR_OK;
}

/* scale * <Q[t,h,:], K[j,g,:]> */
static double score(const elem_t* Q, const elem_t* K, int64_t t, int h, int64_t j, int g,
                    double scale) {
  const elem_t* q = Q + ((int64_t)t * NQH + h) * HD;
  const elem_t* k = K + ((int64_t)j * NKV + g) * HD;
  double acc = 0.0;
  for (int c = 0; c < HD; ++c) acc += ld(q, c) * ld(k, c);
  return scale * acc;
}

/* Forward of one query token t for the 16 heads of index head g:
 * LSE[h] = ln sum_j exp(s_j), P_j = exp(s_j - LSE), O[h] = sum_j P_j V[j,g].
 * o: [16][128], lse: [16].  s: scratch of nkeys doubles. */
static void row_forward(const elem_t* Q, const elem_t* K, const elem_t* V, int64_t t, int g,
                        const int64_t* keys, int64_t nkeys, double scale, double* s, double* o,
                        double* lse) {
  for (int hh = 0; hh < HPG; ++hh) {
    int h = g * HPG + hh;
    double* oh = o + (int64_t)hh * HD;
    for (int c = 0; c < HD; ++c) oh[c] = 0.0;
    if (nkeys == 0) {
      lse[hh] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int64_t i = 0; i < nkeys; ++i) {
      s[i] = score(Q, K, t, h, keys[i], g, scale);
      if (s[i] > m) m = s[i];
    }
    double sum = 0.0;
    for (int64_t i = 0; i < nkeys; ++i) sum += exp(s[i] - m);
    double L = m + log(sum);
    lse[hh] = L;
    for (int64_t i = 0; i < nkeys; ++i) {
      double pr = exp(s[i] - L);
      const elem_t* vr = V + ((int64_t)keys[i] * NKV + g) * HD;
      for (int c = 0; c < HD; ++c) oh[c] += pr * ld(vr, c);
    }
  }
}

/* ------------------------------------------------------------------------
 * Forward on a list of query tokens (all 64 heads each).
 * toks == NULL means every token 0..T-1 (ntoks must equal T).
 * O: [ntoks][64][128], LSE: [ntoks][64].
 */
int oracle_forward(const elem_t* Q, const elem_t* K, const elem_t* V, const int32_t* q2k,
                   int64_t T, const int32_t* offs, int32_t D, double scale, const int64_t* toks,
                   int64_t ntoks, double* O, double* LSE) {
  if (T <= 0 || check_offsets(offs, D, T)) return OR_BAD_ARGS;
  if (check_q2k(q2k, T, offs, D)) return OR_BAD_Q2K;
  int64_t maxlen = 0;
  for (int32_t d = 0; d < D; ++d)
    if (offs[d + 1] - offs[d] > maxlen) maxlen = offs[d + 1] - offs[d];
  int err = 0;
#pragma omp parallel
  {
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)maxlen);
    double* s = (double*)malloc(sizeof(double) * (size_t)maxlen);
    unsigned char* sel = (unsigned char*)malloc((size_t)nblocks((int32_t)maxlen));
#pragma omp for schedule(dynamic, 4)
    for (int64_t i = 0; i < ntoks; ++i) {
      int64_t t = toks ? toks[i] : i;
      for (int g = 0; g < NKV; ++g) {
        int64_t nk;
        if (keys_of(q2k, T, offs, D, g, t, keys, &nk, sel)) {
          err = OR_BAD_Q2K;
          continue;
        }
        row_forward(Q, K, V, t, g, keys, nk, scale, s, O + (i * NQH + g * HPG) * HD,
                    LSE + i * NQH + g * HPG);
      }
    }
    free(keys);
    free(s);
    free(sel);
  }
  return err;
}

/* ------------------------------------------------------------------------
 * dQ on a list of query tokens.  For L = sum(O * dO):
 *   delta = sum_c dO * O,  dP_j = <dO, V_j>,  dS_j = P_j (dP_j - delta),
 *   dQ = scale * sum_j dS_j K_j.
 * O, LSE and delta are recomputed exactly here.  dQ: [ntoks][64][128].
 * If DELTA is not NULL it receives delta [ntoks][64].
 */
int oracle_dq(const elem_t* Q, const elem_t* K, const elem_t* V, const elem_t* dO,
              const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D, double scale,
              const int64_t* toks, int64_t ntoks, double* dQ, double* DELTA) {
  if (T <= 0 || check_offsets(offs, D, T)) return OR_BAD_ARGS;
  if (check_q2k(q2k, T, offs, D)) return OR_BAD_Q2K;
  int64_t maxlen = 0;
  for (int32_t d = 0; d < D; ++d)
    if (offs[d + 1] - offs[d] > maxlen) maxlen = offs[d + 1] - offs[d];
#pragma omp parallel
  {
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)maxlen);
    double* s = (double*)malloc(sizeof(double) * (size_t)maxlen);
    unsigned char* sel = (unsigned char*)malloc((size_t)nblocks((int32_t)maxlen));
    double o[HPG * HD], lse[HPG];
#pragma omp for schedule(dynamic, 4)
    for (int64_t i = 0; i < ntoks; ++i) {
      int64_t t = toks ? toks[i] : i;
      for (int g = 0; g < NKV; ++g) {
        int64_t nk;
        keys_of(q2k, T, offs, D, g, t, keys, &nk, sel);
        row_forward(Q, K, V, t, g, keys, nk, scale, s, o, lse);
        for (int hh = 0; hh < HPG; ++hh) {
          int h = g * HPG + hh;
          const elem_t* dor = dO + ((int64_t)t * NQH + h) * HD;
          double* dq = dQ + (i * NQH + h) * HD;
          double delta = 0.0;
          for (int c = 0; c < HD; ++c) delta += ld(dor, c) * o[hh * HD + c];
          if (DELTA) DELTA[i * NQH + h] = delta;
          for (int c = 0; c < HD; ++c) dq[c] = 0.0;
          for (int64_t kk = 0; kk < nk; ++kk) {
            int64_t j = keys[kk];
            double pr = exp(score(Q, K, t, h, j, g, scale) - lse[hh]);
            const elem_t* vr = V + (j * NKV + g) * HD;
            const elem_t* kr = K + (j * NKV + g) * HD;
            double dp = 0.0;
            for (int c = 0; c < HD; ++c) dp += ld(dor, c) * ld(vr, c);
            double ds = pr * (dp - delta);
            for (int c = 0; c < HD; ++c) dq[c] += scale * ds * ld(kr, c);
          }
        }
      }
    }
    free(keys);
    free(s);
    free(sel);
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * dK and dV of whole key blocks.  blocks: nblk_req pairs (g, global token
 * index of the block's first key).  For each such block, every query t of the
 * same document that sees a key of the block contributes, over its 16 heads:
 *   dV_j += P_tj dO_t,   dK_j += scale * dS_tj Q_t.
 * dK, dV: [nblk_req][128][128] (rows past the document end stay zero).
 */
int oracle_dkv_blocks(const elem_t* Q, const elem_t* K, const elem_t* V,
                      const elem_t* dO, const int32_t* q2k, int64_t T, const int32_t* offs,
                      int32_t D, double scale, const int64_t* blocks, int64_t nblk_req,
                      double* dK, double* dV) {
  if (T <= 0 || check_offsets(offs, D, T)) return OR_BAD_ARGS;
  if (check_q2k(q2k, T, offs, D)) return OR_BAD_Q2K;
  int64_t maxlen = 0;
  for (int32_t d = 0; d < D; ++d)
    if (offs[d + 1] - offs[d] > maxlen) maxlen = offs[d + 1] - offs[d];
  for (int64_t b = 0; b < nblk_req; ++b) {
    int g = (int)blocks[2 * b];
    int64_t k0 = blocks[2 * b + 1];
    int32_t d = doc_of(offs, D, k0);
    int64_t s0 = offs[d], e0 = offs[d + 1];
    if ((k0 - s0) % BLK) return OR_BAD_ARGS;
    int64_t v = (k0 - s0) / BLK;
    int64_t klen = (e0 - k0 < BLK) ? (e0 - k0) : BLK;
    double* dk = dK + b * BLK * HD;
    double* dv = dV + b * BLK * HD;
    memset(dk, 0, sizeof(double) * BLK * HD);
    memset(dv, 0, sizeof(double) * BLK * HD);
    int nthr = 1;
#ifdef _OPENMP
    nthr = omp_get_max_threads();
#endif
    double* part = (double*)calloc((size_t)nthr * 2 * BLK * HD, sizeof(double));
#pragma omp parallel
    {
      int tid = 0;
#ifdef _OPENMP
      tid = omp_get_thread_num();
#endif
      double* pk = part + (size_t)tid * 2 * BLK * HD;
      double* pv = pk + BLK * HD;
      int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)maxlen);
      double* s = (double*)malloc(sizeof(double) * (size_t)maxlen);
      unsigned char* sel = (unsigned char*)malloc((size_t)nblocks((int32_t)maxlen));
      double o[HPG * HD], lse[HPG];
#pragma omp for schedule(static)
      for (int64_t t = k0; t < e0; ++t) {
        selection(q2k, T, g, t, nblocks((int32_t)(e0 - s0)), sel);
        if (!sel[v]) continue;
        int64_t nk;
        keys_of(q2k, T, offs, D, g, t, keys, &nk, sel);
        row_forward(Q, K, V, t, g, keys, nk, scale, s, o, lse);
        for (int hh = 0; hh < HPG; ++hh) {
          int h = g * HPG + hh;
          const elem_t* dor = dO + (t * NQH + h) * HD;
          const elem_t* qr = Q + (t * NQH + h) * HD;
          double delta = 0.0;
          for (int c = 0; c < HD; ++c) delta += ld(dor, c) * o[hh * HD + c];
          for (int64_t r = 0; r < klen && k0 + r <= t; ++r) {
            int64_t j = k0 + r;
            double pr = exp(score(Q, K, t, h, j, g, scale) - lse[hh]);
            const elem_t* vr = V + (j * NKV + g) * HD;
            double dp = 0.0;
            for (int c = 0; c < HD; ++c) dp += ld(dor, c) * ld(vr, c);
            double ds = pr * (dp - delta);
            for (int c = 0; c < HD; ++c) {
              pv[r * HD + c] += pr * ld(dor, c);
              pk[r * HD + c] += scale * ds * ld(qr, c);
            }
          }
        }
      }
      free(keys);
      free(s);
      free(sel);
    }
    for (int th = 0; th < nthr; ++th) {
      const double* pk = part + (size_t)th * 2 * BLK * HD;
      for (int64_t x = 0; x < BLK * HD; ++x) {
        dk[x] += pk[x];
        dv[x] += pk[BLK * HD + x];
      }
    }
    free(part);
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * Full backward: dQ [T][64][128], dK, dV [T][4][128].  dQ comes from
 * oracle_dq over all tokens; dK/dV from oracle_dkv_blocks over every (index
 * head, key block) of every document, scattered back to token rows.
 */
int oracle_backward(const elem_t* Q, const elem_t* K, const elem_t* V, const elem_t* dO,
                    const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D, double scale,
                    double* dQ, double* dK, double* dV) {
  int rc = oracle_dq(Q, K, V, dO, q2k, T, offs, D, scale, NULL, T, dQ, NULL);
  if (rc) return rc;
  memset(dK, 0, sizeof(double) * (size_t)T * NKV * HD);
  memset(dV, 0, sizeof(double) * (size_t)T * NKV * HD);
  double* bk = (double*)malloc(sizeof(double) * BLK * HD);
  double* bv = (double*)malloc(sizeof(double) * BLK * HD);
  for (int32_t d = 0; d < D; ++d) {
    for (int64_t k0 = offs[d]; k0 < offs[d + 1]; k0 += BLK) {
      int64_t klen = offs[d + 1] - k0 < BLK ? offs[d + 1] - k0 : BLK;
      for (int g = 0; g < NKV; ++g) {
        int64_t req[2] = {g, k0};
        rc = oracle_dkv_blocks(Q, K, V, dO, q2k, T, offs, D, scale, req, 1, bk, bv);
        if (rc) break;
        for (int64_t r = 0; r < klen; ++r)
          for (int c = 0; c < HD; ++c) {
            dK[((k0 + r) * NKV + g) * HD + c] = bk[r * HD + c];
            dV[((k0 + r) * NKV + g) * HD + c] = bv[r * HD + c];
          }
      }
    }
  }
  free(bk);
  free(bv);
  return rc;
}

/* ------------------------------------------------------------------------
 * The k2q plan in canonical form.
 *   nblk[d] = ceil(len_d / 128); blk_base[d] = sum_{d'<d} nblk[d'];
 *   NB = sum nblk; bucket(g, d, v) = g*NB + blk_base[d] + v.
 *   The bucket holds every query t of document d with v in Sel(t,g) and
 *   v <= (t - s_d)/128, ascending in t (row_ptr / col CSR, 4*NB buckets).
 *   Tasks: the bucket's queries are cut at super-block boundaries - runs of
 *   Z consecutive query blocks (Z = 0: the whole document) - and each run is
 *   split, in order, into chunks of at most 8 queries.  A task is
 *   (bucket, col index of its first query, query count).
 * Output arrays are caller-allocated; the capacities guard them.
 * counts[0] = NB, counts[1] = nnz, counts[2] = ntasks.
 */
int oracle_plan(const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D, int32_t Z,
                int32_t* nblk, int32_t* blk_base, int64_t* row_ptr, int64_t row_ptr_cap,
                int32_t* col, int64_t col_cap, int64_t* tasks, int64_t task_cap,
                int64_t* counts) {
  if (T <= 0 || Z < 0 || check_offsets(offs, D, T)) return OR_BAD_ARGS;
  if (check_q2k(q2k, T, offs, D)) return OR_BAD_Q2K;
  int64_t NB = 0;
  int32_t maxnb = 0;
  for (int32_t d = 0; d < D; ++d) {
    nblk[d] = nblocks(offs[d + 1] - offs[d]);
    blk_base[d] = (int32_t)NB;
    NB += nblk[d];
    if (nblk[d] > maxnb) maxnb = nblk[d];
  }
  if (4 * NB + 1 > row_ptr_cap) return OR_CAPACITY;
  unsigned char* sel = (unsigned char*)malloc((size_t)maxnb);
  /* count */
  for (int64_t b = 0; b <= 4 * NB; ++b) row_ptr[b] = 0;
  for (int g = 0; g < NKV; ++g)
    for (int64_t t = 0; t < T; ++t) {
      int32_t d = doc_of(offs, D, t);
      int64_t qb = (t - offs[d]) / BLK;
      selection(q2k, T, g, t, nblk[d], sel);
      for (int64_t v = 0; v <= qb; ++v)
        if (sel[v]) row_ptr[g * NB + blk_base[d] + v + 1] += 1;
    }
  for (int64_t b = 0; b < 4 * NB; ++b) row_ptr[b + 1] += row_ptr[b];
  int64_t nnz = row_ptr[4 * NB];
  if (nnz > col_cap) {
    free(sel);
    return OR_CAPACITY;
  }
  /* fill, ascending t within each bucket */
  int64_t* fillpos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(4 * NB));
  for (int64_t b = 0; b < 4 * NB; ++b) fillpos[b] = row_ptr[b];
  for (int g = 0; g < NKV; ++g)
    for (int64_t t = 0; t < T; ++t) {
      int32_t d = doc_of(offs, D, t);
      int64_t qb = (t - offs[d]) / BLK;
      selection(q2k, T, g, t, nblk[d], sel);
      for (int64_t v = 0; v <= qb; ++v)
        if (sel[v]) col[fillpos[g * NB + blk_base[d] + v]++] = (int32_t)t;
    }
  /* tasks */
  int64_t nt = 0;
  int rc = OR_OK;
  for (int g = 0; g < NKV && !rc; ++g)
    for (int32_t d = 0; d < D && !rc; ++d)
      for (int32_t v = 0; v < nblk[d] && !rc; ++v) {
        int64_t b = g * NB + blk_base[d] + v;
        int64_t i = row_ptr[b];
        while (i < row_ptr[b + 1]) {
          int64_t run_sb = Z ? ((col[i] - offs[d]) / BLK) / Z : 0;
          int64_t n = 0;
          while (i + n < row_ptr[b + 1] && n < 8 &&
                 (Z ? ((col[i + n] - offs[d]) / BLK) / Z : 0) == run_sb)
            ++n;
          if (nt >= task_cap) {
            rc = OR_CAPACITY;
            break;
          }
          tasks[3 * nt + 0] = b;
          tasks[3 * nt + 1] = i;
          tasks[3 * nt + 2] = n;
          ++nt;
          i += n;
        }
      }
  counts[0] = NB;
  counts[1] = nnz;
  counts[2] = nt;
  free(fillpos);
  free(sel);
  return rc;
}

/* Number of attended (query, head, key) triples: sum over t, g of
 * 16 * |Keys(t,g)|.  This is the pair count the FLOP metric uses. */
int64_t oracle_pair_count(const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D) {
  if (T <= 0 || check_offsets(offs, D, T) || check_q2k(q2k, T, offs, D)) return -1;
  int32_t maxnb = 0;
  for (int32_t d = 0; d < D; ++d)
    if (nblocks(offs[d + 1] - offs[d]) > maxnb) maxnb = nblocks(offs[d + 1] - offs[d]);
  int64_t total = 0;
#pragma omp parallel reduction(+ : total)
  {
    unsigned char* sel = (unsigned char*)malloc((size_t)maxnb);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      int32_t d = doc_of(offs, D, t);
      int64_t p = t - offs[d];
      for (int g = 0; g < NKV; ++g) {
        selection(q2k, T, g, t, nblocks(offs[d + 1] - offs[d]), sel);
        for (int64_t v = 0; v * BLK <= p; ++v)
          if (sel[v]) {
            int64_t hi = (v + 1) * BLK - 1 < p ? (v + 1) * BLK - 1 : p;
            total += HPG * (hi - v * BLK + 1);
          }
      }
    }
    free(sel);
  }
  return total;
}

/* Number of OpenMP threads the oracle runs with. */
int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Octet groups of the forward schedule (a reading: the pages fix the task
 * tile - 8 queries x the 16 heads of an index head - but not how the tiles
 * of one query set are merged).
 *
 * For index head g, the tokens of document d are cut into aligned octets:
 * document positions 8k .. 8k+7 (fewer at the document's end), all in one
 * block b.  S_t = {v in q2k[g, t, :] : 0 <= v <= b} is token t's set of
 * visible selected blocks.  An octet is
 *   UNIFORM when all its tokens have the same non-empty S_t: its tile walks
 *     exactly those blocks;
 *   DENSE when it is not uniform, b + 1 <= dense_blocks and some S_t is
 *     non-empty: its tile walks all blocks 0 .. b, and a token's rows take
 *     part in block v only where v is in S_t (a per-token bit mask);
 * and GROUPED when it is either: one tile then accumulates its rows block
 * after block without a merge.  Octets 2i and 2i+1 of a document form one
 * item when both are uniform with the same set, or both dense (the same
 * blocks 0 .. b); every other grouped octet is an item alone.
 *   grouped: uint8 [4][T]  (1 = the token's octet is grouped)
 *   items:   int64 [cap][23]: tokA, tokB (-1 if none), nqA, nqB, g, nsel,
 *            dense, then 16 words: uniform - the blocks ascending (-1
 *            padded); dense - the masks (bit v = v in S_t) of tokens
 *            tokA .. tokA+7 and tokB .. tokB+7 (0 past the octet's end);
 *            nsel = |S| (uniform) or b + 1 (dense); items in (g, d, k) order
 *   counts:  [0] = items
 * dense_blocks <= 0 makes no octet dense; it is at most 64 (one 64-bit mask
 * per token).  The forward's task list is then the task list without the
 * tasks all of whose queries are grouped (see oracle/__init__.py).
 */
#define ITEM_WORDS 23
enum { OCT_NONE = 0, OCT_UNIFORM = 1, OCT_DENSE = 2 };

int oracle_groups(const int32_t* q2k, int64_t T, const int32_t* offs, int32_t D,
                  int32_t dense_blocks, unsigned char* grouped, int64_t* items,
                  int64_t item_cap, int64_t* counts) {
  if (T <= 0 || check_offsets(offs, D, T) || dense_blocks > 64) return OR_BAD_ARGS;
  if (check_q2k(q2k, T, offs, D)) return OR_BAD_Q2K;
  int32_t maxnb = 0;
  for (int32_t d = 0; d < D; ++d)
    if (nblocks(offs[d + 1] - offs[d]) > maxnb) maxnb = nblocks(offs[d + 1] - offs[d]);
  unsigned char* s0 = (unsigned char*)malloc((size_t)maxnb);
  unsigned char* s1 = (unsigned char*)malloc((size_t)maxnb);
  memset(grouped, 0, (size_t)(4 * T));
  int64_t n = 0;
  int rc = OR_OK;
  for (int g = 0; g < NKV && !rc; ++g)
    for (int32_t d = 0; d < D && !rc; ++d) {
      const int64_t st = offs[d];
      const int32_t len = offs[d + 1] - offs[d];
      const int32_t nb = nblocks(len);
      /* octet k covers document positions [8k, min(8k + 8, len)) */
      const int32_t noct = (len + 7) / 8;
      int* kind = (int*)malloc(sizeof(int) * (size_t)noct);
      for (int32_t k = 0; k < noct; ++k) {
        const int64_t t0 = st + 8 * (int64_t)k;
        const int64_t t1 = (8 * (int64_t)k + 8 < len) ? t0 + 8 : st + len;
        const int32_t b = (int32_t)(8 * (int64_t)k / BLK);
        int same = 1, any = 0;
        selection(q2k, T, g, t0, nb, s0);
        for (int32_t v = 0; v <= b; ++v) any |= s0[v];
        const int first_nonempty = any;
        for (int64_t t = t0 + 1; t < t1; ++t) {
          selection(q2k, T, g, t, nb, s1);
          for (int32_t v = 0; v <= b; ++v) {
            any |= s1[v];
            if (s1[v] != s0[v]) same = 0;
          }
        }
        if (same && first_nonempty)
          kind[k] = OCT_UNIFORM;
        else if (!same && any && b + 1 <= dense_blocks)
          kind[k] = OCT_DENSE;
        else
          kind[k] = OCT_NONE;
        if (kind[k] != OCT_NONE)
          for (int64_t t = t0; t < t1; ++t) grouped[(int64_t)g * T + t] = 1;
      }
      /* octets k, k+1 (k even) pair when both dense, or both uniform with
         the same set */
      int* paired = (int*)calloc((size_t)noct, sizeof(int));
      for (int32_t k = 0; k + 1 < noct; k += 2) {
        const int32_t b = (int32_t)(8 * (int64_t)k / BLK);
        if (kind[k] == OCT_DENSE && kind[k + 1] == OCT_DENSE) {
          paired[k] = 1;
        } else if (kind[k] == OCT_UNIFORM && kind[k + 1] == OCT_UNIFORM) {
          selection(q2k, T, g, st + 8 * (int64_t)k, nb, s0);
          selection(q2k, T, g, st + 8 * (int64_t)k + 8, nb, s1);
          paired[k] = 1;
          for (int32_t v = 0; v <= b; ++v)
            if (s0[v] != s1[v]) paired[k] = 0;
        }
      }
      for (int32_t k = 0; k < noct && !rc; ++k) {
        if (kind[k] == OCT_NONE || (k % 2 == 1 && paired[k - 1])) continue;
        if (n >= item_cap) {
          rc = OR_CAPACITY;
          break;
        }
        const int pair = k % 2 == 0 && paired[k];
        const int64_t t0 = st + 8 * (int64_t)k;
        const int32_t b = (int32_t)(8 * (int64_t)k / BLK);
        int64_t* it = items + n * ITEM_WORDS;
        const int32_t nqa = (8 * k + 8 < len) ? 8 : len - 8 * k;
        const int32_t nqb = pair ? ((8 * (k + 1) + 8 < len) ? 8 : len - 8 * (k + 1)) : 0;
        it[0] = t0;
        it[1] = pair ? t0 + 8 : -1;
        it[2] = nqa;
        it[3] = nqb;
        it[4] = g;
        it[6] = kind[k] == OCT_DENSE;
        if (kind[k] == OCT_UNIFORM) {
          selection(q2k, T, g, t0, nb, s0);
          int32_t j = 0;
          for (int32_t v = 0; v <= b; ++v)
            if (s0[v]) it[7 + j++] = v;
          it[5] = j;
          for (; j < TOPK; ++j) it[7 + j] = -1;
        } else {
          it[5] = b + 1;
          for (int x = 0; x < 2; ++x)
            for (int i = 0; i < 8; ++i) {
              int64_t mask = 0;
              if (i < (x ? nqb : nqa)) {
                selection(q2k, T, g, t0 + 8 * x + i, nb, s0);
                for (int32_t v = 0; v <= b; ++v)
                  if (s0[v]) mask |= (int64_t)1 << v;
              }
              it[7 + 8 * x + i] = mask;
            }
        }
        ++n;
      }
      free(kind);
      free(paired);
    }
  counts[0] = n;
  free(s0);
  free(s1);
  return rc;
}

/* ------------------------------------------------------------------------
 * Block selection: the index scorer and top-k that produce q2k.
 *
 * The pages name the step (an indexer scores the key blocks, each query
 * keeps the top 16) but print no scoring formula; the plainest reading:
 *   summary(g, d, v)[c] = mean over the keys j of document block v of
 *                         ik[j, g, c]   (block v = document positions
 *                         128v .. 128v+127, the last one may be partial)
 *   score(t, g, v)      = sum_c iq[t, g, c] * summary(g, d, v)[c]
 * over the candidate blocks v = 0 .. b of the query's document (b = its own
 * block).  With b + 1 <= 16 every candidate is selected.  Otherwise the 16
 * best by (score descending, block ascending) are kept; with force_local the
 * sink block 0 and the query's own block b are always kept and 14 are chosen
 * among 1 .. b-1.  Slots hold the chosen blocks in ascending order, then -1.
 *
 * Everything is fp64 on the exactly widened bf16 inputs.  A kernel that ranks
 * in a lower precision can differ from this where two candidates' scores lie
 * within its rounding of each other; the tests check such rows for validity
 * against the fp64 scores (oracle_block_scores) instead of equality.
 * iq, ik: bf16 bit patterns [T][4][dim]; q2k: [4][T][16].
 */
static double bf16_to_f64(uint16_t u) {
  uint32_t w = (uint32_t)u << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* (s1, v1) ranks before (s2, v2)? */
static int sel_better(double s1, int32_t v1, double s2, int32_t v2) {
  return s1 > s2 || (s1 == s2 && v1 < v2);
}

/* summary(g, d, v)[0 .. dim) for every block v of document d. */
static void block_summaries(const uint16_t* ik, int32_t dim, int64_t s0, int32_t len, int g,
                            double* summ) {
  const int32_t nb = nblocks(len);
  for (int32_t v = 0; v < nb; ++v) {
    const int32_t n = (len - v * BLK) < BLK ? (len - v * BLK) : BLK;
    for (int32_t c = 0; c < dim; ++c) {
      double acc = 0.0;
      for (int32_t j = 0; j < n; ++j)
        acc += bf16_to_f64(ik[((s0 + (int64_t)v * BLK + j) * NKV + g) * dim + c]);
      summ[(int64_t)v * dim + c] = acc / (double)n;
    }
  }
}

/* score(t, g, v) for v = 0 .. b. */
static void block_scores(const uint16_t* iq, int32_t dim, int64_t t, int g, int32_t b,
                         const double* summ, double* score) {
  for (int32_t v = 0; v <= b; ++v) {
    double acc = 0.0;
    for (int32_t c = 0; c < dim; ++c)
      acc += bf16_to_f64(iq[(t * NKV + g) * dim + c]) * summ[(int64_t)v * dim + c];
    score[v] = acc;
  }
}

int oracle_select_blocks(const uint16_t* iq, const uint16_t* ik, int64_t T, int32_t dim,
                         const int32_t* offs, int32_t D, int32_t force_local, int32_t* q2k) {
  if (T <= 0 || dim <= 0 || check_offsets(offs, D, T)) return OR_BAD_ARGS;
  int64_t maxnb = 0;
  for (int32_t d = 0; d < D; ++d)
    if (nblocks(offs[d + 1] - offs[d]) > maxnb) maxnb = nblocks(offs[d + 1] - offs[d]);
#pragma omp parallel
  {
    double* summ = (double*)malloc(sizeof(double) * (size_t)maxnb * (size_t)dim);
    double* score = (double*)malloc(sizeof(double) * (size_t)maxnb);
    unsigned char* taken = (unsigned char*)malloc((size_t)maxnb);
    int32_t cached_doc = -1, cached_g = -1;
#pragma omp for schedule(dynamic, 16)
    for (int64_t i = 0; i < 4 * T; ++i) {
      const int g = (int)(i / T);
      const int64_t t = i % T;
      const int32_t d = doc_of(offs, D, t);
      const int64_t s0 = offs[d];
      const int32_t len = offs[d + 1] - offs[d];
      const int32_t b = (int32_t)((t - s0) / BLK);
      int32_t* out = q2k + ((int64_t)g * T + t) * TOPK;
      if (b + 1 <= TOPK) {
        for (int k = 0; k < TOPK; ++k) out[k] = k <= b ? k : -1;
        continue;
      }
      if (d != cached_doc || g != cached_g) {
        block_summaries(ik, dim, s0, len, g, summ);
        cached_doc = d;
        cached_g = g;
      }
      block_scores(iq, dim, t, g, b, summ, score);
      /* selection by repeated best-of-the-rest */
      memset(taken, 0, (size_t)b + 1);
      int32_t chosen[TOPK];
      int nc = 0;
      if (force_local) {
        chosen[nc++] = 0;
        chosen[nc++] = b;
        taken[0] = taken[b] = 1;
      }
      while (nc < TOPK) {
        int32_t best = -1;
        for (int32_t v = 0; v <= b; ++v)
          if (!taken[v] && (best < 0 || sel_better(score[v], v, score[best], best))) best = v;
        if (best < 0) break;
        taken[best] = 1;
        chosen[nc++] = best;
      }
      for (int x = 1; x < nc; ++x) /* ascending */
        for (int y = x; y > 0 && chosen[y - 1] > chosen[y]; --y) {
          int32_t tmp = chosen[y];
          chosen[y] = chosen[y - 1];
          chosen[y - 1] = tmp;
        }
      for (int k = 0; k < TOPK; ++k) out[k] = k < nc ? chosen[k] : -1;
    }
    free(summ);
    free(score);
    free(taken);
  }
  return OR_OK;
}

/* fp64 scores of the candidate blocks 0 .. b of the listed (index head,
 * token) rows: scores[r * maxb + v] for v <= b, NaN after.  rows: n pairs
 * (g, t), best sorted by (g, t) (a thread reuses the summaries of the last
 * (g, document) it met); maxb: the row stride (>= largest b + 1). */
int oracle_block_scores(const uint16_t* iq, const uint16_t* ik, int64_t T, int32_t dim,
                        const int32_t* offs, int32_t D, const int64_t* rows, int64_t n,
                        int64_t maxb, double* scores) {
  if (T <= 0 || dim <= 0 || maxb <= 0 || check_offsets(offs, D, T)) return OR_BAD_ARGS;
  int64_t maxnb = 0;
  for (int32_t d = 0; d < D; ++d)
    if (nblocks(offs[d + 1] - offs[d]) > maxnb) maxnb = nblocks(offs[d + 1] - offs[d]);
  int err = OR_OK;
#pragma omp parallel
  {
    double* summ = (double*)malloc(sizeof(double) * (size_t)maxnb * (size_t)dim);
    int32_t cached_doc = -1, cached_g = -1;
#pragma omp for schedule(dynamic, 64)
    for (int64_t r = 0; r < n; ++r) {
      const int g = (int)rows[2 * r];
      const int64_t t = rows[2 * r + 1];
      double* out = scores + r * maxb;
      for (int64_t v = 0; v < maxb; ++v) out[v] = NAN;
      if (g < 0 || g >= NKV || t < 0 || t >= T) {
#pragma omp atomic write
        err = OR_BAD_ARGS;
        continue;
      }
      const int32_t d = doc_of(offs, D, t);
      const int64_t s0 = offs[d];
      const int32_t len = offs[d + 1] - offs[d];
      const int32_t b = (int32_t)((t - s0) / BLK);
      if (b + 1 > maxb) {
#pragma omp atomic write
        err = OR_BAD_ARGS;
        continue;
      }
      if (d != cached_doc || g != cached_g) {
        block_summaries(ik, dim, s0, len, g, summ);
        cached_doc = d;
        cached_g = g;
      }
      block_scores(iq, dim, t, g, b, summ, out);
    }
    free(summ);
  }
  return err;
}
