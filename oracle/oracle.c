/*
 * oracle.c -- plain, slow CPU reference for the LSA c4 indexer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path (sparse_attention_kv_c4_gb300/csrc) and includes none of its
 * headers.  Every result is the plain definition written out, accumulated in
 * fp64, in the order the pages state it.  OpenMP only splits independent
 * outputs across threads; it never changes a summation order.
 *
 * Sources (page titles as published):
 *   [FM]  "FlashMemory-DeepSeek-V4: Lightning Index Ultra-Long Context via
 *         Lookahead Sparse Attention" (paper summary), sec. 3 "Memory Indexer
 *         scoring function" and sec. 6 "Implementation boundary".
 *   [RM]  "FlashMemory-DeepSeek-V4" (repository README): "Retriever
 *         architecture", "compressed_k format", "Two-level recall algorithm".
 *   [V4]  "DeepSeek-V4 CSA + HCA explained" (yuyanqi.com): sec. 3 "C4Indexer"
 *         (CSA-1 score, CSA-2 top-512), sec. 8 (c4 chunk = 4 tokens).
 *
 * Readings where the pages are silent:
 *   - Ranking is by the pre-sigmoid logit; equal logits are ordered by the
 *     lower chunk id first.  NaN logits rank as -inf.
 *   - The threshold test is inclusive: sigma(x) >= thr.
 *   - Fewer candidates than k: all are returned, padded with id -1.
 *   - Prefill causal limit: chunk s is a candidate of a query at position pos
 *     iff s < min(S, floor(pos / ratio)).
 *   - Selected ids are emitted sorted by ascending chunk id.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Element decoding                                                           */
/* ------------------------------------------------------------------------- */

/* bfloat16: the upper half of an IEEE binary32; the value is exact in fp64. */
ORC_API double orc_bf16(uint16_t bits) {
  union { uint32_t u; float f; } v;
  v.u = (uint32_t)bits << 16;
  return (double)v.f;
}

/* OCP FP8 E4M3 ([RM] "compressed_k format": bytes [:128] are float8_e4m3):
 * sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is
 * subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
ORC_API double orc_e4m3(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xF;
  int m = bits & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* [RM] "compressed_k format": dequant = fp8.float() * scale, an fp32 product. */
static double orc_dequant(uint8_t code, float scale) {
  float kv = (float)orc_e4m3(code) * scale;
  return (double)kv;
}

/* ------------------------------------------------------------------------- */
/* Indexer score                                                              */
/* ------------------------------------------------------------------------- */

/* x = sum_h w_h * ReLU(q_h . k)  -- the argument of sigma in [FM] sec. 3
 * (I_{t,s}) and the native C4Indexer score of [V4] sec. 3 (CSA-1).
 * q is [n_h][d] bf16, w is [n_h] fp32 (already fused with any head scaling,
 * [RM] "fused_w"), k is the dequantised key [d] in fp64. */
static double orc_score_k(const uint16_t* q, const float* w, const double* k, int n_h, int d) {
  double x = 0.0;
  for (int h = 0; h < n_h; ++h) {
    double dot = 0.0;
    for (int j = 0; j < d; ++j) dot += orc_bf16(q[(size_t)h * d + j]) * k[j];
    double relu = dot > 0.0 ? dot : 0.0;
    x += (double)w[h] * relu;
  }
  return x;
}

ORC_API double orc_score_bf16(const uint16_t* q, const float* w, const uint16_t* k, int n_h, int d) {
  double kd[1024];
  if (d > 1024) return NAN;
  for (int j = 0; j < d; ++j) kd[j] = orc_bf16(k[j]);
  return orc_score_k(q, w, kd, n_h, d);
}

ORC_API double orc_score_fp8(const uint16_t* q, const float* w, const uint8_t* k8, float scale, int n_h,
                             int d) {
  double kd[1024];
  if (d > 1024) return NAN;
  for (int j = 0; j < d; ++j) kd[j] = orc_dequant(k8[j], scale);
  return orc_score_k(q, w, kd, n_h, d);
}

/* sigma(x) = 1 / (1 + e^-x), [FM] sec. 3. */
ORC_API double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------- */
/* Memory Indexer: per-layer logits, OR-union over layers, resident bitmask   */
/* ------------------------------------------------------------------------- */

/* x[b][l][s] for q [B][L][n_h][d] bf16, w [B][L][n_h], keys bf16 at
 * K + b*stride_b + l*stride_l + s*d (element strides). */
ORC_API void orc_memindex_logits(const uint16_t* q, const float* w, const uint16_t* K, int64_t stride_b,
                                 int64_t stride_l, int64_t B, int64_t L, int64_t S, int n_h, int d,
                                 double* x_out) {
#pragma omp parallel for collapse(2) schedule(dynamic, 64)
  for (int64_t bl = 0; bl < B * L; ++bl)
    for (int64_t s = 0; s < S; ++s) {
      int64_t b = bl / L, l = bl % L;
      const uint16_t* qb = q + (size_t)bl * n_h * d;
      const float* wb = w + (size_t)bl * n_h;
      const uint16_t* ks = K + b * stride_b + l * stride_l + s * d;
      x_out[(size_t)bl * S + s] = orc_score_bf16(qb, wb, ks, n_h, d);
    }
}

/* The same logits over compressed keys ([FM] sec. 6 and [RM] "compressed_k
 * format": the retriever reads each chunk as 128 E4M3 bytes plus an fp32
 * scale, dequantised as fp8.float() * scale): keys k8 at
 * k8 + b*stride_b + l*stride_l + s*d (byte strides), scales at
 * scale + b*sstride_b + l*sstride_l + s (element strides). */
ORC_API void orc_memindex_logits_fp8(const uint16_t* q, const float* w, const uint8_t* k8, const float* scale,
                                     int64_t stride_b, int64_t stride_l, int64_t sstride_b, int64_t sstride_l,
                                     int64_t B, int64_t L, int64_t S, int n_h, int d, double* x_out) {
#pragma omp parallel for collapse(2) schedule(dynamic, 64)
  for (int64_t bl = 0; bl < B * L; ++bl)
    for (int64_t s = 0; s < S; ++s) {
      int64_t b = bl / L, l = bl % L;
      const uint16_t* qb = q + (size_t)bl * n_h * d;
      const float* wb = w + (size_t)bl * n_h;
      const uint8_t* ks = k8 + b * stride_b + l * stride_l + s * d;
      const float sc = scale[b * sstride_b + l * sstride_l + s];
      x_out[(size_t)bl * S + s] = orc_score_fp8(qb, wb, ks, sc, n_h, d);
    }
}

/* [FM] sec. 3: R[s] = 1(max_l sigma(x_l[s]) >= thr), the OR-union of the
 * per-layer sets {s | I^(l) >= thr}.  mask bit (s & 31) of word s >> 5;
 * bits at s >= S stay zero.  maxsig[b][s] = max_l sigma(x_l[s]). */
ORC_API void orc_memindex_select(const double* x, int64_t B, int64_t L, int64_t S, double thr,
                                 uint32_t* mask, double* maxsig) {
  int64_t words = (S + 31) / 32;
  memset(mask, 0, sizeof(uint32_t) * (size_t)(B * words));
  for (int64_t b = 0; b < B; ++b)
    for (int64_t s = 0; s < S; ++s) {
      double best = -1.0;
      for (int64_t l = 0; l < L; ++l) {
        double sig = orc_sigmoid(x[((size_t)b * L + l) * S + s]);
        if (sig > best) best = sig;
      }
      if (best >= thr) mask[b * words + (s >> 5)] |= 1u << (s & 31);
      if (maxsig) maxsig[b * S + s] = best;
    }
}

/* The retriever's packed compressed_k rows ([RM] "compressed_k format"): a
 * chunk is d + 4 bytes, bytes [0, d) its E4M3 key and bytes [d, d + 4) its
 * fp32 dequant scale, read in the machine's byte order as a tensor view of
 * those bytes reads it.  Splits n packed rows into k8 [n][d] and scale [n]. */
ORC_API void orc_unpack_compressed_k(const uint8_t* ck, int64_t n, int d, uint8_t* k8_out, float* scale_out) {
  for (int64_t i = 0; i < n; ++i) {
    const uint8_t* row = ck + (size_t)i * (size_t)(d + 4);
    memcpy(k8_out + (size_t)i * (size_t)d, row, (size_t)d);
    memcpy(&scale_out[i], row + d, sizeof(float));
  }
}

/* [RM] "Joint checkpoint + ensemble": the per-layer sigmoid scores of a chunk
 * are ensembled -- mode 0: max (the union, the default), mode 1: mean -- into
 * one score e[b][s]; the chunk is resident iff e >= thr.  The mean sums the
 * L sigmoids in layer order and divides by L. */
ORC_API void orc_memindex_ensemble(const double* x, int64_t B, int64_t L, int64_t S, int mode, double thr,
                                   uint32_t* mask, double* ens) {
  int64_t words = (S + 31) / 32;
  memset(mask, 0, sizeof(uint32_t) * (size_t)(B * words));
  for (int64_t b = 0; b < B; ++b)
    for (int64_t s = 0; s < S; ++s) {
      double e;
      if (mode == 0) {
        e = -1.0;
        for (int64_t l = 0; l < L; ++l) {
          double sig = orc_sigmoid(x[((size_t)b * L + l) * S + s]);
          if (sig > e) e = sig;
        }
      } else {
        double sum = 0.0;
        for (int64_t l = 0; l < L; ++l) sum += orc_sigmoid(x[((size_t)b * L + l) * S + s]);
        e = sum / (double)L;
      }
      if (e >= thr) mask[b * words + (s >> 5)] |= 1u << (s & 31);
      if (ens) ens[b * S + s] = e;
    }
}

/* ------------------------------------------------------------------------- */
/* Top-k select                                                               */
/* ------------------------------------------------------------------------- */

typedef struct {
  double x;
  int64_t id;
} orc_cand;

static int orc_rank_cmp(const void* pa, const void* pb) {
  const orc_cand* a = (const orc_cand*)pa;
  const orc_cand* b = (const orc_cand*)pb;
  double xa = isnan(a->x) ? -INFINITY : a->x;
  double xb = isnan(b->x) ? -INFINITY : b->x;
  if (xa > xb) return -1;
  if (xa < xb) return 1;
  if (a->id != b->id) return a->id < b->id ? -1 : 1; /* tie: lower chunk id first */
  return 0;
}

static int orc_id_cmp(const void* pa, const void* pb) {
  const orc_cand* a = (const orc_cand*)pa;
  const orc_cand* b = (const orc_cand*)pb;
  return (a->id > b->id) - (a->id < b->id);
}

/* [FM] sec. 3 (C^CoreComp = Top-k of the native score inside the resident
 * set), [V4] sec. 3 (CSA-2, top-512; fewer than 512 chunks -> take all,
 * sec. 8 worked layout): the min(k, n) best candidates by (x desc, id asc),
 * emitted by ascending id, padded with id -1 / score -inf.  Returns the
 * number selected. */
static int orc_topk_cands(orc_cand* c, int64_t n, int k, int32_t* idx_out, double* score_out) {
  qsort(c, (size_t)n, sizeof(orc_cand), orc_rank_cmp);
  int64_t m = n < k ? n : k;
  qsort(c, (size_t)m, sizeof(orc_cand), orc_id_cmp);
  for (int64_t i = 0; i < k; ++i) {
    idx_out[i] = i < m ? (int32_t)c[i].id : -1;
    if (score_out) score_out[i] = i < m ? c[i].x : -INFINITY;
  }
  return (int)m;
}

ORC_API int orc_topk(const int64_t* ids, const double* x, int64_t n, int k, int32_t* idx_out,
                     double* score_out) {
  orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(n > 0 ? n : 1));
  if (!c) return -1;
  for (int64_t i = 0; i < n; ++i) {
    c[i].x = x[i];
    c[i].id = ids[i];
  }
  int m = orc_topk_cands(c, n, k, idx_out, score_out);
  free(c);
  return m;
}

/* ------------------------------------------------------------------------- */
/* Native paged top-k over the resident pages                                 */
/* ------------------------------------------------------------------------- */

/* [RM] "Two-level recall algorithm", Level 2: the native indexer scores only
 * the resident chunks (read through the page table, [RM] "Page-recall",
 * 64-chunk pages) and keeps the top-k.  Query qi has q [n_h][d] bf16 and w
 * [n_h]; its j-th resident page (j < n_res[qi], or R when n_res is NULL) lives
 * at pool page page_phys[qi][j] and holds logical chunks
 * page_logical[qi][j]*page_size + o.  Pool keys: k8 [P][page_size][d] E4M3,
 * scale [P][page_size] fp32.
 * Level 2 confines the top-k to the resident set by giving non-resident
 * chunks -inf ([RM] Level 2; [FM] sec. 6 Mode A): with res_mask, chunk c of
 * query qi is a candidate only if bit c & 31 of word c >> 5 of mask row
 * qi / mask_group (mask_ld words per row; words past the row read as 0) is
 * set; without it every chunk of the listed pages is.  Reading: a chunk that
 * is not a candidate is never selected (fewer candidates than k -> all of
 * them, padded with -1).  id_mode 0 emits logical chunk ids; id_mode 1 emits
 * reserve cells page_phys*page_size + o ([RM] "Fused remap": top-512 columns
 * map directly to reserve cells).  Reading: the remap only translates the
 * emitted ids -- the selection, its tie-break and its order stay those of
 * the logical chunk ids.
 * logit_out (optional) is [Q][R*page_size] in page-table order: the score of
 * every listed chunk, NaN for slots past n_res. */
/* The pool holds either E4M3 codes with a per-chunk scale (k8, scale) or bf16
 * keys (kbf, no scale); exactly one of k8 / kbf is given. */
static void orc_paged_topk_any(const uint16_t* q, const float* w, const uint8_t* k8, const float* scale,
                               const uint16_t* kbf, const int32_t* page_phys, const int32_t* page_logical,
                               const int32_t* n_res, int64_t Q, int64_t R, int n_h, int d, int page_size, int k,
                               const uint32_t* res_mask, int64_t mask_ld, int mask_group, int id_mode,
                               int32_t* idx_out, double* score_out, double* logit_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t qi = 0; qi < Q; ++qi) {
    int64_t nr = n_res ? n_res[qi] : R;
    if (nr > R) nr = R;
    if (nr < 0) nr = 0;
    orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(nr * page_size > 0 ? nr * page_size : 1));
    int64_t n = 0;
    const uint32_t* mrow = res_mask ? res_mask + (qi / mask_group) * mask_ld : NULL;
    for (int64_t j = 0; j < nr; ++j) {
      int64_t p = page_phys[qi * R + j];
      int64_t lp = page_logical[qi * R + j];
      for (int o = 0; o < page_size; ++o) {
        int64_t row = p * page_size + o;
        double x = kbf ? orc_score_bf16(q + (size_t)qi * n_h * d, w + (size_t)qi * n_h, kbf + (size_t)row * d, n_h, d)
                       : orc_score_fp8(q + (size_t)qi * n_h * d, w + (size_t)qi * n_h, k8 + (size_t)row * d,
                                       scale[row], n_h, d);
        if (logit_out) logit_out[(size_t)qi * R * page_size + j * page_size + o] = x;
        int64_t chunk = lp * page_size + o;
        if (mrow) {
          int64_t word = chunk >> 5;
          uint32_t bits = word < mask_ld ? mrow[word] : 0u;
          if (!((bits >> (chunk & 31)) & 1u)) continue; /* not resident: not a candidate */
        }
        c[n].x = x;
        c[n].id = chunk;
        ++n;
      }
    }
    if (logit_out)
      for (int64_t j = nr; j < R; ++j)
        for (int o = 0; o < page_size; ++o) logit_out[(size_t)qi * R * page_size + j * page_size + o] = NAN;
    int m = orc_topk_cands(c, n, k, idx_out + (size_t)qi * k, score_out ? score_out + (size_t)qi * k : NULL);
    if (id_mode) /* translate each selected logical chunk to its reserve cell */
      for (int i = 0; i < m; ++i) {
        int64_t chunk = idx_out[(size_t)qi * k + i];
        for (int64_t j = 0; j < nr; ++j)
          if (page_logical[qi * R + j] == chunk / page_size) {
            idx_out[(size_t)qi * k + i] = (int32_t)(page_phys[qi * R + j] * page_size + chunk % page_size);
            break;
          }
      }
    free(c);
  }
}

ORC_API void orc_paged_topk_ex(const uint16_t* q, const float* w, const uint8_t* k8, const float* scale,
                               const int32_t* page_phys, const int32_t* page_logical, const int32_t* n_res,
                               int64_t Q, int64_t R, int n_h, int d, int page_size, int k, const uint32_t* res_mask,
                               int64_t mask_ld, int mask_group, int id_mode, int32_t* idx_out, double* score_out,
                               double* logit_out) {
  orc_paged_topk_any(q, w, k8, scale, NULL, page_phys, page_logical, n_res, Q, R, n_h, d, page_size, k, res_mask,
                     mask_ld, mask_group, id_mode, idx_out, score_out, logit_out);
}

/* The same over a pool of bf16 keys kbf [P][page_size][d] (no scale): the
 * native score with the keys as the Memory Indexer reads them ([V4] sec. 3
 * CSA-1 over paged keys; bf16 is the pages' uncompressed key type). */
ORC_API void orc_paged_topk_bf16_ex(const uint16_t* q, const float* w, const uint16_t* kbf,
                                    const int32_t* page_phys, const int32_t* page_logical, const int32_t* n_res,
                                    int64_t Q, int64_t R, int n_h, int d, int page_size, int k,
                                    const uint32_t* res_mask, int64_t mask_ld, int mask_group, int id_mode,
                                    int32_t* idx_out, double* score_out, double* logit_out) {
  orc_paged_topk_any(q, w, NULL, NULL, kbf, page_phys, page_logical, n_res, Q, R, n_h, d, page_size, k, res_mask,
                     mask_ld, mask_group, id_mode, idx_out, score_out, logit_out);
}

ORC_API void orc_paged_topk(const uint16_t* q, const float* w, const uint8_t* k8, const float* scale,
                            const int32_t* page_phys, const int32_t* page_logical, const int32_t* n_res,
                            int64_t Q, int64_t R, int n_h, int d, int page_size, int k, int32_t* idx_out,
                            double* score_out, double* logit_out) {
  orc_paged_topk_ex(q, w, k8, scale, page_phys, page_logical, n_res, Q, R, n_h, d, page_size, k, NULL, 0, 1, 0,
                    idx_out, score_out, logit_out);
}

/* ------------------------------------------------------------------------- */
/* Prefill: many queries against dense chunk keys under the causal limit      */
/* ------------------------------------------------------------------------- */

/* Chunk s covers tokens ratio*s .. ratio*s+ratio-1 ([V4] sec. 1/8: c4 = 4
 * tokens per chunk); it is visible to the query at position pos only when all
 * of its tokens precede pos: s < floor(pos / ratio), and s < S. */
ORC_API int64_t orc_causal_limit(int64_t pos, int64_t S, int ratio) {
  if (pos < 0) return 0;
  int64_t lim = pos / ratio;
  return lim < S ? lim : S;
}

/* q [T][n_h][d] bf16, w [T][n_h], pos [T], K [S][d] bf16. */
ORC_API void orc_prefill_topk(const uint16_t* q, const float* w, const int64_t* pos, const uint16_t* K,
                              int64_t T, int64_t S, int n_h, int d, int ratio, int k, int32_t* idx_out,
                              double* score_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    int64_t n = orc_causal_limit(pos[t], S, ratio);
    orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(n > 0 ? n : 1));
    for (int64_t s = 0; s < n; ++s) {
      c[s].x = orc_score_bf16(q + (size_t)t * n_h * d, w + (size_t)t * n_h, K + (size_t)s * d, n_h, d);
      c[s].id = s;
    }
    orc_topk_cands(c, n, k, idx_out + (size_t)t * k, score_out ? score_out + (size_t)t * k : NULL);
    free(c);
  }
}

/* ------------------------------------------------------------------------- */
/* Page recall: the densest resident pages of each request                    */
/* ------------------------------------------------------------------------- */

/* [RM] "Two-level recall algorithm", Level 1: the resident set is the
 * thresholded Memory-Indexer mask plus the recency tail and the attention
 * sink; [RM] "Page-recall" (64-chunk pages) and the KMAX note under
 * "Reference performance": each request recalls the KMAX pages that hold the
 * most resident chunks (256K -> 96, 512K -> 192, 1M -> 384 pages).
 * Readings where the pages are silent: the sink is chunks [0, sink), the
 * recency tail chunks [S - recent, S); a page's density is its number of
 * resident chunks (the last page may be partial); pages of density 0 are never
 * recalled; equal densities go to the lower page id; the recalled pages are
 * emitted by ascending id, padded with -1 (density -1).
 * mask [B][ceil(S/32)]: bit s & 31 of word s >> 5 is chunk s.  pages_out and
 * density_out are [B][kmax]; n_out[b] is the number of pages recalled. */
ORC_API void orc_page_recall(const uint32_t* mask, int64_t B, int64_t S, int64_t sink, int64_t recent,
                             int page_size, int kmax, int32_t* pages_out, int32_t* density_out, int32_t* n_out) {
  const int64_t words = (S + 31) / 32;
  const int64_t n_pages = (S + page_size - 1) / page_size;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t b = 0; b < B; ++b) {
    orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(n_pages > 0 ? n_pages : 1));
    double* dens = (double*)malloc(sizeof(double) * (size_t)(kmax > 0 ? kmax : 1));
    int64_t n = 0;
    for (int64_t p = 0; p < n_pages; ++p) {
      int64_t density = 0;
      for (int64_t s = p * page_size; s < (p + 1) * page_size && s < S; ++s) {
        int resident = (mask[b * words + (s >> 5)] >> (s & 31)) & 1u;
        if (s < sink || s >= S - recent) resident = 1;
        density += resident;
      }
      if (density > 0) {
        c[n].x = (double)density;
        c[n].id = p;
        ++n;
      }
    }
    n_out[b] = orc_topk_cands(c, n, kmax, pages_out + b * kmax, dens);
    for (int i = 0; i < kmax; ++i) density_out[b * kmax + i] = i < n_out[b] ? (int32_t)dens[i] : -1;
    free(dens);
    free(c);
  }
}

/* ------------------------------------------------------------------------- */
/* Query-side projection chain of one CSA layer ([RM] "Retriever            */
/* architecture" and "Hyperparameters")                                       */
/* ------------------------------------------------------------------------- */

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g. */
ORC_API void orc_rmsnorm(const double* x, const uint16_t* g, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * orc_bf16(g[i]);
}

/* YaRN frequency of rotary pair i of a rope_dim-wide rotary part, the
 * "NTK-by-parts" rule of the YaRN method (Peng et al., 2023): the base
 * frequency theta_i = base^(-2i / rope_dim) has wavelength 2 pi / theta_i and
 * turns r = orig_len / wavelength times over the original context; pairs
 * turning fewer than beta_slow times are interpolated (theta / factor), pairs
 * turning more than beta_fast times keep theta, and in between
 * gamma = (r - beta_slow) / (beta_fast - beta_slow) blends the two:
 * theta' = (1 - gamma) theta / factor + gamma theta. */
ORC_API double orc_yarn_freq(int i, int rope_dim, double base, double factor, double orig_len, double beta_fast,
                             double beta_slow) {
  const double two_pi = 6.283185307179586476925286766559;
  double theta = pow(base, -2.0 * (double)i / (double)rope_dim);
  double r = orig_len * theta / two_pi;
  double gamma = (r - beta_slow) / (beta_fast - beta_slow);
  if (gamma < 0.0) gamma = 0.0;
  if (gamma > 1.0) gamma = 1.0;
  return (1.0 - gamma) * theta / factor + gamma * theta;
}

/* Rotary embedding of the last rope_dim entries of a head_dim vector at
 * position pos: consecutive entries (2i, 2i+1) of the rotary part form pair i
 * and turn by the angle pos * theta'_i (the complex-pair form of rotary
 * embeddings). */
ORC_API void orc_rope_yarn(double* x, int head_dim, int rope_dim, int64_t pos, double base, double factor,
                           double orig_len, double beta_fast, double beta_slow) {
  double* xr = x + head_dim - rope_dim;
  for (int i = 0; i < rope_dim / 2; ++i) {
    double a = (double)pos * orc_yarn_freq(i, rope_dim, base, factor, orig_len, beta_fast, beta_slow);
    double c = cos(a), sn = sin(a);
    double x0 = xr[2 * i], x1 = xr[2 * i + 1];
    xr[2 * i] = x0 * c - x1 * sn;
    xr[2 * i + 1] = x0 * sn + x1 * c;
  }
}

/* Normalised Walsh-Hadamard transform (Sylvester order): y = H x / sqrt(n),
 * H[i][j] = (-1)^popcount(i & j), n a power of two. */
ORC_API void orc_hadamard(const double* x, int n, double* y) {
  double norm = 1.0 / sqrt((double)n);
  for (int i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -x[j] : x[j];
    y[i] = acc * norm;
  }
}

/* The chain for T tokens: for token t,
 *   a = wq_a . hidden_t                     (Linear dim -> r, no bias)
 *   c = RMSNorm(a; q_norm, eps)
 *   u = wq_b . c                            (Linear r -> n_h * head_dim)
 *   q_h = Hadamard(RoPE_yarn(u_h, pos_t))   per head h (u reshaped [n_h, head_dim])
 *   w = (w_proj . hidden_t) * head_dim^-1/2 * n_h^-1/2
 * Weights are row-major [out][in] bf16 (a Linear's weight), hidden [T][dim]
 * bf16; everything is accumulated in fp64 with no intermediate rounding. */
ORC_API void orc_query_chain(const uint16_t* hidden, const uint16_t* wq_a, const uint16_t* q_norm, const uint16_t* wq_b,
                             const uint16_t* w_proj, const int64_t* pos, int64_t T, int dim, int r, int n_h,
                             int head_dim, int rope_dim, double base, double factor, double orig_len, double beta_fast,
                             double beta_slow, double eps, double* q_out, double* w_out) {
  for (int64_t t = 0; t < T; ++t) {
    double* h = (double*)malloc(sizeof(double) * (size_t)dim);
    double* a = (double*)malloc(sizeof(double) * (size_t)r);
    double* c = (double*)malloc(sizeof(double) * (size_t)r);
    double* u = (double*)malloc(sizeof(double) * (size_t)n_h * head_dim);
    for (int i = 0; i < dim; ++i) h[i] = orc_bf16(hidden[(size_t)t * dim + i]);
#pragma omp parallel for schedule(static)
    for (int j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dim; ++i) acc += orc_bf16(wq_a[(size_t)j * dim + i]) * h[i];
      a[j] = acc;
    }
    orc_rmsnorm(a, q_norm, r, eps, c);
#pragma omp parallel for schedule(static)
    for (int j = 0; j < n_h * head_dim; ++j) {
      double acc = 0.0;
      for (int i = 0; i < r; ++i) acc += orc_bf16(wq_b[(size_t)j * r + i]) * c[i];
      u[j] = acc;
    }
    for (int hh = 0; hh < n_h; ++hh) {
      double* uh = u + (size_t)hh * head_dim;
      orc_rope_yarn(uh, head_dim, rope_dim, pos[t], base, factor, orig_len, beta_fast, beta_slow);
      orc_hadamard(uh, head_dim, q_out + ((size_t)t * n_h + hh) * head_dim);
    }
    double ws = 1.0 / sqrt((double)head_dim) / sqrt((double)n_h);
    for (int hh = 0; hh < n_h; ++hh) {
      double acc = 0.0;
      for (int i = 0; i < dim; ++i) acc += orc_bf16(w_proj[(size_t)hh * dim + i]) * h[i];
      w_out[(size_t)t * n_h + hh] = acc * ws;
    }
    free(h);
    free(a);
    free(c);
    free(u);
  }
}

ORC_API int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

ORC_API void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
