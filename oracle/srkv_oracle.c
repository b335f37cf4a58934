/*
 * srkv_oracle.c -- the plain, slow fp64 CPU definition of block-sparse retrieval
 * decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  The GPU library does not link,
 * include or call it, and the two share no code, header, table or constant.
 *
 * Sources (page title, then section):
 *  [OG]  openGauss 7.0.0 DataVec, "KV Cache Query-Based Computation Inference
 *        Acceleration": "Feature Description" (one representation vector per block,
 *        extracted at prefill), "Overall Solution" (initial_tokens / sliding_window /
 *        offload_tokens split; inner-product scoring of the current query against
 *        each representation vector; topK blocks joined with the initial and window
 *        KV for attention), "Configuration Parameters" (INIT_TOKENS_NUM,
 *        LOCAL_TOKENS_NUM, TOPK_PERCENT, block size 128, DENSE_BOUNDARY).
 *  [KVS] "大模型推理百倍加速之KV cache篇" (KV-cache acceleration survey):
 *        "为什么要研究KV cache？" (footprint 4blh(s+n) bytes in fp16) and
 *        "Share--KV cache共享" (GQA: a group of query heads shares one K/V head).
 *  [ATB] rkmt.cn, ATB KV-cache reuse article: §1.1 (Attention = softmax(QK^T/sqrt(d_k))V),
 *        §1.2 (Memory_KV = 2 x layers x seq_len x hidden x precision),
 *        §2.2 (paged attention reads K/V through a page table).
 *
 * Readings where the pages are silent (each repeated at the function it affects):
 *  R1 representation vector = mean of the block's keys, per kv head, over the
 *     tokens of the block that exist (t < L);
 *  R2 GQA: the score of a block for a kv head is the inner product with the SUM of
 *     the group's query vectors (equal to the sum of per-head scores); selection
 *     is per (request, kv head);
 *  R3 "closest" = largest inner product; no scaling is applied to scores;
 *  R4 ties in score go to the lower block index;
 *  R5 k = min(n, ceil(p*n - 1e-9)), and 0 when n = 0;
 *  R6 candidates = blocks that intersect the offload range [INIT, L - LOCAL);
 *  R7 attended tokens = the SET [0, INIT) u (selected blocks n [INIT, W)) u [W, L),
 *     W = L - LOCAL, so no token counts twice;
 *  R8 dense iff prompt length < DENSE_BOUNDARY (then every candidate is selected);
 *  R9 the cache already holds the current token at position L - 1; softmax scale
 *     is 1/sqrt(d); no causal mask is needed at decode; L = 0 gives a zero output.
 *
 * Compressed pages ([KVS] lists KV quantisation among the ways to shrink the cache; the
 * format is the 8-bit floating point "E4M3" of the OCP 8-bit floating point specification,
 * OFP8): with dtype 2 the K and V caches hold one E4M3 code per value and a fp32 scale per
 * (page, kv head, token) row; a value is code x scale.  The query stays bf16.
 *  R10 quantisation of a row x[0..d): scale = max_e |x_e| / 448 in fp32 (1 for an all-zero
 *      row), code_e = E4M3(x_e / scale) with the quotient rounded to fp32 first, then to
 *      the nearest E4M3 value, ties to the even code, finite values past 448 to +-448.
 *  R11 with compressed pages the selection is computed from the representation vectors of
 *      the full-precision keys (they are extracted at prefill, before the pages are
 *      compressed); the attended values are the compressed ones.
 *
 * Arithmetic is fp64 throughout, from the exact input values (bf16 inputs are
 * widened exactly).  The build uses -ffp-contract=off so that the integer
 * decision in R5 is taken with separately rounded multiply and subtract on every
 * host architecture.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t num_q_heads;   /* Hq */
  int32_t num_kv_heads;  /* Hkv; Hq must be a multiple of it */
  int32_t head_dim;      /* d */
  int32_t block_size;    /* S tokens per block (= page) */
  int32_t init_tokens;   /* INIT */
  int32_t local_tokens;  /* LOCAL (sliding window) */
  double topk_percent;   /* p in [0, 1] */
  int32_t dense_boundary;
  int32_t dtype;         /* 0: bf16 bit patterns (uint16), 1: fp32, 2: E4M3 K/V (bf16 q) */
} oracle_cfg;

typedef struct {
  const void* q;               /* [B][Hq][d] */
  const void* k_cache;         /* [P][Hkv][S][d] */
  const void* v_cache;         /* [P][Hkv][S][d] */
  int64_t num_pages;           /* P */
  const int32_t* block_table;  /* [B][max_blocks] logical block -> physical page */
  int32_t max_blocks;
  const int32_t* seq_lens;     /* [B] L: tokens in the cache, current token included */
  const int32_t* prompt_lens;  /* [B] prefill length, compared with DENSE_BOUNDARY */
  int32_t batch;
  const float* k_scale;        /* dtype 2: [P][Hkv][S] scale of each K row */
  const float* v_scale;        /* dtype 2: [P][Hkv][S] scale of each V row */
} oracle_inputs;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_BAD_PAGE = -2, ORACLE_NO_MEM = -3,
       ORACLE_KMAX = -4 };

/* ---- input decoding (exact widening) ------------------------------------------ */

static double value_at(const void* base, int32_t dtype, int64_t i) {
  if (dtype == 1) return (double)((const float*)base)[i];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ---- E4M3 (OCP OFP8): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits -------------
 * Exponent field 0 holds subnormals m/8 x 2^-6; fields 1..15 hold (1 + m/8) x 2^(e-7),
 * except S.1111.111, which is NaN; there are no infinities, the largest finite value is
 * 1.75 x 2^8 = 448. */
double oracle_e4m3_value(uint32_t code) {
  code &= 0xffu;
  const int s = (int)(code >> 7), e = (int)((code >> 3) & 15u), m = (int)(code & 7u);
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* R10: the code of the nearest E4M3 value to x (searched over every finite magnitude),
 * ties to the even code; |x| >= 448 gives +-448; NaN gives 0x7f. */
uint32_t oracle_e4m3_code(double x) {
  if (isnan(x)) return 0x7fu;
  const uint32_t sign = signbit(x) ? 0x80u : 0u;
  const double a = fabs(x);
  if (a >= 448.0) return sign | 0x7eu;
  uint32_t best = 0;
  double bd = INFINITY;
  for (uint32_t code = 0; code <= 0x7eu; ++code) {
    const double dist = fabs(oracle_e4m3_value(code) - a);
    if (dist < bd || (dist == bd && (code & 1u) == 0)) {
      bd = dist;
      best = code;
    }
  }
  return sign | best;
}

void oracle_e4m3_values(const uint8_t* codes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]);
}

void oracle_e4m3_codes(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_code(x[i]);
}

/* R10 for the listed pages of a bf16 cache: codes [n][Hkv][S][d], scales [n][Hkv][S]. */
int oracle_quantize_e4m3(const oracle_cfg* c, const uint16_t* cache, int64_t num_pages,
                         const int32_t* page_ids, int64_t n, uint8_t* codes, float* scales) {
  const int64_t Hkv = c->num_kv_heads, S = c->block_size, d = c->head_dim;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t page = page_ids[i];
    if (page < 0 || page >= num_pages) return ORACLE_BAD_PAGE;
    for (int64_t row = 0; row < Hkv * S; ++row) {
      const uint16_t* x = cache + (page * Hkv * S + row) * d;
      float amax = 0.0f;
      for (int64_t e = 0; e < d; ++e) {
        const float v = fabsf((float)value_at(x, 0, e));
        if (v > amax) amax = v;
      }
      const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
      scales[i * Hkv * S + row] = scale;
      for (int64_t e = 0; e < d; ++e) {
        const float y = (float)value_at(x, 0, e) / scale;  /* fp32 quotient */
        codes[(i * Hkv * S + row) * d + e] = (uint8_t)oracle_e4m3_code((double)y);
      }
    }
  }
  return ORACLE_OK;
}

/* K (which = 0) or V (1) value i of the cache, decoded for the configured dtype. */
static double kv_value(const oracle_cfg* c, const oracle_inputs* in, int which, int64_t i) {
  const void* base = which ? in->v_cache : in->k_cache;
  if (c->dtype != 2) return value_at(base, c->dtype, i);
  const float* sc = which ? in->v_scale : in->k_scale;
  return oracle_e4m3_value(((const uint8_t*)base)[i]) * (double)sc[i / c->head_dim];
}

/* The query's dtype: bf16 when the pages are compressed. */
static int32_t q_dtype(const oracle_cfg* c) { return c->dtype == 2 ? 0 : c->dtype; }

/* ---- closed forms ---------------------------------------------------------------- */

/* KV-cache bytes: 2 (K and V) x batch x layers x tokens x hidden x bytes per value.
 * [ATB] §1.2 writes it per request; [KVS] "为什么要研究KV cache？" writes the fp16
 * case as 4blh(s+n) with tokens = s + n. */
double oracle_kv_cache_bytes(double batch, double layers, double tokens, double hidden,
                             double bytes_per_value) {
  return 2.0 * batch * layers * tokens * hidden * bytes_per_value;
}

/* R5: number of blocks kept out of n candidates for ratio p ([OG] "Configuration
 * Parameters": TOPK_PERCENT is the sparse retrieval ratio). */
int64_t oracle_topk_count(int64_t n, double p) {
  if (n <= 0) return 0;
  double x = ceil(p * (double)n - 1e-9);
  if (!(x > 0.0)) return 0;
  if (x > (double)n) return n;
  return (int64_t)x;
}

/* R6: is block b a candidate, i.e. does [bS, bS+S) meet [INIT, W)? */
static int is_candidate(int64_t b, int64_t S, int64_t INIT, int64_t W) {
  int64_t lo = b * S > INIT ? b * S : INIT;
  int64_t hi = (b + 1) * S < W ? (b + 1) * S : W;
  return lo < hi;
}

/* Count the candidate blocks of a sequence of L tokens by testing every block. */
int64_t oracle_num_candidates(int64_t L, int32_t S, int32_t INIT, int32_t LOCAL) {
  if (L <= 0 || S <= 0) return 0;
  int64_t W = L - LOCAL, n = 0;
  int64_t nblocks = (L + S - 1) / S;
  for (int64_t b = 0; b < nblocks; ++b) n += is_candidate(b, S, INIT, W);
  return n;
}

/* ---- R1: representation vectors ---------------------------------------------------- */

/* Mean over the first valid[i] tokens of physical page page_ids[i], per kv head.
 * reps_out: [n][Hkv][d].  ([OG] "Feature Description": representation vectors are
 * extracted block by block at prefill.) */
int oracle_block_reps(const oracle_cfg* c, const void* k_cache, int64_t num_pages,
                      const int32_t* page_ids, const int32_t* valid, int64_t n,
                      double* reps_out) {
  const int64_t Hkv = c->num_kv_heads, S = c->block_size, d = c->head_dim;
  if (c->dtype == 2) return ORACLE_BAD_ARG;  /* R11: vectors come from the full-precision keys */
  for (int64_t i = 0; i < n; ++i) {
    int64_t page = page_ids[i];
    int64_t v = valid[i];
    if (page < 0 || page >= num_pages) return ORACLE_BAD_PAGE;
    if (v < 0 || v > S) return ORACLE_BAD_ARG;
    for (int64_t h = 0; h < Hkv; ++h) {
      double* rep = reps_out + (i * Hkv + h) * d;
      for (int64_t e = 0; e < d; ++e) {
        double sum = 0.0;
        for (int64_t t = 0; t < v; ++t)
          sum += value_at(k_cache, c->dtype, ((page * Hkv + h) * S + t) * d + e);
        rep[e] = v > 0 ? sum / (double)v : 0.0;
      }
    }
  }
  return ORACLE_OK;
}

/* ---- one (request, kv head) unit ------------------------------------------------------ */

typedef struct {
  double score;
  int32_t block;
} scored_block;

/* R3 + R4: higher score first, then lower block index. */
static int by_score_then_index(const void* pa, const void* pb) {
  const scored_block* a = (const scored_block*)pa;
  const scored_block* b = (const scored_block*)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  return (a->block > b->block) - (a->block < b->block);
}

/* Physical page holding token t of request r, or -1 if out of range. */
static int64_t page_of(const oracle_inputs* in, int32_t r, int64_t t, int64_t S) {
  int64_t b = t / S;
  if (b >= in->max_blocks) return -1;
  int64_t page = in->block_table[(int64_t)r * in->max_blocks + b];
  if (page < 0 || page >= in->num_pages) return -1;
  return page;
}

/*
 * Decode one unit (request r, kv head h): candidate scoring, top-k, attended token
 * set and exact softmax attention for the G query heads of the group.
 *
 *   sel_in / nsel_in : if sel_in != NULL, these logical blocks are taken as the
 *                      selection (the dense rule R8 is then not applied: the given
 *                      selection alone defines the attended set);
 *   sel_out          : [kmax] selected logical blocks, ascending (may be NULL);
 *   nsel_out         : number written to sel_out (may be NULL);
 *   scores_out       : [max_blocks]; candidate scores, NaN for non-candidates (may be NULL);
 *   out              : [G][d] attention output;
 *   weights_out      : [G][L] softmax weight of every token, 0 if not attended (may be NULL).
 */
int oracle_unit(const oracle_cfg* c, const oracle_inputs* in, int32_t r, int32_t h,
                const int32_t* sel_in, int32_t nsel_in, int32_t* sel_out,
                int32_t* nsel_out, int32_t kmax, double* scores_out, double* out,
                double* weights_out) {
  const int64_t Hq = c->num_q_heads, Hkv = c->num_kv_heads, d = c->head_dim;
  const int64_t S = c->block_size, INIT = c->init_tokens, LOCAL = c->local_tokens;
  if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || S <= 0 || r < 0 || r >= in->batch || h < 0 ||
      h >= Hkv)
    return ORACLE_BAD_ARG;
  if (c->dtype == 2 && (!in->k_scale || !in->v_scale)) return ORACLE_BAD_ARG;
  /* R11: over compressed pages the selection comes from the full-precision keys' vectors,
   * which this function does not have: the caller must pass it. */
  if (c->dtype == 2 && !sel_in) return ORACLE_BAD_ARG;
  const int64_t G = Hq / Hkv;
  const int64_t L = in->seq_lens[r];
  const int64_t prompt = in->prompt_lens ? in->prompt_lens[r] : L;
  if (L < 0 || (L + S - 1) / S > in->max_blocks) return ORACLE_BAD_ARG;
  const int64_t W = L - LOCAL;
  const int64_t nblocks = (L + S - 1) / S;
  const int dense = prompt < (int64_t)c->dense_boundary;  /* R8 */

  int rc = ORACLE_OK;
  scored_block* cand = (scored_block*)malloc(sizeof(scored_block) * (size_t)(nblocks + 1));
  char* selected = (char*)calloc((size_t)(nblocks + 1), 1);
  double* qbar = (double*)calloc((size_t)d, sizeof(double));
  double* rep = (double*)calloc((size_t)d, sizeof(double));
  double* logits = (double*)malloc(sizeof(double) * (size_t)(L + 1));
  char* attended = (char*)calloc((size_t)(L + 1), 1);
  if (!cand || !selected || !qbar || !rep || !logits || !attended) {
    rc = ORACLE_NO_MEM;
    goto done;
  }

  /* R2: the group's summed query. */
  for (int64_t j = 0; j < G; ++j)
    for (int64_t e = 0; e < d; ++e)
      qbar[e] += value_at(in->q, q_dtype(c), ((int64_t)r * Hq + h * G + j) * d + e);

  if (scores_out)
    for (int64_t b = 0; b < in->max_blocks; ++b) scores_out[b] = NAN;

  /* R6 + R1 + R3: score every candidate block against the mean of its keys. */
  int64_t n = 0;
  for (int64_t b = 0; b < nblocks; ++b) {
    if (!is_candidate(b, S, INIT, W)) continue;
    int64_t first = b * S;
    int64_t last = (b + 1) * S < L ? (b + 1) * S : L;  /* R1: tokens with t < L */
    int64_t page = page_of(in, r, first, S);
    if (page < 0) {
      rc = ORACLE_BAD_PAGE;
      goto done;
    }
    for (int64_t e = 0; e < d; ++e) {
      double sum = 0.0;
      for (int64_t t = first; t < last; ++t)
        sum += kv_value(c, in, 0, ((page * Hkv + h) * S + (t - first)) * d + e);
      rep[e] = sum / (double)(last - first);
    }
    double s = 0.0;
    for (int64_t e = 0; e < d; ++e) s += qbar[e] * rep[e];
    cand[n].score = s;
    cand[n].block = (int32_t)b;
    ++n;
    if (scores_out) scores_out[b] = s;
  }

  /* Selection: given, dense (R8), or the top k by (score desc, index asc). */
  int64_t nsel = 0;
  if (sel_in) {
    for (int64_t i = 0; i < nsel_in; ++i) {
      int64_t b = sel_in[i];
      if (b < 0 || b >= nblocks) {
        rc = ORACLE_BAD_ARG;
        goto done;
      }
      selected[b] = 1;
    }
  } else if (dense) {
    for (int64_t i = 0; i < n; ++i) selected[cand[i].block] = 1;
  } else {
    int64_t k = oracle_topk_count(n, c->topk_percent);  /* R5 */
    qsort(cand, (size_t)n, sizeof(scored_block), by_score_then_index);
    for (int64_t i = 0; i < k; ++i) selected[cand[i].block] = 1;
  }
  for (int64_t b = 0; b < nblocks; ++b) nsel += selected[b];
  if (sel_out) {
    if (nsel > kmax) {
      rc = ORACLE_KMAX;
      goto done;
    }
    int64_t i = 0;
    for (int64_t b = 0; b < nblocks; ++b)  /* ascending block order */
      if (selected[b]) sel_out[i++] = (int32_t)b;
  }
  if (nsel_out) *nsel_out = (int32_t)nsel;

  /* R7: the attended token set. */
  for (int64_t t = 0; t < L; ++t) attended[t] = (t < INIT) || (t >= W) || selected[t / S];

  /* R9 + [ATB] §1.1: softmax(q K^T / sqrt(d)) V per query head of the group. */
  const double scale = 1.0 / sqrt((double)d);
  for (int64_t j = 0; j < G; ++j) {
    const int64_t qh = h * G + j;
    double* o = out + j * d;
    for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
    double m = -INFINITY;
    for (int64_t t = 0; t < L; ++t) {
      if (!attended[t]) continue;
      int64_t page = page_of(in, r, t, S);
      if (page < 0) {
        rc = ORACLE_BAD_PAGE;
        goto done;
      }
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e)
        dot += value_at(in->q, q_dtype(c), ((int64_t)r * Hq + qh) * d + e) *
               kv_value(c, in, 0, ((page * Hkv + h) * S + t % S) * d + e);
      logits[t] = dot * scale;
      if (logits[t] > m) m = logits[t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t < L; ++t) {
      if (!attended[t]) continue;
      int64_t page = page_of(in, r, t, S);
      double w = exp(logits[t] - m);
      denom += w;
      for (int64_t e = 0; e < d; ++e)
        o[e] += w * kv_value(c, in, 1, ((page * Hkv + h) * S + t % S) * d + e);
    }
    if (denom > 0.0)
      for (int64_t e = 0; e < d; ++e) o[e] /= denom;
    if (weights_out) {
      double* wrow = weights_out + j * L;
      for (int64_t t = 0; t < L; ++t)
        wrow[t] = attended[t] ? exp(logits[t] - m) / denom : 0.0;
    }
  }

done:
  free(cand);
  free(selected);
  free(qbar);
  free(rep);
  free(logits);
  free(attended);
  return rc;
}

/* ---- many units, in parallel over plain threads ------------------------------------------ */

typedef struct {
  const oracle_cfg* c;
  const oracle_inputs* in;
  const int32_t* units;  /* pairs (r, h) */
  int64_t n_units;
  const int32_t* sel_in;
  const int32_t* nsel_in;
  int32_t* sel_out;
  int32_t* nsel_out;
  int32_t kmax;
  double* scores_out;
  double* out;
  int32_t stride, offset;
  int rc;
} unit_job;

static void* run_units(void* arg) {
  unit_job* jb = (unit_job*)arg;
  const int64_t Hkv = jb->c->num_kv_heads, G = jb->c->num_q_heads / Hkv, d = jb->c->head_dim;
  for (int64_t i = jb->offset; i < jb->n_units; i += jb->stride) {
    int32_t r = jb->units[2 * i], h = jb->units[2 * i + 1];
    int64_t u = (int64_t)r * Hkv + h;
    int rc = oracle_unit(
        jb->c, jb->in, r, h, jb->sel_in ? jb->sel_in + u * jb->kmax : NULL,
        jb->nsel_in ? jb->nsel_in[u] : 0, jb->sel_out ? jb->sel_out + u * jb->kmax : NULL,
        jb->nsel_out ? jb->nsel_out + u : NULL, jb->kmax,
        jb->scores_out ? jb->scores_out + u * jb->in->max_blocks : NULL,
        jb->out + ((int64_t)r * jb->c->num_q_heads + h * G) * d, NULL);
    if (rc != ORACLE_OK) {
      jb->rc = rc;
      return NULL;
    }
  }
  return NULL;
}

/* Decode the listed units (pairs (r, h)); outputs are indexed as for the whole batch:
 * sel [B][Hkv][kmax], nsel [B][Hkv], scores [B][Hkv][max_blocks], out [B][Hq][d]. */
int oracle_decode_units(const oracle_cfg* c, const oracle_inputs* in, const int32_t* units,
                        int64_t n_units, const int32_t* sel_in, const int32_t* nsel_in,
                        int32_t* sel_out, int32_t* nsel_out, int32_t kmax,
                        double* scores_out, double* out, int32_t nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t tid[256];
  unit_job jobs[256];
  for (int32_t t = 0; t < nthreads; ++t) {
    jobs[t] = (unit_job){c,      in,      units,      n_units, sel_in, nsel_in, sel_out,
                         nsel_out, kmax, scores_out, out,     nthreads, t,    ORACLE_OK};
  }
  int32_t started = 0;
  for (int32_t t = 1; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, run_units, &jobs[t]) != 0) break;
    started = t;
  }
  run_units(&jobs[0]);
  for (int32_t t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
  /* Any slice whose thread failed to start is done here, serially. */
  for (int32_t t = started + 1; t < nthreads; ++t) run_units(&jobs[t]);
  for (int32_t t = 0; t < nthreads; ++t)
    if (jobs[t].rc != ORACLE_OK) return jobs[t].rc;
  return ORACLE_OK;
}
