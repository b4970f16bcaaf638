/*
 * fp64 CPU oracle for paged decode attention (Gemma-4-12B text path).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes (one output row per (sequence b, query head h)):
 *
 *   Gemma-4-12B model page, "Compute-graph nodes", attn.core rows
 *   (slidingDecodeGQA and decodeGQA):
 *       o[b,h] = sum over visible s of softmax_s(1 * <q[b,h], k[b,s,h/G]>) * v[b,s,h/G]
 *
 *   Attention.lean, `decodeGQA`: the query of a sequence with L cached tokens
 *   sits at position L-1, so with no window every cached key l <= L-1 is
 *   visible, and query head c*G+g reads KV head c.
 *
 *   Attention.lean, `slidingGQA`: the query at position p sees key l iff
 *   l <= p and p < l + window, i.e. p - window < l <= p.  With p = L-1 that is
 *   the last min(L, window) positions (Op Specs page, NOTE on
 *   slidingDecodeGQA: "decode attention over the last w cached positions").
 *
 *   Attention.lean, `softmax`: exp(s_l) / sum over visible m of exp(s_m) for
 *   visible l, 0 otherwise.  This oracle subtracts the largest visible logit
 *   before exponentiating; exp(s_l - M) / sum exp(s_m - M) is the same real
 *   number, and it keeps exp() finite for logits in the hundreds.
 *
 *   Gemma-4-12B model page, "At a glance", shape domain: the KV cache is
 *   paged with page size 16.  Reading (no layout is printed on the pages): a
 *   pool holds pages of `page_size` token rows, each row [Hkv, D], so pool
 *   element (page, slot, c, e) is at ((page*page_size + slot)*Hkv + c)*D + e,
 *   and logical position l of sequence b lives in physical page
 *   block_table[b, l / page_size], slot l % page_size.
 *
 * Inputs are bf16 bit patterns (uint16); each is widened exactly to double.
 * Every sum runs in ascending order of its index, in double precision.
 *
 * Reading of `window`: window > 0 selects the sliding rule above; window <= 0
 * means no window (decodeGQA).  L == 0 gives an all-zero row (an empty sum).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,          /* a size or pointer argument is invalid       */
  ORACLE_ERR_SEQ_LEN = 2,      /* seq_lens[b] < 0 or beyond the block table    */
  ORACLE_ERR_UNMAPPED = 3,     /* a visible position maps to a page id outside [0, num_pages) */
  ORACLE_ERR_NOMEM = 4
};

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t* q;
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t B, Hq, Hkv, D, page_size, max_blocks;
  int64_t num_pages;
  int32_t window;
  const int32_t* rows; /* flat b*Hq+h indices (t*Hq+h for prefill), or NULL for all rows */
  int32_t n_rows;
  const int32_t* cu_q; /* prefill: [B+1] query-row offsets; NULL for decode */
  int32_t T;           /* prefill: cu_q[B], the number of query rows */
  double* out;         /* [n_rows, D] */
  int32_t n_threads;
  int32_t thread_id;
  int status;
} job_t;

/* Index of pool row (token slot) for logical position l of sequence b, or -1. */
static int64_t pool_row(const job_t* j, int b, int l) {
  int page = l / j->page_size;
  if (page >= j->max_blocks) return -1;
  int64_t phys = j->block_table[(int64_t)b * j->max_blocks + page];
  if (phys < 0 || phys >= j->num_pages) return -1;
  return phys * j->page_size + (l % j->page_size);
}

/* The output row of query vector qv (head h) of sequence b sitting at
 * position L-1, over the cached positions l <= L-1 (decodeGQA, or
 * slidingGQA at p = L-1).  L <= seq_lens[b] has been checked by the caller. */
static int attend_one_row(const job_t* j, int b, int h, const uint16_t* qv, int L, double* o, double* logit) {
  const int G = j->Hq / j->Hkv;
  const int c = h / G;               /* query head c*G+g reads KV head c */
  const int D = j->D;

  /* visible positions: p - window < l <= p with p = L-1 (no lower bound when window <= 0) */
  int lo = 0;
  if (j->window > 0 && L > j->window) lo = L - j->window;
  const int n = L - lo;

  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (n <= 0) return ORACLE_OK;

  /* logits s_l = 1 * sum_e q[e] * k[l,c,e]  (scale 1) */
  double m = -INFINITY;
  for (int l = lo; l < L; ++l) {
    int64_t r = pool_row(j, b, l);
    if (r < 0) return ORACLE_ERR_UNMAPPED;
    const uint16_t* kv = j->k_pool + (r * j->Hkv + c) * D;
    double s = 0.0;
    for (int e = 0; e < D; ++e) s += bf16_bits_to_double(qv[e]) * bf16_bits_to_double(kv[e]);
    logit[l - lo] = s;
    if (s > m) m = s;
  }

  /* softmax over the visible set: w_l = exp(s_l - m), Z = sum w_l */
  double Z = 0.0;
  for (int i = 0; i < n; ++i) {
    logit[i] = exp(logit[i] - m);
    Z += logit[i];
  }

  /* o[d] = sum_l w_l * v[l,c,d] / Z */
  for (int l = lo; l < L; ++l) {
    int64_t r = pool_row(j, b, l);
    const uint16_t* vv = j->v_pool + (r * j->Hkv + c) * D;
    const double w = logit[l - lo];
    for (int d = 0; d < D; ++d) o[d] += w * bf16_bits_to_double(vv[d]);
  }
  for (int d = 0; d < D; ++d) o[d] /= Z;
  return ORACLE_OK;
}

/* One output row o[b,h,:] (decodeGQA / slidingGQA at position L-1). */
static int decode_one_row(const job_t* j, int b, int h, double* o, double* logit) {
  const int L = j->seq_lens[b];
  if (L < 0 || (int64_t)L > (int64_t)j->max_blocks * j->page_size) return ORACLE_ERR_SEQ_LEN;
  return attend_one_row(j, b, h, j->q + ((int64_t)b * j->Hq + h) * j->D, L, o, logit);
}

/* One prefill output row o[t,h,:]: query row t belongs to the sequence b with
 * cu_q[b] <= t < cu_q[b+1]; its n = cu_q[b+1] - cu_q[b] queries are the last
 * n tokens of the L = seq_lens[b] cached ones, so query i = t - cu_q[b] sits
 * at position p = L - n + i (causalGQA / slidingGQA with that pos), which is
 * the decode of the sequence cut to its first p + 1 tokens. */
static int prefill_one_row(const job_t* j, int t, int h, double* o, double* logit) {
  int lo = 0, hi = j->B; /* largest b with cu_q[b] <= t */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (j->cu_q[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int n = j->cu_q[b + 1] - j->cu_q[b];
  const int L = j->seq_lens[b];
  if (L < n || (int64_t)L > (int64_t)j->max_blocks * j->page_size) return ORACLE_ERR_SEQ_LEN;
  const int p = L - n + (t - j->cu_q[b]);
  return attend_one_row(j, b, h, j->q + ((int64_t)t * j->Hq + h) * j->D, p + 1, o, logit);
}

static void* worker(void* arg) {
  job_t* j = (job_t*)arg;
  int max_L = 0;
  for (int b = 0; b < j->B; ++b)
    if (j->seq_lens[b] > max_L) max_L = j->seq_lens[b];
  double* logit = (double*)malloc(sizeof(double) * (size_t)(max_L > 0 ? max_L : 1));
  if (!logit) {
    j->status = ORACLE_ERR_NOMEM;
    return NULL;
  }
  const int total = j->rows ? j->n_rows : (j->cu_q ? j->T : j->B) * j->Hq;
  for (int i = j->thread_id; i < total; i += j->n_threads) {
    const int flat = j->rows ? j->rows[i] : i;
    const int b = flat / j->Hq, h = flat % j->Hq; /* b is the query row t for prefill */
    int st = j->cu_q ? prefill_one_row(j, b, h, j->out + (int64_t)i * j->D, logit)
                     : decode_one_row(j, b, h, j->out + (int64_t)i * j->D, logit);
    if (st != ORACLE_OK && j->status == ORACLE_OK) j->status = st;
  }
  free(logit);
  return NULL;
}

/*
 * Paged decode attention, fp64.
 *
 * q           bf16 bits [B, Hq, D]
 * k_pool      bf16 bits [num_pages, page_size, Hkv, D]
 * v_pool      bf16 bits [num_pages, page_size, Hkv, D]
 * block_table int32 [B, max_blocks]; entries of pages that hold no visible
 *             position are never read (they may be -1)
 * seq_lens    int32 [B], 0 <= L <= max_blocks*page_size
 * window      > 0: sliding window; <= 0: none
 * rows        NULL for every (b, h) row in b-major order, else n_rows flat
 *             indices b*Hq + h to compute
 * out         double [n_rows (or B*Hq), D]
 * n_threads   worker threads (>= 1); rows are striped over them
 * returns     ORACLE_OK or an ORACLE_ERR_* code
 */
static int run_jobs(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                    const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q, int32_t T,
                    int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size, int32_t max_blocks,
                    int64_t num_pages, int32_t window, const int32_t* rows, int32_t n_rows, double* out,
                    int32_t n_threads) {
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out) return ORACLE_ERR_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || page_size < 1 || max_blocks < 1 || num_pages < 1)
    return ORACLE_ERR_ARG;
  if (Hq % Hkv != 0) return ORACLE_ERR_ARG;
  const int n_out = cu_q ? T : B; /* output rows per head */
  if (rows) {
    if (n_rows < 0) return ORACLE_ERR_ARG;
    for (int i = 0; i < n_rows; ++i)
      if (rows[i] < 0 || rows[i] >= n_out * Hq) return ORACLE_ERR_ARG;
  }
  if (n_threads < 1) n_threads = 1;

  job_t* jobs = (job_t*)calloc((size_t)n_threads, sizeof(job_t));
  pthread_t* tids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return ORACLE_ERR_NOMEM;
  }
  for (int t = 0; t < n_threads; ++t) {
    job_t* j = &jobs[t];
    j->q = q; j->k_pool = k_pool; j->v_pool = v_pool;
    j->block_table = block_table; j->seq_lens = seq_lens;
    j->B = B; j->Hq = Hq; j->Hkv = Hkv; j->D = D; j->page_size = page_size;
    j->max_blocks = max_blocks; j->num_pages = num_pages; j->window = window;
    j->rows = rows; j->n_rows = n_rows; j->out = out;
    j->cu_q = cu_q; j->T = T;
    j->n_threads = n_threads; j->thread_id = t; j->status = ORACLE_OK;
  }
  int status = ORACLE_OK;
  if (n_threads == 1) {
    worker(&jobs[0]);
  } else {
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
      if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) break;
      ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    /* rows of threads that never started are computed here */
    for (int t = started; t < n_threads; ++t) worker(&jobs[t]);
  }
  for (int t = 0; t < n_threads; ++t)
    if (jobs[t].status != ORACLE_OK && status == ORACLE_OK) status = jobs[t].status;
  free(jobs);
  free(tids);
  return status;
}

int oracle_decode_paged(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                        const int32_t* block_table, const int32_t* seq_lens, int32_t B,
                        int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                        int32_t max_blocks, int64_t num_pages, int32_t window,
                        const int32_t* rows, int32_t n_rows, double* out, int32_t n_threads) {
  return run_jobs(q, k_pool, v_pool, block_table, seq_lens, NULL, 0, B, Hq, Hkv, D, page_size, max_blocks,
                  num_pages, window, rows, n_rows, out, n_threads);
}

/*
 * Multi-query attention over the paged cache (prefill of a chunk of new
 * tokens whose keys and values are already in the cache), fp64.
 *
 * Attention.lean, `causalGQA` and `slidingGQA` with S > 1: query s at
 * position pos s sees key l iff l <= pos s (and pos s < l + window).  Here
 * sequence b holds L = seq_lens[b] cached tokens and n = cu_q[b+1] - cu_q[b]
 * queries, the last n tokens: query i (packed row cu_q[b] + i) sits at
 * position L - n + i.  Query row s of causalGQA depends on pos s alone, so it
 * equals decodeGQA over the first pos s + 1 tokens; that is how each row is
 * computed.
 *
 * q           bf16 bits [T, Hq, D], T = cu_q[B], rows packed sequence by sequence
 * cu_q        int32 [B+1], cu_q[0] = 0, non-decreasing; n <= L for every sequence
 * rows        NULL for every (t, h) row in t-major order, else n_rows flat
 *             indices t*Hq + h
 * out         double [n_rows (or T*Hq), D]
 * the rest as for oracle_decode_paged
 */
int oracle_prefill_paged(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                         const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                         int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size, int32_t max_blocks,
                         int64_t num_pages, int32_t window, const int32_t* rows, int32_t n_rows, double* out,
                         int32_t n_threads) {
  if (!cu_q || B < 1 || cu_q[0] != 0) return ORACLE_ERR_ARG;
  for (int b = 0; b < B; ++b)
    if (cu_q[b + 1] < cu_q[b]) return ORACLE_ERR_ARG;
  return run_jobs(q, k_pool, v_pool, block_table, seq_lens, cu_q, cu_q[B], B, Hq, Hkv, D, page_size, max_blocks,
                  num_pages, window, rows, n_rows, out, n_threads);
}

/* ------------------------------------------------------------------------ */
/*
 * The steps that feed attn.core for one new token per sequence: per-head
 * norms, RoPE, and the append of the token's key and value to the paged
 * cache.  Gemma-4-12B model page, "Compute-graph nodes":
 *
 *   attn.qk_norm  rmsnorm, per head:  y[i] = x[i] / sqrt(sum_j x[j]^2 / D + eps) * w[i]
 *   attn.v_norm   rmsnormUnit, per head:  y[i] = x[i] / sqrt(sum_j x[j]^2 / D + eps)
 *   attn.rope     rotate pairs (i, i + D/2) by pos * theta^(-2i/D), i < active;
 *                 the other coordinates are unchanged
 *   ("What to watch for": sliding layers theta 10,000 with all 128 pairs of
 *   D = 256 active; global layers theta 1,000,000 with the first 64 of the
 *   256 pairs of D = 512 active, and values = keys.)
 *
 * The qkv row of token b (the attn.qkv_proj output) is [q: Hq*D | k: Hkv*D |
 * v: Hkv*D], or with shared_kv [q: Hq*D | x: D], whose one head x gives both
 * the key (qk_norm, RoPE) and the value (v_norm).  Rotating (a, b) by phi is
 * (a cos phi - b sin phi, b cos phi + a sin phi).  The token sits at position
 * pos = positions[b]: its key and value go to page block_table[b, pos/16],
 * slot pos % 16; q leaves normed and rotated.  Everything is computed in
 * double from the exact bf16 inputs and rounded once to bf16 (nearest, ties
 * to even).
 */

/* double -> bf16 bits, round to nearest, ties to even (finite, normal range). */
static uint16_t double_to_bf16_rne(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000u : 0;
  int e;
  const double m = frexp(x, &e);          /* x = m * 2^e, 0.5 <= |m| < 1 */
  const double r = nearbyint(ldexp(m, 8)); /* 8 significant bits, ties to even */
  const float f = (float)ldexp(r, e - 8);  /* exact in binary32 */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* y = x / rms(x) (* w when w != NULL), x and w bf16 bits, D values. */
static void rms_norm(const uint16_t* x, const uint16_t* w, int D, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < D; ++i) {
    const double v = bf16_bits_to_double(x[i]);
    ss += v * v;
  }
  const double inv = 1.0 / sqrt(ss / D + eps);
  for (int i = 0; i < D; ++i) y[i] = bf16_bits_to_double(x[i]) * inv * (w ? bf16_bits_to_double(w[i]) : 1.0);
}

/* Rotate pairs (i, i + D/2), i < pairs, by pos * theta^(-2i/D). */
static void rope(double* y, int D, int pairs, double theta, int pos) {
  const int half = D / 2;
  for (int i = 0; i < pairs; ++i) {
    const double phi = (double)pos * pow(theta, -2.0 * i / D);
    const double c = cos(phi), s = sin(phi);
    const double a = y[i], b = y[i + half];
    y[i] = a * c - b * s;
    y[i + half] = b * c + a * s;
  }
}

/*
 * qkv         bf16 bits [B, Hq*D + (shared_kv ? D : 2*Hkv*D)]
 * w_q, w_k    bf16 bits [D]: the qk_norm weights of q and k
 * block_table int32 [B, max_blocks]; positions int32 [B]
 * q_out       bf16 bits [B, Hq, D] (written)
 * k_pool      bf16 bits [num_pages, page_size, Hkv, D] (the token's slot written)
 * v_pool      likewise
 * returns     ORACLE_OK, ORACLE_ERR_ARG, ORACLE_ERR_SEQ_LEN (a position
 *             beyond the block table) or ORACLE_ERR_UNMAPPED (its page id
 *             outside [0, num_pages)); nothing is written for that sequence
 */
int oracle_qkv_append(const uint16_t* qkv, const uint16_t* w_q, const uint16_t* w_k,
                      const int32_t* block_table, const int32_t* positions, int32_t B, int32_t Hq,
                      int32_t Hkv, int32_t D, int32_t shared_kv, int32_t page_size, int32_t max_blocks,
                      int64_t num_pages, double theta, int32_t rope_pairs, double eps, uint16_t* q_out,
                      uint16_t* k_pool, uint16_t* v_pool) {
  if (!qkv || !w_q || !w_k || !block_table || !positions || !q_out || !k_pool || !v_pool) return ORACLE_ERR_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 2 || (D & 1) || page_size < 1 || max_blocks < 1 || num_pages < 1)
    return ORACLE_ERR_ARG;
  if (rope_pairs < 0 || rope_pairs > D / 2 || (shared_kv && Hkv != 1)) return ORACLE_ERR_ARG;
  const int64_t row_len = (int64_t)Hq * D + (shared_kv ? D : 2 * (int64_t)Hkv * D);
  double* y = (double*)malloc(sizeof(double) * (size_t)D);
  if (!y) return ORACLE_ERR_NOMEM;
  int status = ORACLE_OK;
  for (int b = 0; b < B; ++b) {
    const uint16_t* row = qkv + (int64_t)b * row_len;
    const int pos = positions[b];
    const int page = pos >= 0 ? pos / page_size : -1;
    if (pos < 0 || page >= max_blocks) {
      if (status == ORACLE_OK) status = ORACLE_ERR_SEQ_LEN;
      continue;
    }
    const int64_t phys = block_table[(int64_t)b * max_blocks + page];
    if (phys < 0 || phys >= num_pages) {
      if (status == ORACLE_OK) status = ORACLE_ERR_UNMAPPED;
      continue;
    }
    const int64_t slot = phys * page_size + pos % page_size;
    for (int h = 0; h < Hq; ++h) {
      rms_norm(row + (int64_t)h * D, w_q, D, eps, y);
      rope(y, D, rope_pairs, theta, pos);
      for (int i = 0; i < D; ++i) q_out[((int64_t)b * Hq + h) * D + i] = double_to_bf16_rne(y[i]);
    }
    for (int c = 0; c < Hkv; ++c) {
      const uint16_t* xk = row + (int64_t)Hq * D + (shared_kv ? 0 : (int64_t)c * D);
      const uint16_t* xv = row + (int64_t)Hq * D + (shared_kv ? 0 : ((int64_t)Hkv + c) * D);
      uint16_t* kd = k_pool + (slot * Hkv + c) * D;
      uint16_t* vd = v_pool + (slot * Hkv + c) * D;
      rms_norm(xk, w_k, D, eps, y);
      rope(y, D, rope_pairs, theta, pos);
      for (int i = 0; i < D; ++i) kd[i] = double_to_bf16_rne(y[i]);
      rms_norm(xv, NULL, D, eps, y);
      for (int i = 0; i < D; ++i) vd[i] = double_to_bf16_rne(y[i]);
    }
  }
  free(y);
  return status;
}

/* ------------------------------------------------------------------------ */
/*
 * The keys of a global-layer cache that stores values only.  With "values =
 * keys" (Gemma-4-12B model page, "What to watch for": attention_k_eq_v) one
 * head x gives both, V = rmsnormUnit(x) and K = rope(rmsnorm(x) * w_k), so
 * K = rope(V * w_k): a cache holding V can rebuild K.  Reading: the rebuilt
 * key is V * w_k rotated as attn.rope rotates it at the key's position,
 * computed in double from the stored bf16 V and w_k and rounded once to bf16
 * (the precision keys have in a cache that stores them).
 *
 * v_pool      bf16 bits [num_pages, page_size, Hkv, D]
 * w_k         bf16 bits [D]
 * block_table int32 [B, max_blocks]; seq_lens int32 [B]; window as for
 *             oracle_decode_paged: only the visible positions are rebuilt
 * k_out       bf16 bits, same shape as v_pool: the slot of every visible
 *             position is written, every other slot is left as it is
 */
int oracle_rebuild_keys(const uint16_t* v_pool, const uint16_t* w_k, const int32_t* block_table,
                        const int32_t* seq_lens, int32_t B, int32_t Hkv, int32_t D, int32_t page_size,
                        int32_t max_blocks, int64_t num_pages, int32_t window, double theta, int32_t rope_pairs,
                        uint16_t* k_out) {
  if (!v_pool || !w_k || !block_table || !seq_lens || !k_out) return ORACLE_ERR_ARG;
  if (B < 1 || Hkv < 1 || D < 2 || (D & 1) || page_size < 1 || max_blocks < 1 || num_pages < 1)
    return ORACLE_ERR_ARG;
  if (rope_pairs < 0 || rope_pairs > D / 2) return ORACLE_ERR_ARG;
  double* y = (double*)malloc(sizeof(double) * (size_t)D);
  if (!y) return ORACLE_ERR_NOMEM;
  int status = ORACLE_OK;
  for (int b = 0; b < B && status == ORACLE_OK; ++b) {
    const int L = seq_lens[b];
    if (L < 0 || (int64_t)L > (int64_t)max_blocks * page_size) {
      status = ORACLE_ERR_SEQ_LEN;
      break;
    }
    const int lo = (window > 0 && L > window) ? L - window : 0;
    for (int l = lo; l < L; ++l) {
      const int64_t phys = block_table[(int64_t)b * max_blocks + l / page_size];
      if (phys < 0 || phys >= num_pages) {
        status = ORACLE_ERR_UNMAPPED;
        break;
      }
      const int64_t slot = phys * page_size + l % page_size;
      for (int c = 0; c < Hkv; ++c) {
        const uint16_t* v = v_pool + (slot * Hkv + c) * D;
        for (int i = 0; i < D; ++i) y[i] = bf16_bits_to_double(v[i]) * bf16_bits_to_double(w_k[i]);
        rope(y, D, rope_pairs, theta, l);
        for (int i = 0; i < D; ++i) k_out[(slot * Hkv + c) * D + i] = double_to_bf16_rne(y[i]);
      }
    }
  }
  free(y);
  return status;
}
