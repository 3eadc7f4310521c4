/*
 * pkv_oracle.c -- plain fp64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
 * benchmark's CPU-baseline leg are the only code that may load this file's
 * shared object. The GPU library neither links it nor shares any code,
 * header or constant with it.
 *
 * What it computes, and the passages it follows:
 *
 *  - KV append: each new token's key and value rows are written into the page
 *    slot named by its slot index. The KV cache is paged and grows as decoding
 *    proceeds ("FunASR vLLM Inference Engine Guide", section 2 "vLLM Engine
 *    Architecture", table "Why vLLM?": PagedAttention, on-demand allocation;
 *    "Optimizing ASR for 90-minute multi-speaker audio", section "LLM
 *    prefill": the prompt builds the KV cache that decoding extends).
 *
 *  - Decode attention: one query row per request and query head attends over
 *    every cached position of that request, read through its block table
 *    (same guide, section 2, "PagedAttention + Continuous Batching"). Grouped
 *    query attention with 16 query heads over 8 KV heads ("Fun-ASR-Nano
 *    Native Runtime Design", section "Decoder And Prompt").
 *
 *  - Chunked-prefill attention: a chunk of query rows of one request attends
 *    causally over the request's cached prefix plus the chunk itself; row i of
 *    a chunk that follows P cached tokens sits at absolute position P + i
 *    ("Optimizing ASR for 90-minute multi-speaker audio", section "Chunked
 *    prefill for long audio": 4096-token chunks interleaved with decode).
 *
 *  - Rotary position embedding of the new token's query and key rows, the
 *    step that precedes decode attention in a Qwen3-style decoder with RoPE
 *    theta 1e6 ("Fun-ASR-Nano Native Runtime Design", section "Decoder And
 *    Prompt"). The pages name RoPE and theta only; the rotate-half form of
 *    Qwen3 decoders is taken: dims i and i + head_dim/2 form a pair rotated by
 *    angle pos * theta^(-2i/head_dim).
 *
 * Readings taken where the pages are silent (no page gives a kernel, a page
 * layout or a page size):
 *  - pool layout [num_pages][n_kv_heads][page_size][head_dim], K and V in
 *    separate pools; logical position j of a request lives in page
 *    block_table[j / page_size] at slot j % page_size;
 *  - query head h reads KV head h / (n_q_heads / n_kv_heads);
 *  - plain softmax attention with an explicit scale, no soft-cap, no window;
 *  - a request with zero cached positions yields an all-zero output row;
 *  - bf16 inputs are widened exactly to double; all arithmetic is double,
 *    except where a result is stored as bf16 (a rotated key row written into
 *    the cache): that rotation is evaluated in float with the operation order
 *    stated at pkvo_rope_bf16 and rounded to nearest even, the precision in
 *    which the GPU kernel takes the same rounding decision (the pages fix none);
 *  - the cos/sin table is an input (double angles, rounded to float), as
 *    serving engines precompute it once.
 *
 * The softmax is evaluated as its definition with the maximum subtracted
 * (exp(s_j - m) / sum_k exp(s_k - m) equals exp(s_j) / sum_k exp(s_k)
 * exactly in real arithmetic). Scores are summed over positions in logical
 * order, so the result does not depend on where pages sit in the pool.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PKVO_OK 0
#define PKVO_ERR_ARG (-1)
#define PKVO_ERR_RANGE (-2)
#define PKVO_ERR_NOMEM (-3)

typedef struct {
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int64_t num_pages;
} pkvo_geom;

/* Exact widening of a bf16 bit pattern: bf16 is the top 16 bits of a float. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Element offset of row (page, kv_head, slot) in a pool. */
static int64_t pool_row(const pkvo_geom* g, int64_t page, int32_t kv_head, int32_t slot) {
  return ((page * g->n_kv_heads + kv_head) * (int64_t)g->page_size + slot) * g->head_dim;
}

/*
 * Attention of one query row over logical positions 0 .. n_keys-1 of one
 * request, KV head kv_head. `scores` has room for n_keys doubles.
 * Returns PKVO_ERR_RANGE if the block table names a page outside the pool.
 */
static int attend_row(const pkvo_geom* g, const double* q_row, const uint16_t* k_pages,
                      const uint16_t* v_pages, const int32_t* bt_row, int64_t n_keys,
                      int32_t kv_head, double scale, double* scores, double* out) {
  const int32_t D = g->head_dim;
  for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
  if (n_keys <= 0) return PKVO_OK;

  /* s_j = scale * <q, k_j> */
  for (int64_t j = 0; j < n_keys; ++j) {
    int64_t page = bt_row[j / g->page_size];
    int32_t slot = (int32_t)(j % g->page_size);
    if (page < 0 || page >= g->num_pages) return PKVO_ERR_RANGE;
    const uint16_t* k = k_pages + pool_row(g, page, kv_head, slot);
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d) dot += q_row[d] * bf16_bits_to_double(k[d]);
    scores[j] = scale * dot;
  }

  /* softmax weights w_j = exp(s_j - m) / Z */
  double m = scores[0];
  for (int64_t j = 1; j < n_keys; ++j)
    if (scores[j] > m) m = scores[j];
  double z = 0.0;
  for (int64_t j = 0; j < n_keys; ++j) {
    scores[j] = exp(scores[j] - m);
    z += scores[j];
  }

  /* out = sum_j w_j v_j */
  for (int64_t j = 0; j < n_keys; ++j) {
    int64_t page = bt_row[j / g->page_size];
    int32_t slot = (int32_t)(j % g->page_size);
    const uint16_t* v = v_pages + pool_row(g, page, kv_head, slot);
    double w = scores[j] / z;
    for (int32_t d = 0; d < D; ++d) out[d] += w * bf16_bits_to_double(v[d]);
  }
  return PKVO_OK;
}

static int geom_ok(const pkvo_geom* g) {
  return g && g->n_q_heads > 0 && g->n_kv_heads > 0 && g->head_dim > 0 && g->page_size > 0 &&
         g->num_pages >= 0 && (g->n_q_heads % g->n_kv_heads) == 0;
}

/* ------------------------------------------------------------------------ */
/* KV append                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * k_new, v_new: [n_tokens][n_kv_heads][head_dim] bf16 bits.
 * slot_mapping: [n_tokens]; slot s names page s / page_size, slot s % page_size;
 *               a negative slot skips that token.
 * k_pages, v_pages: pools, updated in place.
 */
int pkvo_append(const pkvo_geom* g, const uint16_t* k_new, const uint16_t* v_new,
                const int32_t* slot_mapping, int64_t n_tokens, uint16_t* k_pages, uint16_t* v_pages) {
  if (!geom_ok(g) || n_tokens < 0) return PKVO_ERR_ARG;
  const int32_t D = g->head_dim;
  for (int64_t t = 0; t < n_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    int64_t page = s / g->page_size;
    int32_t slot = (int32_t)(s % g->page_size);
    if (page >= g->num_pages) return PKVO_ERR_RANGE;
    for (int32_t h = 0; h < g->n_kv_heads; ++h) {
      const uint16_t* ks = k_new + (t * g->n_kv_heads + h) * D;
      const uint16_t* vs = v_new + (t * g->n_kv_heads + h) * D;
      memcpy(k_pages + pool_row(g, page, h, slot), ks, sizeof(uint16_t) * (size_t)D);
      memcpy(v_pages + pool_row(g, page, h, slot), vs, sizeof(uint16_t) * (size_t)D);
    }
  }
  return PKVO_OK;
}

/* ------------------------------------------------------------------------ */
/* Work items shared by the threaded drivers                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
  const pkvo_geom* g;
  const uint16_t* q;      /* [rows][n_q_heads][head_dim] bf16 bits, or NULL when q64 is given */
  const double* q64;      /* [rows][n_q_heads][head_dim] double */
  const uint16_t* k_pages;
  const uint16_t* v_pages;
  const int32_t* block_table;
  int64_t bt_stride;      /* entries per block-table row */
  const int32_t* row_seq;   /* request of each query row */
  const int64_t* row_keys;  /* number of visible keys of each query row */
  const int64_t* row_index; /* row of q to read for each output row */
  int64_t n_rows;
  int64_t max_keys;
  double scale;
  double* out;            /* [n_rows][n_q_heads][head_dim] */
  int64_t next;           /* shared work counter */
  pthread_mutex_t lock;
  int status;
} job_t;

static int64_t take_item(job_t* job) {
  pthread_mutex_lock(&job->lock);
  int64_t it = job->next++;
  pthread_mutex_unlock(&job->lock);
  return it;
}

static void* worker(void* arg) {
  job_t* job = (job_t*)arg;
  const pkvo_geom* g = job->g;
  const int32_t group = g->n_q_heads / g->n_kv_heads;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(job->max_keys > 0 ? job->max_keys : 1));
  double* qbuf = (double*)malloc(sizeof(double) * (size_t)g->head_dim);
  if (!scores || !qbuf) {
    free(scores);
    free(qbuf);
    pthread_mutex_lock(&job->lock);
    job->status = PKVO_ERR_NOMEM;
    pthread_mutex_unlock(&job->lock);
    return NULL;
  }
  const int64_t n_items = job->n_rows * g->n_q_heads;
  for (;;) {
    int64_t it = take_item(job);
    if (it >= n_items) break;
    int64_t r = it / g->n_q_heads;
    int32_t h = (int32_t)(it % g->n_q_heads);
    const int64_t q_off = (job->row_index[r] * g->n_q_heads + h) * g->head_dim;
    const double* q_row = job->q64 ? job->q64 + q_off : qbuf;
    if (!job->q64)
      for (int32_t d = 0; d < g->head_dim; ++d) qbuf[d] = bf16_bits_to_double(job->q[q_off + d]);
    const int32_t* bt_row = job->block_table + (int64_t)job->row_seq[r] * job->bt_stride;
    double* o = job->out + (r * g->n_q_heads + h) * g->head_dim;
    int rc = attend_row(g, q_row, job->k_pages, job->v_pages, bt_row, job->row_keys[r], h / group,
                        job->scale, scores, o);
    if (rc != PKVO_OK) {
      pthread_mutex_lock(&job->lock);
      job->status = rc;
      pthread_mutex_unlock(&job->lock);
    }
  }
  free(scores);
  free(qbuf);
  return NULL;
}

static int run_job(job_t* job, int n_threads) {
  if (n_threads < 1) n_threads = 1;
  job->next = 0;
  job->status = PKVO_OK;
  pthread_mutex_init(&job->lock, NULL);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  if (!th) return PKVO_ERR_NOMEM;
  int started = 0;
  for (int i = 0; i < n_threads; ++i) {
    if (pthread_create(&th[i], NULL, worker, job) != 0) break;
    ++started;
  }
  if (started == 0) worker(job);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&job->lock);
  return job->status;
}

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

/*
 * q: [batch][n_q_heads][head_dim] bf16 bits.
 * block_table: [batch][max_pages] page ids; seq_lens: [batch] visible keys.
 * out: [batch][n_q_heads][head_dim] double.
 */
static int decode_rows(const pkvo_geom* g, const uint16_t* q, const double* q64, const uint16_t* k_pages,
                       const uint16_t* v_pages, const int32_t* block_table, const int32_t* seq_lens, int64_t batch,
                       int64_t max_pages, double scale, double* out, int n_threads) {
  if (!geom_ok(g) || batch < 0 || max_pages < 0) return PKVO_ERR_ARG;
  int32_t* row_seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(batch + 1));
  int64_t* row_keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(batch + 1));
  int64_t* row_index = (int64_t*)malloc(sizeof(int64_t) * (size_t)(batch + 1));
  if (!row_seq || !row_keys || !row_index) {
    free(row_seq); free(row_keys); free(row_index);
    return PKVO_ERR_NOMEM;
  }
  int64_t max_keys = 1;
  int rc = PKVO_OK;
  for (int64_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > max_pages * g->page_size) rc = PKVO_ERR_RANGE;
    row_seq[b] = (int32_t)b;
    row_keys[b] = seq_lens[b];
    row_index[b] = b;
    if (row_keys[b] > max_keys) max_keys = row_keys[b];
  }
  if (rc == PKVO_OK) {
    job_t job;
    memset(&job, 0, sizeof job);
    job.g = g; job.q = q; job.q64 = q64; job.k_pages = k_pages; job.v_pages = v_pages;
    job.block_table = block_table; job.bt_stride = max_pages;
    job.row_seq = row_seq; job.row_keys = row_keys; job.row_index = row_index;
    job.n_rows = batch; job.max_keys = max_keys; job.scale = scale; job.out = out;
    rc = run_job(&job, n_threads);
  }
  free(row_seq); free(row_keys); free(row_index);
  return rc;
}

int pkvo_decode(const pkvo_geom* g, const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                const int32_t* block_table, const int32_t* seq_lens, int64_t batch, int64_t max_pages,
                double scale, double* out, int n_threads) {
  if (!q) return PKVO_ERR_ARG;
  return decode_rows(g, q, NULL, k_pages, v_pages, block_table, seq_lens, batch, max_pages, scale, out, n_threads);
}

/* Same, with the query rows given as doubles (e.g. after the rotation below). */
int pkvo_decode_q64(const pkvo_geom* g, const double* q64, const uint16_t* k_pages, const uint16_t* v_pages,
                    const int32_t* block_table, const int32_t* seq_lens, int64_t batch, int64_t max_pages,
                    double scale, double* out, int n_threads) {
  if (!q64) return PKVO_ERR_ARG;
  return decode_rows(g, NULL, q64, k_pages, v_pages, block_table, seq_lens, batch, max_pages, scale, out,
                     n_threads);
}

/* ------------------------------------------------------------------------ */
/* Rotary position embedding (rotate-half form)                              */
/* ------------------------------------------------------------------------ */

/*
 * cache: [max_pos][head_dim] float; row p holds cos(p w_i) for i < head_dim/2,
 * then sin(p w_i), with w_i = theta^(-2 i / head_dim). Angles and their cosine
 * and sine are evaluated in double and rounded to float once.
 */
int pkvo_rope_cache(double theta, int32_t head_dim, int64_t max_pos, float* cache) {
  if (theta <= 0.0 || head_dim <= 0 || (head_dim % 2) != 0 || max_pos < 0 || !cache) return PKVO_ERR_ARG;
  const int32_t half = head_dim / 2;
  for (int64_t p = 0; p < max_pos; ++p)
    for (int32_t i = 0; i < half; ++i) {
      const double w = pow(theta, -2.0 * (double)i / (double)head_dim);
      const double ang = (double)p * w;
      cache[p * head_dim + i] = (float)cos(ang);
      cache[p * head_dim + half + i] = (float)sin(ang);
    }
  return PKVO_OK;
}

/* Round a float to the nearest bf16, ties to even (finite inputs). */
static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float bf16_bits_to_float(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/*
 * Rotation of rows x [n_rows][n_heads][head_dim] (bf16 bits); row r at
 * position pos[r] (pos[r] < 0: the row is copied unrotated). For each pair
 * (x1, x2) = (x[i], x[i + head_dim/2]) with c, s = cache[pos][i], cache[pos][half + i]:
 *   y1 = x1 c - x2 s,   y2 = x2 c + x1 s.
 * pkvo_rope_f64 evaluates this in double. pkvo_rope_bf16 evaluates it in
 * float as y1 = fmaf(x1, c, -(x2 * s)), y2 = fmaf(x2, c, x1 * s) (each product
 * rounded to float, then one fused multiply-add) and rounds to bf16, ties to even.
 */
static int rope_args_ok(int64_t n_rows, int32_t n_heads, int32_t head_dim, const int32_t* pos, int64_t max_pos) {
  if (n_rows < 0 || n_heads <= 0 || head_dim <= 0 || (head_dim % 2) != 0 || !pos) return 0;
  for (int64_t r = 0; r < n_rows; ++r)
    if (pos[r] >= max_pos) return 0;
  return 1;
}

int pkvo_rope_f64(const uint16_t* x, int64_t n_rows, int32_t n_heads, int32_t head_dim, const int32_t* pos,
                  const float* cache, int64_t max_pos, double* out) {
  if (!rope_args_ok(n_rows, n_heads, head_dim, pos, max_pos)) return PKVO_ERR_ARG;
  const int32_t half = head_dim / 2;
  for (int64_t r = 0; r < n_rows; ++r)
    for (int32_t h = 0; h < n_heads; ++h) {
      const uint16_t* xr = x + (r * n_heads + h) * head_dim;
      double* o = out + (r * n_heads + h) * head_dim;
      for (int32_t i = 0; i < half; ++i) {
        const double x1 = bf16_bits_to_double(xr[i]), x2 = bf16_bits_to_double(xr[half + i]);
        if (pos[r] < 0) {
          o[i] = x1;
          o[half + i] = x2;
          continue;
        }
        const double c = (double)cache[(int64_t)pos[r] * head_dim + i];
        const double s = (double)cache[(int64_t)pos[r] * head_dim + half + i];
        o[i] = x1 * c - x2 * s;
        o[half + i] = x2 * c + x1 * s;
      }
    }
  return PKVO_OK;
}

int pkvo_rope_bf16(const uint16_t* x, int64_t n_rows, int32_t n_heads, int32_t head_dim, const int32_t* pos,
                   const float* cache, int64_t max_pos, uint16_t* out) {
  if (!rope_args_ok(n_rows, n_heads, head_dim, pos, max_pos)) return PKVO_ERR_ARG;
  const int32_t half = head_dim / 2;
  for (int64_t r = 0; r < n_rows; ++r)
    for (int32_t h = 0; h < n_heads; ++h) {
      const uint16_t* xr = x + (r * n_heads + h) * head_dim;
      uint16_t* o = out + (r * n_heads + h) * head_dim;
      for (int32_t i = 0; i < half; ++i) {
        if (pos[r] < 0) {
          o[i] = xr[i];
          o[half + i] = xr[half + i];
          continue;
        }
        const float x1 = bf16_bits_to_float(xr[i]), x2 = bf16_bits_to_float(xr[half + i]);
        const float c = cache[(int64_t)pos[r] * head_dim + i];
        const float s = cache[(int64_t)pos[r] * head_dim + half + i];
        const float p2 = x2 * s, p1 = x1 * s;
        o[i] = float_to_bf16_rne(fmaf(x1, c, -p2));
        o[half + i] = float_to_bf16_rne(fmaf(x2, c, p1));
      }
    }
  return PKVO_OK;
}

/* ------------------------------------------------------------------------ */
/* Chunked-prefill attention                                                 */
/* ------------------------------------------------------------------------ */

/*
 * q: [total_q][n_q_heads][head_dim] bf16 bits, the chunks of num_seqs requests
 *    packed back to back; request n owns rows cu_q_lens[n] .. cu_q_lens[n+1]-1.
 * prefix_lens: [num_seqs] tokens cached before each chunk. The chunk's own K/V
 *    are already in the pool at positions prefix .. prefix + q_len - 1.
 * rows: the global query rows to evaluate (n_rows of them); NULL = all rows.
 * out: [n_rows][n_q_heads][head_dim] double.
 */
int pkvo_prefill(const pkvo_geom* g, const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                 const int32_t* block_table, int64_t max_pages, const int32_t* prefix_lens,
                 const int32_t* cu_q_lens, int64_t num_seqs, const int64_t* rows, int64_t n_rows,
                 double scale, double* out, int n_threads) {
  if (!geom_ok(g) || num_seqs < 0 || max_pages < 0) return PKVO_ERR_ARG;
  const int64_t total_q = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
  if (!rows) n_rows = total_q;
  if (n_rows < 0) return PKVO_ERR_ARG;
  int32_t* row_seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_rows + 1));
  int64_t* row_keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_rows + 1));
  int64_t* row_index = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_rows + 1));
  if (!row_seq || !row_keys || !row_index) {
    free(row_seq); free(row_keys); free(row_index);
    return PKVO_ERR_NOMEM;
  }
  int rc = PKVO_OK;
  int64_t max_keys = 1;
  for (int64_t r = 0; r < n_rows && rc == PKVO_OK; ++r) {
    int64_t t = rows ? rows[r] : r;
    if (t < 0 || t >= total_q) { rc = PKVO_ERR_RANGE; break; }
    int64_t n = 0;
    while (n + 1 < num_seqs && cu_q_lens[n + 1] <= t) ++n;
    int64_t i = t - cu_q_lens[n];
    int64_t keys = (int64_t)prefix_lens[n] + i + 1; /* causal, bottom-right aligned */
    if (keys > max_pages * g->page_size) { rc = PKVO_ERR_RANGE; break; }
    row_seq[r] = (int32_t)n;
    row_keys[r] = keys;
    row_index[r] = t;
    if (keys > max_keys) max_keys = keys;
  }
  if (rc == PKVO_OK) {
    job_t job;
    memset(&job, 0, sizeof job);
    job.g = g; job.q = q; job.k_pages = k_pages; job.v_pages = v_pages;
    job.block_table = block_table; job.bt_stride = max_pages;
    job.row_seq = row_seq; job.row_keys = row_keys; job.row_index = row_index;
    job.n_rows = n_rows; job.max_keys = max_keys; job.scale = scale; job.out = out;
    rc = run_job(&job, n_threads);
  }
  free(row_seq); free(row_keys); free(row_index);
  return rc;
}
