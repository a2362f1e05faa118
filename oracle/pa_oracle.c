/*
 * Oracle for windowed prefill attention over a paged int8 KV pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the bench's CPU
 * baseline use it.  It shares no code, header or table with the CUDA path.
 *
 * Sources (page titles; sections):
 *   [P1] "int8 tensor-core prefill attention", sections "Summary" and
 *        "Why the attention, and why tensor cores"; "Relation to open PRs"
 *        for the window-off case.
 *   [P2] "fp16 shared-memory tiles for windowed prefill attention", "Summary"
 *        (int8 paged KV pool, StreamingLLM sink + window).
 *
 * What is computed (the plain definition, fp64 throughout):
 *   row (sequence s, query token t = q_start + i, q head h), kv head g = h / (HQ/HKV);
 *   key j is visible iff j <= t and, when the window is on (W > 0),
 *   block(j) < S or block(j) >= max(0, block(t) + 1 - W), blocks being 16-token
 *   pages [P1 "Why the attention...": window start constant over a 16-row tile,
 *   only the causal bound varies per row; P1 "Relation to open PRs": W <= 0 is
 *   full causal; P2 "Summary": StreamingLLM window = sink blocks + recent blocks];
 *   K_j = k_code * k_scale, V_j = v_code * v_scale (per token, per kv head) [P1, P2];
 *   s_j = sm_scale * <q, K_j>;  out = sum_j softmax(s)_j V_j (two passes).
 *
 * The method the pages describe approximates this with an int8 query
 * (one scale per row), per-token K scales and the softmax scale applied to the
 * integer scores, an online softmax over key tiles, and the per-token V scale
 * folded into P before P is quantised per row [P1 "Why the attention...",
 * bullets 2-3].  pa_oracle_method() walks those steps in that order so the
 * quantisation error of each choice can be measured against pa_oracle_exact().
 *
 * Built with plain -O2 (no fast-math) into a shared library called via ctypes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int n_q_heads, n_kv_heads, head_dim, page_size;
  const uint16_t* q;           /* bf16 bit patterns [total_q][HQ][D] */
  const int8_t* k_pool;        /* [n_pool][page][HKV][D] */
  const int8_t* v_pool;        /* [n_pool][page][HKV][D] */
  const float* k_scale;        /* [n_pool][page][HKV] */
  const float* v_scale;        /* [n_pool][page][HKV] */
  const int32_t* block_table;  /* [n_seq][bt_stride] */
  int bt_stride;
  int n_seq;
  const int32_t* seqs;         /* [n_seq][4] = q_off, q_start, n_q, n_ctx */
  int n_sink_blk, n_win_blk;
  double sm_scale;
} pa_problem;

static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* The block mask of the pages: causal, plus sink blocks and the last W blocks
 * up to and including the query's own block. */
int pa_oracle_key_visible(int t, int j, int page, int n_sink_blk, int n_win_blk) {
  if (j > t) return 0;
  if (n_win_blk <= 0) return 1;
  int bj = j / page, bt = t / page;
  int lo = bt + 1 - n_win_blk;
  if (lo < 0) lo = 0;
  return bj < n_sink_blk || bj >= lo;
}

/* Number of visible keys of query token t (an enumeration, not a closed form). */
long long pa_oracle_visible_count(int t, int page, int n_sink_blk, int n_win_blk) {
  long long c = 0;
  for (int j = 0; j <= t; ++j) c += pa_oracle_key_visible(t, j, page, n_sink_blk, n_win_blk);
  return c;
}

/* Visible (query token, key) pairs summed over tokens [q_start, q_start + n_q). */
long long pa_oracle_visible_pairs(int q_start, int n_q, int page, int n_sink_blk, int n_win_blk) {
  long long c = 0;
  for (int t = q_start; t < q_start + n_q; ++t)
    c += pa_oracle_visible_count(t, page, n_sink_blk, n_win_blk);
  return c;
}

/* For each query block qb in [qb_first, qb_last]: the key blocks visible to at
 * least one token of that block that lies in [q_start, q_start+n_q), in
 * increasing order, written to out[(qb - qb_first) * cap + k], padded with -1.
 * Returns 0, or -1 if a list does not fit in cap. */
int pa_oracle_block_lists(int q_start, int n_q, int page, int n_sink_blk, int n_win_blk,
                          int cap, int32_t* out) {
  int qb_first = q_start / page, qb_last = (q_start + n_q - 1) / page;
  for (int qb = qb_first; qb <= qb_last; ++qb) {
    int32_t* row = out + (size_t)(qb - qb_first) * cap;
    for (int k = 0; k < cap; ++k) row[k] = -1;
    int t_lo = qb * page, t_hi = qb * page + page - 1;
    if (t_lo < q_start) t_lo = q_start;
    if (t_hi > q_start + n_q - 1) t_hi = q_start + n_q - 1;
    int n = 0;
    for (int kb = 0; kb <= qb; ++kb) {
      int any = 0;
      for (int t = t_lo; t <= t_hi && !any; ++t)
        for (int j = kb * page; j < kb * page + page && !any; ++j)
          any = pa_oracle_key_visible(t, j, page, n_sink_blk, n_win_blk);
      if (any) {
        if (n >= cap) return -1;
        row[n++] = kb;
      }
    }
  }
  return 0;
}

/* Gather through the block table: logical tokens [0, n_tok) of sequence s,
 * kv head g -> codes [n_tok][D] and scales [n_tok]. */
void pa_oracle_gather(const pa_problem* P, int s, int g, int n_tok, int8_t* k_out, int8_t* v_out,
                      float* ks_out, float* vs_out) {
  const int D = P->head_dim, PG = P->page_size, HKV = P->n_kv_heads;
  for (int j = 0; j < n_tok; ++j) {
    int phys = P->block_table[(size_t)s * P->bt_stride + j / PG];
    size_t slot = (size_t)phys * PG + (size_t)(j % PG);
    memcpy(k_out + (size_t)j * D, P->k_pool + (slot * HKV + g) * D, (size_t)D);
    memcpy(v_out + (size_t)j * D, P->v_pool + (slot * HKV + g) * D, (size_t)D);
    ks_out[j] = P->k_scale[slot * HKV + g];
    vs_out[j] = P->v_scale[slot * HKV + g];
  }
}

/* Locate the sequence of global query row i; returns s and the token t. */
static int locate(const pa_problem* P, int i, int* t_out) {
  for (int s = 0; s < P->n_seq; ++s) {
    const int32_t* d = P->seqs + 4 * s;
    if (i >= d[0] && i < d[0] + d[2]) {
      *t_out = d[1] + (i - d[0]);
      return s;
    }
  }
  return -1;
}

/* Dequantised key/value element access. */
static const int8_t* k_code(const pa_problem* P, int s, int g, int j, double* scale) {
  int phys = P->block_table[(size_t)s * P->bt_stride + j / P->page_size];
  size_t slot = (size_t)phys * P->page_size + (size_t)(j % P->page_size);
  *scale = (double)P->k_scale[slot * P->n_kv_heads + g];
  return P->k_pool + (slot * P->n_kv_heads + g) * P->head_dim;
}
static const int8_t* v_code(const pa_problem* P, int s, int g, int j, double* scale) {
  int phys = P->block_table[(size_t)s * P->bt_stride + j / P->page_size];
  size_t slot = (size_t)phys * P->page_size + (size_t)(j % P->page_size);
  *scale = (double)P->v_scale[slot * P->n_kv_heads + g];
  return P->v_pool + (slot * P->n_kv_heads + g) * P->head_dim;
}

/* ---------------------------------------------------------------- exact */
static void exact_row(const pa_problem* P, int i, int h, double* out) {
  const int D = P->head_dim;
  int t;
  int s = locate(P, i, &t);
  int g = h / (P->n_q_heads / P->n_kv_heads);
  const uint16_t* qrow = P->q + ((size_t)i * P->n_q_heads + h) * D;
  double* q = (double*)malloc(sizeof(double) * D);
  double* score = (double*)malloc(sizeof(double) * (size_t)(t + 1));
  for (int d = 0; d < D; ++d) q[d] = bf16_to_double(qrow[d]);
  /* pass 1: scores of visible keys and their maximum */
  double m = -INFINITY;
  for (int j = 0; j <= t; ++j) {
    if (!pa_oracle_key_visible(t, j, P->page_size, P->n_sink_blk, P->n_win_blk)) continue;
    double ks;
    const int8_t* kc = k_code(P, s, g, j, &ks);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * ((double)kc[d] * ks);
    score[j] = P->sm_scale * dot;
    if (score[j] > m) m = score[j];
  }
  /* pass 2: normalised weights times dequantised values */
  double denom = 0.0;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int j = 0; j <= t; ++j) {
    if (!pa_oracle_key_visible(t, j, P->page_size, P->n_sink_blk, P->n_win_blk)) continue;
    double w = exp(score[j] - m);
    double vs;
    const int8_t* vc = v_code(P, s, g, j, &vs);
    denom += w;
    for (int d = 0; d < D; ++d) out[d] += w * ((double)vc[d] * vs);
  }
  for (int d = 0; d < D; ++d) out[d] /= denom;
  free(q);
  free(score);
}

/* ---------------------------------------------------------------- quantisers */
/* Q per row [P1 "Why the attention...": "quantizes Q per query row (one
 * scale/row)"], symmetric int8 with scale absmax/127 and round-half-even.  The
 * decision is taken in float32: inv = 127/absmax, code = rint(q * inv) clamped
 * to +-127.  An all-zero row gets scale 0 and codes 0. */
void pa_oracle_quantize_q_row(const uint16_t* q, int D, int8_t* codes, float* scale) {
  float absmax = 0.0f;
  for (int d = 0; d < D; ++d) {
    float a = fabsf((float)bf16_to_double(q[d]));
    if (a > absmax) absmax = a;
  }
  if (!(absmax > 0.0f)) {
    *scale = 0.0f;
    for (int d = 0; d < D; ++d) codes[d] = 0;
    return;
  }
  float inv = 127.0f / absmax;
  *scale = absmax / 127.0f;
  for (int d = 0; d < D; ++d) {
    float c = rintf((float)bf16_to_double(q[d]) * inv);
    if (c > 127.0f) c = 127.0f;
    if (c < -127.0f) c = -127.0f;
    codes[d] = (int8_t)c;
  }
}

/* P' of one row over one key tile, quantised to u8 with one scale
 * s_p = max P' / 255 [P1 "Why the attention...": "folds the per-token V scale
 * into P and quantizes P per row"; P' >= 0, so the unsigned grid].  Writes the
 * codes (as doubles) to out, returns s_p; a tile with max P' = 0 keeps
 * prev_scale and gets all-zero codes. */
double pa_oracle_quantize_p_u8(const double* p, int n, double prev_scale, double* out) {
  double pmax = 0.0;
  for (int k = 0; k < n; ++k)
    if (p[k] > pmax) pmax = p[k];
  double sp = pmax > 0.0 ? pmax / 255.0 : prev_scale;
  for (int k = 0; k < n; ++k) out[k] = pmax > 0.0 ? rint(p[k] / sp) : 0.0;
  return sp;
}

/* ---------------------------------------------------------------- method */
enum { Q_LOSSLESS = 0, Q_INT8 = 1 };
enum { P_F16 = 0, P_U8 = 1, P_EXACT = 2 };

/* Round to 11 significant bits, nearest-even (fp16 precision, no range limits). */
static double round_sig11(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  double f = frexp(x, &e); /* x = f * 2^e, 0.5 <= |f| < 1 */
  return ldexp(rint(ldexp(f, 11)), e - 11);
}

/* One row through the pages' steps:
 *  a1  Q per-row quantise: s_q = absmax/127, code = rint(q * 127/absmax), in
 *      float32 (the precision the kernel takes that decision in); or, for the
 *      lossless container, q itself;
 *  a4  integer scores S_j = <q_code, k_code_j> (exact);
 *  a5  x_j = S_j * s_q * s_k[j] * sm_scale; online softmax over key tiles:
 *      m' = max(m, max x), alpha = e^(m - m'), p = e^(x - m'), l = alpha l + sum p;
 *  a6  P'_j = p_j * s_v[j] (V scale folded into P); then P' is rounded to fp16
 *      precision, or quantised per row over the tile to u8 with s_p = max P'/255;
 *  a7  O = alpha (s_p_prev / s_p) O + sum_j code(P'_j) v_code_j;
 *  a8  out = O s_p / l.
 * Key tiles: the row's visible keys in increasing order, cut into runs of at
 * most `tile` keys that restart at the start of the sink run and of the
 * window run (each run begins on a 16-token block). */
static void method_row(const pa_problem* P, int i, int h, int q_mode, int p_mode, int tile,
                       double* out) {
  const int D = P->head_dim, PG = P->page_size;
  int t;
  int s = locate(P, i, &t);
  int g = h / (P->n_q_heads / P->n_kv_heads);
  const uint16_t* qrow = P->q + ((size_t)i * P->n_q_heads + h) * D;
  double* qv = (double*)malloc(sizeof(double) * D);
  double* O = (double*)calloc((size_t)D, sizeof(double));
  double* x = (double*)malloc(sizeof(double) * (size_t)tile);
  int* key = (int*)malloc(sizeof(int) * (size_t)tile);
  double* pq = (double*)malloc(sizeof(double) * (size_t)tile);
  double s_q = 1.0;
  if (q_mode == Q_INT8) {
    int8_t* codes = (int8_t*)malloc((size_t)D);
    float sq;
    pa_oracle_quantize_q_row(qrow, D, codes, &sq);
    s_q = (double)sq;
    for (int d = 0; d < D; ++d) qv[d] = (double)codes[d];
    free(codes);
  } else {
    for (int d = 0; d < D; ++d) qv[d] = bf16_to_double(qrow[d]);
  }

  /* runs: [0, sink_end) and [win_start, t] in tokens */
  int bt = t / PG;
  int lo = P->n_win_blk > 0 ? bt + 1 - P->n_win_blk : 0;
  if (lo < 0) lo = 0;
  int sink_end = P->n_win_blk > 0 ? (P->n_sink_blk < lo ? P->n_sink_blk : lo) * PG : 0;
  int runs[2][2] = {{0, sink_end}, {lo * PG, t + 1}};
  if (sink_end == lo * PG) { /* sink run touches the window: one run */
    runs[0][1] = 0;
    runs[1][0] = 0;
  }

  double m = -INFINITY, l = 0.0, sp_prev = 1.0, sp = 1.0;
  for (int r = 0; r < 2; ++r) {
    for (int j0 = runs[r][0]; j0 < runs[r][1]; j0 += tile) {
      int j1 = j0 + tile < runs[r][1] ? j0 + tile : runs[r][1];
      int n = 0;
      double tmax = -INFINITY;
      for (int j = j0; j < j1; ++j) {
        if (!pa_oracle_key_visible(t, j, PG, P->n_sink_blk, P->n_win_blk)) continue;
        double ks;
        const int8_t* kc = k_code(P, s, g, j, &ks);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qv[d] * (double)kc[d];
        key[n] = j;
        x[n] = dot * s_q * ks * P->sm_scale;
        if (x[n] > tmax) tmax = x[n];
        ++n;
      }
      if (n == 0) continue;
      double m_new = tmax > m ? tmax : m;
      double alpha = isinf(m) ? 0.0 : exp(m - m_new);
      double psum = 0.0, pmax = 0.0;
      for (int k = 0; k < n; ++k) {
        double p = exp(x[k] - m_new);
        double vs;
        (void)v_code(P, s, g, key[k], &vs);
        psum += p;
        pq[k] = p * vs; /* V scale folded into P */
        if (pq[k] > pmax) pmax = pq[k];
      }
      l = alpha * l + psum;
      double corr = alpha;
      if (p_mode == P_U8) {
        sp = pa_oracle_quantize_p_u8(pq, n, sp_prev, pq);
        corr = alpha * sp_prev / sp;
      } else if (p_mode == P_F16) {
        for (int k = 0; k < n; ++k) pq[k] = round_sig11(pq[k]);
      }
      for (int d = 0; d < D; ++d) O[d] *= corr;
      for (int k = 0; k < n; ++k) {
        double vs;
        const int8_t* vc = v_code(P, s, g, key[k], &vs);
        for (int d = 0; d < D; ++d) O[d] += pq[k] * (double)vc[d];
      }
      m = m_new;
      sp_prev = sp;
    }
  }
  double fin = (p_mode == P_U8 ? sp : 1.0) / l;
  for (int d = 0; d < D; ++d) out[d] = O[d] * fin;
  free(qv);
  free(O);
  free(x);
  free(key);
  free(pq);
}

/* ---------------------------------------------------------------- threads */
typedef struct {
  const pa_problem* P;
  const int32_t* rows; /* [n_rows][2] = (global q row, q head) */
  int n_rows, kind, q_mode, p_mode, tile;
  double* out;         /* [n_rows][D] */
  int next;
  pthread_mutex_t mu;
} job_t;

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int r = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (r >= J->n_rows) break;
    double* o = J->out + (size_t)r * J->P->head_dim;
    if (J->kind == 0)
      exact_row(J->P, J->rows[2 * r], J->rows[2 * r + 1], o);
    else
      method_row(J->P, J->rows[2 * r], J->rows[2 * r + 1], J->q_mode, J->p_mode, J->tile, o);
  }
  return NULL;
}

static int run_rows(const pa_problem* P, int n_rows, const int32_t* rows, int kind, int q_mode,
                    int p_mode, int tile, double* out, int n_threads) {
  for (int r = 0; r < n_rows; ++r) {
    int t;
    if (locate(P, rows[2 * r], &t) < 0) return -1;
    if (rows[2 * r + 1] < 0 || rows[2 * r + 1] >= P->n_q_heads) return -1;
  }
  job_t J;
  J.P = P;
  J.rows = rows;
  J.n_rows = n_rows;
  J.kind = kind;
  J.q_mode = q_mode;
  J.p_mode = p_mode;
  J.tile = tile;
  J.out = out;
  J.next = 0;
  pthread_mutex_init(&J.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int k = 0; k < n_threads; ++k) pthread_create(&th[k], NULL, worker, &J);
  for (int k = 0; k < n_threads; ++k) pthread_join(th[k], NULL);
  free(th);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

/* Exact fp64 attention for the listed (global q row, q head) pairs. */
int pa_oracle_exact(const pa_problem* P, int n_rows, const int32_t* rows, double* out,
                    int n_threads) {
  return run_rows(P, n_rows, rows, 0, 0, 0, 0, out, n_threads);
}

/* The pages' quantised method for the listed rows (modes as above). */
int pa_oracle_method(const pa_problem* P, int n_rows, const int32_t* rows, int q_mode, int p_mode,
                     int tile, double* out, int n_threads) {
  if (tile < 1) return -1;
  return run_rows(P, n_rows, rows, 1, q_mode, p_mode, tile, out, n_threads);
}
