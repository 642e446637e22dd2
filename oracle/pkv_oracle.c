/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct FP64 CPU statement of what the paged-KV
 * decode path computes.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline arm may call it; the product path (the CUDA library
 * and its Python binding) never links, imports or executes anything here, and
 * nothing here is shared with that path.
 *
 * Sources (page title, section):
 *   [README]  "Hours of YouTube and 85 handtyped pages of notes on LLM
 *             Inference - Start here" (hackernews.jp translation of the
 *             Tiny-vLLM README), section "これまでの進捗" (progress so far):
 *             the shared BF16 KV page pool with one block table per
 *             (sequence, layer) and 16-token pages; decode adds one token per
 *             sequence at its absolute RoPE position; paged decode attention
 *             with an FP32 online softmax in which every query head streams
 *             its own sequence's cached pages without gathering a contiguous
 *             prefix or storing scores.  Section "現在のスコープ" (scope):
 *             model dimensions and the 2048-token context are fixed.
 *   [TINY]    "Tiny-vLLMでゼロから構築する高性能LLM推論エンジン", sections
 *             "Bfloat16の選択" (BF16 = 8-bit exponent, 7-bit mantissa),
 *             "KV Cache" and "Prefill vs. Decode".
 *
 * Readings where the pages are silent (each is a choice, not a quote):
 *   R1  bf16 results are the round-to-nearest-even image of the FP64 value,
 *       rounded once (no detour through FP32).
 *   R2  RoPE is the rotate-half form: element i < D/2 pairs with i + D/2,
 *       inv_freq_i = theta^(-2i/D), angle = pos * inv_freq_i; the rotation is
 *       evaluated in FP64 as (x1*c - x2*s, x2*c + x1*s), each product and the
 *       sum rounded in FP64 (this file is built with -ffp-contract=off), then
 *       rounded once to bf16 (R1).
 *   R3  Query head j reads kv head j / (Hq/Hkv) (consecutive query heads share
 *       a kv head).
 *   R4  seq_lens[b] counts the tokens attended, including the token appended
 *       in the same step; a sequence of length 0 yields a zero output.
 *   R5  Page layout [page][K|V][slot][kv head][d], element index
 *       ((page*2 + kv)*page_size + slot)*Hkv*D + h*D + d.
 *
 * All parity pins for this file live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2
#define ORC_EBADPAGE 4
#define ORC_EBADLEN 8
#define ORC_EBADPOS 16

int orc_version(void) { return 1; }

/* ---------------------------------------------------------------- bf16 -- */

/* [TINY] "Bfloat16の選択": a bf16 is the top half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * R1: round x to the nearest bf16, ties to even, in one step.
 * The bf16 grid in the binade of x has spacing 2^(E-7) for E = floor(log2|x|)
 * >= -126, and 2^-133 below that (subnormals).  Dividing by the spacing is an
 * exact power-of-two scaling, rint() rounds to the nearest integer with ties
 * to even (default rounding mode), and the product back is exact.
 */
uint16_t orc_f64_to_bf16(double x) {
  if (isnan(x)) return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
  if (x == 0.0) return (uint16_t)(signbit(x) ? 0x8000u : 0x0000u);
  double ax = fabs(x);
  if (isinf(ax)) return (uint16_t)(signbit(x) ? 0xFF80u : 0x7F80u);
  int e = ilogb(ax);
  if (e < -126) e = -126;
  double spacing = ldexp(1.0, e - 7);
  double r = rint(ax / spacing) * spacing;
  if (r >= ldexp(1.0, 128)) return (uint16_t)(signbit(x) ? 0xFF80u : 0x7F80u);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint16_t h = (uint16_t)(u >> 16);
  return (uint16_t)(signbit(x) ? (h | 0x8000u) : h);
}

/* ---------------------------------------------------------------- RoPE -- */

/* R2: inv_freq_i = theta^(-2i/D) for i in [0, D/2). */
void orc_rope_inv_freq(double theta, int head_dim, double* inv_freq) {
  for (int i = 0; i < head_dim / 2; ++i)
    inv_freq[i] = pow(theta, -(2.0 * (double)i) / (double)head_dim);
}

/* R2 before the final rounding: y = RoPE(x, pos) in FP64. */
void orc_rope_rotate_f64(const uint16_t* x, int head_dim, int32_t pos,
                         double theta, double* y) {
  int half = head_dim / 2;
  double inv_freq[512];
  orc_rope_inv_freq(theta, head_dim, inv_freq);
  for (int i = 0; i < half; ++i) {
    double angle = (double)pos * inv_freq[i];
    double c = cos(angle);
    double s = sin(angle);
    double x1 = orc_bf16_to_f64(x[i]);
    double x2 = orc_bf16_to_f64(x[i + half]);
    double a = x1 * c;
    double b = x2 * s;
    double p = x2 * c;
    double q = x1 * s;
    y[i] = a - b;
    y[i + half] = p + q;
  }
}

/* R2 with the bf16 rounding of R1: the value a decode step stores for K. */
void orc_rope_rotate(const uint16_t* x, int head_dim, int32_t pos,
                     double theta, uint16_t* y) {
  double tmp[1024];
  orc_rope_rotate_f64(x, head_dim, pos, theta, tmp);
  for (int d = 0; d < head_dim; ++d) y[d] = orc_f64_to_bf16(tmp[d]);
}

/* ------------------------------------------------------------- append -- */

static int64_t orc_slot_index(int64_t page, int kv, int slot, int h, int d,
                              int page_size, int num_kv_heads, int head_dim) {
  /* R5 */
  return ((page * 2 + kv) * page_size + slot) * (int64_t)num_kv_heads *
             head_dim +
         (int64_t)h * head_dim + d;
}

/*
 * [README] "これまでの進捗", KV page pool item: a decode step adds one new
 * token per sequence at its absolute RoPE position.  For each sequence b the
 * token at position positions[b] goes to slot positions[b] % page_size of the
 * page block_table[b][positions[b] / page_size]; K is stored rotated (R2), V
 * as given.  Entries with a bad position or page are skipped and reported in
 * the returned bit set.
 */
int orc_kv_append(const uint16_t* k_new, const uint16_t* v_new, uint16_t* pool,
                  int64_t num_pages, const int32_t* block_table,
                  int max_blocks, const int32_t* positions, int batch,
                  int num_kv_heads, int head_dim, int page_size,
                  double theta) {
  int status = ORC_OK;
  if (head_dim > 1024 || head_dim % 2) return ORC_EINVAL;
  uint16_t rotated[1024];
  for (int b = 0; b < batch; ++b) {
    int32_t pos = positions[b];
    if (pos < 0 || pos >= max_blocks * page_size) {
      status |= ORC_EBADPOS;
      continue;
    }
    int32_t page = block_table[(int64_t)b * max_blocks + pos / page_size];
    if (page < 0 || page >= num_pages) {
      status |= ORC_EBADPAGE;
      continue;
    }
    int slot = pos % page_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const uint16_t* k = k_new + ((int64_t)b * num_kv_heads + h) * head_dim;
      const uint16_t* v = v_new + ((int64_t)b * num_kv_heads + h) * head_dim;
      orc_rope_rotate(k, head_dim, pos, theta, rotated);
      for (int d = 0; d < head_dim; ++d) {
        pool[orc_slot_index(page, 0, slot, h, d, page_size, num_kv_heads,
                            head_dim)] = rotated[d];
        pool[orc_slot_index(page, 1, slot, h, d, page_size, num_kv_heads,
                            head_dim)] = v[d];
      }
    }
  }
  return status;
}

/*
 * [README] "これまでの進捗", KV page pool item: prefill fills the prompt's
 * pages.  Sequence b contributes the tokens [token_offsets[b],
 * token_offsets[b+1]) of k/v ([num_tokens][Hkv][D]); token i of sequence b
 * sits at absolute position start_positions[b] + i and is stored exactly as a
 * one-token append at that position would store it (K rotated by RoPE at its
 * position, V as given).  Tokens with a bad position or page are skipped and
 * reported in the returned bit set.
 */
int orc_kv_write_prefill(const uint16_t* k, const uint16_t* v,
                         const int32_t* token_offsets,
                         const int32_t* start_positions, uint16_t* pool,
                         int64_t num_pages, const int32_t* block_table,
                         int max_blocks, int batch, int num_kv_heads,
                         int head_dim, int page_size, double theta) {
  int status = ORC_OK;
  for (int b = 0; b < batch; ++b) {
    for (int32_t t = token_offsets[b]; t < token_offsets[b + 1]; ++t) {
      int32_t pos = start_positions[b] + (t - token_offsets[b]);
      /* one token of sequence b, appended at pos through b's block table */
      status |= orc_kv_append(k + (int64_t)t * num_kv_heads * head_dim,
                              v + (int64_t)t * num_kv_heads * head_dim, pool,
                              num_pages, block_table + (int64_t)b * max_blocks,
                              max_blocks, &pos, 1, num_kv_heads, head_dim,
                              page_size, theta);
    }
  }
  return status;
}

/* Optional query rotation: q_out[b][j] = RoPE(q_in[b][j], positions[b]). */
void orc_rope_queries(const uint16_t* q_in, uint16_t* q_out,
                      const int32_t* positions, int batch, int num_q_heads,
                      int head_dim, double theta) {
  for (int b = 0; b < batch; ++b)
    for (int j = 0; j < num_q_heads; ++j) {
      int64_t off = ((int64_t)b * num_q_heads + j) * head_dim;
      orc_rope_rotate(q_in + off, head_dim, positions[b], theta, q_out + off);
    }
}

/* ---------------------------------------------------------- attention -- */

typedef struct {
  const uint16_t* q;
  const uint16_t* pool;
  int64_t num_pages;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  int batch, num_q_heads, num_kv_heads, head_dim, page_size;
  double scale;
  double* out;
  int online; /* 0 = two-pass, 1 = one-pass running max */
  int num_threads;
  int thread_id;
  int status;
} orc_job;

/*
 * Walk the block table of sequence b and copy token t's K and V row of kv
 * head g into k_row / v_row as doubles (the materialised cache rows).
 * Returns nonzero if the page id is out of range.
 */
static int orc_read_token(const orc_job* J, int b, int g, int t, double* k_row,
                          double* v_row) {
  int32_t page = J->block_table[(int64_t)b * J->max_blocks + t / J->page_size];
  if (page < 0 || page >= J->num_pages) return 1;
  int slot = t % J->page_size;
  for (int d = 0; d < J->head_dim; ++d) {
    k_row[d] = orc_bf16_to_f64(J->pool[orc_slot_index(
        page, 0, slot, g, d, J->page_size, J->num_kv_heads, J->head_dim)]);
    v_row[d] = orc_bf16_to_f64(J->pool[orc_slot_index(
        page, 1, slot, g, d, J->page_size, J->num_kv_heads, J->head_dim)]);
  }
  return 0;
}

/*
 * One (sequence b, query head j):
 *   o = sum_t softmax_t(scale * q . K_t) V_t   over t < seq_lens[b].
 * two-pass: s_t for every t, m = max s_t, w_t = exp(s_t - m), l = sum w_t,
 *           o = sum w_t V_t / l.
 * online:   one pass keeping (m, l, acc) and rescaling by exp(m_old - m_new)
 *           whenever the running maximum grows ([README] "これまでの進捗",
 *           paged decode attention item).
 */
static int orc_attend_one(const orc_job* J, int b, int j, double* o) {
  int D = J->head_dim;
  int group = J->num_q_heads / J->num_kv_heads;
  int g = j / group; /* R3 */
  int L = J->seq_lens[b];
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (L < 0 || L > J->max_blocks * J->page_size) return ORC_EBADLEN;
  if (L == 0) return ORC_OK; /* R4 */

  double* qd = (double*)malloc(sizeof(double) * D);
  double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
  double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  if (!qd || !K || !V || !s) {
    free(qd); free(K); free(V); free(s);
    return ORC_ENOMEM;
  }
  const uint16_t* qrow = J->q + ((int64_t)b * J->num_q_heads + j) * D;
  for (int d = 0; d < D; ++d) qd[d] = orc_bf16_to_f64(qrow[d]);
  for (int t = 0; t < L; ++t) {
    if (orc_read_token(J, b, g, t, K + (size_t)t * D, V + (size_t)t * D)) {
      free(qd); free(K); free(V); free(s);
      return ORC_EBADPAGE;
    }
  }
  for (int t = 0; t < L; ++t) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qd[d] * K[(size_t)t * D + d];
    s[t] = J->scale * dot;
  }
  if (!J->online) {
    double m = -INFINITY;
    for (int t = 0; t < L; ++t)
      if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int t = 0; t < L; ++t) {
      double w = exp(s[t] - m);
      l += w;
      for (int d = 0; d < D; ++d) o[d] += w * V[(size_t)t * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
  } else {
    double m = -INFINITY, l = 0.0;
    for (int t = 0; t < L; ++t) {
      double m_new = s[t] > m ? s[t] : m;
      double alpha = exp(m - m_new); /* exp(-inf) = 0 on the first token */
      double w = exp(s[t] - m_new);
      l = l * alpha + w;
      for (int d = 0; d < D; ++d)
        o[d] = o[d] * alpha + w * V[(size_t)t * D + d];
      m = m_new;
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
  }
  free(qd); free(K); free(V); free(s);
  return ORC_OK;
}

static void* orc_worker(void* arg) {
  orc_job* J = (orc_job*)arg;
  int pairs = J->batch * J->num_q_heads;
  for (int p = J->thread_id; p < pairs; p += J->num_threads) {
    int b = p / J->num_q_heads, j = p % J->num_q_heads;
    J->status |= orc_attend_one(
        J, b, j, J->out + ((int64_t)b * J->num_q_heads + j) * J->head_dim);
  }
  return NULL;
}

static int orc_run(orc_job proto) {
  if (proto.num_q_heads <= 0 || proto.num_kv_heads <= 0 ||
      proto.num_q_heads % proto.num_kv_heads || proto.head_dim <= 0 ||
      proto.page_size <= 0 || proto.batch < 0)
    return ORC_EINVAL;
  int T = proto.num_threads > 0 ? proto.num_threads : 1;
  if (T > 256) T = 256;
  orc_job jobs[256];
  pthread_t tids[256];
  for (int i = 0; i < T; ++i) {
    jobs[i] = proto;
    jobs[i].num_threads = T;
    jobs[i].thread_id = i;
    jobs[i].status = 0;
  }
  if (T == 1) {
    orc_worker(&jobs[0]);
    return jobs[0].status;
  }
  int started = 0;
  for (int i = 0; i < T; ++i) {
    if (pthread_create(&tids[i], NULL, orc_worker, &jobs[i]) != 0) break;
    ++started;
  }
  for (int i = started; i < T; ++i) orc_worker(&jobs[i]); /* run inline */
  int status = 0;
  for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
  for (int i = 0; i < T; ++i) status |= jobs[i].status;
  return status;
}

/* Two-pass FP64 attention for every (b, j); out is [batch][Hq][D] doubles. */
int orc_decode_attention(const uint16_t* q, const uint16_t* pool,
                         int64_t num_pages, const int32_t* block_table,
                         int max_blocks, const int32_t* seq_lens, int batch,
                         int num_q_heads, int num_kv_heads, int head_dim,
                         int page_size, double scale, double* out,
                         int num_threads) {
  orc_job J = {q, pool, num_pages, block_table, max_blocks, seq_lens,
               batch, num_q_heads, num_kv_heads, head_dim, page_size,
               scale, out, 0, num_threads, 0, 0};
  return orc_run(J);
}

/* The same quantity through the one-pass running-max recurrence. */
int orc_decode_attention_online(const uint16_t* q, const uint16_t* pool,
                                int64_t num_pages, const int32_t* block_table,
                                int max_blocks, const int32_t* seq_lens,
                                int batch, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, double scale,
                                double* out, int num_threads) {
  orc_job J = {q, pool, num_pages, block_table, max_blocks, seq_lens,
               batch, num_q_heads, num_kv_heads, head_dim, page_size,
               scale, out, 1, num_threads, 0, 0};
  return orc_run(J);
}

/* ------------------------------------------------------ split partials -- */

/*
 * Partial state of (b, j) over tokens [t_begin, t_end):
 *   m = max s_t, l = sum exp(s_t - m), acc = sum exp(s_t - m) V_t.
 * An empty range gives m = -inf, l = 0, acc = 0.
 */
int orc_attention_partial(const uint16_t* q, const uint16_t* pool,
                          int64_t num_pages, const int32_t* block_table,
                          int max_blocks, int num_q_heads, int num_kv_heads,
                          int head_dim, int page_size, double scale, int b,
                          int j, int t_begin, int t_end, double* m_out,
                          double* l_out, double* acc) {
  orc_job J = {q, pool, num_pages, block_table, max_blocks, NULL,
               0, num_q_heads, num_kv_heads, head_dim, page_size,
               scale, NULL, 0, 1, 0, 0};
  int D = head_dim;
  int g = j / (num_q_heads / num_kv_heads);
  double m = -INFINITY, l = 0.0;
  for (int d = 0; d < D; ++d) acc[d] = 0.0;
  if (t_end <= t_begin) {
    *m_out = m;
    *l_out = l;
    return ORC_OK;
  }
  int n = t_end - t_begin;
  double* K = (double*)malloc(sizeof(double) * (size_t)n * D);
  double* V = (double*)malloc(sizeof(double) * (size_t)n * D);
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!K || !V || !s) {
    free(K); free(V); free(s);
    return ORC_ENOMEM;
  }
  const uint16_t* qrow = q + ((int64_t)b * num_q_heads + j) * D;
  for (int t = 0; t < n; ++t) {
    if (orc_read_token(&J, b, g, t_begin + t, K + (size_t)t * D,
                       V + (size_t)t * D)) {
      free(K); free(V); free(s);
      return ORC_EBADPAGE;
    }
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += orc_bf16_to_f64(qrow[d]) * K[(size_t)t * D + d];
    s[t] = scale * dot;
    if (s[t] > m) m = s[t];
  }
  for (int t = 0; t < n; ++t) {
    double w = exp(s[t] - m);
    l += w;
    for (int d = 0; d < D; ++d) acc[d] += w * V[(size_t)t * D + d];
  }
  free(K); free(V); free(s);
  *m_out = m;
  *l_out = l;
  return ORC_OK;
}

/*
 * Combine S partial states of one (b, j):
 *   M = max m_i, L = sum l_i exp(m_i - M), o = sum acc_i exp(m_i - M) / L.
 * Partials with l = 0 (empty ranges) are skipped; all empty gives o = 0.
 */
void orc_merge_partials(int num_splits, const double* m, const double* l,
                        const double* acc, int head_dim, double* out) {
  double M = -INFINITY;
  for (int i = 0; i < num_splits; ++i)
    if (l[i] > 0.0 && m[i] > M) M = m[i];
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (M == -INFINITY) return;
  double Lsum = 0.0;
  for (int i = 0; i < num_splits; ++i) {
    if (!(l[i] > 0.0)) continue;
    double w = exp(m[i] - M);
    Lsum += l[i] * w;
    for (int d = 0; d < head_dim; ++d) out[d] += acc[(size_t)i * head_dim + d] * w;
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= Lsum;
}
