/*
 * TEST INFRASTRUCTURE ONLY -- the fp64 CPU oracle for packed variable-length
 * attention.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load this library; the product path never does.
 *
 * It shares no code, header, table or helper with the CUDA path.  It is the
 * plain definition of the operation, written out as a loop nest in double
 * precision, following these passages of the "onnx-runtime-ep-cuda" source
 * pages:
 *
 *   - packed_varlen_attention.rs, module doc "Packed layout & cumulative
 *     offsets": sequence b owns query rows [cu_q[b], cu_q[b+1]) and key/value
 *     rows [cu_kv[b], cu_kv[b+1]); attention is block diagonal.
 *   - same page, "Schema (v1)": Q [total_q, H, d], K [total_kv, Hkv, d],
 *     V [total_kv, Hkv, dv], out [total_q, H, dv]; Hkv divides H; the query
 *     head h reads key/value head h / (H / Hkv) (kernel source, `kvh = qh /
 *     group`).
 *   - same page, "Causal alignment": local query i sees local key j iff
 *     j <= i + (L_kv - L_q).
 *   - attention.rs and group_query_attention.rs, the softmax / reference
 *     kernels' `local_window`: with a window W > 0, keys before
 *     frontier + 1 - W are masked as well (frontier = i + L_kv - L_q, the
 *     causal limit, which sets the window's end whether or not the causal
 *     mask itself is on).  W <= 0 means no window.
 *   - same page, kernel stages 1-5: score = scale * q.k; softcap (when
 *     nonzero) replaces the score by softcap * tanh(score / softcap) before the
 *     mask; max-subtracted exponentials, normalised; a row whose every key is
 *     masked produces zeros; out = sum_j p_j * V[j].
 *
 * The stage order (all scores, then max, then exponentials and their sum, then
 * the weighted sum of V) is the pages' own; nothing is tiled, fused or
 * reordered.  Inputs arrive already widened to double (bf16/f16/f32 -> double
 * is exact), so the oracle sees the very values the GPU sees.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC pva_oracle.c -o libpva_oracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_OOM -4

/* Index of the sequence that owns packed query token `tok`: the b with
 * cu_q[b] <= tok < cu_q[b+1].  Plain binary search over the non-decreasing
 * offsets; empty sequences (cu_q[b] == cu_q[b+1]) are skipped naturally. */
static int owner_sequence(const int32_t* cu_q, int B, int64_t tok) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = lo + (hi - lo + 1) / 2;
    if ((int64_t)cu_q[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/* One output row: query token `tok` (local position i in sequence b), query
 * head h.  `scores` is caller scratch of at least L_kv doubles. */
static void attend_one_row(const double* q, const double* k, const double* v,
                           const int32_t* cu_q, const int32_t* cu_kv,
                           int b, int64_t tok, int h,
                           int H, int Hkv, int d, int dv,
                           double scale, int is_causal, double softcap,
                           int local_window, double* scores, double* out_row) {
  const int group = H / Hkv;
  const int g = h / group;                          /* shared key/value head */
  const int64_t q_start = cu_q[b];
  const int64_t L_q = (int64_t)cu_q[b + 1] - cu_q[b];
  const int64_t kv_start = cu_kv[b];
  const int64_t L_kv = (int64_t)cu_kv[b + 1] - cu_kv[b];
  const int64_t i = tok - q_start;
  const int64_t frontier = i + (L_kv - L_q);        /* tail-aligned causal */
  const double* qrow = q + (tok * H + h) * (int64_t)d;

  /* Stage 1-3: scores of every visible key (invisible keys are skipped, which
   * is what a -inf score contributes to the softmax). */
  int64_t n_visible = 0;
  double m = -INFINITY;
  for (int64_t j = 0; j < L_kv; ++j) {
    if (is_causal && j > frontier) { scores[j] = -INFINITY; continue; }
    if (local_window > 0 && j < frontier + 1 - local_window) { scores[j] = -INFINITY; continue; }
    const double* krow = k + ((kv_start + j) * Hkv + g) * (int64_t)d;
    double dot = 0.0;
    for (int p = 0; p < d; ++p) dot += qrow[p] * krow[p];
    double s = scale * dot;
    if (softcap != 0.0) s = softcap * tanh(s / softcap);
    scores[j] = s;
    if (s > m) m = s;
    ++n_visible;
  }

  for (int c = 0; c < dv; ++c) out_row[c] = 0.0;
  if (n_visible == 0) return;                       /* fully masked -> zeros */

  /* Stage 4: max-subtracted exponentials and their sum. */
  double l = 0.0;
  for (int64_t j = 0; j < L_kv; ++j) {
    if (scores[j] == -INFINITY) { scores[j] = 0.0; continue; }
    scores[j] = exp(scores[j] - m);
    l += scores[j];
  }
  /* Stage 5: normalised weights times V. */
  for (int64_t j = 0; j < L_kv; ++j) {
    const double p = scores[j] / l;
    if (p == 0.0) continue;
    const double* vrow = v + ((kv_start + j) * Hkv + g) * (int64_t)dv;
    for (int c = 0; c < dv; ++c) out_row[c] += p * vrow[c];
  }
}

static int check_args(const int32_t* cu_q, const int32_t* cu_kv, int B, int H,
                      int Hkv, int d, int dv) {
  if (!cu_q || !cu_kv || B < 1 || H <= 0 || Hkv <= 0 || H % Hkv != 0 ||
      d <= 0 || dv <= 0)
    return ORACLE_BAD_ARG;
  if (cu_q[0] != 0 || cu_kv[0] != 0) return ORACLE_BAD_ARG;
  for (int b = 0; b < B; ++b)
    if (cu_q[b + 1] < cu_q[b] || cu_kv[b + 1] < cu_kv[b]) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

static int64_t max_kv_len(const int32_t* cu_kv, int B) {
  int64_t mx = 1;
  for (int b = 0; b < B; ++b) {
    int64_t L = (int64_t)cu_kv[b + 1] - cu_kv[b];
    if (L > mx) mx = L;
  }
  return mx;
}

/* Full forward: every row of `out` [cu_q[B], H, dv] is written. */
int pva_oracle_forward_window(const double* q, const double* k, const double* v,
                              const int32_t* cu_q, const int32_t* cu_kv, double* out,
                              int B, int H, int Hkv, int d, int dv, double scale,
                              int is_causal, double softcap, int local_window,
                              int nthreads) {
  int rc = check_args(cu_q, cu_kv, B, H, Hkv, d, dv);
  if (rc != ORACLE_OK) return rc;
  const int64_t total_q = cu_q[B];
  const int64_t n_rows = total_q * H;
  const int64_t smax = max_kv_len(cu_kv, B);
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)smax);
    if (!scores) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t row = 0; row < n_rows; ++row) {
      if (!scores) continue;
      const int64_t tok = row / H;
      const int h = (int)(row % H);
      const int b = owner_sequence(cu_q, B, tok);
      attend_one_row(q, k, v, cu_q, cu_kv, b, tok, h, H, Hkv, d, dv, scale,
                     is_causal, softcap, local_window, scores, out + row * (int64_t)dv);
    }
    free(scores);
  }
  return failed ? ORACLE_OOM : ORACLE_OK;
}

int pva_oracle_forward(const double* q, const double* k, const double* v,
                       const int32_t* cu_q, const int32_t* cu_kv, double* out,
                       int B, int H, int Hkv, int d, int dv, double scale,
                       int is_causal, double softcap, int nthreads) {
  return pva_oracle_forward_window(q, k, v, cu_q, cu_kv, out, B, H, Hkv, d, dv, scale,
                                   is_causal, softcap, 0, nthreads);
}

/* Sampled forward: only the listed rows, row = token * H + head, written to
 * out_rows [n_rows, dv] in the order given.  Used where the full problem is
 * too large for the CPU. */
int pva_oracle_rows_window(const double* q, const double* k, const double* v,
                           const int32_t* cu_q, const int32_t* cu_kv,
                           const int64_t* rows, int64_t n_rows, double* out_rows,
                           int B, int H, int Hkv, int d, int dv, double scale,
                           int is_causal, double softcap, int local_window, int nthreads) {
  int rc = check_args(cu_q, cu_kv, B, H, Hkv, d, dv);
  if (rc != ORACLE_OK) return rc;
  const int64_t total_rows = (int64_t)cu_q[B] * H;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= total_rows) return ORACLE_BAD_ARG;
  const int64_t smax = max_kv_len(cu_kv, B);
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)smax);
    if (!scores) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
      if (!scores) continue;
      const int64_t tok = rows[r] / H;
      const int h = (int)(rows[r] % H);
      const int b = owner_sequence(cu_q, B, tok);
      attend_one_row(q, k, v, cu_q, cu_kv, b, tok, h, H, Hkv, d, dv, scale,
                     is_causal, softcap, local_window, scores, out_rows + r * (int64_t)dv);
    }
    free(scores);
  }
  return failed ? ORACLE_OOM : ORACLE_OK;
}

int pva_oracle_rows(const double* q, const double* k, const double* v,
                    const int32_t* cu_q, const int32_t* cu_kv,
                    const int64_t* rows, int64_t n_rows, double* out_rows,
                    int B, int H, int Hkv, int d, int dv, double scale,
                    int is_causal, double softcap, int nthreads) {
  return pva_oracle_rows_window(q, k, v, cu_q, cu_kv, rows, n_rows, out_rows, B, H, Hkv, d,
                                dv, scale, is_causal, softcap, 0, nthreads);
}

/* Padded form: the opset-24 Attention input `nonpad_kv_seqlen` (attention.rs,
 * the per-batch causal offset and padding frontier set up before the launch;
 * packed_varlen_attention.rs, module doc "Relationship to ONNX Attention-24
 * nonpad_kv_seqlen").  Batch entry b has q_seq query rows and a slot of kv_seq
 * key/value rows: q [B, q_seq, H, d], k [B, kv_seq, Hkv, d],
 * v [B, kv_seq, Hkv, dv], out [B, q_seq, H, dv].  Query row i of entry b sees
 * slot row j iff j < nonpad[b] (the padding frontier, in every mode) and, when
 * causal, j <= i + offset with offset = nonpad[b] - q_seq.  Written on its own
 * over the padded layout (no packing), so that the tests can hold it against
 * the packed definition above. */
int pva_oracle_forward_padded(const double* q, const double* k, const double* v,
                              const int64_t* nonpad, double* out, int B, int q_seq, int kv_seq,
                              int H, int Hkv, int d, int dv, double scale, int is_causal,
                              double softcap, int nthreads) {
  if (!nonpad || B < 1 || q_seq < 0 || kv_seq < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 ||
      d <= 0 || dv <= 0)
    return ORACLE_BAD_ARG;
  for (int b = 0; b < B; ++b)
    if (nonpad[b] < 0 || nonpad[b] > kv_seq) return ORACLE_BAD_ARG;
  const int group = H / Hkv;
  const int64_t n_rows = (int64_t)B * q_seq * H;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)(kv_seq > 0 ? kv_seq : 1));
    if (!w) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t row = 0; row < n_rows; ++row) {
      if (!w) continue;
      const int h = (int)(row % H);
      const int64_t bi = row / H;               /* b * q_seq + i */
      const int b = (int)(bi / q_seq);
      const int64_t i = bi % q_seq;
      const int g = h / group;
      const int64_t limit = nonpad[b];           /* padding frontier */
      const int64_t offset = nonpad[b] - q_seq;  /* causal offset */
      const double* qrow = q + row * (int64_t)d;
      double* orow = out + row * (int64_t)dv;
      double m = -INFINITY;
      int any = 0;
      for (int64_t j = 0; j < kv_seq; ++j) {
        const int visible = j < limit && (!is_causal || j <= i + offset);
        w[j] = -INFINITY;
        if (!visible) continue;
        const double* krow = k + (((int64_t)b * kv_seq + j) * Hkv + g) * (int64_t)d;
        double dot = 0.0;
        for (int p = 0; p < d; ++p) dot += qrow[p] * krow[p];
        double s = scale * dot;
        if (softcap != 0.0) s = softcap * tanh(s / softcap);
        w[j] = s;
        if (s > m) m = s;
        any = 1;
      }
      for (int c = 0; c < dv; ++c) orow[c] = 0.0;
      if (!any) continue;
      double l = 0.0;
      for (int64_t j = 0; j < kv_seq; ++j) {
        w[j] = w[j] == -INFINITY ? 0.0 : exp(w[j] - m);
        l += w[j];
      }
      for (int64_t j = 0; j < kv_seq; ++j) {
        if (w[j] == 0.0) continue;
        const double* vrow = v + (((int64_t)b * kv_seq + j) * Hkv + g) * (int64_t)dv;
        for (int c = 0; c < dv; ++c) orow[c] += (w[j] / l) * vrow[c];
      }
    }
    free(w);
  }
  return failed ? ORACLE_OOM : ORACLE_OK;
}

/* Threads OpenMP would use by default (reported with CPU timings). */
int pva_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
