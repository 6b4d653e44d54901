/*
 * mca_oracle.c -- fp64 CPU oracle of the FLASH mixed-chunk attention forward core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (plain definition, no blocking, fusion or reordering beyond
 * what the definition states), for every batch element b:
 *
 *  (1) four per-dimension affine maps of the shared Z
 *        T_k[t, :] = Z[t, :] * gamma[k, :] + beta[k, :],   k = 0 quad_q, 1 quad_k,
 *                                                          2 lin_q,  3 lin_k
 *      -- "FLASH: Possibly the Most Interesting Efficient Transformer Design
 *         Recently", section "Weak Attention", eq. (relu-att): Q and K are
 *         simple affine transforms of Z, like gamma/beta in Layer Norm; section
 *         "Mixed Chunk": four such transforms give Q^quad, K^quad, Q^lin, K^lin.
 *
 *  (2) the sequence is cut into G = n / C non-overlapping chunks of C tokens
 *      (same page, "Mixed Chunk", first paragraph; C must divide n).
 *
 *  (3) intra-chunk quadratic attention, for token i of chunk g
 *        quad[i, :] = sum_j relu( T_0[i] . T_1[j] / C )^2 * V[j, :]
 *      with j over the tokens of chunk g, and j <= i in causal mode (the strict
 *      upper triangle of each chunk's score matrix is masked).
 *      -- same page, "Mixed Chunk", equation for V-hat^quad_g and the sentence
 *         on masking the upper triangle for a decoder.  The scale is taken as
 *         relu(x / C)^2, i.e. the appendix form relu(x/n)^2 of "Weak Attention"
 *         applied to a chunk of length C.
 *
 *  (4) global linear attention through per-chunk states
 *        state_h = sum_{t in chunk h} T_3[t]^T V[t, :]                  (s x e)
 *      non-causal:  glob[i, :] = T_2[i] . (sum over all chunks h of state_h) / n
 *      causal:      glob[i, :] = T_2[i] . (sum over chunks h < g of state_h) / n
 *      -- same page, "Mixed Chunk", the non-causal equation for V-hat^lin_g and
 *         its cumsum (decoder) form; the sum over h < g is exclusive, so chunk 0
 *         has no global term in causal mode; the normaliser is 1/n in both
 *         modes.
 *
 *  (5) gate:  O[i, :] = U[i, :] * (quad[i, :] + glob[i, :])
 *      -- same page, "Mixed Chunk", final equation for O_g (W_o is applied
 *         outside this core).
 *
 * Variants (the *_ex entry points), for where the page's own formulas differ
 * from the reading above ("Mixed Chunk", the equations for V-hat^quad_g and
 * the decoder form of V-hat^lin_g; "Extended Thoughts", the remark on the
 * decoder's normalisation factor):
 *   quad_scale  the weight is quad_scale * relu(T_0[i] . T_1[j])^2; the page's
 *               1/(cs) relu^2(Q K^T) is quad_scale = 1/(C s), and the default
 *               relu(x / C)^2 above is quad_scale = 1/C^2.
 *   lin_norm    0: the global term is divided by n (as above);
 *               1: by the number of tokens its sum covers -- g*C for chunk g
 *                  (counted from 0) in causal mode, which is the decoder
 *                  equation's 1/((g-1)c) with chunks counted from 1, and n
 *                  otherwise; chunk 0's causal sum is empty, so its term is 0;
 *               2: by t+1 for the token at position t (counted from 0) of its
 *                  sequence, i.e. by its position counted from 1 ("the sum of
 *                  the first t items should be divided by t");
 *               3: no global term at all -- with C = n this is the
 *                  quadratic-only model of "Weak Attention" (FLASH-Quad:
 *                  relu(q.k / n)^2 over the whole sequence, masked for a
 *                  decoder).
 *
 * All arithmetic is fp64.  Arrays are row-major and contiguous:
 *   Z[B][n][s], V[B][n][e], U[B][n][e], gamma[4][s], beta[4][s], O[B][n][e].
 *
 * Return codes: 0 ok, -1 bad arguments (non-positive sizes, C not dividing n,
 * NULL pointers, s > 4096, a negative or non-finite quad_scale, an unknown
 * lin_norm), -2 out of host memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double relu(double x) { return x > 0.0 ? x : 0.0; }

/* (1): T_k[t, :] for one token t of batch element b. */
static void affine_row(const double *Z, const double *gamma, const double *beta,
                       int s, int64_t row, int k, double *out) {
  const double *z = Z + row * (int64_t)s;
  for (int c = 0; c < s; ++c) out[c] = z[c] * gamma[k * s + c] + beta[k * s + c];
}

static double dot(const double *a, const double *b, int s) {
  double acc = 0.0;
  for (int c = 0; c < s; ++c) acc += a[c] * b[c];
  return acc;
}

/* (4): state_h = sum over the C tokens of chunk h of T_3[t]^T V[t, :]; result
 * written to st[s][e] (overwritten). */
static void chunk_state(const double *Z, const double *V, const double *gamma,
                        const double *beta, int b, int n, int s, int e, int C, int h,
                        double *st, double *tk) {
  memset(st, 0, sizeof(double) * (size_t)s * (size_t)e);
  for (int j = 0; j < C; ++j) {
    int64_t row = (int64_t)b * n + (int64_t)h * C + j;
    affine_row(Z, gamma, beta, s, row, 3, tk);
    const double *v = V + row * (int64_t)e;
    for (int a = 0; a < s; ++a) {
      double ka = tk[a];
      double *sr = st + (size_t)a * e;
      for (int c = 0; c < e; ++c) sr[c] += ka * v[c];
    }
  }
}

/* (3) + (4) + (5) for one token: row = b*n + g*C + i.  `glob_state` is the
 * state sum the global term reads for this token's chunk (already chosen by
 * the caller per causal / non-causal).  Writes O[row, :] into out[e]. */
static void output_row(const double *Z, const double *V, const double *U,
                       const double *gamma, const double *beta, const double *glob_state,
                       int b, int n, int s, int e, int C, int causal, int g, int i,
                       double *out, double *q0, double *k1, double *q2) {
  int64_t row = (int64_t)b * n + (int64_t)g * C + i;
  affine_row(Z, gamma, beta, s, row, 0, q0);
  affine_row(Z, gamma, beta, s, row, 2, q2);
  for (int c = 0; c < e; ++c) out[c] = 0.0;
  /* (3) intra-chunk relu^2 attention */
  int jmax = causal ? i : C - 1;
  for (int j = 0; j <= jmax; ++j) {
    int64_t krow = (int64_t)b * n + (int64_t)g * C + j;
    affine_row(Z, gamma, beta, s, krow, 1, k1);
    double r = relu(dot(q0, k1, s) / (double)C);
    double w = r * r;
    const double *v = V + krow * (int64_t)e;
    for (int c = 0; c < e; ++c) out[c] += w * v[c];
  }
  /* (4) global linear attention: T_2[row] . state / n */
  for (int a = 0; a < s; ++a) {
    double qa = q2[a] / (double)n;
    const double *sr = glob_state + (size_t)a * e;
    for (int c = 0; c < e; ++c) out[c] += qa * sr[c];
  }
  /* (5) gate */
  const double *u = U + row * (int64_t)e;
  for (int c = 0; c < e; ++c) out[c] *= u[c];
}

/* The variants: the divisor of the global term of token i of chunk g. */
static double lin_factor(int lin_norm, int causal, int n, int C, int g, int i) {
  if (lin_norm == 1) {
    if (!causal) return 1.0 / (double)n;
    return g > 0 ? 1.0 / ((double)g * (double)C) : 0.0; /* chunk 0: empty sum */
  }
  if (lin_norm == 2) return 1.0 / ((double)g * (double)C + (double)i + 1.0);
  if (lin_norm == 3) return 0.0; /* no global term */
  return 1.0 / (double)n;
}

/* output_row with the variant weight quad_scale * relu(q . k)^2 and divisor
 * lin_factor(...). */
static void output_row_ex(const double *Z, const double *V, const double *U,
                          const double *gamma, const double *beta, const double *glob_state,
                          int b, int n, int s, int e, int C, int causal, int g, int i,
                          double quad_scale, int lin_norm, double *out, double *q0,
                          double *k1, double *q2) {
  int64_t row = (int64_t)b * n + (int64_t)g * C + i;
  affine_row(Z, gamma, beta, s, row, 0, q0);
  affine_row(Z, gamma, beta, s, row, 2, q2);
  for (int c = 0; c < e; ++c) out[c] = 0.0;
  int jmax = causal ? i : C - 1;
  for (int j = 0; j <= jmax; ++j) {
    int64_t krow = (int64_t)b * n + (int64_t)g * C + j;
    affine_row(Z, gamma, beta, s, krow, 1, k1);
    double r = relu(dot(q0, k1, s));
    double w = quad_scale * r * r;
    const double *v = V + krow * (int64_t)e;
    for (int c = 0; c < e; ++c) out[c] += w * v[c];
  }
  double f = lin_factor(lin_norm, causal, n, C, g, i);
  for (int a = 0; a < s; ++a) {
    double qa = q2[a] * f;
    const double *sr = glob_state + (size_t)a * e;
    for (int c = 0; c < e; ++c) out[c] += qa * sr[c];
  }
  const double *u = U + row * (int64_t)e;
  for (int c = 0; c < e; ++c) out[c] *= u[c];
}

/* Which formula a driver applies: NULL = the definition at the top. */
struct variant {
  double quad_scale;
  int lin_norm;
};

static void row_of(const double *Z, const double *V, const double *U, const double *gamma,
                   const double *beta, const double *glob_state, int b, int n, int s, int e,
                   int C, int causal, int g, int i, const struct variant *v, double *out,
                   double *q0, double *k1, double *q2) {
  if (v)
    output_row_ex(Z, V, U, gamma, beta, glob_state, b, n, s, e, C, causal, g, i,
                  v->quad_scale, v->lin_norm, out, q0, k1, q2);
  else
    output_row(Z, V, U, gamma, beta, glob_state, b, n, s, e, C, causal, g, i, out, q0, k1, q2);
}

static int check_variant(double quad_scale, int lin_norm) {
  if (!(quad_scale >= 0.0) || !isfinite(quad_scale)) return -1;
  if (lin_norm < 0 || lin_norm > 3) return -1;
  return 0;
}

static int check_args(const void *Z, const void *V, const void *U, const void *gamma,
                      const void *beta, int B, int n, int s, int e, int C) {
  if (!Z || !V || !U || !gamma || !beta) return -1;
  if (B <= 0 || n <= 0 || s <= 0 || e <= 0 || C <= 0) return -1;
  if (C > n || n % C != 0) return -1;
  if (s > 4096) return -1; /* per-token scratch lives on the stack */
  return 0;
}

/* Whole output O[B][n][e].  nthreads <= 0 means the OpenMP default. */
static int forward_impl(const double *Z, const double *V, const double *U,
                        const double *gamma, const double *beta, double *O, int B, int n,
                        int s, int e, int C, int causal, const struct variant *var,
                        int nthreads) {
  if (check_args(Z, V, U, gamma, beta, B, n, s, e, C) || !O) return -1;
  const int G = n / C;
  const size_t se = (size_t)s * (size_t)e;
  /* glob[b][g] = the state sum chunk g reads, (4). */
  double *states = (double *)malloc(sizeof(double) * se * (size_t)G);
  double *glob = (double *)malloc(sizeof(double) * se * (size_t)G);
  if (!states || !glob) {
    free(states);
    free(glob);
    return -2;
  }
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  for (int b = 0; b < B; ++b) {
    /* per-chunk states */
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < G; ++h) {
      double tk[s];
      chunk_state(Z, V, gamma, beta, b, n, s, e, C, h, states + se * h, tk);
    }
    /* the sum each chunk's global term reads */
    for (int g = 0; g < G; ++g) {
      double *dst = glob + se * g;
      memset(dst, 0, sizeof(double) * se);
      int hend = causal ? g : G; /* causal: h < g (exclusive); else all h */
      for (int h = 0; h < hend; ++h) {
        const double *src = states + se * h;
        for (size_t x = 0; x < se; ++x) dst[x] += src[x];
      }
    }
    /* every output row */
#pragma omp parallel for schedule(dynamic)
    for (int g = 0; g < G; ++g) {
      double q0[s], k1[s], q2[s];
      for (int i = 0; i < C; ++i) {
        int64_t row = (int64_t)b * n + (int64_t)g * C + i;
        row_of(Z, V, U, gamma, beta, glob + se * g, b, n, s, e, C, causal, g, i, var,
               O + row * (int64_t)e, q0, k1, q2);
      }
    }
  }
  free(states);
  free(glob);
  return 0;
}

int mca_oracle_forward(const double *Z, const double *V, const double *U,
                       const double *gamma, const double *beta, double *O, int B, int n,
                       int s, int e, int C, int causal, int nthreads) {
  return forward_impl(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, NULL, nthreads);
}

/* The variants (see the top of this file). */
int mca_oracle_forward_ex(const double *Z, const double *V, const double *U,
                          const double *gamma, const double *beta, double *O, int B, int n,
                          int s, int e, int C, int causal, double quad_scale, int lin_norm,
                          int nthreads) {
  if (check_variant(quad_scale, lin_norm)) return -1;
  struct variant v = {quad_scale, lin_norm};
  return forward_impl(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, &v, nthreads);
}

/* Selected output rows only.  rows[r] is a flat token index b*n + t; the
 * result for rows[r] goes to Orows[r][0..e).  Same definition as above: the
 * state sum a row reads is built from the chunk states of its own batch
 * element, chunk by chunk, up to the row's chunk (causal) or over all chunks
 * (non-causal). */
static int rows_impl(const double *Z, const double *V, const double *U, const double *gamma,
                     const double *beta, int B, int n, int s, int e, int C, int causal,
                     int nrows, const int64_t *rows, double *Orows, const struct variant *var,
                     int nthreads) {
  if (check_args(Z, V, U, gamma, beta, B, n, s, e, C) || !rows || !Orows || nrows < 0)
    return -1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= (int64_t)B * n) return -1;
  const int G = n / C;
  const size_t se = (size_t)s * (size_t)e;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  double *states = (double *)malloc(sizeof(double) * se * (size_t)G);
  double *acc = (double *)malloc(sizeof(double) * se);
  if (!states || !acc) {
    free(states);
    free(acc);
    return -2;
  }
  for (int b = 0; b < B; ++b) {
    /* which chunks of this batch element hold requested rows */
    int gmax = -1;
    for (int r = 0; r < nrows; ++r)
      if (rows[r] / n == b) {
        int g = (int)((rows[r] % n) / C);
        if (g > gmax) gmax = g;
      }
    if (gmax < 0) continue;
    int hneed = causal ? gmax : G - 1; /* highest chunk whose state is read */
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h <= hneed; ++h) {
      double tk[s];
      chunk_state(Z, V, gamma, beta, b, n, s, e, C, h, states + se * h, tk);
    }
    for (int g = 0; g <= gmax; ++g) {
      int any = 0;
      for (int r = 0; r < nrows; ++r)
        if (rows[r] / n == b && (int)((rows[r] % n) / C) == g) any = 1;
      if (!any) continue;
      memset(acc, 0, sizeof(double) * se);
      int hend = causal ? g : G;
      for (int h = 0; h < hend; ++h) {
        const double *src = states + se * h;
        for (size_t x = 0; x < se; ++x) acc[x] += src[x];
      }
#pragma omp parallel for schedule(dynamic)
      for (int r = 0; r < nrows; ++r) {
        if (rows[r] / n != b || (int)((rows[r] % n) / C) != g) continue;
        double q0[s], k1[s], q2[s];
        int i = (int)((rows[r] % n) % C);
        row_of(Z, V, U, gamma, beta, acc, b, n, s, e, C, causal, g, i, var,
               Orows + (int64_t)r * e, q0, k1, q2);
      }
    }
  }
  free(states);
  free(acc);
  return 0;
}

int mca_oracle_rows(const double *Z, const double *V, const double *U,
                    const double *gamma, const double *beta, int B, int n, int s, int e,
                    int C, int causal, int nrows, const int64_t *rows, double *Orows,
                    int nthreads) {
  return rows_impl(Z, V, U, gamma, beta, B, n, s, e, C, causal, nrows, rows, Orows, NULL,
                   nthreads);
}

int mca_oracle_rows_ex(const double *Z, const double *V, const double *U,
                       const double *gamma, const double *beta, int B, int n, int s, int e,
                       int C, int causal, double quad_scale, int lin_norm, int nrows,
                       const int64_t *rows, double *Orows, int nthreads) {
  if (check_variant(quad_scale, lin_norm)) return -1;
  struct variant v = {quad_scale, lin_norm};
  return rows_impl(Z, V, U, gamma, beta, B, n, s, e, C, causal, nrows, rows, Orows, &v,
                   nthreads);
}

int mca_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
