/*
 * qref.c -- the CPU oracle for the Q4_0 / Q8_0 block-quantised products.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; it exists so that tests, the smoke check and the CPU-baseline leg
 * of the bench have an independent, plainly correct reference. It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Everything is computed in f64, in plain loops, in k order, with no blocking
 * or fusion beyond what the definitions state:
 *
 *  - Block format ("Engine and kernels", pooled.run, section "What it runs"):
 *    a block is 32 weights plus one f16 scale d. Q4_0 stores 4-bit quants q
 *    with weight (q - 8) * d, byte j of the block holding element j in its
 *    low nibble and element j + 16 in its high nibble; Q8_0 stores int8 q with
 *    weight q * d.
 *  - Product: the plain matrix-vector definition (one output element owns one
 *    row and loops over the input: "Running LLMs in the browser with
 *    Three.js", section "Expressing the model as TSL compute", the linear
 *    layer), applied to the dequantised weights, per column, plus an optional
 *    residual: y += W x ("Engine and kernels", section "Fewer passes",
 *    accumulate into the residual).
 *  - Fused gate/up: both projections of one input, SiLU of the gate
 *    multiplying the up projection ("Engine and kernels", section "Kernel
 *    families", fused gate/up; "Running LLMs in the browser with Three.js",
 *    section "From GPT-2 to SmolLM2", the gated MLP).
 *  - MoE: for each column, the chosen experts of the stacked [E, rows, cols]
 *    gate/up/down tensors run as gated FFNs, weighted by the routing weights
 *    and summed, plus a shared expert ("Engine and kernels", sections "What
 *    it runs" and "Kernel families", MoE; "A 235B model in a browser window",
 *    section "A mixture of experts is a different animal").
 *  - Repack: GGUF interleaved blocks into separate quant and scale arrays
 *    ("Architecture", section "Memory and caching").
 *  - Sampling: greedy argmax and top-k over f32 logits, lowest index on ties
 *    ("Engine and kernels", sections "Kernel families", sampling, and "Fewer
 *    passes", GPU argmax and top-k).
 *  - MoE router: logits = W_router x per column (f32 router weights, the
 *    f16/bf16 -> f32 conversion of "Architecture", section "Memory and
 *    caching"), top-k experts in the sampling order, routing weights = a
 *    softmax over the selected logits ("Engine and kernels", section "Kernel
 *    families", MoE: router and top-k on the GPU).
 *
 * Pins (tests/test_oracle_pins.py): hand-worked blocks, x = e_j returning
 * dequantised column j, nibble 8 / scale 0 giving zero, linearity in x,
 * brute force on 4x64 matrices built from logical integer weights, the f16
 * decoder against numpy for all 65,536 patterns, SiLU closed forms and MoE
 * reductions to a single FFN.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_Q4_0 2
#define ORACLE_Q8_0 8
#define ORACLE_QK 32

/* ---------------------------------------------------------------- f16 */

/* IEEE 754 binary16 -> binary64: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 is subnormal, exponent 31 is inf/NaN. */
double qref_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* f * 2^-10 * 2^-14 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)f / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

/* ------------------------------------------------------------ dequant */

static int qbytes_per_block(int type) {
  if (type == ORACLE_Q4_0) return 16;
  if (type == ORACLE_Q8_0) return 32;
  return -1;
}

/* Dequantise one row of k weights from its quant bytes and f16 scales. */
int qref_dequant_row(int type, const uint8_t *qrow, const uint16_t *srow, int k,
                     double *w) {
  if (k % ORACLE_QK) return 1;
  int nb = k / ORACLE_QK;
  for (int b = 0; b < nb; ++b) {
    double d = qref_f16_to_f64(srow[b]);
    if (type == ORACLE_Q4_0) {
      const uint8_t *blk = qrow + (size_t)b * 16;
      for (int i = 0; i < 16; ++i) {
        int lo = blk[i] & 0x0f;
        int hi = blk[i] >> 4;
        w[b * 32 + i] = (double)(lo - 8) * d;
        w[b * 32 + 16 + i] = (double)(hi - 8) * d;
      }
    } else if (type == ORACLE_Q8_0) {
      const int8_t *blk = (const int8_t *)(qrow + (size_t)b * 32);
      for (int i = 0; i < 32; ++i) w[b * 32 + i] = (double)blk[i] * d;
    } else {
      return 2;
    }
  }
  return 0;
}

/* -------------------------------------------------------- matrix apply */

typedef struct {
  int type;
  const uint8_t *q;
  const uint16_t *scl;
  int rows, k;
  const uint16_t *x; /* f16 [ncols][k] */
  int ncols;
  const float *y0;   /* f32 [ncols][rows] or NULL */
  double *y;         /* f64 [ncols][rows] */
  double *S;         /* f64 [ncols][rows] or NULL: sum_k |w||x| */
  const int64_t *row_idx; /* NULL: all rows; else the selected rows */
  int64_t nsel;
  int64_t lo, hi;    /* range of output rows (or of selections) */
  double *xd;        /* decoded x, shared read-only */
} mm_job;

static void *mm_worker(void *arg) {
  mm_job *j = (mm_job *)arg;
  double *w = (double *)malloc(sizeof(double) * (size_t)j->k);
  size_t rowbytes = (size_t)(j->k / ORACLE_QK) * (size_t)qbytes_per_block(j->type);
  size_t nsc = (size_t)(j->k / ORACLE_QK);
  int64_t nout = j->row_idx ? j->nsel : j->rows;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    int64_t r = j->row_idx ? j->row_idx[i] : i;
    qref_dequant_row(j->type, j->q + (size_t)r * rowbytes, j->scl + (size_t)r * nsc,
                     j->k, w);
    for (int c = 0; c < j->ncols; ++c) {
      const double *xc = j->xd + (size_t)c * j->k;
      double acc = 0.0, s = 0.0;
      for (int kk = 0; kk < j->k; ++kk) {
        acc += w[kk] * xc[kk];
        s += fabs(w[kk]) * fabs(xc[kk]);
      }
      if (j->y0) acc += (double)j->y0[(size_t)c * j->rows + r];
      j->y[(size_t)c * nout + i] = acc;
      if (j->S) j->S[(size_t)c * nout + i] = s;
    }
  }
  free(w);
  return NULL;
}

static int run_matmul(int type, const void *q, const uint16_t *scl, int rows, int k,
                      const uint16_t *x, int ncols, const float *y0, double *y,
                      double *S, const int64_t *row_idx, int64_t nsel, int nthreads) {
  if (qbytes_per_block(type) < 0) return 2;
  if (k <= 0 || k % ORACLE_QK || rows < 0 || ncols < 0) return 1;
  double *xd = (double *)malloc(sizeof(double) * (size_t)ncols * (size_t)k + 1);
  for (size_t i = 0; i < (size_t)ncols * (size_t)k; ++i) xd[i] = qref_f16_to_f64(x[i]);
  int64_t nout = row_idx ? nsel : rows;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nout < nthreads) nthreads = nout > 0 ? (int)nout : 1;
  mm_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    mm_job *j = &jobs[t];
    j->type = type; j->q = (const uint8_t *)q; j->scl = scl; j->rows = rows; j->k = k;
    j->x = x; j->ncols = ncols; j->y0 = y0; j->y = y; j->S = S;
    j->row_idx = row_idx; j->nsel = nsel; j->xd = xd;
    j->lo = nout * t / nthreads;
    j->hi = nout * (t + 1) / nthreads;
  }
  if (nthreads == 1) {
    mm_worker(&jobs[0]);
  } else {
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, mm_worker, &jobs[t]);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  }
  free(xd);
  return 0;
}

/* y[c][r] = (y0[c][r]) + sum_k w[r][k] x[c][k];  S[c][r] = sum_k |w[r][k]| |x[c][k]|. */
int qref_matmul(int type, const void *q, const uint16_t *scl, int rows, int k,
                const uint16_t *x, int ncols, const float *y0, double *y, double *S,
                int nthreads) {
  return run_matmul(type, q, scl, rows, k, x, ncols, y0, y, S, NULL, 0, nthreads);
}

/* The same, for a list of selected rows only: y and S are [ncols][nsel]. */
int qref_matmul_rows(int type, const void *q, const uint16_t *scl, int rows, int k,
                     const uint16_t *x, int ncols, const float *y0, const int64_t *row_idx,
                     int64_t nsel, double *y, double *S, int nthreads) {
  for (int64_t i = 0; i < nsel; ++i)
    if (row_idx[i] < 0 || row_idx[i] >= rows) return 1;
  return run_matmul(type, q, scl, rows, k, x, ncols, y0, y, S, row_idx, nsel, nthreads);
}

/* --------------------------------------------------------------- SiLU */

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^-z). */
double qref_silu(double z) { return z / (1.0 + exp(-z)); }

/* Fused gate/up: g = Wg x, u = Wu x (f64), h = SiLU(g) * u. All outputs are
 * [ncols][rows]; Sg, Su are the sum_k |w||x| of each projection. */
int qref_ffn_gate_up_silu(int type, const void *qg, const uint16_t *sg, const void *qu,
                          const uint16_t *su, int rows, int k, const uint16_t *x,
                          int ncols, double *h, double *g, double *u, double *Sg,
                          double *Su, int nthreads) {
  int rc = qref_matmul(type, qg, sg, rows, k, x, ncols, NULL, g, Sg, nthreads);
  if (rc) return rc;
  rc = qref_matmul(type, qu, su, rows, k, x, ncols, NULL, u, Su, nthreads);
  if (rc) return rc;
  for (size_t i = 0; i < (size_t)ncols * (size_t)rows; ++i) h[i] = qref_silu(g[i]) * u[i];
  return 0;
}

/* ---------------------------------------------------------------- MoE */

/* SiLU'(z) = sigma(z) (1 + z (1 - sigma(z))), sigma(z) = 1 / (1 + e^-z): the
 * product rule applied to z * sigma(z), with sigma' = sigma (1 - sigma). */
double qref_silu_prime(double z) {
  double s = 1.0 / (1.0 + exp(-z));
  return s * (1.0 + z * (1.0 - s));
}

/* The one critical point of SiLU: SiLU'(z) = sigma(z) f(z) with
 * f(z) = 1 + z (1 - sigma(z)); f > 0 for z >= 0, and on z < 0 f is increasing
 * (f' = (1 - sigma)(1 - z sigma) > 0) from -inf to 1, so it has exactly one
 * root, between -2 and -1 (f(-2) < 0 < f(-1)). Found by bisection. */
static double silu_critical_point(void) {
  double a = -2.0, b = -1.0;
  for (int i = 0; i < 200 && b - a > 0.0; ++i) {
    double m = 0.5 * (a + b);
    if (m == a || m == b) break;
    if (qref_silu_prime(m) < 0.0) a = m; else b = m;
  }
  return 0.5 * (a + b);
}

/* Bound on |h_gpu - h| for one element of a gated FFN whose projections each
 * carry the GEMV tolerance e = 1e-3 * S + 1e-6 (g' = g + dg, |dg| <= eg; the
 * same for u), followed by SiLU * up in f32 and one rounding to f16.
 * SiLU is monotone on each side of its critical point z0, so over the interval
 * [g - eg, g + eg] its extremes lie at the two ends or at z0 (if inside), and
 *   D = max |SiLU(g') - SiLU(g)| = max(|SiLU(g + eg) - SiLU(g)|,
 *                                      |SiLU(g - eg) - SiLU(g)|,
 *                                      |SiLU(z0) - SiLU(g)| if z0 is inside)
 * exactly. With |u'| <= |u| + eu:
 *   |SiLU(g') u' - SiLU(g) u| <= D (|u| + eu) + |SiLU(g)| eu,
 * which to first order is 1e-3 (|SiLU'(g)| |u| Sg + |SiLU(g)| Su). Added: one
 * f16 rounding of the result (2^-11 relative, 2^-24 absolute for subnormals)
 * and 1e-6 relative for the f32 evaluation of SiLU(g) * u. */
double qref_h_bound(double g, double u, double Sg, double Su) {
  static double z0 = 0.0;
  if (z0 == 0.0) z0 = silu_critical_point();
  double eg = 1e-3 * Sg + 1e-6, eu = 1e-3 * Su + 1e-6;
  double sg = qref_silu(g);
  double h = sg * u;
  double D = fmax(fabs(qref_silu(g + eg) - sg), fabs(qref_silu(g - eg) - sg));
  if (g - eg <= z0 && z0 <= g + eg) D = fmax(D, fabs(qref_silu(z0) - sg));
  double prop = D * (fabs(u) + eu) + fabs(sg) * eu;
  return prop + ldexp(fabs(h) + prop, -11) + ldexp(1.0, -24) + 1e-6 * (fabs(h) + prop);
}

typedef struct {
  const void *qg; const uint16_t *sg;
  const void *qu; const uint16_t *su;
  const void *qd; const uint16_t *sd;
} qref_expert;

static size_t mat_qbytes(int type, int rows, int k) {
  return (size_t)rows * (size_t)(k / ORACLE_QK) * (size_t)qbytes_per_block(type);
}
static size_t mat_scales(int rows, int k) { return (size_t)rows * (size_t)(k / ORACLE_QK); }

/* One gated expert on one column: out = D (SiLU(G x) * (U x)).
 * hsrc, if not NULL, replaces h by the given f16 values (the staged check).
 * bnd receives, per output row, the propagated error bound of the expert. */
static int expert_apply(int type, const qref_expert *e, int ffn, int hidden,
                        const uint16_t *xc, const uint16_t *hsrc, double *out,
                        double *bnd, int nthreads) {
  double *g = malloc(sizeof(double) * ffn), *u = malloc(sizeof(double) * ffn);
  double *Sg = malloc(sizeof(double) * ffn), *Su = malloc(sizeof(double) * ffn);
  double *h = malloc(sizeof(double) * ffn), *th = malloc(sizeof(double) * ffn);
  double *w = malloc(sizeof(double) * ffn);
  int rc = qref_ffn_gate_up_silu(type, e->qg, e->sg, e->qu, e->su, ffn, hidden, xc, 1, h,
                                 g, u, Sg, Su, nthreads);
  if (!rc) {
    for (int i = 0; i < ffn; ++i) {
      th[i] = qref_h_bound(g[i], u[i], Sg[i], Su[i]);
      if (hsrc) { h[i] = qref_f16_to_f64(hsrc[i]); th[i] = 0.0; }
    }
    size_t rowbytes = (size_t)(ffn / ORACLE_QK) * (size_t)qbytes_per_block(type);
    for (int r = 0; r < hidden; ++r) {
      qref_dequant_row(type, (const uint8_t *)e->qd + (size_t)r * rowbytes,
                       e->sd + (size_t)r * (ffn / ORACLE_QK), ffn, w);
      double acc = 0.0, b = 0.0;
      for (int i = 0; i < ffn; ++i) {
        acc += w[i] * h[i];
        /* down-GEMV tolerance on the device's h plus the error carried by h */
        b += fabs(w[i]) * (th[i] + 1e-3 * (fabs(h[i]) + th[i]));
      }
      out[r] = acc;
      bnd[r] = b + 1e-6;
    }
  }
  free(g); free(u); free(Sg); free(Su); free(h); free(th); free(w);
  return rc;
}

/* Stacked-expert MoE layer.
 *   ids [ncols][topk] int32, rw [ncols][topk] f32; x [ncols][hidden] f16;
 *   stacks: gate/up [E][ffn][hidden], down [E][hidden][ffn] (quants + scales);
 *   shared: NULL or one more expert of the same shape, added with weight 1.
 *   y [ncols][hidden] f64 = y0 + sum_j rw[c][j] * expert_{ids[c][j]}(x_c) + shared(x_c)
 *   bound [ncols][hidden]: the propagated per-element error bound.
 *   h_in (optional): f16 [ncols][topk + 1][ffn] intermediate h to use instead of
 *   the f64 one, slot topk being the shared expert (staged check).
 *   uniq [ncols*topk]: sorted unique valid ids, padded with -1; *n_uniq its count.
 * Returns 0, or 3 if any id is outside [0, E) (that slot then contributes 0). */
int qref_moe(int type, const void *qg, const uint16_t *sg, const void *qu,
             const uint16_t *su, const void *qd, const uint16_t *sd, int n_expert,
             int ffn, int hidden, const int32_t *ids, const float *rw, int topk,
             const qref_expert *shared, const uint16_t *x, int ncols, const float *y0,
             const uint16_t *h_in, double *y, double *bound, int32_t *uniq,
             int *n_uniq, int nthreads) {
  if (qbytes_per_block(type) < 0) return 2;
  if (ffn % ORACLE_QK || hidden % ORACLE_QK) return 1;
  int bad = 0;
  double *out = malloc(sizeof(double) * hidden), *bnd = malloc(sizeof(double) * hidden);
  for (int c = 0; c < ncols; ++c) {
    const uint16_t *xc = x + (size_t)c * hidden;
    for (int r = 0; r < hidden; ++r) {
      y[(size_t)c * hidden + r] = y0 ? (double)y0[(size_t)c * hidden + r] : 0.0;
      bound[(size_t)c * hidden + r] = 1e-6;
    }
    for (int j = 0; j <= topk; ++j) {
      qref_expert e;
      double wgt;
      if (j < topk) {
        int id = ids[(size_t)c * topk + j];
        if (id < 0 || id >= n_expert) { bad = 1; continue; }
        e.qg = (const uint8_t *)qg + (size_t)id * mat_qbytes(type, ffn, hidden);
        e.sg = sg + (size_t)id * mat_scales(ffn, hidden);
        e.qu = (const uint8_t *)qu + (size_t)id * mat_qbytes(type, ffn, hidden);
        e.su = su + (size_t)id * mat_scales(ffn, hidden);
        e.qd = (const uint8_t *)qd + (size_t)id * mat_qbytes(type, hidden, ffn);
        e.sd = sd + (size_t)id * mat_scales(hidden, ffn);
        wgt = (double)rw[(size_t)c * topk + j];
      } else {
        if (!shared) continue;
        e = *shared;
        wgt = 1.0;
      }
      const uint16_t *hs = h_in ? h_in + ((size_t)c * (topk + 1) + j) * ffn : NULL;
      int rc = expert_apply(type, &e, ffn, hidden, xc, hs, out, bnd, nthreads);
      if (rc) { free(out); free(bnd); return rc; }
      for (int r = 0; r < hidden; ++r) {
        y[(size_t)c * hidden + r] += wgt * out[r];
        bound[(size_t)c * hidden + r] += fabs(wgt) * bnd[r] + 1e-7 * fabs(wgt * out[r]);
      }
    }
  }
  /* sorted unique valid ids (insertion into a sorted list without repeats) */
  int n = 0;
  for (int i = 0; i < ncols * topk; ++i) {
    int id = ids[i];
    if (id < 0 || id >= n_expert) continue;
    int pos = 0;
    while (pos < n && uniq[pos] < id) ++pos;
    if (pos < n && uniq[pos] == id) continue;
    for (int t = n; t > pos; --t) uniq[t] = uniq[t - 1];
    uniq[pos] = id;
    ++n;
  }
  for (int i = n; i < ncols * topk; ++i) uniq[i] = -1;
  *n_uniq = n;
  free(out); free(bnd);
  return bad ? 3 : 0;
}

/* ------------------------------------------------------------- repack */

/* GGUF interleaved blocks (per block: f16 d little endian, then the quant
 * bytes) -> separate quant array [rows][k/32 * qbytes] and scale array
 * [rows][k/32]. The stored quant order is the library's: in every 16-byte
 * group of a block's quants, stored byte 2m + h is GGUF byte m + 8h
 * (m = 0..7, h = 0..1), i.e. the two 8-byte halves interleaved byte by byte.
 * Test infrastructure: this is the oracle's statement of that layout. */
int qref_repack(int type, const uint8_t *gguf, int rows, int k, uint8_t *q_out,
                uint16_t *scl_out) {
  int qb = qbytes_per_block(type);
  if (qb < 0) return 2;
  if (k % ORACLE_QK || rows < 0) return 1;
  int nb = k / ORACLE_QK;
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < nb; ++b) {
      const uint8_t *blk = gguf + ((size_t)r * nb + b) * (size_t)(2 + qb);
      scl_out[(size_t)r * nb + b] = (uint16_t)(blk[0] | (blk[1] << 8));
      uint8_t *dst = q_out + ((size_t)r * nb + b) * (size_t)qb;
      for (int g = 0; g < qb; g += 16)
        for (int m = 0; m < 8; ++m)
          for (int h = 0; h < 2; ++h) dst[g + 2 * m + h] = blk[2 + g + m + 8 * h];
    }
  }
  return 0;
}

/* ----------------------------------------------------------- sampling */

/* Order of the sampling calls ("Engine and kernels", section "Fewer passes":
 * lowest-index tie-breaking, as a CPU loop would do it): a number ranks before
 * NaN; among numbers the larger value ranks first (+0 and -0 are equal); equal
 * values, and two NaNs, rank by the lower index. Returns 1 when element i
 * ranks before element j. */
static int qref_before(const float *v, int64_t i, int64_t j) {
  const float a = v[i], b = v[j];
  const int na = isnan(a) != 0, nb = isnan(b) != 0;
  if (na != nb) return nb;
  if (!na && a != b) return a > b;
  return i < j;
}

/* Greedy argmax of every column of x [ncols][n]: the first-ranked element. */
int qref_argmax(const float *x, int n, int ncols, int32_t *idx, float *val) {
  if (n < 1 || ncols < 1) return 1;
  for (int c = 0; c < ncols; ++c) {
    const float *v = x + (size_t)c * n;
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
      if (qref_before(v, i, best)) best = i;
    idx[c] = (int32_t)best;
    if (val) val[c] = v[best];
  }
  return 0;
}

/* Top-k of every column: k selection passes, each taking the first-ranked
 * element not yet taken; outputs [ncols][k] in rank order. */
int qref_topk(const float *x, int n, int ncols, int k, int32_t *idx, float *val) {
  if (n < 1 || ncols < 1 || k < 1 || k > n) return 1;
  unsigned char *taken = (unsigned char *)malloc((size_t)n);
  if (!taken) return 2;
  for (int c = 0; c < ncols; ++c) {
    const float *v = x + (size_t)c * n;
    memset(taken, 0, (size_t)n);
    for (int r = 0; r < k; ++r) {
      int64_t best = -1;
      for (int64_t i = 0; i < n; ++i)
        if (!taken[i] && (best < 0 || qref_before(v, i, best))) best = i;
      taken[best] = 1;
      idx[(size_t)c * k + r] = (int32_t)best;
      if (val) val[(size_t)c * k + r] = v[best];
    }
  }
  free(taken);
  return 0;
}

/* ---------------------------------------------------------- MoE router */

/* Router logits in f64: logits[c][e] = sum_k w[e][k] * x[c][k] (w f32
 * [E][hidden], x f16 bits [ncols][hidden]), k order; S[c][e] = sum |w||x|. */
int qref_router_logits(const float *w, const uint16_t *x, int E, int hidden, int ncols,
                       double *logits, double *S) {
  if (E < 1 || hidden < 1 || ncols < 1) return 1;
  for (int c = 0; c < ncols; ++c)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0, sa = 0.0;
      for (int k = 0; k < hidden; ++k) {
        const double p = (double)w[(size_t)e * hidden + k] * qref_f16_to_f64(x[(size_t)c * hidden + k]);
        acc += p;
        sa += fabs(p);
      }
      logits[(size_t)c * E + e] = acc;
      if (S) S[(size_t)c * E + e] = sa;
    }
  return 0;
}

/* Softmax of k values in f64: out[i] = exp(v[i] - max) / sum_j exp(v[j] - max). */
int qref_softmax(const float *v, int k, double *out) {
  if (k < 1) return 1;
  double m = v[0];
  for (int i = 1; i < k; ++i)
    if (v[i] > m) m = v[i];
  double sum = 0.0;
  for (int i = 0; i < k; ++i) {
    out[i] = exp((double)v[i] - m);
    sum += out[i];
  }
  for (int i = 0; i < k; ++i) out[i] /= sum;
  return 0;
}
