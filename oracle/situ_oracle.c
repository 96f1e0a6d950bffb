/*
 * situ_oracle.c -- FP64 CPU oracle for the SiTU-GLU expert feed-forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement
 * of what the GPU library computes.  It is built into its own shared object and
 * may be loaded only by the test suite, by the package's smoke check and by the
 * benchmark's CPU-baseline leg.  The GPU library never links, loads or calls it,
 * and it shares no code, header, table or helper with the GPU library.
 *
 * Sources (web pages on SiTU-GLU, cited by title and section):
 *   [problem]  "SiTU-GLU" problem page (ai-engineer-exhaustive.pages.dev, Kimi K3):
 *              "Theory" formula, "Implementation order", "A scalar example",
 *              "Requirements", "Constraints".
 *   [bound]    "Kimi K3 - Bound the up branch" (atlas.klimoza.dev): the up-branch
 *              formula, and its code excerpts of the activation module
 *              (SituAndMul) and the expert MLP (KimiBlockSparseMLP).
 *   [dense]    "DenseFFN and SituGLU - Docs - Kimi K3 from Scratch": "SiTU-GLU: one
 *              split, two softly bounded branches" and "Two linear maps and a
 *              guarded compiled branch".
 *   [chapter]  "SiTU-GLU" architecture chapter (mkdocs.reaper.mx, in French): the
 *              boxed SiTU-GLU equation of "La construction de SiTU-GLU", "Les
 *              valeurs chez Kimi K3", "La borne de sortie".
 *
 * Every value is carried in IEEE double.  Inputs may be given as double, float or
 * bfloat16 bit patterns; all three convert to double exactly.  Nothing is fused,
 * blocked or reordered beyond what the definitions state: each projection is a
 * plain dot product over the input features in ascending order.
 *
 * Parity pins: every function here is pinned by the CPU test suite against values
 * the pages print and against closed forms (worked example, the beta1*beta2 bound,
 * first-order agreement with SwiGLU, the SwiGLU limit, basis-vector projections,
 * brute-force recounts of the expert index).  None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Input element types accepted by the oracle (its own enum; unrelated to the
 * GPU library's dtype codes). */
enum { ORACLE_F64 = 0, ORACLE_BF16 = 1, ORACLE_F32 = 2 };

/* Status codes returned by the oracle. */
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_INDEX = 2 };

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
static double oracle_bf16_to_double(uint16_t v) {
  uint32_t bits = ((uint32_t)v) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double oracle_load(const void* p, int dt, int64_t i) {
  if (dt == ORACLE_F64) return ((const double*)p)[i];
  if (dt == ORACLE_F32) return (double)((const float*)p)[i];
  return oracle_bf16_to_double(((const uint16_t*)p)[i]);
}

static int oracle_dtype_ok(int dt) {
  return dt == ORACLE_F64 || dt == ORACLE_BF16 || dt == ORACLE_F32;
}

/* Soft cap beta * tanh(x / beta): divide by the cap, take tanh, multiply back
 * ([problem] "Implementation order", second bullet; "Why scaled tanh is
 * useful").  A cap of zero or below stands for "no cap" and returns x unchanged,
 * the behaviour of the activation module when its linear_beta is unset ([bound]
 * code excerpt of SituAndMul). */
double oracle_softcap(double x, double beta) {
  if (!(beta > 0.0)) return x;
  return beta * tanh(x / beta);
}

/* Logistic sigmoid 1 / (1 + exp(-g)).  For g < 0 the same value is written as
 * exp(g) / (1 + exp(g)) so that exp never overflows. */
double oracle_sigmoid(double g) {
  if (g >= 0.0) return 1.0 / (1.0 + exp(-g));
  double e = exp(g);
  return e / (1.0 + e);
}

/* Gate branch a = beta1 * tanh(g / beta1) * sigmoid(g).  The sigmoid takes the
 * UNCAPPED gate projection ([problem] "Implementation order", third bullet). */
double oracle_gate_branch(double g, double beta) {
  return oracle_softcap(g, beta) * oracle_sigmoid(g);
}

/* Up branch b = beta2 * tanh(u / beta2) ([bound] page formula; [problem]
 * "Implementation order", fourth bullet). */
double oracle_up_branch(double u, double linear_beta) {
  return oracle_softcap(u, linear_beta);
}

/* One output coordinate h = a(g) * b(u) ([chapter] boxed SiTU-GLU equation;
 * [problem] "Implementation order", last bullet). */
double oracle_situ_pair(double g, double u, double beta, double linear_beta) {
  return oracle_gate_branch(g, beta) * oracle_up_branch(u, linear_beta);
}

/* Standalone activation over rows of a packed [rows, 2I] tensor: the first I
 * columns are the gate projection g, the last I the up projection u ([dense]
 * "one split, two softly bounded branches": chunk(2) along the last dimension;
 * [bound] SituAndMul slices at d = width / 2).  out is [rows, I], row-major. */
int oracle_situ_glu_act(const void* gate_up, int in_dt, double* out, int64_t rows,
                        int64_t I, double beta, double linear_beta) {
  if (!oracle_dtype_ok(in_dt) || rows < 0 || I < 0) return ORACLE_BAD_ARG;
  if (rows > 0 && I > 0 && (gate_up == 0 || out == 0)) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < I; ++j) {
      double g = oracle_load(gate_up, in_dt, r * 2 * I + j);
      double u = oracle_load(gate_up, in_dt, r * 2 * I + I + j);
      out[r * I + j] = oracle_situ_pair(g, u, beta, linear_beta);
    }
  }
  return ORACLE_OK;
}

/* The SiTU-GLU feed-forward of one row.  x_row holds M doubles; w_gate_up is
 * [2I, M] (rows 0..I-1 gate, rows I..2I-1 up), w_down is [M, I]; both use the
 * [out, in] orientation of a bias-free linear map ([dense] "Two linear maps":
 * gate_up_proj M -> 2I, down_proj I -> M).  gu is scratch of 2I doubles. */
static void oracle_ffn_row(const double* x_row, const void* w_gate_up,
                           const void* w_down, int w_dt, int64_t M, int64_t I,
                           double beta, double linear_beta, double* gu,
                           double* h_row, double* y_row) {
  for (int64_t n = 0; n < 2 * I; ++n) {
    double s = 0.0;
    for (int64_t k = 0; k < M; ++k) s += x_row[k] * oracle_load(w_gate_up, w_dt, n * M + k);
    gu[n] = s;
  }
  for (int64_t j = 0; j < I; ++j) h_row[j] = oracle_situ_pair(gu[j], gu[I + j], beta, linear_beta);
  for (int64_t m = 0; m < M; ++m) {
    double s = 0.0;
    for (int64_t j = 0; j < I; ++j) s += h_row[j] * oracle_load(w_down, w_dt, m * I + j);
    y_row[m] = s;
  }
}

/* Dense expert FFN over R rows: gu = x W_gate_up^T, h = SiTU-GLU(gu),
 * y = h W_down^T, all in FP64 with no rounding of gu or h ([dense] forward:
 * packed projection, activation, down projection; [bound] KimiBlockSparseMLP
 * forward, where concatenating the separate gate and up outputs gives the same
 * packed tensor).  x is [R, M]; h_out ([R, I]) may be NULL; y is [R, M]. */
int oracle_ffn_forward(const void* x, int x_dt, const void* w_gate_up,
                       const void* w_down, int w_dt, double* h_out, double* y,
                       int64_t R, int64_t M, int64_t I, double beta,
                       double linear_beta) {
  if (!oracle_dtype_ok(x_dt) || !oracle_dtype_ok(w_dt)) return ORACLE_BAD_ARG;
  if (R < 0 || M <= 0 || I <= 0) return ORACLE_BAD_ARG;
  if (R == 0) return ORACLE_OK;
  if (!x || !w_gate_up || !w_down || !y) return ORACLE_BAD_ARG;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < R; ++r) {
    double* xr = (double*)malloc(sizeof(double) * (size_t)(M + 3 * I));
    if (!xr) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    double* gu = xr + M;
    double* hr = gu + 2 * I;
    for (int64_t k = 0; k < M; ++k) xr[k] = oracle_load(x, x_dt, r * M + k);
    oracle_ffn_row(xr, w_gate_up, w_down, w_dt, M, I, beta, linear_beta, gu, hr, y + r * M);
    if (h_out) memcpy(h_out + r * I, hr, sizeof(double) * (size_t)I);
    free(xr);
  }
  return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* Expert index: a stable counting sort of the n = T * k_eff flat (token, slot)
 * routes by expert id.  offsets[e] .. offsets[e+1]-1 are the positions of expert
 * e's routes in token_index, and within one expert the flat indices ascend.
 * The pages show no router; variable per-expert row counts are what the expert
 * FFN is called on ([dense] "a varying number of expert-token rows"). */
int oracle_moe_build_index(const int32_t* expert_ids, int64_t n, int32_t E,
                           int32_t* offsets, int32_t* token_index) {
  if (n < 0 || E <= 0 || !offsets || (n > 0 && (!expert_ids || !token_index)))
    return ORACLE_BAD_ARG;
  if (n > INT32_MAX) return ORACLE_BAD_ARG;
  for (int32_t e = 0; e <= E; ++e) offsets[e] = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t e = expert_ids[i];
    if (e < 0 || e >= E) return ORACLE_BAD_INDEX;
    offsets[e + 1] += 1;
  }
  for (int32_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  if (!cursor) return ORACLE_BAD_ARG;
  for (int32_t e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t i = 0; i < n; ++i) token_index[cursor[expert_ids[i]]++] = (int32_t)i;
  free(cursor);
  return ORACLE_OK;
}

/* Grouped routed experts: build the expert index, then for every expert e and
 * every route r in its group, gather the token row x[token_index[r] / k_eff],
 * run expert e's SiTU-GLU FFN on it and write the result to flat slot
 * token_index[r] of y ([T * k_eff, M], no combine weights).  Expert weights are
 * stacked: w_gate_up is [E, 2I, M], w_down is [E, M, I]. */
int oracle_moe_grouped_forward(const void* x, int x_dt, const int32_t* expert_ids,
                               const void* w_gate_up, const void* w_down, int w_dt,
                               double* y, int64_t T, int32_t k_eff, int32_t E,
                               int64_t M, int64_t I, double beta, double linear_beta) {
  if (!oracle_dtype_ok(x_dt) || !oracle_dtype_ok(w_dt)) return ORACLE_BAD_ARG;
  if (T < 0 || k_eff <= 0 || E <= 0 || M <= 0 || I <= 0) return ORACLE_BAD_ARG;
  int64_t n = T * (int64_t)k_eff;
  if (n == 0) return ORACLE_OK;
  if (!x || !expert_ids || !w_gate_up || !w_down || !y) return ORACLE_BAD_ARG;
  int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t* token_index = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  if (!offsets || !token_index) {
    free(offsets);
    free(token_index);
    return ORACLE_BAD_ARG;
  }
  int st = oracle_moe_build_index(expert_ids, n, E, offsets, token_index);
  if (st != ORACLE_OK) {
    free(offsets);
    free(token_index);
    return st;
  }
  size_t wgu_elems = (size_t)(2 * I * M), wd_elems = (size_t)(M * I);
  size_t esz = w_dt == ORACLE_F64 ? 8 : (w_dt == ORACLE_F32 ? 4 : 2);
  int bad = 0;
  for (int32_t e = 0; e < E; ++e) {
    const char* wgu_e = (const char*)w_gate_up + (size_t)e * wgu_elems * esz;
    const char* wd_e = (const char*)w_down + (size_t)e * wd_elems * esz;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) {
      int64_t flat = token_index[r];
      int64_t t = flat / k_eff;
      double* xr = (double*)malloc(sizeof(double) * (size_t)(M + 3 * I));
      if (!xr) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      double* gu = xr + M;
      double* hr = gu + 2 * I;
      for (int64_t k = 0; k < M; ++k) xr[k] = oracle_load(x, x_dt, t * M + k);
      oracle_ffn_row(xr, wgu_e, wd_e, w_dt, M, I, beta, linear_beta, gu, hr, y + flat * M);
      free(xr);
    }
  }
  free(offsets);
  free(token_index);
  return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* Partial derivatives of one output coordinate h = a(g) b(u):
 *   dh/dg = b(u) a'(g),  a'(g) = sech^2(g/b1) sigmoid(g)
 *                                + b1 tanh(g/b1) sigmoid(g) (1 - sigmoid(g)),
 *   dh/du = a(g) b'(u),  b'(u) = sech^2(u/b2).
 * (Differentiation of the "Implementation order" steps of the problem page; the
 * chapter's "Pourquoi un plafond doux" section notes that the soft cap keeps these
 * gradients nonzero where a hard clamp would zero them.)  sech^2 is written
 * 1 / cosh^2 and 1 - sigmoid(g) as sigmoid(-g), so neither cancels.  A cap <= 0
 * means no cap: a = g sigmoid(g), a' = sigmoid(g) + g sigmoid(g) sigmoid(-g);
 * b = u, b' = 1. */
void oracle_situ_pair_grad(double g, double u, double beta, double linear_beta, double* dh_dg,
                           double* dh_du) {
  const double sg = oracle_sigmoid(g), sgm = oracle_sigmoid(-g);
  double da;
  if (beta > 0.0) {
    const double c = cosh(g / beta);
    da = sg / (c * c) + beta * tanh(g / beta) * sg * sgm;
  } else {
    da = sg + g * sg * sgm;
  }
  double db = 1.0;
  if (linear_beta > 0.0) {
    const double c = cosh(u / linear_beta);
    db = 1.0 / (c * c);
  }
  *dh_dg = oracle_up_branch(u, linear_beta) * da;
  *dh_du = oracle_gate_branch(g, beta) * db;
}

/* Backward of the dense FFN y = h W_down^T, h = SiTU-GLU(x W_gate_up^T), for a
 * given upstream gradient dy [R, M], in FP64 with no intermediate rounding:
 *   dh    = dy W_down                        [R, I]
 *   dg_j  = dh_j dh/dg(g_j, u_j), du_j = dh_j dh/du(g_j, u_j)   (dgu = [dg, du])
 *   dx    = dgu W_gate_up                    [R, M]
 *   dW_down    = dy^T h                      [M, I]
 *   dW_gate_up = dgu^T x                     [2I, M]
 * dgu_out ([R, 2I]) may be NULL.  Plain loops; the weight gradients sum over the
 * rows in ascending order. */
int oracle_ffn_backward(const void* x, int x_dt, const void* w_gate_up, const void* w_down,
                        int w_dt, const void* dy, int dy_dt, double* dx, double* dw_gate_up,
                        double* dw_down, double* dgu_out, int64_t R, int64_t M, int64_t I,
                        double beta, double linear_beta) {
  if (!oracle_dtype_ok(x_dt) || !oracle_dtype_ok(w_dt) || !oracle_dtype_ok(dy_dt))
    return ORACLE_BAD_ARG;
  if (R < 0 || M <= 0 || I <= 0) return ORACLE_BAD_ARG;
  if (!x || !w_gate_up || !w_down || !dy || !dx || !dw_gate_up || !dw_down) return ORACLE_BAD_ARG;
  double* h = (double*)malloc(sizeof(double) * (size_t)(R * I + 1));
  double* dgu = (double*)malloc(sizeof(double) * (size_t)(R * 2 * I + 1));
  if (!h || !dgu) {
    free(h);
    free(dgu);
    return ORACLE_BAD_ARG;
  }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < R; ++r) {
    double* gu = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    if (!gu) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    for (int64_t n = 0; n < 2 * I; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < M; ++k)
        s += oracle_load(x, x_dt, r * M + k) * oracle_load(w_gate_up, w_dt, n * M + k);
      gu[n] = s;
    }
    for (int64_t j = 0; j < I; ++j) {
      h[r * I + j] = oracle_situ_pair(gu[j], gu[I + j], beta, linear_beta);
      double dhj = 0.0;
      for (int64_t m = 0; m < M; ++m)
        dhj += oracle_load(dy, dy_dt, r * M + m) * oracle_load(w_down, w_dt, m * I + j);
      double pg, pu;
      oracle_situ_pair_grad(gu[j], gu[I + j], beta, linear_beta, &pg, &pu);
      dgu[r * 2 * I + j] = dhj * pg;
      dgu[r * 2 * I + I + j] = dhj * pu;
    }
    for (int64_t k = 0; k < M; ++k) {
      double s = 0.0;
      for (int64_t n = 0; n < 2 * I; ++n)
        s += dgu[r * 2 * I + n] * oracle_load(w_gate_up, w_dt, n * M + k);
      dx[r * M + k] = s;
    }
    free(gu);
  }
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t j = 0; j < I; ++j) {
      double s = 0.0;
      for (int64_t r = 0; r < R; ++r) s += oracle_load(dy, dy_dt, r * M + m) * h[r * I + j];
      dw_down[m * I + j] = s;
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < 2 * I; ++n) {
    for (int64_t k = 0; k < M; ++k) {
      double s = 0.0;
      for (int64_t r = 0; r < R; ++r) s += dgu[r * 2 * I + n] * oracle_load(x, x_dt, r * M + k);
      dw_gate_up[n * M + k] = s;
    }
  }
  if (dgu_out) memcpy(dgu_out, dgu, sizeof(double) * (size_t)(R * 2 * I));
  free(h);
  free(dgu);
  return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* Backward of the grouped experts, for upstream gradients dy [T, k_eff, M] of the
 * per-(token, slot) outputs: every route (t, s) with expert e = expert_ids[t, s]
 * is one row of expert e's dense FFN on x[t], so, routes taken in ascending flat
 * order,
 *   dx[t]         += the dense backward's dx for (x[t], dy[t, s], expert e)
 *   dW_gate_up[e] += dgu^T x[t],   dW_down[e] += dy[t, s]^T h
 * (the dense backward of oracle_ffn_backward, row by row).  dx is [T, M],
 * dw_gate_up [E, 2I, M], dw_down [E, M, I]; all are overwritten. */
int oracle_moe_grouped_backward(const void* x, int x_dt, const int32_t* expert_ids,
                                const void* w_gate_up, const void* w_down, int w_dt,
                                const void* dy, int dy_dt, double* dx, double* dw_gate_up,
                                double* dw_down, int64_t T, int32_t k_eff, int32_t E, int64_t M,
                                int64_t I, double beta, double linear_beta) {
  if (!oracle_dtype_ok(x_dt) || !oracle_dtype_ok(w_dt) || !oracle_dtype_ok(dy_dt))
    return ORACLE_BAD_ARG;
  if (T < 0 || k_eff <= 0 || E <= 0 || M <= 0 || I <= 0) return ORACLE_BAD_ARG;
  if (!x || !expert_ids || !w_gate_up || !w_down || !dy || !dx || !dw_gate_up || !dw_down)
    return ORACLE_BAD_ARG;
  memset(dx, 0, sizeof(double) * (size_t)(T * M));
  memset(dw_gate_up, 0, sizeof(double) * (size_t)(E * 2 * I * M));
  memset(dw_down, 0, sizeof(double) * (size_t)(E * M * I));
  double* gu = (double*)malloc(sizeof(double) * (size_t)(2 * I));
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* dgu = (double*)malloc(sizeof(double) * (size_t)(2 * I));
  if (!gu || !h || !dgu) {
    free(gu);
    free(h);
    free(dgu);
    return ORACLE_BAD_ARG;
  }
  const size_t esz = w_dt == ORACLE_F64 ? 8 : (w_dt == ORACLE_F32 ? 4 : 2);
  int st = ORACLE_OK;
  for (int64_t f = 0; f < T * k_eff && st == ORACLE_OK; ++f) {
    const int64_t t = f / k_eff;
    const int32_t e = expert_ids[f];
    if (e < 0 || e >= E) {
      st = ORACLE_BAD_INDEX;
      break;
    }
    const char* wg = (const char*)w_gate_up + (size_t)e * (size_t)(2 * I * M) * esz;
    const char* wd = (const char*)w_down + (size_t)e * (size_t)(M * I) * esz;
    for (int64_t n = 0; n < 2 * I; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < M; ++k)
        acc += oracle_load(x, x_dt, t * M + k) * oracle_load(wg, w_dt, n * M + k);
      gu[n] = acc;
    }
    for (int64_t j = 0; j < I; ++j) {
      h[j] = oracle_situ_pair(gu[j], gu[I + j], beta, linear_beta);
      double dhj = 0.0;
      for (int64_t m = 0; m < M; ++m)
        dhj += oracle_load(dy, dy_dt, f * M + m) * oracle_load(wd, w_dt, m * I + j);
      double pg, pu;
      oracle_situ_pair_grad(gu[j], gu[I + j], beta, linear_beta, &pg, &pu);
      dgu[j] = dhj * pg;
      dgu[I + j] = dhj * pu;
    }
    for (int64_t k = 0; k < M; ++k) {
      double acc = 0.0;
      for (int64_t n = 0; n < 2 * I; ++n) acc += dgu[n] * oracle_load(wg, w_dt, n * M + k);
      dx[t * M + k] += acc;
    }
    double* dwd_e = dw_down + (size_t)e * (size_t)(M * I);
    for (int64_t m = 0; m < M; ++m)
      for (int64_t j = 0; j < I; ++j) dwd_e[m * I + j] += oracle_load(dy, dy_dt, f * M + m) * h[j];
    double* dwg_e = dw_gate_up + (size_t)e * (size_t)(2 * I * M);
    for (int64_t n = 0; n < 2 * I; ++n)
      for (int64_t k = 0; k < M; ++k) dwg_e[n * M + k] += dgu[n] * oracle_load(x, x_dt, t * M + k);
  }
  free(gu);
  free(h);
  free(dgu);
  return st;
}

/* Combine of a routed layer: out[t, :] = sum over slots s of w[t, s] * y[t, s, :]
 * in slot order, FP64.  The pages' MoE calls each routed and shared expert on its
 * token rows ("SiTU-GLU" chapter, "Ou SiTU-GLU est utilise": 896 routed plus 2
 * shared experts per layer; docs page: DenseFFN is the expert network inside the
 * MoE); the layer output is the router-weighted sum of a token's expert outputs,
 * with the shared experts as extra slots.  y is [T, k_eff, M] (double), w is
 * [T, k_eff] (any accepted input type), out is [T, M]. */
int oracle_moe_combine(const double* y, const void* w, int w_dt, double* out, int64_t T,
                       int32_t k_eff, int64_t M) {
  if (!oracle_dtype_ok(w_dt) || T < 0 || k_eff <= 0 || M <= 0) return ORACLE_BAD_ARG;
  if (T == 0) return ORACLE_OK;
  if (!y || !w || !out) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t m = 0; m < M; ++m) {
      double s = 0.0;
      for (int32_t k = 0; k < k_eff; ++k)
        s += oracle_load(w, w_dt, t * k_eff + k) * y[(t * k_eff + k) * M + m];
      out[t * M + m] = s;
    }
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * MXFP8: the block-scaled 8-bit format of the OCP Microscaling Formats (MX) v1.0
 * specification.  The SiTU-GLU chapter ("Pourquoi un plafond doux", "Ou SiTU-GLU
 * est utilise") motivates the activation's bound by experts that run in MXFP8 /
 * MXFP4; the format is the specification's:
 *   element E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field
 *     0 holds the subnormals m/8 * 2^-6; there are no infinities, and exponent 15
 *     with mantissa 7 is NaN, so the largest magnitude is 1.75 * 2^8 = 448;
 *   scale E8M0: an exponent alone, code c standing for 2^(c - 127) (255 is NaN);
 *   a block of 32 consecutive elements shares one scale X = 2^(floor(log2 amax) - 8),
 *     amax the block's largest magnitude and 8 the largest exponent of E4M3; each
 *     element is stored as v / X rounded to E4M3, magnitudes past 448 clamped to 448.
 * Readings where the specification leaves a choice: rounding is to nearest with
 * ties to the even mantissa; a block of zeros (log2 0 = -inf) and any scale
 * exponent below -127 take the smallest scale 2^-127, exponents above 127 the
 * largest; an element that rounds to zero keeps its sign bit.
 * ------------------------------------------------------------------------- */
double oracle_e4m3_decode(uint32_t code) {
  const uint32_t c = code & 0xFFu;
  const double sign = (c & 0x80u) ? -1.0 : 1.0;
  const int e = (int)((c >> 3) & 0xFu), m = (int)(c & 7u);
  if (e == 15 && m == 7) return NAN;
  if (e == 0) return sign * ldexp((double)m, -9);  /* m/8 * 2^-6 */
  return sign * ldexp(8.0 + m, e - 10);             /* (1 + m/8) * 2^(e-7) */
}

uint32_t oracle_e4m3_encode(double v) {
  const uint32_t s = signbit(v) ? 0x80u : 0u;
  const double a = fabs(v);
  if (isnan(v)) return s | 0x7Fu;
  if (a == 0.0) return s;
  /* The quantum of a's binade (3 mantissa bits); below 2^-6 the subnormal
   * quantum 2^-9.  a / q is exact, so the rounding is the only rounding. */
  int ea;
  frexp(a, &ea);
  int fl = ea - 1; /* floor(log2 a) */
  if (fl < -6) fl = -6;
  const double r = nearbyint(a / ldexp(1.0, fl - 3)) * ldexp(1.0, fl - 3);
  if (r == 0.0) return s;
  if (r >= 448.0) return s | 0x7Eu; /* clamped to the largest magnitude */
  int er;
  frexp(r, &er);
  const int flr = er - 1;
  if (flr < -6) return s | (uint32_t)(r / ldexp(1.0, -9)); /* subnormal: m * 2^-9 */
  const uint32_t mant = (uint32_t)(r / ldexp(1.0, flr - 3)) - 8u;
  return s | ((uint32_t)(flr + 7) << 3) | mant;
}

double oracle_e8m0_decode(uint32_t code) {
  const uint32_t c = code & 0xFFu;
  return c == 255u ? NAN : ldexp(1.0, (int)c - 127);
}

/* Scale code of a block whose largest magnitude is amax. */
uint32_t oracle_mx_scale_code(double amax) {
  if (!(amax > 0.0)) return 0u;
  int e;
  frexp(amax, &e);
  int x = (e - 1) - 8;
  if (x < -127) x = -127;
  if (x > 127) x = 127;
  return (uint32_t)(x + 127);
}

/* MX quantization of a row-major [R, K] tensor (K a multiple of 32): codes
 * [R, K] E4M3, scales [R, K/32] E8M0, block b of row r = columns 32b .. 32b+31. */
int oracle_mx_quantize(const void* src, int dt, int64_t R, int64_t K, uint8_t* codes,
                       uint8_t* scales) {
  if (!oracle_dtype_ok(dt) || R < 0 || K <= 0 || K % 32 != 0) return ORACLE_BAD_ARG;
  if (R == 0) return ORACLE_OK;
  if (!src || !codes || !scales) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < K / 32; ++b) {
      double amax = 0.0;
      for (int64_t i = 0; i < 32; ++i) {
        const double a = fabs(oracle_load(src, dt, r * K + 32 * b + i));
        if (a > amax) amax = a;
      }
      const uint32_t c = oracle_mx_scale_code(amax);
      const double X = oracle_e8m0_decode(c);
      scales[r * (K / 32) + b] = (uint8_t)c;
      for (int64_t i = 0; i < 32; ++i)
        codes[r * K + 32 * b + i] = (uint8_t)oracle_e4m3_encode(oracle_load(src, dt, r * K + 32 * b + i) / X);
    }
  }
  return ORACLE_OK;
}

/* The values an MX tensor stands for: code * scale of its block, in FP64. */
int oracle_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t K,
                         double* out) {
  if (R < 0 || K <= 0 || K % 32 != 0) return ORACLE_BAD_ARG;
  if (R == 0) return ORACLE_OK;
  if (!codes || !scales || !out) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k)
      out[r * K + k] = oracle_e4m3_decode(codes[r * K + k]) * oracle_e8m0_decode(scales[r * (K / 32) + k / 32]);
  return ORACLE_OK;
}

/* MXFP4 (OCP MX v1.0): element E2M1 -- sign, 2 exponent bits (bias 1), 1 mantissa
 * bit; exponent field 0 holds the subnormal 0.5 (m * 2^-1); magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6; no infinities or NaN.  A block of 32 shares the E8M0 scale
 * X = 2^(floor(log2 amax) - 2) (2 = the largest exponent of E2M1); each element is
 * v / X rounded to E2M1 (ties to the even mantissa), magnitudes past 6 clamped.
 * Codes are packed two to a byte, element 2j in the low nibble of byte j (the order
 * the block-scaled MMA reads). */
double oracle_e2m1_decode(uint32_t code) {
  const uint32_t c = code & 0xFu;
  const double sign = (c & 8u) ? -1.0 : 1.0;
  const int e = (int)((c >> 1) & 3u), m = (int)(c & 1u);
  if (e == 0) return sign * 0.5 * m;
  return sign * ldexp(2.0 + m, e - 2); /* (1 + m/2) * 2^(e-1) */
}

uint32_t oracle_e2m1_encode(double v) {
  const uint32_t s = signbit(v) ? 8u : 0u;
  const double a = fabs(v);
  if (isnan(v)) return s | 7u;
  if (a == 0.0) return s;
  int ea;
  frexp(a, &ea);
  int fl = ea - 1;
  if (fl < 0) fl = 0; /* below 1 the subnormal quantum 0.5 */
  const double q = ldexp(1.0, fl - 1);
  const double r = nearbyint(a / q) * q;
  if (r == 0.0) return s;
  if (r >= 6.0) return s | 7u; /* clamped to the largest magnitude */
  if (r < 1.0) return s | 1u;  /* 0.5 */
  int er;
  frexp(r, &er);
  const int flr = er - 1;
  const uint32_t mant = (uint32_t)(r / ldexp(1.0, flr - 1)) - 2u;
  return s | ((uint32_t)(flr + 1) << 1) | mant;
}

/* Scale code of a block of elements whose largest exponent is emax_elem. */
static uint32_t oracle_mx_scale_code_emax(double amax, int emax_elem) {
  if (!(amax > 0.0)) return 0u;
  int e;
  frexp(amax, &e);
  int x = (e - 1) - emax_elem;
  if (x < -127) x = -127;
  if (x > 127) x = 127;
  return (uint32_t)(x + 127);
}

/* MXFP4 quantization of a row-major [R, K] tensor (K a multiple of 32): codes
 * [R, K/2] bytes (two E2M1 codes each), scales [R, K/32] E8M0. */
int oracle_mxfp4_quantize(const void* src, int dt, int64_t R, int64_t K, uint8_t* codes,
                          uint8_t* scales) {
  if (!oracle_dtype_ok(dt) || R < 0 || K <= 0 || K % 32 != 0) return ORACLE_BAD_ARG;
  if (R == 0) return ORACLE_OK;
  if (!src || !codes || !scales) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < K / 32; ++b) {
      double amax = 0.0;
      for (int64_t i = 0; i < 32; ++i) {
        const double a = fabs(oracle_load(src, dt, r * K + 32 * b + i));
        if (a > amax) amax = a;
      }
      const uint32_t c = oracle_mx_scale_code_emax(amax, 2);
      const double X = oracle_e8m0_decode(c);
      scales[r * (K / 32) + b] = (uint8_t)c;
      for (int64_t i = 0; i < 32; i += 2) {
        const uint32_t lo = oracle_e2m1_encode(oracle_load(src, dt, r * K + 32 * b + i) / X);
        const uint32_t hi = oracle_e2m1_encode(oracle_load(src, dt, r * K + 32 * b + i + 1) / X);
        codes[(r * K + 32 * b + i) / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
  return ORACLE_OK;
}

int oracle_mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t K,
                            double* out) {
  if (R < 0 || K <= 0 || K % 32 != 0) return ORACLE_BAD_ARG;
  if (R == 0) return ORACLE_OK;
  if (!codes || !scales || !out) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t byte = codes[(r * K + k) / 2];
      const uint32_t c = (k % 2 == 0) ? (byte & 0xFu) : (uint32_t)(byte >> 4);
      out[r * K + k] = oracle_e2m1_decode(c) * oracle_e8m0_decode(scales[r * (K / 32) + k / 32]);
    }
  return ORACLE_OK;
}

int oracle_e2m1_encode_array(const double* v, int64_t n, uint8_t* out) {
  if (n < 0 || (n > 0 && (!v || !out))) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e2m1_encode(v[i]);
  return ORACLE_OK;
}

/* Elementwise E4M3 encode / decode of arrays (for the tests). */
int oracle_e4m3_encode_array(const double* v, int64_t n, uint8_t* out) {
  if (n < 0 || (n > 0 && (!v || !out))) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_encode(v[i]);
  return ORACLE_OK;
}

int oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
  if (n < 0 || (n > 0 && (!c || !out))) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
  return ORACLE_OK;
}

/* bfloat16 rounding of doubles, to nearest with ties to the even last bit: the
 * cast of h back to the input dtype ([dense] "SiTU-GLU: one split, two softly
 * bounded branches").  bf16 keeps 8 significant bits down to 2^-126 and the
 * fixed quantum 2^-133 below; magnitudes that round past the largest finite value
 * become infinities.  Returned as bit patterns. */
int oracle_round_bf16_array(const double* v, int64_t n, uint16_t* out) {
  if (n < 0 || (n > 0 && (!v || !out))) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    const double a = fabs(v[i]);
    const uint16_t s = signbit(v[i]) ? 0x8000u : 0u;
    if (isnan(v[i])) {
      out[i] = (uint16_t)(s | 0x7FC0u);
      continue;
    }
    double r = a;
    if (a != 0.0 && !isinf(a)) {
      int e;
      frexp(a, &e);
      int fl = e - 1;
      if (fl < -126) fl = -126;
      const double q = ldexp(1.0, fl - 7);
      r = nearbyint(a / q) * q;
    }
    if (r >= ldexp(1.0, 128)) {
      out[i] = (uint16_t)(s | 0x7F80u);
      continue;
    }
    const float f = (float)r; /* exact: r is a bf16 value */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    out[i] = (uint16_t)(s | (uint16_t)((bits >> 16) & 0x7FFFu));
  }
  return ORACLE_OK;
}

/* Number of threads the oracle's parallel loops use. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
