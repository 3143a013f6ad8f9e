/*
 * oracle.c -- fp64 reference for the SP-region hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain nested loops, one thread,
 * no blocking or fusion beyond what the definitions state, so each step can
 * be checked against the pages by eye.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* Scalar conversions                                                        */
/* ======================================================================== */

double orc_f64_from_bf16(uint16_t b) {
  /* bf16 is the top half of an IEEE binary32; widening is exact. */
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t orc_bf16_from_f64(double x) {
  /* Round a double to bf16 (8 significant bits, binary32 exponent range)
   * with round-to-nearest-even in ONE step.  Going through binary32 first
   * would round twice. */
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  double ax = fabs(x);
  /* Halfway between the largest finite bf16, (2 - 2^-7) * 2^127, and 2^128:
   * from here on RNE gives infinity (2^128 has the even significand). */
  if (ax >= ldexp(2.0 - ldexp(1.0, -8), 127)) return (uint16_t)(sign | 0x7F80u);
  double r;
  if (ax < ldexp(1.0, -126)) {
    /* subnormal bf16: fixed spacing 2^-133 */
    r = ldexp(nearbyint(ldexp(ax, 133)), -133);
  } else {
    int e;
    double m = frexp(ax, &e);                  /* ax = m * 2^e, m in [0.5, 1) */
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8);  /* 8 significant bits, RNE */
  }
  /* r has at most 8 significant bits and lies in binary32 range, so the
   * conversion below is exact and the top 16 bits are the bf16 pattern. */
  float f = (float)r;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (uint16_t)(u >> 16));
}

int32_t orc_elem_bytes(int32_t dtype) {
  switch (dtype) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_F64: return 8;
    default: return 0;
  }
}

double orc_load(int32_t dtype, const void* base, int64_t idx) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[idx];
    case ORC_BF16: return orc_f64_from_bf16(((const uint16_t*)base)[idx]);
    default: return ((const double*)base)[idx];
  }
}

void orc_store(int32_t dtype, void* base, int64_t idx, double v) {
  switch (dtype) {
    case ORC_F32: ((float*)base)[idx] = (float)v; break; /* C conversion: RNE */
    case ORC_BF16: ((uint16_t*)base)[idx] = orc_bf16_from_f64(v); break;
    default: ((double*)base)[idx] = v; break;
  }
}

/* ======================================================================== */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel Random Numbers: As  */
/* Easy as 1, 2, 3", SC'11).  Each round multiplies counter words 0 and 2 by */
/* the two round multipliers, keeps both halves of each 64-bit product and  */
/* mixes them with the other two words and the round key; the key is bumped */
/* by the two Weyl constants between rounds.                                 */
/* ======================================================================== */

static const uint32_t ORC_PHILOX_M0 = 0xD2511F53u;
static const uint32_t ORC_PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t ORC_PHILOX_W0 = 0x9E3779B9u;
static const uint32_t ORC_PHILOX_W1 = 0xBB67AE85u;

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += ORC_PHILOX_W0;
      k1 += ORC_PHILOX_W1;
    }
    uint64_t prod0 = (uint64_t)ORC_PHILOX_M0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)ORC_PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

uint32_t orc_mask_word(uint64_t seed, uint64_t g) {
  uint64_t q = g >> 2;
  uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[g & 3u];
}

uint32_t orc_keep_threshold(double p) {
  /* p < 1 so the product is below 2^32 */
  return (uint32_t)floor(p * 4294967296.0);
}

uint8_t orc_keep(uint64_t seed, uint32_t thr, uint64_t g) {
  return orc_mask_word(seed, g) >= thr ? 1u : 0u;
}

/* ======================================================================== */
/* Forward: reduce -> dropout -> residual add -> norm                        */
/* ======================================================================== */

static int orc_check_problem(const orc_problem* pr) {
  if (!pr) return -1;
  if (pr->T < 1 || pr->j < 0 || pr->j >= pr->T) return -2;
  if (pr->nshards < 1 || pr->j + pr->nshards > pr->T) return -3;
  if (pr->S < 0 || pr->B < 0 || pr->H < 1) return -4;
  if (pr->S % pr->T != 0) return -5; /* contiguous equal split */
  if (orc_elem_bytes(pr->dtype) == 0) return -6;
  if (pr->norm != ORC_RMS && pr->norm != ORC_LN) return -7;
  if (!(pr->p >= 0.0 && pr->p < 1.0)) return -8;
  if (!(pr->eps > 0.0)) return -9;
  return 0;
}

void orc_fwd_row(const orc_problem* pr, int64_t grow, const void* const* prow,
                 const void* res_row, const void* gamma, const void* beta,
                 void* h_row, void* y_row, uint8_t* mask_row, double* rstd,
                 double* mean, double* h_exact, double* y_exact) {
  const int64_t H = pr->H;
  const int32_t dt = pr->dtype;
  const uint32_t thr = orc_keep_threshold(pr->p);
  double* h = (double*)malloc((size_t)H * sizeof(double));

  for (int64_t c = 0; c < H; ++c) {
    /* (1) reduce: Y^(j) = sum over t = 0..T-1 of P_t, in rank order */
    double y = 0.0;
    for (int32_t t = 0; t < pr->T; ++t) y += orc_load(dt, prow[t], c);
    /* (2) mask from the counter-based generator at the global element index */
    const uint64_t g = (uint64_t)grow * (uint64_t)H + (uint64_t)c;
    const uint8_t m = orc_keep(pr->seed, thr, g);
    /* (3) inverted dropout, then the residual add */
    const double z = y * (double)m / (1.0 - pr->p);
    const double hx = orc_load(dt, res_row, c) + z;
    /* the residual stream is stored once, rounded to the activation dtype;
     * the norm reads the stored value */
    if (h_exact) h_exact[c] = hx;
    if (mask_row) mask_row[c] = m;
    if (h_row) orc_store(dt, h_row, c, hx);
    h[c] = (dt == ORC_F64) ? hx : (dt == ORC_F32 ? (double)(float)hx : orc_f64_from_bf16(orc_bf16_from_f64(hx)));
  }

  /* (4) norm over the hidden dim of the stored row */
  double mu = 0.0, r;
  if (pr->norm == ORC_LN) {
    for (int64_t c = 0; c < H; ++c) mu += h[c];
    mu /= (double)H;
    double var = 0.0; /* population variance */
    for (int64_t c = 0; c < H; ++c) var += (h[c] - mu) * (h[c] - mu);
    var /= (double)H;
    r = 1.0 / sqrt(var + pr->eps);
  } else {
    double ms = 0.0;
    for (int64_t c = 0; c < H; ++c) ms += h[c] * h[c];
    ms /= (double)H;
    r = 1.0 / sqrt(ms + pr->eps);
  }
  for (int64_t c = 0; c < H; ++c) {
    const double gm = orc_load(dt, gamma, c);
    double yv;
    if (pr->norm == ORC_LN)
      yv = gm * (h[c] - mu) * r + orc_load(dt, beta, c);
    else
      yv = gm * h[c] * r;
    if (y_exact) y_exact[c] = yv;
    if (y_row) orc_store(dt, y_row, c, yv);
  }
  if (rstd) *rstd = r;
  if (mean) *mean = mu;
  free(h);
}

int orc_fwd(const orc_problem* pr, const void* const* partials,
            const void* residual, const void* gamma, const void* beta,
            void* h_out, void* y_out, uint8_t* mask_out, double* rstd_out,
            double* mean_out, double* h_exact, double* y_exact) {
  int err = orc_check_problem(pr);
  if (err) return err;
  if (!partials || !residual || !gamma || (pr->norm == ORC_LN && !beta)) return -10;
  const int64_t R = (pr->S / pr->T) * pr->B;
  const int64_t H = pr->H;
  const int32_t es = orc_elem_bytes(pr->dtype);
  const int64_t rows = R * pr->nshards;
  const void* prow[64];
  if (pr->T > 64) return -11;
  for (int64_t r = 0; r < rows; ++r) {
    const int64_t grow = (int64_t)pr->j * R + r;
    for (int32_t t = 0; t < pr->T; ++t)
      prow[t] = (const char*)partials[t] + (size_t)(grow * H) * es;
    const size_t off = (size_t)(r * H);
    orc_fwd_row(pr, grow, prow, (const char*)residual + off * es, gamma, beta,
                h_out ? (char*)h_out + off * es : NULL,
                y_out ? (char*)y_out + off * es : NULL,
                mask_out ? mask_out + off : NULL,
                rstd_out ? rstd_out + r : NULL, mean_out ? mean_out + r : NULL,
                h_exact ? h_exact + off : NULL, y_exact ? y_exact + off : NULL);
  }
  return 0;
}

/* ======================================================================== */
/* Backward                                                                  */
/* ======================================================================== */
/* Gradient of L with respect to the inputs of the forward above, given the
 * upstream dL/dy (dy) and the gradient flowing along the residual stream
 * (dh_out):
 *   g = gamma * dy
 *   RMS:  xhat = h r,        dh = r (g - xhat mean(g xhat))
 *   LN:   xhat = (h - mu) r, dh = r (g - mean(g) - xhat mean(g xhat))
 *   dH = dh + dh_out
 *   d_residual = dH                       (the add passes its gradient on)
 *   d_sum = dH * M / (1 - p)              (dropout backward uses only M)
 *   dgamma += dy xhat,  dbeta += dy
 * d_sum is the gradient of the reduced sum and therefore of every partial
 * P_t of this shard (the add node copies its gradient to each input). */
void orc_bwd_row(const orc_problem* pr, const void* dy_row, const void* dh_row,
                 const void* h_row, const void* gamma, const uint8_t* mask_row,
                 void* dres_row, void* dsum_row, double* dres_exact,
                 double* dsum_exact, double* dgamma_acc, double* dbeta_acc) {
  const int64_t H = pr->H;
  const int32_t dt = pr->dtype;
  double* h = (double*)malloc((size_t)H * sizeof(double));
  double* xhat = (double*)malloc((size_t)H * sizeof(double));
  double* g = (double*)malloc((size_t)H * sizeof(double));

  for (int64_t c = 0; c < H; ++c) h[c] = orc_load(dt, h_row, c);
  double mu = 0.0, r;
  if (pr->norm == ORC_LN) {
    for (int64_t c = 0; c < H; ++c) mu += h[c];
    mu /= (double)H;
    double var = 0.0;
    for (int64_t c = 0; c < H; ++c) var += (h[c] - mu) * (h[c] - mu);
    var /= (double)H;
    r = 1.0 / sqrt(var + pr->eps);
  } else {
    double ms = 0.0;
    for (int64_t c = 0; c < H; ++c) ms += h[c] * h[c];
    ms /= (double)H;
    r = 1.0 / sqrt(ms + pr->eps);
  }
  double mean_g = 0.0, mean_gx = 0.0;
  for (int64_t c = 0; c < H; ++c) {
    xhat[c] = (h[c] - mu) * r;
    g[c] = orc_load(dt, gamma, c) * orc_load(dt, dy_row, c);
    mean_g += g[c];
    mean_gx += g[c] * xhat[c];
  }
  mean_g /= (double)H;
  mean_gx /= (double)H;
  if (pr->norm != ORC_LN) mean_g = 0.0;

  for (int64_t c = 0; c < H; ++c) {
    double dH = r * (g[c] - mean_g - xhat[c] * mean_gx);
    if (dh_row) dH += orc_load(dt, dh_row, c);
    const double m = mask_row ? (double)mask_row[c] : 1.0;
    const double ds = dH * m / (1.0 - pr->p);
    if (dres_exact) dres_exact[c] = dH;
    if (dsum_exact) dsum_exact[c] = ds;
    if (dres_row) orc_store(dt, dres_row, c, dH);
    if (dsum_row) orc_store(dt, dsum_row, c, ds);
    const double dyv = orc_load(dt, dy_row, c);
    if (dgamma_acc) dgamma_acc[c] += dyv * xhat[c];
    if (dbeta_acc) dbeta_acc[c] += dyv;
  }
  free(h);
  free(xhat);
  free(g);
}

int orc_bwd(const orc_problem* pr, const void* dy, const void* dh_out,
            const void* h_saved, const void* gamma, const uint8_t* mask,
            void* d_residual, void* d_sum, double* dres_exact,
            double* dsum_exact, double* dgamma, double* dbeta) {
  int err = orc_check_problem(pr);
  if (err) return err;
  if (!dy || !h_saved || !gamma) return -10;
  if (!mask && pr->p != 0.0) return -12;
  const int64_t R = (pr->S / pr->T) * pr->B;
  const int64_t H = pr->H;
  const int32_t es = orc_elem_bytes(pr->dtype);
  const int64_t rows = R * pr->nshards;
  if (dgamma) memset(dgamma, 0, (size_t)H * sizeof(double));
  if (dbeta) memset(dbeta, 0, (size_t)H * sizeof(double));
  for (int64_t r = 0; r < rows; ++r) {
    const size_t off = (size_t)(r * H);
    orc_bwd_row(pr, (const char*)dy + off * es,
                dh_out ? (const char*)dh_out + off * es : NULL,
                (const char*)h_saved + off * es, gamma, mask ? mask + off : NULL,
                d_residual ? (char*)d_residual + off * es : NULL,
                d_sum ? (char*)d_sum + off * es : NULL,
                dres_exact ? dres_exact + off : NULL,
                dsum_exact ? dsum_exact + off : NULL, dgamma, dbeta);
  }
  return 0;
}

/* ======================================================================== */
/* Simulated collectives (MiniMind-tron ch.3, §3.2.1 and §3.2.3)             */
/* ======================================================================== */

int orc_reduce_scatter(int32_t T, int64_t n, const double* const* P, int32_t j, double* out) {
  if (T < 1 || n % T != 0 || j < 0 || j >= T) return -1;
  const int64_t m = n / T;
  for (int64_t i = 0; i < m; ++i) {
    double s = 0.0;
    for (int32_t t = 0; t < T; ++t) s += P[t][(int64_t)j * m + i];
    out[i] = s;
  }
  return 0;
}

int orc_all_gather(int32_t T, int64_t m, const double* const* blocks, double* out) {
  if (T < 1 || m < 0) return -1;
  for (int32_t t = 0; t < T; ++t)
    for (int64_t i = 0; i < m; ++i) out[(int64_t)t * m + i] = blocks[t][i];
  return 0;
}

int orc_all_reduce(int32_t T, int64_t n, const double* const* P, double* out) {
  if (T < 1 || n < 0) return -1;
  for (int64_t i = 0; i < n; ++i) {
    double s = 0.0;
    for (int32_t t = 0; t < T; ++t) s += P[t][i];
    out[i] = s;
  }
  return 0;
}

static int32_t orc_mod(int32_t a, int32_t T) { return ((a % T) + T) % T; }

int orc_ring_reduce_scatter(int32_t T, int64_t n, double* const* work, int64_t* sent) {
  if (T < 1 || n % T != 0) return -1;
  const int64_t m = n / T;
  double* msg = (double*)malloc((size_t)(T * m > 0 ? T * m : 1) * sizeof(double));
  for (int32_t t = 0; t < T; ++t) sent[t] = 0;
  /* step k: every rank r sends its running partial of block (r - k) mod T to
   * rank r + 1, which adds it into the same block; all links move at once */
  for (int32_t k = 1; k < T; ++k) {
    for (int32_t r = 0; r < T; ++r) {
      const int32_t b = orc_mod(r - k, T);
      memcpy(msg + (int64_t)r * m, work[r] + (int64_t)b * m, (size_t)m * sizeof(double));
      sent[r] += m;
    }
    for (int32_t r = 0; r < T; ++r) {
      const int32_t b = orc_mod(r - k, T);
      const int32_t dst = orc_mod(r + 1, T);
      for (int64_t i = 0; i < m; ++i) work[dst][(int64_t)b * m + i] += msg[(int64_t)r * m + i];
    }
  }
  free(msg);
  return 0;
}

int orc_ring_reduce_scatter_symbolic(int32_t T, int32_t steps, uint64_t* contrib, uint8_t* used) {
  if (T < 1 || T > 64 || steps < 0 || steps > T - 1) return -1;
  for (int32_t r = 0; r < T; ++r)
    for (int32_t b = 0; b < T; ++b) {
      contrib[r * T + b] = (uint64_t)1 << r;
      used[r * T + b] = 0;
    }
  uint64_t* msg = (uint64_t*)malloc((size_t)T * sizeof(uint64_t));
  for (int32_t k = 1; k <= steps; ++k) {
    for (int32_t r = 0; r < T; ++r) {
      const int32_t b = orc_mod(r - k, T);
      msg[r] = contrib[r * T + b];
      used[r * T + b] = 1;
    }
    for (int32_t r = 0; r < T; ++r) {
      const int32_t b = orc_mod(r - k, T);
      const int32_t dst = orc_mod(r + 1, T);
      contrib[dst * T + b] |= msg[r];
    }
  }
  free(msg);
  return 0;
}

/* ======================================================================== */
/* Layout transforms (LLM Infra Atlas "03 · Sequence Parallelism", §5)       */
/* ======================================================================== */

static int orc_layout_check(int64_t N, int64_t H, int32_t T, int32_t es) {
  if (T < 1 || N < 0 || H < 0 || N % T != 0 || H % T != 0) return -1;
  if (es != 1 && es != 2 && es != 4 && es != 8) return -2;
  return 0;
}

/* out[r][n][c] = in[n][r*Hc + c] */
int orc_sp2hp(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t es) {
  int err = orc_layout_check(N, H, T, es);
  if (err) return err;
  const int64_t Hc = H / T;
  for (int32_t r = 0; r < T; ++r)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t c = 0; c < Hc; ++c)
        memcpy((char*)out + (((int64_t)r * N + n) * Hc + c) * es,
               (const char*)in + (n * H + (int64_t)r * Hc + c) * es, (size_t)es);
  return 0;
}

/* out[n][r*Hc + c] = in[r][n][c] */
int orc_hp2sp(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t es) {
  int err = orc_layout_check(N, H, T, es);
  if (err) return err;
  const int64_t Hc = H / T;
  for (int32_t r = 0; r < T; ++r)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t c = 0; c < Hc; ++c)
        memcpy((char*)out + (n * H + (int64_t)r * Hc + c) * es,
               (const char*)in + (((int64_t)r * N + n) * Hc + c) * es, (size_t)es);
  return 0;
}

/* Rank r holds token rows [r*N/T, (r+1)*N/T) with the full hidden dim.  It
 * splits its rows along hidden into T pieces, sends piece s to rank s, and
 * every rank concatenates what it received along tokens, in rank order. */
int orc_sp2hp_all_to_all(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t es) {
  int err = orc_layout_check(N, H, T, es);
  if (err) return err;
  const int64_t Nl = N / T, Hc = H / T;
  const size_t piece = (size_t)(Nl * Hc * es);
  char* sendbuf = (char*)malloc(piece * (size_t)T * (size_t)T + 1);
  char* recvbuf = (char*)malloc(piece * (size_t)T * (size_t)T + 1);
  /* split: sendbuf[r][s] = rows of rank r, hidden columns of piece s */
  for (int32_t r = 0; r < T; ++r)
    for (int32_t s = 0; s < T; ++s)
      for (int64_t n = 0; n < Nl; ++n)
        memcpy(sendbuf + ((size_t)r * T + s) * piece + (size_t)(n * Hc * es),
               (const char*)in + (((int64_t)r * Nl + n) * H + (int64_t)s * Hc) * es,
               (size_t)(Hc * es));
  /* exchange: rank s receives piece s of every rank r */
  for (int32_t r = 0; r < T; ++r)
    for (int32_t s = 0; s < T; ++s)
      memcpy(recvbuf + ((size_t)s * T + r) * piece, sendbuf + ((size_t)r * T + s) * piece, piece);
  /* cat along tokens in rank order: out[s] = [recv[s][0]; recv[s][1]; ...] */
  for (int32_t s = 0; s < T; ++s)
    for (int32_t r = 0; r < T; ++r)
      memcpy((char*)out + ((size_t)s * T + r) * piece, recvbuf + ((size_t)s * T + r) * piece, piece);
  free(sendbuf);
  free(recvbuf);
  return 0;
}

/* Rank r holds all tokens with hidden piece r.  It splits along tokens into
 * T pieces, sends piece s to rank s, and every rank concatenates what it
 * received along hidden, in rank order; the rank outputs stacked in rank
 * order form [N, H]. */
int orc_hp2sp_all_to_all(const void* in, void* out, int64_t N, int64_t H, int32_t T, int32_t es) {
  int err = orc_layout_check(N, H, T, es);
  if (err) return err;
  const int64_t Nl = N / T, Hc = H / T;
  const size_t piece = (size_t)(Nl * Hc * es);
  char* sendbuf = (char*)malloc(piece * (size_t)T * (size_t)T + 1);
  char* recvbuf = (char*)malloc(piece * (size_t)T * (size_t)T + 1);
  /* split: sendbuf[r][s] = token rows [s*Nl, (s+1)*Nl) of rank r's [N, Hc] */
  for (int32_t r = 0; r < T; ++r)
    for (int32_t s = 0; s < T; ++s)
      memcpy(sendbuf + ((size_t)r * T + s) * piece,
             (const char*)in + (((int64_t)r * N + (int64_t)s * Nl) * Hc) * es, piece);
  for (int32_t r = 0; r < T; ++r)
    for (int32_t s = 0; s < T; ++s)
      memcpy(recvbuf + ((size_t)s * T + r) * piece, sendbuf + ((size_t)r * T + s) * piece, piece);
  /* cat along hidden: out rows of rank s, columns [r*Hc, (r+1)*Hc) from r */
  for (int32_t s = 0; s < T; ++s)
    for (int32_t r = 0; r < T; ++r)
      for (int64_t n = 0; n < Nl; ++n)
        memcpy((char*)out + (((int64_t)s * Nl + n) * H + (int64_t)r * Hc) * es,
               recvbuf + ((size_t)s * T + r) * piece + (size_t)(n * Hc * es),
               (size_t)(Hc * es));
  free(sendbuf);
  free(recvbuf);
  return 0;
}

/* ======================================================================== */
/* Helpers for the bindings                                                  */
/* ======================================================================== */

void orc_norm_stats_row(const orc_problem* pr, const void* h_row, double* rstd, double* mean) {
  const int64_t H = pr->H;
  double mu = 0.0;
  if (pr->norm == ORC_LN) {
    for (int64_t c = 0; c < H; ++c) mu += orc_load(pr->dtype, h_row, c);
    mu /= (double)H;
  }
  double v = 0.0;
  for (int64_t c = 0; c < H; ++c) {
    const double d = orc_load(pr->dtype, h_row, c) - mu;
    v += d * d;
  }
  v /= (double)H;
  if (rstd) *rstd = 1.0 / sqrt(v + pr->eps);
  if (mean) *mean = mu;
}

void orc_bf16_from_f64_array(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_f64(x[i]);
}

void orc_f64_from_bf16_array(const uint16_t* x, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_from_bf16(x[i]);
}

void orc_mask_range(uint64_t seed, double p, uint64_t g0, int64_t n, uint8_t* out) {
  const uint32_t thr = orc_keep_threshold(p);
  for (int64_t i = 0; i < n; ++i) out[i] = orc_keep(seed, thr, g0 + (uint64_t)i);
}
