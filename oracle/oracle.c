/*
 * CPU ORACLE for the DiffusionGemma uniform-state denoise step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is plain, slow, obviously correct C in
 * double precision.  It shares no code with the CUDA path and is never called
 * by it; only the tests, the package's smoke check and the benchmark's CPU
 * baseline run it.
 *
 * What each function computes, and where the pages define it:
 *
 *   or_rmsnorm_bf16 -- the final RMSNorm, w * x * sqrt(D) / (||x||_2 + eps),
 *       cast back to the model dtype (bf16).  "The Annotated DiffusionGemma",
 *       section "RMSNorm"; applied before the tied LM head in "Complete
 *       DiffusionGemma model".  Norm and scaling are taken in fp64 here and
 *       rounded once, to nearest-even, to bf16.
 *
 *   or_stats -- for one canvas position, given its logits z_v = h . W_v (the
 *       tied LM head, "Complete DiffusionGemma model"), the temperature
 *       softmax softmax(z/T) ("Apply temperature"), its entropy
 *       H = -sum_v p_v ln p_v in nats ("Compute entropy"), log Z, the argmax,
 *       and one categorical sample.  The sample is drawn by the Gumbel-max
 *       rule (Gumbel 1954; e.g. Maddison, Tarlow, Minka, "A* Sampling", 2014):
 *       y = argmax_v (z_v/T + G_v), G_v = -ln E_v with E_v i.i.d. Exp(1),
 *       which has the law of a draw from the categorical distribution with
 *       logits z/T, the draw "Denoise, stage, commit, and generate" makes.
 *
 *   or_exp_variates -- the Exp(1) variates E_v of one position.  The
 *       vocabulary is cut into groups of 16 entries, j = v >> 4, and each
 *       group's sixteen i.i.d. Exp(1) variates are drawn in increasing order
 *       by Renyi's representation of exponential order statistics (A. Renyi,
 *       "On the theory of order statistics", 1953): the k-th smallest of n is
 *       E_(k) = E_(k-1) + X_k / (n - k), k = 0 .. n-1, E_(-1) = 0, with
 *       X_k i.i.d. Exp(1); and since the variates are exchangeable, the
 *       slots that receive E_(0), E_(1), ... are a uniformly random
 *       permutation, drawn here one slot at a time without replacement.  With
 *       U(w) = (w + 0.5) 2^-32 for a Philox4x32-10 word w (Salmon et al.,
 *       SC'11), key = canvas seed, step k of group j reads the words of
 *         b = Philox((8 j + k / 2, p, (block<<16)|step, 5)):
 *       X_k = -ln U(b[2 (k & 1)]) and, from w = b[2 (k & 1) + 1],
 *       r = (w (16 - k)) >> 32 (Lemire's multiply-shift), so that E_(k) goes
 *       to the r-th (from 0, in increasing order) slot not yet given a value.
 *       Entries of the last group at or beyond V are simply not used.
 *
 *   or_draw_u32 -- one Philox word for the uniform re-noise ("Keep a
 *       low-entropy prefix and renoise the rest") and the uniform initial
 *       canvas ("Lazy Sampling": the first input is a uniform categorical).
 *       key = canvas seed, counter = (0, p, (block<<16)|step, purpose),
 *       purpose 2 = initial canvas, 4 = re-noise; lane 0.  A word u maps to a
 *       token by Lemire's multiply-shift, (u * V) >> 32.
 *
 * Parity pins for every function are in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_PURPOSE_INIT = 2, OR_PURPOSE_RENOISE = 4, OR_PURPOSE_GUMBEL_ORDER = 5 };

/* ---------------------------------------------------------------- Philox -- */

/* Philox4x32-10: ten rounds of the Philox S-box with the Weyl key schedule. */
void or_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t x[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k[2] = {key[0], key[1]};
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)M0 * x[0];
    uint64_t p1 = (uint64_t)M1 * x[2];
    uint32_t y0 = (uint32_t)(p1 >> 32) ^ x[1] ^ k[0];
    uint32_t y1 = (uint32_t)p1;
    uint32_t y2 = (uint32_t)(p0 >> 32) ^ x[3] ^ k[1];
    uint32_t y3 = (uint32_t)p0;
    x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
    k[0] += W0;
    k[1] += W1;
  }
  memcpy(out, x, sizeof x);
}

uint32_t or_draw_u32(uint64_t seed, uint32_t purpose, int32_t block, int32_t step, int32_t p) {
  uint32_t ctr[4] = {0u, (uint32_t)p, ((uint32_t)block << 16) | (uint32_t)step, purpose};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  or_philox(ctr, key, out);
  return out[0];
}

/* Uniform token in [0, V): Lemire (2019), "Fast random integer generation in an interval". */
int32_t or_uniform_token(uint32_t u, int32_t V) { return (int32_t)(((uint64_t)u * (uint64_t)(uint32_t)V) >> 32); }

/* -------------------------------------------------------------- RMSNorm -- */

/* Round a double to the nearest bfloat16, ties to even: |x| is rounded to a
 * multiple of the bf16 quantum of its binade (2^(e-8) for normals, 2^-133 for
 * subnormals) with nearbyint() in the default round-to-nearest-even mode. */
uint16_t or_bf16_rne(double x) {
  float f;
  uint32_t bits;
  if (isnan(x)) return 0x7FC0u;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs(x);
  if (a == 0.0) return (uint16_t)(neg << 15);
  int e;
  (void)frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
  int q = (e + 126 >= 1) ? e - 8 : -133;
  double rounded = ldexp(nearbyint(ldexp(a, -q)), q);
  f = (float)rounded; /* exact: a bf16 value, or +inf on overflow */
  memcpy(&bits, &f, 4);
  return (uint16_t)((bits >> 16) | (uint32_t)(neg << 15));
}

double or_bf16_value(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/* h[i,:] = bf16( w * r * sqrt(d) / (||r[i,:]||_2 + eps) ), fp64 throughout. */
void or_rmsnorm_bf16(int64_t n_rows, int64_t d, const float* r, const float* w, double eps, uint16_t* h) {
  for (int64_t i = 0; i < n_rows; ++i) {
    const float* x = r + i * d;
    double ss = 0.0;
    for (int64_t k = 0; k < d; ++k) ss += (double)x[k] * (double)x[k];
    double norm = sqrt(ss);
    double sqrt_d = sqrt((double)d);
    for (int64_t k = 0; k < d; ++k) {
      double wk = w ? (double)w[k] : 1.0;
      double val = wk * (double)x[k] * sqrt_d / (norm + eps);
      h[i * d + k] = or_bf16_rne(val);
    }
  }
}

/* ---------------------------------------------------- per-position stats -- */

typedef struct or_pos {
  double logZ;      /* ln sum_v exp(z_v / T)                               */
  double H;         /* -sum_v p_v ln p_v, computed directly                */
  double H_online;  /* the same entropy through the max/sum rescaling form */
  double zmax;      /* max_v z_v / T                                       */
  double zgap;      /* zmax minus the largest z_v / T at another index     */
  double gbest;     /* max_v (z_v / T + G_v)                               */
  double ggap;      /* gbest minus the runner-up perturbed score           */
  int32_t amax;     /* argmax_v z_v / T, lowest index on ties              */
  int32_t y;        /* argmax_v (z_v / T + G_v), lowest index on ties      */
} or_pos;

static double or_unit(uint32_t w) { return ((double)w + 0.5) / 4294967296.0; }

/* E[v] for v in [0, V): the Exp(1) variates of position p's Gumbel draws (see the header). */
void or_exp_variates(uint64_t seed, int32_t block, int32_t step, int32_t p, int64_t V, double* E) {
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  const uint32_t bs = ((uint32_t)block << 16) | (uint32_t)step;
  for (int64_t j = 0; 16 * j < V; ++j) {
    double ek = 0.0;    /* E_(k-1) */
    int taken[16] = {0};
    for (int k = 0; k < 16; ++k) {
      const uint32_t c[4] = {(uint32_t)(8 * j + k / 2), (uint32_t)p, bs, OR_PURPOSE_GUMBEL_ORDER};
      uint32_t b[4];
      or_philox(c, key, b);
      ek += -log(or_unit(b[2 * (k & 1)])) / (double)(16 - k);
      const uint32_t r = (uint32_t)(((uint64_t)b[2 * (k & 1) + 1] * (uint64_t)(16 - k)) >> 32);
      /* the r-th free slot */
      int slot = -1;
      for (int i = 0, seen = 0; i < 16; ++i) {
        if (taken[i]) continue;
        if (seen == (int)r) {
          slot = i;
          break;
        }
        ++seen;
      }
      taken[slot] = 1;
      if (16 * j + slot < V) E[16 * j + slot] = ek;
    }
  }
}

static void or_stats_row(int64_t V, const double* z, double T, uint64_t seed, int32_t block, int32_t step, int32_t p,
                         or_pos* o) {
  /* temperature-scaled logits and their maximum */
  double m = -INFINITY, m2 = -INFINITY;
  int32_t amax = 0;
  for (int64_t v = 0; v < V; ++v) {
    double zp = z[v] / T;
    if (zp > m) {
      m2 = m;
      m = zp;
      amax = (int32_t)v;
    } else if (zp > m2) {
      m2 = zp;
    }
  }
  /* normaliser */
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) S += exp(z[v] / T - m);
  double logZ = m + log(S);
  /* entropy, directly from the probabilities */
  double H = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double pv = exp(z[v] / T - logZ);
    if (pv > 0.0) H -= pv * log(pv);
  }
  /* the same entropy through running (max, sum, sum*shift) merges over blocks
   * of 256 entries; H = ln S - A / S with A = sum e^(z-m) (z-m) */
  double om = -INFINITY, oS = 0.0, oA = 0.0;
  for (int64_t v0 = 0; v0 < V; v0 += 256) {
    int64_t v1 = v0 + 256 < V ? v0 + 256 : V;
    double bm = -INFINITY;
    for (int64_t v = v0; v < v1; ++v) bm = fmax(bm, z[v] / T);
    double bS = 0.0, bA = 0.0;
    for (int64_t v = v0; v < v1; ++v) {
      double t = z[v] / T - bm;
      bS += exp(t);
      bA += exp(t) * t;
    }
    double nm = fmax(om, bm);
    double so = (oS > 0.0) ? exp(om - nm) : 0.0;
    double sb = exp(bm - nm);
    double nA = (oS > 0.0 ? so * (oA + (om - nm) * oS) : 0.0) + sb * (bA + (bm - nm) * bS);
    double nS = so * oS + sb * bS;
    om = nm;
    oS = nS;
    oA = nA;
  }
  /* Gumbel-max sample, G_v = -ln E_v */
  double* E = (double*)malloc(sizeof(double) * (size_t)V);
  or_exp_variates(seed, block, step, p, V, E);
  double g1 = -INFINITY, g2 = -INFINITY;
  int32_t y = 0;
  for (int64_t v = 0; v < V; ++v) {
    double s = z[v] / T - log(E[v]);
    if (s > g1) {
      g2 = g1;
      g1 = s;
      y = (int32_t)v;
    } else if (s > g2) {
      g2 = s;
    }
  }
  free(E);
  o->logZ = logZ;
  o->H = H;
  o->H_online = log(oS) - oA / oS;
  o->zmax = m;
  o->zgap = m - m2;
  o->gbest = g1;
  o->ggap = g1 - g2;
  o->amax = amax;
  o->y = y;
}

/* Statistics for n_rows positions; z is [n_rows, V] raw logits (before /T). */
void or_stats(int64_t n_rows, int64_t V, const double* z, const double* T, const uint64_t* seed, const int32_t* block,
              const int32_t* step, const int32_t* pos, or_pos* out, int nthreads) {
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#else
  (void)nthreads;
#endif
  for (int64_t i = 0; i < n_rows; ++i)
    or_stats_row(V, z + i * V, T[i], seed[i], block[i], step[i], pos[i], out + i);
}

/* Logits z[i, v] = sum_k h[i,k] W[v,k] in fp64 from the bf16 values (the tied
 * LM head).  Plain triple loop; rows of W outermost so that each W row is read
 * once per call. */
void or_logits(int64_t n_rows, int64_t V, int64_t d, const uint16_t* h, const uint16_t* W, double* z, int nthreads) {
  double* hv = (double*)malloc(sizeof(double) * (size_t)(n_rows * d));
  for (int64_t i = 0; i < n_rows * d; ++i) hv[i] = or_bf16_value(h[i]);
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#else
  (void)nthreads;
#endif
  {
    double* wrow = (double*)malloc(sizeof(double) * (size_t)d);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
    for (int64_t v = 0; v < V; ++v) {
      for (int64_t k = 0; k < d; ++k) wrow[k] = or_bf16_value(W[v * d + k]);
      for (int64_t i = 0; i < n_rows; ++i) {
        const double* hi = hv + i * d;
        double acc = 0.0;
        for (int64_t k = 0; k < d; ++k) acc += hi[k] * wrow[k];
        z[i * V + v] = acc;
      }
    }
    free(wrow);
  }
  free(hv);
}
