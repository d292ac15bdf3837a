/*
 * Seeded synthetic inputs for the denoise step (test and benchmark harness).
 *
 * This file generates INPUTS only: the tied vocabulary matrix W_vocab and the
 * per-step residual stream r that stands in for the DiffusionGemma backbone.
 * It holds none of the sampler's arithmetic (no RMSNorm, no logits, no
 * softmax, no sampling, no commit).  Both the CPU oracle and the CUDA path are
 * fed from here, so that the two see bit-identical inputs.
 *
 * Definitions (the workload the pages size: canvas of 256 positions, V = 2^18,
 * N(0, 0.02^2) weights, hidden built from the current token plus noise):
 *
 *   W[v,k]   = bf16_rne( fp32_rne( sigma_w * n_W(v*d + k) ) )
 *   r[p,k]   = fp32_rne( double(W[x_p,k]) + sigma * n_H(p, k) )
 *
 * where n_W and n_H are standard normals from Box-Muller (Box & Muller 1958,
 * "A note on the generation of random normal deviates") applied to pairs of
 * uniforms U = (u + 0.5) * 2^-32 drawn from Philox4x32-10 (Salmon, Moraes,
 * Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11):
 *
 *   W:  key = seed,    counter = (e>>2 lo, e>>2 hi, 0, 0),      e = v*d + k
 *   H:  key = seed_c,  counter = (k>>2, p, (block<<16)|step, 1)
 *
 * One Philox call yields four 32-bit words (x0,x1,x2,x3); (x0,x1) give the
 * normals of lanes 0 and 1, (x2,x3) those of lanes 2 and 3, and element e
 * (or k) takes lane e&3 (k&3).  Box-Muller is evaluated in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYN_PURPOSE_W 0u
#define SYN_PURPOSE_HIDDEN 1u

static inline uint32_t syn_mulhi(uint32_t a, uint32_t b, uint32_t* lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *lo = (uint32_t)p;
  return (uint32_t)(p >> 32);
}

/* Philox4x32 with 10 rounds, as defined in Salmon et al. (SC'11). */
void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint32_t lo0, lo1;
    uint32_t hi0 = syn_mulhi(0xD2511F53u, c0, &lo0);
    uint32_t hi1 = syn_mulhi(0xCD9E8D57u, c2, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static inline double syn_unit(uint32_t u) { return ((double)u + 0.5) * (1.0 / 4294967296.0); }

/* Box-Muller on one Philox block: four normals. */
static void syn_normals4(const uint32_t x[4], double n[4]) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = 0; j < 2; ++j) {
    double u1 = syn_unit(x[2 * j]);
    double u2 = syn_unit(x[2 * j + 1]);
    double rad = sqrt(-2.0 * log(u1));
    n[2 * j] = rad * cos(two_pi * u2);
    n[2 * j + 1] = rad * sin(two_pi * u2);
  }
}

/* Round-to-nearest-even from binary32 to bfloat16 (finite inputs). */
static inline uint16_t syn_bf16_from_f32(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

static inline float syn_f32_from_bf16(uint16_t h) {
  uint32_t b = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

/*
 * W_vocab [V, d] row-major.  w_f32 (nullable) receives the fp32 values,
 * w_bf16 (nullable) their bf16 rounding.  Rows [row0, row1) only, so callers
 * can split the work across threads.
 */
void synth_wvocab_rows(uint64_t seed, int64_t V, int64_t d, double sigma_w, int64_t row0, int64_t row1,
                       float* w_f32, uint16_t* w_bf16) {
  (void)V;
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint64_t e_begin = (uint64_t)row0 * (uint64_t)d, e_end = (uint64_t)row1 * (uint64_t)d;
  uint64_t g = e_begin >> 2;
  while ((g << 2) < e_end) {
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), 0u, SYN_PURPOSE_W};
    uint32_t x[4];
    double n[4];
    synth_philox4x32_10(ctr, key, x);
    syn_normals4(x, n);
    for (uint64_t j = 0; j < 4; ++j) {
      uint64_t e = (g << 2) + j;
      if (e < e_begin || e >= e_end) continue;
      float f = (float)(sigma_w * n[j]);
      if (w_f32) w_f32[e] = f;
      if (w_bf16) w_bf16[e] = syn_bf16_from_f32(f);
    }
    ++g;
  }
}

void synth_wvocab(uint64_t seed, int64_t V, int64_t d, double sigma_w, float* w_f32, uint16_t* w_bf16,
                  int nthreads) {
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = 1;
  int64_t chunk = 256;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
  for (int64_t v0 = 0; v0 < V; v0 += chunk)
    synth_wvocab_rows(seed, V, d, sigma_w, v0, v0 + chunk < V ? v0 + chunk : V, w_f32, w_bf16);
#else
  (void)nthreads;
  synth_wvocab_rows(seed, V, d, sigma_w, 0, V, w_f32, w_bf16);
#endif
}

/*
 * Residual rows standing in for the backbone output at one denoising step:
 * out[i, k] = fp32( W_bf16[tok[i], k] + sigma * n_H(pos[i], k) ) with Philox key
 * seeds[i] and counter word 2 = (block[i] << 16) | step[i].
 */
void synth_resid_rows(int64_t n_rows, const uint64_t* seeds, const int32_t* block, const int32_t* step,
                      const int32_t* pos, const int32_t* tok, const uint16_t* w_bf16, int64_t d, double sigma,
                      float* out, int nthreads) {
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
  for (int64_t i = 0; i < n_rows; ++i) {
    uint32_t key[2] = {(uint32_t)seeds[i], (uint32_t)(seeds[i] >> 32)};
    uint32_t bs = ((uint32_t)block[i] << 16) | (uint32_t)step[i];
    const uint16_t* wrow = w_bf16 + (int64_t)tok[i] * d;
    for (int64_t k0 = 0; k0 < d; k0 += 4) {
      uint32_t ctr[4] = {(uint32_t)(k0 >> 2), (uint32_t)pos[i], bs, SYN_PURPOSE_HIDDEN};
      uint32_t x[4];
      double n[4];
      synth_philox4x32_10(ctr, key, x);
      syn_normals4(x, n);
      for (int64_t j = 0; j < 4 && k0 + j < d; ++j) {
        double val = (double)syn_f32_from_bf16(wrow[k0 + j]) + sigma * n[j];
        out[i * d + k0 + j] = (float)val;
      }
    }
  }
}
