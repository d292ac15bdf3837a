// Device version of the residual generator in synth.c (benchmark harness):
// r[c, p, k] = fp32( W_bf16[x[c,p], k] + sigma * n_H(c, p, k) ), with n_H the
// Box-Muller normal of Philox4x32-10 keyed by the canvas seed and counter
// (k>>2, p, (block<<16)|step, 1) -- the same definition as the host code,
// evaluated in fp64.  Reads the per-canvas state through the public dg_slot
// layout; canvases that are not active are skipped.  A token outside [0, V)
// is never used as a W row: its residual row is written as zeros.  Inputs
// only: none of the sampler's arithmetic is here.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_sampler.h"

namespace {

__device__ __forceinline__ uint4 syn_philox(uint4 c, uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__global__ void syn_resid_kernel(const uint16_t* __restrict__ w, const int32_t* __restrict__ tokens,
                                 const dg_slot* __restrict__ slots, int B, int L, int V, int d, double sigma,
                                 float* __restrict__ out) {
  const int groups = d >> 2;
  const long long n = (long long)B * L * groups;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(t % groups);
    const long long cp = t / groups;
    const int c = (int)(cp / L), p = (int)(cp % L);
    const dg_slot sl = slots[c];
    if (sl.state != 1) continue;
    const int32_t tok = tokens[cp];
    if (tok < 0 || tok >= V) {
      reinterpret_cast<float4*>(out + (size_t)cp * d)[g] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const uint32_t bs = ((uint32_t)sl.block << 16) | (uint32_t)sl.step;
    const uint4 x = syn_philox(make_uint4((uint32_t)g, (uint32_t)p, bs, 1u), (uint32_t)sl.seed,
                               (uint32_t)(sl.seed >> 32));
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
    double nrm[4];
    for (int j = 0; j < 2; ++j) {
      const double u1 = ((double)xs[2 * j] + 0.5) * (1.0 / 4294967296.0);
      const double u2 = ((double)xs[2 * j + 1] + 0.5) * (1.0 / 4294967296.0);
      const double rad = sqrt(-2.0 * log(u1));
      double s, co;
      sincos(6.283185307179586476925286766559 * u2, &s, &co);
      nrm[2 * j] = rad * co;
      nrm[2 * j + 1] = rad * s;
    }
    const uint16_t* wrow = w + (size_t)tok * d + 4 * g;
    float4 o;
    float* of = &o.x;
    for (int j = 0; j < 4; ++j) {
      const float wf = __uint_as_float((uint32_t)wrow[j] << 16);
      of[j] = __double2float_rn(__dadd_rn((double)wf, __dmul_rn(sigma, nrm[j])));
    }
    reinterpret_cast<float4*>(out + (size_t)cp * d)[g] = o;
  }
}

}  // namespace

extern "C" int synth_resid_device(const void* w_bf16, const int32_t* tokens, const dg_slot* slots, int B, int L,
                                  int V, int d, double sigma, float* out, void* stream) {
  if (d % 4 || V < 1) return -1;
  const long long n = (long long)B * L * (d / 4);
  long long blocks = (n + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  syn_resid_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w_bf16), tokens, slots, B, L, V, d, sigma, out);
  return (int)cudaGetLastError();
}
