// K1 RMSNorm, K3 split-vocabulary combine, K4 entropy-bounded commit +
// uniform re-noise + schedule advance, and the tick planner.
#include <cuda_runtime.h>
#include <math.h>

#include "dg_internal.cuh"

namespace dg {
namespace {

// Round a double to the nearest bfloat16, ties to even, from its bit pattern:
// keep the top 7 fraction bits and round on the 45 bits below (normal range),
// or on the bits below the 2^-133 quantum (subnormal range).
__device__ __forceinline__ uint16_t bf16_rne(double x) {
  const uint64_t b = (uint64_t)__double_as_longlong(x);
  const uint32_t sign = (uint32_t)(b >> 63) << 15;
  const int e = (int)((b >> 52) & 0x7FF);
  const uint64_t frac = b & 0xFFFFFFFFFFFFFull;
  if (e == 0x7FF) return (uint16_t)(sign | (frac ? 0x7FC0u : 0x7F80u));
  if (e == 0) return (uint16_t)sign;  // zero or a double subnormal (far below the bf16 range)
  int E = e - 1023 + 127;
  if (E >= 1) {
    uint32_t m7 = (uint32_t)(frac >> 45);
    const uint64_t rem = frac & ((1ull << 45) - 1);
    const uint64_t halfway = 1ull << 44;
    if (rem > halfway || (rem == halfway && (m7 & 1u))) {
      if (++m7 == 128u) {
        m7 = 0;
        ++E;
      }
    }
    if (E >= 255) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | ((uint32_t)E << 7) | m7);
  }
  // value = sig * 2^(e-1075); in quanta of 2^-133 that is sig >> (942 - e)
  const uint64_t sig = frac | (1ull << 52);
  const int shift = 942 - e;
  if (shift >= 64) return (uint16_t)sign;
  uint64_t m = sig >> shift;
  const uint64_t rem = sig & ((1ull << shift) - 1);
  const uint64_t halfway = 1ull << (shift - 1);
  if (rem > halfway || (rem == halfway && (m & 1ull))) ++m;
  return (uint16_t)(sign | (uint32_t)m);  // m == 128 rolls into the smallest normal
}

// ------------------------------------------------------------------- K1
// h = bf16( w * r * sqrt(d) / (||r||_2 + eps) ) per active row, one warp per
// row.  The norm and the scaling are carried in fp64 so the bf16 rounding of
// every element is the one the exact quotient gives.
__global__ void __launch_bounds__(256) k_rmsnorm(const float* __restrict__ resid, const Dev dv) {
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int n_rows = dv.plan->n_active * dv.L;
  if (row >= n_rows) return;
  const int a = row / dv.L, p = row - a * dv.L;
  const int c = dv.active[a];
  const float4* r4 = reinterpret_cast<const float4*>(resid + ((size_t)c * dv.L + p) * dv.d);
  const int n4 = dv.d >> 2;
  double ss = 0.0;
  for (int i = lane; i < n4; i += 32) {
    const float4 v = __ldg(r4 + i);
    ss = fma((double)v.x, (double)v.x, ss);
    ss = fma((double)v.y, (double)v.y, ss);
    ss = fma((double)v.z, (double)v.z, ss);
    ss = fma((double)v.w, (double)v.w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const double inv = sqrt((double)dv.d) / (sqrt(ss) + (double)dv.eps);
  uint2* out = reinterpret_cast<uint2*>(dv.h + (size_t)row * dv.d);
  for (int i = lane; i < n4; i += 32) {
    const float4 v = __ldg(r4 + i);
    double w0 = 1.0, w1 = 1.0, w2 = 1.0, w3 = 1.0;
    if (dv.norm_w) {
      w0 = dv.norm_w[4 * i];
      w1 = dv.norm_w[4 * i + 1];
      w2 = dv.norm_w[4 * i + 2];
      w3 = dv.norm_w[4 * i + 3];
    }
    const uint32_t h0 = bf16_rne(w0 * (double)v.x * inv), h1 = bf16_rne(w1 * (double)v.y * inv);
    const uint32_t h2 = bf16_rne(w2 * (double)v.z * inv), h3 = bf16_rne(w3 * (double)v.w * inv);
    out[i] = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
  }
}

// ------------------------------------------------------------------- K3
__device__ __forceinline__ Partial shfl_partial(const Partial& a, int o) {
  Partial b;
  b.m = __shfl_xor_sync(0xFFFFFFFFu, a.m, o);
  b.S = __shfl_xor_sync(0xFFFFFFFFu, a.S, o);
  b.A = __shfl_xor_sync(0xFFFFFFFFu, a.A, o);
  b.g = __shfl_xor_sync(0xFFFFFFFFu, a.g, o);
  b.amax = __shfl_xor_sync(0xFFFFFFFFu, a.amax, o);
  b.gidx = __shfl_xor_sync(0xFFFFFFFFu, a.gidx, o);
  b.pad0 = b.pad1 = 0;
  return b;
}

// Combine the split-vocabulary partials of each active position:
// log2 Z = m + log2 S,  H = ln 2 (log2 S - A / S)  (= log Z - E_p[z/T] in nats),
// the sample is the index of the largest perturbed score, the argmax the index
// of the largest logit.  One warp per position.
__global__ void __launch_bounds__(256) k_combine(const Dev dv) {
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int n_rows = dv.plan->n_active * dv.L;
  if (row >= n_rows) return;
  Partial acc = empty_partial();
  const Partial* src = dv.part + (size_t)row * dv.n_sub;
  for (int i = lane; i < dv.n_sub; i += 32) acc = merge_partial(acc, src[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = merge_partial(acc, shfl_partial(acc, o));
  if (lane == 0) {
    const int a = row / dv.L, p = row - a * dv.L;
    const int c = dv.active[a];
    const float l2S = log2f(acc.S);
    const float H = 0.69314718055994531f * (l2S - acc.A / acc.S);
    const float lz = 0.69314718055994531f * (acc.m + l2S);
    const size_t o = (size_t)c * dv.L + p;
    dv.H[o] = fmaxf(H, 0.f);
    dv.logZ[o] = lz;
    dv.y[o] = acc.gidx;
    dv.amax[o] = acc.amax;
    if (!isfinite(H) || !isfinite(lz) || !isfinite(acc.g) || acc.gidx < 0 || acc.gidx >= dv.V) {
      if (atomicCAS(&dv.plan->err, kErrNone, kErrNonFinite) == kErrNone) dv.plan->err_info[1] = (int)o;
    }
  }
}

// ------------------------------------------------------------------- K4
constexpr int kCommitThreads = 256;
constexpr int kMaxL = 1024;

__device__ void init_canvas(const Dev& dv, int c, int block) {
  const uint64_t seed = dv.slots[c].seed;
  for (int p = threadIdx.x; p < dv.L; p += blockDim.x) {
    const size_t o = (size_t)c * dv.L + p;
    dv.x[o] = uniform_token(draw_u32(seed, kPurposeInit, block, 0, p), dv.V);
    dv.committed[o] = 0;
    dv.commit_step[o] = -1;
    dv.prev_amax[o] = 0;
  }
}

// Admit the canvases due by `tick` (admit_tick <= tick), in canvas order, while
// fewer than max_active are running; refresh temperatures; rebuild the active
// list in canvas order.  Run by every thread of one CTA.
__device__ void plan_tick(const Dev& dv, int tick) {
  __shared__ int s_running;
  // Slots were written by other CTAs of this grid: read them at L2 (ld.global.cg), not L1.
  if (threadIdx.x == 0) {
    int n = 0;
    for (int c = 0; c < dv.B; ++c) n += (__ldcg(&dv.slots[c].state) == kActive) ? 1 : 0;
    s_running = n;
  }
  __syncthreads();
  int running = s_running;
  for (int c = 0; c < dv.B && running < dv.max_active; ++c) {
    const int state = __ldcg(&dv.slots[c].state);
    const int admit = __ldcg(&dv.slots[c].admit_tick);
    if (state == kWaiting && admit <= tick) {
      init_canvas(dv, c, 0);
      __syncthreads();
      if (threadIdx.x == 0) {
        dg_slot& s = dv.slots[c];
        s.state = kActive;
        s.block = 0;
        s.step = 0;
        s.n_committed = 0;
      }
      ++running;
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {
    int n = 0;
    for (int c = 0; c < dv.B; ++c) {
      dg_slot& s = dv.slots[c];
      if (__ldcg(&s.state) == kActive) {
        s.temperature = temperature(__ldcg(&s.step), dv.N, dv.t_min, dv.t_max);
        if (n < dv.max_active) dv.active[n] = c;
        ++n;
      }
    }
    if (n > dv.max_active) n = dv.max_active;  // only reachable through an inconsistent dg_set_state
    dv.plan->n_active = n;
    dv.plan->tick = tick;
    dv.plan->k4_counter = 0u;
  }
  __syncthreads();
}

__device__ __forceinline__ double block_sum_double(double v, double* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += scratch[i];
    scratch[32] = t;
  }
  __syncthreads();
  return scratch[32];
}

// One CTA per active canvas:
//  (i)   early stop: s >= 1, mean_p H < confidence and argmax == previous argmax at every p;
//  (ii)  otherwise sort the uncommitted positions by (H, p) and accept the prefix whose
//        exclusive entropy sums (fp64) stay <= entropy_bound; accepted take the sample;
//  (iii) on early stop or at s = N-1 every uncommitted position takes its sample and the
//        block ends (tokens copied out, next block or done);
//  (iv)  every other uncommitted position is re-noised to a uniform token.
// The CTA that finishes last plans the next tick.
__global__ void __launch_bounds__(kCommitThreads) k_commit(const Dev dv) {
  __shared__ unsigned long long keys[kMaxL];
  __shared__ double red[33];
  __shared__ int s_k;
  const int n_active = dv.plan->n_active;
  const int a = blockIdx.x;
  const int L = dv.L;

  if (a < n_active) {
    const int c = dv.active[a];
    const dg_slot sl = dv.slots[c];
    const int s = sl.step, b = sl.block;
    const size_t base = (size_t)c * L;

    // (i) early-stop test
    double hsum = 0.0;
    int stable = 1;
    for (int p = threadIdx.x; p < L; p += blockDim.x) {
      hsum += (double)dv.H[base + p];
      stable &= (dv.amax[base + p] == dv.prev_amax[base + p]) ? 1 : 0;
    }
    const double mean_H = block_sum_double(hsum, red) / (double)L;
    stable = __syncthreads_and(stable);
    const bool converged = (s >= 1) && (mean_H < (double)dv.conf) && stable;
    const bool final_step = converged || (s == dv.N - 1);

    int n_acc = 0;
    if (!final_step) {
      // (ii) keys (H bits, p) for uncommitted positions, all-ones padding otherwise; H >= 0 so
      // the float bit pattern orders like the value
      int n2 = 1;
      while (n2 < L) n2 <<= 1;
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        unsigned long long k = ~0ull;
        if (i < L && !dv.committed[base + i])
          k = ((unsigned long long)__float_as_uint(dv.H[base + i]) << 32) | (unsigned)i;
        keys[i] = k;
      }
      __syncthreads();
      // bitonic sort, ascending
      for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int t = threadIdx.x; t < (n2 >> 1); t += blockDim.x) {
            const int i = 2 * t - (t & (stride - 1));
            const int j = i + stride;
            const bool up = ((i & size) == 0);
            const unsigned long long ki = keys[i], kj = keys[j];
            if ((ki > kj) == up) {
              keys[i] = kj;
              keys[j] = ki;
            }
          }
          __syncthreads();
        }
      }
      // walk the sorted entries in order, summing their entropies in fp64: entry j is
      // accepted while the sum of the entries before it is <= entropy_bound.  fp64
      // sums of non-negative terms never decrease, so the first refusal ends the walk.
      if (threadIdx.x == 0) {
        double E = 0.0;
        int k = 0;
        for (int j = 0; j < n2; ++j) {
          const unsigned long long kj = keys[j];
          if (kj == ~0ull || !(E <= (double)dv.bound)) break;
          ++k;
          E += (double)__uint_as_float((unsigned)(kj >> 32));
        }
        s_k = k;
      }
      __syncthreads();
      n_acc = s_k;
      for (int j = threadIdx.x; j < n_acc; j += blockDim.x) {
        const int p = (int)(keys[j] & 0xFFFFFFFFu);
        dv.x[base + p] = dv.y[base + p];
        dv.committed[base + p] = 1;
        dv.commit_step[base + p] = (int16_t)s;
      }
      __syncthreads();
      // (iv) uniform re-noise of everything still uncommitted; keep the argmax canvas
      for (int p = threadIdx.x; p < L; p += blockDim.x) {
        if (!dv.committed[base + p]) dv.x[base + p] = uniform_token(draw_u32(sl.seed, kPurposeRenoise, b, s, p), dv.V);
        dv.prev_amax[base + p] = dv.amax[base + p];
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        dg_slot& so = dv.slots[c];
        so.step = s + 1;
        so.n_committed = sl.n_committed + n_acc;
        so.mean_entropy = (float)mean_H;
      }
    } else {
      // (iii) finish the block
      for (int p = threadIdx.x; p < L; p += blockDim.x) {
        if (!dv.committed[base + p]) {
          dv.x[base + p] = dv.y[base + p];
          dv.committed[base + p] = 1;
          dv.commit_step[base + p] = (int16_t)s;
        }
        dv.tokens_out[((size_t)c * dv.G + b) * L + p] = dv.x[base + p];
      }
      __syncthreads();
      const bool more = (b + 1 < dv.G);
      if (more) init_canvas(dv, c, b + 1);
      __syncthreads();
      if (threadIdx.x == 0) {
        dg_slot& so = dv.slots[c];
        so.steps_used = sl.steps_used + s + 1;
        so.converged_blocks = sl.converged_blocks + (converged ? 1 : 0);
        so.mean_entropy = (float)mean_H;
        if (more) {
          so.block = b + 1;
          so.step = 0;
          so.n_committed = 0;
        } else {
          so.n_committed = L;
          so.state = kDone;
        }
      }
    }
  }

  // last CTA to finish plans the next tick
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&dv.plan->k4_counter, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (s_last) {
    __threadfence();
    plan_tick(dv, __ldcg(&dv.plan->tick) + 1);
  }
}

__global__ void __launch_bounds__(kCommitThreads) k_plan(const Dev dv, int tick) { plan_tick(dv, tick); }

}  // namespace

cudaError_t launch_rmsnorm(const Dev& dv, const float* resid, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;
  const int blocks = (rows + 7) / 8;
  k_rmsnorm<<<blocks, 256, 0, st>>>(resid, dv);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Dev& dv, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;
  k_combine<<<(rows + 7) / 8, 256, 0, st>>>(dv);
  return cudaGetLastError();
}

cudaError_t launch_commit(const Dev& dv, cudaStream_t st) {
  k_commit<<<dv.max_active, kCommitThreads, 0, st>>>(dv);
  return cudaGetLastError();
}

cudaError_t launch_plan(const Dev& dv, int tick, cudaStream_t st) {
  k_plan<<<1, kCommitThreads, 0, st>>>(dv, tick);
  return cudaGetLastError();
}

}  // namespace dg
