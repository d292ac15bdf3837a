// K1 RMSNorm, K3 split-vocabulary combine, K4 entropy-bounded commit +
// uniform re-noise + schedule advance, and the tick planner.
#include <cuda_runtime.h>
#include <math.h>

#include <utility>

#include "dg_internal.cuh"

namespace dg {
namespace {

// ------------------------------------------------------------------- K1
// Error-free transformations in fp32 (the fp64 pipe of this part is slow):
// Knuth's TwoSum gives a + b = s + e exactly; an FMA gives x*y = p + e exactly
// (Dekker's product).  Carried as unevaluated pairs (hi, lo) they hold the sum
// of squares and the scaled value to ~2^-46 relative accuracy.  __f*_rn
// intrinsics keep the compiler from contracting the steps into other FMAs.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float z = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

// bf16 nearest-even of the exact value hi + lo, where hi = fl(hi + lo) (so
// |lo| <= half an fp32 ulp of hi): hi's own rounding decides unless hi sits
// exactly on a bf16 midpoint, where the sign of lo decides and 0 means a tie.
__device__ __forceinline__ uint32_t bf16_rne_pair(float hi, float lo) {
  const uint32_t b = __float_as_uint(hi);
  const uint32_t rem = b & 0xFFFFu;
  uint32_t up;
  if (rem != 0x8000u) {
    up = rem > 0x8000u ? 1u : 0u;
  } else if (lo == 0.f) {
    up = (b >> 16) & 1u;
  } else {
    up = ((lo > 0.f) == (hi > 0.f)) ? 1u : 0u;  // lo moves |value| above the midpoint
  }
  return (b >> 16) + up;
}

// h = bf16( w * r * sqrt(d) / (||r||_2 + eps) ) per active row, one warp per
// row.  The rounding of every element is the one the exact quotient gives
// (up to ~2^-46 relative): sum of squares in TwoSum pairs, the per-row
// scale sqrt(d) / (norm + eps) in fp64 (two operations per row), split into
// an fp32 pair, and each product carried exactly before the bf16 rounding.
__global__ void __launch_bounds__(256) k_rmsnorm(const float* __restrict__ resid, const Dev dv) {
  pdl_wait();
  pdl_allow_next();
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int n_rows = dv.plan->n_active * dv.L;
  if (row >= n_rows) return;
  const int a = row / dv.L, p = row - a * dv.L;
  const int c = dv.active[a];
  const float4* r4 = reinterpret_cast<const float4*>(resid + ((size_t)c * dv.L + p) * dv.d);
  const int n4 = dv.d >> 2;
  float sh = 0.f, sl = 0.f;
  for (int i = lane; i < n4; i += 32) {
    const float4 v = __ldg(r4 + i);
    const float xs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float sq = __fmul_rn(xs[j], xs[j]);
      const float sq_err = fmaf(xs[j], xs[j], -sq);
      float e;
      two_sum(sh, sq, sh, e);
      sl = __fadd_rn(sl, __fadd_rn(e, sq_err));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, sh, o);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, sl, o);
    float e;
    two_sum(sh, oh, sh, e);
    sl = __fadd_rn(__fadd_rn(sl, ol), e);
  }
  const double inv = sqrt((double)dv.d) / (sqrt((double)sh + (double)sl) + (double)dv.eps);
  const float inv_hi = __double2float_rn(inv);
  const float inv_lo = __double2float_rn(inv - (double)inv_hi);
  uint2* out = reinterpret_cast<uint2*>(dv.h + (size_t)row * dv.d);
  const float4* w4 = reinterpret_cast<const float4*>(dv.norm_w);
  for (int i = lane; i < n4; i += 32) {
    const float4 v = __ldg(r4 + i);
    const float4 w = w4 ? __ldg(w4 + i) : make_float4(1.f, 1.f, 1.f, 1.f);
    const float xs[4] = {v.x, v.y, v.z, v.w};
    const float ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t hb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float xw = __fmul_rn(ws[j], xs[j]);            // w x = xw + xw_err exactly
      const float xw_err = fmaf(ws[j], xs[j], -xw);
      const float ph = __fmul_rn(xw, inv_hi);               // (w x) inv ~= ph + pl
      const float pe = fmaf(xw, inv_hi, -ph);
      const float pl = fmaf(xw, inv_lo, fmaf(xw_err, inv_hi, pe));
      const float hi = __fadd_rn(ph, pl);                   // renormalise: |lo| <= ulp(hi)/2
      const float lo = __fsub_rn(pl, __fsub_rn(hi, ph));
      hb[j] = bf16_rne_pair(hi, lo) & 0xFFFFu;
    }
    out[i] = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
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
  pdl_wait();
  pdl_allow_next();
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
    dv.H[o] = H > 0.f ? H : 0.f;  // +0 for rounding below zero (and never -0: its bits would sort last)
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

// Block-wide helpers for the commit kernel (blockDim.x = kCommitThreads).
__device__ __forceinline__ float block_sum_f32(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kCommitThreads / 32; ++i) t += scratch[i];
  return t;
}

__device__ __forceinline__ unsigned long long block_min_u64(unsigned long long v, unsigned long long* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w < v ? w : v;
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  unsigned long long t = ~0ull;
#pragma unroll
  for (int i = 0; i < kCommitThreads / 32; ++i) t = scratch[i] < t ? scratch[i] : t;
  return t;
}

// Sort 32 keys held one per lane, ascending (bitonic network over shuffles).
__device__ __forceinline__ unsigned long long warp_sort_u64(unsigned long long key) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, key, stride);
      const bool keep_min = ((lane & stride) == 0) == ((lane & size) == 0);
      key = keep_min ? (other < key ? other : key) : (other > key ? other : key);
    }
  }
  return key;
}

// Accepted entries among `n` ascending keys (H bits << 32 | p): the walk sums
// the entropies in fp64, in order; entry j is accepted while the sum of the
// entries before it is <= bound.  fp64 sums of non-negative terms never
// decrease, so the first refusal ends the walk.
__device__ __forceinline__ int accept_walk(const unsigned long long* keys, int n, float bound) {
  double E = 0.0;
  int k = 0;
  for (int j = 0; j < n; ++j) {
    if (keys[j] == ~0ull || !(E <= (double)bound)) break;
    ++k;
    E += (double)__uint_as_float((unsigned)(keys[j] >> 32));
  }
  return k;
}

// One CTA per active canvas:
//  (i)   early stop: s >= 1, mean_p H < confidence and argmax == previous argmax at every p;
//  (ii)  otherwise order the uncommitted positions by (H, p) and accept the prefix whose
//        exclusive entropy sums stay <= entropy_bound; accepted positions take their sample;
//  (iii) on early stop or at s = N-1 every uncommitted position takes its sample and the
//        block ends (tokens copied out, next block or done);
//  (iv)  every other uncommitted position is re-noised to a uniform token.
// Only entries whose entropy is <= bound, plus the smallest one above it, can be
// accepted, so the common case sorts at most 32 candidates in one warp; more than
// 31 entropies within the bound fall back to a bitonic sort of the canvas.
// The CTA that finishes last plans the next tick.
__global__ void __launch_bounds__(kCommitThreads) k_commit(const Dev dv) {
  __shared__ unsigned long long keys[kMaxL];
  __shared__ float redf[kCommitThreads / 32];
  __shared__ unsigned long long redk[kCommitThreads / 32];
  __shared__ unsigned long long cand[32];
  __shared__ int s_cnt, s_k;
  pdl_wait();
  pdl_allow_next();
  const int n_active = dv.plan->n_active;
  const int a = blockIdx.x;
  const int L = dv.L;

  if (a < n_active) {
    const int c = dv.active[a];
    const dg_slot sl = dv.slots[c];
    const int s = sl.step, b = sl.block;
    const size_t base = (size_t)c * L;
    const float bound = dv.bound;

    // (i) early-stop test, and the keys of the uncommitted positions
    float hsum = 0.f, n_le = 0.f;
    int stable = 1;
    unsigned long long kmin_above = ~0ull;
    for (int p = threadIdx.x; p < L; p += blockDim.x) {
      const float H = dv.H[base + p];
      hsum += H;
      stable &= (dv.amax[base + p] == dv.prev_amax[base + p]) ? 1 : 0;
      if (!dv.committed[base + p]) {
        const unsigned long long k = ((unsigned long long)__float_as_uint(H) << 32) | (unsigned)p;
        if (H <= bound) n_le += 1.f;
        else kmin_above = k < kmin_above ? k : kmin_above;
      }
    }
    const float mean_H = block_sum_f32(hsum, redf) / (float)L;
    const int count_le = (int)block_sum_f32(n_le, redf);
    kmin_above = block_min_u64(kmin_above, redk);
    stable = __syncthreads_and(stable);
    const bool converged = (s >= 1) && (mean_H < dv.conf) && stable;
    const bool final_step = converged || (s == dv.N - 1);

    int n_acc = 0;
    if (!final_step) {
      // (ii) the accepted prefix of the (H, p) order
      if (count_le < 32) {
        if (threadIdx.x == 0) s_cnt = 0;
        __syncthreads();
        for (int p = threadIdx.x; p < L; p += blockDim.x) {
          const float H = dv.H[base + p];
          if (!dv.committed[base + p] && H <= bound)
            cand[atomicAdd(&s_cnt, 1)] = ((unsigned long long)__float_as_uint(H) << 32) | (unsigned)p;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
          const int lane = threadIdx.x;
          unsigned long long k = lane < count_le ? cand[lane] : (lane == count_le ? kmin_above : ~0ull);
          k = warp_sort_u64(k);
          cand[lane] = k;
          __syncwarp();
          if (lane == 0) s_k = accept_walk(cand, 32, bound);
        }
        __syncthreads();
        n_acc = s_k;
        for (int j = threadIdx.x; j < n_acc; j += blockDim.x) keys[j] = cand[j];
      } else {
        int n2 = 1;
        while (n2 < L) n2 <<= 1;
        for (int i = threadIdx.x; i < n2; i += blockDim.x) {
          unsigned long long k = ~0ull;
          if (i < L && !dv.committed[base + i])
            k = ((unsigned long long)__float_as_uint(dv.H[base + i]) << 32) | (unsigned)i;
          keys[i] = k;
        }
        __syncthreads();
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
        if (threadIdx.x == 0) s_k = accept_walk(keys, n2, bound);
        __syncthreads();
        n_acc = s_k;
      }
      __syncthreads();
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
        so.mean_entropy = mean_H;
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
        so.mean_entropy = mean_H;
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

// Launch with programmatic stream serialization (see pdl_wait / pdl_allow_next).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_rmsnorm(const Dev& dv, const float* resid, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;
  return launch_pdl(k_rmsnorm, dim3((rows + 7) / 8), dim3(256), 0, st, resid, dv);
}

cudaError_t launch_combine(const Dev& dv, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;
  return launch_pdl(k_combine, dim3((rows + 7) / 8), dim3(256), 0, st, dv);
}

cudaError_t launch_commit(const Dev& dv, cudaStream_t st) {
  return launch_pdl(k_commit, dim3(dv.max_active), dim3(kCommitThreads), 0, st, dv);
}

cudaError_t launch_plan(const Dev& dv, int tick, cudaStream_t st) {
  k_plan<<<1, kCommitThreads, 0, st>>>(dv, tick);
  return cudaGetLastError();
}

}  // namespace dg
