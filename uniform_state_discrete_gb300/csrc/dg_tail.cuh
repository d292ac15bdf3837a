// The per-tick tail of the denoise step, run by a group of threads of one CTA:
// the entropy-bounded commit of a canvas and the planning of the next tick.
// Used by the finishing kernel and the stand-alone planner kernel.
#pragma once

#include "dg_internal.cuh"

namespace dg {

// A set of threads of one CTA that synchronise together: named barrier `bar`
// over `n` threads (bar 0 = __syncthreads for the whole CTA).
struct Group {
  int tid, n, bar;
  __device__ __forceinline__ void sync() const {
    if (bar == 0) {
      __syncthreads();
    } else {
      asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(n) : "memory");
    }
  }
};

constexpr int kMaxL = 1024;
constexpr int kTailMaxThreads = 1024;

// Shared-memory scratch of the tail.
struct TailScratch {
  unsigned long long keys[kMaxL];
  unsigned long long cand[32];
  unsigned long long redk[kTailMaxThreads / 32];
  float redf[kTailMaxThreads / 32];
  int flags[4];
  int done_list[64];  // canvases completed by one CTA's rows (at most 8 / L + 2)
};

__device__ __forceinline__ float group_sum_f32(float v, const Group& g, TailScratch* sc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = g.tid >> 5, lane = g.tid & 31;
  g.sync();
  if (lane == 0) sc->redf[w] = v;
  g.sync();
  float t = 0.f;
  for (int i = 0; i < g.n / 32; ++i) t += sc->redf[i];
  return t;
}

__device__ __forceinline__ unsigned long long group_min_u64(unsigned long long v, const Group& g, TailScratch* sc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w < v ? w : v;
  }
  const int w = g.tid >> 5, lane = g.tid & 31;
  g.sync();
  if (lane == 0) sc->redk[w] = v;
  g.sync();
  unsigned long long t = ~0ull;
  for (int i = 0; i < g.n / 32; ++i) t = sc->redk[i] < t ? sc->redk[i] : t;
  return t;
}

__device__ __forceinline__ int group_and(int v, const Group& g, TailScratch* sc) {
  return group_sum_f32(v ? 0.f : 1.f, g, sc) == 0.f ? 1 : 0;
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

// Accepted entries among `n` ascending keys (H bits << 32 | p): the walk sums the
// entropies in fp64, in order; entry j is accepted while the sum of the entries
// before it is <= bound.  fp64 sums of non-negative terms never decrease, so the
// first refusal ends the walk.
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

__device__ __forceinline__ void init_canvas(const Dev& dv, int c, int block, const Group& g) {
  const uint64_t seed = dv.slots[c].seed;
  for (int p = g.tid; p < dv.L; p += g.n) {
    const size_t o = (size_t)c * dv.L + p;
    dv.x[o] = uniform_token(draw_u32(seed, kPurposeInit, block, 0, p), dv.V);
    dv.committed[o] = 0;
    dv.commit_step[o] = -1;
    dv.prev_amax[o] = 0;
  }
}

// Admit the canvases due by `tick` (admit_tick <= tick), in canvas order, while
// fewer than max_active are running; refresh temperatures; rebuild the active
// list in canvas order; reset the tick's counters.  Slots may have been written
// by other CTAs of the grid, so they are read at L2 (ld.global.cg).
static __device__ void plan_tick(const Dev& dv, int tick, const Group& g, TailScratch* sc) {
  if (g.tid == 0) {
    int n = 0;
    for (int c = 0; c < dv.B; ++c) n += (__ldcg(&dv.slots[c].state) == kActive) ? 1 : 0;
    sc->flags[0] = n;
  }
  g.sync();
  int running = sc->flags[0];
  for (int c = 0; c < dv.B && running < dv.max_active; ++c) {
    const int state = __ldcg(&dv.slots[c].state);
    const int admit = __ldcg(&dv.slots[c].admit_tick);
    if (state == kWaiting && admit <= tick) {
      init_canvas(dv, c, 0, g);
      g.sync();
      if (g.tid == 0) {
        dg_slot& s = dv.slots[c];
        s.state = kActive;
        s.block = 0;
        s.step = 0;
        s.n_committed = 0;
      }
      ++running;
      g.sync();
    }
  }
  if (g.tid == 0) {
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
    dv.plan->commits = 0u;
  }
  g.sync();
}

// The commit step of canvas c for this tick:
//  (i)   early stop: s >= 1, mean_p H < confidence and argmax == previous argmax at every p;
//  (ii)  otherwise order the uncommitted positions by (H, p) and accept the prefix whose
//        exclusive entropy sums stay <= entropy_bound; accepted positions take their sample;
//  (iii) on early stop or at s = N-1 every uncommitted position takes its sample and the
//        block ends (tokens copied out, next block or done);
//  (iv)  every other uncommitted position is re-noised to a uniform token.
// Only entries whose entropy is <= bound, plus the smallest one above it, can be
// accepted, so the common case sorts at most 32 candidates in one warp; more than
// 31 entropies within the bound fall back to a bitonic sort of the canvas.
// Per-position data of this tick were written by other CTAs: read at L2.
static __device__ void commit_canvas(const Dev& dv, int c, const Group& g, TailScratch* sc) {
  const int L = dv.L;
  const dg_slot sl = dv.slots[c];
  const int s = sl.step, b = sl.block;
  const size_t base = (size_t)c * L;
  const float bound = dv.bound;

  float hsum = 0.f, n_le = 0.f;
  int stable = 1;
  unsigned long long kmin_above = ~0ull;
  for (int p = g.tid; p < L; p += g.n) {
    const float H = __ldcg(dv.H + base + p);
    hsum += H;
    stable &= (__ldcg(dv.amax + base + p) == dv.prev_amax[base + p]) ? 1 : 0;
    if (!dv.committed[base + p]) {
      const unsigned long long k = ((unsigned long long)__float_as_uint(H) << 32) | (unsigned)p;
      if (H <= bound) n_le += 1.f;
      else kmin_above = k < kmin_above ? k : kmin_above;
    }
  }
  const float mean_H = group_sum_f32(hsum, g, sc) / (float)L;
  const int count_le = (int)group_sum_f32(n_le, g, sc);
  kmin_above = group_min_u64(kmin_above, g, sc);
  stable = group_and(stable, g, sc);
  const bool converged = (s >= 1) && (mean_H < dv.conf) && stable;
  const bool final_step = converged || (s == dv.N - 1);

  if (!final_step) {
    int n_acc;
    if (count_le < 32) {
      if (g.tid == 0) sc->flags[1] = 0;
      g.sync();
      for (int p = g.tid; p < L; p += g.n) {
        const float H = __ldcg(dv.H + base + p);
        if (!dv.committed[base + p] && H <= bound)
          sc->cand[atomicAdd(&sc->flags[1], 1)] = ((unsigned long long)__float_as_uint(H) << 32) | (unsigned)p;
      }
      g.sync();
      if (g.tid < 32) {
        const int lane = g.tid;
        unsigned long long k = lane < count_le ? sc->cand[lane] : (lane == count_le ? kmin_above : ~0ull);
        k = warp_sort_u64(k);
        sc->keys[lane] = k;
        __syncwarp();
        if (lane == 0) sc->flags[2] = accept_walk(sc->keys, 32, bound);
      }
      g.sync();
      n_acc = sc->flags[2];
    } else {
      int n2 = 1;
      while (n2 < L) n2 <<= 1;
      for (int i = g.tid; i < n2; i += g.n) {
        unsigned long long k = ~0ull;
        if (i < L && !dv.committed[base + i])
          k = ((unsigned long long)__float_as_uint(__ldcg(dv.H + base + i)) << 32) | (unsigned)i;
        sc->keys[i] = k;
      }
      g.sync();
      for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int t = g.tid; t < (n2 >> 1); t += g.n) {
            const int i = 2 * t - (t & (stride - 1));
            const int j = i + stride;
            const bool up = ((i & size) == 0);
            const unsigned long long ki = sc->keys[i], kj = sc->keys[j];
            if ((ki > kj) == up) {
              sc->keys[i] = kj;
              sc->keys[j] = ki;
            }
          }
          g.sync();
        }
      }
      if (g.tid == 0) sc->flags[2] = accept_walk(sc->keys, n2, bound);
      g.sync();
      n_acc = sc->flags[2];
    }
    for (int j = g.tid; j < n_acc; j += g.n) {
      const int p = (int)(sc->keys[j] & 0xFFFFFFFFu);
      dv.x[base + p] = __ldcg(dv.y + base + p);
      dv.committed[base + p] = 1;
      dv.commit_step[base + p] = (int16_t)s;
    }
    g.sync();
    for (int p = g.tid; p < L; p += g.n) {
      if (!dv.committed[base + p]) dv.x[base + p] = uniform_token(draw_u32(sl.seed, kPurposeRenoise, b, s, p), dv.V);
      dv.prev_amax[base + p] = __ldcg(dv.amax + base + p);
    }
    g.sync();
    if (g.tid == 0) {
      dg_slot& so = dv.slots[c];
      so.step = s + 1;
      so.n_committed = sl.n_committed + n_acc;
      so.mean_entropy = mean_H;
    }
  } else {
    for (int p = g.tid; p < L; p += g.n) {
      if (!dv.committed[base + p]) {
        dv.x[base + p] = __ldcg(dv.y + base + p);
        dv.committed[base + p] = 1;
        dv.commit_step[base + p] = (int16_t)s;
      }
      dv.tokens_out[((size_t)c * dv.G + b) * L + p] = dv.x[base + p];
    }
    g.sync();
    const bool more = (b + 1 < dv.G);
    if (more) init_canvas(dv, c, b + 1, g);
    g.sync();
    if (g.tid == 0) {
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
  g.sync();
}

}  // namespace dg
