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
constexpr int kTailThreads = 256;               // threads of every group that runs the tail
constexpr int kTailPer = kMaxL / kTailThreads;  // canvas positions per thread

// Shared-memory scratch of the tail.
struct TailScratch {
  unsigned long long keys[kMaxL];  // (H bits << 32 | p) of each uncommitted position, ~0 otherwise
  unsigned char acc[kMaxL];        // accepted this tick
  unsigned long long cand[32];
  unsigned long long redk[kTailThreads / 32];
  float redf[kTailThreads / 32][2];
  int redi[kTailThreads / 32][2];
  int flags[4];
  int remasked;        // DG_REACCEPT: positions accepted at the previous step and re-noised now
  int done_list[64];   // canvases completed by one CTA's rows (at most 8 / L + 2)
  int row_canvas[8];   // canvas of each of a finishing CTA's rows
};

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
  if (!DG_IN_BOUNDS(dv.plan, c >= 0 && c < dv.B && block >= 0 && block < dv.G, 1, c)) return;
  const uint64_t seed = __ldcg(&dv.slots[c].seed);
  for (int p = g.tid; p < dv.L; p += g.n) {
    const size_t o = (size_t)c * dv.L + p;
    dv.x[o] = uniform_token(draw_u32(seed, kPurposeInit, block, 0, p), dv.V);
    dv.committed[o] = 0;
    dv.commit_step[o] = -1;
    dv.prev_amax[o] = 0;
  }
}

// Admit the canvases due by `tick` (admit_tick <= tick), in canvas order, while
// fewer than max_active are running; rebuild the active list in canvas order;
// reset the tick's counters.  A canvas's temperature is written by whoever
// writes its step (the commit, an admission); `refresh_temps` rewrites it for
// every active canvas, for a state loaded from the host.  Slots may have been
// written by other CTAs of the grid, so they are read at L2 (ld.global.cg).
// The group has kTailThreads threads; with at most that many canvases the
// slots are read once.  The state of canvas `known_c` (if >= 0), which the
// calling group has just written itself, is taken as `known_state`.
static __device__ void plan_tick(const Dev& dv, int tick, const Group& g, TailScratch* sc, bool refresh_temps,
                                 int known_c = -1, int known_state = kDone) {
  const int lane = g.tid & 31, w = g.tid >> 5;
  int st0 = kDone;  // state of canvas g.tid (first round)
  int run = 0, due = 0;
  for (int c = g.tid; c < dv.B; c += g.n) {
    const int st = c == known_c ? known_state : __ldcg(&dv.slots[c].state);
    if (c == g.tid) st0 = st;
    run += st == kActive ? 1 : 0;
    due |= (st == kWaiting && __ldcg(&dv.slots[c].admit_tick) <= tick) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    run += __shfl_xor_sync(0xFFFFFFFFu, run, o);
    due |= __shfl_xor_sync(0xFFFFFFFFu, due, o);
  }
  if (lane == 0) {
    sc->redi[w][0] = run;
    sc->redi[w][1] = due;
  }
  g.sync();
  int running = 0, any_due = 0;
  for (int k = 0; k < kTailThreads / 32; ++k) {
    running += sc->redi[k][0];
    any_due |= sc->redi[k][1];
  }
  bool admitted = false;
  if (any_due) {
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
          s.n_remasked = 0;
          s.stable_steps = 0;
          s.temperature = dv.temps[0];
        }
        ++running;
        admitted = true;
        g.sync();
      }
    }
  }
  // active list in canvas order
  int base = 0;
  for (int c0 = 0; c0 < dv.B; c0 += g.n) {
    const int c = c0 + g.tid;
    bool act = false;
    if (c < dv.B) act = (c0 == 0 && !admitted ? st0 : __ldcg(&dv.slots[c].state)) == kActive;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, act);
    g.sync();  // the previous round's counts have been read
    if (lane == 0) sc->redi[w][0] = __popc(bal);
    g.sync();
    int off = base, tot = 0;
    for (int k = 0; k < kTailThreads / 32; ++k) {
      off += k < w ? sc->redi[k][0] : 0;
      tot += sc->redi[k][0];
    }
    if (act) {
      const int idx = off + __popc(bal & ((1u << lane) - 1u));
      if (idx < dv.max_active && DG_IN_BOUNDS(dv.plan, c < dv.B, 2, c)) dv.active[idx] = c;
      if (refresh_temps) {
        int st = __ldcg(&dv.slots[c].step);
        st = st < 0 ? 0 : (st >= dv.N ? dv.N - 1 : st);
        dv.slots[c].temperature = dv.temps[st];
      }
    }
    base += tot;
  }
  // the tick's hand-off counters: every kernel that waited on them is past its wait
  // and fin_started, slab_done, units_done
  for (int i = g.tid; i < 3 + dv.rows_cap / 128; i += g.n) dv.rows_ready[i] = 0u;
  if (g.tid == 0) {
    dv.plan->n_active = base < dv.max_active ? base : dv.max_active;  // above it only after an inconsistent dg_set_state
    dv.plan->tick = tick;
    dv.plan->commits = 0u;
    dv.plan->epoch += 1u;  // the per-row best scores of earlier ticks no longer count
  }
  g.sync();
}

// The commit step of canvas c for this tick:
//  (i)   early stop: mean_p H < confidence and the argmax canvas equal to the previous one
//        at every p for the last `stability` steps in a row (s >= stability);
//  (ii)  otherwise order the open positions by (H, p) and accept the prefix whose
//        exclusive entropy sums stay <= entropy_bound; accepted positions take their sample;
//  (iii) on early stop or at s = N-1 every open position takes its sample and the
//        block ends (tokens copied out, next block or done);
//  (iv)  every other open position is re-noised to a uniform token.
// The open positions are the uncommitted ones under DG_FREEZE and all of them
// under DG_REACCEPT, where the committed mask becomes this step's accepted set.
// Only entries whose entropy is <= bound, plus the smallest one above it, can be
// accepted, so the common case sorts at most 32 candidates in one warp; more than
// 31 entropies within the bound fall back to a bitonic sort of the canvas.
// Every per-position input is read once, up front, into registers (this tick's
// values were written by other CTAs: read at L2); the group has kTailThreads
// threads, so each holds at most kTailPer positions.  Returns the canvas's
// state after the commit (kActive, or kDone after its last block).
static __device__ int commit_canvas(const Dev& dv, int c, const Group& g, TailScratch* sc) {
  const int L = dv.L;
  dg_slot sl;
  sl.seed = __ldcg(&dv.slots[c].seed);
  sl.step = __ldcg(&dv.slots[c].step);
  sl.block = __ldcg(&dv.slots[c].block);
  sl.n_committed = __ldcg(&dv.slots[c].n_committed);
  sl.steps_used = __ldcg(&dv.slots[c].steps_used);
  sl.converged_blocks = __ldcg(&dv.slots[c].converged_blocks);
  sl.stable_steps = __ldcg(&dv.slots[c].stable_steps);
  const int s = sl.step, b = sl.block;
  if (!DG_IN_BOUNDS(dv.plan, c >= 0 && c < dv.B && b >= 0 && b < dv.G && s >= 0 && s < dv.N, 3,
                    c < 0 || c >= dv.B ? c : (b < 0 || b >= dv.G ? b : s)))
    return kActive;  // the group skips the commit (every thread takes the same branch)
  const size_t base = (size_t)c * L;
  const float bound = dv.bound;
  const int lane = g.tid & 31, w = g.tid >> 5;

  const float t_next = dv.temps[s + 1 < dv.N ? s + 1 : dv.N - 1], t_first = dv.temps[0];
  float Hv[kTailPer];
  int yv[kTailPer], av[kTailPer], pv[kTailPer], xv[kTailPer];
  bool cm[kTailPer], was[kTailPer];
#pragma unroll
  for (int i = 0; i < kTailPer; ++i) {
    const int p = g.tid + i * kTailThreads;
    if (p < L) {
      Hv[i] = __ldcg(dv.H + base + p);
      yv[i] = __ldcg(dv.y + base + p);
      av[i] = __ldcg(dv.amax + base + p);
      pv[i] = __ldcg(dv.prev_amax + base + p);
      xv[i] = __ldcg(dv.x + base + p);
      was[i] = __ldcg(dv.committed + base + p) != 0;
      cm[i] = was[i] && !dv.reaccept;  // frozen
    }
  }
  float hsum = 0.f, n_le = 0.f;
  int stable = 1;
  unsigned long long kmin_above = ~0ull;
#pragma unroll
  for (int i = 0; i < kTailPer; ++i) {
    const int p = g.tid + i * kTailThreads;
    if (p < L) {
      hsum += Hv[i];
      stable &= av[i] == pv[i] ? 1 : 0;
      const unsigned long long k = ((unsigned long long)__float_as_uint(Hv[i]) << 32) | (unsigned)p;
      sc->keys[p] = cm[i] ? ~0ull : k;
      sc->acc[p] = 0;
      if (!cm[i]) {
        if (Hv[i] <= bound) n_le += 1.f;
        else kmin_above = k < kmin_above ? k : kmin_above;
      }
    }
  }
  // the four canvas-wide reductions share one exchange through shared memory
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    hsum += __shfl_xor_sync(0xFFFFFFFFu, hsum, o);
    n_le += __shfl_xor_sync(0xFFFFFFFFu, n_le, o);
    stable &= __shfl_xor_sync(0xFFFFFFFFu, stable, o);
    const unsigned long long ko = __shfl_xor_sync(0xFFFFFFFFu, kmin_above, o);
    kmin_above = ko < kmin_above ? ko : kmin_above;
  }
  if (lane == 0) {
    sc->redf[w][0] = hsum;
    sc->redf[w][1] = n_le;
    sc->redi[w][0] = stable;
    sc->redk[w] = kmin_above;
  }
  if (g.tid == 0) {
    sc->flags[1] = 0;
    sc->remasked = 0;
  }
  g.sync();
  float tot_h = 0.f, tot_le = 0.f;
  for (int k = 0; k < kTailThreads / 32; ++k) {
    tot_h += sc->redf[k][0];
    tot_le += sc->redf[k][1];
    stable &= sc->redi[k][0];
    kmin_above = sc->redk[k] < kmin_above ? sc->redk[k] : kmin_above;
  }
  const float mean_H = tot_h / (float)L;
  const int count_le = (int)tot_le;
  // steps in a row whose argmax canvas equalled the one before (none before step 1)
  const int run = (s >= 1 && stable) ? sl.stable_steps + 1 : 0;
  const bool converged = run >= dv.stability && mean_H < dv.conf;
  const bool final_step = converged || (s == dv.N - 1);

  if (!final_step) {
    int n_acc;
    if (count_le < 32) {
#pragma unroll
      for (int i = 0; i < kTailPer; ++i) {
        const int p = g.tid + i * kTailThreads;
        if (p < L && !cm[i] && Hv[i] <= bound)
          sc->cand[atomicAdd(&sc->flags[1], 1)] = ((unsigned long long)__float_as_uint(Hv[i]) << 32) | (unsigned)p;
      }
      g.sync();
      if (g.tid < 32) {
        unsigned long long k = lane < count_le ? sc->cand[lane] : (lane == count_le ? kmin_above : ~0ull);
        k = warp_sort_u64(k);
        sc->cand[lane] = k;
        __syncwarp();
        const int na = accept_walk(sc->cand, 32, bound);  // every lane walks the same keys
        if (lane < na) sc->acc[(unsigned)(k & 0xFFFFFFFFu)] = 1;
        if (lane == 0) sc->flags[2] = na;
      }
      g.sync();
      n_acc = sc->flags[2];
    } else {
      int n2 = 1;
      while (n2 < L) n2 <<= 1;
      for (int i = L + g.tid; i < n2; i += g.n) sc->keys[i] = ~0ull;
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
      for (int j = g.tid; j < n_acc; j += g.n) sc->acc[(unsigned)(sc->keys[j] & 0xFFFFFFFFu)] = 1;
      g.sync();
    }
    int remasked = 0;
#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
      const int p = g.tid + i * kTailThreads;
      if (p < L) {
        if (!cm[i]) {
          if (sc->acc[p]) {
            if (DG_IN_BOUNDS(dv.plan, yv[i] >= 0 && yv[i] < dv.V, 4, yv[i])) dv.x[base + p] = yv[i];
            dv.committed[base + p] = 1;
            dv.commit_step[base + p] = (int16_t)s;
          } else {
            dv.x[base + p] = uniform_token(draw_u32(sl.seed, kPurposeRenoise, b, s, p), dv.V);
            if (was[i]) {  // only under DG_REACCEPT: accepted before, re-noised now
              dv.committed[base + p] = 0;
              ++remasked;
            }
          }
        }
        dv.prev_amax[base + p] = av[i];
      }
    }
    if (dv.reaccept && remasked) atomicAdd(&sc->remasked, remasked);
    g.sync();
    if (g.tid == 0) {
      dg_slot& so = dv.slots[c];
      so.step = s + 1;
      so.temperature = t_next;
      so.n_committed = dv.reaccept ? n_acc : sl.n_committed + n_acc;
      so.n_remasked = sc->remasked;
      so.stable_steps = run;
      so.mean_entropy = mean_H;
    }
    g.sync();
    return kActive;
  } else {
#pragma unroll
    for (int i = 0; i < kTailPer; ++i) {
      const int p = g.tid + i * kTailThreads;
      if (p < L) {
        int xo = xv[i];
        int16_t cs = (int16_t)s;
        if (!cm[i]) {
          xo = DG_IN_BOUNDS(dv.plan, yv[i] >= 0 && yv[i] < dv.V, 4, yv[i]) ? yv[i] : xv[i];
          dv.x[base + p] = xo;
          dv.committed[base + p] = 1;
          dv.commit_step[base + p] = cs;
        } else {
          cs = __ldcg(dv.commit_step + base + p);
        }
        dv.tokens_out[((size_t)c * dv.G + b) * L + p] = xo;
        dv.commit_steps_out[((size_t)c * dv.G + b) * L + p] = cs;
      }
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
      so.n_remasked = 0;
      so.stable_steps = 0;
      if (more) {
        so.block = b + 1;
        so.step = 0;
        so.temperature = t_first;
        so.n_committed = 0;
      } else {
        so.n_committed = L;
        so.state = kDone;
      }
    }
    g.sync();
    return more ? kActive : kDone;
  }
}

}  // namespace dg
