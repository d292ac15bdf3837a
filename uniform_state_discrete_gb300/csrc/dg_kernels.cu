// The RMSNorm kernel (K1, for the single-CTA LM head), the finishing kernel
// (K3: split-vocabulary combine, entropy-bounded commit, re-noise and
// next-tick plan) and the stand-alone tick planner.
#include <cuda_runtime.h>
#include <math.h>

#include <utility>

#include "dg_internal.cuh"
#include "dg_norm.cuh"
#include "dg_tail.cuh"

namespace dg {
namespace {

// ------------------------------------------------------------------- K1
// RMSNorm per active row, for the single-CTA LM head (the kernel on SM pairs
// forms its rows itself).  Layout for latency: one CTA of kNormThreads (four
// warps) per row; a row of up to kNormThreads * kNormVec float4 (d <= 3072)
// is held in registers, so the kernel costs about one memory round trip.
constexpr int kNormThreads = 128;
constexpr int kNormVec = 6;

__global__ void __launch_bounds__(kNormThreads) k_rmsnorm(const float* __restrict__ resid, const Dev dv) {
  __shared__ float red[kNormThreads / 32][2];
  pdl_wait();
  pdl_allow_next();
  const int n_rows = dv.plan->n_active * dv.L;
  if ((int)blockIdx.x >= n_rows) return;  // uniform per CTA
  const int row = blockIdx.x;
  const int a = row / dv.L, p = row - a * dv.L;
  if (!DG_IN_BOUNDS(dv.plan, row < dv.rows_cap && dv.active[a] >= 0 && dv.active[a] < dv.B, 9, row)) return;
  norm_row<kNormThreads, kNormVec>(resid + ((size_t)dv.active[a] * dv.L + p) * dv.d, dv.norm_w,
                                   dv.h + (size_t)row * dv.d, dv.d, dv.eps, (int)threadIdx.x, red,
                                   [] { __syncthreads(); });
  // the row is written: count it for the LM head, which waits for all rows
  if (threadIdx.x == 0) red_release_add(dv.rows_ready, 1u);
}

// Finishing kernel of a tick.  Each warp combines the split-vocabulary partial
// records of one active position: log2 Z = m + log2 S, H = ln 2 (log2 S - A/S)
// (= log Z - E_p[z/T] in nats), the sample is the index of the largest
// perturbed score and the argmax the index of the largest logit.  Each CTA then
// credits its positions to their canvases; the CTA that completes a canvas
// commits it (dg_tail.cuh), and the last commit plans the next tick.  No CTA
// waits for another: the last arrival at a counter does the work.
constexpr int kFinishRows = 8;  // positions (warps) per CTA

static_assert(kFinishRows <= (int)(sizeof(TailScratch::row_canvas) / sizeof(int)), "row_canvas holds a CTA's rows");

// The planner of k_finish: waits (bounded) until every CTA of the grid has read
// this tick's plan, then plans the next tick.  `started` says that thread 0
// already saw every CTA counted, with an acquire load, so no wait is needed;
// known_c / known_state pass on a slot the group wrote.
__device__ __forceinline__ void plan_next_tick(const Dev& dv, int tick, const Group& g, TailScratch* sc,
                                               bool started = false, int known_c = -1, int known_state = kDone) {
  if (g.tid == 0 && !started) {
    if (!wait_count(dv.fin_started, gridDim.x))
      timeout_latch(dv.plan, (int)blockIdx.x, kWaitFinStarted, *(volatile uint32_t*)dv.fin_started);
  }
  g.sync();
  plan_tick(dv, tick + 1, g, sc, false, known_c, known_state);
}

// It does not wait for the whole LM-head grid: each CTA waits for the LM-head
// units of its rows' 128-row slab (dv.slab_done), so it starts combining as
// soon as the last partial record of those rows is written.  Data of earlier
// kernels is read at L2.
__global__ void __launch_bounds__(256) k_finish(const Dev dv) {
  __shared__ TailScratch sc;
  const Group g{(int)threadIdx.x, (int)blockDim.x, 0};
  // Each CTA reads the tick's plan, then counts itself as started; the planner of
  // the next tick rewrites the plan only once every CTA of this grid has started,
  // so a CTA that starts late cannot mistake the next tick's plan for this one's.
  const int n_rows = __ldcg(&dv.plan->n_active) * dv.L;
  const int tick = __ldcg(&dv.plan->tick);
  if (dv.sc_rows && blockIdx.x == 0 && threadIdx.x == 0) *dv.sc_rows = (uint32_t)n_rows;  // for self-conditioning
  __syncthreads();
  if (threadIdx.x == 0) red_release_add(dv.fin_started, 1u);  // after every thread's reads of the plan
  pdl_allow_next();
  if (n_rows == 0) {
    if (blockIdx.x == 0) plan_next_tick(dv, tick, g, &sc);
    return;
  }
  const int row0 = blockIdx.x * kFinishRows;
  if (row0 >= n_rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = row0 + warp;
  // the canvas of this warp's row, read before the wait so its latency is hidden
  int row_c = (lane == 0 && row < n_rows) ? __ldcg(dv.active + row / dv.L) : 0;
  if (lane == 0 && !DG_IN_BOUNDS(dv.plan, row_c >= 0 && row_c < dv.B, 5, row_c)) row_c = 0;
  if (threadIdx.x == 0) {
    const bool ok = wait_count(dv.slab_done + row0 / 128, (uint32_t)(dv.chunk_end - dv.chunk_begin));
    if (!ok) timeout_latch(dv.plan, (int)blockIdx.x, kWaitSlab, row0 / 128);
  }
  __syncthreads();
  const int row1 = min(row0 + kFinishRows, n_rows);
  if (row < row1) {
    Partial acc = empty_partial();
    const Partial* src = dv.part + (size_t)row * dv.n_sub;
    for (int i = lane; i < dv.n_sub; i += 32) acc = merge_partial(acc, load_partial(src + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Partial b;
      b.m = __shfl_xor_sync(0xFFFFFFFFu, acc.m, o);
      b.S = __shfl_xor_sync(0xFFFFFFFFu, acc.S, o);
      b.A = __shfl_xor_sync(0xFFFFFFFFu, acc.A, o);
      b.g = __shfl_xor_sync(0xFFFFFFFFu, acc.g, o);
      b.amax = __shfl_xor_sync(0xFFFFFFFFu, acc.amax, o);
      b.gidx = __shfl_xor_sync(0xFFFFFFFFu, acc.gidx, o);
      b.pad0 = b.pad1 = 0;
      acc = merge_partial(acc, b);
    }
    if (lane == 0) {
      const int a = row / dv.L, p = row - a * dv.L;
      const int c = row_c;
      sc.row_canvas[warp] = c;
      const float l2S = log2f(acc.S);
      const float H = 0.69314718055994531f * (l2S - acc.A / acc.S);
      const float lz = 0.69314718055994531f * (acc.m + l2S);
      const size_t o = (size_t)c * dv.L + p;
      dv.H[o] = H > 0.f ? H : 0.f;  // +0 for rounding below zero (and never -0: its bits would sort last)
      dv.logZ[o] = lz;
      if (dv.row_log2z) {  // what the self-conditioning pass reads after the tick
        dv.row_log2z[row] = acc.m + l2S;
        if (p == 0) dv.row_canvas[a] = c;
      }
      // a row without valid statistics latches an error and never hands an
      // out-of-range token to the canvas (callers index embeddings with it)
      const bool y_ok = acc.gidx >= 0 && acc.gidx < dv.V, a_ok = acc.amax >= 0 && acc.amax < dv.V;
      dv.y[o] = y_ok ? acc.gidx : 0;
      dv.amax[o] = a_ok ? acc.amax : 0;
      if (!isfinite(H) || !isfinite(lz) || !isfinite(acc.g) || !y_ok || !a_ok) {
        if (atomicCAS(&dv.plan->err, kErrNone, kErrNonFinite) == kErrNone) dv.plan->err_info[1] = (int)o;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Release this CTA's rows to the canvas counter; the CTA that completes a canvas
    // acquires every other CTA's rows of it with the same access.
    int nd = 0;
    for (int a = row0 / dv.L; a * dv.L < row1; ++a) {
      const int lo = max(a * dv.L, row0), hi = min((a + 1) * dv.L, row1);
      const int c = sc.row_canvas[lo - row0];
      const unsigned old = atom_add_acq_rel(&dv.canvas_rows[c], (unsigned)(hi - lo));
      if (old + (unsigned)(hi - lo) == (unsigned)dv.L) {
        dv.canvas_rows[c] = 0u;  // every row of this canvas is combined: reset for the next tick
        sc.done_list[nd++] = c;
      }
    }
    sc.flags[3] = nd;
  }
  __syncthreads();
  const int nd = sc.flags[3];
  const int na = n_rows / dv.L;  // canvases active this tick
  for (int i = 0; i < nd; ++i) {
    const int c = sc.done_list[i];
    // whether every CTA of the grid has started (an acquire: the plan is rewritten after it)
    const bool started = threadIdx.x == 0 && ld_acquire(dv.fin_started) >= gridDim.x;
    const int state = commit_canvas(dv, c, g, &sc);
    __syncthreads();
    if (threadIdx.x == 0) {
      // The last commit of the tick plans the next; alone, this one is the last and
      // plans right away from what it wrote itself.  With several canvases the
      // commit counter releases this commit's writes and acquires the others'.
      sc.flags[1] = (na == 1 || atom_add_acq_rel(&dv.plan->commits, 1u) == (unsigned)(na - 1)) ? 1 : 0;
    }
    __syncthreads();
    const int plan_now = sc.flags[1];
    __syncthreads();
    if (plan_now) plan_next_tick(dv, tick, g, &sc, started, c, state);
  }
}

// Planner kernel (sampler creation and dg_set_state): clears the tick's
// counters and the error latch, which an interrupted tick may have left
// behind, then plans `tick`.
__global__ void __launch_bounds__(256) k_plan(const Dev dv, int tick) {
  __shared__ TailScratch sc;
  for (int i = threadIdx.x; i < dv.B; i += blockDim.x) dv.canvas_rows[i] = 0u;
  if (threadIdx.x == 0) {
    dv.plan->err = kErrNone;
    for (int i = 0; i < 4; ++i) dv.plan->err_info[i] = 0;
  }
  __syncthreads();
  plan_tick(dv, tick, Group{(int)threadIdx.x, (int)blockDim.x, 0}, &sc, true);
}

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

}  // namespace

cudaError_t launch_rmsnorm(const Dev& dv, const float* resid, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;
  return launch_pdl(k_rmsnorm, dim3(rows), dim3(kNormThreads), 0, st, resid, dv);
}

cudaError_t launch_finish(const Dev& dv, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;
  return launch_pdl(k_finish, dim3((rows + kFinishRows - 1) / kFinishRows), dim3(256), 0, st, dv);
}

cudaError_t launch_plan(const Dev& dv, int tick, cudaStream_t st) {
  k_plan<<<1, 256, 0, st>>>(dv, tick);
  return cudaGetLastError();
}

}  // namespace dg
