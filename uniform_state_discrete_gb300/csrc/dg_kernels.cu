// K1 RMSNorm, the finishing kernel (split-vocabulary combine, entropy-bounded
// commit, re-noise and next-tick plan) and the stand-alone tick planner.
#include <cuda_runtime.h>
#include <math.h>

#include <utility>

#include "dg_internal.cuh"
#include "dg_tail.cuh"

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

// Accumulate x^2 into the unevaluated pair (sh, sl): the square is split
// exactly by an FMA, its high part added by TwoSum, all low parts summed.
__device__ __forceinline__ void acc_square(float x, float& sh, float& sl) {
  const float sq = __fmul_rn(x, x);
  const float sq_err = fmaf(x, x, -sq);
  float e;
  two_sum(sh, sq, sh, e);
  sl = __fadd_rn(sl, __fadd_rn(e, sq_err));
}

// bf16 bits of w x (inv_hi + inv_lo), rounded as the exact product would be.
__device__ __forceinline__ uint32_t scaled_bf16(float x, float w, float inv_hi, float inv_lo) {
  const float xw = __fmul_rn(w, x);  // w x = xw + xw_err exactly
  const float xw_err = fmaf(w, x, -xw);
  const float ph = __fmul_rn(xw, inv_hi);  // (w x) inv ~= ph + pl
  const float pe = fmaf(xw, inv_hi, -ph);
  const float pl = fmaf(xw, inv_lo, fmaf(xw_err, inv_hi, pe));
  const float hi = __fadd_rn(ph, pl);  // renormalise: |lo| <= ulp(hi)/2
  const float lo = __fsub_rn(pl, __fsub_rn(hi, ph));
  return bf16_rne_pair(hi, lo) & 0xFFFFu;
}

// sqrt(d) / (sqrt(h + l) + eps) as an unevaluated fp32 pair, to ~2^-46
// relative, in double-float arithmetic (Dekker 1971): a square root and a
// quotient rounded in fp32 and corrected by their exact FMA residues.
__device__ __forceinline__ void row_scale(float h, float l, int d, float eps, float& inv_hi, float& inv_lo) {
  // norm = sqrt(h + l): r = fl(sqrt(h)), then r + (h + l - r^2) / (2r)
  const float r = __fsqrt_rn(h);
  const float p = __fmul_rn(r, r);
  const float pe = fmaf(r, r, -p);  // r^2 = p + pe exactly
  const float r_lo = __fdiv_rn(__fadd_rn(__fsub_rn(__fsub_rn(h, p), pe), l), __fmul_rn(2.f, r));
  // den = norm + eps, renormalised
  float dh, de;
  two_sum(r, eps, dh, de);
  de = __fadd_rn(de, r_lo);
  const float den_hi = __fadd_rn(dh, de);
  const float den_lo = __fsub_rn(de, __fsub_rn(den_hi, dh));
  // sqrt(d) = sd + sd_lo (d is an integer, exact in fp32)
  const float fd = (float)d;
  const float sd = __fsqrt_rn(fd);
  const float sd_lo = __fdiv_rn(fmaf(-sd, sd, fd), __fmul_rn(2.f, sd));
  // quotient: q = fl(sd / den_hi), remainder sd - q den_hi exact by FMA
  const float q = __fdiv_rn(sd, den_hi);
  const float rem = __fadd_rn(fmaf(-q, den_hi, sd), fmaf(-q, den_lo, sd_lo));
  const float q_lo = __fdiv_rn(rem, den_hi);
  inv_hi = __fadd_rn(q, q_lo);
  inv_lo = __fsub_rn(q_lo, __fsub_rn(inv_hi, q));
}

// h = bf16( w * r * sqrt(d) / (||r||_2 + eps) ) per active row.  The rounding
// of every element is the one the exact quotient gives (up to ~2^-46
// relative): sum of squares in TwoSum pairs, the per-row scale sqrt(d) /
// (norm + eps) as a double-float fp32 pair (row_scale), and each product
// carried exactly before the bf16 rounding.
//
// Layout for latency: one CTA of kNormThreads (four warps) per row.  A row
// of up to kNormThreads * kNormVec float4 (d <= 3072) is loaded into
// registers with every load issued before the first use, so the kernel costs
// about one memory round trip; longer rows are read twice.  At most 40
// registers a thread: two of these CTAs fit on an SM beside an LM-head CTA, so
// the LM head starts, and loads its first W stages, while the rows are formed.
constexpr int kNormThreads = 128;
constexpr int kNormVec = 6;

__global__ void __launch_bounds__(kNormThreads, 12) k_rmsnorm(const float* __restrict__ resid, const Dev dv) {
  __shared__ float red[kNormThreads / 32][2];
  pdl_wait();
  pdl_allow_next();
  const int n_rows = dv.plan->n_active * dv.L;
  if ((int)blockIdx.x >= n_rows) return;  // uniform per CTA
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int row = blockIdx.x;
  const int n4 = dv.d >> 2;
  const bool in_regs = n4 <= kNormThreads * kNormVec;
  const int a = row / dv.L, p = row - a * dv.L;
  const float4* r4 = reinterpret_cast<const float4*>(resid + ((size_t)dv.active[a] * dv.L + p) * dv.d);
  float4 v[kNormVec];
  float sh = 0.f, sl = 0.f;
  if (in_regs) {
#pragma unroll
    for (int k = 0; k < kNormVec; ++k) {
      const int i = t + k * kNormThreads;
      v[k] = i < n4 ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kNormVec; ++k) {
      acc_square(v[k].x, sh, sl);
      acc_square(v[k].y, sh, sl);
      acc_square(v[k].z, sh, sl);
      acc_square(v[k].w, sh, sl);
    }
  } else {
    for (int i0 = t; i0 < n4; i0 += kNormThreads * kNormVec) {
#pragma unroll
      for (int k = 0; k < kNormVec; ++k) {
        const int i = i0 + k * kNormThreads;
        v[k] = i < n4 ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kNormVec; ++k) {
        acc_square(v[k].x, sh, sl);
        acc_square(v[k].y, sh, sl);
        acc_square(v[k].z, sh, sl);
        acc_square(v[k].w, sh, sl);
      }
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
  if (lane == 0) {
    red[warp][0] = sh;
    red[warp][1] = sl;
  }
  __syncthreads();
  // every thread forms the row's sum of squares and scale itself
  float h = red[0][0], l = red[0][1];
#pragma unroll
  for (int w = 1; w < kNormThreads / 32; ++w) {
    float e;
    two_sum(h, red[w][0], h, e);
    l = __fadd_rn(__fadd_rn(l, red[w][1]), e);
  }
  float inv_hi, inv_lo;
  row_scale(h, l, dv.d, dv.eps, inv_hi, inv_lo);
  uint2* out = reinterpret_cast<uint2*>(dv.h + (size_t)row * dv.d);
  const float4* w4 = reinterpret_cast<const float4*>(dv.norm_w);
  if (in_regs) {
#pragma unroll
    for (int k = 0; k < kNormVec; ++k) {
      const int i = t + k * kNormThreads;
      if (i < n4) {
        const float4 w = w4 ? __ldg(w4 + i) : make_float4(1.f, 1.f, 1.f, 1.f);
        out[i] = make_uint2(scaled_bf16(v[k].x, w.x, inv_hi, inv_lo) | (scaled_bf16(v[k].y, w.y, inv_hi, inv_lo) << 16),
                            scaled_bf16(v[k].z, w.z, inv_hi, inv_lo) | (scaled_bf16(v[k].w, w.w, inv_hi, inv_lo) << 16));
      }
    }
  } else {
    for (int i = t; i < n4; i += kNormThreads) {
      const float4 x = __ldg(r4 + i);
      const float4 w = w4 ? __ldg(w4 + i) : make_float4(1.f, 1.f, 1.f, 1.f);
      out[i] = make_uint2(scaled_bf16(x.x, w.x, inv_hi, inv_lo) | (scaled_bf16(x.y, w.y, inv_hi, inv_lo) << 16),
                          scaled_bf16(x.z, w.z, inv_hi, inv_lo) | (scaled_bf16(x.w, w.w, inv_hi, inv_lo) << 16));
    }
  }
  // the row is written: count it for the LM head, which waits for all rows
  __syncthreads();
  if (t == 0) {
    __threadfence();
    atomicAdd(dv.rows_ready, 1u);
  }
}

// Finishing kernel of a tick.  Each warp combines the split-vocabulary partial
// records of one active position: log2 Z = m + log2 S, H = ln 2 (log2 S - A/S)
// (= log Z - E_p[z/T] in nats), the sample is the index of the largest
// perturbed score and the argmax the index of the largest logit.  Each CTA then
// credits its positions to their canvases; the CTA that completes a canvas
// commits it (dg_tail.cuh), and the last commit plans the next tick.  No CTA
// waits for another: the last arrival at a counter does the work.
constexpr int kFinishRows = 8;  // positions (warps) per CTA

// The planner of k_finish: waits (bounded) until every CTA of the grid has read
// this tick's plan, then plans the next tick.
__device__ __forceinline__ void plan_next_tick(const Dev& dv, int tick, const Group& g, TailScratch* sc) {
  if (g.tid == 0) {
    if (!wait_count(dv.fin_started, gridDim.x) && atomicCAS(&dv.plan->err, kErrNone, kErrTimeout) == kErrNone)
      dv.plan->err_info[0] = -2;
  }
  g.sync();
  plan_tick(dv, tick + 1, g, sc, false);
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
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(dv.fin_started, 1u);
  }
  pdl_allow_next();
  if (n_rows == 0) {
    if (blockIdx.x == 0) plan_next_tick(dv, tick, g, &sc);
    return;
  }
  const int row0 = blockIdx.x * kFinishRows;
  if (row0 >= n_rows) return;
  if (threadIdx.x == 0) {
    const bool ok = wait_count(dv.slab_done + row0 / 128, (uint32_t)dv.n_chunks);
    if (!ok && atomicCAS(&dv.plan->err, kErrNone, kErrTimeout) == kErrNone) dv.plan->err_info[0] = -1 - (int)blockIdx.x;
  }
  __syncthreads();
  const int row1 = min(row0 + kFinishRows, n_rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = row0 + warp;
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
      const int c = __ldcg(dv.active + a);
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
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int nd = 0;
    for (int a = row0 / dv.L; a * dv.L < row1; ++a) {
      const int lo = max(a * dv.L, row0), hi = min((a + 1) * dv.L, row1);
      const int c = __ldcg(dv.active + a);
      const unsigned old = atomicAdd(&dv.canvas_rows[c], (unsigned)(hi - lo));
      if (old + (unsigned)(hi - lo) == (unsigned)dv.L) {
        dv.canvas_rows[c] = 0u;  // every row of this canvas is combined: reset for the next tick
        sc.done_list[nd++] = c;
      }
    }
    sc.flags[3] = nd;
  }
  __syncthreads();
  const int nd = sc.flags[3];
  for (int i = 0; i < nd; ++i) {
    const int c = sc.done_list[i];
    __threadfence();
    commit_canvas(dv, c, g, &sc);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      // the last commit of the tick plans the next; alone, this one is the last
      const int na = __ldcg(&dv.plan->n_active);
      sc.flags[1] = (na == 1 || atomicAdd(&dv.plan->commits, 1u) == (unsigned)(na - 1)) ? 1 : 0;
    }
    __syncthreads();
    const int plan_now = sc.flags[1];
    __syncthreads();
    if (plan_now) {
      __threadfence();
      plan_next_tick(dv, tick, g, &sc);
    }
  }
}

// Planner kernel (sampler creation and dg_set_state): clears the tick's
// counters, which an interrupted tick may have left behind, then plans `tick`.
__global__ void __launch_bounds__(256) k_plan(const Dev dv, int tick) {
  __shared__ TailScratch sc;
  for (int i = threadIdx.x; i < dv.B; i += blockDim.x) dv.canvas_rows[i] = 0u;
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
