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

// Finishing kernel of a tick.  Each warp combines the split-vocabulary partial
// records of one active position: log2 Z = m + log2 S, H = ln 2 (log2 S - A/S)
// (= log Z - E_p[z/T] in nats), the sample is the index of the largest
// perturbed score and the argmax the index of the largest logit.  Each CTA then
// credits its positions to their canvases; the CTA that completes a canvas
// commits it (dg_tail.cuh), and the last commit plans the next tick.  No CTA
// waits for another: the last arrival at a counter does the work.
constexpr int kFinishRows = 8;  // positions (warps) per CTA

__global__ void __launch_bounds__(256) k_finish(const Dev dv) {
  __shared__ TailScratch sc;
  pdl_wait();
  pdl_allow_next();
  const Group g{(int)threadIdx.x, (int)blockDim.x, 0};
  const int n_rows = dv.plan->n_active * dv.L;
  if (n_rows == 0) {
    if (blockIdx.x == 0) plan_tick(dv, dv.plan->tick + 1, g, &sc);
    return;
  }
  const int row0 = blockIdx.x * kFinishRows;
  if (row0 >= n_rows) return;
  const int row1 = min(row0 + kFinishRows, n_rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = row0 + warp;
  if (row < row1) {
    Partial acc = empty_partial();
    const Partial* src = dv.part + (size_t)row * dv.n_sub;
    for (int i = lane; i < dv.n_sub; i += 32) acc = merge_partial(acc, src[i]);
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
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int nd = 0;
    for (int a = row0 / dv.L; a * dv.L < row1; ++a) {
      const int lo = max(a * dv.L, row0), hi = min((a + 1) * dv.L, row1);
      const int c = dv.active[a];
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
    if (threadIdx.x == 0)
      sc.flags[1] = (atomicAdd(&dv.plan->commits, 1u) == (unsigned)(__ldcg(&dv.plan->n_active) - 1)) ? 1 : 0;
    __syncthreads();
    const int plan_now = sc.flags[1];
    __syncthreads();
    if (plan_now) {
      __threadfence();
      plan_tick(dv, __ldcg(&dv.plan->tick) + 1, g, &sc);
    }
  }
}

// Planner kernel (sampler creation and dg_set_state): clears the tick's
// counters, which an interrupted tick may have left behind, then plans `tick`.
__global__ void __launch_bounds__(256) k_plan(const Dev dv, int tick) {
  __shared__ TailScratch sc;
  for (int i = threadIdx.x; i < dv.B; i += blockDim.x) dv.canvas_rows[i] = 0u;
  __syncthreads();
  plan_tick(dv, tick, Group{(int)threadIdx.x, (int)blockDim.x, 0}, &sc);
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
  return launch_pdl(k_rmsnorm, dim3((rows + 7) / 8), dim3(256), 0, st, resid, dv);
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
