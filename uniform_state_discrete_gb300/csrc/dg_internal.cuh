// Internal declarations of the denoise-step library (sm_103a): workspace
// view, device helpers and the PTX wrappers the kernels use.  Not part of the
// public ABI (include/dg_sampler.h is).
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver entry point is looked up at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_sampler.h"

namespace dg {

// ---------------------------------------------------------------- tiling
// LM-head GEMM tile: 128 canvas positions (TMEM lanes) x 256 vocabulary rows
// (TMEM columns) per accumulator, K staged 64 bf16 (one 128-byte swizzle row)
// at a time.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kStageA = kBM * kBK * 2;  // 16 KB
constexpr int kStageB = kBN * kBK * 2;  // 32 KB
// on SM pairs (cta_group::2) each CTA stages its own 128 rows of A and its own 128-row half of B
constexpr int kStagesPair = 6;
constexpr int kStagePairA = kBM * kBK * 2;        // 16 KB
constexpr int kStagePairB = (kBN / 2) * kBK * 2;  // 16 KB
constexpr int kEpiWarps = 16;           // four per TMEM lane quadrant, each owning 64 of the 256 columns
constexpr int kThreadsLM = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 2 * kBN;      // double-buffered accumulator
// The vocabulary is cut into this many chunks (fewer when V is small),
// independent of how many canvases are active, so a position's statistics do
// not depend on the batch it runs in.
constexpr int kChunkTarget = 76;
constexpr int kColGroups = kEpiWarps / 4;
constexpr int kColsPerWarp = kBN / kColGroups;  // 64
constexpr int kSubPerChunk = 1;                 // column groups are merged in the CTA before writing

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits give up after 1 s

// Philox counter "purpose" word (word 3); see the oracle's definition.
enum : uint32_t { kPurposeInit = 2u, kPurposeRenoise = 4u, kPurposeGumbelOrder = 5u };
enum : int32_t { kWaiting = 0, kActive = 1, kDone = 2 };
// Device error codes latched in Plan::err.
enum : int32_t { kErrNone = 0, kErrNonFinite = 1, kErrTimeout = 2, kErrBounds = 3 };

// Split-vocabulary partial statistics of one position over one column range,
// in base-2 units: u = z * log2(e) / T.
//   m = max u, S = sum 2^(u-m), A = sum 2^(u-m) (u-m),
//   g = max (u - log2 E_v) with E_v the Exp(1) variate of the Gumbel draw.
struct Partial {
  float m, S, A, g;
  int32_t amax, gidx, pad0, pad1;
};
static_assert(sizeof(Partial) == 32, "partial record is 32 bytes");

struct Plan {
  int32_t tick;
  int32_t n_active;
  uint32_t commits;  // canvases committed so far this tick
  int32_t err;
  int32_t err_info[4];
  uint32_t epoch;    // advanced by every planning; tags this tick's per-row best Gumbel scores
};

// Everything a kernel needs, by value.
struct Dev {
  dg_slot* slots;       // [B]
  Plan* plan;
  int32_t* active;      // [B] active canvas ids, in canvas order
  int32_t* x;           // [B, L]
  uint8_t* committed;   // [B, L]
  int16_t* commit_step; // [B, L]
  int32_t* prev_amax;   // [B, L]
  int32_t* tokens_out;  // [B, G, L]
  int16_t* commit_steps_out; // [B, G, L] commit step of each position of each finished block
  float* H;             // [B, L]
  float* logZ;          // [B, L]
  int32_t* y;           // [B, L]
  int32_t* amax;        // [B, L]
  uint16_t* h;          // [rows_cap, d] bf16 bits, compact active rows
  Partial* part;        // [rows_cap, n_sub]
  unsigned long long* row_best; // [rows_cap] best perturbed score found so far for each row this tick,
                                //   (epoch << 32) | ordered score bits; other epochs read as none
  uint32_t* canvas_rows;// [B] rows combined per canvas this tick
  uint32_t* rows_ready; // normalised rows written this tick (RMSNorm -> LM-head producers)
  uint32_t* fin_started;// finishing-kernel CTAs that have read this tick's plan
  uint32_t* slab_done;  // [rows_cap / 128] LM-head units finished per 128-row slab (-> finishing kernel)
  uint32_t* units_done; // LM-head units finished this tick, counted by the rank-0 CTA of a pair (paces the producers)
  float* resid_stage;   // [B, L, d]
  const float* norm_w;  // [d] or null
  const float* temps;   // [N] temperature of each step, T_s = t_max + (s/N)(t_min - t_max)
  int32_t V, d, L, B, G, N;
  float t_min, t_max, bound, conf, eps;
  int32_t n_vtiles, tiles_per_chunk, n_chunks, n_sub, rows_cap, max_active;
  // vocabulary chunks this LM head computes, [chunk_begin, chunk_end) of the n_chunks (all of them
  // unless the vocabulary is split across ranks), and the first vocabulary tile of the W rows the
  // tensor map covers (its row 0 is vocabulary entry vt_base * kBN)
  int32_t chunk_begin, chunk_end, vt_base;
  // self-conditioning (dg_self_condition; all null / 0 when the sampler was created without it):
  // what a tick leaves for it -- each row's temperature factor log2(e)/T (LM head), its log2 Z
  // and canvas (finishing kernel) and the tick's row count -- and its buffers
  float* row_scale;        // [rows_cap]
  float* row_log2z;        // [rows_cap]
  int32_t* row_canvas;     // [B] canvas of each active slot a (rows a L .. a L + L - 1)
  uint32_t* sc_rows;       // rows of the last tick
  uint16_t* sc_probs;      // [rows_cap, sc_vpad] bf16 P
  float* sc_part;          // [sc_kc, rows_cap, d] per-chunk shares of P W
  int32_t sc_vpad, sc_kc, sc_kbpc;  // V rounded up to 256; vocabulary chunks of the contraction, 64-wide K blocks each
  bool reaccept;        // DG_REACCEPT: every step re-sorts all positions (see dg_mode)
  int32_t stability;    // early stop needs this many consecutive steps with an unchanged argmax canvas
  float softcap;        // final logit softcap c (0 = off): z -> c tanh(z / c) before the temperature
  float inv_softcap;    // 1 / c (0 when off)
  int32_t hold_slabs;   // test hook (dg_debug_hold_slabs): the LM head does not count finished units
};

// ------------------------------------------------------------ expired waits
// Where a bounded wait gave up.  The first wait to give up latches DG_ERR_TIMEOUT with
// its CTA (err_info[0]), its site (err_info[2]) and a detail (err_info[3]: a barrier's
// shared-memory offset times 2 plus the parity waited for, or the counter's value);
// later ones, which usually wait on the first, leave the latch as it is.
enum : int32_t {
  kWaitRowsReady = 1,   // LM-head producer: normalised rows of the tick
  kWaitPacing = 2,      // LM-head producer: units of the previous round
  kWaitBarrier = 3,     // LM-head: an mbarrier phase (stage ring, TMEM buffers)
  kWaitFinStarted = 4,  // finishing kernel: every CTA has read the plan
  kWaitSlab = 5,        // finishing kernel: LM-head units of a 128-row slab
};
inline const char* wait_site_name(int site) {
  switch (site) {
    case kWaitRowsReady: return "LM head, normalised rows";
    case kWaitPacing: return "LM head, pacing of the unit rounds";
    case kWaitBarrier: return "LM head, stage or TMEM barrier";
    case kWaitFinStarted: return "finishing kernel, plan read by every CTA";
    case kWaitSlab: return "finishing kernel, LM-head units of a slab";
    default: return "unknown site";
  }
}
__device__ __noinline__ inline void timeout_latch(Plan* plan, int cta, int site, long long detail) {
  if (atomicCAS(&plan->err, kErrNone, kErrTimeout) == kErrNone) {
    plan->err_info[0] = cta;
    plan->err_info[2] = site;
    plan->err_info[3] = (int)detail;
  }
}

// ------------------------------------------------------------ debug index checks
// In the debug build (DG_DEBUG_CHECKS) an index check that fails latches
// DG_ERR_BOUNDS with the check's site number and the offending value in the
// plan and makes the caller skip the access; nothing traps.  In the release
// build the checks compile to nothing.
__device__ __noinline__ inline bool bounds_fail(Plan* plan, int site, long long value) {
  if (atomicCAS(&plan->err, kErrNone, kErrBounds) == kErrNone) {
    plan->err_info[2] = site;
    plan->err_info[3] = (int)value;
  }
  return false;
}
#ifdef DG_DEBUG_CHECKS
#define DG_IN_BOUNDS(plan, cond, site, value) ((cond) || ::dg::bounds_fail((plan), (site), (long long)(value)))
#else
#define DG_IN_BOUNDS(plan, cond, site, value) true
#endif

// ------------------------------------------------------------ Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): ten rounds of two 32x32->64 multiplies, key bumped by the Weyl
// constants between rounds.
__device__ __forceinline__ uint4 philox(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;  // one 32x32->64 multiply each
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ (k0 + (uint32_t)r * 0x9E3779B9u), (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ (k1 + (uint32_t)r * 0xBB67AE85u), (uint32_t)p0);
  }
  return c;
}

// One word for a per-position draw (initial canvas, re-noise): counter
// (0, p, (block<<16)|step, purpose), key = canvas seed, lane 0.
__device__ __forceinline__ uint32_t draw_u32(uint64_t seed, uint32_t purpose, int block, int step, int p) {
  return philox(make_uint4(0u, (uint32_t)p, ((uint32_t)block << 16) | (uint32_t)step, purpose), (uint32_t)seed,
                (uint32_t)(seed >> 32)).x;
}

// Uniform token in [0, V): Lemire's multiply-shift.
__device__ __forceinline__ int32_t uniform_token(uint32_t u, int32_t V) {
  return (int32_t)(((uint64_t)u * (uint64_t)(uint32_t)V) >> 32);
}

// ------------------------------------------------------------ small PTX
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream still runs;
// pdl_wait() blocks until that predecessor has completed and its memory is
// visible (it returns at once when there is none), pdl_allow_next() lets the
// successor begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// The same, issued only once `v` is in a register: a value read from the plan
// before this call has arrived, so a dependent kernel that rewrites the plan
// cannot change what this thread saw.
__device__ __forceinline__ void pdl_allow_next_after(int v) {
  asm volatile("griddepcontrol.launch_dependents;" ::"r"(v) : "memory");
}

// Counters that hand data from one CTA or kernel of a tick to another without
// waiting for a whole grid: after a CTA barrier one thread of the writer adds
// to the counter with release semantics, so the CTA's earlier memory
// operations are visible before the addition is; the reader acquires it (one
// thread, followed by a CTA barrier), spinning until the count it needs is
// reached and giving up after kWaitLimitNs.  The planner of the next tick
// resets them.  Release and acquire each fold the fence into the one access.
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Both at once, for a counter whose old value elects the CTA that goes on with
// every contributor's data: returns the value before the addition.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait until *cnt >= target; false if kWaitLimitNs passed first.
__device__ __forceinline__ bool wait_count(const uint32_t* cnt, uint32_t target) {
  if (ld_acquire(cnt) >= target) return true;
  const uint64_t t0 = now_ns();
  while (ld_acquire(cnt) < target) {
    if (now_ns() - t0 > kWaitLimitNs) return false;
    __nanosleep(64);
  }
  return true;
}

// Merge two partial records (base-2 units).  Ties keep the lower vocabulary index.
__device__ __forceinline__ Partial merge_partial(const Partial& a, const Partial& b) {
  Partial r;
  r.m = fmaxf(a.m, b.m);
  const float fa = a.S > 0.f ? ex2_approx(a.m - r.m) : 0.f;
  const float fb = b.S > 0.f ? ex2_approx(b.m - r.m) : 0.f;
  r.S = fa * a.S + fb * b.S;
  r.A = (a.S > 0.f ? fa * fmaf(a.m - r.m, a.S, a.A) : 0.f) + (b.S > 0.f ? fb * fmaf(b.m - r.m, b.S, b.A) : 0.f);
  const bool ta = (a.m > b.m) || (a.m == b.m && a.amax < b.amax);
  r.amax = ta ? a.amax : b.amax;
  const bool ga = (a.g > b.g) || (a.g == b.g && a.gidx < b.gidx);
  r.g = ga ? a.g : b.g;
  r.gidx = ga ? a.gidx : b.gidx;
  r.pad0 = r.pad1 = 0;
  return r;
}

// A partial record written by another kernel, read at L2.
__device__ __forceinline__ Partial load_partial(const Partial* p) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  Partial r;
  r.m = a.x;
  r.S = a.y;
  r.A = a.z;
  r.g = a.w;
  r.amax = b.x;
  r.gidx = b.y;
  r.pad0 = b.z;
  r.pad1 = b.w;
  return r;
}

// Order-preserving unsigned image of a float (for atomicMax on scores) and back.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// The best score a row's word records for this epoch, or -inf.
__device__ __forceinline__ float row_best_decode(unsigned long long v, uint32_t epoch) {
  return (uint32_t)(v >> 32) == epoch ? key_score((uint32_t)v) : -INFINITY;
}
__device__ __forceinline__ float row_best_score(const unsigned long long* e, uint32_t epoch) {
  return row_best_decode(__ldcg(e), epoch);
}
__device__ __forceinline__ void row_best_raise(unsigned long long* e, uint32_t epoch, float score) {
  atomicMax(e, ((unsigned long long)epoch << 32) | score_key(score));
}

__device__ __forceinline__ Partial empty_partial() {
  Partial p;
  p.m = -INFINITY;
  p.S = 0.f;
  p.A = 0.f;
  p.g = -INFINITY;
  p.amax = 0x7FFFFFFF;
  p.gidx = 0x7FFFFFFF;
  p.pad0 = p.pad1 = 0;
  return p;
}

// ------------------------------------------------------------- launchers
// Implemented in dg_kernels.cu / dg_lmhead.cu; all enqueue on `st`.
cudaError_t launch_rmsnorm(const Dev& dv, const float* resid, cudaStream_t st);
cudaError_t launch_lmhead(const Dev& dv, const CUtensorMap* tmA, const CUtensorMap* tmB, int num_sms,
                          cudaStream_t st);
cudaError_t launch_lmhead_pair(const Dev& dv, const float* resid, const CUtensorMap* tmA, const CUtensorMap* tmB, int num_sms,
                               cudaStream_t st);
cudaError_t launch_finish(const Dev& dv, cudaStream_t st);
cudaError_t launch_plan(const Dev& dv, int tick, cudaStream_t st);
cudaError_t lmhead_configure();
cudaError_t selfcond_configure();
cudaError_t launch_transpose_w(const void* w, uint16_t* wt, int V, int d, int v_pad, cudaStream_t st);
// pair: the sampler runs its LM head on SM pairs (256 positions and up); tm_w and tm_wt then have
// 128-row boxes, else 256-row ones
cudaError_t launch_selfcond(const Dev& dv, bool pair, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                            const CUtensorMap* tm_p, const CUtensorMap* tm_wt, float* out, int num_sms, cudaStream_t st);

}  // namespace dg
