// K2: the tied LM head z = h W^T on the 5th-generation tensor cores, fused
// with the temperature-softmax statistics and the Gumbel-max sample, so the
// [positions x V] logits never leave the SM.
//
// Pages: "The Annotated DiffusionGemma" -- the tied LM head at the end of
// "Complete DiffusionGemma model", the temperature divisor of "Apply
// temperature", the entropy of "Compute entropy", the sample drawn in
// "Denoise, stage, commit, and generate".  TensorSharp's DiffusionGemma doc
// ("5. Acceleration status") fuses output-norm + lm-head and then reduces
// per position on the device; here the reduction moves into the GEMM's own
// epilogue so the logits are never written.
//
// Two kernels share the epilogue.  k_lmhead_pair (256 positions and up) runs
// persistent clusters of two CTAs, one per SM, 576 threads each:
//   warp 0      TMA producer: this CTA's 128 rows of h and its 128-row half of
//               the 256-row W tile per K stage of 64, 128-byte swizzle,
//               6-stage mbarrier ring (completion on the leader's barriers);
//               the first W stages are loaded before the kernel waits for
//               anything, since W depends on no earlier kernel.
//   warp 1      allocates 512 TMEM columns for the pair; the leader's lane 0
//               issues tcgen05.mma.cta_group::2.kind::f16 (bf16 x bf16 -> fp32,
//               M=256, N=256, K=16) into one of two TMEM accumulators and
//               commits stage-release / accumulator-ready barriers to both CTAs.
//   warps 2..17 first form this CTA's share of the RMSNorm rows (dg_norm.cuh)
//               and count them; then the epilogue: four warps per TMEM lane
//               quadrant (rows), each owning 64 of the 256 columns; per element
//                 u = z * log2(e)/T, running (max, sum 2^(u-m), sum 2^(u-m)(u-m)),
//                 argmax, and the perturbed score u - log2 E_v of the
//                 Gumbel draw (E_v = -ln U_v, U_v from Philox).
// k_lmhead (fewer positions) is the same on one CTA: M=128, a 4-stage ring,
// rows formed beforehand by the RMSNorm kernel.
// Work unit = (row tile, vocabulary chunk); the epilogue keeps its running
// statistics in registers across the chunk's tiles, merges the four column
// groups in shared memory and writes one 32-byte partial record per row and
// chunk, then counts the unit on its 128-row slab for the finishing kernel.
// Every wait is bounded (1 s); on expiry the CTA latches an error, drains what
// it issued and frees TMEM.
#include <cuda_runtime.h>

#include "dg_gumbel.cuh"
#include "dg_internal.cuh"
#include "dg_norm.cuh"
#include "dg_tc.cuh"

namespace dg {
namespace {

struct RowMeta {
  GumbelStream gs;  // this position's Philox stream of Gumbel words
  float scale;      // log2(e) / T
  bool valid;
};

// Meta data of TMEM lane `row` of the current unit: the position's canvas
// seed, block, step and temperature.
__device__ __forceinline__ RowMeta row_meta(const Dev& dv, int row, int n_rows) {
  RowMeta rm;
  rm.valid = row < n_rows;
  rm.scale = 0.f;
  if (rm.valid) {
    const int a = row / dv.L;
    int c = __ldcg(dv.active + a);
    if (!DG_IN_BOUNDS(dv.plan, c >= 0 && c < dv.B, 7, c)) c = 0;
    const dg_slot* sl = dv.slots + c;
    rm.gs.init(__ldcg(&sl->seed), (uint32_t)(row - a * dv.L),
               ((uint32_t)__ldcg(&sl->block) << 16) | (uint32_t)__ldcg(&sl->step), kPurposeGumbelOrder);
    rm.scale = 1.4426950408889634f / __ldcg(&sl->temperature);
  } else {
    rm.gs.init(0ull, 0u, 0u, kPurposeGumbelOrder);
  }
  return rm;
}

// Screen factor K ~ 2^(m - g).  An entry can raise the best perturbed score g
// only if its Exp(1) variate E < 2^(u - g) = e 2^(m - g), where e = 2^(u - m) is
// its softmax weight.  The factor carries 0.2 % slack for the approximate
// exponentials and logarithms, plus the rounding of scores of magnitude up to
// |m| + 64, so the screen never drops an entry that could win.
__device__ __forceinline__ float screen_factor(float m, float g) {
  return ex2_approx(m - g) * fmaf(fabsf(m) + 64.f, 0x1p-20f, 1.002f);
}

// A lower bound of q = 1 - U without an integer-to-float conversion: with
// Ut = (r >> 9) 2^-23, U - Ut < 2^-23, so q >= 2 - f - 2^-23 for f = 1 + Ut, which
// one funnel shift builds exactly (and the subtraction from 2 - 2^-23 is exact).
__device__ __forceinline__ float screen_word(uint32_t r) { return __uint_as_float(__funnelshift_r(r, 0x7Fu, 9)); }

// The Exp(1) variate E = -ln U of a word r, U = (r + 0.5) 2^-32.  For U < 3/4,
// E comes from lg2(U).  For U >= 3/4, E = -ln(1 - q) with q = 1 - U taken
// exactly from the integer, through the series -ln(1-q) = 2 atanh(s) =
// 2 (s + s^3/3 + s^5/5 + ...), s = q / (2 - q) <= 1/7, truncated after s^9
// (relative error < 4e-10), which keeps small variates (large Gumbel values)
// accurate where lg2(U) would lose them.  Both branches are evaluated and one
// kept, so a warp scores in lockstep.
__device__ __forceinline__ float exp_variate(uint32_t r) {
  const float U = fmaf(__uint2float_rn(r), 0x1p-32f, 0x1p-33f);
  const float Eu = -0.69314718055994531f * lg2_approx(U);
  const float q = fmaf(__uint2float_rn(~r), 0x1p-32f, 0x1p-33f);
  const float sq = __fdividef(q, 2.0f - q);
  const float s2 = sq * sq;
  float t = fmaf(s2, 1.0f / 9.0f, 1.0f / 7.0f);
  t = fmaf(s2, t, 1.0f / 5.0f);
  t = fmaf(s2, t, 1.0f / 3.0f);
  t = fmaf(s2, t, 1.0f);
  const float Eq = 2.0f * sq * t;
  return r < 0xC0000000u ? Eu : Eq;
}

// Order-preserving int image of a float (for atomicMax on shared scores).
__device__ __forceinline__ int ord_key(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : (b ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float key_ord(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF)); }

// z[j] for a lane-varying j, by a four-level select tree (registers cannot be indexed).
__device__ __forceinline__ float select16(const float (&z)[16], uint32_t j) {
  float a[8];
  const bool b0 = j & 1u, b1 = j & 2u, b2 = j & 4u, b3 = j & 8u;
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = b0 ? z[2 * i + 1] : z[2 * i];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = b1 ? a[2 * i + 1] : a[2 * i];
#pragma unroll
  for (int i = 0; i < 2; ++i) a[i] = b2 ? a[2 * i + 1] : a[2 * i];
  return b3 ? a[1] : a[0];
}

// Index of the r-th set bit (from 0, lowest first) of a 16-bit mask holding more than r set bits.
__device__ __forceinline__ uint32_t nth_set_bit16(uint32_t mask, uint32_t r) {
  uint32_t pos = 0u, c = __popc(mask & 0xFFu);
  if (r >= c) {
    r -= c;
    pos = 8u;
  }
  c = __popc((mask >> pos) & 0xFu);
  if (r >= c) {
    r -= c;
    pos += 4u;
  }
  c = __popc((mask >> pos) & 0x3u);
  if (r >= c) {
    r -= c;
    pos += 2u;
  }
  return pos + (r >= ((mask >> pos) & 1u) ? 1u : 0u);
}

// Where a row's best perturbed score is kept: this CTA's column groups share
// `cta` (shared memory), every unit of the row in the tick shares `glob`
// (global memory, tagged with the tick's epoch).  `known` is the largest global
// value read so far, refreshed before every group; a stream publishes its own
// best to the global value as soon as it rises (its seed, then each fold that
// raised it), so the units of a row that run at the same time -- at small V,
// all of them -- screen against each other's finds within the same tile.
struct BestScore {
  int* cta;
  unsigned long long* glob;
  uint32_t epoch;
  float known;
  bool raised;  // this stream's best rose in the last fold and raised the CTA's (published right after)
};

// Fold 16 columns [v0, v0+16) of one row (raw fp32 logits z) into its running
// statistics and Gumbel sample (fold16 below: group_prep, then stats16, then
// screen16).  v0 is a multiple of 16, so the columns are one group of the
// Gumbel draws.  kTail: some of the columns lie at or beyond V.
//
// With a final logit softcap c > 0 each logit first becomes c tanh(z / c)
// ("The Annotated DiffusionGemma", "Logit Softcapping": part of the model,
// applied before the temperature); tanhf is CUDA's, within 2 ulp.  kCap
// selects the kernels compiled with the cap, so the uncapped ones carry none
// of its code.
//
// Softmax statistics in base 2 with u = z log2(e)/T: running max m, S = sum
// 2^(u-m), A = sum 2^(u-m)(u-m), formed from d = u - m = fma(z, log2(e)/T, -m).
// The argmax index is looked up only when the fold raises the running max.
//
// Gumbel-max sample: the perturbed score of entry v is (m + d) - log2 E_v with
// E_v its Exp(1) variate.  A group's sixteen variates are drawn in increasing
// order, E_(k) = E_(k-1) + X_k / (16 - k), each placed in a slot drawn
// uniformly from those still free (Renyi's representation of exponential
// order statistics; the counters are in dg_gumbel.cuh), so the group is walked
// from its smallest variate up and the walk stops as soon as
// E_(k) >= 2^(u_max - g): every entry not yet scored then scores below g, the
// best score known for the row -- this stream's own, one another column group
// of the CTA found (shared memory), or one any unit of the row found this tick
// (global memory).  Each is the score of a real entry, so the row's winner is
// always scored and the result equals the unscreened maximum.  The walk is
// started only if its first entry or the second order statistic can pass,
// tested on words of the first Philox block alone -- one block for sixteen
// entries, drawn before the tile's accumulator is ready (first_blocks).  Walks
// run one step per lane per round, all lanes of the warp together.  Equal
// scores keep the lower index.

// The logits of a group as the statistics and the screen take them: capped (kCap), with
// columns at or beyond V set to -inf (kTail); returns the group's maximum logit in `cmz`, or
// false when the whole group lies beyond V.
template <bool kTail, bool kCap>
__device__ __forceinline__ bool group_prep(float (&z)[16], int v0, int V, float cap, float inv_cap, float& cmz) {
  if (kCap) {
#pragma unroll
    for (int j = 0; j < 16; ++j) z[j] = cap * tanhf(z[j] * inv_cap);
  }
  if (kTail) {
    if (v0 >= V) return false;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (v0 + j >= V) z[j] = -INFINITY;
  }
  float t8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) t8[i] = fmaxf(z[i], z[i + 8]);
#pragma unroll
  for (int i = 0; i < 4; ++i) t8[i] = fmaxf(t8[i], t8[i + 4]);
  cmz = fmaxf(fmaxf(t8[0], t8[2]), fmaxf(t8[1], t8[3]));
  return true;
}

// The softmax statistics of a prepared group (the running max, S, A and the argmax).
template <bool kTail>
__device__ __forceinline__ void stats16(const float (&z)[16], float cmz, int v0, int V, const RowMeta& rm,
                                        Partial& st) {
  const float cm = cmz * rm.scale;
  if (cm > st.m) {
    const float f = ex2_approx(st.m - cm);
    st.A = st.S > 0.f ? f * fmaf(st.m - cm, st.S, st.A) : 0.f;
    st.S = f * st.S;
    st.m = cm;
    int ci = 15;
#pragma unroll
    for (int j = 15; j >= 0; --j)
      if (z[j] == cmz) ci = j;  // first index holding the maximum
    st.amax = v0 + ci;
  }
  const float nm = -st.m;
  float S[4] = {0.f, 0.f, 0.f, 0.f}, A[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float d = fmaf(z[j], rm.scale, nm);
    const float e = ex2_approx(d);  // +0 for a masked column (d = -inf)
    S[j & 3] += e;
    if (!kTail || v0 + j < V) A[j & 3] = fmaf(e, d, A[j & 3]);
  }
  st.S += (S[0] + S[1]) + (S[2] + S[3]);
  st.A += (A[0] + A[1]) + (A[2] + A[3]);
}

// The Gumbel screen and walk of a prepared group against the best score known for the row
// (the running max m only scales the test: any m gives the same decisions up to the slack).
template <bool kTail>
__device__ __forceinline__ void screen16(const float (&z)[16], float cmz, int v0, int V, const RowMeta& rm,
                                         Partial& st, BestScore& bs, const uint32_t (&pw)[2]) {
  const uint32_t x0 = 8u * ((uint32_t)v0 >> 4);
  const float m = st.m, nm = -st.m;
  // Can any entry of the group beat g?  The entry holding E_(0) = X_0 / 16 (slot r_0, known from
  // the first slot word alone) only if X_0 / 16 < 2^(u_slot - g); every other entry only if
  // E_(1) = X_0 / 16 + X_1 / 15 < 2^(u_max - g).  With X >= q = 1 - U and, from the funnel-shift
  // word f = 1 + Ut, q >= 2 - f - 2^-23, both tests take the first Philox block alone.
  const float emax = ex2_approx(fmaf(cmz, rm.scale, nm));  // 2^(u_max - m)
  const float g0 = fmaxf(fmaxf(st.g, bs.known), key_ord(*(volatile int*)bs.cta));
  bool live = true;
  if (g0 != -INFINITY) {
    const float K = screen_factor(m, g0);
    const float q0 = (2.f - 0x1p-23f) - screen_word(pw[0]), q1 = (2.f - 0x1p-23f) - screen_word(pw[1]);
    const float e0 = ex2_approx(fmaf(select16(z, pw[1] & 15u), rm.scale, nm));  // 2^(u_slot - m)
    live = q0 * 0.0625f < e0 * K || fmaf(q1, 1.f / 15.f, q0 * 0.0625f) < emax * K;
  }
  const unsigned act = __activemask();
  if (!__any_sync(act, live)) return;
  uint32_t w4[4];
  rm.gs.draw(x0, w4);  // a walk takes the whole first block: its fourth word is the second slot word
  bool improved = false;
  float E = 0.f;
  uint32_t rem = 0xFFFFu;  // slots not yet given a variate
  uint32_t k = 0u;
  while (__any_sync(act, live)) {
    if (live) {
      const uint32_t xw = (k & 1u) ? w4[2] : w4[0], rw = (k & 1u) ? w4[3] : w4[1];
      E = fmaf(exp_variate(xw), __frcp_rn((float)(16u - k)), E);  // E_(k)
      const float g = fmaxf(g0, st.g);
      if (g != -INFINITY && !(E < emax * screen_factor(m, g))) {
        live = false;  // no entry left in the group can score above g
      } else {
        const uint32_t slot = nth_set_bit16(rem, __umulhi(rw, 16u - k));
        rem &= ~(1u << slot);
        const int idx = v0 + (int)slot;
        if (!kTail || idx < V) {
          const float sc = fmaf(select16(z, slot), rm.scale, -lg2_approx(E));
          if (sc > st.g || (sc == st.g && idx < st.gidx)) {
            st.g = sc;
            st.gidx = idx;
            improved = true;
          }
        }
        if (++k == 16u) {
          live = false;
        } else if (!(k & 1u)) {
          rm.gs.draw(x0 + (k >> 1), w4);
        }
      }
    }
  }
  // the column group that raises the CTA's best publishes it (the word's other writers already hold
  // no more than the CTA's best, which its raiser published)
  if (improved && atomicMax(bs.cta, ord_key(st.g)) < ord_key(st.g)) bs.raised = true;
}

template <bool kTail, bool kCap>
__device__ __forceinline__ void fold16(float (&z)[16], int v0, int V, const RowMeta& rm, Partial& st, BestScore& bs,
                                       const uint32_t (&pw)[2], float cap, float inv_cap) {
  float cmz;
  if (!group_prep<kTail, kCap>(z, v0, V, cap, inv_cap, cmz)) return;
  stats16<kTail>(z, cmz, v0, V, rm, st);
  screen16<kTail>(z, cmz, v0, V, rm, st, bs, pw);
}

// A first score for a row whose unit has none yet: the entry holding its
// group's smallest variate, E_(0) = X_0 / 16 at slot r_0 (the first Philox block
// of the group alone), scored exactly as the walk in fold16 scores it.  Run
// over a tile's groups before they are folded, it gives the folds the best of
// those entries to screen against instead of starting from nothing.
template <bool kCap>
__device__ __forceinline__ void seed16(float (&z)[16], int v0, int V, const RowMeta& rm, Partial& st,
                                       const uint32_t (&pw)[2], float cap, float inv_cap) {
  if (v0 >= V) return;
  const uint32_t slot = pw[1] & 15u;
  const int idx = v0 + (int)slot;
  if (idx >= V) return;
  float zs = select16(z, slot);
  if (kCap) zs = cap * tanhf(zs * inv_cap);
  const float sc = fmaf(zs, rm.scale, -lg2_approx(exp_variate(pw[0]) * 0.0625f));
  if (sc > st.g || (sc == st.g && idx < st.gidx)) {
    st.g = sc;
    st.gidx = idx;
  }
}

// The fold of this warp's 16 columns of one accumulator tile.
template <bool kCap>
__device__ __forceinline__ void fold_cols(float (&acc)[16], int v0, int V, const RowMeta& rm, Partial& st,
                                          BestScore& bs, const uint32_t (&pw)[2], float cap, float inv_cap) {
  if (v0 + 16 <= V)
    fold16<false, kCap>(acc, v0, V, rm, st, bs, pw, cap, inv_cap);
  else
    fold16<true, kCap>(acc, v0, V, rm, st, bs, pw, cap, inv_cap);
}

// A unit's first tile in two passes: the statistics of every group first (while the seeds just
// published by the row's other units reach L2), then the screens and walks against the best of
// them.  Neither pass changes what the other computes, so the results equal fold_cols's.
template <bool kCap>
__device__ __forceinline__ void stats_cols(float (&acc)[16], int v0, int V, const RowMeta& rm, Partial& st, float cap,
                                           float inv_cap) {
  float cmz;
  if (v0 + 16 <= V) {
    if (group_prep<false, kCap>(acc, v0, V, cap, inv_cap, cmz)) stats16<false>(acc, cmz, v0, V, rm, st);
  } else {
    if (group_prep<true, kCap>(acc, v0, V, cap, inv_cap, cmz)) stats16<true>(acc, cmz, v0, V, rm, st);
  }
}
template <bool kCap>
__device__ __forceinline__ void screen_cols(float (&acc)[16], int v0, int V, const RowMeta& rm, Partial& st,
                                            BestScore& bs, const uint32_t (&pw)[2], float cap, float inv_cap) {
  float cmz;
  if (v0 + 16 <= V) {
    if (group_prep<false, kCap>(acc, v0, V, cap, inv_cap, cmz)) screen16<false>(acc, cmz, v0, V, rm, st, bs, pw);
  } else {
    if (group_prep<true, kCap>(acc, v0, V, cap, inv_cap, cmz)) screen16<true>(acc, cmz, v0, V, rm, st, bs, pw);
  }
}

// What the screens take from the first Philox block of each of a warp's four 16-column groups
// of a tile, drawn before the tile's accumulator is ready: four independent chains interleave
// and overlap the tile's MMAs, and no fold draws for its screen.  pw[0] is word 0 (the smallest
// variate's); pw[1] is word 2 (the second's: only its bits 9-31 are read) with the first slot,
// the top four bits of word 1, in its low four bits.
constexpr int kGroupsPerWarp = kColsPerWarp / 16;
__device__ __forceinline__ void first_blocks(const RowMeta& rm, int v0, uint32_t (&pw)[kGroupsPerWarp][2]) {
#pragma unroll
  for (int c = 0; c < kGroupsPerWarp; ++c) {
    uint32_t w[4];
    rm.gs.draw(8u * ((uint32_t)(v0 + 16 * c) >> 4), w);
    pw[c][0] = w[0];
    pw[c][1] = (w[2] & ~15u) | (w[1] >> 28);
  }
}
// Brings the next group's words to the front (registers cannot be indexed by a loop counter).
__device__ __forceinline__ void rotate_blocks(uint32_t (&pw)[kGroupsPerWarp][2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t t = pw[0][i];
#pragma unroll
    for (int c = 0; c + 1 < kGroupsPerWarp; ++c) pw[c][i] = pw[c + 1][i];
    pw[kGroupsPerWarp - 1][i] = t;
  }
}

// Before the first h copy: wait until RMSNorm has counted every active row as
// written, then order those generic-proxy stores before this thread's TMA
// (async-proxy) reads.  On expiry the CTA latches DG_ERR_TIMEOUT and aborts.
__device__ __forceinline__ bool rows_written(const Dev& dv, int n_rows, volatile int* abort_flag) {
  if (!wait_count(dv.rows_ready, (uint32_t)n_rows)) {
    *abort_flag = 1;
    timeout_latch(dv.plan, (int)blockIdx.x, kWaitRowsReady, *(volatile uint32_t*)dv.rows_ready);
    return false;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// Work units (row tile, vocabulary chunk) in the order the persistent grid takes
// them.  Row tiles are taken in groups whose rows of h fit in about 48 MB of L2,
// and each group runs through all of this rank's chunks before the next
// starts: every unit re-reads its rows of h once per vocabulary tile, so the
// rows the grid works on at any time have to stay in L2 beside the W tiles
// streaming through, and W is then read from DRAM once per group.  The order
// decides nothing about the results: a unit's partial record depends only on
// its rows and chunk.
struct UnitMap {
  int n_mt, n_local, group;  // row tiles, chunks of this rank, row tiles per group
  __device__ __forceinline__ UnitMap(const Dev& dv, int n_mt_, int rows_per_tile) {
    n_mt = n_mt_;
    n_local = dv.chunk_end - dv.chunk_begin;
    const long long bytes_per_tile = (long long)rows_per_tile * dv.d * 2;
    const long long g = (48ll << 20) / (bytes_per_tile > 0 ? bytes_per_tile : 1);
    group = (int)(g < 1 ? 1 : (g > n_mt ? n_mt : g));
  }
  __device__ __forceinline__ int units() const { return n_mt * n_local; }
  __device__ __forceinline__ void at(const Dev& dv, int u, int& chunk, int& mt) const {
    const int g = u / (group * n_local);
    const int g0 = g * group;
    const int rows_g = min(group, n_mt - g0);  // the last group may hold fewer row tiles
    const int r = u - g0 * n_local;
    chunk = dv.chunk_begin + r / rows_g;
    mt = g0 + r % rows_g;
  }
};

template <bool kCap>
__global__ void __launch_bounds__(kThreadsLM, 1)
    k_lmhead(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Dev dv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int tile_ok[2];  // the epilogue's poller found the tile's accumulator ready (per TMEM buffer)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kStageB);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // column-group merge area: the four warps of a row quadrant leave their records here
  Partial* mrg = reinterpret_cast<Partial*>(reinterpret_cast<uint8_t*>(sB + kStages * kStageB) + 256);
  int* gbest = reinterpret_cast<int*>(mrg + kColGroups * kBM);  // best score per row, shared by the column groups

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (dv.d + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    for (int i = 0; i < kBM; ++i) gbest[i] = ord_key(-INFINITY);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above overlaps the previous kernel.  There is no wait for the whole
  // RMSNorm grid: the producer waits for the count of written rows instead, and
  // data of earlier kernels is read at L2.
  // the plan is read before the next kernel may launch, so its planner cannot have
  // rewritten it for the next tick yet
  const int n_rows = __ldcg(&dv.plan->n_active) * dv.L;
  const uint32_t epoch = __ldcg(&dv.plan->epoch);
  pdl_allow_next();
  const int n_mt = (n_rows + kBM - 1) / kBM;
  const UnitMap um(dv, n_mt, kBM);
  const int n_units = um.units();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued_parity[kStages];
      for (int s = 0; s < kStages; ++s) issued_parity[s] = -1;
      bool ok = rows_written(dv, n_rows, abort_flag);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int chunk, mt;
        um.at(dv, u, chunk, mt);
        const int vt0 = chunk * dv.tiles_per_chunk;
        const int vt1 = min(vt0 + dv.tiles_per_chunk, dv.n_vtiles);
        (void)DG_IN_BOUNDS(dv.plan, mt * kBM < dv.rows_cap && vt0 >= dv.vt_base && vt1 <= dv.n_vtiles, 8, mt);
        for (int vt = vt0; vt < vt1 && ok; ++vt) {
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, dv.plan)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&full[stage], (uint32_t)(kStageA + kStageB));
            tma_load_2d(sA + stage * kStageA, &tmA, kb * kBK, mt * kBM, &full[stage]);
            tma_load_2d(sB + stage * kStageB, &tmB, kb * kBK, (vt - dv.vt_base) * kBN, &full[stage]);
            issued_parity[stage] = (int)phase;
            if (++stage == (uint32_t)kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before shared memory is released
        for (int s = 0; s < kStages; ++s) {
          if (issued_parity[s] < 0) continue;
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(&full[s], (uint32_t)issued_parity[s]) && global_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // descriptors of stage 0; a stage or K offset adds to the low word only (as on pairs)
      const DescPair dA(sw128_desc(smem_u32(sA))), dB(sw128_desc(smem_u32(sB)));
      uint32_t stage = 0, phase = 0, tcount = 0;
      bool ok = true, any = false;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int chunk, mt;
        um.at(dv, u, chunk, mt);
        const int vt0 = chunk * dv.tiles_per_chunk;
        const int vt1 = min(vt0 + dv.tiles_per_chunk, dv.n_vtiles);
        for (int vt = vt0; vt < vt1 && ok; ++vt, ++tcount) {
          const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
          if (!mbar_wait(&tempty[ab], aph ^ 1u, abort_flag, dv.plan)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * (uint32_t)kBN;
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, dv.plan)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t alo = dA.lo + (uint32_t)((stage * kStageA) >> 4);
            const uint32_t blo = dB.lo + (uint32_t)((stage * kStageB) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              // advance K by 16 bf16 = 32 bytes inside the swizzled 128-byte row
              mma_bf16(d_tmem, dA.at(alo + (uint32_t)(kk * 2)), dB.at(blo + (uint32_t)(kk * 2)), (kb | kk) != 0 ? 1u : 0u);
            }
            mma_commit(&empty[stage]);
            any = true;
            if (++stage == (uint32_t)kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&tfull[ab]);
        }
      }
      if (!ok && any) {
        // wait (bounded) for the MMAs already issued before TMEM is freed
        mma_commit(drain);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(drain, 0u) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int cg = (warp - 2) >> 2;         // which 64 of the 256 columns
    uint32_t tcount = 0;
    bool aborted = false;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      int chunk, mt;
        um.at(dv, u, chunk, mt);
      const int vt0 = chunk * dv.tiles_per_chunk;
      const int vt1 = min(vt0 + dv.tiles_per_chunk, dv.n_vtiles);
      const int rl = q * 32 + lane;         // row within the tile
      const int row = mt * kBM + rl;
      const RowMeta rm = row_meta(dv, row, n_rows);
      if (dv.row_scale && rm.valid && cg == 0) dv.row_scale[row] = rm.scale;  // for the self-conditioning pass
      BestScore bs{gbest + rl, dv.row_best + row, epoch, -INFINITY, false};
      Partial st = empty_partial();
      for (int vt = vt0; vt < vt1; ++vt, ++tcount) {
        if (aborted) continue;
        const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
        // the best score other units of this row have found so far (read while the tile completes)
        if (rm.valid) bs.known = row_best_score(bs.glob, epoch);
        uint32_t pw[kGroupsPerWarp][2];
        first_blocks(rm, vt * kBN + cg * kColsPerWarp, pw);
        // One warp polls for the tile; the other fifteen wait on a hardware barrier, which issues
        // nothing (sixteen pollers took issue slots from the MMA and producer warps).  The result
        // goes through shared memory, double-buffered: the poller cannot write this slot again
        // before every warp has passed the next tile's barrier, so after reading it.
        if (warp == 2) {
          if (lane == 0) tile_ok[ab] = mbar_wait_poll(&tfull[ab], aph, 256u, abort_flag, dv.plan) ? 1 : 0;
          __syncwarp();
        }
        asm volatile("bar.sync 4, %0;" ::"r"(32 * kEpiWarps) : "memory");
        const int got = *(volatile int*)&tile_ok[ab];
        if (!got) {
          aborted = true;
          continue;
        }
        tc_fence_after();
        const uint32_t tbase =
            tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBN + (uint32_t)(cg * kColsPerWarp);
        // No score known for the row yet (its unit's first tile, no other unit ahead of it): seed
        // one and publish it, then form the tile's statistics, and only then screen (below) --
        // against the seeds the row's other units have published meanwhile.
        const bool seeding = __any_sync(0xFFFFFFFFu, rm.valid && st.g == -INFINITY && bs.known == -INFINITY);
        if (seeding) {
          const bool seed = rm.valid && st.g == -INFINITY && bs.known == -INFINITY;
#pragma unroll 1
          for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
            float acc[16];
            __syncwarp();
            tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
            if (seed)
              seed16<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, pw[0], dv.softcap,
                           dv.inv_softcap);
            rotate_blocks(pw);  // four turns: back in order for the screens
          }
          if (seed && st.g != -INFINITY) {
            // published at once, by the column group whose seed raised the CTA's best only (a few
            // atomics per row, not one per column group): the other units of the row, folding
            // their own tiles now, screen against it
            if (atomicMax(bs.cta, ord_key(st.g)) < ord_key(st.g)) row_best_raise(bs.glob, epoch, st.g);
          }
#pragma unroll 1
          for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
            float acc[16];
            __syncwarp();
            tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
            if (rm.valid)
              stats_cols<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, dv.softcap, dv.inv_softcap);
          }
        }
        // the best score any unit of the row has published, refreshed for every group: the value
        // a group screens against is loaded one group ahead, so its latency overlaps a fold (and a
        // load never follows this lane's own atomic on the same word, which it would wait for)
        // (the raw word is carried and decoded where it is used, so nothing waits on the load early)
        unsigned long long known_next = (unsigned long long)(epoch ^ 1u) << 32;  // another epoch: no score
        if (seeding && rm.valid) known_next = __ldcg(bs.glob);  // the seeds published meanwhile
#pragma unroll 1
        for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
          float acc[16];
          const unsigned long long known = known_next;
          if (rm.valid && cc + 1 < kColsPerWarp / 16) known_next = __ldcg(bs.glob);
          __syncwarp();  // tcgen05.ld is .sync.aligned: the fold below may leave lanes diverged
          tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
          if (cc == kColsPerWarp / 16 - 1) {
            // the accumulator is in registers: hand the buffer back to the MMA warp early
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
          }
          bs.known = fmaxf(bs.known, row_best_decode(known, epoch));
          if (rm.valid) {
            if (seeding)
              screen_cols<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, bs, pw[0], dv.softcap,
                                dv.inv_softcap);
            else
              fold_cols<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, bs, pw[0], dv.softcap,
                              dv.inv_softcap);
          }
          if (bs.raised) {  // published as soon as it rises, for the same reason
            row_best_raise(bs.glob, epoch, st.g);
            bs.raised = false;
          }
          rotate_blocks(pw);
        }
      }
      // merge the four column groups of each row; one record per row and chunk.  Every
      // epilogue warp reaches both barriers once per unit, aborted or not (named barrier 1,
      // the 512 epilogue threads).
      mrg[cg * kBM + rl] = st;
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (cg == 0 && rm.valid) {
        Partial m = st;
#pragma unroll
        for (int k = 1; k < kColGroups; ++k) m = merge_partial(m, mrg[k * kBM + rl]);
        if (DG_IN_BOUNDS(dv.plan, row < dv.rows_cap && chunk >= 0 && chunk < dv.n_sub, 6, row))
          dv.part[(size_t)row * dv.n_sub + chunk] = m;
      }
      if (cg == 0) gbest[rl] = ord_key(-INFINITY);  // the next unit may hold other rows
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (warp == 2 && lane == 0 && mt * kBM < n_rows && !dv.hold_slabs)
        red_release_add(dv.slab_done + mt, 1u);  // after this unit's partial records of the slab
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)kTmemCols)
                 : "memory");
  }
}

// The same LM head on SM pairs: a cluster of two CTAs computes M = 256 rows x
// N = 256 vocabulary entries per tcgen05.mma.cta_group::2 instruction, issued
// by one thread of the leader CTA (rank 0).  Each CTA stages its own 128 rows
// of A and its own 128-row half of the W tile (32 KB per stage, 6 stages), so
// a pair streams W once for 256 rows; the accumulator of each CTA's 128 rows
// lands in its own TMEM, and each CTA runs the same epilogue on its rows.
//   full[s]   (leader)  both CTAs' TMA bytes; the leader arms it with the total
//   empty[s]  (both)    released by the leader's commit, multicast to the pair
//   tfull[b]  (both)    accumulator ready, multicast from the leader's commit
//   tempty[b] (leader)  both CTAs' 16 epilogue warps release the accumulator

template <bool kCap>
__global__ void __launch_bounds__(kThreadsLM, 1)
    k_lmhead_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Dev dv,
                  const float* __restrict__ resid) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red_norm[2][8][2];  // RMSNorm reductions of the two row groups
  __shared__ int tile_ok[2];           // the epilogue's poller found the tile's accumulator ready (per TMEM buffer)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStagesPair * kStagePairA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStagesPair * kStagePairB);
  uint64_t* empty = full + kStagesPair;
  uint64_t* tfull = empty + kStagesPair;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  Partial* mrg = reinterpret_cast<Partial*>(reinterpret_cast<uint8_t*>(sB + kStagesPair * kStagePairB) + 256);
  int* gbest = reinterpret_cast<int*>(mrg + kColGroups * kBM);  // best score per row, shared by the column groups

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int KB = (dv.d + kBK - 1) / kBK;

  // The epilogue warps start the loads of the RMSNorm phase below before the
  // set-up, so their latency overlaps it: the norm weights (constant), then,
  // once the previous kernel of the stream (the last tick's planner) has
  // completed, the plan, the canvas of the group's first row and an L2
  // prefetch of that row as it lies when canvas k is the k-th active one.
  const int et = (int)threadIdx.x - 64, grp = et >> 8, r_first = (int)blockIdx.x + grp * (int)gridDim.x;
  int n_active = 0, c_first = 0;
  uint32_t epoch = 0;
  if (warp >= 2) {
    if (dv.norm_w) prefetch_row<256>(dv.norm_w, dv.d >> 2, et & 255);
    pdl_wait();
    n_active = __ldcg(&dv.plan->n_active);
    epoch = __ldcg(&dv.plan->epoch);
    if (r_first < dv.max_active * dv.L) {
      const int a = r_first / dv.L;
      c_first = __ldcg(dv.active + a);
      prefetch_row<256>(resid + (size_t)r_first * dv.d, dv.d >> 2, et & 255);
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesPair; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    for (int i = 0; i < kBM; ++i) gbest[i] = ord_key(-INFINITY);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before anything arrives on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  // W does not depend on the previous kernel, so its first stages are loaded
  // before the wait below.  This needs the pair's first unit to be known
  // already, which holds when one 256-row pair tile covers every position the
  // sampler can hold: the unit is then vocabulary chunk `cid` whenever any
  // canvas is active.  The leader raises the stage's expected bytes by the W
  // halves now and arrives, with the h halves, after the wait.
  int pre = 0;
  if ((dv.max_active * dv.L + 2 * kBM - 1) / (2 * kBM) == 1 && cid < dv.chunk_end - dv.chunk_begin) {
    const int vt0 = (dv.chunk_begin + cid) * dv.tiles_per_chunk;
    pre = min(kStagesPair, KB * (min(vt0 + dv.tiles_per_chunk, dv.n_vtiles) - vt0));
    if (warp == 0 && lane == 0) {
      for (int it = 0; it < pre; ++it) {
        const int vt = vt0 + it / KB, kb = it % KB;
        if (leader) mbar_expect_tx_only(&full[it], (uint32_t)(2 * kStagePairB));
        tma_load_2d_pair(sB + it * kStagePairB, &tmB, kb * kBK, (vt - dv.vt_base) * kBN + (int)rank * (kBN / 2),
                         peer_addr(smem_u32(&full[it]), 0));
      }
    }
  }
  // The previous kernel of the stream (the last tick's planner) has completed:
  // the plan, the active list and the slots are current.  The plan is read
  // before the next kernel may launch, so its planner cannot rewrite it first.
  if (warp < 2) {
    pdl_wait();
    n_active = __ldcg(&dv.plan->n_active);
  }
  const int n_rows = n_active * dv.L;
  pdl_allow_next_after(n_rows);
  const int n_mt = (n_rows + 2 * kBM - 1) / (2 * kBM);  // 256-row pair tiles
  const UnitMap um(dv, n_mt, 2 * kBM);
  const int n_units = um.units();

  if (warp >= 2) {
    // RMSNorm: the epilogue warps form rows blockIdx.x + j * gridDim.x of h, two
    // at a time (eight warps a row), and count them; every CTA's producer then
    // waits for all rows (rows_written).  The grid is at most one CTA per SM, so
    // all of its CTAs can be resident at once; one kept waiting for an SM longer
    // than the bounded wait fails the tick with a timeout instead of hanging it.
    for (int r = r_first; r < n_rows; r += 2 * (int)gridDim.x) {
      const int a = r / dv.L, p = r - a * dv.L;
      int c = r == r_first ? c_first : __ldcg(dv.active + a);
      if (!DG_IN_BOUNDS(dv.plan, c >= 0 && c < dv.B && r < dv.rows_cap, 9, c)) c = 0;
      norm_row<256, 4>(resid + ((size_t)c * dv.L + p) * dv.d, dv.norm_w, dv.h + (size_t)r * dv.d,
                       dv.d, dv.eps, et & 255, red_norm[grp],
                       [grp] {
                         if (grp == 0)
                           asm volatile("bar.sync 2, 256;" ::: "memory");
                         else
                           asm volatile("bar.sync 3, 256;" ::: "memory");
                       });
    }
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
    if (warp == 2 && lane == 0 && n_rows > (int)blockIdx.x) {
      // this CTA's rows (written by all its epilogue warps, ordered before this thread by the
      // barrier above) are released with the count, in one reduction
      red_release_add(dv.rows_ready, (unsigned)((n_rows - 1 - (int)blockIdx.x) / (int)gridDim.x + 1));
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = rows_written(dv, n_rows, abort_flag);
      int issued = 0, round = 0;
      for (int u = cid; u < n_units && ok; u += n_clusters, ++round) {
        // Pacing, when the row tiles span more than one L2-sized group: a pair starts its unit of
        // round r only once every unit of round r - 1 is finished.  Left alone, the pairs drift apart over the rounds and the W and h tiles they
        // share leave L2 between their reads: at 64 x 256 rows, 32-55 GB of DRAM reads a launch
        // instead of 4.9 GB.  With one group (16 x 256 rows and fewer) the drift costs little
        // and the pacing's pause at each round boundary costs more.  The slowest pair never waits.
        if (round > 0 && um.group < n_mt &&
            !wait_count(dv.units_done, (uint32_t)min(round * n_clusters, n_units))) {
          *abort_flag = 1;
          timeout_latch(dv.plan, (int)blockIdx.x, kWaitPacing, *(volatile uint32_t*)dv.units_done);
          ok = false;
          break;
        }
        int chunk, mt;
        um.at(dv, u, chunk, mt);
        const int vt0 = chunk * dv.tiles_per_chunk;
        const int vt1 = min(vt0 + dv.tiles_per_chunk, dv.n_vtiles);
        (void)DG_IN_BOUNDS(dv.plan, (mt * 2 + 1) * kBM < dv.rows_cap && vt0 >= dv.vt_base && vt1 <= dv.n_vtiles, 8, mt);
        for (int vt = vt0; vt < vt1 && ok; ++vt) {
          for (int kb = 0; kb < KB; ++kb) {
            const uint32_t full_leader = peer_addr(smem_u32(&full[stage]), 0);
            if (issued < pre) {
              // first lap, W half already in flight: the h half and the leader's arrival
              if (leader) mbar_expect_tx(&full[stage], (uint32_t)(2 * kStagePairA));
              tma_load_2d_pair(sA + stage * kStagePairA, &tmA, kb * kBK, mt * 2 * kBM + (int)rank * kBM,
                                    full_leader);
            } else {
              // Both CTAs' loads complete the leader's full barrier, so the leader's MMAs never
              // run a lap ahead of either producer: the commits arriving on this CTA's empty
              // barrier stay within one phase of this wait, and its parity cannot alias.
              if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, dv.plan)) {
                ok = false;
                break;
              }
              if (leader) mbar_expect_tx(&full[stage], (uint32_t)(2 * (kStagePairA + kStagePairB)));
              tma_load_2d_pair(sA + stage * kStagePairA, &tmA, kb * kBK, mt * 2 * kBM + (int)rank * kBM,
                                    full_leader);
              tma_load_2d_pair(sB + stage * kStagePairB, &tmB, kb * kBK, (vt - dv.vt_base) * kBN + (int)rank * (kBN / 2),
                               full_leader);
            }
            ++issued;
            if (++stage == (uint32_t)kStagesPair) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (issued == 0 && pre > 0 && leader) {
        // no active canvas: close the preloaded stages and let their copies land
        for (int it = 0; it < pre; ++it) {
          mbar_arrive(&full[it]);
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(&full[it], 0u) && global_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
      // drain: one more lap of the ring's waits covers the releases of the last
      // kStagesPair loads (laps before the first load pass at once), so no copy or
      // release is still in flight toward this CTA when the pair exits
      (void)issued;
      for (int i = 0; i < kStagesPair; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, dv.plan)) break;
        if (++stage == (uint32_t)kStagesPair) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && leader) {
      // descriptors of stage 0; a stage or K offset adds its 16-byte count to the
      // start-address field, which stays below 2^14 for any shared-memory address,
      // so only the low word changes (32-bit adds: fewer instructions from a warp
      // whose issue slots the epilogue warps of its sub-partition contend for)
      const DescPair dA(sw128_desc(smem_u32(sA))), dB(sw128_desc(smem_u32(sB)));
      uint32_t stage = 0, phase = 0, tcount = 0;
      bool ok = true, any = false;
      for (int u = cid; u < n_units && ok; u += n_clusters) {
        int chunk, mt;
        um.at(dv, u, chunk, mt);
        const int vt0 = chunk * dv.tiles_per_chunk;
        const int vt1 = min(vt0 + dv.tiles_per_chunk, dv.n_vtiles);
        for (int vt = vt0; vt < vt1 && ok; ++vt, ++tcount) {
          const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
          if (!mbar_wait(&tempty[ab], aph ^ 1u, abort_flag, dv.plan)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * (uint32_t)kBN;
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, dv.plan)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t alo = dA.lo + (uint32_t)((stage * kStagePairA) >> 4);
            const uint32_t blo = dB.lo + (uint32_t)((stage * kStagePairB) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_pair(d_tmem, dA.at(alo + (uint32_t)(kk * 2)), dB.at(blo + (uint32_t)(kk * 2)),
                            (kb | kk) != 0 ? 1u : 0u);
            mma_commit_pair(&empty[stage], (uint16_t)0x3);
            any = true;
            if (++stage == (uint32_t)kStagesPair) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(&tfull[ab], (uint16_t)0x3);
        }
      }
      if (!ok && any) {
        mma_commit_pair(drain, (uint16_t)0x1);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(drain, 0u) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int cg = (warp - 2) >> 2;
    const uint32_t tempty_leader[2] = {peer_addr(smem_u32(&tempty[0]), 0), peer_addr(smem_u32(&tempty[1]), 0)};
    uint32_t tcount = 0;
    bool aborted = false;
    for (int u = cid; u < n_units; u += n_clusters) {
      int chunk, mt;
        um.at(dv, u, chunk, mt);
      const int vt0 = chunk * dv.tiles_per_chunk;
      const int vt1 = min(vt0 + dv.tiles_per_chunk, dv.n_vtiles);
      const int rl = q * 32 + lane;
      const int row = mt * 2 * kBM + (int)rank * kBM + rl;
      const RowMeta rm = row_meta(dv, row, n_rows);
      if (dv.row_scale && rm.valid && cg == 0) dv.row_scale[row] = rm.scale;  // for the self-conditioning pass
      BestScore bs{gbest + rl, dv.row_best + row, epoch, -INFINITY, false};
      Partial st = empty_partial();
      for (int vt = vt0; vt < vt1; ++vt, ++tcount) {
        if (aborted) continue;
        const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
        // the best score other units of this row have found so far (read while the tile completes)
        if (rm.valid) bs.known = row_best_score(bs.glob, epoch);
        uint32_t pw[kGroupsPerWarp][2];
        first_blocks(rm, vt * kBN + cg * kColsPerWarp, pw);
        // One warp polls for the tile; the other fifteen wait on a hardware barrier, which issues
        // nothing (sixteen pollers took issue slots from the MMA and producer warps).  The result
        // goes through shared memory, double-buffered: the poller cannot write this slot again
        // before every warp has passed the next tile's barrier, so after reading it.
        if (warp == 2) {
          if (lane == 0) tile_ok[ab] = mbar_wait_poll(&tfull[ab], aph, 256u, abort_flag, dv.plan) ? 1 : 0;
          __syncwarp();
        }
        asm volatile("bar.sync 4, %0;" ::"r"(32 * kEpiWarps) : "memory");
        const int got = *(volatile int*)&tile_ok[ab];
        if (!got) {
          aborted = true;
          continue;
        }
        tc_fence_after();
        const uint32_t tbase =
            tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBN + (uint32_t)(cg * kColsPerWarp);
        // No score known for the row yet (its unit's first tile, no other unit ahead of it): seed
        // one and publish it, then form the tile's statistics, and only then screen (below) --
        // against the seeds the row's other units have published meanwhile.
        const bool seeding = __any_sync(0xFFFFFFFFu, rm.valid && st.g == -INFINITY && bs.known == -INFINITY);
        if (seeding) {
          const bool seed = rm.valid && st.g == -INFINITY && bs.known == -INFINITY;
#pragma unroll 1
          for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
            float acc[16];
            __syncwarp();
            tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
            if (seed)
              seed16<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, pw[0], dv.softcap,
                           dv.inv_softcap);
            rotate_blocks(pw);  // four turns: back in order for the screens
          }
          if (seed && st.g != -INFINITY) {
            // published at once, by the column group whose seed raised the CTA's best only (a few
            // atomics per row, not one per column group): the other units of the row, folding
            // their own tiles now, screen against it
            if (atomicMax(bs.cta, ord_key(st.g)) < ord_key(st.g)) row_best_raise(bs.glob, epoch, st.g);
          }
#pragma unroll 1
          for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
            float acc[16];
            __syncwarp();
            tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
            if (rm.valid)
              stats_cols<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, dv.softcap, dv.inv_softcap);
          }
        }
        // the best score any unit of the row has published, refreshed for every group: the value
        // a group screens against is loaded one group ahead, so its latency overlaps a fold (and a
        // load never follows this lane's own atomic on the same word, which it would wait for)
        // (the raw word is carried and decoded where it is used, so nothing waits on the load early)
        unsigned long long known_next = (unsigned long long)(epoch ^ 1u) << 32;  // another epoch: no score
        if (seeding && rm.valid) known_next = __ldcg(bs.glob);  // the seeds published meanwhile
#pragma unroll 1
        for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
          float acc[16];
          const unsigned long long known = known_next;
          if (rm.valid && cc + 1 < kColsPerWarp / 16) known_next = __ldcg(bs.glob);
          __syncwarp();  // tcgen05.ld is .sync.aligned: the fold below may leave lanes diverged
          tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
          if (cc == kColsPerWarp / 16 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader[ab]);
          }
          bs.known = fmaxf(bs.known, row_best_decode(known, epoch));
          if (rm.valid) {
            if (seeding)
              screen_cols<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, bs, pw[0], dv.softcap,
                                dv.inv_softcap);
            else
              fold_cols<kCap>(acc, vt * kBN + cg * kColsPerWarp + cc * 16, dv.V, rm, st, bs, pw[0], dv.softcap,
                              dv.inv_softcap);
          }
          if (bs.raised) {  // published as soon as it rises, for the same reason
            row_best_raise(bs.glob, epoch, st.g);
            bs.raised = false;
          }
          rotate_blocks(pw);
        }
      }
      mrg[cg * kBM + rl] = st;
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (cg == 0 && rm.valid) {
        Partial m = st;
#pragma unroll
        for (int k = 1; k < kColGroups; ++k) m = merge_partial(m, mrg[k * kBM + rl]);
        if (DG_IN_BOUNDS(dv.plan, row < dv.rows_cap && chunk >= 0 && chunk < dv.n_sub, 6, row))
          dv.part[(size_t)row * dv.n_sub + chunk] = m;
      }
      if (cg == 0) gbest[rl] = ord_key(-INFINITY);  // the next unit may hold other rows
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (warp == 2 && lane == 0) {
        // The pacing count, one per unit from the CTA whose rows always lie below n_rows, comes
        // before that CTA's slab count: once the finishing kernel has seen every slab done it
        // may reset the tick's counters, and a later increment would carry into the next tick.
        if (rank == 0) atomicAdd(dv.units_done, 1u);
        if ((mt * 2 + (int)rank) * kBM < n_rows && !dv.hold_slabs)
          red_release_add(dv.slab_done + mt * 2 + (int)rank, 1u);  // after the records and the pacing count
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs are done with the pair's TMEM and barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)kTmemCols)
                 : "memory");
  }
}

constexpr size_t kSmemBytesPair = 1024 + (size_t)kStagesPair * (kStagePairA + kStagePairB) + 256 +
                                  sizeof(Partial) * kColGroups * kBM + sizeof(int) * kBM;
static_assert(kSmemBytesPair <= 232448, "shared memory per CTA");

constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * (kStageA + kStageB) + 256 + sizeof(Partial) * kColGroups * kBM + sizeof(int) * kBM;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

}  // namespace

cudaError_t lmhead_configure() {
  cudaError_t e = cudaFuncSetAttribute(k_lmhead<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_lmhead<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_lmhead_pair<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesPair);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_lmhead_pair<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesPair);
  return e;
}

cudaError_t launch_lmhead_pair(const Dev& dv, const float* resid, const CUtensorMap* tmA, const CUtensorMap* tmB,
                               int num_sms, cudaStream_t st) {
  // persistent grid of CTA pairs, never more pairs than the largest number of work units
  const int max_mt = (dv.max_active * dv.L + 2 * kBM - 1) / (2 * kBM);
  int pairs = max_mt * (dv.chunk_end - dv.chunk_begin);
  if (pairs > num_sms / 2) pairs = num_sms / 2;
  if (pairs < 1) pairs = 1;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreadsLM);
  cfg.dynamicSmemBytes = kSmemBytesPair;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return dv.softcap > 0.f ? cudaLaunchKernelEx(&cfg, k_lmhead_pair<true>, *tmA, *tmB, dv, resid)
                          : cudaLaunchKernelEx(&cfg, k_lmhead_pair<false>, *tmA, *tmB, dv, resid);
}

cudaError_t launch_lmhead(const Dev& dv, const CUtensorMap* tmA, const CUtensorMap* tmB, int num_sms,
                          cudaStream_t st) {
  // Persistent grid: one CTA per SM (the shared-memory ring keeps it at one),
  // never more CTAs than the largest number of work units.
  const int max_mt = (dv.max_active * dv.L + kBM - 1) / kBM;
  int grid = max_mt * (dv.chunk_end - dv.chunk_begin);
  if (grid > num_sms) grid = num_sms;
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsLM);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return dv.softcap > 0.f ? cudaLaunchKernelEx(&cfg, k_lmhead<true>, *tmA, *tmB, dv)
                          : cudaLaunchKernelEx(&cfg, k_lmhead<false>, *tmA, *tmB, dv);
}

}  // namespace dg
