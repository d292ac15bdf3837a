// Self-conditioning input for the next denoising step: the expected token
// embedding under this step's distribution,
//   e[p, :] = sum_v P[p, v] W[v, :],  P[p, :] = softmax(z[p, :] / T),
// "The Annotated DiffusionGemma", decode mode (the previous step's
// probabilities times the embedding matrix, one convex combination of
// embedding rows per position) and `_forward`'s condition_x, before the
// embedding scale; P is the same distribution whose entropy the commit uses
// (the page's denoise loop builds a categorical distribution from the model
// output divided by the temperature and hands its probabilities to the next
// decode), cast to bf16 before the contraction as the page casts it to the
// activation dtype.
//
// It runs after a tick, from what the tick left: the normalised rows h, each
// row's temperature factor (LM head) and log2 Z (finishing kernel).  Three
// kernels on the sampler's stream:
//   k_selfcond<kProbs>  the tied LM head again (tcgen05, M = 128, N = 256),
//                       whose epilogue writes P = 2^(z log2(e)/T - log2 Z) in
//                       bf16 to a [rows, V_pad] buffer (zeros past V);
//   k_selfcond<kGemm>   E_part[kc] = P[:, chunk kc] W^T[:, chunk kc]^T on the
//                       same tensor-core mainloop, A = P and B = W^T (a
//                       transposed copy of W made at sampler creation), both
//                       K-major along the vocabulary, split into vocabulary
//                       chunks kc so the grid fills the GPU;
//   k_selfcond_reduce   e = sum over kc in order (deterministic), written to
//                       the caller's [B, L, d] array at each row's canvas.
// The top-K variant (further down) keeps each position's K most probable
// tokens only: k_topk_prep bounds each row's K-th largest logit from the
// tick's chunk maxima, k_selfcond<kCands> is the LM head again listing the
// entries that reach the bound (and writing P), and k_selfcond_topk ranks a
// row's list and sums the kept rows of W.
// Producer (warp 0), MMA issuer (warp 1) and 16 epilogue warps as in the LM
// head; every wait is bounded (1 s) and latches DG_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dg_internal.cuh"
#include "dg_tc.cuh"

namespace dg {
namespace {

// kProbs: the LM head again, writing P.  kCands: the same, also listing each row's top-K
// candidates with their logits (the top-K variant, below).  kGemm: P W^T.
enum : int { kProbs = 0, kGemm = 1, kCands = 2 };

// The top-K variant's candidate lists live in the dense variant's per-chunk shares (which it does
// not use), one region of sc_kc * d floats per row: a 16-byte header {count, bound, dense, -} and
// then (token, u) pairs.  `bound` is the row's lower bound of the K-th largest u = z log2(e)/T;
// `dense` marks a row whose bound is not known (K above the number of vocabulary chunks).
constexpr int kTopKCand = 2048;  // candidates a row can list, at most
struct CandHeader {
  uint32_t count;
  float bound;
  uint32_t dense;
  uint32_t pad;
};
static_assert(sizeof(CandHeader) == 16, "candidate header is 16 bytes");
__device__ __forceinline__ CandHeader* cand_header(const Dev& dv, int row) {
  return reinterpret_cast<CandHeader*>(dv.sc_part + (size_t)row * dv.sc_kc * dv.d);
}
__device__ __forceinline__ int2* cand_list(const Dev& dv, int row) { return reinterpret_cast<int2*>(cand_header(dv, row) + 1); }
__device__ __forceinline__ uint32_t cand_capacity(const Dev& dv) {
  const size_t pairs = ((size_t)dv.sc_kc * dv.d * 4 - sizeof(CandHeader)) / 8;
  return (uint32_t)(pairs < (size_t)kTopKCand ? pairs : (size_t)kTopKCand);
}

// The units of one launch: kProbs (row tile, vocabulary chunk) with the chunk's
// vocabulary tiles as N tiles and the hidden dimension as K; kGemm (row tile,
// d tile, vocabulary chunk kc) with one N tile and the chunk's vocabulary
// columns as K.
struct ScUnits {
  int n_mt, n_dt, KB;
  __device__ __forceinline__ int units(const Dev& dv, int mode) const {
    return mode != kGemm ? n_mt * dv.n_chunks : n_mt * n_dt * dv.sc_kc;
  }
  // first/last N tile and first/last K block of unit u, and its row tile
  __device__ __forceinline__ void at(const Dev& dv, int mode, int u, int& mt, int& t0, int& t1, int& kb0,
                                     int& kb1) const {
    if (mode != kGemm) {
      const int chunk = u / n_mt;
      mt = u - chunk * n_mt;
      t0 = chunk * dv.tiles_per_chunk;
      t1 = min(t0 + dv.tiles_per_chunk, dv.n_vtiles);
      kb0 = 0;
      kb1 = KB;
    } else {
      const int kc = u / (n_mt * n_dt), r = u - kc * n_mt * n_dt;
      const int dt = r / n_mt;
      mt = r - dt * n_mt;
      t0 = dt;
      t1 = dt + 1;
      kb0 = kc * dv.sc_kbpc;
      kb1 = min(kb0 + dv.sc_kbpc, dv.sc_vpad / kBK);
    }
  }
};

// An epilogue's 16 accumulator columns [c0, c0 + 16) of `row`: kProbs writes P = 2^(u - log2 Z),
// u = z log2(e)/T, rounded to bf16 (zero past V); kCands also lists the columns whose u reaches
// the row's bound `cand` (with u as the tick forms its maxima: the capped logit times log2(e)/T);
// kGemm writes the vocabulary chunk's share of e for hidden columns [c0, c0 + 16).
template <int kMode, bool kCap>
__device__ __forceinline__ void store_cols(const Dev& dv, const float (&acc)[16], int row, int c0, int kb0,
                                           float scale, float l2z, float cand) {
  if (kMode != kGemm) {
    uint32_t pk[8];
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float z0 = acc[j], z1 = acc[j + 1];
      if (kCap) {
        z0 = dv.softcap * tanhf(z0 * dv.inv_softcap);
        z1 = dv.softcap * tanhf(z1 * dv.inv_softcap);
      }
      if (kMode == kCands) {
        const float u0 = z0 * scale, u1 = z1 * scale;
        const bool t0 = c0 + j < dv.V && u0 >= cand, t1 = c0 + j + 1 < dv.V && u1 >= cand;
        if (t0 || t1) {
          CandHeader* hd = cand_header(dv, row);
          const uint32_t cap = cand_capacity(dv);
          if (t0) {
            const uint32_t at = atomicAdd(&hd->count, 1u);
            if (at < cap) cand_list(dv, row)[at] = make_int2(c0 + j, __float_as_int(u0));
          }
          if (t1) {
            const uint32_t at = atomicAdd(&hd->count, 1u);
            if (at < cap) cand_list(dv, row)[at] = make_int2(c0 + j + 1, __float_as_int(u1));
          }
        }
      }
      const float p0 = c0 + j < dv.V ? ex2_approx(fmaf(z0, scale, -l2z)) : 0.f;
      const float p1 = c0 + j + 1 < dv.V ? ex2_approx(fmaf(z1, scale, -l2z)) : 0.f;
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
      pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    uint4* dst = reinterpret_cast<uint4*>(dv.sc_probs + (size_t)row * dv.sc_vpad + c0);
    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  } else {
    const int kc = kb0 / dv.sc_kbpc;
    float* dst = dv.sc_part + ((size_t)kc * dv.rows_cap + row) * dv.d + c0;
#pragma unroll
    for (int j = 0; j < 16; j += 4)
      if (c0 + j < dv.d) *reinterpret_cast<float4*>(dst + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
  }
}

template <int kMode, bool kCap>
__global__ void __launch_bounds__(kThreadsLM, 1)
    k_selfcond(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Dev dv) {
  extern __shared__ uint8_t smem_raw[];
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
  // rows of the tick that left h, the temperature factors and log2 Z behind
  const int n_rows = (int)__ldcg(dv.sc_rows);
  const ScUnits su{(n_rows + kBM - 1) / kBM, (dv.d + kBN - 1) / kBN, (dv.d + kBK - 1) / kBK};
  const int n_units = su.units(dv, kMode);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued_parity[kStages];
      for (int s = 0; s < kStages; ++s) issued_parity[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int mt, t0, t1, kb0, kb1;
        su.at(dv, kMode, u, mt, t0, t1, kb0, kb1);
        for (int t = t0; t < t1 && ok; ++t) {
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, dv.plan)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&full[stage], (uint32_t)(kStageA + kStageB));
            tma_load_2d(sA + stage * kStageA, &tmA, kb * kBK, mt * kBM, &full[stage]);
            tma_load_2d(sB + stage * kStageB, &tmB, kb * kBK, t * kBN, &full[stage]);
            issued_parity[stage] = (int)phase;
            if (++stage == (uint32_t)kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
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
      const DescPair dA(sw128_desc(smem_u32(sA))), dB(sw128_desc(smem_u32(sB)));
      uint32_t stage = 0, phase = 0, tcount = 0;
      bool ok = true, any = false;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int mt, t0, t1, kb0, kb1;
        su.at(dv, kMode, u, mt, t0, t1, kb0, kb1);
        for (int t = t0; t < t1 && ok; ++t, ++tcount) {
          const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
          if (!mbar_wait(&tempty[ab], aph ^ 1u, abort_flag, dv.plan)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * (uint32_t)kBN;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, dv.plan)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t alo = dA.lo + (uint32_t)((stage * kStageA) >> 4);
            const uint32_t blo = dB.lo + (uint32_t)((stage * kStageB) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16(d_tmem, dA.at(alo + (uint32_t)(kk * 2)), dB.at(blo + (uint32_t)(kk * 2)),
                       (kb != kb0 || kk != 0) ? 1u : 0u);
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
        mma_commit(drain);
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
    uint32_t tcount = 0;
    bool aborted = false;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      int mt, t0, t1, kb0, kb1;
      su.at(dv, kMode, u, mt, t0, t1, kb0, kb1);
      const int row = mt * kBM + q * 32 + lane;
      const bool valid = row < n_rows;
      const float scale = valid && kMode != kGemm ? __ldcg(dv.row_scale + row) : 0.f;
      const float l2z = valid && kMode != kGemm ? __ldcg(dv.row_log2z + row) : 0.f;
      const float cand = valid && kMode == kCands ? __ldcg(&cand_header(dv, row)->bound) : INFINITY;
      for (int t = t0; t < t1; ++t, ++tcount) {
        if (aborted) continue;
        const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
        int got = 0;
        if (lane == 0) got = mbar_wait(&tfull[ab], aph, abort_flag, dv.plan) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          aborted = true;
          continue;
        }
        tc_fence_after();
        const uint32_t tbase =
            tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBN + (uint32_t)(cg * kColsPerWarp);
#pragma unroll 1
        for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
          float acc[16];
          __syncwarp();
          tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
          if (cc == kColsPerWarp / 16 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
          }
          if (!valid) continue;
          store_cols<kMode, kCap>(dv, acc, row, t * kBN + cg * kColsPerWarp + cc * 16, kb0, scale, l2z, cand);
        }
      }
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

// The same two contractions on SM pairs, as the LM head runs above 256 positions: M = 256 rows
// per tcgen05.mma.cta_group::2 instruction, each CTA staging its own 128 rows of A (h, or P) and
// its own 128-row half of the 256-row B tile (W, or W^T), so B is streamed once for 256 rows and
// each SM takes in 32 KB from L2 per K block instead of 48 (the single-CTA form, whose 256-row
// B stage beside a 128-row A stage asks more of an SM's L2 ingress than the MMA rate allows).
// Units as ScUnits with 256-row tiles; barriers as in the LM head on pairs:
//   full[s]   (leader)  both CTAs' TMA bytes; the leader arms it with the total
//   empty[s]  (both)    released by the leader's commit, multicast to the pair
//   tfull[b]  (both)    accumulator ready, multicast from the leader's commit
//   tempty[b] (leader)  both CTAs' 16 epilogue warps release the accumulator
template <int kMode, bool kCap>
__global__ void __launch_bounds__(kThreadsLM, 1)
    k_selfcond_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Dev dv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int tile_ok[2];  // the epilogue's poller found the tile's accumulator ready (per TMEM buffer)
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
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
  // rows of the tick that left h, the temperature factors and log2 Z behind
  const int n_rows = (int)__ldcg(dv.sc_rows);
  const ScUnits su{(n_rows + 2 * kBM - 1) / (2 * kBM), (dv.d + kBN - 1) / kBN, (dv.d + kBK - 1) / kBK};
  const int n_units = su.units(dv, kMode);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int u = cid; u < n_units && ok; u += n_clusters) {
        int mt, t0, t1, kb0, kb1;
        su.at(dv, kMode, u, mt, t0, t1, kb0, kb1);
        for (int t = t0; t < t1 && ok; ++t) {
          for (int kb = kb0; kb < kb1; ++kb) {
            // both CTAs' loads complete the leader's full barrier, so the leader's MMAs never run a
            // lap ahead of either producer and this parity wait cannot alias
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, dv.plan)) {
              ok = false;
              break;
            }
            const uint32_t full_leader = peer_addr(smem_u32(&full[stage]), 0);
            if (leader) mbar_expect_tx(&full[stage], (uint32_t)(2 * (kStagePairA + kStagePairB)));
            tma_load_2d_pair(sA + stage * kStagePairA, &tmA, kb * kBK, mt * 2 * kBM + (int)rank * kBM, full_leader);
            tma_load_2d_pair(sB + stage * kStagePairB, &tmB, kb * kBK, t * kBN + (int)rank * (kBN / 2), full_leader);
            if (++stage == (uint32_t)kStagesPair) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // drain: one more lap of the ring's waits covers the releases of the last kStagesPair loads
      // (laps before the first load pass at once), so no copy or release is still in flight toward
      // this CTA when the pair exits
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
      const DescPair dA(sw128_desc(smem_u32(sA))), dB(sw128_desc(smem_u32(sB)));
      uint32_t stage = 0, phase = 0, tcount = 0;
      bool ok = true, any = false;
      for (int u = cid; u < n_units && ok; u += n_clusters) {
        int mt, t0, t1, kb0, kb1;
        su.at(dv, kMode, u, mt, t0, t1, kb0, kb1);
        for (int t = t0; t < t1 && ok; ++t, ++tcount) {
          const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
          if (!mbar_wait(&tempty[ab], aph ^ 1u, abort_flag, dv.plan)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * (uint32_t)kBN;
          for (int kb = kb0; kb < kb1; ++kb) {
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
                            (kb != kb0 || kk != 0) ? 1u : 0u);
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
        // wait (bounded) for the MMAs already issued before TMEM is freed
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
      int mt, t0, t1, kb0, kb1;
      su.at(dv, kMode, u, mt, t0, t1, kb0, kb1);
      const int row = mt * 2 * kBM + (int)rank * kBM + q * 32 + lane;
      const bool valid = row < n_rows;
      const float scale = valid && kMode != kGemm ? __ldcg(dv.row_scale + row) : 0.f;
      const float l2z = valid && kMode != kGemm ? __ldcg(dv.row_log2z + row) : 0.f;
      const float cand = valid && kMode == kCands ? __ldcg(&cand_header(dv, row)->bound) : INFINITY;
      for (int t = t0; t < t1; ++t, ++tcount) {
        if (aborted) continue;
        const uint32_t ab = tcount & 1u, aph = (tcount >> 1) & 1u;
        // one warp polls for the tile, the other fifteen wait on a named barrier (as in the LM head)
        if (warp == 2) {
          if (lane == 0) tile_ok[ab] = mbar_wait_poll(&tfull[ab], aph, 256u, abort_flag, dv.plan) ? 1 : 0;
          __syncwarp();
        }
        asm volatile("bar.sync 4, %0;" ::"r"(32 * kEpiWarps) : "memory");
        if (!*(volatile int*)&tile_ok[ab]) {
          aborted = true;
          continue;
        }
        tc_fence_after();
        const uint32_t tbase =
            tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBN + (uint32_t)(cg * kColsPerWarp);
#pragma unroll 1
        for (int cc = 0; cc < kColsPerWarp / 16; ++cc) {
          float acc[16];
          __syncwarp();
          tmem_ld16(tbase + (uint32_t)(cc * 16), acc);
          if (cc == kColsPerWarp / 16 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader[ab]);
          }
          if (!valid) continue;
          store_cols<kMode, kCap>(dv, acc, row, t * kBN + cg * kColsPerWarp + cc * 16, kb0, scale, l2z, cand);
        }
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

// e[c, p, :] = sum over the vocabulary chunks, in chunk order, of their shares
// of row a L + p, written where canvas c = row_canvas[a] keeps its positions.
__global__ void __launch_bounds__(256) k_selfcond_reduce(const Dev dv, float* __restrict__ out) {
  const int n_rows = (int)__ldcg(dv.sc_rows);
  const int d4 = dv.d >> 2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)n_rows * d4;
       i += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(i / d4), k = (int)(i - (long long)row * d4) * 4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int kc = 0; kc < dv.sc_kc; ++kc) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(dv.sc_part + ((size_t)kc * dv.rows_cap + row) * dv.d + k));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    const int a = row / dv.L, p = row - a * dv.L;
    const int c = __ldcg(dv.row_canvas + a);
    if (DG_IN_BOUNDS(dv.plan, c >= 0 && c < dv.B && row < dv.rows_cap, 10, c))
      *reinterpret_cast<float4*>(out + ((size_t)c * dv.L + p) * dv.d + k) = s;
  }
}

// ------------------------------------------------------------- top-K variant
// e[p, :] = sum over the K most probable tokens v of position p of q_v W[v, :],
// q the tick's softmax restricted to those K tokens and renormalised.
// TensorSharp's DiffusionGemma doc ("5. Acceleration status", its toggles)
// lists this cutoff of the self-conditioning input (experimental, K = 32 by
// default); the renormalisation keeps the one
// convex combination of embedding rows per position that the Annotated page's
// decode mode describes.  Tokens rank by z / T, equal values by the lower
// index.
//
// The tick's partial records hold each vocabulary chunk's largest u = z
// log2(e)/T of every row: when K is at most the number of chunks, the K-th
// largest of those maxima is a lower bound of the K-th largest u (K chunks
// each hold an entry at least as large).  k_topk_prep writes that bound (less
// a margin) into each row's candidate header, k_selfcond<kCands> -- the LM
// head again -- lists every entry that reaches it with its fp32 u from the
// accumulator, and k_selfcond_topk ranks the row's list (about K entries for a
// smooth distribution).  A row with more candidates than its list holds, or K
// above the number of chunks, takes the path below instead, from the bf16 P
// that the same launch wrote.
//
// That path takes one CTA per position (P >= 0, so a bf16 bit pattern orders
// like its value, and the rounding keeps order):
//   1. each thread's largest P over its entries; the K-th largest of these
//      maxima, s, is a lower bound of the K-th largest P (K threads each hold
//      an entry >= s), so every entry of the top K has P >= s;
//   2. the entries with P >= s (and P > 0) are the candidates -- about K of
//      them for any smooth distribution;
//   3. each candidate's logit again in fp32 (one warp per candidate: h . W[v],
//      the softcap, the row's temperature factor), and the K best by
//      (z desc, v asc), which ranks them;
//   4. q = 2^(u - u_max) / (sum over the K), e = sum_j q_j W[v_j, :] in rank
//      order (a fixed order: the result does not depend on the schedule).
// Entries whose P rounds to zero (p < 2^-126) are never kept: their weights
// would be below 2^-108 of the largest.  When more than kTopKCand entries are
// candidates (a plateau of equal probabilities at the top, as with equal
// logits), the row is taken in windows of kTopKWin entries and each window's
// candidates are merged into the running K best: slower, the same result.
constexpr int kTopKThreads = 256;
constexpr int kTopKWarps = kTopKThreads / 32;
constexpr int kTopKWin = kTopKThreads * 8;  // one 16-byte group of P per thread
static_assert(kTopKWin <= kTopKCand, "a window's candidates fit the candidate list");

// The 16-bit keys of entries [8 i, 8 i + 8) of a row of P, -1 past V.
__device__ __forceinline__ void p_keys8(const uint16_t* __restrict__ prow, int i, int V, int (&key)[8]) {
  const uint4 q = __ldcg(reinterpret_cast<const uint4*>(prow) + i);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int v = 8 * i + j;
    key[j] = v < V ? (int)((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu) : -1;
  }
}

// (u, v) ranks before (u2, v2): larger logit first, equal logits by the lower index.
__device__ __forceinline__ bool topk_before(float u, int v, float u2, int v2) { return u > u2 || (u == u2 && v < v2); }

// u = z' log2(e) for each of cand[i0, i1): one warp per candidate, fp32 h . W[v] accumulated in
// a fixed order, then the softcap and the row's factor log2(e) / T (as the tick forms them).
__device__ __forceinline__ void topk_logits(const Dev& dv, const uint16_t* __restrict__ W,
                                            const uint16_t* __restrict__ hrow, float scale, const int* cand_v,
                                            float* cand_u, int i0, int i1) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d8 = dv.d >> 3;
  for (int i = i0 + warp; i < i1; i += kTopKWarps) {
    const int v = cand_v[i];
    const uint4* wr = reinterpret_cast<const uint4*>(W + (size_t)v * dv.d);
    const uint4* hr = reinterpret_cast<const uint4*>(hrow);
    float acc = 0.f;
    for (int k = lane; k < d8; k += 32) {
      const uint4 a = __ldg(hr + k), b = __ldg(wr + k);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = fmaf(__uint_as_float(aw[j] << 16), __uint_as_float(bw[j] << 16), acc);
        acc = fmaf(__uint_as_float(aw[j] & 0xFFFF0000u), __uint_as_float(bw[j] & 0xFFFF0000u), acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) {
      float z = acc;
      if (dv.softcap > 0.f) z = dv.softcap * tanhf(z * dv.inv_softcap);
      const float u = z * scale;
      cand_u[i] = u == u ? u : -INFINITY;  // a non-finite logit ranks last
    }
  }
}

// Keeps the best min(K, n) of cand[0, n) in rank order at cand[0, ...); returns how many.
__device__ __forceinline__ int topk_select(int* cand_v, float* cand_u, int n, int K, int* sel_v, float* sel_u) {
  for (int i = threadIdx.x; i < n; i += kTopKThreads) {
    const float u = cand_u[i];
    const int v = cand_v[i];
    int r = 0;
    for (int j = 0; j < n && r < K; ++j) r += topk_before(cand_u[j], cand_v[j], u, v) ? 1 : 0;
    if (r < K) {
      sel_v[r] = v;
      sel_u[r] = u;
    }
  }
  __syncthreads();
  const int m = n < K ? n : K;
  for (int i = threadIdx.x; i < m; i += kTopKThreads) {
    cand_v[i] = sel_v[i];
    cand_u[i] = sel_u[i];
  }
  __syncthreads();
  return m;
}

// One warp per row: the row's bound -- the K-th largest of its chunk maxima (ties by chunk), less
// a margin of 2^-12 (|bound| + 1), and no lower than log2 Z - 126, below which P rounds to zero --
// and an empty candidate list.
__global__ void __launch_bounds__(256) k_topk_prep(const Dev dv, int top_k) {
  __shared__ float m_s[8][kChunkTarget];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  const int n_rows = (int)__ldcg(dv.sc_rows);
  if (row >= n_rows) return;
  const int nc = dv.n_chunks, K = top_k < dv.V ? top_k : dv.V;
  CandHeader* hd = cand_header(dv, row);
  if (K > nc || nc > kChunkTarget) {
    if (lane == 0) *hd = CandHeader{0u, INFINITY, 1u, 0u};
    return;
  }
  for (int c = lane; c < nc; c += 32) {
    const float m = __ldcg(&dv.part[(size_t)row * dv.n_sub + c].m);
    m_s[warp][c] = m == m ? m : -INFINITY;
  }
  __syncwarp();
  for (int c = lane; c < nc; c += 32) {
    const float m = m_s[warp][c];
    int r = 0;
    for (int j = 0; j < nc; ++j) r += (m_s[warp][j] > m || (m_s[warp][j] == m && j < c)) ? 1 : 0;
    if (r == K - 1) {
      const float floor_u = __ldcg(dv.row_log2z + row) - 126.f;
      const float b = m - 0x1p-12f * (fabsf(m) + 1.f);
      *hd = CandHeader{0u, b > floor_u ? b : floor_u, 0u, 0u};
    }
  }
}

// The K best of a row from its bf16 probabilities (the path described above); they are left in
// rank order at cand[0, n_keep).
__device__ __noinline__ int topk_from_probs(const Dev& dv, const uint16_t* __restrict__ W,
                                            const uint16_t* __restrict__ prow, const uint16_t* __restrict__ hrow,
                                            float scale, int K, int* tmax, int* cand_v, float* cand_u, int* sel_v,
                                            float* sel_u, int* s_thresh_p, int* s_count_p) {
  int& s_thresh = *s_thresh_p;
  int& s_count = *s_count_p;
  const int tid = threadIdx.x;
  const int V = dv.V;
  const int n8 = dv.sc_vpad >> 3;

  // 1. this thread's largest key; s = the K-th largest of the threads' maxima (ties by thread)
  int mx = -1;
#pragma unroll 4
  for (int i = tid; i < n8; i += kTopKThreads) {
    int key[8];
    p_keys8(prow, i, V, key);
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = max(mx, key[j]);
  }
  tmax[tid] = mx;
  if (tid == 0) s_count = 0;
  __syncthreads();
  {
    int r = 0;
    for (int j = 0; j < kTopKThreads; ++j) r += (tmax[j] > mx || (tmax[j] == mx && j < tid)) ? 1 : 0;
    if (r == K - 1) s_thresh = mx > 1 ? mx : 1;  // entries whose P rounds to zero are never kept
  }
  __syncthreads();
  const int s = s_thresh;

  // 2. the candidates: entries with key >= s
#pragma unroll 4
  for (int i = tid; i < n8; i += kTopKThreads) {
    int key[8];
    p_keys8(prow, i, V, key);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (key[j] >= s) {
        const int at = atomicAdd(&s_count, 1);
        if (at < kTopKCand) cand_v[at] = 8 * i + j;
      }
  }
  __syncthreads();
  const int n_cand = s_count;

  // 3. exact logits of the candidates and the K best
  int n_keep;
  if (n_cand <= kTopKCand) {
    topk_logits(dv, W, hrow, scale, cand_v, cand_u, 0, n_cand);
    __syncthreads();
    n_keep = topk_select(cand_v, cand_u, n_cand, K, sel_v, sel_u);
  } else {
    // a plateau at the top: windows of kTopKWin entries in index order, each window's
    // candidates merged into the running K best (held at cand[0, n_keep))
    n_keep = 0;
    for (int w0 = 0; w0 < n8; w0 += kTopKThreads) {
      __syncthreads();
      if (tid == 0) s_count = 0;
      __syncthreads();
      const int i = w0 + tid;
      if (i < n8) {
        int key[8];
        p_keys8(prow, i, V, key);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (key[j] >= s) cand_v[n_keep + atomicAdd(&s_count, 1)] = 8 * i + j;
      }
      __syncthreads();
      const int n_new = s_count;
      if (n_new == 0) continue;
      topk_logits(dv, W, hrow, scale, cand_v, cand_u, n_keep, n_keep + n_new);
      __syncthreads();
      n_keep = topk_select(cand_v, cand_u, n_keep + n_new, K, sel_v, sel_u);
    }
  }

  return n_keep;
}

// 4. the weights of the kept cand[0, n_keep) (rank order, largest u first), summed in rank order,
// and the weighted rows of W, written where the row's canvas keeps its positions.
__device__ __noinline__ void topk_write(const Dev& dv, const uint16_t* __restrict__ W, int row, int n_keep,
                                        const int* cand_v, const float* cand_u, float* sel_u, float* s_sum_p,
                                        float* __restrict__ out) {
  float& s_sum = *s_sum_p;
  const int tid = threadIdx.x;
  if (tid == 0) {
    float S = 0.f;
    for (int j = 0; j < n_keep; ++j) S += exp2f(cand_u[j] - cand_u[0]);
    s_sum = S;
  }
  __syncthreads();
  for (int j = tid; j < n_keep; j += kTopKThreads) sel_u[j] = exp2f(cand_u[j] - cand_u[0]) / s_sum;
  __syncthreads();
  const int a = row / dv.L, p = row - a * dv.L;
  const int c = __ldcg(dv.row_canvas + a);
  if (!DG_IN_BOUNDS(dv.plan, c >= 0 && c < dv.B && row < dv.rows_cap, 10, c)) return;
  float* orow = out + ((size_t)c * dv.L + p) * dv.d;
  for (int k8 = tid; k8 < (dv.d >> 3); k8 += kTopKThreads) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < n_keep; ++j) {
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(W + (size_t)cand_v[j] * dv.d) + k8);
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
      const float q = sel_u[j];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        acc[2 * t] = fmaf(q, __uint_as_float(bw[t] << 16), acc[2 * t]);
        acc[2 * t + 1] = fmaf(q, __uint_as_float(bw[t] & 0xFFFF0000u), acc[2 * t + 1]);
      }
    }
    float4* o = reinterpret_cast<float4*>(orow + 8 * k8);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

__global__ void __launch_bounds__(kTopKThreads)
    k_selfcond_topk(const Dev dv, const uint16_t* __restrict__ W, int top_k, float* __restrict__ out) {
  __shared__ int tmax[kTopKThreads];
  __shared__ int cand_v[kTopKCand + DG_SC_TOPK_MAX];
  __shared__ float cand_u[kTopKCand + DG_SC_TOPK_MAX];
  __shared__ int sel_v[DG_SC_TOPK_MAX];
  __shared__ float sel_u[DG_SC_TOPK_MAX];
  __shared__ int s_thresh, s_count;
  __shared__ float s_sum;

  const int row = blockIdx.x;
  const int n_rows = (int)__ldcg(dv.sc_rows);
  if (row >= n_rows) return;
  const int tid = threadIdx.x;
  const int K = top_k < dv.V ? top_k : dv.V;
  const uint16_t* prow = dv.sc_probs + (size_t)row * dv.sc_vpad;
  const uint16_t* hrow = dv.h + (size_t)row * dv.d;
  const float scale = __ldcg(dv.row_scale + row);

  int n_keep;
  const uint4 hd = __ldcg(reinterpret_cast<const uint4*>(cand_header(dv, row)));  // {count, bound, dense, -}
  if (hd.z == 0u && hd.x >= 1u && hd.x <= cand_capacity(dv)) {
    // the row's candidates as the LM head listed them, with their fp32 u
    const int2* lst = cand_list(dv, row);
    const int n = (int)hd.x;
    for (int i = tid; i < n; i += kTopKThreads) {
      const int2 e = __ldcg(lst + i);
      cand_v[i] = e.x;
      const float u = __int_as_float(e.y);
      cand_u[i] = u == u ? u : -INFINITY;
    }
    __syncthreads();
    n_keep = topk_select(cand_v, cand_u, n, K, sel_v, sel_u);
  } else {
    n_keep = topk_from_probs(dv, W, prow, hrow, scale, K, tmax, cand_v, cand_u, sel_v, sel_u, &s_thresh, &s_count);
  }
  topk_write(dv, W, row, n_keep, cand_v, cand_u, sel_u, &s_sum, out);
}

// W [V, d] -> W^T [d, V_pad], zero past V, through 32 x 32 tiles in shared memory.
__global__ void __launch_bounds__(256) k_transpose_w(const uint16_t* __restrict__ W, uint16_t* __restrict__ WT, int V,
                                                     int d, int v_pad) {
  __shared__ uint16_t t[32][33];
  const int v0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int v = v0 + i, k = k0 + (int)threadIdx.x;
    t[i][threadIdx.x] = (v < V && k < d) ? W[(size_t)v * d + k] : (uint16_t)0;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int k = k0 + i, v = v0 + (int)threadIdx.x;
    if (k < d && v < v_pad) WT[(size_t)k * v_pad + v] = t[threadIdx.x][i];
  }
}

constexpr size_t kSmemBytesSc = 1024 + (size_t)kStages * (kStageA + kStageB) + 256;
constexpr size_t kSmemBytesScPair = 1024 + (size_t)kStagesPair * (kStagePairA + kStagePairB) + 256;
static_assert(kSmemBytesSc <= 232448 && kSmemBytesScPair <= 232448, "shared memory per CTA");

template <int kMode, bool kCap>
cudaError_t launch_pair(int units, int num_sms, const CUtensorMap* tmA, const CUtensorMap* tmB, const Dev& dv,
                        cudaStream_t st) {
  int pairs = units < num_sms / 2 ? units : num_sms / 2;
  if (pairs < 1) pairs = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreadsLM);
  cfg.dynamicSmemBytes = kSmemBytesScPair;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_selfcond_pair<kMode, kCap>, *tmA, *tmB, dv);
}

// The LM head again, its epilogue writing P in bf16 (the first kernel of either variant; kMode
// kCands also lists the top-K candidates).
template <int kMode>
cudaError_t launch_probs(const Dev& dv, bool pair, const CUtensorMap* tm_h, const CUtensorMap* tm_w, int num_sms,
                         cudaStream_t st) {
  const bool cap = dv.softcap > 0.f;
  if (pair) {
    // 256-row tiles on SM pairs; the maps' B boxes are 128 rows (each CTA's half of a tile)
    const int max_mt = (dv.max_active * dv.L + 2 * kBM - 1) / (2 * kBM);
    return cap ? launch_pair<kMode, true>(max_mt * dv.n_chunks, num_sms, tm_h, tm_w, dv, st)
               : launch_pair<kMode, false>(max_mt * dv.n_chunks, num_sms, tm_h, tm_w, dv, st);
  }
  const int max_mt = (dv.max_active * dv.L + kBM - 1) / kBM;
  int g1 = max_mt * dv.n_chunks;
  g1 = g1 < num_sms ? g1 : num_sms;
  if (cap)
    k_selfcond<kMode, true><<<g1, kThreadsLM, kSmemBytesSc, st>>>(*tm_h, *tm_w, dv);
  else
    k_selfcond<kMode, false><<<g1, kThreadsLM, kSmemBytesSc, st>>>(*tm_h, *tm_w, dv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t selfcond_configure() {
  cudaError_t e = cudaSuccess;
  for (auto k : {k_selfcond<kProbs, false>, k_selfcond<kProbs, true>, k_selfcond<kGemm, false>,
                 k_selfcond<kGemm, true>, k_selfcond<kCands, false>, k_selfcond<kCands, true>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesSc);
  for (auto k : {k_selfcond_pair<kProbs, false>, k_selfcond_pair<kProbs, true>, k_selfcond_pair<kGemm, false>,
                 k_selfcond_pair<kCands, false>, k_selfcond_pair<kCands, true>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesScPair);
  return e;
}

cudaError_t launch_transpose_w(const void* w, uint16_t* wt, int V, int d, int v_pad, cudaStream_t st) {
  k_transpose_w<<<dim3(v_pad / 32, (d + 31) / 32), dim3(32, 8), 0, st>>>(static_cast<const uint16_t*>(w), wt, V, d,
                                                                        v_pad);
  return cudaGetLastError();
}

cudaError_t launch_selfcond(const Dev& dv, bool pair, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                            const CUtensorMap* tm_p, const CUtensorMap* tm_wt, float* out, int num_sms, cudaStream_t st) {
  const int n_dt = (dv.d + kBN - 1) / kBN;
  cudaError_t e = launch_probs<kProbs>(dv, pair, tm_h, tm_w, num_sms, st);
  if (e != cudaSuccess) return e;
  if (pair) {
    const int max_mt = (dv.max_active * dv.L + 2 * kBM - 1) / (2 * kBM);
    e = launch_pair<kGemm, false>(max_mt * n_dt * dv.sc_kc, num_sms, tm_p, tm_wt, dv, st);
    if (e != cudaSuccess) return e;
  } else {
    const int max_mt = (dv.max_active * dv.L + kBM - 1) / kBM;
    int g2 = max_mt * n_dt * dv.sc_kc;
    g2 = g2 < num_sms ? g2 : num_sms;
    k_selfcond<kGemm, false><<<g2, kThreadsLM, kSmemBytesSc, st>>>(*tm_p, *tm_wt, dv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long long work = (long long)dv.max_active * dv.L * (dv.d >> 2);
  long long blocks = (work + 255) / 256;
  if (blocks > 8 * num_sms) blocks = 8 * num_sms;
  k_selfcond_reduce<<<(int)(blocks > 0 ? blocks : 1), 256, 0, st>>>(dv, out);
  return cudaGetLastError();
}

cudaError_t launch_selfcond_topk(const Dev& dv, bool pair, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                                 const void* w, int top_k, float* out, int num_sms, cudaStream_t st) {
  const int rows = dv.max_active * dv.L;  // CTAs past the tick's rows return at once
  k_topk_prep<<<(rows + 7) / 8 > 0 ? (rows + 7) / 8 : 1, 256, 0, st>>>(dv, top_k);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_probs<kCands>(dv, pair, tm_h, tm_w, num_sms, st);
  if (e != cudaSuccess) return e;
  k_selfcond_topk<<<rows > 0 ? rows : 1, kTopKThreads, 0, st>>>(dv, static_cast<const uint16_t*>(w), top_k, out);
  return cudaGetLastError();
}

}  // namespace dg
