// Host side of the C ABI in include/dg_sampler.h: config validation,
// workspace layout, TMA tensor maps, the per-tick launch sequence and state
// transfer.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "dg_internal.cuh"

namespace dg {
// defined with the other self-conditioning kernels (dg_selfcond.cu)
cudaError_t launch_selfcond_topk(const Dev& dv, bool pair, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                                 const void* w, int top_k, float* out, int num_sms, cudaStream_t st);
}  // namespace dg

struct dg_sampler {
  dg_config cfg;
  std::vector<uint64_t> seeds;
  std::vector<int32_t> admit;
  dg::Dev dv;
  CUtensorMap tmA, tmB;
  CUtensorMap tmP, tmWT;  // self-conditioning: P, and W^T in boxes of the LM head's B rows
  const void* w_vocab = nullptr;  // the borrowed W rows (the top-K self-conditioning variant reads them directly)
  bool pair;  // LM head on CTA pairs (tcgen05 cta_group::2), chosen when a tick can hold >= 256 rows
  bool split = false;            // the vocabulary is split across ranks (dg_denoise_step_partial / _finish)
  bool partial_pending = false;  // a partial tick waits for its finishing step
  cudaStream_t stream;
  int num_sms;
  int64_t host_tick;
  int64_t tick_bound;
  void* ws;
  size_t ws_bytes;
  std::vector<size_t> guards;  // debug build: workspace offsets of the canary guards
  cudaEvent_t timing[4];
  bool timed;
  char err[512];
  // pinned copy of the plan's error latch: reading it back does not go through
  // a staged pageable copy, so a step that returns results synchronizes once
  dg::Plan* pl_host = nullptr;
  // pinned staging of the plan .. entropies span for dg_denoise_step_host, made on its first call
  uint8_t* stage_host = nullptr;
  size_t stage_bytes = 0, stage_x = 0, stage_H = 0;  // span size and offsets of x and H in it
  ~dg_sampler() {
    if (pl_host) cudaFreeHost(pl_host);
    if (stage_host) cudaFreeHost(stage_host);
  }
};

namespace {

char g_create_err[512] = "";

void set_err(char* buf, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, 512, fmt, ap);
  va_end(ap);
}

struct Layout {
  size_t slots, plan, active, x, committed, commit_step, prev_amax, tokens_out, commit_steps_out, H, logZ, y, amax, h,
      part, row_best, resid,
      canvas_rows, temps, sync;
  size_t total;
  std::vector<size_t> guards;  // debug build: offsets of the 256-byte canary guards
  int rows_cap, n_vtiles, tiles_per_chunk, n_chunks, n_sub, max_active;
  int chunk_begin, chunk_end;  // this rank's vocabulary chunks
  // self-conditioning buffers (0 when off)
  size_t wt, probs, sc_part, row_scale, row_log2z, row_canvas, sc_rows;
  int sc_vpad, sc_kc, sc_kbpc;
};

// The LM head's vocabulary chunking, which depends on V only: 256-entry tiles,
// at most kChunkTarget chunks of equally many tiles (the last may be shorter).
void vocab_chunking(int32_t V, int* n_vtiles, int* tiles_per_chunk, int* n_chunks) {
  *n_vtiles = (V + dg::kBN - 1) / dg::kBN;
  const int target = *n_vtiles < dg::kChunkTarget ? *n_vtiles : dg::kChunkTarget;
  *tiles_per_chunk = (*n_vtiles + target - 1) / target;
  *n_chunks = (*n_vtiles + *tiles_per_chunk - 1) / *tiles_per_chunk;
}

// Chunks [c0, c1) of rank r of G (G <= 1: all of them).
void rank_chunks(int n_chunks, int G, int r, int* c0, int* c1) {
  if (G <= 1) {
    *c0 = 0;
    *c1 = n_chunks;
    return;
  }
  *c0 = (int)((int64_t)r * n_chunks / G);
  *c1 = (int)((int64_t)(r + 1) * n_chunks / G);
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
constexpr size_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;

bool validate(const dg_config* c, char* why) {
  if (!c) return set_err(why, "config is NULL"), false;
  if (c->vocab < 2) return set_err(why, "vocab must be >= 2 (got %d)", c->vocab), false;
  if (c->hidden < 8 || c->hidden > 16384 || c->hidden % 8)
    return set_err(why, "hidden must be a multiple of 8 in [8, 16384] (got %d)", c->hidden), false;
  if (c->canvas_len < 1 || c->canvas_len > 1024)
    return set_err(why, "canvas_len must be in [1, 1024] (got %d)", c->canvas_len), false;
  if (c->n_canvases < 1) return set_err(why, "n_canvases must be >= 1"), false;
  if (c->gen_blocks < 1 || c->gen_blocks > 65535) return set_err(why, "gen_blocks must be in [1, 65535]"), false;
  if (c->num_inference_steps < 1 || c->num_inference_steps > 1024)
    return set_err(why, "num_inference_steps must be in [1, 1024] (got %d)", c->num_inference_steps), false;
  if (!(c->t_min > 0.f) || !(c->t_max > 0.f) || !std::isfinite(c->t_min) || !std::isfinite(c->t_max))
    return set_err(why, "t_min and t_max must be finite and > 0"), false;
  if (!(c->entropy_bound >= 0.f) || !std::isfinite(c->entropy_bound))
    return set_err(why, "entropy_bound must be finite and >= 0"), false;
  if (!(c->confidence >= 0.f) || !std::isfinite(c->confidence))
    return set_err(why, "confidence must be finite and >= 0"), false;
  if (!(c->rms_eps >= 0.f) || !std::isfinite(c->rms_eps)) return set_err(why, "rms_eps must be finite and >= 0"), false;
  if (!(c->softcap >= 0.f) || !std::isfinite(c->softcap)) return set_err(why, "softcap must be finite and >= 0"), false;
  if (c->max_active < 0 || c->max_active > c->n_canvases)
    return set_err(why, "max_active must be in [0, n_canvases]"), false;
  if ((int64_t)c->n_canvases * c->canvas_len > (int64_t)1 << 24)
    return set_err(why, "n_canvases * canvas_len must be <= 2^24"), false;
  if (c->admit_tick)
    for (int i = 0; i < c->n_canvases; ++i)
      if (c->admit_tick[i] < 0) return set_err(why, "admit_tick[%d] is negative", i), false;
  if (c->self_cond != 0 && c->self_cond != 1) return set_err(why, "self_cond must be 0 or 1"), false;
  if (c->self_cond && c->vocab_ranks > 1)
    return set_err(why, "self_cond needs the whole vocabulary (vocab_ranks <= 1)"), false;
  if (c->vocab_ranks < 0 || c->vocab_rank < 0 || c->vocab_rank >= (c->vocab_ranks > 1 ? c->vocab_ranks : 1))
    return set_err(why, "vocab_rank must be in [0, vocab_ranks) (got %d of %d)", c->vocab_rank, c->vocab_ranks),
           false;
  return true;
}

// Returns 1 ok, 0 invalid, -1 unsupported.
int make_layout(const dg_config* c, Layout* L, char* why) {
  if (!validate(c, why)) return 0;
  if (c->stability < 1 || c->stability > 1024)
    return set_err(why, "stability must be in [1, 1024] (got %d)", c->stability), 0;
  if (c->mode != DG_FREEZE && c->mode != DG_REACCEPT)
    return set_err(why, "mode must be DG_FREEZE or DG_REACCEPT (got %d)", c->mode), 0;
  const size_t B = c->n_canvases, Lc = c->canvas_len, d = c->hidden, G = c->gen_blocks;
  L->max_active = c->max_active ? c->max_active : c->n_canvases;
  const size_t rows = (size_t)L->max_active * Lc;
  L->rows_cap = (int)((rows + 255) / 256 * 256);
  vocab_chunking(c->vocab, &L->n_vtiles, &L->tiles_per_chunk, &L->n_chunks);
  L->n_sub = L->n_chunks * dg::kSubPerChunk;
  if (c->vocab_ranks > L->n_chunks)
    return set_err(why, "vocab_ranks must be at most the %d vocabulary chunks (got %d)", L->n_chunks, c->vocab_ranks),
           0;
  rank_chunks(L->n_chunks, c->vocab_ranks, c->vocab_rank, &L->chunk_begin, &L->chunk_end);
  size_t o = 0;
  L->guards.clear();
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
#ifdef DG_DEBUG_CHECKS
    L->guards.push_back(o);  // a guard after every sub-buffer
    o += kGuardBytes;
#endif
    return at;
  };
  L->slots = take(sizeof(dg_slot) * B);
  // plan, canvas and entropies adjacent: a host step reads all three back in one copy
  L->plan = take(sizeof(dg::Plan));
  L->x = take(4 * B * Lc);
  L->H = take(4 * B * Lc);
  L->active = take(sizeof(int32_t) * B);
  L->committed = take(B * Lc);
  L->commit_step = take(2 * B * Lc);
  L->prev_amax = take(4 * B * Lc);
  L->tokens_out = take(4 * B * G * Lc);
  L->commit_steps_out = take(2 * B * G * Lc);
  L->logZ = take(4 * B * Lc);
  L->y = take(4 * B * Lc);
  L->amax = take(4 * B * Lc);
  L->h = take(2 * (size_t)L->rows_cap * d);
  L->part = take(sizeof(dg::Partial) * (size_t)L->rows_cap * L->n_sub);
  L->row_best = take(sizeof(unsigned long long) * (size_t)L->rows_cap);
  L->resid = take(4 * B * Lc * d);
  L->canvas_rows = take(4 * B);
  L->temps = take(4 * (size_t)c->num_inference_steps);
  // rows_ready, fin_started, slab_done[rows_cap / 128], units_done
  L->sync = take(4 * (3 + (size_t)L->rows_cap / 128));
  L->wt = L->probs = L->sc_part = L->row_scale = L->row_log2z = L->row_canvas = L->sc_rows = 0;
  L->sc_vpad = L->sc_kc = L->sc_kbpc = 0;
  if (c->self_cond) {
    // the contraction's grid: row tiles x 256-wide d tiles x vocabulary chunks, about two units per
    // SM (single CTAs) or per SM pair (256 positions and up, the sampler's rule), rounded so that no
    // pair takes a third
    L->sc_vpad = L->n_vtiles * dg::kBN;
    const bool pair = rows >= 2 * dg::kBM;
    const int kbv = L->sc_vpad / dg::kBK, n_dt = (int)((d + 255) / 256);
    const int n_mt = (int)((rows + (pair ? 2 : 1) * dg::kBM - 1) / ((pair ? 2 : 1) * dg::kBM));
    int kc = pair ? 152 / (n_mt * n_dt) : (304 + n_mt * n_dt - 1) / (n_mt * n_dt);
    kc = kc < 1 ? 1 : (kc > kbv ? kbv : kc);
    L->sc_kbpc = (kbv + kc - 1) / kc;
    L->sc_kc = (kbv + L->sc_kbpc - 1) / L->sc_kbpc;  // every chunk holds at least one K block
    L->wt = take(2 * d * (size_t)L->sc_vpad);
    L->probs = take(2 * (size_t)L->rows_cap * L->sc_vpad);
    L->sc_part = take(4 * (size_t)L->sc_kc * L->rows_cap * d);
    L->row_scale = take(4 * (size_t)L->rows_cap);
    L->row_log2z = take(4 * (size_t)L->rows_cap);
    L->row_canvas = take(4 * B);
    L->sc_rows = take(4);
  }
  L->total = o;
  return 1;
}

dg_status cuda_fail(char* buf, cudaError_t e, const char* what) {
  set_err(buf, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return DG_ERR_CUDA;
}

// dg_debug_fail_cuda_call: how many more checked CUDA calls run before one is
// replaced by a reported failure (-1: none).
std::atomic<int> g_fail_after{-1};

// Whether this checked CUDA call is the one to fail (it is then not made).
bool injected_failure() {
  int v = g_fail_after.load();
  while (v >= 0) {
    if (g_fail_after.compare_exchange_weak(v, v - 1)) return v == 0;
  }
  return false;
}

#define DG_CUDA(s, call, what)                                                          \
  do {                                                                                  \
    if (injected_failure()) return cuda_fail((s), cudaErrorLaunchFailure, (what));     \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess) return cuda_fail((s), e_, (what));                           \
  } while (0)

// An NVTX range over one entry point (shown by profilers that collect NVTX; free otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

PFN_cuTensorMapEncodeTiled_v12000 get_encode(char* why) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
    set_err(why, "cuTensorMapEncodeTiled not available from the driver");
    return nullptr;
  }
  fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box [box_rows, 64],
// 128-byte swizzle (the layout the MMA descriptors expect), zero fill outside.
bool encode_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, char* why) {
  auto enc = get_encode(why);
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)dg::kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_err(why, "cuTensorMapEncodeTiled failed (CUresult %d) for a [%llu x %llu] matrix", (int)r,
            (unsigned long long)rows, (unsigned long long)cols);
    return false;
  }
  return true;
}

// The status a latched device error in the plan stands for.
dg_status latched_status(dg_sampler* s, const dg::Plan& pl);

dg_status check_device_error(dg_sampler* s) {
  DG_CUDA(s->err, cudaMemcpyAsync(s->pl_host, s->dv.plan, sizeof(dg::Plan), cudaMemcpyDeviceToHost, s->stream),
          "read plan");
  DG_CUDA(s->err, cudaStreamSynchronize(s->stream), "synchronize");
  return latched_status(s, *s->pl_host);
}

dg_status latched_status(dg_sampler* s, const dg::Plan& pl) {
  if (pl.err == dg::kErrNonFinite) {
    set_err(s->err, "non-finite logit statistics at position index %d", pl.err_info[1]);
    return DG_ERR_NONFINITE;
  }
  if (pl.err == dg::kErrTimeout) {
    set_err(s->err, "a bounded wait expired: %s (CTA %d, detail %d)", dg::wait_site_name(pl.err_info[2]),
            pl.err_info[0], pl.err_info[3]);
    return DG_ERR_TIMEOUT;
  }
  if (pl.err == dg::kErrBounds) {
    set_err(s->err, "a debug index check failed at site %d (value %d); the access was skipped", pl.err_info[2],
            pl.err_info[3]);
    return DG_ERR_BOUNDS;
  }
  return DG_OK;
}

// The first part of a tick: RMSNorm and the LM head (with the timing marks 0..2).
dg_status tick_front(dg_sampler* s, const float* resid);
// The finishing kernel of a tick (timing mark 3).
dg_status tick_back(dg_sampler* s);

dg_status tick(dg_sampler* s, const float* resid) {
  dg_status st = tick_front(s, resid);
  return st == DG_OK ? tick_back(s) : st;
}

dg_status mark_event(dg_sampler* s, int i) {
  // external event nodes when the tick is captured in a CUDA graph, plain records otherwise
  if (!s->timed) return DG_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  DG_CUDA(s->err, cudaStreamIsCapturing(s->stream, &cap), "query stream capture");
  const unsigned rec_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  DG_CUDA(s->err, cudaEventRecordWithFlags(s->timing[i], s->stream, rec_flags), "record timing event");
  return DG_OK;
}

dg_status tick_back(dg_sampler* s) {
  DG_CUDA(s->err, dg::launch_finish(s->dv, s->stream), "launch finish");
  dg_status st = mark_event(s, 3);
  if (st != DG_OK) return st;
  ++s->host_tick;
  return DG_OK;
}

dg_status tick_front(dg_sampler* s, const float* resid) {
  if (s->host_tick >= s->tick_bound) {
    set_err(s->err, "every canvas has finished (tick %lld)", (long long)s->host_tick);
    return DG_ERR_STATE;
  }
  dg_status st = mark_event(s, 0);
  if (st != DG_OK) return st;
  // the LM head on SM pairs forms the RMSNorm rows itself
  if (!s->pair) DG_CUDA(s->err, dg::launch_rmsnorm(s->dv, resid, s->stream), "launch rmsnorm");
  if ((st = mark_event(s, 1)) != DG_OK) return st;
  DG_CUDA(s->err,
          s->pair ? dg::launch_lmhead_pair(s->dv, resid, &s->tmA, &s->tmB, s->num_sms, s->stream)
                  : dg::launch_lmhead(s->dv, &s->tmA, &s->tmB, s->num_sms, s->stream),
          "launch lm head");
  return mark_event(s, 2);
}

}  // namespace

extern "C" {

size_t dg_workspace_size(const dg_config* cfg) {
  Layout L;
  char why[512];
  if (make_layout(cfg, &L, why) != 1) return 0;
  return L.total;
}

dg_status dg_sampler_create(const dg_config* cfg, const void* w_vocab, const float* norm_w, void* workspace,
                            size_t ws_bytes, dg_stream_t stream, dg_sampler** out) {
  NvtxRange nvtx_("dg_sampler_create");
  g_create_err[0] = 0;
  if (!out) return set_err(g_create_err, "out is NULL"), DG_ERR_ARG;
  *out = nullptr;
  Layout L;
  const int lr = make_layout(cfg, &L, g_create_err);
  if (lr == 0) return DG_ERR_ARG;
  if (lr < 0) return DG_ERR_UNSUPPORTED;
  if (!w_vocab) return set_err(g_create_err, "w_vocab is NULL"), DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(w_vocab) % 16)
    return set_err(g_create_err, "w_vocab must be 16-byte aligned"), DG_ERR_ALIGN;
  if (norm_w && reinterpret_cast<uintptr_t>(norm_w) % 16)
    return set_err(g_create_err, "norm_w must be 16-byte aligned"), DG_ERR_ALIGN;
  if (!workspace || ws_bytes < L.total)
    return set_err(g_create_err, "workspace needs %zu bytes (got %zu)", L.total, workspace ? ws_bytes : 0),
           DG_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return set_err(g_create_err, "workspace must be 256-byte aligned"), DG_ERR_ALIGN;

  int dev = 0, major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(g_create_err, e, "query device");
  if (major != 10 || minor != 3) {
    set_err(g_create_err, "this library is built for sm_103a (GB300); device is sm_%d%d", major, minor);
    return DG_ERR_UNSUPPORTED;
  }

  dg_sampler* s = new (std::nothrow) dg_sampler();
  if (!s) return set_err(g_create_err, "out of host memory"), DG_ERR_ARG;
  s->cfg = *cfg;
  s->w_vocab = w_vocab;
  const int B = cfg->n_canvases;
  s->seeds.resize(B);
  s->admit.resize(B);
  for (int c = 0; c < B; ++c) {
    s->seeds[c] = cfg->seeds ? cfg->seeds[c] : (uint64_t)c;
    s->admit[c] = cfg->admit_tick ? cfg->admit_tick[c] : 0;
  }
  s->cfg.seeds = nullptr;
  s->cfg.admit_tick = nullptr;
  s->stream = reinterpret_cast<cudaStream_t>(stream);
  s->num_sms = sms;
  s->ws = workspace;
  s->ws_bytes = ws_bytes;
  s->err[0] = 0;
  s->host_tick = 0;
  int32_t max_admit = 0;
  for (int c = 0; c < B; ++c) max_admit = s->admit[c] > max_admit ? s->admit[c] : max_admit;
  // every canvas has finished by then, even if it waited for a free slot behind all others
  s->tick_bound = (int64_t)max_admit + (int64_t)cfg->gen_blocks * cfg->num_inference_steps * B;

  uint8_t* w = static_cast<uint8_t*>(workspace);
  dg::Dev& dv = s->dv;
  dv.slots = reinterpret_cast<dg_slot*>(w + L.slots);
  dv.plan = reinterpret_cast<dg::Plan*>(w + L.plan);
  dv.active = reinterpret_cast<int32_t*>(w + L.active);
  dv.x = reinterpret_cast<int32_t*>(w + L.x);
  dv.committed = w + L.committed;
  dv.commit_step = reinterpret_cast<int16_t*>(w + L.commit_step);
  dv.prev_amax = reinterpret_cast<int32_t*>(w + L.prev_amax);
  dv.tokens_out = reinterpret_cast<int32_t*>(w + L.tokens_out);
  dv.commit_steps_out = reinterpret_cast<int16_t*>(w + L.commit_steps_out);
  dv.H = reinterpret_cast<float*>(w + L.H);
  dv.logZ = reinterpret_cast<float*>(w + L.logZ);
  dv.y = reinterpret_cast<int32_t*>(w + L.y);
  dv.amax = reinterpret_cast<int32_t*>(w + L.amax);
  dv.h = reinterpret_cast<uint16_t*>(w + L.h);
  dv.part = reinterpret_cast<dg::Partial*>(w + L.part);
  dv.row_best = reinterpret_cast<unsigned long long*>(w + L.row_best);
  dv.resid_stage = reinterpret_cast<float*>(w + L.resid);
  dv.canvas_rows = reinterpret_cast<uint32_t*>(w + L.canvas_rows);
  dv.rows_ready = reinterpret_cast<uint32_t*>(w + L.sync);
  dv.fin_started = dv.rows_ready + 1;
  dv.slab_done = dv.rows_ready + 2;
  dv.units_done = dv.slab_done + L.rows_cap / 128;
  dv.norm_w = norm_w;
  dv.temps = reinterpret_cast<const float*>(w + L.temps);
  dv.V = cfg->vocab;
  dv.d = cfg->hidden;
  dv.L = cfg->canvas_len;
  dv.B = B;
  dv.G = cfg->gen_blocks;
  dv.N = cfg->num_inference_steps;
  dv.t_min = cfg->t_min;
  dv.t_max = cfg->t_max;
  dv.bound = cfg->entropy_bound;
  dv.reaccept = cfg->mode == DG_REACCEPT;
  dv.stability = cfg->stability;
  dv.conf = cfg->confidence;
  dv.eps = cfg->rms_eps;
  dv.softcap = cfg->softcap;
  dv.inv_softcap = cfg->softcap > 0.f ? 1.f / cfg->softcap : 0.f;
  dv.n_vtiles = L.n_vtiles;
  dv.tiles_per_chunk = L.tiles_per_chunk;
  dv.n_chunks = L.n_chunks;
  dv.n_sub = L.n_sub;
  dv.rows_cap = L.rows_cap;
  dv.max_active = L.max_active;
  dv.chunk_begin = L.chunk_begin;
  dv.chunk_end = L.chunk_end;
  dv.vt_base = L.chunk_begin * L.tiles_per_chunk;
  s->split = cfg->vocab_ranks > 1;
  if (cfg->self_cond) {
    dv.row_scale = reinterpret_cast<float*>(w + L.row_scale);
    dv.row_log2z = reinterpret_cast<float*>(w + L.row_log2z);
    dv.row_canvas = reinterpret_cast<int32_t*>(w + L.row_canvas);
    dv.sc_rows = reinterpret_cast<uint32_t*>(w + L.sc_rows);
    dv.sc_probs = reinterpret_cast<uint16_t*>(w + L.probs);
    dv.sc_part = reinterpret_cast<float*>(w + L.sc_part);
    dv.sc_vpad = L.sc_vpad;
    dv.sc_kc = L.sc_kc;
    dv.sc_kbpc = L.sc_kbpc;
  }

  auto fail = [&](dg_status st) {
    memcpy(g_create_err, s->err, sizeof g_create_err);
    delete s;
    return st;
  };
  if (!encode_2d(&s->tmA, dv.h, (uint64_t)L.rows_cap, (uint64_t)dv.d, dg::kBM, s->err)) return fail(DG_ERR_ARG);
  s->pair = (int64_t)L.max_active * cfg->canvas_len >= 2 * dg::kBM && sms >= 2;
  // W: the whole matrix, or this rank's slice of whole chunks
  const int64_t v_begin = (int64_t)dv.vt_base * dg::kBN;
  const int64_t v_end = std::min<int64_t>((int64_t)L.chunk_end * L.tiles_per_chunk * dg::kBN, dv.V);
  if (!encode_2d(&s->tmB, w_vocab, (uint64_t)(v_end - v_begin), (uint64_t)dv.d, s->pair ? dg::kBN / 2 : dg::kBN,
                 s->err))
    return fail(DG_ERR_ARG);
  cudaError_t ce = dg::lmhead_configure();
  if (ce != cudaSuccess) return fail(cuda_fail(s->err, ce, "configure kernels"));
  if (cfg->self_cond) {
    uint16_t* wt = reinterpret_cast<uint16_t*>(w + L.wt);
    if (!encode_2d(&s->tmP, dv.sc_probs, (uint64_t)L.rows_cap, (uint64_t)L.sc_vpad, dg::kBM, s->err) ||
        !encode_2d(&s->tmWT, wt, (uint64_t)dv.d, (uint64_t)L.sc_vpad, s->pair ? dg::kBN / 2 : dg::kBN, s->err))
      return fail(DG_ERR_ARG);
    ce = dg::selfcond_configure();
    if (ce != cudaSuccess) return fail(cuda_fail(s->err, ce, "configure self-conditioning kernels"));
  }

  std::vector<dg_slot> slots(B);
  for (int c = 0; c < B; ++c) {
    dg_slot& sl = slots[c];
    memset(&sl, 0, sizeof sl);
    sl.seed = s->seeds[c];
    sl.admit_tick = s->admit[c];
    sl.state = dg::kWaiting;
    sl.temperature = cfg->t_max;
  }
  // T_s = t_max + (s/N)(t_min - t_max) for every step: fp64, one IEEE operation at a time
  // (this file is compiled without contraction), rounded once to fp32
  std::vector<float> temps(cfg->num_inference_steps);
  for (int st = 0; st < cfg->num_inference_steps; ++st) {
    const double frac = (double)st / (double)cfg->num_inference_steps;
    const double span = (double)cfg->t_min - (double)cfg->t_max;
    const double prod = frac * span;
    temps[st] = (float)((double)cfg->t_max + prod);
  }
  ce = cudaHostAlloc(reinterpret_cast<void**>(&s->pl_host), sizeof(dg::Plan), cudaHostAllocDefault);
  if (ce != cudaSuccess) return fail(cuda_fail(s->err, ce, "allocate the pinned error latch copy"));
  // the host step's result staging: plan, canvas and entropies lie next to each
  // other in the workspace, and one copy into this buffer brings back all three.
  // Allocated here, so no host step pays for a page-locked allocation.
  {
    const uint8_t* p0 = reinterpret_cast<const uint8_t*>(dv.plan);
    s->stage_x = (size_t)(reinterpret_cast<const uint8_t*>(dv.x) - p0);
    s->stage_H = (size_t)(reinterpret_cast<const uint8_t*>(dv.H) - p0);
    s->stage_bytes = s->stage_H + (size_t)B * cfg->canvas_len * 4;
    ce = cudaHostAlloc(reinterpret_cast<void**>(&s->stage_host), s->stage_bytes, cudaHostAllocDefault);
    if (ce != cudaSuccess) return fail(cuda_fail(s->err, ce, "allocate the pinned result staging"));
  }
  ce = cudaMemsetAsync(workspace, 0, L.total, s->stream);
  s->guards = L.guards;
  for (size_t g : L.guards)
    if (ce == cudaSuccess) ce = cudaMemsetAsync(w + g, kGuardByte, kGuardBytes, s->stream);
  if (ce == cudaSuccess && cfg->self_cond)
    ce = dg::launch_transpose_w(w_vocab, reinterpret_cast<uint16_t*>(w + L.wt), dv.V, dv.d, L.sc_vpad, s->stream);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(dv.slots, slots.data(), sizeof(dg_slot) * B, cudaMemcpyHostToDevice, s->stream);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(w + L.temps, temps.data(), 4 * temps.size(), cudaMemcpyHostToDevice, s->stream);
  if (ce == cudaSuccess) ce = dg::launch_plan(dv, 0, s->stream);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s->stream);
  if (ce != cudaSuccess) return fail(cuda_fail(s->err, ce, "initialise sampler state"));
  *out = s;
  return DG_OK;
}

static dg_status refuse_split(dg_sampler* s) {
  set_err(s->err, "the vocabulary of this sampler is split across ranks: tick with dg_denoise_step_partial, "
                  "exchange the partial records, then dg_denoise_step_finish");
  return DG_ERR_STATE;
}

dg_status dg_denoise_step_partial(dg_sampler* s, const float* resid) {
  NvtxRange nvtx_("dg_denoise_step_partial");
  if (!s) return DG_ERR_ARG;
  if (!resid) return set_err(s->err, "resid is NULL"), DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(resid) % 16) return set_err(s->err, "resid must be 16-byte aligned"), DG_ERR_ALIGN;
  if (s->partial_pending)
    return set_err(s->err, "the previous partial tick has not been finished (dg_denoise_step_finish)"), DG_ERR_STATE;
  dg_status st = tick_front(s, resid);
  if (st == DG_OK) s->partial_pending = true;
  return st;
}

dg_status dg_denoise_step_finish(dg_sampler* s) {
  NvtxRange nvtx_("dg_denoise_step_finish");
  if (!s) return DG_ERR_ARG;
  if (!s->partial_pending) return set_err(s->err, "no partial tick to finish"), DG_ERR_STATE;
  s->partial_pending = false;
  return tick_back(s);
}

dg_status dg_partial_records(const dg_sampler* s, void** records_dev, int32_t* rows_cap, int32_t* n_chunks,
                             int32_t* chunk_begin, int32_t* chunk_end) {
  if (!s) return DG_ERR_ARG;
  if (records_dev) *records_dev = s->dv.part;
  if (rows_cap) *rows_cap = s->dv.rows_cap;
  if (n_chunks) *n_chunks = s->dv.n_sub;
  if (chunk_begin) *chunk_begin = s->dv.chunk_begin;
  if (chunk_end) *chunk_end = s->dv.chunk_end;
  return DG_OK;
}

dg_status dg_vocab_slice(int32_t vocab, int32_t ranks, int32_t rank, int32_t* v_begin, int32_t* v_end) {
  if (vocab < 2 || ranks < 0 || rank < 0 || rank >= (ranks > 1 ? ranks : 1) || !v_begin || !v_end) return DG_ERR_ARG;
  int n_vtiles, tpc, n_chunks, c0, c1;
  vocab_chunking(vocab, &n_vtiles, &tpc, &n_chunks);
  if (ranks > n_chunks) return DG_ERR_ARG;
  rank_chunks(n_chunks, ranks, rank, &c0, &c1);
  *v_begin = c0 * tpc * dg::kBN;
  *v_end = std::min(c1 * tpc * dg::kBN, vocab);
  return DG_OK;
}

dg_status dg_self_condition(dg_sampler* s, float* out) {
  NvtxRange nvtx_("dg_self_condition");
  if (!s) return DG_ERR_ARG;
  if (!out) return set_err(s->err, "out is NULL"), DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(out) % 16) return set_err(s->err, "out must be 16-byte aligned"), DG_ERR_ALIGN;
  if (!s->dv.sc_probs) return set_err(s->err, "the sampler was created without self_cond"), DG_ERR_STATE;
  if (s->partial_pending) return set_err(s->err, "a partial tick is not finished"), DG_ERR_STATE;
  DG_CUDA(s->err,
          dg::launch_selfcond(s->dv, s->pair, &s->tmA, &s->tmB, &s->tmP, &s->tmWT, out, s->num_sms, s->stream),
          "launch self-conditioning");
  return DG_OK;
}

dg_status dg_self_condition_topk(dg_sampler* s, int32_t top_k, float* out) {
  NvtxRange nvtx_("dg_self_condition_topk");
  if (!s) return DG_ERR_ARG;
  if (!out) return set_err(s->err, "out is NULL"), DG_ERR_ARG;
  if (top_k < 1 || top_k > DG_SC_TOPK_MAX)
    return set_err(s->err, "top_k must be in [1, %d] (got %d)", DG_SC_TOPK_MAX, top_k), DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(out) % 16) return set_err(s->err, "out must be 16-byte aligned"), DG_ERR_ALIGN;
  if (!s->dv.sc_probs) return set_err(s->err, "the sampler was created without self_cond"), DG_ERR_STATE;
  if (s->partial_pending) return set_err(s->err, "a partial tick is not finished"), DG_ERR_STATE;
  DG_CUDA(s->err,
          dg::launch_selfcond_topk(s->dv, s->pair, &s->tmA, &s->tmB, s->w_vocab, top_k, out, s->num_sms, s->stream),
          "launch top-K self-conditioning");
  return DG_OK;
}

dg_status dg_denoise_step(dg_sampler* s, const float* resid) {
  NvtxRange nvtx_("dg_denoise_step");
  if (!s) return DG_ERR_ARG;
  if (s->split) return refuse_split(s);
  if (!resid) return set_err(s->err, "resid is NULL"), DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(resid) % 16) return set_err(s->err, "resid must be 16-byte aligned"), DG_ERR_ALIGN;
  return tick(s, resid);
}

dg_status dg_denoise_step_host(dg_sampler* s, const float* resid_host, int32_t* canvas_host, float* entropy_host) {
  NvtxRange nvtx_("dg_denoise_step_host");
  if (!s) return DG_ERR_ARG;
  if (s->split) return refuse_split(s);
  if (!resid_host) return set_err(s->err, "resid_host is NULL"), DG_ERR_ARG;
  const size_t BL = (size_t)s->dv.B * s->dv.L;
  // Page-locked input mapped into the device's address space is read by the
  // RMSNorm straight from host memory (zero-copy: the rows cross the host link
  // once, while the LM head sets up); anything else is copied into the workspace.
  const float* resid = s->dv.resid_stage;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, resid_host) == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer &&
      reinterpret_cast<uintptr_t>(pa.devicePointer) % 16 == 0) {
    resid = static_cast<const float*>(pa.devicePointer);
  } else {
    (void)cudaGetLastError();  // an unregistered pointer is not an error
    DG_CUDA(s->err,
            cudaMemcpyAsync(s->dv.resid_stage, resid_host, BL * s->dv.d * sizeof(float), cudaMemcpyHostToDevice,
                            s->stream),
            "copy resid to device");
  }
  dg_status st = tick(s, resid);
  if (st != DG_OK) return st;
  if (!canvas_host && !entropy_host) return check_device_error(s);
  // plan, canvas and entropies in one copy into the pinned staging buffer
  DG_CUDA(s->err, cudaMemcpyAsync(s->stage_host, s->dv.plan, s->stage_bytes, cudaMemcpyDeviceToHost, s->stream),
          "copy results");
  DG_CUDA(s->err, cudaStreamSynchronize(s->stream), "synchronize");
  if (canvas_host) memcpy(canvas_host, s->stage_host + s->stage_x, BL * 4);
  if (entropy_host) memcpy(entropy_host, s->stage_host + s->stage_H, BL * 4);
  return latched_status(s, *reinterpret_cast<const dg::Plan*>(s->stage_host));
}

dg_status dg_set_timing_events(dg_sampler* s, void* const* events) {
  if (!s) return DG_ERR_ARG;
  s->timed = events != nullptr;
  if (events)
    for (int i = 0; i < 4; ++i) {
      if (!events[i]) return s->timed = false, set_err(s->err, "timing event %d is NULL", i), DG_ERR_ARG;
      s->timing[i] = static_cast<cudaEvent_t>(events[i]);
    }
  return DG_OK;
}

dg_status dg_sync_info(dg_sampler* s, dg_slot* slots_host) {
  if (!s || !slots_host) return DG_ERR_ARG;
  DG_CUDA(s->err,
          cudaMemcpyAsync(slots_host, s->dv.slots, sizeof(dg_slot) * s->dv.B, cudaMemcpyDeviceToHost, s->stream),
          "copy slots");
  return check_device_error(s);
}

dg_status dg_run(dg_sampler* s, dg_resid_fn fn, void* user, float* resid_dev, int32_t* tokens_host,
                 dg_slot* slots_host) {
  NvtxRange nvtx_("dg_run");
  if (!s || !fn) return DG_ERR_ARG;
  if (s->split) return refuse_split(s);
  float* resid = resid_dev ? resid_dev : s->dv.resid_stage;
  if (reinterpret_cast<uintptr_t>(resid) % 16) return set_err(s->err, "resid_dev must be 16-byte aligned"), DG_ERR_ALIGN;
  std::vector<dg_slot> sl(s->dv.B);
  for (;;) {
    for (int i = 0; i < s->dv.N && s->host_tick < s->tick_bound; ++i) {
      if (fn(user, (int32_t)s->host_tick, s->dv.x, s->dv.slots, resid, reinterpret_cast<dg_stream_t>(s->stream)) != 0)
        return set_err(s->err, "residual callback failed at tick %lld", (long long)s->host_tick), DG_ERR_ARG;
      dg_status st = tick(s, resid);
      if (st != DG_OK) return st;
    }
    dg_status st = dg_sync_info(s, sl.data());
    if (st != DG_OK) return st;
    bool done = true;
    for (const dg_slot& x : sl) done = done && x.state == dg::kDone;
    if (done || s->host_tick >= s->tick_bound) break;
  }
  if (tokens_host)
    DG_CUDA(s->err,
            cudaMemcpyAsync(tokens_host, s->dv.tokens_out, sizeof(int32_t) * s->dv.B * s->dv.G * s->dv.L,
                            cudaMemcpyDeviceToHost, s->stream),
            "copy tokens");
  if (slots_host) memcpy(slots_host, sl.data(), sizeof(dg_slot) * s->dv.B);
  return check_device_error(s);
}

dg_status dg_get_state(dg_sampler* s, dg_state* h) {
  if (!s || !h) return DG_ERR_ARG;
  const size_t B = s->dv.B, BL = B * s->dv.L;
  dg::Plan pl;
  struct {
    void* dst;
    const void* src;
    size_t n;
  } cp[] = {{h->slots, s->dv.slots, sizeof(dg_slot) * B},    {h->tokens, s->dv.x, 4 * BL},
            {h->committed, s->dv.committed, BL},             {h->commit_step, s->dv.commit_step, 2 * BL},
            {h->prev_argmax, s->dv.prev_amax, 4 * BL},       {h->tokens_out, s->dv.tokens_out, 4 * BL * s->dv.G},
            {h->commit_steps_out, s->dv.commit_steps_out, 2 * BL * s->dv.G},
            {&pl, s->dv.plan, sizeof pl}};
  for (auto& c : cp)
    if (c.dst) DG_CUDA(s->err, cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyDeviceToHost, s->stream), "copy state");
  DG_CUDA(s->err, cudaStreamSynchronize(s->stream), "synchronize");
  h->tick = pl.tick;
  return check_device_error(s);
}

dg_status dg_set_state(dg_sampler* s, const dg_state* h) {
  NvtxRange nvtx_("dg_set_state");
  if (!s || !h || !h->slots || !h->tokens || !h->committed || !h->commit_step || !h->prev_argmax)
    return DG_ERR_ARG;
  if (h->tick < 0) return set_err(s->err, "tick must be >= 0"), DG_ERR_ARG;
  const size_t B = s->dv.B, BL = B * s->dv.L;
  std::vector<dg_slot> sl(h->slots, h->slots + B);
  int active = 0;
  for (size_t c = 0; c < B; ++c) {
    sl[c].seed = s->seeds[c];
    sl[c].admit_tick = s->admit[c];
    if (sl[c].state < dg::kWaiting || sl[c].state > dg::kDone || sl[c].block < 0 || sl[c].block >= s->dv.G ||
        sl[c].step < 0 || sl[c].step >= s->dv.N)
      return set_err(s->err, "slot %zu holds an invalid state/block/step", c), DG_ERR_ARG;
    active += sl[c].state == dg::kActive;
  }
  if (active > s->dv.max_active) return set_err(s->err, "more active canvases than max_active"), DG_ERR_ARG;
  for (size_t i = 0; i < BL; ++i)
    if (h->tokens[i] < 0 || h->tokens[i] >= s->dv.V) return set_err(s->err, "token out of range"), DG_ERR_ARG;
  struct {
    void* dst;
    const void* src;
    size_t n;
  } cp[] = {{s->dv.slots, sl.data(), sizeof(dg_slot) * B},  {s->dv.x, h->tokens, 4 * BL},
            {s->dv.committed, h->committed, BL},            {s->dv.commit_step, h->commit_step, 2 * BL},
            {s->dv.prev_amax, h->prev_argmax, 4 * BL},      {s->dv.tokens_out, h->tokens_out, 4 * BL * s->dv.G},
            {s->dv.commit_steps_out, h->commit_steps_out, 2 * BL * s->dv.G}};
  for (auto& c : cp)
    if (c.src) DG_CUDA(s->err, cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, s->stream), "copy state");
  DG_CUDA(s->err, dg::launch_plan(s->dv, h->tick, s->stream), "launch plan");
  DG_CUDA(s->err, cudaStreamSynchronize(s->stream), "synchronize");
  s->host_tick = h->tick;
  s->partial_pending = false;  // a partial tick of the replaced state is dropped
  int32_t max_admit = 0;
  for (int32_t a : s->admit) max_admit = a > max_admit ? a : max_admit;
  s->tick_bound = (int64_t)(h->tick > max_admit ? h->tick : max_admit) +
                  (int64_t)s->dv.G * s->dv.N * (int64_t)s->dv.B;
  return DG_OK;
}

void dg_destroy(dg_sampler* s) {
  if (!s) return;
  cudaStreamSynchronize(s->stream);
  delete s;
}

dg_status dg_debug_fail_cuda_call(int32_t after) {
  if (after < -1) return DG_ERR_ARG;
  g_fail_after.store(after);
  return DG_OK;
}

dg_status dg_debug_hold_slabs(dg_sampler* s, int on) {
  if (!s) return DG_ERR_ARG;
  s->dv.hold_slabs = on ? 1 : 0;
  return DG_OK;
}

const int32_t* dg_canvas(const dg_sampler* s) { return s ? s->dv.x : nullptr; }
const uint8_t* dg_committed(const dg_sampler* s) { return s ? s->dv.committed : nullptr; }
const int16_t* dg_commit_step(const dg_sampler* s) { return s ? s->dv.commit_step : nullptr; }
const float* dg_entropy(const dg_sampler* s) { return s ? s->dv.H : nullptr; }
const float* dg_logz(const dg_sampler* s) { return s ? s->dv.logZ : nullptr; }
const int32_t* dg_sample(const dg_sampler* s) { return s ? s->dv.y : nullptr; }
const int32_t* dg_argmax(const dg_sampler* s) { return s ? s->dv.amax : nullptr; }
const int32_t* dg_tokens_out(const dg_sampler* s) { return s ? s->dv.tokens_out : nullptr; }
const int16_t* dg_commit_steps_out(const dg_sampler* s) { return s ? s->dv.commit_steps_out : nullptr; }
const dg_slot* dg_slots(const dg_sampler* s) { return s ? s->dv.slots : nullptr; }
const uint16_t* dg_normed(const dg_sampler* s) { return s ? s->dv.h : nullptr; }

dg_status dg_debug_check(dg_sampler* s, uint64_t* first_bad) {
  if (!s) return DG_ERR_ARG;
  if (first_bad) *first_bad = 0;
#ifndef DG_DEBUG_CHECKS
  set_err(s->err, "this library was built without DG_DEBUG_CHECKS");
  return DG_ERR_UNSUPPORTED;
#else
  std::vector<unsigned char> host(s->guards.size() * kGuardBytes);
  for (size_t i = 0; i < s->guards.size(); ++i)
    DG_CUDA(s->err,
            cudaMemcpyAsync(host.data() + i * kGuardBytes, static_cast<uint8_t*>(s->ws) + s->guards[i], kGuardBytes,
                            cudaMemcpyDeviceToHost, s->stream),
            "copy guards");
  dg_status st = check_device_error(s);  // synchronizes the copies too
  if (st != DG_OK) return st;
  for (size_t i = 0; i < host.size(); ++i)
    if (host[i] != kGuardByte) {
      const uint64_t off = s->guards[i / kGuardBytes] + i % kGuardBytes;
      if (first_bad) *first_bad = off;
      set_err(s->err, "workspace guard damaged at offset %llu", (unsigned long long)off);
      return DG_ERR_BOUNDS;
    }
  return DG_OK;
#endif
}

const char* dg_status_string(dg_status st) {
  switch (st) {
    case DG_OK: return "DG_OK";
    case DG_ERR_ARG: return "DG_ERR_ARG";
    case DG_ERR_ALIGN: return "DG_ERR_ALIGN";
    case DG_ERR_WORKSPACE: return "DG_ERR_WORKSPACE";
    case DG_ERR_CUDA: return "DG_ERR_CUDA";
    case DG_ERR_STATE: return "DG_ERR_STATE";
    case DG_ERR_NONFINITE: return "DG_ERR_NONFINITE";
    case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED";
    case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT";
    case DG_ERR_BOUNDS: return "DG_ERR_BOUNDS";
  }
  return "unknown dg_status";
}

const char* dg_last_error(const dg_sampler* s) { return s ? s->err : g_create_err; }

}  // extern "C"
