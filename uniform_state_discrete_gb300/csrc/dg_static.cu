// dg_lmhead_stats_static: the LM-head statistics of one canvas (RMSNorm, tied
// LM head, temperature softmax entropy / log Z / argmax, Gumbel-max sample)
// computed without allocating any device memory.
//
// The sampler's entry points take a caller-allocated workspace.  This one is
// for callers that cannot hand one over: programs that reserve the whole
// device for their own memory pool at start-up (so a later cudaMalloc fails),
// and code running where cudaMalloc is not allowed or would stall the device,
// such as allocator callbacks.  Its scratch -- the normalised rows, the
// split-vocabulary partial records and the rows' best Gumbel scores -- lives in
// one fixed-size array in device global memory, declared below, which every
// GPU that loads this library holds until the process exits.  The call waits
// for its stream before it returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "dg_internal.cuh"

namespace {

// Layout of the static scratch: per-call canvas state the kernels read, then
// the normalised rows (bf16 [256, 4096] at most), then the partial records
// ([256 rows, at most kChunkTarget chunks]).
constexpr size_t kOffSlot = 0;
constexpr size_t kOffPlan = 256;
constexpr size_t kOffActive = 512;
constexpr size_t kOffSync = 768;  // rows written by RMSNorm, (unused here), LM-head units per 128-row slab (2), units done
constexpr size_t kOffH = 1024;
constexpr size_t kBytesH = (size_t)2 * DG_STATIC_MAX_ROWS * DG_STATIC_MAX_HIDDEN;
constexpr size_t kOffPart = kOffH + kBytesH;
constexpr size_t kBytesPart = sizeof(dg::Partial) * DG_STATIC_MAX_ROWS * dg::kChunkTarget;
constexpr size_t kOffRowBest = kOffPart + kBytesPart;
constexpr size_t kBytesRowBest = sizeof(unsigned long long) * DG_STATIC_MAX_ROWS;
constexpr size_t kStaticBytes = (kOffRowBest + kBytesRowBest + 255) & ~size_t(255);
static_assert(sizeof(dg_slot) <= 256 && sizeof(dg::Plan) <= 256, "scratch header fits");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  bool ready;
  unsigned char* base;  // device address of g_static_scratch on this device
  int num_sms;
  PFN_cuTensorMapEncodeTiled_v12000 encode;  // the driver's tensor-map encoder
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;  // guards g_setup: every call reads its device's entry under it

void put_err(char* buf, size_t len, const char* fmt, ...) {
  if (!buf || len == 0) return;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, len, fmt, ap);
  va_end(ap);
}

// Writes this call's canvas state and clears the error latch: the kernels read
// one active canvas (id 0) at the given seed, block, step and temperature.
__global__ void k_static_prep(unsigned char* base, uint64_t seed, int block, int step, float T) {
  if (threadIdx.x != 0) return;
  dg_slot* sl = reinterpret_cast<dg_slot*>(base + kOffSlot);
  dg::Plan* pl = reinterpret_cast<dg::Plan*>(base + kOffPlan);
  int32_t* active = reinterpret_cast<int32_t*>(base + kOffActive);
  sl->seed = seed;
  sl->admit_tick = 0;
  sl->state = dg::kActive;
  sl->block = block;
  sl->step = step;
  sl->n_committed = 0;
  sl->steps_used = 0;
  sl->converged_blocks = 0;
  sl->temperature = T;
  sl->mean_entropy = 0.f;
  sl->n_remasked = 0;
  sl->stable_steps = 0;
  pl->tick = 0;
  pl->n_active = 1;
  pl->epoch += 1u;  // the per-row best scores of earlier calls no longer count
  pl->commits = 0u;
  pl->err = dg::kErrNone;
  for (int i = 0; i < 4; ++i) pl->err_info[i] = 0;
  active[0] = 0;
  uint32_t* sync = reinterpret_cast<uint32_t*>(base + kOffSync);
  for (int i = 0; i < 5; ++i) sync[i] = 0u;  // rows_ready, fin_started, slab_done[2], units_done
}

// One warp per position: merge its split-vocabulary partial records into the
// entropy (nats), log Z, sampled token and argmax written to the caller's
// arrays (same arithmetic as the sampler's finishing kernel).
__global__ void __launch_bounds__(256) k_static_combine(const dg::Dev dv, int rows, float* H, float* logZ,
                                                        int32_t* y, int32_t* amax) {
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  dg::Partial acc = dg::empty_partial();
  const dg::Partial* src = dv.part + (size_t)row * dv.n_sub;
  for (int i = lane; i < dv.n_sub; i += 32) acc = dg::merge_partial(acc, src[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dg::Partial b;
    b.m = __shfl_xor_sync(0xFFFFFFFFu, acc.m, o);
    b.S = __shfl_xor_sync(0xFFFFFFFFu, acc.S, o);
    b.A = __shfl_xor_sync(0xFFFFFFFFu, acc.A, o);
    b.g = __shfl_xor_sync(0xFFFFFFFFu, acc.g, o);
    b.amax = __shfl_xor_sync(0xFFFFFFFFu, acc.amax, o);
    b.gidx = __shfl_xor_sync(0xFFFFFFFFu, acc.gidx, o);
    b.pad0 = b.pad1 = 0;
    acc = dg::merge_partial(acc, b);
  }
  if (lane == 0) {
    const float l2S = log2f(acc.S);
    const float h = 0.69314718055994531f * (l2S - acc.A / acc.S);
    const float lz = 0.69314718055994531f * (acc.m + l2S);
    H[row] = h > 0.f ? h : 0.f;
    logZ[row] = lz;
    const bool y_ok = acc.gidx >= 0 && acc.gidx < dv.V, a_ok = acc.amax >= 0 && acc.amax < dv.V;
    y[row] = y_ok ? acc.gidx : 0;  // never an out-of-range token, even on the error path
    amax[row] = a_ok ? acc.amax : 0;
    if (!isfinite(h) || !isfinite(lz) || !isfinite(acc.g) || !y_ok || !a_ok) {
      if (atomicCAS(&dv.plan->err, dg::kErrNone, dg::kErrNonFinite) == dg::kErrNone) dv.plan->err_info[1] = row;
    }
  }
}

bool encode(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
            uint32_t box_rows, char* err, size_t err_len) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)dg::kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  if (fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    put_err(err, err_len, "cuTensorMapEncodeTiled failed for a [%llu x %llu] matrix", (unsigned long long)rows,
            (unsigned long long)cols);
    return false;
  }
  return true;
}

dg_status cuda_err(cudaError_t e, const char* what, char* err, size_t err_len) {
  put_err(err, err_len, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return DG_ERR_CUDA;
}

}  // namespace

extern "C" dg_status dg_lmhead_stats_static(const float* resid, int32_t rows, const void* w_vocab, int32_t vocab,
                                            int32_t hidden, const float* norm_w, float rms_eps, float temperature,
                                            uint64_t seed, int32_t block, int32_t step, float* entropy, float* logz,
                                            int32_t* sample, int32_t* argmax, dg_stream_t stream, char* err,
                                            size_t err_len) {
  if (err && err_len) err[0] = 0;
  // sizes first, before any CUDA call
  if (rows < 1 || rows > DG_STATIC_MAX_ROWS) {
    put_err(err, err_len, "rows must be in [1, %d] (got %d): the static scratch holds at most %d positions",
            DG_STATIC_MAX_ROWS, rows, DG_STATIC_MAX_ROWS);
    return DG_ERR_ARG;
  }
  if (hidden < 8 || hidden > DG_STATIC_MAX_HIDDEN || hidden % 8) {
    put_err(err, err_len, "hidden must be a multiple of 8 in [8, %d] (got %d): the static scratch holds %d columns",
            DG_STATIC_MAX_HIDDEN, hidden, DG_STATIC_MAX_HIDDEN);
    return DG_ERR_ARG;
  }
  if (vocab < 2) return put_err(err, err_len, "vocab must be >= 2 (got %d)", vocab), DG_ERR_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !(rms_eps >= 0.f) || !std::isfinite(rms_eps) ||
      block < 0 || block > 65535 || step < 0 || step > 65535)
    return put_err(err, err_len, "temperature must be finite and > 0, rms_eps finite and >= 0, block and step in "
                   "[0, 65535]"), DG_ERR_ARG;
  if (!resid || !w_vocab || !entropy || !logz || !sample || !argmax)
    return put_err(err, err_len, "resid, w_vocab and the four output arrays must not be NULL"), DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(resid) % 16 || reinterpret_cast<uintptr_t>(w_vocab) % 16 ||
      (norm_w && reinterpret_cast<uintptr_t>(norm_w) % 16))
    return put_err(err, err_len, "resid, w_vocab and norm_w must be 16-byte aligned"), DG_ERR_ALIGN;

  // once per device, with that device current: the scratch array's device address
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_err(e, "query device", err, err_len);
  if (dev < 0 || dev >= kMaxDevices) return put_err(err, err_len, "device %d out of range", dev), DG_ERR_UNSUPPORTED;
  DeviceSetup su;
  try {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_setup[dev].ready) {
      int major = 0, minor = 0, sms = 0;
      e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_err(e, "query device", err, err_len);
      if (major != 10 || minor != 3) {
        put_err(err, err_len, "this library is built for sm_103a (GB300); device is sm_%d%d", major, minor);
        return DG_ERR_UNSUPPORTED;
      }
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_scratch);
      if (e != cudaSuccess || !ptr) return cuda_err(e, "cudaGetSymbolAddress of the static scratch", err, err_len);
      e = dg::lmhead_configure();
      if (e != cudaSuccess) return cuda_err(e, "configure kernels", err, err_len);
      void* enc = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &enc, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !enc) {
        put_err(err, err_len, "cuTensorMapEncodeTiled not available from the driver");
        return DG_ERR_CUDA;
      }
      g_setup[dev].encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(enc);
      g_setup[dev].base = static_cast<unsigned char*>(ptr);
      g_setup[dev].num_sms = sms;
      g_setup[dev].ready = true;
    }
    su = g_setup[dev];
  } catch (...) {
    put_err(err, err_len, "could not take the set-up lock");
    return DG_ERR_CUDA;
  }

  // the same vocabulary chunking as the sampler (it depends on V only)
  const int n_vtiles = (vocab + dg::kBN - 1) / dg::kBN;
  const int target = n_vtiles < dg::kChunkTarget ? n_vtiles : dg::kChunkTarget;
  const int tpc = (n_vtiles + target - 1) / target;
  const int n_chunks = (n_vtiles + tpc - 1) / tpc;

  dg::Dev dv = {};
  dv.slots = reinterpret_cast<dg_slot*>(su.base + kOffSlot);
  dv.plan = reinterpret_cast<dg::Plan*>(su.base + kOffPlan);
  dv.active = reinterpret_cast<int32_t*>(su.base + kOffActive);
  dv.rows_ready = reinterpret_cast<uint32_t*>(su.base + kOffSync);
  dv.fin_started = dv.rows_ready + 1;
  dv.slab_done = dv.rows_ready + 2;
  dv.units_done = dv.slab_done + 2;
  dv.h = reinterpret_cast<uint16_t*>(su.base + kOffH);
  dv.part = reinterpret_cast<dg::Partial*>(su.base + kOffPart);
  dv.row_best = reinterpret_cast<unsigned long long*>(su.base + kOffRowBest);
  dv.norm_w = norm_w;
  dv.V = vocab;
  dv.d = hidden;
  dv.L = rows;
  dv.B = 1;
  dv.G = 1;
  dv.N = 1;
  dv.t_min = temperature;
  dv.t_max = temperature;
  dv.eps = rms_eps;
  dv.n_vtiles = n_vtiles;
  dv.tiles_per_chunk = tpc;
  dv.n_chunks = n_chunks;
  dv.n_sub = n_chunks * dg::kSubPerChunk;
  dv.chunk_begin = 0;
  dv.chunk_end = n_chunks;
  dv.vt_base = 0;
  dv.rows_cap = DG_STATIC_MAX_ROWS;
  dv.max_active = 1;

  // the pair kernel when the rows fill a 256-row pair tile, as the sampler chooses
  const bool pair = rows >= 2 * dg::kBM && su.num_sms >= 2;
  CUtensorMap tmA, tmB;
  if (!encode(su.encode, &tmA, dv.h, (uint64_t)DG_STATIC_MAX_ROWS, (uint64_t)hidden, dg::kBM, err, err_len))
    return DG_ERR_ARG;
  if (!encode(su.encode, &tmB, w_vocab, (uint64_t)vocab, (uint64_t)hidden, pair ? dg::kBN / 2 : dg::kBN, err,
              err_len))
    return DG_ERR_ARG;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  k_static_prep<<<1, 32, 0, st>>>(su.base, seed, (int)block, (int)step, temperature);
  e = cudaGetLastError();
  if (e == cudaSuccess && !pair) e = dg::launch_rmsnorm(dv, resid, st);  // the pair kernel forms its rows itself
  if (e == cudaSuccess)
    e = pair ? dg::launch_lmhead_pair(dv, resid, &tmA, &tmB, su.num_sms, st)
             : dg::launch_lmhead(dv, &tmA, &tmB, su.num_sms, st);
  if (e == cudaSuccess) {
    k_static_combine<<<(rows + 7) / 8, 256, 0, st>>>(dv, rows, entropy, logz, sample, argmax);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return cuda_err(e, "launch", err, err_len);
  // the error latch comes back on the caller's stream, so no other stream is waited for
  dg::Plan pl;
  e = cudaMemcpyAsync(&pl, dv.plan, sizeof pl, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_err(e, "read the error latch", err, err_len);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_err(e, "synchronize", err, err_len);
  if (pl.err == dg::kErrNonFinite) {
    put_err(err, err_len, "non-finite logit statistics at row %d", pl.err_info[1]);
    return DG_ERR_NONFINITE;
  }
  if (pl.err == dg::kErrTimeout) {
    put_err(err, err_len, "a bounded wait expired: %s (CTA %d, detail %d)", dg::wait_site_name(pl.err_info[2]),
            pl.err_info[0], pl.err_info[3]);
    return DG_ERR_TIMEOUT;
  }
  if (pl.err == dg::kErrBounds) {
    put_err(err, err_len, "a debug index check failed at site %d (value %d)", pl.err_info[2], pl.err_info[3]);
    return DG_ERR_BOUNDS;
  }
  return DG_OK;
}
