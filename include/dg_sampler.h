/*
 * dg_sampler.h -- C ABI of the GB300 (sm_103a) denoise-step library for the
 * uniform-state discrete-diffusion sampler of DiffusionGemma.
 *
 * One denoising step ("tick") runs, for every active canvas:
 *   1. the final RMSNorm of the residual stream, w * x * sqrt(D) / (||x||_2 + eps),
 *      cast to bf16                 ("The Annotated DiffusionGemma", "RMSNorm")
 *   2. the tied LM head z = h W_vocab^T, fp32 accumulate, never stored, with an
 *      optional final logit softcap c tanh(z / c)
 *                                   (same page, "Complete DiffusionGemma model",
 *                                    "Logit Softcapping")
 *   3. softmax(z / T) with the per-position entropy H (nats), log Z, the argmax
 *      and one sampled token        (same page, "Apply temperature", "Compute
 *                                    entropy")
 *   4. the entropy-bounded commit: the open positions sorted by entropy, the
 *      prefix whose exclusive entropy sum stays <= entropy_bound takes its
 *      sampled tokens and, under DG_FREEZE, freezes (dg_mode)
 *                                   (same page, "Keep a low-entropy prefix and
 *                                    renoise the rest"; ComfyUI-DiffusionGemma,
 *                                    "What it is")
 *   5. the early-stop test (mean H < confidence and an unchanged argmax canvas)
 *      and the uniform re-noise of every position still uncommitted
 *                                   (same page, "Check for early stopping")
 * with the temperature cooling T_s = t_max + (s/N)(t_min - t_max), s = 0..N-1
 * ("Apply temperature"; DiffusionGemma Denoise node, "Inputs": t_min / t_max).
 *
 * Conventions for every entry point:
 *   - "dev" pointers are CUDA device pointers, "host" pointers host memory.
 *   - The library never allocates device memory.  The caller allocates one
 *     workspace of dg_workspace_size() bytes and keeps it alive until
 *     dg_destroy().  Device buffers passed in are borrowed, not owned.  A
 *     sampler holds two small page-locked host buffers of its own (the error
 *     latch read-back and the result staging of dg_denoise_step_host), both
 *     made by dg_sampler_create() and freed by dg_destroy().
 *   - Work is enqueued on the stream given to dg_sampler_create().  Calls
 *     marked "asynchronous" return before the GPU work ends; calls marked
 *     "synchronizing" wait for the stream.
 *   - Errors are returned as dg_status; no C++ exception crosses the ABI.  A
 *     failed call leaves a message readable by dg_last_error().  A device-side
 *     fault condition found by a kernel (non-finite logits, a bounded wait that
 *     ran out) is latched on the device and reported by the next synchronizing
 *     call.
 *   - A sampler is not thread-safe; distinct samplers are independent.
 */
#ifndef DG_SAMPLER_H
#define DG_SAMPLER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  NULL selects the legacy default stream. */
typedef struct CUstream_st* dg_stream_t;

typedef enum dg_status {
  DG_OK = 0,
  DG_ERR_ARG = 1,         /* an argument or config field is out of range          */
  DG_ERR_ALIGN = 2,       /* a pointer lacks the alignment the kernels need        */
  DG_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than dg_workspace_size()    */
  DG_ERR_CUDA = 4,        /* a CUDA runtime call failed (message in dg_last_error) */
  DG_ERR_STATE = 5,       /* call not valid in the sampler's state (e.g. all done) */
  DG_ERR_NONFINITE = 6,   /* a kernel met a non-finite logit statistic             */
  DG_ERR_UNSUPPORTED = 7, /* a valid request this build does not implement         */
  DG_ERR_TIMEOUT = 8,     /* a kernel's bounded wait ran out (pipeline stalled)    */
  DG_ERR_BOUNDS = 9       /* debug build: an index check failed, the access was
                             skipped (dg_debug_check)                             */
} dg_status;

/* Commit semantics.
 * DG_FREEZE: a committed position keeps its token for the rest of the block
 *   and only uncommitted positions enter each step's sort
 *   (ComfyUI-DiffusionGemma, "What it is": confident positions freeze).
 * DG_REACCEPT: every step sorts all positions of the canvas afresh and accepts
 *   the low-entropy prefix; accepted positions take this step's sample and all
 *   others, including positions accepted at earlier steps, are re-noised (The
 *   Annotated DiffusionGemma, "Keep a low-entropy prefix and renoise the rest"
 *   and its "Denoise, stage, commit, and generate" code).  The committed mask
 *   is then the set accepted at the latest step, commit_step the last step a
 *   position was accepted, and the slot's n_remasked the positions accepted at
 *   the previous step and re-noised at the latest one.  At the final step
 *   every position takes its sample in both modes. */
typedef enum dg_mode { DG_FREEZE = 0, DG_REACCEPT = 1 } dg_mode;

/*
 * Sampler configuration.  Field names follow the pages' knobs (DiffusionGemma
 * Denoise node, "Inputs (11)"; TensorSharp DiffusionGemma doc, "3. Sampler
 * contract"); defaults there: num_inference_steps 48, t_min 0.4, t_max 0.8,
 * entropy_bound 0.1 nats, confidence 0.005, canvas length 256, stability 1.
 */
typedef struct dg_config {
  int32_t vocab;               /* V >= 2 (the pages' model: 2^18)                                */
  int32_t hidden;              /* d, a multiple of 8 (16-byte rows for TMA), <= 16384            */
  int32_t canvas_len;          /* L positions per canvas, 1..1024 (pages: 256)                  */
  int32_t n_canvases;          /* B >= 1 independent canvases                                    */
  int32_t gen_blocks;          /* blocks per canvas, denoised one after another, >= 1           */
  int32_t num_inference_steps; /* N, 1..1024: steps per block                                   */
  float t_min;                 /* cold temperature endpoint, > 0                                 */
  float t_max;                 /* hot temperature endpoint (step 0), > 0                         */
  float entropy_bound;         /* per-step acceptance budget in nats, >= 0                       */
  float confidence;            /* early stop when mean H (nats) falls below this, >= 0           */
  int32_t stability;           /* k, 1..1024: the early stop also needs the argmax canvas equal
                                  to each of the k previous steps' (the pages use 1)             */
  float rms_eps;               /* RMSNorm epsilon, added to ||x||_2, >= 0                        */
  int32_t mode;                /* dg_mode: DG_FREEZE or DG_REACCEPT                              */
  int32_t max_active;          /* most canvases active in one tick, 1..B (0 = B); sizes buffers  */
  const uint64_t* seeds;       /* host [B]: per-canvas Philox key; NULL = seed c for canvas c    */
  const int32_t* admit_tick;   /* host [B]: tick at which canvas c joins, >= 0; NULL = all at 0  */
  float softcap;               /* final logit softcap c >= 0: logits become c tanh(z / c) before
                                  the temperature (The Annotated DiffusionGemma, "Logit
                                  Softcapping"); 0 = off                                        */
  int32_t vocab_ranks;         /* G: ranks the vocabulary is split across, 0 or 1 = not split;
                                  at most the number of vocabulary chunks (see
                                  dg_denoise_step_partial)                                       */
  int32_t vocab_rank;          /* this sampler's rank r in [0, G)                                */
  int32_t self_cond;           /* 1: also hold what dg_self_condition needs (a transposed copy of
                                  W and a bf16 [rows, V] buffer for the probabilities); 0: off.
                                  Not with vocab_ranks > 1                                        */
} dg_config;

/* Per-canvas state, the layout of the device array returned by dg_slots().
 * state: 0 waiting for admission, 1 active, 2 done (all blocks finished). */
typedef struct dg_slot {
  uint64_t seed;
  int32_t admit_tick;
  int32_t state;
  int32_t block;            /* current block (gen_blocks - 1 after the last one)      */
  int32_t step;             /* step of the current block the next tick runs           */
  int32_t n_committed;      /* committed positions of the current block (DG_REACCEPT:
                               positions accepted at the latest step)                 */
  int32_t steps_used;       /* steps run over all finished blocks                     */
  int32_t converged_blocks; /* blocks ended by the early-stop test                    */
  float temperature;        /* T the next tick applies to this canvas                 */
  float mean_entropy;       /* mean H (nats) over the canvas at its last tick         */
  int32_t n_remasked;       /* DG_REACCEPT: positions accepted at the previous step and
                               re-noised at the latest one; 0 under DG_FREEZE          */
  int32_t stable_steps;     /* consecutive latest steps whose argmax canvas equalled the
                               one before (reset at each block start)                  */
} dg_slot;

typedef struct dg_sampler dg_sampler;

/* Bytes of device workspace a sampler with this config needs; 0 if the
 * config is invalid (dg_sampler_create then reports why). */
size_t dg_workspace_size(const dg_config* cfg);

/*
 * Create a sampler.  Synchronizing.
 *   w_vocab   dev, bf16 [V, d] row-major, 16-byte aligned: the tied embedding /
 *             LM-head matrix.  Borrowed; must stay valid and unchanged.
 *   norm_w    dev, fp32 [d]: RMSNorm weight, or NULL for all ones.  Borrowed.
 *   workspace dev, >= dg_workspace_size(cfg) bytes, 256-byte aligned.  Borrowed.
 *   stream    stream all later work of this sampler is enqueued on.
 * Canvases whose admit_tick is 0 receive their uniform initial canvas.
 */
dg_status dg_sampler_create(const dg_config* cfg, const void* w_vocab, const float* norm_w, void* workspace,
                            size_t ws_bytes, dg_stream_t stream, dg_sampler** out);

/*
 * Run one tick (steps 1-5 above) for every active canvas.  Asynchronous: no
 * host synchronization inside, so a tick can be captured in a CUDA graph.
 *   resid  dev, fp32 [B, L, d]: the residual stream entering the final norm;
 *          rows of canvases not active this tick are not read.
 * Returns DG_ERR_STATE when the host can tell every canvas has finished.
 */
dg_status dg_denoise_step(dg_sampler* s, const float* resid);

/*
 * The same tick from host memory.  Synchronizing.  resid_host (fp32 [B, L, d])
 * in page-locked memory mapped into the device's address space (cudaHostAlloc,
 * cudaHostRegister, torch pin_memory) is read by the kernels directly; other
 * host memory is first copied into the workspace.  The call runs the tick,
 * copies back the canvas after the tick (int32 [B, L], nullable) and this
 * tick's entropies (fp32 [B, L], nullable) in one copy, and waits once for the
 * stream; resid_host must stay unchanged until it returns.
 */
dg_status dg_denoise_step_host(dg_sampler* s, const float* resid_host, int32_t* canvas_host, float* entropy_host);

/*
 * Vocabulary-parallel ticks.  The LM head cuts the vocabulary into chunks of
 * whole 256-entry tiles (the chunking depends on V only) and writes one 32-byte
 * partial record of softmax statistics and Gumbel-max candidate per position
 * and chunk; the finishing step merges a position's records in chunk order
 * (log Z = m + ln S, H = ln S - A/S with "The Annotated DiffusionGemma",
 * "Compute entropy"), then commits and re-noises.  With vocab_ranks = G > 1 the
 * chunks are split into G contiguous ranges, rank r taking chunks
 * [floor(r n / G), floor((r + 1) n / G)) of the n, and each rank holds only the
 * W rows of its range: w_vocab given to dg_sampler_create is then that slice,
 * rows [chunk_begin * tiles_per_chunk * 256, min(chunk_end * tiles_per_chunk *
 * 256, V)) of the whole matrix (dg_vocab_slice gives both ends).  Vocabulary
 * indices stay global (Philox counters, tie-breaks, tokens), so a tick split
 * this way gives bit for bit what one unsplit sampler gives.  A tick is then:
 *   1. dg_denoise_step_partial on every rank (RMSNorm and the LM head over its
 *      chunks; asynchronous);
 *   2. the caller copies each rank's records -- rows [0, rows_cap), chunk
 *      columns [chunk_begin, chunk_end) of the [rows_cap, n_chunks] array
 *      that dg_partial_records describes -- into every other rank's array
 *      (a collective across GPUs, or device copies on one GPU), ordered on
 *      the samplers' streams after step 1;
 *   3. dg_denoise_step_finish on every rank (asynchronous): each merges all n
 *      records and commits, so every rank holds the same canvas state.
 * dg_denoise_step, dg_denoise_step_host and dg_run refuse a split sampler
 * (DG_ERR_STATE).  Without the exchange of step 2 the finishing step merges
 * stale records.
 */
dg_status dg_denoise_step_partial(dg_sampler* s, const float* resid);
dg_status dg_denoise_step_finish(dg_sampler* s);

/* Layout of the partial records for the exchange: records_dev (dev, 32-byte
 * records, [rows_cap, n_chunks] row-major, inside the workspace), the row
 * capacity, the number of vocabulary chunks and this rank's chunk range.  Any
 * output pointer may be NULL. */
dg_status dg_partial_records(const dg_sampler* s, void** records_dev, int32_t* rows_cap, int32_t* n_chunks,
                             int32_t* chunk_begin, int32_t* chunk_end);

/* The rows [v_begin, v_end) of W_vocab that rank `rank` of `ranks` holds for a
 * vocabulary of `vocab` entries (any hidden size), so a caller can cut W
 * before creating the rank's sampler.  DG_ERR_ARG for an invalid split. */
dg_status dg_vocab_slice(int32_t vocab, int32_t ranks, int32_t rank, int32_t* v_begin, int32_t* v_end);

/*
 * Self-conditioning input of the next step ("The Annotated DiffusionGemma",
 * decode mode: the previous step's probabilities times the embedding matrix
 * give each position's expected token embedding; `_forward`'s condition_x
 * before the embedding scale): for every
 * position of the canvases active at the last tick,
 *   out[c, p, :] = sum_v P[v] W[v, :],  P = softmax(z / T) of that tick
 * (after the softcap, at the tick's temperature: the distribution whose
 * entropy the commit used), with P rounded to bf16 before the contraction, as
 * the page casts it to the activation dtype, and fp32 accumulation.
 *   out  dev, fp32 [B, L, d]; rows of canvases not active at the last tick are
 *        left as they are.
 * Asynchronous.  Call it after a tick and before the next one (it reads what
 * the tick left in the workspace); needs a sampler created with self_cond = 1,
 * else DG_ERR_STATE.  It runs the LM head once more (its epilogue writes P) and
 * a tensor-core contraction of P with W, so it costs about two LM heads.
 */
dg_status dg_self_condition(dg_sampler* s, float* out);

/*
 * Top-K variant of the self-conditioning input (TensorSharp's DiffusionGemma
 * doc, "5. Acceleration status", its toggles: an experimental cutoff of the
 * self-conditioning input, K = 32 by default).  For every position of the canvases active at the last tick,
 *   out[c, p, :] = sum over the K most probable tokens v of q[v] W[v, :],
 * q = softmax(z / T) of that tick restricted to those K tokens and
 * renormalised to sum 1, which keeps the input a convex combination of
 * embedding rows as in the Annotated page's decode mode.  Tokens rank by
 * z / T (after the softcap), equal values by the lower token index; top_k >= V
 * keeps every token.  The weights come from the kept tokens' logits in fp32
 * (not from bf16 probabilities) and the sum accumulates in fp32.  Tokens whose
 * probability is below 2^-126 are never kept (their weights would be below
 * 2^-108 of the largest), so fewer than K tokens may be kept.
 *   top_k  1 <= top_k <= DG_SC_TOPK_MAX, else DG_ERR_ARG.
 *   out    dev, fp32 [B, L, d], 16-byte aligned; rows of canvases not active
 *          at the last tick are left as they are.
 * Asynchronous.  Call it after a tick and before the next one; needs a
 * sampler created with self_cond = 1, else DG_ERR_STATE.  It runs the LM head
 * once more (its epilogue writes the probabilities in bf16, which only narrow
 * down the candidates), then one CTA per position recomputes the candidates'
 * logits and sums the kept rows of W: about one LM head in all.
 */
#define DG_SC_TOPK_MAX 256
dg_status dg_self_condition_topk(dg_sampler* s, int32_t top_k, float* out);

/* Residual supplier for dg_run: the backbone's place in the loop.  Must fill
 * resid_dev [B, L, d] for the active canvases of this tick from their current
 * canvas_dev [B, L] and slots_dev [B], enqueueing work on `stream`.  Returns
 * 0 on success; anything else stops dg_run with DG_ERR_ARG. */
typedef int (*dg_resid_fn)(void* user, int32_t tick, const int32_t* canvas_dev, const dg_slot* slots_dev,
                           float* resid_dev, dg_stream_t stream);

/*
 * Drive ticks until every canvas is done: fn, then dg_denoise_step, repeated.
 * Synchronizes once every num_inference_steps ticks to test for completion.
 *   resid_dev   dev, fp32 [B, L, d] scratch the callback writes
 *   tokens_host host int32 [B, gen_blocks, L] final tokens, or NULL
 *   slots_host  host dg_slot [B] final per-canvas readout, or NULL
 */
dg_status dg_run(dg_sampler* s, dg_resid_fn fn, void* user, float* resid_dev, int32_t* tokens_host,
                 dg_slot* slots_host);

/* Free the host-side sampler object (the workspace belongs to the caller).
 * NULL-safe.  Waits for the sampler's stream first. */
void dg_destroy(dg_sampler* s);

/* Device views into the workspace, valid until dg_destroy.  [B, L] row-major. */
const int32_t* dg_canvas(const dg_sampler* s);      /* current tokens                                 */
const uint8_t* dg_committed(const dg_sampler* s);   /* 1 where frozen in the current block            */
const int16_t* dg_commit_step(const dg_sampler* s); /* step at which each position froze, -1 if not  */
const float* dg_entropy(const dg_sampler* s);       /* H (nats) from the last tick                    */
const float* dg_logz(const dg_sampler* s);          /* log Z of softmax(z/T) from the last tick       */
const int32_t* dg_sample(const dg_sampler* s);      /* sampled token from the last tick               */
const int32_t* dg_argmax(const dg_sampler* s);      /* argmax token from the last tick                */
const int32_t* dg_tokens_out(const dg_sampler* s);  /* [B, gen_blocks, L] tokens of finished blocks   */
/* [B, gen_blocks, L] commit heatmap of finished blocks: the step at which each
 * position took its final token (under DG_REACCEPT, the block's last step). */
const int16_t* dg_commit_steps_out(const dg_sampler* s);
const dg_slot* dg_slots(const dg_sampler* s);       /* [B] per-canvas state                           */
/* bf16 [rows, d] normalised hidden rows of the last tick (the LM head's input), one row per
 * position of the active canvases in canvas order (active canvas a, position p -> row a*L + p). */
const uint16_t* dg_normed(const dg_sampler* s);

/* Per-kernel timing: with events set (four cudaEvent_t created by the caller),
 * every later tick records events[0] before the RMSNorm kernel, events[1] after
 * it, events[2] after the LM-head kernel (LM head fused with the softmax
 * statistics and the sample) and events[3] after the finishing kernel (combine,
 * commit, re-noise, next-tick plan), on the sampler's stream (as external event
 * nodes when the tick is being captured into a CUDA graph).  NULL turns it off.
 * The events stay owned by the caller. */
dg_status dg_set_timing_events(dg_sampler* s, void* const* events);

/* Copy the per-canvas state to host memory (dg_slot [B]).  Synchronizing;
 * also reports a latched device fault. */
dg_status dg_sync_info(dg_sampler* s, dg_slot* slots_host);

/* Whole sampler state in host arrays ([B] and [B, L] row-major, [B, G, L] for
 * tokens_out and commit_steps_out), for checkpoint and resume.  prev_argmax is the argmax canvas of
 * each canvas's previous step (the early-stop test compares against it). */
typedef struct dg_state {
  int32_t tick;
  dg_slot* slots;       /* [B]        */
  int32_t* tokens;      /* [B, L]     */
  uint8_t* committed;   /* [B, L]     */
  int16_t* commit_step; /* [B, L]     */
  int32_t* prev_argmax; /* [B, L]     */
  int32_t* tokens_out;  /* [B, G, L]  */
  int16_t* commit_steps_out; /* [B, G, L]; NULL: not copied */
} dg_state;

/* Copy out the state (synchronizing). */
dg_status dg_get_state(dg_sampler* s, dg_state* host);

/* Replace the state (synchronizing); the next tick resumes from it.  The
 * active set is rebuilt from the slots' states; per-canvas seeds, admit ticks
 * and temperatures are taken from the config and the slots' steps. */
dg_status dg_set_state(dg_sampler* s, const dg_state* host);

/* Test hook for failure detection.  While on, the LM-head kernel does not
 * count its finished units, so the finishing kernel's bounded wait for them
 * runs out after about a second; the kernels then finish, the tick latches
 * DG_ERR_TIMEOUT and the next synchronizing call reports it.  No wait hangs
 * and nothing faults.  The sampler's state after such a tick is undefined;
 * dg_set_state (which also clears the latch) makes it usable again. */
dg_status dg_debug_hold_slabs(dg_sampler* s, int on);

/* Test hook for failure detection, process-wide: after `after` more CUDA
 * calls that the library checks (0: the next one), one is not made and is
 * reported as failed with cudaErrorLaunchFailure, as the real call would
 * report a failure -- the entry point returns DG_ERR_CUDA with the call named
 * in dg_last_error.  The hook then turns itself off; after = -1 turns it off
 * at once.  Nothing reaches the GPU.  A failure between the kernels of a tick
 * leaves the sampler's state undefined, as a real one would; dg_set_state
 * makes it usable again.  DG_ERR_ARG for after < -1. */
dg_status dg_debug_fail_cuda_call(int32_t after);

/*
 * Race and bounds checks of the debug build (the library compiled with
 * DG_DEBUG_CHECKS; the release build returns DG_ERR_UNSUPPORTED).  In that
 * build every sub-buffer of the workspace is followed by a 256-byte guard
 * filled with 0xA5 at creation, and the kernels check their indices (canvas,
 * position, block and token ranges, row tiles, vocabulary tiles and partial
 * records) before they touch memory: a failed check skips the access and
 * latches DG_ERR_BOUNDS with the check's site and value instead of faulting.
 * dg_debug_check (synchronizing) reads every guard back: DG_OK when all are
 * intact, else DG_ERR_BOUNDS with the workspace offset of the first damaged
 * guard in *first_bad (NULL allowed); a latched index failure is reported the
 * same way, with its site and value in the message.
 */
dg_status dg_debug_check(dg_sampler* s, uint64_t* first_bad);

const char* dg_status_string(dg_status st);
const char* dg_last_error(const dg_sampler* s); /* "" when none; s may be NULL (last create failure) */

/*
 * Stateless LM-head statistics without any workspace.  The paper has no
 * counterpart: this is a library convenience, not a step of the method.
 *
 * Computes steps 1-3 above for the positions of ONE canvas -- RMSNorm, tied LM
 * head, and at temperature T the entropy H (nats), log Z, the sampled token
 * and the argmax of every position -- as a sampler tick computes them for an
 * active canvas with this seed, block, step and temperature (position p is
 * row p of resid), for a sampler whose final logit softcap is off (softcap 0;
 * this call applies none).  Nothing is committed or re-noised and no sampler
 * is needed.
 *
 * Who it is for: callers that cannot allocate device memory at the point of
 * the call, such as engines that reserve the whole device for their own pool
 * at start-up (a later cudaMalloc fails), or code where cudaMalloc/cudaFree
 * would synchronize the device.  The scratch this call needs (the normalised
 * rows, the split-vocabulary partial records and each row's best Gumbel score)
 * is one fixed array in device global memory inside the library, about
 * 2.7 MB on each device the library is loaded on, held until the process
 * exits.  Nothing is allocated per call, by this function or by anything it
 * calls.
 *
 * Limits: 1 <= rows <= DG_STATIC_MAX_ROWS; hidden a multiple of 8 and
 * <= DG_STATIC_MAX_HIDDEN; vocab >= 2; temperature > 0; block and step in
 * [0, 65535].  Larger sizes are rejected with DG_ERR_ARG and a message saying
 * which limit was passed; nothing is launched then.
 *
 *   resid     dev, fp32 [rows, hidden], 16-byte aligned.
 *   w_vocab   dev, bf16 [vocab, hidden] row-major, 16-byte aligned.
 *   norm_w    dev, fp32 [hidden] (16-byte aligned), or NULL for all ones.
 *   entropy, logz      dev, fp32 [rows] outputs.
 *   sample, argmax     dev, int32 [rows] outputs.
 *   stream    the work is enqueued on this stream, then the call waits for it.
 *   err       host buffer of err_len bytes for a message on failure, or NULL.
 *
 * Synchronizing: it enqueues the work on `stream`, copies the device error
 * latch back and waits for the stream before it returns, reporting a
 * non-finite statistic (DG_ERR_NONFINITE) or an expired bounded wait
 * (DG_ERR_TIMEOUT) found on the device.
 *
 * The first call on each device (with that device current) does a one-time
 * set-up: it looks up the scratch array's device address and sets the
 * kernels' shared-memory limits.  Make that first call before capturing any
 * stream, e.g. once at start-up.
 *
 * Every call on a device shares the one scratch array, and each call resets
 * the parts of it that must start cleared.  Calls that overlap in time --
 * from two host threads, or on two streams -- race on it and give wrong
 * results: serialize them.  The sampler entry points do not use this array.
 */
#define DG_STATIC_MAX_ROWS 256
#define DG_STATIC_MAX_HIDDEN 4096
dg_status dg_lmhead_stats_static(const float* resid, int32_t rows, const void* w_vocab, int32_t vocab,
                                 int32_t hidden, const float* norm_w, float rms_eps, float temperature,
                                 uint64_t seed, int32_t block, int32_t step, float* entropy, float* logz,
                                 int32_t* sample, int32_t* argmax, dg_stream_t stream, char* err, size_t err_len);

#ifdef __cplusplus
}
#endif

#endif /* DG_SAMPLER_H */
