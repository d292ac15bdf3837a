"""GB300 (sm_103a) denoise step of DiffusionGemma's uniform-state discrete-diffusion sampler.

A thin ctypes binding over the C ABI in ``include/dg_sampler.h`` (library
``_build/libdgsampler.so``): argument marshalling only, every step of the path
runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no CPU fallback: if the library is missing, importing the
binding raises.

Names match the C ABI (``dg_sampler_create``, ``dg_denoise_step``, ``dg_run``,
``dg_destroy`` ...).  ``Sampler`` bundles them for Python callers.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# DG_LIBRARY=debug selects the index-checking build (libdgsampler_debug.so, build.py --debug)
LIB_PATH = os.path.join(_PKG, "_build", "libdgsampler_debug.so" if os.environ.get("DG_LIBRARY") == "debug"
                        else "libdgsampler.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "dg_sampler.h")

DG_OK, DG_ERR_ARG, DG_ERR_ALIGN, DG_ERR_WORKSPACE, DG_ERR_CUDA, DG_ERR_STATE, DG_ERR_NONFINITE, \
    DG_ERR_UNSUPPORTED, DG_ERR_TIMEOUT, DG_ERR_BOUNDS = range(10)
DG_FREEZE = 0
DG_REACCEPT = 1
WAITING, ACTIVE, DONE = 0, 1, 2


class dg_config(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int32), ("hidden", ctypes.c_int32), ("canvas_len", ctypes.c_int32),
                ("n_canvases", ctypes.c_int32), ("gen_blocks", ctypes.c_int32),
                ("num_inference_steps", ctypes.c_int32), ("t_min", ctypes.c_float), ("t_max", ctypes.c_float),
                ("entropy_bound", ctypes.c_float), ("confidence", ctypes.c_float), ("stability", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("mode", ctypes.c_int32), ("max_active", ctypes.c_int32),
                ("seeds", ctypes.POINTER(ctypes.c_uint64)), ("admit_tick", ctypes.POINTER(ctypes.c_int32)),
                ("softcap", ctypes.c_float), ("vocab_ranks", ctypes.c_int32), ("vocab_rank", ctypes.c_int32),
                ("self_cond", ctypes.c_int32)]


class dg_slot(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("admit_tick", ctypes.c_int32), ("state", ctypes.c_int32),
                ("block", ctypes.c_int32), ("step", ctypes.c_int32), ("n_committed", ctypes.c_int32),
                ("steps_used", ctypes.c_int32), ("converged_blocks", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("mean_entropy", ctypes.c_float), ("n_remasked", ctypes.c_int32),
                ("stable_steps", ctypes.c_int32)]


SLOT_DTYPE = np.dtype([("seed", "u8"), ("admit_tick", "i4"), ("state", "i4"), ("block", "i4"), ("step", "i4"),
                       ("n_committed", "i4"), ("steps_used", "i4"), ("converged_blocks", "i4"),
                       ("temperature", "f4"), ("mean_entropy", "f4"), ("n_remasked", "i4"),
                       ("stable_steps", "i4")], align=True)
assert SLOT_DTYPE.itemsize == ctypes.sizeof(dg_slot) == 56


class dg_state(ctypes.Structure):
    _fields_ = [("tick", ctypes.c_int32), ("slots", ctypes.c_void_p), ("tokens", ctypes.c_void_p),
                ("committed", ctypes.c_void_p), ("commit_step", ctypes.c_void_p),
                ("prev_argmax", ctypes.c_void_p), ("tokens_out", ctypes.c_void_p), ("commit_steps_out", ctypes.c_void_p)]


DG_RESID_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p)

# exported name -> (restype, argtypes)
_SIGS = {
    "dg_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(dg_config)]),
    "dg_sampler_create": (ctypes.c_int, [ctypes.POINTER(dg_config), ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                         ctypes.POINTER(ctypes.c_void_p)]),
    "dg_denoise_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "dg_denoise_step_partial": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "dg_denoise_step_finish": (ctypes.c_int, [ctypes.c_void_p]),
    "dg_self_condition": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "dg_self_condition_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "dg_debug_fail_cuda_call": (ctypes.c_int, [ctypes.c_int32]),
    "dg_partial_records": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
                                          ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "dg_vocab_slice": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "dg_denoise_step_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "dg_run": (ctypes.c_int, [ctypes.c_void_p, DG_RESID_FN, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p]),
    "dg_destroy": (None, [ctypes.c_void_p]),
    "dg_canvas": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_committed": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_commit_step": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_entropy": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_logz": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_sample": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_argmax": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_tokens_out": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_commit_steps_out": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_slots": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_normed": (ctypes.c_void_p, [ctypes.c_void_p]),
    "dg_sync_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "dg_set_timing_events": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "dg_debug_hold_slabs": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "dg_get_state": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(dg_state)]),
    "dg_set_state": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(dg_state)]),
    "dg_debug_check": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64)]),
    "dg_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dg_last_error": (ctypes.c_char_p, [ctypes.c_void_p]),
    "dg_lmhead_stats_static": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_float, ctypes.c_float,
                                              ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_char_p, ctypes.c_size_t]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'); "
                          "there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class DGError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{lib.dg_status_string(status).decode()}: {msg}")
        self.status = status


def _check(st: int, handle=None):
    if st != DG_OK:
        raise DGError(st, (lib.dg_last_error(handle) or b"").decode())


def make_config(vocab, hidden, canvas_len, n_canvases=1, gen_blocks=1, num_inference_steps=48, t_min=0.4,
                t_max=0.8, entropy_bound=0.1, confidence=0.005, stability=1, rms_eps=1e-6, mode=DG_FREEZE,
                max_active=0, seeds=None, admit_tick=None, softcap=0.0, vocab_ranks=0, vocab_rank=0, self_cond=0):
    """Build a ``dg_config``; the returned object keeps the seed/admit arrays alive."""
    cfg = dg_config(vocab, hidden, canvas_len, n_canvases, gen_blocks, num_inference_steps, t_min, t_max,
                    entropy_bound, confidence, stability, rms_eps, mode, max_active)
    cfg.softcap = softcap
    cfg.vocab_ranks = vocab_ranks
    cfg.vocab_rank = vocab_rank
    cfg.self_cond = self_cond
    keep = []
    if seeds is not None:
        a = (ctypes.c_uint64 * n_canvases)(*[int(s) for s in seeds])
        cfg.seeds = ctypes.cast(a, ctypes.POINTER(ctypes.c_uint64))
        keep.append(a)
    if admit_tick is not None:
        a = (ctypes.c_int32 * n_canvases)(*[int(t) for t in admit_tick])
        cfg.admit_tick = ctypes.cast(a, ctypes.POINTER(ctypes.c_int32))
        keep.append(a)
    cfg._keep = keep
    return cfg


def dg_workspace_size(cfg: dg_config) -> int:
    return int(lib.dg_workspace_size(ctypes.byref(cfg)))


def vocab_slice(vocab: int, ranks: int, rank: int):
    """dg_vocab_slice: the W rows [v_begin, v_end) rank ``rank`` of ``ranks`` holds."""
    b, e = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.dg_vocab_slice(vocab, ranks, rank, ctypes.byref(b), ctypes.byref(e)))
    return b.value, e.value


def exchange_partials(samplers) -> None:
    """The exchange of a vocabulary-parallel tick for ranks that share one GPU: every rank's chunk
    columns of the partial records are copied into every other rank's array, each copy ordered after
    both samplers' partial ticks (device copies only)."""
    import torch
    for dst in samplers:
        rec_d, (b_d, e_d) = dst.partial_records(), dst.chunk_range()
        for src in samplers:
            if src is dst:
                continue
            rec_s, (b, e) = src.partial_records(), src.chunk_range()
            dst.stream.wait_stream(src.stream)
            with torch.cuda.stream(dst.stream):
                rec_d[:, b:e].copy_(rec_s[:, b:e])
            src.stream.wait_stream(dst.stream)


def all_gather_partials(records, chunk_ranges, rank: int, group=None) -> None:
    """The exchange of a vocabulary-parallel tick across processes (torch.distributed): ``records`` is
    this rank's [rows_cap, n_chunks, 8] record array (a view of the workspace, or any tensor of that
    layout), ``chunk_ranges`` every rank's (chunk_begin, chunk_end).  Each rank's columns are packed,
    all-gathered and written into every rank's array in place.  The collective and the copies run on
    torch's current stream: call it under ``torch.cuda.stream(sampler.stream)`` (or after synchronizing
    the sampler's stream) so that they follow the partial tick, and before dg_denoise_step_finish."""
    import torch
    import torch.distributed as dist
    b, e = chunk_ranges[rank]
    mine = records[:, b:e].contiguous()
    parts = [torch.empty((records.shape[0], e1 - b1, records.shape[2]), dtype=records.dtype, device=records.device)
             for b1, e1 in chunk_ranges]
    dist.all_gather(parts, mine, group=group)
    for (b1, e1), part in zip(chunk_ranges, parts):
        records[:, b1:e1].copy_(part)


def dg_lmhead_stats_static(resid, w_vocab, norm_w, rms_eps, temperature, seed, block, step, entropy, logz, sample,
                           argmax, stream=None):
    """LM-head statistics of one canvas into caller-provided outputs, with no device allocation.

    ``resid`` fp32 [rows, d], ``w_vocab`` bf16 [V, d], ``norm_w`` fp32 [d] or None; ``entropy``/``logz`` fp32
    [rows] and ``sample``/``argmax`` int32 [rows] are written.  Raises ``DGError`` with the library's message.
    """
    import torch
    rows, d = resid.shape
    st = stream if stream is not None else torch.cuda.current_stream(resid.device)
    msg = ctypes.create_string_buffer(512)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    status = lib.dg_lmhead_stats_static(ptr(resid), rows, ptr(w_vocab), w_vocab.shape[0], d, ptr(norm_w),
                                        float(rms_eps), float(temperature), int(seed), int(block), int(step),
                                        ptr(entropy), ptr(logz), ptr(sample), ptr(argmax),
                                        ctypes.c_void_p(st.cuda_stream), msg, len(msg))
    if status != DG_OK:
        raise DGError(status, msg.value.decode())


class Sampler:
    """One sampler: owns its workspace (a torch uint8 CUDA tensor) and borrows ``w_vocab``."""

    def __init__(self, cfg: dg_config, w_vocab, norm_w=None, stream=None):
        import torch
        assert w_vocab.is_cuda and w_vocab.dtype == torch.bfloat16 and w_vocab.is_contiguous()
        self.cfg = cfg
        self.device = w_vocab.device
        self.w_vocab = w_vocab
        self.norm_w = norm_w
        self.B, self.L, self.d, self.V, self.G = (cfg.n_canvases, cfg.canvas_len, cfg.hidden, cfg.vocab,
                                                  cfg.gen_blocks)
        nbytes = dg_workspace_size(cfg)
        if nbytes == 0:
            h = ctypes.c_void_p()
            st = lib.dg_sampler_create(ctypes.byref(cfg), None, None, None, 0, None, ctypes.byref(h))
            _check(st if st != DG_OK else DG_ERR_ARG)
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.workspace.data_ptr()) % 256
        self._ws_off = off
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        h = ctypes.c_void_p()
        st = lib.dg_sampler_create(ctypes.byref(cfg), ctypes.c_void_p(w_vocab.data_ptr()),
                                   ctypes.c_void_p(norm_w.data_ptr()) if norm_w is not None else None,
                                   ctypes.c_void_p(self.workspace.data_ptr() + off), nbytes,
                                   ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h))
        _check(st)
        self.handle = h
        # page-locked result buffers of step_host, allocated once here rather than in a step
        self._host_out = (torch.empty((self.B, self.L), dtype=torch.int32).pin_memory(),
                          torch.empty((self.B, self.L), dtype=torch.float32).pin_memory())

    # --------------------------------------------------------------- calls
    def dg_denoise_step(self, resid) -> int:
        return lib.dg_denoise_step(self.handle, ctypes.c_void_p(resid.data_ptr()))

    def step(self, resid):
        _check(self.dg_denoise_step(resid), self.handle)

    def self_condition(self, out):
        """dg_self_condition: the expected embedding softmax(z/T) W of every position of the canvases
        active at the last tick, into ``out`` (fp32 [B, L, d] on the device)."""
        assert out.dtype.itemsize == 4 and out.is_contiguous() and out.numel() == self.B * self.L * self.d
        _check(lib.dg_self_condition(self.handle, ctypes.c_void_p(out.data_ptr())), self.handle)

    def self_condition_topk(self, out, top_k=32):
        """dg_self_condition_topk: the same input restricted to each position's ``top_k`` most probable
        tokens, renormalised, into ``out`` (fp32 [B, L, d] on the device)."""
        assert out.dtype.itemsize == 4 and out.is_contiguous() and out.numel() == self.B * self.L * self.d
        _check(lib.dg_self_condition_topk(self.handle, int(top_k), ctypes.c_void_p(out.data_ptr())), self.handle)

    def step_partial(self, resid):
        """dg_denoise_step_partial: RMSNorm and the LM head over this rank's vocabulary chunks."""
        _check(lib.dg_denoise_step_partial(self.handle, ctypes.c_void_p(resid.data_ptr())), self.handle)

    def step_finish(self):
        """dg_denoise_step_finish: merge every chunk's records, commit and re-noise."""
        _check(lib.dg_denoise_step_finish(self.handle), self.handle)

    def _records_layout(self):
        ptr, rows, n, b, e = ctypes.c_void_p(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib.dg_partial_records(self.handle, ctypes.byref(ptr), ctypes.byref(rows), ctypes.byref(n),
                                      ctypes.byref(b), ctypes.byref(e)), self.handle)
        return ptr.value, rows.value, n.value, b.value, e.value

    def partial_records(self):
        """The [rows_cap, n_chunks, 8] int32 view of the 32-byte partial records (dg_partial_records)."""
        import torch
        ptr, rows, n, _, _ = self._records_layout()
        off = ptr - self.workspace.data_ptr()
        return self.workspace[off:off + rows * n * 32].view(torch.int32).view(rows, n, 8)

    def chunk_range(self):
        """This rank's vocabulary chunks [chunk_begin, chunk_end)."""
        _, _, _, b, e = self._records_layout()
        return b, e

    def step_host(self, resid_host: np.ndarray, want_canvas=True, want_entropy=True):
        """dg_denoise_step_host; the results land in page-locked buffers kept by the sampler and are
        returned as copies.  Pass a page-locked ``resid_host`` for an asynchronous input copy."""
        assert resid_host.dtype == np.float32 and resid_host.flags["C_CONTIGUOUS"]
        canvas, ent = self._host_out
        _check(lib.dg_denoise_step_host(self.handle, ctypes.c_void_p(resid_host.ctypes.data),
                                        ctypes.c_void_p(canvas.data_ptr()) if want_canvas else None,
                                        ctypes.c_void_p(ent.data_ptr()) if want_entropy else None), self.handle)
        return (canvas.numpy().copy() if want_canvas else None), (ent.numpy().copy() if want_entropy else None)

    def run(self, resid_fn, resid_dev=None):
        """dg_run with a Python callback ``resid_fn(tick, canvas_ptr, slots_ptr, resid_ptr, stream_ptr) -> int``."""
        cb = DG_RESID_FN(lambda user, tick, canvas, slots, resid, stream: int(resid_fn(tick, canvas, slots, resid,
                                                                                          stream)))
        tokens = np.empty((self.B, self.G, self.L), np.int32)
        slots = np.empty(self.B, SLOT_DTYPE)
        _check(lib.dg_run(self.handle, cb, None, ctypes.c_void_p(resid_dev.data_ptr()) if resid_dev is not None
                          else None, ctypes.c_void_p(tokens.ctypes.data), ctypes.c_void_p(slots.ctypes.data)),
               self.handle)
        return tokens, slots

    def set_timing_events(self, events):
        """Four torch.cuda.Event(enable_timing=True) recorded on every tick: before the RMSNorm kernel,
        after it, after the LM-head kernel and after the finishing kernel; or None."""
        if events is None:
            _check(lib.dg_set_timing_events(self.handle, None), self.handle)
            self._timing = None
            return
        assert len(events) == 4
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
                e.record(self.stream)
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        self._timing = (events, arr)
        _check(lib.dg_set_timing_events(self.handle, arr), self.handle)

    def debug_hold_slabs(self, on: bool):
        """Failure-detection test hook (dg_debug_hold_slabs): the next ticks' bounded waits run out."""
        _check(lib.dg_debug_hold_slabs(self.handle, 1 if on else 0), self.handle)

    def debug_check(self):
        """dg_debug_check (debug build): raises DGError(DG_ERR_BOUNDS) on a damaged workspace guard or a
        failed index check; returns None when all is intact."""
        off = ctypes.c_uint64()
        _check(lib.dg_debug_check(self.handle, ctypes.byref(off)), self.handle)

    def sync_info(self) -> np.ndarray:
        slots = np.empty(self.B, SLOT_DTYPE)
        _check(lib.dg_sync_info(self.handle, ctypes.c_void_p(slots.ctypes.data)), self.handle)
        return slots

    def get_state(self) -> dict:
        B, L, G = self.B, self.L, self.G
        st = {"slots": np.empty(B, SLOT_DTYPE), "tokens": np.empty((B, L), np.int32),
              "committed": np.empty((B, L), np.uint8), "commit_step": np.empty((B, L), np.int16),
              "prev_argmax": np.empty((B, L), np.int32), "tokens_out": np.empty((B, G, L), np.int32),
              "commit_steps_out": np.empty((B, G, L), np.int16)}
        s = dg_state(0, *[ctypes.c_void_p(st[k].ctypes.data) for k in ("slots", "tokens", "committed", "commit_step",
                                                                       "prev_argmax", "tokens_out",
                                                                       "commit_steps_out")])
        _check(lib.dg_get_state(self.handle, ctypes.byref(s)), self.handle)
        st["tick"] = s.tick
        return st

    def set_state(self, st: dict):
        names = ("slots", "tokens", "committed", "commit_step", "prev_argmax", "tokens_out", "commit_steps_out")
        dts = (SLOT_DTYPE, np.int32, np.uint8, np.int16, np.int32, np.int32, np.int16)
        arrs = {k: np.ascontiguousarray(st[k], dtype=dt) for k, dt in zip(names, dts) if st.get(k) is not None}
        s = dg_state(int(st["tick"]), *[ctypes.c_void_p(arrs[k].ctypes.data) if k in arrs else None for k in names])
        _check(lib.dg_set_state(self.handle, ctypes.byref(s)), self.handle)

    # --------------------------------------------------------------- views
    def _view(self, fn, dtype, shape):
        import torch
        ptr = getattr(lib, fn)(self.handle)
        off = ptr - self.workspace.data_ptr()
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        return self.workspace[off:off + n].view(dtype).view(*shape)

    def canvas(self):
        import torch
        return self._view("dg_canvas", torch.int32, (self.B, self.L))

    def committed(self):
        import torch
        return self._view("dg_committed", torch.uint8, (self.B, self.L))

    def commit_step(self):
        import torch
        return self._view("dg_commit_step", torch.int16, (self.B, self.L))

    def entropy(self):
        import torch
        return self._view("dg_entropy", torch.float32, (self.B, self.L))

    def logz(self):
        import torch
        return self._view("dg_logz", torch.float32, (self.B, self.L))

    def sample(self):
        import torch
        return self._view("dg_sample", torch.int32, (self.B, self.L))

    def argmax(self):
        import torch
        return self._view("dg_argmax", torch.int32, (self.B, self.L))

    def tokens_out(self):
        import torch
        return self._view("dg_tokens_out", torch.int32, (self.B, self.G, self.L))

    def commit_steps_out(self):
        """[B, G, L] int16: the step at which each position of each finished block took its final token."""
        import torch
        return self._view("dg_commit_steps_out", torch.int16, (self.B, self.G, self.L))

    def normed(self, n_rows: int):
        """bf16 bit patterns (int16) of the first n_rows normalised hidden rows of the last tick."""
        import torch
        return self._view("dg_normed", torch.int16, (n_rows, self.d))

    def slots_ptr(self) -> int:
        return int(lib.dg_slots(self.handle))

    def close(self):
        if getattr(self, "handle", None):
            lib.dg_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
