"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Only inputs live here: the tied vocabulary matrix ``W_vocab`` and the residual
rows that stand in for the backbone's output at each denoising step.  None of
the sampler's arithmetic is in this module.  The definitions are in
``synth.c``; this file compiles it once and marshals numpy arrays.

The workload shapes follow the pages: a 256-position canvas (TensorSharp
DiffusionGemma doc, "4. Architecture details", ``diffusion.canvas_length``),
V = 2^18 (ComfyUI-DiffusionGemma, "Terms and units": 18 bits per position),
and weights drawn from N(0, 0.02^2).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")
_SO_GPU = os.path.join(_BUILD, "libsynth_gpu.so")
_lib = None
_lib_gpu = None

PURPOSE_W = 0
PURPOSE_HIDDEN = 1


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def build_gpu(force: bool = False) -> str:
    """Compile the device residual generator ``synth_gpu.cu`` (nvcc, sm_103a) into ``_build/libsynth_gpu.so``."""
    src = os.path.join(_HERE, "synth_gpu.cu")
    hdr = os.path.join(os.path.dirname(_HERE), "include", "dg_sampler.h")
    if force or not os.path.exists(_SO_GPU) or os.path.getmtime(_SO_GPU) < max(os.path.getmtime(src),
                                                                                   os.path.getmtime(hdr)):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO_GPU + f".tmp{os.getpid()}"
        nvcc = os.environ.get("NVCC") or "/usr/local/cuda/bin/nvcc"
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-Xcompiler", "-fPIC",
                        "-Xcompiler", "-ffp-contract=off", "-I", os.path.dirname(hdr), "-shared", "-o", tmp, src],
                       check=True)
        os.replace(tmp, _SO_GPU)
    return _SO_GPU


def resid_device(w_bf16_ptr: int, tokens_ptr: int, slots_ptr: int, B: int, L: int, V: int, d: int, sigma: float,
                 out_ptr: int, stream_ptr: int) -> None:
    """Device residual rows for every active canvas (same definition as ``resid_rows``), enqueued on a stream."""
    global _lib_gpu
    if _lib_gpu is None:
        lib = ctypes.CDLL(build_gpu())
        lib.synth_resid_device.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_double,
                                                                                          ctypes.c_void_p,
                                                                                          ctypes.c_void_p]
        lib.synth_resid_device.restype = ctypes.c_int
        _lib_gpu = lib
    rc = _lib_gpu.synth_resid_device(w_bf16_ptr, tokens_ptr, slots_ptr, B, L, V, d, sigma, out_ptr, stream_ptr)
    if rc != 0:
        raise RuntimeError(f"synth_resid_device failed with CUDA error {rc}")


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.synth_philox4x32_10.argtypes = [u32p, u32p, u32p]
        lib.synth_philox4x32_10.restype = None
        lib.synth_wvocab.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.synth_wvocab.restype = None
        lib.synth_resid_rows.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
        lib.synth_resid_rows.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox4x32-10 block (Salmon et al., SC'11): 4 counter words, 2 key words."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    _load().synth_philox4x32_10(c.ctypes.data_as(u32p), k.ctypes.data_as(u32p), out.ctypes.data_as(u32p))
    return out


def wvocab(seed: int, V: int, d: int, sigma_w: float = 0.02, want_f32: bool = False, nthreads: int = 0):
    """W_vocab [V, d]: returns the bf16 bit patterns (uint16), and the fp32 values if asked."""
    w16 = np.empty((V, d), dtype=np.uint16)
    w32 = np.empty((V, d), dtype=np.float32) if want_f32 else None
    _load().synth_wvocab(seed, V, d, sigma_w, _ptr(w32) if w32 is not None else None, _ptr(w16),
                         nthreads or default_threads())
    return (w16, w32) if want_f32 else w16


def norm_weight(seed: int, d: int, spread: float = 0.1) -> np.ndarray:
    """An RMSNorm weight vector [d] in fp32: 1 + spread * N(0,1), drawn from the W stream of ``seed``."""
    _, w32 = wvocab(seed, 1, d, sigma_w=spread, want_f32=True)
    return (np.float32(1.0) + w32[0]).astype(np.float32)


def resid_rows(seeds, block, step, pos, tok, w_bf16: np.ndarray, sigma: float, nthreads: int = 0) -> np.ndarray:
    """Residual rows r[i, :] = W[tok[i]] + sigma * N(0,1) noise keyed by (seed, block, step, pos)."""
    seeds = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint64))
    n = seeds.shape[0]
    block = np.ascontiguousarray(np.broadcast_to(np.asarray(block, dtype=np.int32), (n,)))
    step = np.ascontiguousarray(np.broadcast_to(np.asarray(step, dtype=np.int32), (n,)))
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
    tok = np.ascontiguousarray(np.asarray(tok, dtype=np.int32))
    assert pos.shape == (n,) and tok.shape == (n,)
    V, d = w_bf16.shape
    assert tok.min(initial=0) >= 0 and tok.max(initial=0) < V
    out = np.empty((n, d), dtype=np.float32)
    _load().synth_resid_rows(n, _ptr(seeds), _ptr(block), _ptr(step), _ptr(pos), _ptr(tok),
                             _ptr(np.ascontiguousarray(w_bf16)), d, sigma, _ptr(out), nthreads or default_threads())
    return out


def canvas_resid(seed: int, block: int, step: int, tokens: np.ndarray, w_bf16: np.ndarray, sigma: float) -> np.ndarray:
    """Residual [L, d] for one canvas whose current tokens are ``tokens`` [L]."""
    L = tokens.shape[0]
    return resid_rows(np.full(L, seed, dtype=np.uint64), block, step, np.arange(L, dtype=np.int32), tokens,
                      w_bf16, sigma)


def bf16_to_f32(w16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (w16.astype(np.uint32) << np.uint32(16)).view(np.float32)
