"""CPU oracle for the DiffusionGemma uniform-state denoise step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA path.  Its inputs come from the seeded generators in ``synth`` (a module
that holds none of the method's arithmetic) and its random draws from its own
Philox4x32-10 in ``oracle.c``.

Layout:
  oracle.c    -- fp64 arithmetic of one position (RMSNorm, logits, temperature
                 softmax, entropy, log Z, argmax, Gumbel-max sample, Philox).
  sampler.py  -- the denoising loop (schedule, early stop, entropy-bounded
                 commit, uniform re-noise, blocks, staggered admission).

Stored values under tests/golden/ are the pages' printed figures, published
known-answer vectors, hand-worked values, or oracle states written by the
script beside them that calls only this package and ``synth``.

Every function is pinned by tests in tests/test_oracle_*.py against closed
forms, brute force on tiny inputs, published known-answer vectors and
invariants; nothing here is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None

PURPOSE_INIT = 2
PURPOSE_RENOISE = 4
PURPOSE_GUMBEL_ORDER = 5

# numpy mirror of ``struct or_pos`` in oracle.c
POS_DTYPE = np.dtype([("logZ", "f8"), ("H", "f8"), ("H_online", "f8"), ("zmax", "f8"), ("zgap", "f8"),
                      ("gbest", "f8"), ("ggap", "f8"), ("amax", "i4"), ("y", "i4")])
assert POS_DTYPE.itemsize == 64


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP).  Building is not running."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64, i32, u32, u64, dbl = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                                       ctypes.c_uint64, ctypes.c_double)
        lib.or_philox.argtypes = [vp, vp, vp]
        lib.or_philox.restype = None
        lib.or_draw_u32.argtypes = [u64, u32, i32, i32, i32]
        lib.or_draw_u32.restype = u32
        lib.or_uniform_token.argtypes = [u32, i32]
        lib.or_uniform_token.restype = i32
        lib.or_bf16_rne.argtypes = [dbl]
        lib.or_bf16_rne.restype = ctypes.c_uint16
        lib.or_rmsnorm_bf16.argtypes = [i64, i64, vp, vp, dbl, vp]
        lib.or_rmsnorm_bf16.restype = None
        lib.or_stats.argtypes = [i64, i64, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
        lib.or_stats.restype = None
        lib.or_logits.argtypes = [i64, i64, i64, vp, vp, vp, ctypes.c_int]
        lib.or_logits.restype = None
        lib.or_exp_variates.argtypes = [u64, i32, i32, i32, i64, vp]
        lib.or_exp_variates.restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def threads() -> int:
    """Threads the oracle's OpenMP loops use (every core this process may run on)."""
    return max(1, len(os.sched_getaffinity(0)))


def philox(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().or_philox(_p(c), _p(k), _p(out))
    return out


def draw_u32(seed: int, purpose: int, block: int, step: int, p: int) -> int:
    return int(_load().or_draw_u32(seed, purpose, block, step, p))


def exp_variates(seed: int, block: int, step: int, p: int, V: int) -> np.ndarray:
    """The Exp(1) variates E_v (fp64 [V]) behind position p's Gumbel draws, G_v = -ln E_v: per group
    of 16 entries the sixteen order statistics in increasing order, placed in a uniformly random
    permutation of the slots (Renyi's representation of exponential order statistics; oracle.c
    gives the counters)."""
    E = np.empty(V, dtype=np.float64)
    _load().or_exp_variates(seed, block, step, p, V, _p(E))
    return E


def uniform_token(u: int, V: int) -> int:
    return int(_load().or_uniform_token(u, V))


def bf16_rne(x: float) -> int:
    return int(_load().or_bf16_rne(float(x)))


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def rmsnorm_bf16(r: np.ndarray, eps: float, w: np.ndarray | None = None) -> np.ndarray:
    """Final RMSNorm of each row of ``r`` (fp32 [n, d]) -> bf16 bit patterns [n, d]."""
    r = np.ascontiguousarray(r, dtype=np.float32)
    n, d = r.shape
    h = np.empty((n, d), dtype=np.uint16)
    wv = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    _load().or_rmsnorm_bf16(n, d, _p(r), _p(wv) if wv is not None else None, eps, _p(h))
    return h


def logits(h: np.ndarray, W: np.ndarray, block_rows: int = 8192) -> np.ndarray:
    """z = h . W^T in fp64 from bf16 operands (the tied LM head), via a BLAS matmul.

    h: bf16 bits [n, d]; W: bf16 bits [V, d].  Returns fp64 [n, V].  The bf16
    products are exact in fp64, so the only rounding is fp64 summation.
    """
    hv = bf16_value(h)
    V = W.shape[0]
    z = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, block_rows):
        z[:, v0:v0 + block_rows] = hv @ bf16_value(W[v0:v0 + block_rows]).T
    return z


def logits_loop(h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """The same logits by the plain triple loop in oracle.c (used to pin ``logits``)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    n, d = h.shape
    V = W.shape[0]
    z = np.empty((n, V), dtype=np.float64)
    _load().or_logits(n, V, d, _p(h), _p(W), _p(z), threads())
    return z


def softcap(z: np.ndarray, c: float) -> np.ndarray:
    """Final logit softcap z -> c tanh(z / c) in fp64 ("The Annotated DiffusionGemma", "Logit
    Softcapping": part of the model, applied to the final logits before the temperature).  c = 0
    leaves the logits unchanged."""
    z = np.asarray(z, dtype=np.float64)
    return z if c == 0 else c * np.tanh(z / c)


def expected_embedding(z: np.ndarray, T, W: np.ndarray, block_rows: int = 8192):
    """Self-conditioning input: e[p, :] = sum_v P[p, v] W[v, :] with P = softmax(z / T) row by row, in
    fp64 from the bf16 values of W ("The Annotated DiffusionGemma", decode mode: the previous step's
    probabilities times the embedding matrix give each position's expected token embedding, the
    probabilities being the categorical distribution its denoise loop forms from the model output
    divided by the temperature; `_forward`'s condition_x before the embedding scale).  ``z`` are the logits after the final softcap.  Returns
    (e, a): e fp64 [n, d], and a[p, k] = sum_v P[p, v] |W[v, k]|, the scale of each coordinate."""
    z = np.asarray(z, dtype=np.float64)
    T = np.broadcast_to(np.asarray(T, dtype=np.float64), (z.shape[0],))[:, None]
    zz = z / T
    P = np.exp(zz - zz.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    V, d = W.shape
    e = np.zeros((z.shape[0], d))
    a = np.zeros((z.shape[0], d))
    for v0 in range(0, V, block_rows):
        Wv = bf16_value(W[v0:v0 + block_rows])
        e += P[:, v0:v0 + block_rows] @ Wv
        a += P[:, v0:v0 + block_rows] @ np.abs(Wv)
    return e, a


def expected_embedding_topk(z: np.ndarray, T, W: np.ndarray, k: int):
    """Top-K self-conditioning input: e[p, :] = sum over the K most probable tokens v of row p of
    q[p, v] W[v, :], q = softmax(z / T) restricted to those K tokens and renormalised to sum 1.

    TensorSharp's DiffusionGemma doc ("5. Acceleration status", its toggles) lists an experimental
    top-K cutoff of the self-conditioning input (DIFFUSION_SC_TOPK, default 32) beside its on-device
    sampling; the Annotated page's decode mode describes the input as one convex combination of
    embedding rows per position, which the renormalisation keeps.  Ranking: larger z / T first, equal values by the lower token index (the
    tie rule used everywhere else); k >= V keeps every token, giving ``expected_embedding``.  In
    fp64 from the bf16 values of W; ``z`` are the logits after the final softcap.

    Returns (e, a, gap, sel): e fp64 [n, d]; a[p, k] = sum_v q[p, v] |W[v, k]|; gap[p] = the K-th
    largest z / T minus the (K+1)-th (inf when k >= V), the margin by which the kept set is
    decided; sel [n, K] the kept token indices, most probable first."""
    z = np.asarray(z, dtype=np.float64)
    n, V = z.shape
    T = np.broadcast_to(np.asarray(T, dtype=np.float64), (n,))
    kk = min(int(k), V)
    d = W.shape[1]
    e = np.zeros((n, d))
    a = np.zeros((n, d))
    gap = np.full(n, np.inf)
    sel = np.zeros((n, kk), dtype=np.int64)
    idx = np.arange(V)
    for p in range(n):
        u = z[p] / T[p]
        order = np.lexsort((idx, -u))  # by u descending, then index ascending
        keep = order[:kk]
        if kk < V:
            gap[p] = u[order[kk - 1]] - u[order[kk]]
        w = np.exp(u[keep] - u[keep].max())
        q = w / w.sum()
        Wk = bf16_value(W[keep])
        e[p] = q @ Wk
        a[p] = q @ np.abs(Wk)
        sel[p] = keep
    return e, a, gap, sel


def stats(z: np.ndarray, T, seed, block, step, pos) -> np.ndarray:
    """Per-row temperature softmax statistics and Gumbel-max sample; returns POS_DTYPE [n]."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    n, V = z.shape
    bc = lambda a, dt: np.ascontiguousarray(np.broadcast_to(np.asarray(a, dtype=dt), (n,)))
    Tv, sv, bv, stv, pv = bc(T, np.float64), bc(seed, np.uint64), bc(block, np.int32), bc(step, np.int32), bc(pos, np.int32)
    out = np.zeros(n, dtype=POS_DTYPE)
    _load().or_stats(n, V, _p(z), _p(Tv), _p(sv), _p(bv), _p(stv), _p(pv), _p(out), threads())
    return out


from .sampler import OracleConfig, OracleSampler, temperature  # noqa: E402,F401
