"""The oracle's denoising loop (TEST INFRASTRUCTURE ONLY; see the package docstring).

The loop follows "The Annotated DiffusionGemma" (mlberkeley), section
"Sampling" and its code "Denoise, stage, commit, and generate", written in the
eager order (forward -> sample -> commit -> re-noise), which the section "Lazy
Sampling" states is the same procedure as its lazy order.  One tick runs, for
every active canvas, at its own step s of its own block b:

  1. temperature T_s = t_max + (s/N)(t_min - t_max)        ("Apply temperature")
  2. h = RMSNorm(r), z = h W^T (with the final softcap c tanh(z/c) when c > 0),
     softmax(z/T): H, log Z, argmax, sample y
                       ("RMSNorm", "Logit Softcapping", "Compute entropy")
  3. early stop when s >= 1, mean_p H < confidence and the argmax canvas
     equals the previous step's                   ("Check for early stopping")
  4. otherwise sort the open positions by (H, p) ascending and accept
     position j of that order iff the sum of the entropies before it is
     <= entropy_bound; accepted positions take y
                            ("Keep a low-entropy prefix and renoise the rest")
  5. on early stop or at s = N-1 every open position takes y and the
     block is finished ("On convergence or after N steps, we commit")
  6. every other open position is re-noised to a uniform token.

Two commit modes.  "freeze": accepted positions freeze and only uncommitted
positions are open.  "reaccept": every position is open at every step, as the
Annotated page's denoise code computes it (its `accepted` mask is recomputed
from all entropies each step and `torch.where(accepted, sample, randint)`
rebuilds the whole canvas); the committed mask is then the latest step's
accepted set and commit_step the last step a position was accepted.

Readings where the pages are silent or disagree:
by default committed positions stay frozen (ComfyUI-DiffusionGemma, "What it
is": positions committed at low entropy are not revisited) and only uncommitted
positions enter the per-step sort; the prefix is exclusive and compared with <=; ties in
H go to the lower position; the early-stop test is skipped at s = 0; the last
step commits every remaining position to its sample; blocks of one canvas run
one after another with a fresh uniform canvas each (DiffusionGemma Denoise
node, "gen_length" input); canvas c joins at the first tick >= admit_tick[c]
with a free running slot (at most max_active canvases run at once).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Optional

import numpy as np

WAITING, ACTIVE, DONE = 0, 1, 2


def temperature(s: int, N: int, t_min: float, t_max: float) -> float:
    """T_s = t_max + (s/N)(t_min - t_max), s = 0..N-1, in fp64 ("Apply temperature")."""
    return t_max + (s / N) * (t_min - t_max)


def entropy_bounded_accept(H, candidates, bound: float):
    """Entropy-bounded acceptance ("Keep a low-entropy prefix and renoise the rest").

    The candidate positions are ordered by (H, p) ascending; position j of that
    order is accepted iff E_j = sum_{i<j} H_(i) <= bound, summed in fp64 in
    sorted order.  Returns (order, E, k): the order, the exclusive prefix sums,
    and the number k of accepted positions (the first k of the order).
    """
    order = sorted([int(p) for p in candidates], key=lambda p: (float(H[p]), p))
    E = 0.0
    k = 0
    excl = []
    for p in order:
        excl.append(E)
        if E <= bound:
            k += 1
        E += float(H[p])
    return order, excl, k


@dataclasses.dataclass
class OracleConfig:
    vocab: int
    hidden: int
    canvas_len: int
    n_canvases: int = 1
    gen_blocks: int = 1
    num_inference_steps: int = 48
    t_min: float = 0.4
    t_max: float = 0.8
    entropy_bound: float = 0.1
    confidence: float = 0.005
    rms_eps: float = 1e-6
    seeds: Optional[list] = None
    admit_tick: Optional[list] = None
    max_active: Optional[int] = None  # most canvases running in one tick (None: all)
    mode: str = "freeze"  # "freeze" or "reaccept" (see the module docstring)
    softcap: float = 0.0  # final logit softcap c (0 = off): z -> c tanh(z / c) before the temperature
    stability: int = 1  # steps in a row the argmax canvas must equal the one before for an early stop
    # parity margins stated by the task for flagging near-ties
    margin_H: float = 1e-3
    margin_gap: float = 1e-4

    def seed(self, c: int) -> int:
        return int(self.seeds[c]) if self.seeds is not None else c

    def admit(self, c: int) -> int:
        return int(self.admit_tick[c]) if self.admit_tick is not None else 0


@dataclasses.dataclass
class TickRecord:
    """What one tick computed, for every row of every canvas that was active."""
    tick: int
    canvases: np.ndarray          # [n_active] canvas ids, in row order
    block: np.ndarray             # [n_active]
    step: np.ndarray              # [n_active]
    T: np.ndarray                 # [n_active] fp64
    stats: np.ndarray             # [n_active*L] POS_DTYPE
    mean_H: np.ndarray            # [n_active]
    converged: np.ndarray         # [n_active] bool
    final: np.ndarray             # [n_active] bool (early stop or last step)
    accepted: np.ndarray          # [n_active, L] bool: committed at this tick
    n_accepted: np.ndarray        # [n_active]
    flag_y: np.ndarray            # [n_active*L] sample top-2 gap below margin
    flag_amax: np.ndarray         # [n_active*L] argmax top-2 gap below margin
    flag_commit: np.ndarray       # [n_active, L] position sits on a commit-boundary near-tie
    flag_canvas: np.ndarray       # [n_active] canvas-level near-tie (prefix sum or early-stop test)
    n_remasked: np.ndarray = None  # [n_active] reaccept: accepted at the previous step, re-noised now


class OracleSampler:
    """Free-running oracle over B canvases.  ``resid_fn(canvases, blocks, steps, tokens) -> r``
    supplies the residual rows [n_active*L, d] (the backbone stand-in from ``synth``)."""

    def __init__(self, cfg: OracleConfig, W_bf16: np.ndarray, norm_w: Optional[np.ndarray] = None):
        from . import PURPOSE_INIT, draw_u32, uniform_token  # noqa: F401
        self.cfg = cfg
        self.W = W_bf16
        self.norm_w = norm_w
        B, L = cfg.n_canvases, cfg.canvas_len
        assert W_bf16.shape == (cfg.vocab, cfg.hidden)
        self.tick_no = 0
        self.status = np.full(B, WAITING, dtype=np.int32)
        self.block = np.zeros(B, dtype=np.int32)
        self.step_no = np.zeros(B, dtype=np.int32)
        self.x = np.zeros((B, L), dtype=np.int32)
        self.committed = np.zeros((B, L), dtype=bool)
        self.commit_step = np.full((B, L), -1, dtype=np.int16)
        self.prev_amax = np.zeros((B, L), dtype=np.int32)
        self.stable_run = np.zeros(B, dtype=np.int32)  # steps in a row with an unchanged argmax canvas
        self.steps_used = np.zeros(B, dtype=np.int32)
        self.converged_blocks = np.zeros(B, dtype=np.int32)
        self.tokens_out = np.full((B, cfg.gen_blocks, L), -1, dtype=np.int32)
        # commit heatmap of each finished block: the step at which each position took its final token
        self.commit_steps_out = np.full((B, cfg.gen_blocks, L), -1, dtype=np.int16)
        self._admit(0)

    # ---------------------------------------------------------------- state
    def _init_canvas(self, c: int, b: int):
        """Uniform initial canvas of block b ("Lazy Sampling": the first input is uniform)."""
        from . import PURPOSE_INIT, draw_u32, uniform_token
        cfg = self.cfg
        for p in range(cfg.canvas_len):
            self.x[c, p] = uniform_token(draw_u32(cfg.seed(c), PURPOSE_INIT, b, 0, p), cfg.vocab)
        self.committed[c] = False
        self.commit_step[c] = -1
        self.prev_amax[c] = 0
        self.stable_run[c] = 0
        self.block[c] = b
        self.step_no[c] = 0

    def _admit(self, tick: int):
        """Canvases due by this tick join in canvas order while a running slot is free."""
        cap = self.cfg.max_active if self.cfg.max_active is not None else self.cfg.n_canvases
        running = int(np.sum(self.status == ACTIVE))
        for c in range(self.cfg.n_canvases):
            if running >= cap:
                break
            if self.status[c] == WAITING and self.cfg.admit(c) <= tick:
                self._init_canvas(c, 0)
                self.status[c] = ACTIVE
                running += 1

    def active(self) -> np.ndarray:
        return np.nonzero(self.status == ACTIVE)[0].astype(np.int32)

    def done(self) -> bool:
        return bool(np.all(self.status == DONE))

    def snapshot(self) -> dict:
        """Copy of the whole state (used to teacher-force the CUDA path from the oracle)."""
        return {k: getattr(self, k).copy() for k in ("status", "block", "step_no", "x", "committed", "commit_step",
                                                     "prev_amax", "steps_used", "converged_blocks", "tokens_out",
                                                     "commit_steps_out", "stable_run")} | {
            "tick": self.tick_no}

    # ----------------------------------------------------------------- tick
    def tick(self, resid_fn: Callable) -> Optional[TickRecord]:
        from . import PURPOSE_RENOISE, draw_u32, logits, rmsnorm_bf16, softcap, stats, uniform_token
        cfg = self.cfg
        L, V, N = cfg.canvas_len, cfg.vocab, cfg.num_inference_steps
        act = self.active()
        rec = None
        if act.size:
            blocks, steps = self.block[act].copy(), self.step_no[act].copy()
            r = resid_fn(act, blocks, steps, self.x[act].copy())
            assert r.shape == (act.size * L, cfg.hidden)
            h = rmsnorm_bf16(r, cfg.rms_eps, self.norm_w)
            z = softcap(logits(h, self.W), cfg.softcap)
            T = np.array([temperature(int(s), N, cfg.t_min, cfg.t_max) for s in steps])
            rows = lambda a: np.repeat(a, L)
            st = stats(z, rows(T), rows(np.array([cfg.seed(int(c)) for c in act], dtype=np.uint64)), rows(blocks),
                       rows(steps), np.tile(np.arange(L, dtype=np.int32), act.size))
            n = act.size
            rec = TickRecord(tick=self.tick_no, canvases=act, block=blocks, step=steps, T=T, stats=st,
                             mean_H=np.zeros(n), converged=np.zeros(n, bool), final=np.zeros(n, bool),
                             accepted=np.zeros((n, L), bool), n_accepted=np.zeros(n, np.int32),
                             flag_y=st["ggap"] < cfg.margin_gap, flag_amax=st["zgap"] < cfg.margin_gap,
                             flag_commit=np.zeros((n, L), bool), flag_canvas=np.zeros(n, bool),
                             n_remasked=np.zeros(n, np.int32))
            for i, c in enumerate(act):
                self._commit(int(c), st[i * L:(i + 1) * L], rec, i, draw_u32, uniform_token, PURPOSE_RENOISE)
        self.tick_no += 1
        self._admit(self.tick_no)
        return rec

    def _commit(self, c, st, rec, i, draw_u32, uniform_token, PURPOSE_RENOISE):
        cfg = self.cfg
        L, V, N = cfg.canvas_len, cfg.vocab, cfg.num_inference_steps
        s, b = int(self.step_no[c]), int(self.block[c])
        H, y, amax = st["H"], st["y"], st["amax"]
        mean_H = float(np.mean(H))
        rec.mean_H[i] = mean_H
        # early stop: confident (mean entropy below the threshold) and stable (the argmax canvas
        # unchanged from the previous step's for `stability` steps in a row; none before step 1)
        run = int(self.stable_run[c]) + 1 if (s >= 1 and bool(np.all(amax == self.prev_amax[c]))) else 0
        converged = run >= cfg.stability and mean_H < cfg.confidence
        if s >= 1 and (abs(mean_H - cfg.confidence) < cfg.margin_H or
                       (mean_H < cfg.confidence + cfg.margin_H and bool(np.any(rec.flag_amax[i * L:(i + 1) * L])))):
            rec.flag_canvas[i] = True
        final = converged or s == N - 1
        rec.converged[i], rec.final[i] = converged, final
        reaccept = cfg.mode == "reaccept"
        assert cfg.mode in ("freeze", "reaccept"), cfg.mode
        # the open positions: under "reaccept" every position, else the uncommitted ones
        unc = np.arange(L) if reaccept else np.nonzero(~self.committed[c])[0]
        if not final:
            order, excl, k = entropy_bounded_accept(H, unc, cfg.entropy_bound)
            acc = np.array(order[:k], dtype=np.int64)
            # near-tie flags: a prefix sum within margin of the bound, or entropies across the boundary within margin
            for j in (k - 1, k):
                if 1 <= j < len(order) and abs(excl[j] - cfg.entropy_bound) < cfg.margin_H:
                    rec.flag_canvas[i] = True
            if k < len(order):
                h_last_acc, h_first_rej = H[order[k - 1]], H[order[k]]
                for p in order[:k]:
                    if H[p] > h_first_rej - cfg.margin_H:
                        rec.flag_commit[i, p] = True
                for p in order[k:]:
                    if H[p] < h_last_acc + cfg.margin_H:
                        rec.flag_commit[i, p] = True
            if reaccept:
                was = self.committed[c].copy()
                self.committed[c] = False
            self.x[c, acc] = y[acc]
            self.committed[c, acc] = True
            self.commit_step[c, acc] = s
            rec.accepted[i, acc] = True
            rec.n_accepted[i] = k
            if reaccept:
                rec.n_remasked[i] = int(np.sum(was & ~self.committed[c]))
            # uniform re-noise of every open position not accepted
            for p in unc:
                if not self.committed[c, p]:
                    self.x[c, p] = uniform_token(draw_u32(cfg.seed(c), PURPOSE_RENOISE, b, s, int(p)), V)
            self.prev_amax[c] = amax
            self.stable_run[c] = run
            self.step_no[c] = s + 1
        else:
            # finish the block: every remaining position takes its sample
            self.x[c, unc] = y[unc]
            self.committed[c, unc] = True
            self.commit_step[c, unc] = s
            rec.accepted[i, unc] = True
            rec.n_accepted[i] = unc.size
            self.tokens_out[c, b] = self.x[c]
            self.commit_steps_out[c, b] = self.commit_step[c]
            self.steps_used[c] += s + 1
            self.converged_blocks[c] += int(converged)
            self.stable_run[c] = 0  # the count restarts with each block (and stays 0 once done)
            if b + 1 < cfg.gen_blocks:
                self._init_canvas(c, b + 1)
            else:
                self.status[c] = DONE

    def run(self, resid_fn: Callable, max_ticks: int = 1 << 30, on_tick: Optional[Callable] = None):
        while not self.done() and self.tick_no < max_ticks:
            rec = self.tick(resid_fn)
            if on_tick is not None and rec is not None:
                on_tick(rec)
        return self.tokens_out


def synth_resid_fn(cfg: OracleConfig, W_bf16: np.ndarray, sigma: float) -> Callable:
    """Residual supplier built on the shared seeded generator ``synth``."""
    import synth

    def fn(canvases, blocks, steps, tokens):
        L = cfg.canvas_len
        n = canvases.size
        return synth.resid_rows(np.repeat([cfg.seed(int(c)) for c in canvases], L).astype(np.uint64),
                                np.repeat(blocks, L), np.repeat(steps, L), np.tile(np.arange(L), n),
                                tokens.reshape(-1), W_bf16, sigma)

    return fn
