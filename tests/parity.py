"""Parity harness: the CUDA path against the CPU oracle on the same seeded inputs.

Inputs (W_vocab and the per-step residual rows) come from ``synth`` only.  For
a teacher-forced tick the oracle's state before the tick is loaded into the
CUDA sampler (dg_set_state), both sides run the tick on the same residual, and
every output is compared:

  entropy H       |H_gpu - H_oracle| <= 1e-3 nats            (task tolerance)
  log Z           |dlogZ| <= 1e-3 |logZ|                      (task tolerance)
  sample, argmax  bit-exact unless the oracle's top-2 gap < 1e-4 (flagged)
  state after     tokens / committed / commit_step bit-exact except flagged
                  positions (sample near-tie on an accepted position, or an
                  entropy within 1e-3 nats of the other side of the accept
                  boundary) and flagged canvases (a prefix sum within 1e-3 of
                  the bound, or the early-stop test within 1e-3 of its
                  threshold)

Nothing the CUDA path produces is fed to the oracle.
"""
from __future__ import annotations

import dataclasses
import os

import numpy as np

import oracle
import synth
from oracle.sampler import ACTIVE, DONE, WAITING, OracleConfig, OracleSampler

TOL_H = 1e-3
TOL_LOGZ_REL = 1e-3


def f32(x: float) -> float:
    """The fp32 value the C ABI will hold for a config float."""
    return float(np.float32(x))


@dataclasses.dataclass
class Case:
    vocab: int
    hidden: int
    canvas_len: int
    n_canvases: int = 1
    gen_blocks: int = 1
    steps: int = 48
    t_min: float = 0.4
    t_max: float = 0.8
    bound: float = 0.1
    conf: float = 0.005
    sigma: float = 0.5
    sigma_w: float = 0.02
    w_seed: int = 0
    seeds: tuple = None
    admit: tuple = None
    max_active: int = 0
    norm_seed: int = None  # RMSNorm weight from synth.norm_weight, or all ones
    rms_eps: float = 1e-6
    mode: str = "freeze"  # commit mode: "freeze" (DG_FREEZE) or "reaccept" (DG_REACCEPT)
    softcap: float = 0.0  # final logit softcap c (0 = off)
    stability: int = 1  # steps in a row with an unchanged argmax canvas needed for an early stop

    def oracle_cfg(self) -> OracleConfig:
        return OracleConfig(vocab=self.vocab, hidden=self.hidden, canvas_len=self.canvas_len,
                            n_canvases=self.n_canvases, gen_blocks=self.gen_blocks, num_inference_steps=self.steps,
                            t_min=f32(self.t_min), t_max=f32(self.t_max), entropy_bound=f32(self.bound),
                            confidence=f32(self.conf), rms_eps=f32(self.rms_eps),
                            seeds=list(self.seeds) if self.seeds else list(range(self.n_canvases)),
                            admit_tick=list(self.admit) if self.admit else None,
                            max_active=self.max_active or None, mode=self.mode, softcap=f32(self.softcap),
                            stability=self.stability)

    def gpu_cfg(self):
        import uniform_state_discrete_gb300 as dg
        return dg.make_config(self.vocab, self.hidden, self.canvas_len, n_canvases=self.n_canvases,
                              gen_blocks=self.gen_blocks, num_inference_steps=self.steps, t_min=self.t_min,
                              t_max=self.t_max, entropy_bound=self.bound, confidence=self.conf, rms_eps=self.rms_eps,
                              max_active=self.max_active,
                              mode=dg.DG_REACCEPT if self.mode == "reaccept" else dg.DG_FREEZE, softcap=self.softcap,
                              stability=self.stability,
                              seeds=list(self.seeds) if self.seeds else list(range(self.n_canvases)),
                              admit_tick=list(self.admit) if self.admit else None)


def weights(case: Case) -> np.ndarray:
    return synth.wvocab(case.w_seed, case.vocab, case.hidden, sigma_w=case.sigma_w)


def norm_w(case: Case):
    return None if case.norm_seed is None else synth.norm_weight(case.norm_seed, case.hidden)


def resid_slots(case: Case, ocfg: OracleConfig, W: np.ndarray, canvases, blocks, steps, tokens) -> np.ndarray:
    """Residual rows for the given canvases, placed in the [B, L, d] slot layout the ABI reads."""
    full = np.zeros((case.n_canvases, case.canvas_len, case.hidden), np.float32)
    rows = oracle.sampler.synth_resid_fn(ocfg, W, case.sigma)(np.asarray(canvases), np.asarray(blocks),
                                                              np.asarray(steps), np.asarray(tokens))
    full[np.asarray(canvases)] = rows.reshape(len(canvases), case.canvas_len, case.hidden)
    return full


def oracle_state_to_gpu(o: OracleSampler, case: Case) -> dict:
    import uniform_state_discrete_gb300 as dg
    B = case.n_canvases
    slots = np.zeros(B, dg.SLOT_DTYPE)
    slots["state"] = o.status
    slots["block"] = o.block
    slots["step"] = o.step_no
    slots["n_committed"] = o.committed.sum(axis=1)
    slots["steps_used"] = o.steps_used
    slots["converged_blocks"] = o.converged_blocks
    slots["stable_steps"] = o.stable_run
    return {"tick": o.tick_no, "slots": slots, "tokens": o.x.astype(np.int32),
            "committed": o.committed.astype(np.uint8), "commit_step": o.commit_step.astype(np.int16),
            "prev_argmax": o.prev_amax.astype(np.int32), "tokens_out": o.tokens_out.astype(np.int32),
            "commit_steps_out": o.commit_steps_out.astype(np.int16)}


@dataclasses.dataclass
class Report:
    ticks: int = 0
    positions: int = 0
    max_dH: float = 0.0
    max_dlogZ_rel: float = 0.0
    y_mismatch: int = 0
    y_flagged: int = 0
    amax_mismatch: int = 0
    amax_flagged: int = 0
    state_mismatch_unflagged: int = 0
    state_flagged_positions: int = 0
    canvas_flagged: int = 0
    errors: list = dataclasses.field(default_factory=list)

    def ok(self) -> bool:
        return not self.errors


def teacher_forced(case: Case, ticks: int = 1 << 30, gpu=None, W=None, check_every: int = 1) -> Report:
    """Run the oracle free; before each checked tick load its state into the CUDA sampler, run both
    on the same residual and compare.  Returns a Report; ``errors`` lists every violation."""
    import torch
    import uniform_state_discrete_gb300 as dg
    W = weights(case) if W is None else W
    ocfg = case.oracle_cfg()
    nw = norm_w(case)
    o = OracleSampler(ocfg, W, norm_w=nw)
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    s = gpu or dg.Sampler(case.gpu_cfg(), w_dev, norm_w=None if nw is None else torch.from_numpy(nw).to(dev))
    rep = Report()
    L = case.canvas_len
    t = 0
    while not o.done() and t < ticks:
        act = o.active()
        check = (t % check_every == 0) or o.step_no[act].max(initial=0) >= case.steps - 1
        resid = resid_slots(case, ocfg, W, act, o.block[act], o.step_no[act], o.x[act]) if act.size else None
        if check and act.size:
            s.set_state(oracle_state_to_gpu(o, case))
            s.step(torch.from_numpy(resid).to(dev))
        rec = o.tick(lambda canv, blocks, steps, tok: resid[canv].reshape(-1, case.hidden))
        if check and rec is not None:
            compare_tick(s, o, rec, case, rep)
        t += 1
    return rep


def compare_tick(s, o: OracleSampler, rec, case: Case, rep: Report, cmap=None):
    """Compare the CUDA sampler's outputs and state after a tick with the oracle's.  ``cmap`` maps an
    oracle canvas to the CUDA sampler's canvas (default: the same index)."""
    L = case.canvas_len
    H_all = s.entropy().cpu().numpy()
    lz_all = s.logz().cpu().numpy()
    y_all = s.sample().cpu().numpy()
    am_all = s.argmax().cpu().numpy()
    gst_all = s.get_state()
    rep.ticks += 1
    for i, c in enumerate(rec.canvases):
        g = c if cmap is None else cmap[int(c)]
        H, lz, y, am = {c: H_all[g]}, {c: lz_all[g]}, {c: y_all[g]}, {c: am_all[g]}
        gst = {k: ({c: v[g]} if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == case.n_canvases
                   else v) for k, v in gst_all.items()}
        st = rec.stats[i * L:(i + 1) * L]
        rep.positions += L
        dH = np.abs(H[c].astype(np.float64) - st["H"])
        dZ = np.abs(lz[c].astype(np.float64) - st["logZ"]) / np.maximum(np.abs(st["logZ"]), 1e-30)
        rep.max_dH = max(rep.max_dH, float(dH.max()))
        rep.max_dlogZ_rel = max(rep.max_dlogZ_rel, float(dZ.max()))
        if dH.max() > TOL_H:
            rep.errors.append(f"tick {rec.tick} canvas {c}: |dH| {dH.max():.3g} > {TOL_H}")
        if dZ.max() > TOL_LOGZ_REL:
            rep.errors.append(f"tick {rec.tick} canvas {c}: |dlogZ|/|logZ| {dZ.max():.3g} > {TOL_LOGZ_REL}")
        fy = rec.flag_y[i * L:(i + 1) * L]
        fa = rec.flag_amax[i * L:(i + 1) * L]
        ym = y[c] != st["y"]
        amm = am[c] != st["amax"]
        rep.y_mismatch += int(ym.sum())
        rep.y_flagged += int(fy.sum())
        rep.amax_mismatch += int(amm.sum())
        rep.amax_flagged += int(fa.sum())
        if np.any(ym & ~fy):
            rep.errors.append(f"tick {rec.tick} canvas {c}: sample differs at unflagged positions "
                              f"{np.nonzero(ym & ~fy)[0][:8].tolist()}")
        if np.any(amm & ~fa):
            rep.errors.append(f"tick {rec.tick} canvas {c}: argmax differs at unflagged positions "
                              f"{np.nonzero(amm & ~fa)[0][:8].tolist()}")
        if rec.flag_canvas[i]:
            rep.canvas_flagged += 1
            continue
        # state after the tick
        pos_flag = rec.flag_commit[i] | (rec.accepted[i] & fy)
        rep.state_flagged_positions += int(pos_flag.sum())
        for name, gv, ov in (("tokens", gst["tokens"][c], o.x[c]), ("committed", gst["committed"][c],
                                                                     o.committed[c].astype(np.uint8)),
                             ("commit_step", gst["commit_step"][c], o.commit_step[c])):
            bad = (gv != ov) & ~pos_flag
            if rec.final[i] and not np.any(pos_flag):
                bad = gv != ov
            if np.any(bad):
                rep.state_mismatch_unflagged += int(bad.sum())
                rep.errors.append(f"tick {rec.tick} canvas {c}: {name} differs at {np.nonzero(bad)[0][:8].tolist()}")
        if not np.any(pos_flag):
            gs = gst["slots"][c]
            for fld, ov in (("state", o.status[c]), ("block", o.block[c]), ("step", o.step_no[c]),
                            ("steps_used", o.steps_used[c]), ("converged_blocks", o.converged_blocks[c]),
                            ("n_committed", o.committed[c].sum()), ("n_remasked", rec.n_remasked[i]),
                            ("stable_steps", o.stable_run[c])):
                if int(gs[fld]) != int(ov):
                    rep.errors.append(f"tick {rec.tick} canvas {c}: slot {fld} {int(gs[fld])} != oracle {int(ov)}")
            if rec.final[i]:
                b = rec.block[i]
                if not np.array_equal(gst["tokens_out"][c][b], o.tokens_out[c, b]):
                    rep.errors.append(f"tick {rec.tick} canvas {c}: finished block tokens differ")
                if not np.array_equal(gst["commit_steps_out"][c][b], o.commit_steps_out[c, b]):
                    rep.errors.append(f"tick {rec.tick} canvas {c}: finished block commit heatmap differs")


# --------------------------------------------------------------------------- stored oracle states
STATES_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "model_scale_states.npz")
STATE_FIELDS = ("x", "committed", "commit_step", "prev_amax", "stable_run", "step_no", "block", "status",
                "steps_used", "converged_blocks")
_STATES = {}


def _load_states() -> dict:
    if not _STATES:
        with np.load(STATES_PATH) as z:
            for k in z.files:
                traj, step, field = k.split("/")
                _STATES.setdefault(traj, {}).setdefault(step, {})[field] = z[k]
    return _STATES


def stored_state(name: str, key: str) -> dict:
    """One canvas's oracle state before a tick, as written by tests/golden/make_model_scale_states.py
    (``key`` is "s<step>" or "stop")."""
    return {f: np.array(v) for f, v in _load_states()[name][key].items()}


def stored_keys(name: str) -> list:
    """The states stored for one trajectory ("s<step>" and, where its early stop fired, "stop")."""
    return sorted(_load_states().get(name, {}))


def init_state(case: Case, c: int, block: int = 0, step: int = 0) -> dict:
    """Canvas c at the start of a block (its uniform initial canvas), as the oracle draws it; the slot
    step may be set past 0 for a stand-in canvas whose outputs are not compared."""
    cfg = case.oracle_cfg()
    L = case.canvas_len
    x = np.array([oracle.uniform_token(oracle.draw_u32(cfg.seed(c), oracle.PURPOSE_INIT, block, 0, p), case.vocab)
                  for p in range(L)], dtype=np.int32)
    return {"x": x, "committed": np.zeros(L, bool), "commit_step": np.full(L, -1, np.int16),
            "prev_amax": np.zeros(L, np.int32), "stable_run": np.array(0), "step_no": np.array(step),
            "block": np.array(block), "status": np.array(ACTIVE), "steps_used": np.array(0),
            "converged_blocks": np.array(0)}


def oracle_from_state(case: Case, W: np.ndarray, c: int, st: dict, tick: int) -> OracleSampler:
    """A one-canvas oracle for canvas c of the case (its seed and knobs), holding the state ``st``."""
    cfg = dataclasses.replace(case.oracle_cfg(), n_canvases=1, seeds=[case.oracle_cfg().seed(c)], admit_tick=None,
                              max_active=None)
    o = OracleSampler(cfg, W)
    for f in STATE_FIELDS:
        getattr(o, f)[0] = st[f]
    o.tick_no = tick
    return o


def batch_state(case: Case, states: dict, tick: int) -> dict:
    """The CUDA sampler's state for a whole batch: ``states[c]`` is canvas c's state (fields of
    STATE_FIELDS); canvases not listed wait for admission."""
    import uniform_state_discrete_gb300 as dg
    B, L, G = case.n_canvases, case.canvas_len, case.gen_blocks
    slots = np.zeros(B, dg.SLOT_DTYPE)
    out = {"tick": tick, "slots": slots, "tokens": np.zeros((B, L), np.int32),
           "committed": np.zeros((B, L), np.uint8), "commit_step": np.full((B, L), -1, np.int16),
           "prev_argmax": np.zeros((B, L), np.int32), "tokens_out": np.zeros((B, G, L), np.int32),
           "commit_steps_out": np.zeros((B, G, L), np.int16)}
    slots["state"] = WAITING
    for c, st in states.items():
        slots["state"][c] = int(st["status"])
        slots["block"][c] = int(st["block"])
        slots["step"][c] = int(st["step_no"])
        slots["n_committed"][c] = int(np.sum(st["committed"]))
        slots["steps_used"][c] = int(st["steps_used"])
        slots["converged_blocks"][c] = int(st["converged_blocks"])
        slots["stable_steps"][c] = int(st["stable_run"])
        out["tokens"][c] = st["x"]
        out["committed"][c] = np.asarray(st["committed"], bool).astype(np.uint8)
        out["commit_step"][c] = st["commit_step"]
        out["prev_argmax"][c] = st["prev_amax"]
    return out


def tick_from_states(s, case: Case, W: np.ndarray, states: dict, tick: int, check, rep: Report):
    """Load a batch state into the CUDA sampler, run one tick of it on synth's residual rows, and
    compare the canvases in ``check`` with one-canvas oracles started from the same states."""
    import torch
    ocfg = case.oracle_cfg()
    act = np.array(sorted(c for c, st in states.items() if int(st["status"]) == ACTIVE))
    resid = resid_slots(case, ocfg, W, act, [int(states[c]["block"]) for c in act],
                        [int(states[c]["step_no"]) for c in act], np.stack([states[c]["x"] for c in act]))
    s.set_state(batch_state(case, states, tick))
    s.step(torch.from_numpy(resid).to(getattr(s, "device", "cuda:0")))
    for c in check:
        o = oracle_from_state(case, W, c, states[c], tick)
        rec = o.tick(lambda canv, blocks, steps, tok: resid[c].reshape(-1, case.hidden))
        compare_tick(s, o, rec, case, rep, cmap={0: c})
