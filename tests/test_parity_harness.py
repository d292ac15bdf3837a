"""The parity harness itself, on the CPU: a stand-in sampler whose ticks are computed by a second
copy of the oracle must pass every comparison of tests/parity.py, and one with a planted
difference must fail them.  This checks the harness's bookkeeping (state loading, canvas
mapping, flag rules), not the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
from oracle.sampler import OracleSampler
from parity import Case, Report, batch_state, compare_tick, init_state, tick_from_states, weights


class OracleBackedSampler:
    """Implements the parts of the CUDA sampler's Python API the harness uses, on the CPU."""
    device = "cpu"

    def __init__(self, case: Case, W: np.ndarray, plant=None):
        import uniform_state_discrete_gb300 as dg
        self.dg, self.case, self.plant = dg, case, plant
        self.o = OracleSampler(case.oracle_cfg(), W)
        B, L = case.n_canvases, case.canvas_len
        self.out = {k: np.zeros((B, L), dt) for k, dt in (("H", np.float32), ("logZ", np.float32), ("y", np.int32),
                                                            ("amax", np.int32))}
        self.remasked = np.zeros(B, np.int32)

    def set_state(self, st):
        o, sl = self.o, st["slots"]
        o.status[:], o.block[:], o.step_no[:] = sl["state"], sl["block"], sl["step"]
        o.steps_used[:], o.converged_blocks[:], o.stable_run[:] = sl["steps_used"], sl["converged_blocks"], \
            sl["stable_steps"]
        o.x[:], o.committed[:], o.commit_step[:] = st["tokens"], st["committed"] != 0, st["commit_step"]
        o.prev_amax[:], o.tokens_out[:], o.commit_steps_out[:] = st["prev_argmax"], st["tokens_out"], \
            st["commit_steps_out"]
        o.tick_no = int(st["tick"])

    def step(self, resid):
        r = resid.numpy()
        rec = self.o.tick(lambda canv, blocks, steps, tok: r[canv].reshape(-1, self.case.hidden))
        L = self.case.canvas_len
        for i, c in enumerate(rec.canvases):
            st = rec.stats[i * L:(i + 1) * L]
            self.out["H"][c], self.out["logZ"][c] = st["H"], st["logZ"]
            self.out["y"][c], self.out["amax"][c] = st["y"], st["amax"]
            self.remasked[c] = rec.n_remasked[i]
        if self.plant == "token":
            c = int(rec.canvases[-1])
            self.o.x[c, 3] = (self.o.x[c, 3] + 1) % self.case.vocab

    def entropy(self):
        return torch.from_numpy(self.out["H"].copy())

    def logz(self):
        return torch.from_numpy(self.out["logZ"].copy())

    def sample(self):
        return torch.from_numpy(self.out["y"].copy())

    def argmax(self):
        return torch.from_numpy(self.out["amax"].copy())

    def get_state(self):
        o, B = self.o, self.case.n_canvases
        slots = np.zeros(B, self.dg.SLOT_DTYPE)
        slots["state"], slots["block"], slots["step"] = o.status, o.block, o.step_no
        slots["n_committed"] = o.committed.sum(axis=1)
        slots["steps_used"], slots["converged_blocks"] = o.steps_used, o.converged_blocks
        slots["stable_steps"], slots["n_remasked"] = o.stable_run, self.remasked
        return {"tick": o.tick_no, "slots": slots, "tokens": o.x.copy(), "committed": o.committed.astype(np.uint8),
                "commit_step": o.commit_step.copy(), "prev_argmax": o.prev_amax.copy(),
                "tokens_out": o.tokens_out.copy(), "commit_steps_out": o.commit_steps_out.copy()}


def _staggered_case():
    return Case(vocab=512, hidden=64, canvas_len=16, n_canvases=6, gen_blocks=2, steps=5, seeds=tuple(range(6)),
                admit=(0, 0, 2, 2, 4, 4), sigma=0.3, bound=0.5)


def _run_states(plant):
    case = _staggered_case()
    W = weights(case)
    s = OracleBackedSampler(case, W, plant=plant)
    # a free oracle run supplies the states the checks start from
    ref = OracleSampler(case.oracle_cfg(), W)
    fn = oracle.sampler.synth_resid_fn(case.oracle_cfg(), W, case.sigma)
    rep = Report()
    for tick in range(8):
        snap = ref.snapshot()
        states = {}
        for c in range(case.n_canvases):
            if snap["status"][c] == 0:
                continue
            states[c] = {"x": snap["x"][c], "committed": snap["committed"][c], "commit_step": snap["commit_step"][c],
                         "prev_amax": snap["prev_amax"][c], "stable_run": snap["stable_run"][c],
                         "step_no": snap["step_no"][c], "block": snap["block"][c], "status": snap["status"][c],
                         "steps_used": snap["steps_used"][c], "converged_blocks": snap["converged_blocks"][c]}
        active = [c for c, st in states.items() if int(st["status"]) == 1]
        if active:
            tick_from_states(s, case, W, states, tick, active[-2:], rep)
        ref.tick(fn)
    return rep


def test_harness_accepts_an_identical_sampler():
    rep = _run_states(plant=None)
    assert rep.ticks >= 6 and rep.ok(), rep.errors[:5]
    assert rep.max_dH < 1e-6


def test_harness_reports_a_planted_token_difference():
    rep = _run_states(plant="token")
    assert not rep.ok()
    assert any("tokens differ" in e for e in rep.errors)


def test_batch_state_round_trips_initial_canvases():
    case = _staggered_case()
    st = batch_state(case, {c: init_state(case, c) for c in (0, 2)}, 3)
    assert st["slots"]["state"].tolist() == [1, 0, 1, 0, 0, 0]
    for c in (0, 2):
        want = [oracle.uniform_token(oracle.draw_u32(c, oracle.PURPOSE_INIT, 0, 0, p), case.vocab) for p in range(16)]
        assert st["tokens"][c].tolist() == want
