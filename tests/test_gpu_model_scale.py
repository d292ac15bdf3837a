"""Teacher-forced parity at model scale (V = 2^18, d = 2816): the single canvas, the staggered batch
of 16 canvases and every point of the 64-canvas stress sweep, across the temperature schedule.

Each check loads oracle states into the CUDA sampler (dg_set_state) -- states the oracle reached
itself, stored by tests/golden/make_model_scale_states.py, or initial canvases -- runs one tick of
the whole batch in the launch configuration of its workload, and compares the checked canvases
with one-canvas oracles started from the same states (tests/parity.py, compare_tick): entropy within
1e-3 nats, log Z within 1e-3 relative, sample, argmax, committed mask, tokens, commit steps and
slot counters bit-exact outside the flagged near-ties.
"""
import numpy as np
import pytest

import synth

from parity import DONE, Case, Report, init_state, stored_keys, stored_state, tick_from_states

pytestmark = pytest.mark.gpu

V, D, L, N = 262144, 2816, 256, 48
_W = {}


def _weights():
    if "w" not in _W:
        _W["w"] = synth.wvocab(0, V, D)
    return _W["w"]


def _sampler(case):
    import torch
    import uniform_state_discrete_gb300 as dg
    W = _weights()
    w_dev = torch.from_numpy(W.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    return dg.Sampler(case.gpu_cfg(), w_dev), w_dev


def _report(rep, label):
    print(f"\n[{label}] ticks={rep.ticks} positions={rep.positions} max|dH|={rep.max_dH:.3g} "
          f"max|dlogZ|/|logZ|={rep.max_dlogZ_rel:.3g} y mismatch={rep.y_mismatch} (flagged {rep.y_flagged}) "
          f"argmax mismatch={rep.amax_mismatch} (flagged {rep.amax_flagged}) "
          f"flagged positions={rep.state_flagged_positions} flagged canvases={rep.canvas_flagged}")
    assert rep.ticks > 0
    assert rep.ok(), "\n".join(rep.errors[:20])


def _with_seed_state(st: dict) -> dict:
    return {k: np.array(v) for k, v in st.items()}


def test_single_canvas_across_the_schedule():
    """1 canvas x 256 positions (the single-canvas model-scale configuration): steps 0, 1, 16, 32 and
    the last two, where the temperature has cooled to 0.408 and the final step commits the rest."""
    case = Case(vocab=V, hidden=D, canvas_len=L, steps=N, seeds=(0,))
    s, _ = _sampler(case)
    W = _weights()
    rep = Report()
    name = "b0.1_t0.8-0.4_s0.5_seed0"
    for key in ("s0", "s1", "s16", "s32", "s46", "s47"):
        st = init_state(case, 0) if key == "s0" else stored_state(name, key)
        tick_from_states(s, case, W, {0: st}, int(st["step_no"]), [0], rep)
    s.close()
    _report(rep, "1 canvas, V=2^18")
    assert rep.ticks == 6


def test_batched_staggered_admission_across_the_schedule():
    """16 canvases x 256 positions, seeds 0..15 admitted at ticks 0, 12, 24, 36: at each checked tick
    the batch holds exactly the canvases the staggered schedule has running (4 to 16, one 256-row
    pair tile each), finished canvases done and later ones waiting; canvas 0 is checked along its
    whole block and the canvases of each later group at their admission and later."""
    B = 16
    admit = tuple(12 * (c // 4) for c in range(B))
    case = Case(vocab=V, hidden=D, canvas_len=L, n_canvases=B, steps=N, seeds=tuple(range(B)), admit=admit)
    s, _ = _sampler(case)
    W = _weights()
    traj = "b0.1_t0.8-0.4_s0.5_seed{}"
    # tick -> {canvas: state key} for the checked canvases ("s0": initial canvas)
    plan = {0: {0: "s0", 3: "s0"}, 12: {0: "s12", 4: "s0"}, 24: {0: "s24", 4: "s12", 8: "s0"},
            36: {0: "s36", 8: "s12", 12: "s0"}, 47: {0: "s47", 12: "s11"}, 48: {4: "s36"}, 83: {12: "s47"}}
    rep = Report()
    for tick, checked in plan.items():
        states = {}
        for c in range(B):
            step = tick - admit[c]
            if step < 0:
                continue  # waiting for admission
            if step >= N:
                states[c] = dict(init_state(case, c), status=np.array(DONE), steps_used=np.array(N))
                continue
            key = checked.get(c)
            if key is None:
                states[c] = init_state(case, c, step=step)  # a running stand-in, not compared
            elif key == "s0":
                states[c] = init_state(case, c)
            else:
                states[c] = stored_state(traj.format(c), key)
            assert int(states[c]["step_no"]) == step
        tick_from_states(s, case, W, states, tick, sorted(checked), rep)
    s.close()
    _report(rep, "16 canvases staggered")


@pytest.mark.parametrize("sigma", [0.1, 2.0])
@pytest.mark.parametrize("t_max,t_min", [(0.8, 0.4), (1.5, 0.1)])
@pytest.mark.parametrize("bound", [0.01, 0.1, 1.0])
def test_stress_sweep_point_across_the_schedule(bound, t_max, t_min, sigma):
    """64 canvases x 4 blocks x 256 positions at one point of the stress sweep, all 64 canvases
    running (64 pair tiles per vocabulary chunk): the first tick, steps 8, 24 and 47 of block 0 that
    the run reaches, the tick at which the early-stop test ends the block (where it fires), and the
    first tick of block 1.  Canvas 0 is checked throughout and canvas 63 (the last row tile) at the
    first tick and at the early stop; the other canvases hold canvas 0's state under their own seeds."""
    B, G = 64, 4
    case = Case(vocab=V, hidden=D, canvas_len=L, n_canvases=B, gen_blocks=G, steps=N, bound=bound, t_max=t_max,
                t_min=t_min, sigma=sigma, seeds=tuple(range(B)))
    s, _ = _sampler(case)
    W = _weights()
    name = f"b{bound}_t{t_max}-{t_min}_s{sigma}_seed0"
    keys = stored_keys(name)
    assert keys, f"no stored oracle states for {name}"
    rep = Report()
    # the first tick: every canvas at its own initial canvas
    tick_from_states(s, case, W, {c: init_state(case, c) for c in range(B)}, 0, [0, B - 1], rep)
    for key in keys:
        st = stored_state(name, key)
        states = {c: _with_seed_state(st) for c in range(B)}
        tick_from_states(s, case, W, states, int(st["step_no"]), [0, B - 1] if key == "stop" else [0], rep)
    # the first tick of block 1 (block 0 finished and frozen)
    tick_from_states(s, case, W, {c: dict(init_state(case, c, block=1), steps_used=np.array(N)) for c in range(B)},
                     N, [0], rep)
    s.close()
    _report(rep, f"stress bound={bound} t={t_max}->{t_min} sigma={sigma} ({', '.join(keys)})")
    if sigma == 0.1 and bound == 1.0:
        assert "stop" in keys  # peaked distributions stop early
