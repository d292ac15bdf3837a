"""Write ``model_scale_states.npz``: CPU-oracle states of model-scale runs, for teacher forcing.

A teacher-forced parity check loads the oracle's state before a tick into the CUDA sampler and
compares the tick's outputs.  Reaching the state before step 47 of a model-scale canvas
(V = 2^18, d = 2816) takes the oracle 47 ticks of a full fp64 LM head, minutes of CPU time per
canvas, so the states the GPU tests start from are written here once.  At test time the oracle
recomputes each checked tick itself from the stored state; only the states before those ticks
are stored.

Every value comes from ``oracle`` and ``synth`` alone: each trajectory is one canvas run free by
``oracle.OracleSampler`` on the residual rows of ``synth`` (r = W[x_p] + sigma n), the pages'
knobs (canvas 256, V = 2^18, N = 48, confidence 0.005; "DiffusionGemma Denoise" node, "Inputs")
and the configuration's temperature, bound and hidden noise.  Trajectories:

  canvas seeds 0, 4, 8, 12 at sigma 0.5, t 0.8 -> 0.4, bound 0.1 (the single-canvas model-scale
      configuration and canvases of the batched one);
  seed 0 at each of the 12 points of the stress sweep: bound in {0.01, 0.1, 1.0},
      (t_max, t_min) in {(0.8, 0.4), (1.5, 0.1)}, sigma in {0.1, 2.0};

each stored before the listed steps of block 0 that the run reaches, and, where the early-stop
test ends the block, before that tick ("stop").

    python tests/golden/make_model_scale_states.py [--only NAME] [--out PATH]
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

V, D, L, N = 262144, 2816, 256, 48
OUT = os.path.join(HERE, "model_scale_states.npz")
FIELDS = ("x", "committed", "commit_step", "prev_amax", "stable_run", "step_no", "block", "status", "steps_used",
          "converged_blocks")


def trajectories() -> dict:
    t = {}
    for seed, steps in ((0, (1, 12, 16, 24, 32, 36, 46, 47)), (4, (12, 36)), (8, (12,)), (12, (11, 47))):
        t[f"b0.1_t0.8-0.4_s0.5_seed{seed}"] = dict(seed=seed, bound=0.1, t_max=0.8, t_min=0.4, sigma=0.5,
                                                  steps=steps)
    for bound in (0.01, 0.1, 1.0):
        for t_max, t_min in ((0.8, 0.4), (1.5, 0.1)):
            for sigma in (0.1, 2.0):
                t[f"b{bound}_t{t_max}-{t_min}_s{sigma}_seed0"] = dict(seed=0, bound=bound, t_max=t_max, t_min=t_min,
                                                                      sigma=sigma, steps=(8, 24, 47))
    return t


def run_one(name: str, spec: dict, W: np.ndarray) -> dict:
    import oracle
    f32 = lambda x: float(np.float32(x))
    cfg = oracle.OracleConfig(vocab=V, hidden=D, canvas_len=L, n_canvases=1, gen_blocks=1, num_inference_steps=N,
                              t_min=f32(spec["t_min"]), t_max=f32(spec["t_max"]), entropy_bound=f32(spec["bound"]),
                              confidence=f32(0.005), rms_eps=f32(1e-6), seeds=[spec["seed"]])
    o = oracle.OracleSampler(cfg, W)
    fn = oracle.sampler.synth_resid_fn(cfg, W, spec["sigma"])
    want = set(spec["steps"])
    out = {}
    t0 = time.time()
    while not o.done():
        s = int(o.step_no[0])
        pre = {f: np.array(getattr(o, f)[0]).copy() for f in FIELDS}
        if s in want:
            out[f"{name}/s{s}"] = pre
        rec = o.tick(fn)
        if rec is not None and rec.converged[0]:
            out[f"{name}/stop"] = dict(pre, stop_step=np.array(s))
    print(f"{name}: {o.steps_used[0]} steps, converged {int(o.converged_blocks[0])}, stored "
          f"{sorted(k.split('/')[1] for k in out)} in {time.time() - t0:.0f} s", flush=True)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", default=None, help="write only the trajectories whose name contains this")
    ap.add_argument("--out", default=OUT)
    args = ap.parse_args()
    import synth
    W = synth.wvocab(0, V, D)
    arrays = {}
    if os.path.exists(args.out) and args.only:
        with np.load(args.out) as z:
            arrays = {k: z[k] for k in z.files}
    for name, spec in trajectories().items():
        if args.only and args.only not in name:
            continue
        arrays = {k: v for k, v in arrays.items() if not k.startswith(name + "/")}
        for key, st in run_one(name, spec, W).items():
            for f, v in st.items():
                arrays[f"{key}/{f}"] = v
    tmp = args.out + ".tmp.npz"
    np.savez_compressed(tmp, **arrays)
    os.replace(tmp, args.out)


if __name__ == "__main__":
    main()
