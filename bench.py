#!/usr/bin/env python
"""Benchmark of the GB300 denoise step: canvas positions denoised per second.

One bench step is one tick of the whole hot path (RMSNorm -> tied LM head fused
with softmax statistics and the Gumbel-max sample -> split-vocabulary combine ->
entropy-bounded commit and uniform re-noise) over every active canvas, through
the C ABI (dg_denoise_step).  Inputs are synthetic and seeded (``synth``):
W_vocab ~ N(0, 0.02^2) in bf16 and, before every tick, the residual rows
W[x_p] + N(0, 0.5^2) built on the device from the current canvas (the backbone
stand-in, outside the timed kernels).

Timing: CUDA events on the sampler's stream around the four kernels of each
tick (device time); L2 is flushed by a 256 MB write before every timed tick,
outside the events.  ``e2e`` repeats the metric through dg_denoise_step_host
with the residual in pinned host memory: host->device copy, tick, and the
device->host read of the canvas and entropies inside the host-clocked window.
``roofline`` reports the LM-head kernel against the measured peaks;
``cpu_baseline`` times the CPU oracle on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle as the reference arm (rank 0 only).
Under torchrun each rank runs an independent replica (canvases seeded by rank);
the timed region is bracketed by a barrier and the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# OpenMP worker threads of the host-side input generator and the CPU oracle sleep as soon as a
# parallel region ends, instead of spinning on the cores the timed host steps run on (set before
# any OpenMP runtime loads; an explicit setting in the environment wins)
os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")

import numpy as np  # noqa: E402

METRIC = "canvas positions denoised/sec (LM head+entropy+commit); % of bf16/HBM roofline"
UNIT = "positions/s"
L2_FLUSH_BYTES = 256 << 20

# The workloads of the pages' sampler at the sizes this benchmark knows.  The default is the
# largest single-GPU configuration (the stress workload); the others are selectable.  Knobs not
# given take the pages' defaults: entropy_bound 0.1 nats, t 0.8 -> 0.4, hidden noise sigma 0.5.
WORKLOADS = {
    "stress64x4_v262k": dict(vocab=262144, hidden=2816, canvas_len=256, n_canvases=64, gen_blocks=4, steps=48,
                             bound=0.1, t_max=0.8, t_min=0.4, sigma=2.0,
                             text="stress: 64 canvases x gen_length 4 blocks x 256 positions (earlier blocks "
                                  "committed and frozen), V=262144, d=2816, bf16 W_vocab N(0,0.02^2), 48 steps per "
                                  "block; sweep point entropy_bound 0.1, t 0.8->0.4, hidden noise sigma 2.0"),
    "batched16_stagger_v262k": dict(vocab=262144, hidden=2816, canvas_len=256, n_canvases=16, gen_blocks=1, steps=48,
                                    admit=tuple(12 * (c // 4) for c in range(16)),
                                    text="batched: 16 canvases x 256 positions, V=262144, d=2816, seeds 0..15 "
                                         "admitted at ticks 0,12,24,36 (four per offset), 48 steps, t 0.8->0.4, "
                                         "entropy_bound 0.1, confidence 0.005"),
    "canvas256_v262k": dict(vocab=262144, hidden=2816, canvas_len=256, n_canvases=1, steps=48,
                            text="1 canvas x 256 positions, V=262144, d=2816 (model-scale LM head), bf16 W_vocab "
                                 "N(0,0.02^2), hidden W[x_p]+N(0,0.5^2), 48 steps, t 0.8->0.4, entropy_bound 0.1, "
                                 "confidence 0.005"),
    "canvas256_v32k": dict(vocab=32768, hidden=1024, canvas_len=256, n_canvases=1, steps=48,
                           text="1 canvas x 256 positions, V=32768, d=1024, bf16 W_vocab N(0,0.02^2), hidden "
                                "W[x_p]+N(0,0.5^2), 48 steps, T 0.8->0.4, entropy_bound 0.1, confidence 0.005"),
    "tiny": dict(vocab=2048, hidden=128, canvas_len=16, n_canvases=1, steps=8,
                 text="1 canvas x 16 positions, V=2048, d=128, 8 steps"),
    # the batched configuration with every canvas active from the first tick (4096 positions a tick)
    "batched16_v262k": dict(vocab=262144, hidden=2816, canvas_len=256, n_canvases=16, steps=48,
                            text="16 canvases x 256 positions, V=262144, d=2816, per-canvas seeds, all active"),
}
DEFAULT_WORKLOAD = "stress64x4_v262k"
SIGMA_HIDDEN = 0.5


def strip_comments(src: str) -> str:
    """C/CUDA source without its comments and blank lines (string literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':  # a string literal, escapes included
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_digest() -> str:
    """Digest of the LM-head kernel sources, comments left out; a stored ncu traffic figure is valid
    only for this digest."""
    h = hashlib.sha256()
    for rel in ("uniform_state_discrete_gb300/csrc/dg_lmhead.cu", "uniform_state_discrete_gb300/csrc/dg_internal.cuh",
                "uniform_state_discrete_gb300/csrc/dg_gumbel.cuh", "uniform_state_discrete_gb300/csrc/dg_norm.cuh",
                "uniform_state_discrete_gb300/csrc/dg_tc.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """DRAM bytes per LM-head launch from the committed ncu summary, if it matches the current kernel."""
    path = os.path.join(ROOT, "profiles", f"k_lmhead_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_digest") != kernel_source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def vocab_chunks(V: int) -> int:
    """Vocabulary chunks of the LM head: 256-column tiles, at most 76 chunks, the library's layout."""
    tiles = math.ceil(V / 256)
    per_chunk = math.ceil(tiles / min(tiles, 76))
    return math.ceil(tiles / per_chunk)


def lmhead_roofline(V: int, d: int, P: int, pair: bool, seconds: float, peaks: dict):
    """Roofline of one LM-head launch over P positions taking `seconds`.

    Algorithmic bytes: W once (V d bf16), the kernel's input rows (the fp32 residual and the norm
    weights when the SM-pair kernel forms the RMSNorm rows itself, else the bf16 rows h) and the
    32-byte partial records it writes (one per position and vocabulary chunk).  Algorithmic flops:
    2 P V d.  The bound is whichever of the two takes longer at its peak.  Returns (roof, t_hbm, t_tc).
    """
    alg_bytes = V * d * 2 + (P * d * 4 + d * 4 if pair else P * d * 2) + P * vocab_chunks(V) * 32
    alg_flops = 2.0 * P * V * d
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg_flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": alg_bytes / seconds / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": alg_flops / seconds / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["algorithmic_bytes_per_launch"] = alg_bytes
    roof["algorithmic_flops_per_launch"] = alg_flops
    return roof, t_hbm, t_tc


def self_cond_topk_roofline(V: int, d: int, P: float, K: int, seconds: float, peaks: dict) -> dict:
    """Roofline of one dg_self_condition_topk call over P positions taking `seconds`: the logits
    z = h W^T formed again (2 P V d flops) and the K kept rows of W summed per position.
    Algorithmic bytes: W once, the bf16 rows h, the K gathered bf16 rows of W per position and the
    fp32 output (the bf16 probabilities the implementation writes and re-reads are not counted)."""
    k = min(K, V)
    alg_bytes = V * d * 2 + P * d * (2 + 4) + P * k * d * 2
    alg_flops = 2.0 * P * V * d
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg_flops / (peaks["bf16_tflops"] * 1e12)
    r = {"ms_mean": seconds * 1e3, "positions_per_call": P, "top_k": K, "algorithmic_bytes_per_call": alg_bytes,
         "algorithmic_flops_per_call": alg_flops,
         "kernels": "k_topk_prep (each row's bound from the tick's chunk maxima), k_selfcond (the LM head again, "
                    "writing P = softmax(z/T) in bf16 and listing each row's candidates with their logits), "
                    "k_selfcond_topk (one CTA per position: the K best of the list, their weights and rows)",
         "timing": "CUDA events around the call on the sampler stream, after a tick, L2 flushed before it"}
    if t_hbm >= t_tc:
        r.update(bound="hbm", achieved=alg_bytes / seconds / 1e9, peak=peaks["hbm_gbs"], unit="GB/s")
    else:
        r.update(bound="tensor", achieved=alg_flops / seconds / 1e12, peak=peaks["bf16_tflops"], unit="TFLOP/s")
    r["frac"] = r["achieved"] / r["peak"]
    r["roofline_time_ms"] = max(t_hbm, t_tc) * 1e3
    return r


def self_cond_roofline(V: int, d: int, P: float, seconds: float, peaks: dict) -> dict:
    """Roofline of one dg_self_condition call over P positions taking `seconds`: the expected
    embedding softmax(z/T) W, with z = h W^T formed again.  Algorithmic bytes: W once, the bf16
    rows h and the fp32 output; flops: the two contractions, 4 P V d."""
    alg_bytes = V * d * 2 + P * d * (2 + 4)
    alg_flops = 4.0 * P * V * d
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg_flops / (peaks["bf16_tflops"] * 1e12)
    r = {"ms_mean": seconds * 1e3, "positions_per_call": P, "algorithmic_bytes_per_call": alg_bytes,
         "algorithmic_flops_per_call": alg_flops,
         "kernels": "k_selfcond (the LM head again, writing P = softmax(z/T) in bf16), k_selfcond (P W over "
                    "vocabulary chunks, tcgen05), k_selfcond_reduce (fixed-order sum of the chunks)",
         "timing": "CUDA events around the call on the sampler stream, after a tick, L2 flushed before it"}
    if t_hbm >= t_tc:
        r.update(bound="hbm", achieved=alg_bytes / seconds / 1e9, peak=peaks["hbm_gbs"], unit="GB/s")
    else:
        r.update(bound="tensor", achieved=alg_flops / seconds / 1e12, peak=peaks["bf16_tflops"], unit="TFLOP/s")
    r["frac"] = r["achieved"] / r["peak"]
    r["roofline_time_ms"] = max(t_hbm, t_tc) * 1e3
    return r


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_path: str | None):
        self.gpu = gpu_index
        self.out_path = out_path
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "25"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write(self.QUERY + "\n" + "\n".join(self.lines) + "\n")
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seeds(rank: int, n_canvases: int) -> list:
    """Canvas seeds of one replica: ranks take disjoint seed ranges, so N GPUs denoise N*B distinct canvases."""
    return [rank * n_canvases + c for c in range(n_canvases)]


def whole_job_rate(units_per_rank_step: int, steps: int, world: int, max_s: float) -> float:
    """Units all ranks processed, divided by the slowest rank's time (weak scaling: fixed work per rank)."""
    return units_per_rank_step * steps * world / max_s


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- CPU oracle timing
def wl_knob(wl: dict, name: str):
    """A workload knob, or the pages' default (entropy_bound 0.1, t 0.8 -> 0.4, sigma 0.5, one block)."""
    return wl.get(name, {"bound": 0.1, "t_max": 0.8, "t_min": 0.4, "sigma": SIGMA_HIDDEN, "gen_blocks": 1,
                         "admit": None}[name])


def oracle_cfg_for(wl: dict, n_canvases: int, seed_base: int):
    import oracle
    return oracle.OracleConfig(vocab=wl["vocab"], hidden=wl["hidden"], canvas_len=wl["canvas_len"],
                               n_canvases=n_canvases, num_inference_steps=wl["steps"], gen_blocks=1 << 10,
                               t_min=float(np.float32(wl_knob(wl, "t_min"))),
                               t_max=float(np.float32(wl_knob(wl, "t_max"))),
                               entropy_bound=float(np.float32(wl_knob(wl, "bound"))),
                               seeds=[seed_base + c for c in range(n_canvases)], mode=wl.get("mode", "freeze"),
                               softcap=float(wl.get("softcap", 0.0)))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_positions_per_s(wl: dict, budget_s: float, seed_base: int, W16=None, max_ticks=None) -> dict:
    """Time the CPU oracle, as it stands, on whole ticks of the workload until the budget is spent.

    The oracle's work per position is the same whatever the batch, so a workload of more than one
    canvas is timed on its first canvas alone and the rate is extrapolated to the whole batch."""
    import oracle
    import synth
    W16 = synth.wvocab(0, wl["vocab"], wl["hidden"]) if W16 is None else W16
    n_timed = 1 if wl["n_canvases"] > 1 else wl["n_canvases"]
    cfg = oracle_cfg_for(wl, n_timed, seed_base)
    o = oracle.OracleSampler(cfg, W16)
    fn = oracle.sampler.synth_resid_fn(cfg, W16, wl_knob(wl, "sigma"))
    positions, busy, ticks = 0, 0.0, 0
    while (ticks == 0 or busy < budget_s) and (max_ticks is None or ticks < max_ticks):
        act = o.active()
        r = fn(act, o.block[act], o.step_no[act], o.x[act])  # input generation is not timed
        t0 = time.perf_counter()
        o.tick(lambda *a: r)
        busy += time.perf_counter() - t0
        positions += act.size * wl["canvas_len"]
        ticks += 1
    what = (f"{ticks} whole oracle ticks ({positions} positions) of the workload from tick 0" if n_timed ==
            wl["n_canvases"] else
            f"{ticks} whole oracle ticks of canvas 0 alone ({positions} positions), extrapolated to the "
            f"{wl['n_canvases']}-canvas batch (the oracle's work per position does not depend on the batch)")
    return {"value": positions / busy, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{what}; fp64, OpenMP + BLAS on all cores; input generation untimed", "seconds": busy,
            "extrapolated": n_timed != wl["n_canvases"]}


def oracle_rows_per_s(wl: dict, n_rows: int, W16=None, seed: int = 0) -> float:
    """Oracle positions/s on n_rows positions of the first tick of one canvas: RMSNorm, fp64 LM head,
    softmax statistics, Gumbel sample and the entropy-bounded acceptance over those rows."""
    import oracle
    import synth
    W16 = synth.wvocab(0, wl["vocab"], wl["hidden"]) if W16 is None else W16
    cfg = oracle_cfg_for(wl, 1, seed)
    o = oracle.OracleSampler(cfg, W16)
    fn = oracle.sampler.synth_resid_fn(cfg, W16, wl_knob(wl, "sigma"))
    act = o.active()
    rows = np.arange(n_rows)
    r = fn(act, o.block[act], o.step_no[act], o.x[act])[rows]
    t0 = time.perf_counter()
    h = oracle.rmsnorm_bf16(r, cfg.rms_eps)
    z = oracle.softcap(oracle.logits(h, W16), cfg.softcap)
    T = oracle.temperature(0, cfg.num_inference_steps, cfg.t_min, cfg.t_max)
    st = oracle.stats(z, T, cfg.seed(0), 0, 0, rows)
    oracle.sampler.entropy_bounded_accept(st["H"], range(n_rows), cfg.entropy_bound)
    return n_rows / (time.perf_counter() - t0)


def oracle_one_core(workload: str, n_rows: int) -> dict | None:
    """The oracle on one host core (a child process pinned to one CPU, one OpenMP and BLAS thread)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-one-core", "--workload", workload,
                              "--cpu-rows", str(n_rows)], capture_output=True, text=True, env=env, timeout=600)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def cpu_one_core_main(args):
    cpu = sorted(os.sched_getaffinity(0))[0]
    os.sched_setaffinity(0, {cpu})
    import synth
    wl = WORKLOADS[args.workload]
    W16 = synth.wvocab(0, wl["vocab"], wl["hidden"])
    v = oracle_rows_per_s(wl, args.cpu_rows, W16=W16)
    print(json.dumps({"value": v, "cores": 1, "rows": args.cpu_rows}), flush=True)


def cpu_baseline(args, wl, W16) -> dict:
    """cpu_baseline: the oracle on all host cores (whole ticks, extrapolated for a batch) and on one core
    (a subset of one tick's positions), with the host CPU named."""
    base = oracle_positions_per_s(wl, args.cpu_budget, 0, W16=W16)
    # one core: about a tenth of the all-core budget, in positions of one tick
    rows = int(max(1, min(wl["canvas_len"], base["value"] / max(1, base["cores"]) * args.cpu_budget / 10)))
    one = oracle_one_core(args.workload, rows)
    base["cpu_model"] = cpu_model()
    if one is not None:
        base["one_core"] = {"value": one["value"], "unit": UNIT, "cores": 1,
                            "sample": f"{rows} positions of canvas 0's first tick (RMSNorm, fp64 LM head, softmax "
                                      f"statistics, Gumbel sample, acceptance), one thread pinned to one CPU"}
    return base


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    import oracle
    import synth
    W16 = synth.wvocab(0, wl["vocab"], wl["hidden"])
    # each bench step is one oracle tick of canvas 0 restricted to a bounded sample of its positions,
    # sized so the whole --steps/--warmup run stays within a few minutes (the probe times a whole
    # canvas: the oracle's fixed cost per call, converting W to fp64, is then spread as in a tick)
    per_pos = 1.0 / oracle_rows_per_s(wl, wl["canvas_len"], W16=W16)
    budget = 150.0
    sample = max(1, min(wl["canvas_len"], int(budget / max(1, args.steps + args.warmup) / per_pos)))
    cfg = oracle_cfg_for(wl, 1, 0)
    o = oracle.OracleSampler(cfg, W16)
    fn = oracle.sampler.synth_resid_fn(cfg, W16, wl_knob(wl, "sigma"))
    rows = np.arange(sample)
    busy = 0.0
    for k in range(args.warmup + args.steps):
        act = o.active()
        r = fn(act, o.block[act], o.step_no[act], o.x[act])[rows]
        s = int(o.step_no[act[0]])
        t0 = time.perf_counter()
        h = oracle.rmsnorm_bf16(r, cfg.rms_eps)
        z = oracle.softcap(oracle.logits(h, W16), cfg.softcap)
        T = oracle.temperature(s, cfg.num_inference_steps, cfg.t_min, cfg.t_max)
        st = oracle.stats(z, T, cfg.seed(int(act[0])), int(o.block[act[0]]), s, rows)
        oracle.sampler.entropy_bounded_accept(st["H"], range(sample), cfg.entropy_bound)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            busy += dt
        o.step_no[act] = (o.step_no[act] + 1) % cfg.num_inference_steps
    value = sample * args.steps / busy
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * busy / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "description": wl["text"], "commit_mode": wl["mode"],
                       "softcap": wl["softcap"]},
            "cpu_baseline": {"kind": "oracle", "cores": oracle.threads(), "value": value, "unit": UNIT,
                             "cpu_model": cpu_model(),
                             "sample": f"each step: {sample} of the {wl['canvas_len']} positions of one tick of "
                                       f"canvas 0 (RMSNorm, fp64 LM head, softmax statistics, Gumbel sample, "
                                       f"acceptance), oracle as it stands; the rate per position does not depend "
                                       f"on the batch of {wl['n_canvases']} canvases"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def canvas_steps(info) -> int:
    """Canvas-steps run so far: steps of finished blocks plus the steps of each running block."""
    import uniform_state_discrete_gb300 as dg
    return int(info["steps_used"].sum()) + int(info["step"][info["state"] == dg.ACTIVE].sum())


def run_ours(args, wl, world, rank, local):
    import torch
    import synth
    import uniform_state_discrete_gb300 as dg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(dev)  # a capturable (non-default) stream owns the sampler's work

    V, d, L, B, N = wl["vocab"], wl["hidden"], wl["canvas_len"], wl["n_canvases"], wl["steps"]
    sigma = wl_knob(wl, "sigma")
    W16 = synth.wvocab(0, V, d)
    w_dev = torch.from_numpy(W16.view(np.int16)).to(dev).view(torch.bfloat16)
    torch.cuda.synchronize(dev)
    # every canvas keeps running blocks until the bench ends (a block is 48 steps whatever its index;
    # the workload's own gen_length is the lower bound)
    total_ticks = args.warmup + args.steps + args.kernel_steps + args.warmup + args.e2e_steps + 2
    admit = wl_knob(wl, "admit")
    blocks = max(wl_knob(wl, "gen_blocks"), (total_ticks + (max(admit) if admit else 0)) // N + 2)
    seeds = replica_seeds(rank, B)
    cfg = dg.make_config(V, d, L, n_canvases=B, gen_blocks=blocks, num_inference_steps=N, seeds=seeds,
                         t_min=wl_knob(wl, "t_min"), t_max=wl_knob(wl, "t_max"), entropy_bound=wl_knob(wl, "bound"),
                         admit_tick=list(admit) if admit else None,
                         mode=dg.DG_REACCEPT if wl.get("mode") == "reaccept" else dg.DG_FREEZE,
                         softcap=float(wl.get("softcap", 0.0)), self_cond=1 if args.self_cond else 0)
    s = dg.Sampler(cfg, w_dev, stream=stream)
    resid = torch.empty(B, L, d, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    slots_ptr = s.slots_ptr()
    canvas_ptr = s.canvas().data_ptr()

    def make_resid():
        synth.resid_device(w_dev.data_ptr(), canvas_ptr, slots_ptr, B, L, V, d, sigma, resid.data_ptr(),
                           stream.cuda_stream)

    def flush_l2():
        # write a buffer twice the L2, then read it back, so L2 holds only clean lines of the
        # flush buffer: the timed tick starts cold and pays no write-back of the flush
        flush.fill_(1)
        if args.flush == "writeread":
            flush.view(torch.int32).sum()  # reads the 256 MB as int32 words, no converted copy

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:  # torch creates the CUDA event on first record
        e.record(stream)

    def capture(timed_kernels: bool):
        s.set_timing_events(ev if timed_kernels else None)
        make_resid()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            s.step(resid)
        return g

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            make_resid()
            flush_l2()
            s.step(resid)
        graph = capture(False) if args.graph else None
        torch.cuda.synchronize(dev)
        cs0 = canvas_steps(s.sync_info())
        barrier(world)
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(local, args.clocks_csv)
        clocks.start()
        time.sleep(0.3)
        # timed region: whole ticks only, so nothing separates the kernels of a tick.  The
        # ticks are enqueued back to back, as a serving loop would issue them, and every
        # tick is bracketed by its own pair of events; the host reads them at the end.
        tick_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
        for a, b in tick_ev:
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            make_resid()
            flush_l2()
            tick_ev[k][0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                s.step(resid)
            tick_ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        tick_ms = np.array([a.elapsed_time(b) for a, b in tick_ev])
        barrier(world)
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        cs1 = canvas_steps(s.sync_info())
        # per-kernel pass: the same ticks with events between the three kernels (which
        # serialise them); the LM-head kernel's mean is the roofline's launch duration
        kgraph = capture(True) if args.graph else None
        if kgraph is None:
            s.set_timing_events(ev)
        per_kernel = np.zeros((args.kernel_steps, 3))
        for k in range(args.kernel_steps):
            make_resid()
            flush_l2()
            if kgraph is not None:
                kgraph.replay()
            else:
                s.step(resid)
            ev[3].synchronize()
            per_kernel[k] = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
        s.set_timing_events(None)
        cs2 = canvas_steps(s.sync_info())  # also surfaces a latched device fault
        sc_ms, sc_rows, sck_ms = [], [], []
        if args.self_cond:
            # the self-conditioning input after a tick (dg_self_condition), timed alone, L2 flushed
            sc_out = torch.empty(B, L, d, dtype=torch.float32, device=dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for k in range(args.kernel_steps):
                make_resid()
                flush_l2()
                before = canvas_steps(s.sync_info())
                s.step(resid)
                flush_l2()
                e0.record(stream)
                s.self_condition(sc_out)
                e1.record(stream)
                e1.synchronize()
                sc_ms.append(e0.elapsed_time(e1))
                sc_rows.append((canvas_steps(s.sync_info()) - before) * L)
                if args.self_cond_topk:
                    # the top-K variant after the same tick (it reads what the tick left), L2 flushed
                    flush_l2()
                    e0.record(stream)
                    s.self_condition_topk(sc_out, args.self_cond_topk)
                    e1.record(stream)
                    e1.synchronize()
                    sck_ms.append(e0.elapsed_time(e1))
    s.sync_info()  # a fault latched by the self-conditioning calls
    device_s = float(tick_ms.sum()) / 1e3
    # positions denoised in the timed ticks, counted from the sampler's own step counters
    positions_timed = (cs1 - cs0) * L
    max_s = reduce_max(device_s, world)
    value = world * positions_timed / max_s
    positions_per_tick = positions_timed / args.steps
    kernel_positions = (cs2 - cs1) * L / max(1, args.kernel_steps)

    # roofline of the LM-head kernel (K2).  On SM pairs (256 positions or more, the
    # sampler's choice) it also forms the RMSNorm rows, and no RMSNorm kernel runs:
    # the first event interval is then empty and is counted with K2.
    pair = B * L >= 256  # the sampler's rule: SM pairs once a tick can hold 256 rows
    peaks = measured_peaks()
    k2_s = float((per_kernel[:, 0] + per_kernel[:, 1]).mean() if pair else per_kernel[:, 1].mean()) / 1e3
    roof, t_hbm, t_tc = lmhead_roofline(V, d, int(round(kernel_positions)), pair, k2_s, peaks)
    alg_bytes, alg_flops = roof["algorithmic_bytes_per_launch"], roof["algorithmic_flops_per_launch"]
    roof["positions_per_launch"] = kernel_positions
    roof["traffic"] = stored_traffic(args.workload)
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "fallback"
    roof["kernel"] = "k_lmhead_pair" if pair else "k_lmhead"  # the sampler's choice for these sizes
    roof["kernel_ms_mean"] = k2_s * 1e3
    roof["tensor_frac"] = alg_flops / k2_s / 1e12 / peaks["bf16_tflops"]
    roof["tensor_frac_sustained"] = alg_flops / k2_s / 1e12 / peaks["bf16_tflops_sustained"]
    roof["hbm_frac"] = alg_bytes / k2_s / 1e9 / peaks["hbm_gbs"]
    roof["hbm_frac_of_nominal_7_9_tbs"] = alg_bytes / k2_s / 7.9e12
    # the whole tick against the LM head's roofline at this tick's mean positions
    t_roof_tick = max(2.0 * positions_per_tick * V * d / (peaks["bf16_tflops"] * 1e12),
                      (V * d * 2 + positions_per_tick * d * 4) / (peaks["hbm_gbs"] * 1e9))
    roof["step_roofline_frac"] = t_roof_tick / (device_s / args.steps)

    # e2e through the host-buffer entry point, after the same number of untimed warm-up steps
    e2e_steps = min(args.steps, args.e2e_steps)
    host_resid = torch.empty(B, L, d, dtype=torch.float32).pin_memory()
    hr = host_resid.numpy()
    e2e_s, e2e_pos, h2d = 0.0, 0, 0
    for k in range(-args.warmup, e2e_steps):
        info = s.sync_info()
        act = np.nonzero(info["state"] == dg.ACTIVE)[0]
        tok = s.canvas().cpu().numpy()
        rows = synth.resid_rows(np.repeat(info["seed"][act], L), np.repeat(info["block"][act], L),
                                np.repeat(info["step"][act], L), np.tile(np.arange(L), act.size),
                                tok[act].reshape(-1), W16, sigma)
        hr[act] = rows.reshape(act.size, L, d)
        t0 = time.perf_counter()
        canvas_h, ent_h = s.step_host(hr)
        if k >= 0:
            e2e_s += time.perf_counter() - t0
            e2e_pos += act.size * L
            h2d += act.size * L * d * 4
    e2e_max = reduce_max(e2e_s, world)
    e2e = {"value": world * e2e_pos / e2e_max, "unit": UNIT,
           # the active canvases' rows cross the host link; the result copy spans the plan's error latch
           # (256-byte slot), the canvas and the entropies
           "h2d_bytes_per_step": h2d // max(1, e2e_steps),
           "d2h_bytes_per_step": 256 + -(-B * L * 4 // 256) * 256 + B * L * 4,
           "steps": e2e_steps,
           "api": "dg_denoise_step_host",
           "h2d": "the page-locked residual rows of the active canvases are read by the kernels in place over the "
                  "host link (zero-copy)"}

    line = None
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": args.workload, "description": wl["text"], "commit_mode": wl["mode"],
                           "softcap": wl["softcap"], "canvases": B, "canvas_len": L, "vocab": V, "hidden": d,
                           "steps_per_block": N, "entropy_bound": wl_knob(wl, "bound"),
                           "t_max": wl_knob(wl, "t_max"), "t_min": wl_knob(wl, "t_min"), "hidden_sigma": sigma,
                           "admit_ticks": list(admit) if admit else None,
                           "blocks_per_canvas_run": blocks,
                           "positions_per_step": positions_per_tick,
                           "l2": "flushed before every timed tick: 256 MB device write, then read back (outside the "
                                 "events)" if args.flush == "writeread" else "flushed by a 256 MB write",
                           "graph": bool(args.graph),
                           "parallelism": f"replicas x{world} (independent canvases per GPU)" if world > 1 else "1 GPU",
                           "timing": "CUDA events around each whole tick on the sampler stream, ticks enqueued back "
                                     "to back without host synchronisation (timed region); positions counted from "
                                     "the sampler's step counters; a second pass with events between the kernels "
                                     "gives ms_per_kernel"},
                "ms_per_kernel": ({"k_lmhead_pair (RMSNorm fused)": k2_s * 1e3,
                                   "k_finish": float(per_kernel[:, 2].mean())} if pair else
                                  {n: float(per_kernel[:, i].mean()) for i, n in
                                   enumerate(("k_rmsnorm", "k_lmhead", "k_finish"))}),
                "tick_ms_p50": float(np.percentile(tick_ms, 50)), "tick_ms_p99": float(np.percentile(tick_ms, 99)),
                "kernel_pass_steps": args.kernel_steps,
                "wall_s_timed_region": t_wall, "gpu_launches": args.steps * (3 if pair else 4),
                "gpu_launches_detail": ("per step: 2 sampler kernels (LM head on SM pairs fused with RMSNorm, "
                                        "softmax statistics and sample; combine + commit + re-noise + plan) + 1 "
                                        "residual generator" if pair else
                                        "per step: 3 sampler kernels (RMSNorm; LM head fused with softmax "
                                        "statistics and sample; combine + commit + re-noise + plan) + 1 residual "
                                        "generator"),
                "roofline": roof, "e2e": e2e, "clocks": clk}
        if sc_ms:
            line["self_cond"] = self_cond_roofline(V, d, float(np.mean(sc_rows)), float(np.mean(sc_ms)) / 1e3, peaks)
        if sck_ms:
            line["self_cond_topk"] = self_cond_topk_roofline(V, d, float(np.mean(sc_rows)), args.self_cond_topk,
                                                             float(np.mean(sck_ms)) / 1e3, peaks)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args, wl, W16)
        print(json.dumps(line), flush=True)
    s.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed ticks (default: 200 on the model-scale workloads, 3000 on the small ones)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush", choices=["write", "writeread"], default="writeread")
    ap.add_argument("--graph", type=int, default=0,
                    help="1: replay each tick as a captured CUDA graph (measured about 2 %% slower than the "
                         "default stream launches, which programmatic dependent launch already overlaps)")
    ap.add_argument("--mode", choices=["freeze", "reaccept"], default="freeze",
                    help="commit mode: committed positions freeze (default), or every step re-accepts all positions")
    ap.add_argument("--softcap", type=float, default=0.0, help="final logit softcap c (0 = off, the workloads' setting)")
    ap.add_argument("--kernel-steps", type=int, default=None,
                    help="ticks of the per-kernel timing pass (default: 50 on the model-scale workloads, else 200)")
    ap.add_argument("--clocks-csv", default=None, help="also write the raw clock samples of the timed region here")
    ap.add_argument("--self-cond-topk", type=int, default=0, metavar="K",
                    help="with --self-cond, also time dg_self_condition_topk with this K and report its roofline")
    ap.add_argument("--self-cond", action="store_true",
                    help="also time dg_self_condition after the per-kernel pass and report its roofline")
    ap.add_argument("--cpu-one-core", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-rows", type=int, default=8, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_one_core:
        return cpu_one_core_main(args)
    big = WORKLOADS[args.workload]["vocab"] * WORKLOADS[args.workload]["hidden"] >= 1 << 28
    if args.steps is None:
        args.steps = 200 if big else 3000
    if args.kernel_steps is None:
        args.kernel_steps = 50 if big else 200
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if world != args.gpus and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    wl = dict(WORKLOADS[args.workload], mode=args.mode, softcap=args.softcap)
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
    else:
        run_ours(args, wl, world, rank, local)


if __name__ == "__main__":
    main()
