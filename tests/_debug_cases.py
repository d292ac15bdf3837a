"""Cases run against the index-checking build of the library (DG_LIBRARY=debug), in a process of
their own (tests/test_gpu_debug_checks.py starts it): small parity cases through every kernel
path, each followed by dg_debug_check -- every workspace guard intact and no index check failed --
and one planted overflow, a byte written past the first workspace buffer from the host, which the
check must find.  Prints "debug cases ok" and exits 0 when all pass."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)
assert os.environ.get("DG_LIBRARY") == "debug"

import torch  # noqa: E402

import uniform_state_discrete_gb300 as dg  # noqa: E402
from parity import Case, resid_slots, teacher_forced, weights  # noqa: E402

assert dg.LIB_PATH.endswith("libdgsampler_debug.so")


def forced(case, label):
    W = weights(case)
    w_dev = torch.from_numpy(W.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    s = dg.Sampler(case.gpu_cfg(), w_dev)
    rep = teacher_forced(case, gpu=s, W=W)
    assert rep.ok(), (label, rep.errors[:5])
    s.debug_check()
    print(f"{label}: {rep.ticks} ticks, guards intact, no index check failed", flush=True)
    s.close()


CASES = {
    "tiny": Case(vocab=2048, hidden=128, canvas_len=16, steps=8),
    "ragged-staggered": Case(vocab=1000, hidden=200, canvas_len=37, n_canvases=3, gen_blocks=2, steps=5,
                             seeds=(5, 6, 7), admit=(0, 2, 3)),
    "pair-ragged": Case(vocab=1000, hidden=200, canvas_len=100, n_canvases=3, gen_blocks=2, steps=4, seeds=(1, 2, 3),
                        admit=(0, 1, 2)),
    "capacity-limited": Case(vocab=4096, hidden=64, canvas_len=1, n_canvases=5, steps=4, admit=(0, 0, 1, 1, 1),
                             max_active=2),
    "reaccept": Case(vocab=512, hidden=256, canvas_len=32, steps=12, bound=1.0, sigma=0.3, sigma_w=0.1, w_seed=2,
                     seeds=(9,), gen_blocks=2, mode="reaccept"),
    "softcap": Case(vocab=2048, hidden=128, canvas_len=32, steps=6, softcap=2.0, sigma_w=0.2, w_seed=4, t_max=1.5,
                    t_min=0.1),
    "V2": Case(vocab=2, hidden=64, canvas_len=256, steps=4, bound=1.0),
    "L1024": Case(vocab=512, hidden=128, canvas_len=1024, steps=6, bound=200.0, sigma=0.02),
}

for name, case in CASES.items():
    forced(case, name)

# the split vocabulary and self-conditioning paths, a few ticks each
case = Case(vocab=4096, hidden=256, canvas_len=256, n_canvases=2, steps=4, seeds=(3, 4))
W = weights(case)
w_full = torch.from_numpy(W.view(np.int16)).to("cuda:0").view(torch.bfloat16)
ranks = []
for r in range(2):
    v0, v1 = dg.vocab_slice(case.vocab, 2, r)
    cfg = case.gpu_cfg()
    cfg.vocab_ranks, cfg.vocab_rank = 2, r
    ranks.append(dg.Sampler(cfg, w_full[v0:v1].clone()))
cfg = case.gpu_cfg()
cfg.self_cond = 1
sc = dg.Sampler(cfg, w_full)
out = torch.zeros(case.n_canvases, case.canvas_len, case.hidden, device="cuda:0")
ocfg = case.oracle_cfg()
for _ in range(3):
    info = sc.sync_info()
    act = np.nonzero(info["state"] == dg.ACTIVE)[0]
    resid = torch.from_numpy(resid_slots(case, ocfg, W, act, info["block"][act], info["step"][act],
                                         sc.canvas().cpu().numpy()[act])).to("cuda:0")
    sc.step(resid)
    sc.self_condition(out)
    sc.self_condition_topk(out, 32)
    for s in ranks:
        s.step_partial(resid)
    dg.exchange_partials(ranks)
    for s in ranks:
        s.step_finish()
    torch.cuda.synchronize()
    assert all(torch.equal(s.canvas(), sc.canvas()) for s in ranks)
for s in ranks + [sc]:
    s.debug_check()
print("split vocabulary and self-conditioning (dense and top-K): guards intact, no index check failed", flush=True)

# a planted overflow: one byte past the first workspace buffer (the per-canvas slots), from the host
s = ranks[0]
first_guard = (dg.SLOT_DTYPE.itemsize * case.n_canvases + 255) // 256 * 256
s.workspace[s._ws_off + first_guard] = 0
try:
    s.debug_check()
    raise AssertionError("a damaged guard went unnoticed")
except dg.DGError as e:
    assert e.status == dg.DG_ERR_BOUNDS and str(first_guard) in str(e), str(e)
print("planted overflow found at offset", first_guard, flush=True)
for s in ranks + [sc]:
    s.close()
print("debug cases ok", flush=True)
