"""Self-conditioning input (dg_self_condition) against the CPU oracle, through the C ABI.

After a tick, every position of the canvases active in it gets e = softmax(z/T) W, the expected
token embedding under that tick's distribution ("The Annotated DiffusionGemma", decode mode).
The oracle computes it in fp64 from exact probabilities; the CUDA path rounds P to bf16 before
the tensor-core contraction (relative error at most 2^-9 per probability) and accumulates in
fp32, so each coordinate k must lie within 2^-8 a_k + 1e-7 of the oracle's, a_k = sum_v p_v |W_vk|.
"""
import numpy as np
import pytest

import oracle

from parity import Case, resid_slots, weights

pytestmark = pytest.mark.gpu


def _check_ticks(case, ticks):
    import torch
    import uniform_state_discrete_gb300 as dg
    W = weights(case)
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    cfg = case.gpu_cfg()
    cfg.self_cond = 1
    s = dg.Sampler(cfg, w_dev)
    ocfg = case.oracle_cfg()
    out = torch.full((case.n_canvases, case.canvas_len, case.hidden), float("nan"), device=dev)
    worst = 0.0
    for _ in range(ticks):
        info = s.sync_info()
        act = np.nonzero(info["state"] == dg.ACTIVE)[0]
        if act.size == 0:
            break
        steps = info["step"][act]
        resid = resid_slots(case, ocfg, W, act, info["block"][act], steps, s.canvas().cpu().numpy()[act])
        s.step(torch.from_numpy(resid).to(dev))
        s.self_condition(out)
        got = out.cpu().numpy()
        for c, st in zip(act, steps):
            z = oracle.softcap(oracle.logits(oracle.rmsnorm_bf16(resid[c], ocfg.rms_eps), W), ocfg.softcap)
            e, a = oracle.expected_embedding(z, oracle.temperature(int(st), ocfg.num_inference_steps, ocfg.t_min,
                                                                   ocfg.t_max), W)
            err = np.abs(got[c].astype(np.float64) - e)
            tol = 2.0 ** -8 * a + 1e-7
            assert np.all(err <= tol), f"canvas {c}: max excess {np.max(err - tol):.3g}"
            worst = max(worst, float(np.max(err / tol)))
    s.close()
    return worst


@pytest.mark.parametrize("case,ticks", [
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=16, steps=8), 3, id="tiny"),
    pytest.param(Case(vocab=1000, hidden=200, canvas_len=37, n_canvases=3, steps=5, seeds=(5, 6, 7), admit=(0, 1, 1),
                      gen_blocks=2), 4, id="ragged-staggered"),
    pytest.param(Case(vocab=4096, hidden=256, canvas_len=256, n_canvases=2, steps=4, seeds=(3, 4)), 2,
                 id="pair-256-rows"),
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=32, steps=6, softcap=2.0, sigma_w=0.2, w_seed=4,
                      t_max=1.5, t_min=0.1), 2, id="softcap"),
    pytest.param(Case(vocab=262144, hidden=2816, canvas_len=256, steps=48), 1, id="model-scale"),
])
def test_self_condition_matches_oracle(case, ticks):
    worst = _check_ticks(case, ticks)
    print(f"\n[self-cond {case.vocab}x{case.hidden}] worst error / tolerance = {worst:.3g}")


def test_self_condition_needs_the_option():
    import torch
    import uniform_state_discrete_gb300 as dg
    case = Case(vocab=2048, hidden=128, canvas_len=16, steps=8)
    W = weights(case)
    s = dg.Sampler(case.gpu_cfg(), torch.from_numpy(W.view(np.int16)).to("cuda:0").view(torch.bfloat16))
    with pytest.raises(dg.DGError) as e:
        s.self_condition(torch.zeros(1, 16, 128, device="cuda:0"))
    assert e.value.status == dg.DG_ERR_STATE
    s.close()
