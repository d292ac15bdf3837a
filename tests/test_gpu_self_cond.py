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


# ----------------------------------------------------------------------------- top-K variant
# dg_self_condition_topk keeps each position's K most probable tokens (ties to the lower index)
# and renormalises their probabilities.  The CUDA path ranks and weights them by fp32 logits
# recomputed from h and W (a summation error of order 1e-6 of |z|), so e must lie within
# 2^-12 a_k + 1e-7 of the oracle's, a_k = sum_j q_j |W_jk| over the kept tokens -- sixteen times
# tighter than the dense input's bf16 bound.  Where the oracle's K-th and (K+1)-th largest z / T
# differ by less than 1e-4 the kept set is a near-tie: such positions are counted, not compared.
# K at most the number of 256-wide vocabulary chunks (V / 256, at most 74) takes the path where the
# LM head lists the candidates; a larger K, and a row with too many candidates (the plateau), the
# path that ranks them from the bf16 probabilities: the cases cover both.
TOPK_GAP = 1e-4


def _check_topk(case, ticks, ks, resid_fn=None, expect=None):
    import torch
    import uniform_state_discrete_gb300 as dg
    W = weights(case) if expect is None else expect["W"]
    dev = torch.device("cuda:0")
    cfg = case.gpu_cfg()
    cfg.self_cond = 1
    s = dg.Sampler(cfg, torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16))
    ocfg = case.oracle_cfg()
    out = torch.full((case.n_canvases, case.canvas_len, case.hidden), float("nan"), device=dev)
    worst, flagged, checked = 0.0, 0, 0
    for _ in range(ticks):
        info = s.sync_info()
        act = np.nonzero(info["state"] == dg.ACTIVE)[0]
        if act.size == 0:
            break
        steps = info["step"][act]
        if resid_fn is None:
            resid = resid_slots(case, ocfg, W, act, info["block"][act], steps, s.canvas().cpu().numpy()[act])
        else:
            resid = resid_fn(case)
        s.step(torch.from_numpy(resid).to(dev))
        for K in ks:
            out.fill_(float("nan"))
            s.self_condition_topk(out, K)
            got = out.cpu().numpy().astype(np.float64)
            for c, st in zip(act, steps):
                T = oracle.temperature(int(st), ocfg.num_inference_steps, ocfg.t_min, ocfg.t_max)
                if expect is not None:
                    want = expect["e"](K)
                    tol = 2.0 ** -12 * np.abs(want) + 1e-7
                    assert np.all(np.abs(got[c] - want[None, :]) <= tol), f"K={K} canvas {c}"
                    checked += case.canvas_len
                    continue
                z = oracle.softcap(oracle.logits(oracle.rmsnorm_bf16(resid[c], ocfg.rms_eps), W), ocfg.softcap)
                e, a, gap, _ = oracle.expected_embedding_topk(z, T, W, K)
                ok = gap >= TOPK_GAP
                flagged += int(np.sum(~ok))
                checked += int(np.sum(ok))
                err = np.abs(got[c] - e)[ok]
                tol = 2.0 ** -12 * a[ok] + 1e-7
                assert np.all(np.isfinite(got[c])), f"K={K} canvas {c}: row not written"
                assert np.all(err <= tol), f"K={K} canvas {c}: max excess {np.max(err - tol):.3g}"
                worst = max(worst, float(np.max(err / tol)) if err.size else 0.0)
    s.close()
    return worst, flagged, checked


@pytest.mark.parametrize("case,ticks,ks", [
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=16, steps=8), 2, (1, 32, 256), id="tiny"),
    pytest.param(Case(vocab=1000, hidden=200, canvas_len=37, n_canvases=3, steps=5, seeds=(5, 6, 7), admit=(0, 1, 1),
                      gen_blocks=2), 3, (32, 100), id="ragged-staggered"),
    pytest.param(Case(vocab=200, hidden=64, canvas_len=16, steps=4), 1, (256,), id="k-above-vocab"),
    pytest.param(Case(vocab=4096, hidden=256, canvas_len=256, n_canvases=2, steps=4, seeds=(3, 4)), 1, (8, 32),
                 id="pair-256-rows"),
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=32, steps=6, softcap=2.0, sigma_w=0.2, w_seed=4,
                      t_max=1.5, t_min=0.1), 2, (4, 32), id="softcap"),
    pytest.param(Case(vocab=32768, hidden=1024, canvas_len=256, steps=4, sigma=0.1, t_max=0.1, t_min=0.05), 1, (32,),
                 id="peaked-rows"),
    pytest.param(Case(vocab=262144, hidden=2816, canvas_len=256, steps=48), 1, (32, 256), id="model-scale"),
])
def test_self_condition_topk_matches_oracle(case, ticks, ks):
    worst, flagged, checked = _check_topk(case, ticks, ks)
    print(f"\n[self-cond top-K {case.vocab}x{case.hidden} K={ks}] worst error / tolerance = {worst:.3g}; "
          f"{checked} positions compared, {flagged} near-ties at the cut")
    assert checked > 0


def test_self_condition_topk_plateau_keeps_the_lowest_indices():
    """Every logit equal (W rows share the coordinates h lives on; h is zero elsewhere): more than
    2048 tokens tie at the top, the kernel takes the row in windows, and the kept tokens must be the
    K lowest indices, so e is the mean of the first K rows (the oracle's equal-logits pin)."""
    import synth
    V, d, L = 4096, 128, 16
    case = Case(vocab=V, hidden=d, canvas_len=L, steps=4)
    W = synth.wvocab(21, V, d, sigma_w=0.3)
    W[:, : d // 2] = W[0, : d // 2]  # every row equal where h is non-zero
    Wv = oracle.bf16_value(W)

    def resid_fn(case):
        r = np.zeros((1, L, d), np.float32)
        r[0, :, : d // 2] = np.random.default_rng(22).standard_normal((L, d // 2))
        return r

    expect = {"W": W, "e": lambda K: Wv[:K].mean(axis=0)}
    _, _, checked = _check_topk(case, 1, (1, 32, 256), resid_fn=resid_fn, expect=expect)
    assert checked == 3 * L


def test_self_condition_topk_rejects_bad_arguments():
    import torch
    import uniform_state_discrete_gb300 as dg
    case = Case(vocab=2048, hidden=128, canvas_len=16, steps=8)
    W = torch.from_numpy(weights(case).view(np.int16)).to("cuda:0").view(torch.bfloat16)
    s = dg.Sampler(case.gpu_cfg(), W)
    out = torch.zeros(1, 16, 128, device="cuda:0")
    with pytest.raises(dg.DGError) as e:
        s.self_condition_topk(out, 32)
    assert e.value.status == dg.DG_ERR_STATE  # created without self_cond
    s.close()
    cfg = case.gpu_cfg()
    cfg.self_cond = 1
    s = dg.Sampler(cfg, W)
    for k in (0, 257):
        with pytest.raises(dg.DGError) as e:
            s.self_condition_topk(out, k)
        assert e.value.status == dg.DG_ERR_ARG
    s.close()
