"""Vocabulary-parallel ticks on one GPU: G samplers, each holding only the W rows of its
vocabulary chunks (a copy of its slice), run the LM head over their chunks, exchange their partial
records by device copies and finish the tick; every rank must then hold, bit for bit, the state
and outputs of one sampler that holds the whole vocabulary.  The ranks run on their own streams,
one after another on the device: no kernel of one rank waits for another rank's kernel."""
import numpy as np
import pytest

import synth

from parity import Case, resid_slots, weights

pytestmark = pytest.mark.gpu


def _views(s):
    return {"canvas": s.canvas(), "committed": s.committed(), "commit_step": s.commit_step(),
            "entropy": s.entropy(), "logz": s.logz(), "sample": s.sample(), "argmax": s.argmax(),
            "tokens_out": s.tokens_out()}


@pytest.mark.parametrize("case,G,ticks", [
    pytest.param(Case(vocab=4096, hidden=256, canvas_len=256, n_canvases=2, steps=4, seeds=(3, 4), gen_blocks=2),
                 2, 6, id="pair-G2"),
    pytest.param(Case(vocab=4096, hidden=256, canvas_len=256, n_canvases=2, steps=4, seeds=(3, 4), gen_blocks=2),
                 3, 6, id="pair-G3"),
    pytest.param(Case(vocab=1000, hidden=200, canvas_len=37, n_canvases=3, steps=5, seeds=(5, 6, 7),
                      admit=(0, 1, 2)), 3, 7, id="single-cta-ragged-G3"),
    pytest.param(Case(vocab=262144, hidden=2816, canvas_len=256, steps=48, seeds=(0,)), 4, 2, id="model-scale-G4"),
])
def test_split_vocabulary_matches_one_sampler(case, G, ticks):
    import torch
    import uniform_state_discrete_gb300 as dg
    W = weights(case)
    dev = torch.device("cuda:0")
    w_full = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    ref = dg.Sampler(case.gpu_cfg(), w_full, stream=torch.cuda.Stream(dev))
    ranks = []
    for r in range(G):
        v0, v1 = dg.vocab_slice(case.vocab, G, r)
        cfg = case.gpu_cfg()
        cfg.vocab_ranks, cfg.vocab_rank = G, r
        ranks.append(dg.Sampler(cfg, w_full[v0:v1].clone(), stream=torch.cuda.Stream(dev)))
    with pytest.raises(dg.DGError) as e:
        ranks[0].step(torch.zeros(case.n_canvases, case.canvas_len, case.hidden, device=dev))
    assert e.value.status == dg.DG_ERR_STATE
    ocfg = case.oracle_cfg()
    for t in range(ticks):
        info = ref.sync_info()
        if np.all(info["state"] == dg.DONE):
            break
        act = np.nonzero(info["state"] == dg.ACTIVE)[0]
        resid = torch.from_numpy(resid_slots(case, ocfg, W, act, info["block"][act], info["step"][act],
                                             ref.canvas().cpu().numpy()[act])).to(dev)
        torch.cuda.synchronize(dev)
        ref.step(resid)
        for s in ranks:
            s.step_partial(resid)
        dg.exchange_partials(ranks)
        for s in ranks:
            s.step_finish()
        torch.cuda.synchronize(dev)
        want = _views(ref)
        for r, s in enumerate(ranks):
            got = _views(s)
            for k, v in want.items():
                assert torch.equal(got[k], v), f"tick {t} rank {r}: {k} differs"
            assert np.array_equal(s.sync_info(), ref.sync_info()), f"tick {t} rank {r}: slots differ"
    for s in ranks + [ref]:
        s.close()


def test_two_replicas_equal_one_sampler_on_the_union_of_canvases():
    """The replicas path of the multi-GPU benchmark on one GPU: two samplers seeded as bench.py seeds
    ranks 0 and 1 (disjoint seed ranges) finish with exactly the tokens, heatmaps and step counts of
    one sampler holding all their canvases (canvases are independent; no collective is needed)."""
    import torch
    import bench
    import uniform_state_discrete_gb300 as dg
    B, V, d, L = 3, 4096, 256, 64
    W = synth.wvocab(0, V, d)
    dev = torch.device("cuda:0")
    w = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)

    def run(seeds):
        case = Case(vocab=V, hidden=d, canvas_len=L, n_canvases=len(seeds), steps=6, gen_blocks=2, seeds=tuple(seeds))
        s = dg.Sampler(case.gpu_cfg(), w, stream=torch.cuda.Stream(dev))
        resid = torch.empty(len(seeds), L, d, device=dev)
        for _ in range(64):
            if np.all(s.sync_info()["state"] == dg.DONE):
                break
            with torch.cuda.stream(s.stream):
                synth.resid_device(w.data_ptr(), s.canvas().data_ptr(), s.slots_ptr(), len(seeds), L, V, d, 0.5,
                                   resid.data_ptr(), s.stream.cuda_stream)
                s.step(resid)
        out = (s.tokens_out().cpu().numpy(), s.commit_steps_out().cpu().numpy(), s.sync_info()["steps_used"])
        s.close()
        return out

    reps = [run(bench.replica_seeds(r, B)) for r in range(2)]
    union = run(bench.replica_seeds(0, B) + bench.replica_seeds(1, B))
    for k in range(3):
        assert np.array_equal(np.concatenate([reps[0][k], reps[1][k]]), union[k])
