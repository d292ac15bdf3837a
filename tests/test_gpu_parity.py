"""CUDA path vs CPU oracle, element by element, through the C ABI (GB300 only)."""
import numpy as np
import pytest

import oracle
import synth

from parity import Case, f32, oracle_state_to_gpu, resid_slots, teacher_forced, weights

pytestmark = pytest.mark.gpu


def _assert_report(rep, label):
    print(f"\n[{label}] ticks={rep.ticks} positions={rep.positions} max|dH|={rep.max_dH:.3g} "
          f"max|dlogZ|/|logZ|={rep.max_dlogZ_rel:.3g} y mismatch={rep.y_mismatch} (flagged {rep.y_flagged}) "
          f"argmax mismatch={rep.amax_mismatch} (flagged {rep.amax_flagged}) "
          f"flagged positions={rep.state_flagged_positions} flagged canvases={rep.canvas_flagged}")
    assert rep.ticks > 0
    assert rep.ok(), "\n".join(rep.errors[:20])


def test_tiny_config_teacher_forced():
    """1 canvas x 16 positions, V=2048, d=128, 8 steps (W drawn in fp32, rounded once to bf16)."""
    rep = teacher_forced(Case(vocab=2048, hidden=128, canvas_len=16, steps=8))
    _assert_report(rep, "tiny")
    assert rep.max_dH < 1e-4


def test_canvas256_v32k_teacher_forced():
    """1 canvas x 256 positions, V=32768, d=1024, 48 steps, every tick checked."""
    rep = teacher_forced(Case(vocab=32768, hidden=1024, canvas_len=256, steps=48))
    _assert_report(rep, "V32k")
    assert rep.max_dH < 1e-4


def test_ragged_shapes_and_staggered_admission():
    """V not a multiple of the 256-wide tile, d not a multiple of the 64-wide K stage, a canvas
    length that splits M tiles, three canvases admitted at different ticks, two blocks each."""
    case = Case(vocab=1000, hidden=200, canvas_len=37, n_canvases=3, gen_blocks=2, steps=5, seeds=(5, 6, 7),
                admit=(0, 2, 3))
    _assert_report(teacher_forced(case), "ragged")


def test_rmsnorm_weight_vector():
    """A non-trivial RMSNorm weight w (the pages' rms(x, w) with w != 1)."""
    case = Case(vocab=4096, hidden=512, canvas_len=64, steps=4, norm_seed=17, seeds=(2,))
    rep = teacher_forced(case)
    _assert_report(rep, "norm-weight")


@pytest.mark.parametrize("hidden,norm_seed,sigma,eps", [(1024, None, 0.5, 1e-6), (2816, 5, 0.5, 1e-6),
                                                        (200, None, 2.0, 1e-6), (512, 7, 1e-3, 1e-6),
                                                        (1024, 3, 0.05, 0.25), (4096, 9, 0.5, 1e-6)])
def test_rmsnorm_bf16_bit_exact(hidden, norm_seed, sigma, eps):
    """K1's bf16 rows equal the oracle's RMSNorm bit for bit (both round the exact quotient)."""
    import torch
    import uniform_state_discrete_gb300 as dg
    from parity import norm_w
    case = Case(vocab=1024, hidden=hidden, canvas_len=96, n_canvases=3, steps=4, sigma=sigma, norm_seed=norm_seed,
                rms_eps=eps)
    W = weights(case)
    ocfg = case.oracle_cfg()
    nw = norm_w(case)
    o = oracle.OracleSampler(ocfg, W, norm_w=nw)
    dev = torch.device("cuda:0")
    s = dg.Sampler(case.gpu_cfg(), torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16),
                   norm_w=None if nw is None else torch.from_numpy(nw).to(dev))
    act = o.active()
    resid = resid_slots(case, ocfg, W, act, o.block[act], o.step_no[act], o.x[act])
    s.step(torch.from_numpy(resid).to(dev))
    got = s.normed(act.size * case.canvas_len).cpu().numpy().view(np.uint16)
    want = oracle.rmsnorm_bf16(resid[act].reshape(-1, hidden), ocfg.rms_eps, nw)
    assert np.array_equal(got, want), f"{int((got != want).sum())} of {got.size} bf16 values differ"


def test_pair_tiles_ragged_rows_and_tails():
    """>= 256 rows per tick selects the SM-pair LM head: 3 canvases x 100 positions (a second,
    partly empty 256-row pair tile), V and d not multiples of the tile sizes, staggered admission."""
    case = Case(vocab=1000, hidden=200, canvas_len=100, n_canvases=3, gen_blocks=2, steps=4, seeds=(1, 2, 3),
                admit=(0, 1, 2))
    _assert_report(teacher_forced(case), "pair-ragged")


def test_pair_tiles_many_canvases():
    """Five 256-position canvases in one tick: five pair tiles per vocabulary chunk."""
    case = Case(vocab=4096, hidden=256, canvas_len=256, n_canvases=5, steps=3, seeds=(11, 12, 13, 14, 15))
    _assert_report(teacher_forced(case), "pair-many")


def test_single_position_canvases_capacity_limited():
    case = Case(vocab=4096, hidden=64, canvas_len=1, n_canvases=5, steps=4, admit=(0, 0, 1, 1, 1), max_active=2)
    _assert_report(teacher_forced(case), "L1")


@pytest.mark.parametrize("mode", ["freeze", "reaccept"])
def test_maximum_canvas_length_sorts_whole_canvas(mode):
    """The largest canvas the ABI takes (1024 positions) with an entropy budget far above every
    single entropy: all 1024 positions are candidates, so the commit sorts the whole canvas
    (bitonic, 1024 keys) and walks ~33 acceptances a step; the last step commits the rest."""
    case = Case(vocab=512, hidden=128, canvas_len=1024, steps=6, bound=200.0, sigma=0.02, mode=mode)
    _assert_report(teacher_forced(case), f"L1024-{mode}")


@pytest.mark.parametrize("vocab,canvas_len", [(2, 16), (3, 16), (2, 256)], ids=["V2", "V3", "V2-pair"])
def test_smallest_vocabularies(vocab, canvas_len):
    """The smallest vocabularies (V = 2 is the ABI's minimum): one vocabulary chunk holding a single
    ragged tile of 2 or 3 valid columns, on the single-CTA and the SM-pair LM head; entropies
    bounded by ln V, and a budget of 1 nat, so two positions commit a step at V = 2, one at V = 3."""
    case = Case(vocab=vocab, hidden=64, canvas_len=canvas_len, steps=4, bound=1.0)
    _assert_report(teacher_forced(case), f"V{vocab}-L{canvas_len}")


def test_step_after_every_canvas_finished_is_a_state_error():
    """One canvas, one block, two steps: the third tick is refused with DG_ERR_STATE (the host can
    tell that every canvas has finished), through both step entry points, and the finished block's
    tokens stay readable."""
    import torch
    import uniform_state_discrete_gb300 as dg
    case = Case(vocab=512, hidden=64, canvas_len=16, steps=2)
    W = weights(case)
    dev = torch.device("cuda:0")
    s = dg.Sampler(case.gpu_cfg(), torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16))
    resid = torch.zeros(1, case.canvas_len, case.hidden, device=dev)
    s.step(resid)
    s.step(resid)
    with pytest.raises(dg.DGError) as e:
        s.step(resid)
    assert e.value.status == dg.DG_ERR_STATE
    with pytest.raises(dg.DGError) as e:
        s.step_host(np.zeros((1, case.canvas_len, case.hidden), np.float32))
    assert e.value.status == dg.DG_ERR_STATE
    info = s.sync_info()
    assert int(info["state"][0]) == dg.DONE
    toks = s.get_state()["tokens_out"][0, 0]
    assert ((toks >= 0) & (toks < case.vocab)).all()
    s.close()


def test_maximum_step_count():
    """The largest num_inference_steps the ABI takes (1024) on a 1024-position canvas: one commit per
    step (every entropy is far above the budget), the temperature table's last entries, and the final
    step committing the last position; every 64th tick and the last ones are checked."""
    case = Case(vocab=64, hidden=64, canvas_len=1024, steps=1024, bound=0.1)
    rep = teacher_forced(case, check_every=64)
    _assert_report(rep, "N1024")
    assert rep.ticks >= 16


def test_low_entropy_multi_commit_and_early_stop():
    """Peaked distributions: several positions fit the bound per step and the early-stop test fires."""
    case = Case(vocab=512, hidden=256, canvas_len=32, steps=24, bound=1.0, sigma=0.1, sigma_w=0.1, w_seed=2,
                seeds=(9,), gen_blocks=3)
    rep = teacher_forced(case)
    _assert_report(rep, "low-entropy")


@pytest.mark.parametrize("stability", [2, 3])
def test_early_stop_with_longer_stability(stability):
    """Early stop after `stability` steps in a row with an unchanged argmax canvas: the stable-step
    counter, the convergence and the block hand-over against the oracle, teacher-forced."""
    case = Case(vocab=512, hidden=256, canvas_len=32, steps=24, bound=1.0, sigma=0.1, sigma_w=0.1, w_seed=2,
                seeds=(9,), gen_blocks=3, stability=stability)
    _assert_report(teacher_forced(case), f"stability {stability}")


def test_hot_schedule_noise_driven_regime():
    """t 1.5 -> 0.1 with large hidden noise: sampling ties get exercised."""
    case = Case(vocab=2048, hidden=256, canvas_len=64, steps=12, t_max=1.5, t_min=0.1, sigma=2.0, bound=0.01,
                n_canvases=2, seeds=(3, 4))
    _assert_report(teacher_forced(case), "hot")


def test_reaccept_tiny_config_teacher_forced():
    """DG_REACCEPT at the tiny config: one position accepted per step (every entropy far above the
    bound), every other position, earlier acceptances included, re-noised."""
    rep = teacher_forced(Case(vocab=2048, hidden=128, canvas_len=16, steps=8, mode="reaccept"))
    _assert_report(rep, "reaccept tiny")


def test_reaccept_many_accepted_and_remasked():
    """DG_REACCEPT with moderate hidden noise: several accepted positions per step, accepted sets
    that change between steps (re-masking), two blocks; 256 positions take the SM-pair LM head and
    more than 31 candidates take the commit's full sort."""
    for L, bound in ((32, 1.0), (256, 3.0)):
        case = Case(vocab=512, hidden=256, canvas_len=L, steps=12, bound=bound, sigma=0.3, sigma_w=0.1, w_seed=2,
                    seeds=(9,), gen_blocks=2, mode="reaccept")
        _assert_report(teacher_forced(case), f"reaccept L={L}")


@pytest.mark.parametrize("case", [
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=16, steps=8, softcap=30.0), id="tiny-c30"),
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=32, steps=6, softcap=2.0, sigma_w=0.2, w_seed=4,
                      t_max=1.5, t_min=0.1), id="tanh-saturating-c2"),
    pytest.param(Case(vocab=4096, hidden=256, canvas_len=256, steps=4, softcap=3.0, sigma_w=0.1, w_seed=5,
                      seeds=(7,)), id="pair-c3"),
])
def test_final_logit_softcap(case):
    """Final logit softcap c tanh(z/c) before the temperature, from a barely active cap (c = 30 on
    logits of order 0.2) to a saturating one (|z/c| around 1 and above), on both LM-head kernels."""
    _assert_report(teacher_forced(case), f"softcap c={case.softcap}")


def _gpu_free_run(case, W):
    import torch
    import uniform_state_discrete_gb300 as dg
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    s = dg.Sampler(case.gpu_cfg(), w_dev)
    ocfg = case.oracle_cfg()
    for _ in range(10000):
        info = s.sync_info()
        if np.all(info["state"] == dg.DONE):
            break
        act = np.nonzero(info["state"] == dg.ACTIVE)[0]
        tok = s.canvas().cpu().numpy()
        resid = resid_slots(case, ocfg, W, act, info["block"][act], info["step"][act], tok[act])
        s.step(torch.from_numpy(resid).to(dev))
    return s, s.tokens_out().cpu().numpy(), s.sync_info()


def test_free_run_tiny_matches_oracle():
    case = Case(vocab=2048, hidden=128, canvas_len=16, steps=8, n_canvases=2, seeds=(0, 1))
    W = weights(case)
    o = oracle.OracleSampler(case.oracle_cfg(), W)
    o.run(oracle.sampler.synth_resid_fn(case.oracle_cfg(), W, case.sigma))
    s, tok, info = _gpu_free_run(case, W)
    assert np.array_equal(tok, o.tokens_out)
    assert np.array_equal(s.commit_steps_out().cpu().numpy(), o.commit_steps_out)
    assert np.array_equal(info["steps_used"], o.steps_used)


def test_idle_ticks_before_admission_pair_kernel():
    """256 positions of one canvas admitted at tick 2: the SM-pair LM head loads its first W stages
    before it knows whether any canvas is active, so on ticks 0 and 1 it must let those copies land
    with nothing to consume them; the run must then match the oracle."""
    case = Case(vocab=4096, hidden=256, canvas_len=256, steps=5, seeds=(3,), admit=(2,))
    W = weights(case)
    o = oracle.OracleSampler(case.oracle_cfg(), W)
    o.run(oracle.sampler.synth_resid_fn(case.oracle_cfg(), W, case.sigma))
    s, tok, info = _gpu_free_run(case, W)
    assert np.array_equal(tok, o.tokens_out)
    assert np.array_equal(s.commit_steps_out().cpu().numpy(), o.commit_steps_out)
    assert np.array_equal(info["steps_used"], o.steps_used)


@pytest.mark.parametrize("canvas_len", [16, 256], ids=["single-cta", "pair"])
def test_maximum_hidden_size(canvas_len):
    """The largest hidden size the ABI takes (d = 16384): rows longer than the RMSNorm forms keep in
    registers (they loop over the row), 256 K stages per LM-head tile, on both LM-head kernels."""
    case = Case(vocab=1024, hidden=16384, canvas_len=canvas_len, steps=3, seeds=(8,))
    _assert_report(teacher_forced(case), f"d16384-L{canvas_len}")


def test_idle_ticks_before_admission_single_cta_kernels():
    """16 positions of two canvases admitted at ticks 2 and 3: the RMSNorm, single-CTA LM head and
    finishing kernels run ticks with no active canvas (and then with one) before both run; the free
    run must match the oracle's."""
    case = Case(vocab=2048, hidden=128, canvas_len=16, n_canvases=2, steps=4, seeds=(6, 7), admit=(2, 3))
    W = weights(case)
    o = oracle.OracleSampler(case.oracle_cfg(), W)
    o.run(oracle.sampler.synth_resid_fn(case.oracle_cfg(), W, case.sigma))
    s, tok, info = _gpu_free_run(case, W)
    assert np.array_equal(tok, o.tokens_out)
    assert np.array_equal(s.commit_steps_out().cpu().numpy(), o.commit_steps_out)
    assert np.array_equal(info["steps_used"], o.steps_used)


def _random_cases(n, seed=2026):
    """Small configurations drawn at random (fixed seed): every knob of the ABI varied together."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        L = int(rng.choice([1, 7, 16, 33, 100, 256, 300]))
        t_max = float(rng.choice([0.5, 0.8, 1.5]))
        out.append(Case(vocab=int(rng.choice([2, 37, 256, 1000, 2048, 4099])),
                        hidden=int(rng.choice([8, 64, 120, 256, 520])),
                        canvas_len=L, n_canvases=B, gen_blocks=int(rng.integers(1, 3)),
                        steps=int(rng.integers(2, 6)), t_max=t_max, t_min=float(t_max * rng.choice([0.2, 0.5, 1.0])),
                        bound=float(rng.choice([0.0, 0.1, 2.0, 50.0])), conf=float(rng.choice([0.0, 0.005, 0.5])),
                        sigma=float(rng.choice([0.05, 0.5, 2.0])), sigma_w=float(rng.choice([0.02, 0.2])),
                        w_seed=int(rng.integers(0, 100)), seeds=tuple(int(x) for x in rng.integers(0, 2**63, B)),
                        admit=tuple(int(x) for x in rng.integers(0, 3, B)),
                        max_active=int(rng.integers(0, B + 1)),
                        mode=str(rng.choice(["freeze", "reaccept"])), softcap=float(rng.choice([0.0, 0.0, 3.0])),
                        stability=int(rng.integers(1, 3))))
    return out


@pytest.mark.parametrize("case", _random_cases(16), ids=[f"random{i}" for i in range(16)])
def test_randomized_configurations_teacher_forced(case):
    """Sixteen small configurations with every knob drawn at random (vocabulary and hidden sizes
    including ragged and minimal ones, canvas counts and lengths on both LM-head kernels, staggered
    admission under a slot limit, both commit modes, softcap, stability, temperatures, budgets and
    confidence thresholds including 0), each teacher-forced on every tick against the oracle."""
    _assert_report(teacher_forced(case), f"V{case.vocab} d{case.hidden} L{case.canvas_len} B{case.n_canvases} "
                   f"{case.mode} cap{case.softcap}")


def test_batch_and_admission_invariance_bitwise():
    """A canvas gives the same tokens and entropies alone or inside a staggered batch
    (TensorSharp doc, "7. Test coverage": batched decode equals per-sequence decode)."""
    base = dict(vocab=4096, hidden=256, canvas_len=64, steps=6)
    W = weights(Case(**base))
    _, alone, _ = _gpu_free_run(Case(**base, seeds=(21,)), W)
    _, batch, _ = _gpu_free_run(Case(**base, n_canvases=3, seeds=(20, 21, 22), admit=(0, 2, 4)), W)
    assert np.array_equal(batch[1], alone[0])


def test_dg_run_callback_and_host_step():
    import torch
    import uniform_state_discrete_gb300 as dg
    case = Case(vocab=2048, hidden=128, canvas_len=16, steps=8, n_canvases=2, seeds=(0, 1))
    W = weights(case)
    ocfg = case.oracle_cfg()
    o = oracle.OracleSampler(ocfg, W)
    o.run(oracle.sampler.synth_resid_fn(ocfg, W, case.sigma))
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    s = dg.Sampler(case.gpu_cfg(), w_dev)
    resid_dev = torch.zeros(case.n_canvases, case.canvas_len, case.hidden, device=dev)

    def cb(tick, canvas_ptr, slots_ptr, resid_ptr, stream_ptr):
        info = s.sync_info()
        act = np.nonzero(info["state"] == dg.ACTIVE)[0]
        if act.size == 0:
            return 0
        tok = s.canvas().cpu().numpy()
        r = resid_slots(case, ocfg, W, act, info["block"][act], info["step"][act], tok[act])
        assert resid_ptr == resid_dev.data_ptr()
        resid_dev.copy_(torch.from_numpy(r))
        torch.cuda.synchronize()
        return 0

    tokens, slots = s.run(cb, resid_dev)
    assert np.array_equal(tokens, o.tokens_out)
    assert np.all(slots["state"] == dg.DONE)
    # the host-buffer tick gives what the device tick gives, from pageable memory (copied into the
    # workspace) and from page-locked memory (read by the kernels in place), on both LM-head kernels
    for c2 in (case, Case(vocab=4096, hidden=256, canvas_len=256, steps=4, seeds=(5,))):
        W2 = weights(c2)
        w2 = torch.from_numpy(W2.view(np.int16)).to(dev).view(torch.bfloat16)
        o2 = c2.oracle_cfg()
        s2 = dg.Sampler(c2.gpu_cfg(), w2)
        s3 = dg.Sampler(c2.gpu_cfg(), w2)
        for k in range(3):
            info = s2.sync_info()
            act = np.nonzero(info["state"] == dg.ACTIVE)[0]
            r = resid_slots(c2, o2, W2, act, info["block"][act], info["step"][act], s2.canvas().cpu().numpy()[act])
            if k % 2:
                r = torch.from_numpy(r).pin_memory().numpy()
            canvas_h, ent_h = s2.step_host(r)
            s3.step(torch.from_numpy(r).to(dev))
            assert np.array_equal(canvas_h, s3.canvas().cpu().numpy())
            assert np.array_equal(ent_h, s3.entropy().cpu().numpy())


@pytest.mark.parametrize("canvas_len,vocab", [(16, 2048), (256, 4096)], ids=["single-cta", "pair"])
def test_bounded_wait_runs_out_and_sampler_recovers(canvas_len, vocab):
    """Failure detection without a GPU fault: with the LM head holding back its unit counts, the
    finishing kernel's bounded wait runs out after about a second, the tick reports DG_ERR_TIMEOUT
    and the context stays usable; after dg_set_state the next tick matches a fresh sampler's."""
    import time
    import torch
    import uniform_state_discrete_gb300 as dg
    case = Case(vocab=vocab, hidden=128, canvas_len=canvas_len, steps=6, seeds=(4,))
    W = weights(case)
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    ocfg = case.oracle_cfg()
    s = dg.Sampler(case.gpu_cfg(), w_dev)
    st0 = s.get_state()
    r = torch.from_numpy(resid_slots(case, ocfg, W, np.array([0]), np.array([0]), np.array([0]),
                                     st0["tokens"][:1])).to(dev)
    s.debug_hold_slabs(True)
    t0 = time.perf_counter()
    s.step(r)
    with pytest.raises(dg.DGError) as err:
        s.sync_info()
    waited = time.perf_counter() - t0
    assert err.value.status == dg.DG_ERR_TIMEOUT
    # the first wait to give up is latched: the finishing kernel's, not the LM head's
    assert "finishing kernel, LM-head units of a slab" in str(err.value)
    assert 0.9 < waited < 30.0
    s.debug_hold_slabs(False)
    s.set_state(st0)
    s.step(r)
    s.sync_info()
    fresh = dg.Sampler(case.gpu_cfg(), w_dev)
    fresh.step(r)
    fresh.sync_info()
    for view in ("canvas", "entropy", "sample"):
        assert torch.equal(getattr(s, view)(), getattr(fresh, view)())


@pytest.mark.parametrize("canvas_len,vocab", [(16, 2048), (256, 4096)])
def test_failed_cuda_call_is_reported_and_sampler_recovers(canvas_len, vocab):
    """Failure detection with a fake of the failing call, on the host: the library's next checked CUDA
    call is not made and reports a failure.  A step whose first launch fails returns DG_ERR_CUDA
    naming the launch and changes nothing, so retrying it gives a fresh sampler's tick; one that
    fails between the kernels of a tick is brought back by dg_set_state."""
    import torch
    import uniform_state_discrete_gb300 as dg
    case = Case(vocab=vocab, hidden=128, canvas_len=canvas_len, steps=6, seeds=(4,))
    W = weights(case)
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    ocfg = case.oracle_cfg()
    fresh = dg.Sampler(case.gpu_cfg(), w_dev)
    st0 = fresh.get_state()
    r = torch.from_numpy(resid_slots(case, ocfg, W, np.array([0]), np.array([0]), np.array([0]),
                                     st0["tokens"][:1])).to(dev)
    fresh.step(r)
    fresh.sync_info()
    s = dg.Sampler(case.gpu_cfg(), w_dev)
    try:
        # the first checked call of the step fails: nothing was launched
        assert dg.lib.dg_debug_fail_cuda_call(0) == dg.DG_OK
        with pytest.raises(dg.DGError) as err:
            s.step(r)
        assert err.value.status == dg.DG_ERR_CUDA and "cudaErrorLaunchFailure" in str(err.value)
        assert "launch" in str(err.value)
        s.step(r)  # the hook turned itself off
        s.sync_info()
        for view in ("canvas", "entropy", "sample"):
            assert torch.equal(getattr(s, view)(), getattr(fresh, view)())
        # the second checked call fails: the tick is cut between its kernels
        s.set_state(st0)
        assert dg.lib.dg_debug_fail_cuda_call(1) == dg.DG_OK
        with pytest.raises(dg.DGError) as err:
            s.step(r)
        assert err.value.status == dg.DG_ERR_CUDA
        s.set_state(st0)
        s.step(r)
        s.sync_info()
        for view in ("canvas", "entropy", "sample"):
            assert torch.equal(getattr(s, view)(), getattr(fresh, view)())
        assert dg.lib.dg_debug_fail_cuda_call(-2) == dg.DG_ERR_ARG
    finally:
        dg.lib.dg_debug_fail_cuda_call(-1)
        s.close()
        fresh.close()


def test_batched_model_scale_sampled_rows():
    """16 canvases x 256 positions at V=2^18, d=2816 (the batched configuration with every canvas
    active: 16 row tiles of the SM-pair LM head per vocabulary chunk), one tick; sampled positions
    across the canvases against the oracle computed for those rows alone."""
    import torch
    import uniform_state_discrete_gb300 as dg
    B, L, V, d = 16, 256, 262144, 2816
    case = Case(vocab=V, hidden=d, canvas_len=L, n_canvases=B, steps=48, seeds=tuple(range(B)))
    W = weights(case)
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    ocfg = case.oracle_cfg()
    s = dg.Sampler(case.gpu_cfg(), w_dev)
    st = s.get_state()
    canv = np.arange(B)
    resid = resid_slots(case, ocfg, W, canv, np.zeros(B, np.int64), np.zeros(B, np.int64), st["tokens"])
    s.step(torch.from_numpy(resid).to(dev))
    H, lz = s.entropy().cpu().numpy(), s.logz().cpu().numpy()
    y, am = s.sample().cpu().numpy(), s.argmax().cpu().numpy()
    rng = np.random.default_rng(3)
    pick = [(c, int(p)) for c in range(B) for p in rng.choice(L, 2, replace=False)]
    r = np.stack([resid[c, p] for c, p in pick])
    h = oracle.rmsnorm_bf16(r, ocfg.rms_eps)
    z = oracle.logits(h, W)
    T = oracle.temperature(0, ocfg.num_inference_steps, ocfg.t_min, ocfg.t_max)
    ref = oracle.stats(z, T, np.array([ocfg.seed(c) for c, _ in pick], np.uint64), 0, 0,
                       np.array([p for _, p in pick], np.int32))
    for i, (c, p) in enumerate(pick):
        assert abs(float(H[c, p]) - ref["H"][i]) <= 1e-3
        assert abs(float(lz[c, p]) - ref["logZ"][i]) <= 1e-3 * abs(ref["logZ"][i])
        assert y[c, p] == ref["y"][i] or ref["ggap"][i] < 1e-4
        assert am[c, p] == ref["amax"][i] or ref["zgap"][i] < 1e-4


_W_MODEL = {}


def _model_weights():
    """The model-scale W (V=2^18, d=2816, seed 0), generated once per session."""
    if "w" not in _W_MODEL:
        _W_MODEL["w"] = synth.wvocab(0, 262144, 2816)
    return _W_MODEL["w"]


@pytest.mark.parametrize("sigma", [0.1, 2.0])
@pytest.mark.parametrize("t_max,t_min", [(0.8, 0.4), (1.5, 0.1)])
@pytest.mark.parametrize("bound", [0.01, 0.1, 1.0])
def test_stress_config_sweep_point(bound, t_max, t_min, sigma):
    """The stress configuration at full size: 64 canvases x 4 blocks x 256 positions, V=2^18,
    d=2816, one point of its sweep.  The first tick's sampled positions against the oracle; then
    the whole run with the device residual generator, checking at every tick what holds at any
    size: frozen positions keep their tokens, every step commits at least one position while any is
    open, tokens stay in [0, V), and each finished block's heatmap holds steps of that block."""
    import torch
    import uniform_state_discrete_gb300 as dg
    B, G, L, V, d, N = 64, 4, 256, 262144, 2816, 48
    W = _model_weights()
    case = Case(vocab=V, hidden=d, canvas_len=L, n_canvases=B, gen_blocks=G, steps=N, bound=bound, t_max=t_max,
                t_min=t_min, sigma=sigma, seeds=tuple(range(B)))
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    ocfg = case.oracle_cfg()
    stream = torch.cuda.Stream(dev)
    s = dg.Sampler(case.gpu_cfg(), w_dev, stream=stream)
    resid = torch.empty(B, L, d, dtype=torch.float32, device=dev)

    def make_resid():
        synth.resid_device(w_dev.data_ptr(), s.canvas().data_ptr(), s.slots_ptr(), B, L, V, d, sigma, resid.data_ptr(),
                           stream.cuda_stream)

    prev = s.get_state()
    with torch.cuda.stream(stream):
        make_resid()
    stream.synchronize()
    # first tick: sampled positions against the oracle on the same residual rows
    r0 = resid.cpu().numpy()
    with torch.cuda.stream(stream):
        s.step(resid)
    s.sync_info()
    H, y = s.entropy().cpu().numpy(), s.sample().cpu().numpy()
    lz, am = s.logz().cpu().numpy(), s.argmax().cpu().numpy()
    pick = [(c, p) for c, p in zip(range(0, B, 8), (0, 37, 74, 111, 148, 185, 222, 255))]
    h = oracle.rmsnorm_bf16(np.stack([r0[c, p] for c, p in pick]), ocfg.rms_eps)
    ref = oracle.stats(oracle.logits(h, W), oracle.temperature(0, N, ocfg.t_min, ocfg.t_max),
                       np.array([ocfg.seed(c) for c, _ in pick], np.uint64), 0, 0,
                       np.array([p for _, p in pick], np.int32))
    for i, (c, p) in enumerate(pick):
        assert abs(float(H[c, p]) - ref["H"][i]) <= 1e-3
        assert abs(float(lz[c, p]) - ref["logZ"][i]) <= 1e-3 * abs(ref["logZ"][i])
        assert y[c, p] == ref["y"][i] or ref["ggap"][i] < 1e-4
        assert am[c, p] == ref["amax"][i] or ref["zgap"][i] < 1e-4
    # the whole run
    for tick in range(1, G * N + 2):
        cur = s.get_state()
        for c in range(B):
            a, b = prev["slots"][c], cur["slots"][c]
            assert np.all((cur["tokens"][c] >= 0) & (cur["tokens"][c] < V))
            if a["state"] != dg.ACTIVE:
                continue
            if b["block"] == a["block"] and b["state"] == dg.ACTIVE:
                frozen = prev["committed"][c] != 0
                assert np.array_equal(cur["tokens"][c][frozen], prev["tokens"][c][frozen])
                assert np.all(cur["committed"][c][frozen] != 0)
                # at least one commit per step while any position is open
                assert b["n_committed"] > a["n_committed"] or a["n_committed"] == L
                assert b["step"] == a["step"] + 1
            else:  # the block ended at this tick
                blk = a["block"]
                assert np.all((cur["tokens_out"][c, blk] >= 0) & (cur["tokens_out"][c, blk] < V))
                hm = cur["commit_steps_out"][c, blk]
                assert np.all((hm >= 0) & (hm <= a["step"]))
        prev = cur
        if np.all(cur["slots"]["state"] == dg.DONE):
            break
        with torch.cuda.stream(stream):
            make_resid()
            s.step(resid)
    info = s.sync_info()
    assert np.all(info["state"] == dg.DONE)
    assert np.all(info["steps_used"] <= G * N)
    if sigma == 0.1 and bound == 1.0:
        assert info["converged_blocks"].sum() > 0  # peaked distributions stop early
    s.close()


def _final_state_of_run(case, W, sigma, mode):
    """Run a sampler to completion with the device residual generator and return its final state.
    mode "serial": the host waits for every tick; "async": ticks are enqueued back to back with no
    host synchronisation until the end (each LM head starts under the previous tick's finishing
    kernel); "graph": each tick is a replay of one captured CUDA graph of dg_denoise_step."""
    import torch
    import uniform_state_discrete_gb300 as dg
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.Stream(dev)
    s = dg.Sampler(case.gpu_cfg(), w_dev, stream=stream)
    B, L, V, d = case.n_canvases, case.canvas_len, case.vocab, case.hidden
    resid = torch.empty(B, L, d, dtype=torch.float32, device=dev)
    ticks = case.gen_blocks * case.steps + (max(case.admit) if case.admit else 0)

    def gen():
        synth.resid_device(w_dev.data_ptr(), s.canvas().data_ptr(), s.slots_ptr(), B, L, V, d, sigma, resid.data_ptr(),
                           stream.cuda_stream)

    graph = None
    if mode == "graph":
        with torch.cuda.stream(stream):
            gen()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            s.step(resid)  # captured, not run
    for t in range(ticks):
        with torch.cuda.stream(stream):
            gen()
            if graph is not None:
                graph.replay()
            else:
                s.step(resid)
        if mode == "serial":
            s.sync_info()
    info = s.sync_info()  # also reports any error latched on the way
    assert np.all(info["state"] == dg.DONE)
    st = s.get_state()
    s.close()
    return st


@pytest.mark.parametrize("case,sigma", [
    pytest.param(Case(vocab=2048, hidden=128, canvas_len=16, n_canvases=3, gen_blocks=3, steps=8, seeds=(1, 2, 3),
                      admit=(0, 2, 5)), 0.5, id="single-cta"),
    pytest.param(Case(vocab=32768, hidden=1024, canvas_len=256, gen_blocks=2, steps=48), 0.5, id="canvas256-v32k"),
    pytest.param(Case(vocab=262144, hidden=2816, canvas_len=256, n_canvases=64, gen_blocks=4, steps=48,
                      seeds=tuple(range(64))), 2.0, id="stress64x4-v262k"),
])
def test_back_to_back_ticks_equal_serialised_ticks(case, sigma):
    """The hand-off between a tick's kernels and the next tick's (counters released and acquired on
    the device, the next LM head launched under the finishing kernel) gives the same run whether
    the host waits after every tick, enqueues every tick back to back, or replays a captured CUDA
    graph of the tick: every token, heatmap entry and slot counter of the final state is equal."""
    W = _model_weights() if case.vocab == 262144 else weights(case)
    modes = ("serial", "async", "graph") if case.vocab < 262144 else ("serial", "async")
    runs = {m: _final_state_of_run(case, W, sigma, m) for m in modes}
    ref = runs["serial"]
    for m in modes[1:]:
        for key in ("tokens_out", "commit_steps_out", "tokens", "committed"):
            assert np.array_equal(runs[m][key], ref[key]), f"{m}: {key} differs from the serialised run"
        for f in ("state", "block", "step", "steps_used", "n_committed", "converged_blocks"):
            assert np.array_equal(runs[m]["slots"][f], ref["slots"][f]), f"{m}: slot field {f} differs"


def _device_free_run(case, W, sigma, max_ticks):
    """Run a sampler to completion with the device residual generator; returns it."""
    import torch
    import uniform_state_discrete_gb300 as dg
    dev = torch.device("cuda:0")
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.Stream(dev)
    s = dg.Sampler(case.gpu_cfg(), w_dev, stream=stream)
    resid = torch.empty(case.n_canvases, case.canvas_len, case.hidden, dtype=torch.float32, device=dev)
    for _ in range(max_ticks):
        if np.all(s.sync_info()["state"] == dg.DONE):
            break
        with torch.cuda.stream(stream):
            synth.resid_device(w_dev.data_ptr(), s.canvas().data_ptr(), s.slots_ptr(), case.n_canvases,
                               case.canvas_len, case.vocab, case.hidden, sigma, resid.data_ptr(), stream.cuda_stream)
            s.step(resid)
    return s


def test_batched_config_staggered_admission_invariance():
    """The batched configuration as specified: 16 canvases x 256 positions at V=2^18, d=2816, seeds
    0..15 admitted at ticks 12 * (c // 4).  Each canvas's tokens equal those of the same canvas
    run alone (TensorSharp doc, "7. Test coverage": batched decode equals per-sequence decode)."""
    import uniform_state_discrete_gb300 as dg
    W = _model_weights()
    B = 16
    batch = Case(vocab=262144, hidden=2816, canvas_len=256, n_canvases=B, steps=48, seeds=tuple(range(B)),
                 admit=tuple(12 * (c // 4) for c in range(B)))
    s = _device_free_run(batch, W, 0.5, 48 + 36 + 2)
    info = s.sync_info()
    assert np.all(info["state"] == dg.DONE) and np.all(info["steps_used"] == 48)
    tok = s.tokens_out().cpu().numpy()
    s.close()
    for c in (0, 5, 15):
        alone = _device_free_run(Case(vocab=262144, hidden=2816, canvas_len=256, steps=48, seeds=(c,)), W, 0.5, 50)
        assert np.array_equal(alone.tokens_out().cpu().numpy()[0], tok[c])
        alone.close()
