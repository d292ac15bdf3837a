"""The workspace-free LM-head statistics entry point against a sampler tick, through the C ABI.

``dg_lmhead_stats_static`` keeps its scratch in one array inside the library
that every call shares, so this file is named to be collected last: it has to
pass alone and after every other test of the session has run in the same
process.  Its GPU test runs two calls in a row (two consecutive ticks of one
canvas) and compares each against the sampler's own outputs for that tick:
entropy and log Z within the parity tolerances, sample and argmax exactly
(both sides merge the same partial records in the same order); and against the
CPU oracle on the same rows, under the parity rules of tests/parity.py.
"""
import gc

import numpy as np
import pytest

import oracle
import synth

TOL_H = 1e-3
TOL_LOGZ_REL = 1e-3


def test_static_entry_rejects_sizes_beyond_its_scratch():
    """Sizes above the static scratch are refused with DG_ERR_ARG before anything touches the device."""
    import uniform_state_discrete_gb300 as dg
    import ctypes

    msg = ctypes.create_string_buffer(256)
    fake = ctypes.c_void_p(256)

    def call(rows, hidden, vocab=1000):
        return dg.lib.dg_lmhead_stats_static(fake, rows, fake, vocab, hidden, None, 1e-6, 1.0, 0, 0, 0, fake, fake,
                                             fake, fake, None, msg, len(msg))

    assert call(257, 1024) == dg.DG_ERR_ARG and b"256" in msg.value
    assert call(0, 1024) == dg.DG_ERR_ARG
    assert call(128, 4104) == dg.DG_ERR_ARG and b"4096" in msg.value
    assert call(128, 1020) == dg.DG_ERR_ARG  # not a multiple of 8
    assert call(128, 1024, vocab=1) == dg.DG_ERR_ARG


CASES = [
    # rows, vocab, hidden, RMSNorm weight seed (None: all ones)
    pytest.param(256, 32768, 1024, None, id="pair-lmhead-256x32k"),
    pytest.param(100, 1000, 200, 3, id="single-lmhead-ragged"),
    pytest.param(256, 262144, 2816, None, id="pair-lmhead-256x262k"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("rows,vocab,hidden,norm_seed", CASES)
def test_static_entry_matches_sampler_on_two_calls(rows, vocab, hidden, norm_seed):
    import torch
    import uniform_state_discrete_gb300 as dg

    dev = torch.device("cuda:0")
    seed, sigma, eps = 11, 0.5, float(np.float32(1e-6))
    w16 = synth.wvocab(0, vocab, hidden)
    W = torch.from_numpy(w16.view(np.int16)).to(dev).view(torch.bfloat16)
    nw = torch.from_numpy(synth.norm_weight(norm_seed, hidden)).to(dev) if norm_seed is not None else None
    s = dg.Sampler(dg.make_config(vocab, hidden, rows, n_canvases=1, num_inference_steps=8, rms_eps=eps,
                                  seeds=[seed]), W, nw)
    H = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
    lz = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
    y = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    am = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    temps = []
    for call in range(2):
        st = s.get_state()
        slot = st["slots"][0]
        assert slot["state"] == dg.ACTIVE and int(slot["step"]) == call
        block, step, T = int(slot["block"]), int(slot["step"]), float(slot["temperature"])
        temps.append(T)
        resid = torch.from_numpy(synth.canvas_resid(seed, block, step, st["tokens"][0], w16, sigma)).to(dev)
        s.step(resid)
        gc.collect()  # objects of earlier tests freed now, not during the call
        torch.cuda.synchronize(dev)
        torch_bytes = torch.cuda.memory_allocated(dev)
        free_before = torch.cuda.mem_get_info(dev)[0]
        dg.dg_lmhead_stats_static(resid, W, nw, eps, T, seed, block, step, H, lz, y, am, stream=s.stream)
        torch.cuda.synchronize(dev)
        assert torch.cuda.memory_allocated(dev) <= torch_bytes
        # nothing allocated outside torch either.  The first call on the device looks up the static
        # array's address, which makes the driver load the library's module that holds it (the
        # array itself, 2.7 MB, and the module's code); in a fresh process that is this call.  The
        # second call allocates nothing at all.
        slack = (16 << 20) if call == 0 else (1 << 20)
        assert torch.cuda.mem_get_info(dev)[0] >= free_before - slack
        ref_H, ref_lz = s.entropy()[0].cpu().numpy(), s.logz()[0].cpu().numpy()
        ref_y, ref_am = s.sample()[0].cpu().numpy(), s.argmax()[0].cpu().numpy()
        got_H, got_lz, got_y, got_am = H.cpu().numpy(), lz.cpu().numpy(), y.cpu().numpy(), am.cpu().numpy()
        dH = np.abs(got_H - ref_H).max()
        dlz = (np.abs(got_lz - ref_lz) / np.abs(ref_lz)).max()
        print(f"\n[{rows}x{vocab}x{hidden} call {call}] T={T} max|dH|={dH:.3g} max|dlogZ|/|logZ|={dlz:.3g} "
              f"H bit-equal={np.array_equal(got_H, ref_H)}")
        assert np.isfinite(got_H).all() and np.isfinite(got_lz).all()
        assert dH <= TOL_H and dlz <= TOL_LOGZ_REL
        np.testing.assert_array_equal(got_y, ref_y)
        np.testing.assert_array_equal(got_am, ref_am)
        # and against the CPU oracle directly, on the same rows
        r = resid.cpu().numpy().reshape(rows, hidden)
        want = oracle.stats(oracle.logits(oracle.rmsnorm_bf16(r, eps, None if nw is None else nw.cpu().numpy()), w16),
                            T, seed, block, step, np.arange(rows, dtype=np.int32))
        assert np.abs(got_H - want["H"]).max() <= TOL_H
        assert (np.abs(got_lz - want["logZ"]) / np.abs(want["logZ"])).max() <= TOL_LOGZ_REL
        assert np.all((got_y == want["y"]) | (want["ggap"] < 1e-4))
        assert np.all((got_am == want["amax"]) | (want["zgap"] < 1e-4))
    assert temps[0] != temps[1]  # the second call runs at the next step's temperature
    s.close()
