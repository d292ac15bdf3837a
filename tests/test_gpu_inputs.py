"""The benchmark's device residual generator (synth/synth_gpu.cu) against the host generator the
parity tests use (synth/synth.c): both evaluate r = fp32(W_bf16[x_p] + sigma n) with n the
Box-Muller normal of the same Philox counter, in fp64, but with different math libraries (CUDA's on
the device, the C library's on the host), so a value may differ in its last fp32 bit where the fp64
results round differently; every other value is equal.  Rows of canvases that are not active are
left alone."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V,d,L,sigma", [(2048, 128, 16, 0.5), (32768, 1024, 256, 2.0), (1000, 200, 37, 0.1)])
def test_device_residuals_equal_host_residuals(V, d, L, sigma):
    import torch
    import uniform_state_discrete_gb300 as dg
    dev = torch.device("cuda:0")
    B = 3
    W = synth.wvocab(5, V, d)
    w_dev = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    # canvases 0 and 1 active from the first tick, canvas 2 admitted later (not active yet)
    s = dg.Sampler(dg.make_config(V, d, L, n_canvases=B, num_inference_steps=8, seeds=[11, 12, 13],
                                  admit_tick=[0, 0, 5]), w_dev)
    out = torch.full((B, L, d), 7.0, dtype=torch.float32, device=dev)
    info = s.sync_info()
    tok = s.canvas().cpu().numpy()
    stream = torch.cuda.current_stream(dev)
    synth.resid_device(w_dev.data_ptr(), s.canvas().data_ptr(), s.slots_ptr(), B, L, V, d, sigma, out.data_ptr(),
                       stream.cuda_stream)
    got = out.cpu().numpy()
    act = np.nonzero(info["state"] == dg.ACTIVE)[0]
    assert list(act) == [0, 1]
    want = synth.resid_rows(np.repeat(info["seed"][act], L), np.repeat(info["block"][act], L),
                            np.repeat(info["step"][act], L), np.tile(np.arange(L), act.size),
                            tok[act].reshape(-1), W, sigma).reshape(act.size, L, d)
    g = got[act]
    same = g.view(np.int32) == want.view(np.int32)
    ulps = np.abs(g.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    print(f"\n[inputs V={V} d={d}] equal bit for bit: {same.mean():.6f}; largest difference {ulps.max()} ulp")
    assert ulps.max() <= 1 and same.mean() > 0.999
    assert np.all(got[2] == 7.0)  # the canvas not yet admitted is not written
    s.close()
