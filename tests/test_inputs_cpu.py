"""The seeded input generator (synth/) produces the workloads' stated distributions: W_vocab entries
N(0, 0.02^2) rounded to bf16, and hidden residual rows W[x_p] + sigma N(0, 1) noise, the noise
independent across positions, steps and seeds.  Kolmogorov-Smirnov tests against the normal law,
moments, and re-keying checks; no GPU."""
import numpy as np
import scipy.stats

import synth


def test_wvocab_entries_are_normal_with_the_stated_spread():
    W = synth.bf16_to_f32(synth.wvocab(0, 4096, 64))
    x = W.reshape(-1).astype(np.float64)
    assert abs(x.mean()) < 3 * 0.02 / np.sqrt(x.size)
    assert abs(x.std() / 0.02 - 1.0) < 0.01
    # bf16 keeps 8 significant bits: test against the normal law at a resolution above that rounding
    assert scipy.stats.kstest(x / 0.02, "norm").pvalue > 1e-3
    # another seed gives other values, the same seed the same
    assert not np.array_equal(synth.wvocab(1, 64, 64), synth.wvocab(0, 64, 64))
    assert np.array_equal(synth.wvocab(0, 64, 64), synth.wvocab(0, 64, 64))


def test_residual_noise_is_normal_and_keyed_by_seed_block_step_and_position():
    V, d, n = 512, 256, 400
    W16 = synth.wvocab(3, V, d)
    Wf = synth.bf16_to_f32(W16)
    rng = np.random.default_rng(0)
    tok = rng.integers(0, V, n).astype(np.int32)
    pos = np.arange(n, dtype=np.int32)
    for sigma in (0.1, 0.5, 2.0):
        r = synth.resid_rows(np.full(n, 7, np.uint64), 1, 5, pos, tok, W16, sigma)
        noise = (r.astype(np.float64) - Wf[tok]) / sigma
        assert scipy.stats.kstest(noise.reshape(-1), "norm").pvalue > 1e-3
        # independent across positions: neighbouring rows uncorrelated
        c = np.corrcoef(noise[:-1].reshape(-1), noise[1:].reshape(-1))[0, 1]
        assert abs(c) < 4 / np.sqrt(noise[1:].size)
    base = synth.resid_rows(np.full(n, 7, np.uint64), 1, 5, pos, tok, W16, 0.5)
    for kw in (dict(seeds=np.full(n, 8, np.uint64), block=1, step=5), dict(seeds=np.full(n, 7, np.uint64), block=2,
                                                                           step=5),
               dict(seeds=np.full(n, 7, np.uint64), block=1, step=6)):
        other = synth.resid_rows(kw["seeds"], kw["block"], kw["step"], pos, tok, W16, 0.5)
        assert np.mean(other == base) < 0.01  # re-keyed noise: almost no value repeats
