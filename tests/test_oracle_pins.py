"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks one oracle function against something other than itself:
published known-answer vectors, closed forms, library routines for special
cases, brute force on tiny inputs, statistical laws, and the pages' own
printed defaults and figures (tests/golden/, each file citing its source).
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
import synth
from oracle.sampler import entropy_bounded_accept, temperature


# --------------------------------------------------------------------------- Philox
def test_philox_known_answer_vectors(golden):
    rows = golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for row in rows:
        v = [int(x, 16) for x in row]
        assert list(oracle.philox(v[:4], v[4:6])) == v[6:10]
        # the shared input generator carries its own Philox; pin it to the same vectors
        assert list(synth.philox4x32_10(v[:4], v[4:6])) == v[6:10]


# ------------------------------------------------------------- uniform integers
def test_uniform_token_power_of_two_is_top_bits():
    rng = np.random.default_rng(0)
    for k in (1, 11, 15, 18):
        for u in rng.integers(0, 2 ** 32, size=200):
            assert oracle.uniform_token(int(u), 1 << k) == int(u) >> (32 - k)


def test_uniform_token_interval_edges():
    for V in (2, 3, 1000, 262144, 2 ** 31 - 1):
        assert oracle.uniform_token(0, V) == 0
        assert oracle.uniform_token(2 ** 32 - 1, V) == V - 1
        for j in (1, V // 2, V - 1):
            u = -(-(j << 32) // V)  # first word that maps to j
            assert oracle.uniform_token(u, V) == j
            assert oracle.uniform_token(u - 1, V) == j - 1


def test_renoise_tokens_are_uniform():
    V = 16
    counts = np.zeros(V)
    for s in range(40):
        for p in range(256):
            counts[oracle.uniform_token(oracle.draw_u32(7, oracle.PURPOSE_RENOISE, 0, s, p), V)] += 1
    assert scipy.stats.chisquare(counts).pvalue > 1e-3
    init = [oracle.draw_u32(7, oracle.PURPOSE_INIT, 0, 0, p) for p in range(64)]
    ren = [oracle.draw_u32(7, oracle.PURPOSE_RENOISE, 0, 0, p) for p in range(64)]
    blk = [oracle.draw_u32(7, oracle.PURPOSE_INIT, 1, 0, p) for p in range(64)]
    assert init != ren and init != blk


# ----------------------------------------------------------------------- bf16 RNE
def test_bf16_rne_ties_and_double_rounding():
    assert oracle.bf16_rne(1.0) == 0x3F80
    assert oracle.bf16_rne(-1.0) == 0xBF80
    assert oracle.bf16_rne(1 + 2 ** -8) == 0x3F80            # tie -> even (down)
    assert oracle.bf16_rne(1 + 3 * 2 ** -8) == 0x3F82        # tie -> even (up)
    assert oracle.bf16_rne(1 + 2 ** -8 + 2 ** -30) == 0x3F81  # above the tie; an fp32 detour would say 0x3F80
    assert oracle.bf16_rne(2.0 ** -130) == 0x0008            # subnormal: 8 quanta of 2^-133
    assert oracle.bf16_rne(3.3895313892515355e38) == 0x7F7F  # largest finite bf16
    assert oracle.bf16_rne(3.4e38) == 0x7F80                 # past the halfway point -> +inf
    assert oracle.bf16_rne(0.0) == 0


def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------------ RMSNorm
def test_rmsnorm_constant_vector_gives_weight():
    d = 128
    for a in (0.5, -3.0, 1e-3):
        h = oracle.rmsnorm_bf16(np.full((1, d), a, np.float32), eps=0.0)
        assert np.all(h == (0x3F80 if a > 0 else 0xBF80))
    w = np.linspace(-2, 2, d).astype(np.float32)
    h = oracle.rmsnorm_bf16(np.full((1, d), 0.25, np.float32), eps=0.0, w=w)
    assert np.array_equal(h[0], np.array([oracle.bf16_rne(float(v)) for v in w], dtype=np.uint16))


def test_rmsnorm_unit_rms_scale_invariance_and_nearest():
    rng = np.random.default_rng(2)
    r = rng.standard_normal((6, 1024)).astype(np.float32) * 3.0
    h = oracle.rmsnorm_bf16(r, eps=0.0)
    hv = oracle.bf16_value(h)
    # output has unit root-mean-square (the sqrt(D) factor), up to bf16 rounding
    assert np.allclose(np.sqrt(np.mean(hv ** 2, axis=1)), 1.0, rtol=2 ** -8)
    # exact power-of-two rescaling of the input leaves every bit unchanged
    assert np.array_equal(oracle.rmsnorm_bf16(r * np.float32(8.0), eps=0.0), h)
    # each output is the bf16 value nearest to the fp64 quotient
    exact = r.astype(np.float64) * math.sqrt(1024) / np.sqrt(np.sum(r.astype(np.float64) ** 2, axis=1, keepdims=True))
    ulp = 2.0 ** (np.floor(np.log2(np.abs(exact))) - 7)
    assert np.all(np.abs(hv - exact) <= ulp / 2 + 1e-300)
    # eps enters next to the norm: a large eps shrinks the output by norm / (norm + eps)
    h_eps = oracle.bf16_value(oracle.rmsnorm_bf16(r[:1], eps=float(np.linalg.norm(r[0].astype(np.float64)))))
    assert np.allclose(h_eps, oracle.bf16_value(oracle.rmsnorm_bf16(r[:1], eps=0.0)) / 2, rtol=2 ** -7)


# ------------------------------------------------------------------------- logits
def test_logits_hand_case():
    h = np.array([[oracle.bf16_rne(1.0), oracle.bf16_rne(2.0)]], dtype=np.uint16)
    Wv = [[1, 0], [0, 1], [1, 1], [0.5, -2]]
    W = np.array([[oracle.bf16_rne(a) for a in row] for row in Wv], dtype=np.uint16)
    assert np.array_equal(oracle.logits(h, W), [[1.0, 2.0, 3.0, -3.5]])
    assert np.array_equal(oracle.logits_loop(h, W), [[1.0, 2.0, 3.0, -3.5]])


def test_logits_blas_matches_triple_loop():
    h = synth.wvocab(11, 5, 192, sigma_w=1.0)
    W = synth.wvocab(12, 777, 192)
    a, b = oracle.logits(h, W, block_rows=100), oracle.logits_loop(h, W)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------- softmax / entropy / log Z
def _stats1(z, T=1.0, seed=0, block=0, step=0, pos=0):
    return oracle.stats(np.atleast_2d(np.asarray(z, np.float64)), T, seed, block, step, pos)


def test_uniform_logits_entropy_is_log_V(golden):
    for V_s, lnV_s, printed in golden("uniform_entropy.txt"):
        V, lnV = int(V_s), float(lnV_s)
        st = _stats1(np.full(V, 0.3), T=0.8)
        assert abs(st["H"][0] - lnV) < 5e-7
        assert abs(st["H"][0] - math.log(V)) < 1e-9
        assert abs(st["logZ"][0] - (math.log(V) + 0.3 / 0.8)) < 1e-9
        assert st["amax"][0] == 0 and st["zgap"][0] == 0.0  # ties resolve to the lowest index
        if printed != "-":
            assert round(st["H"][0], 2) == float(printed)


def test_one_hot_limit_closed_form():
    V = 1000
    for delta in (0.5, 3.0, 12.0, 40.0):
        z = np.zeros(V)
        z[17] = delta * 0.7
        st = _stats1(z, T=0.7)
        q = (V - 1) * math.exp(-delta)
        H = math.log1p(q) + q * delta / (1 + q)
        assert abs(st["H"][0] - H) < 1e-12 + 1e-10 * H
        assert st["amax"][0] == 17 and abs(st["zgap"][0] - delta) < 1e-12


def test_two_point_is_binary_entropy():
    for a in (-4.0, -0.3, 0.0, 1.7, 9.0):
        st = _stats1([0.0, a])
        p = 1 / (1 + math.exp(-a))
        Hb = -(p * math.log(p) + (1 - p) * math.log(1 - p))
        assert abs(st["H"][0] - Hb) < 1e-12


def test_entropy_and_logz_match_library_routines():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((4, 3000)) * np.array([[0.1], [1.0], [4.0], [20.0]])
    T = 0.6
    st = oracle.stats(z, T, 0, 0, 0, np.arange(4))
    p = scipy.special.softmax(z / T, axis=1)
    assert np.allclose(st["H"], scipy.stats.entropy(p, axis=1), rtol=1e-10, atol=1e-12)
    assert np.allclose(st["H_online"], st["H"], rtol=1e-10, atol=1e-12)
    assert np.allclose(st["logZ"], scipy.special.logsumexp(z / T, axis=1), rtol=1e-13)
    assert np.array_equal(st["amax"], np.argmax(z, axis=1))


def test_temperature_divides_logits():
    rng = np.random.default_rng(4)
    z = rng.standard_normal((3, 500)) * 2
    a = oracle.stats(z, 0.45, 9, 1, 5, np.arange(3))
    b = oracle.stats(z / 0.45, 1.0, 9, 1, 5, np.arange(3))
    for f in ("H", "logZ", "gbest"):
        assert np.allclose(a[f], b[f], rtol=1e-12)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["amax"], b["amax"])


def test_gumbel_sample_follows_softmax():
    V, n, T = 8, 16000, 0.7
    z = np.array([0.0, 0.4, -1.0, 1.1, 0.2, -0.3, 0.9, 0.05])
    st = oracle.stats(np.tile(z, (n, 1)), T, 123, 0, 3, np.arange(n))
    counts = np.bincount(st["y"], minlength=V)
    expect = scipy.special.softmax(z / T) * n
    assert scipy.stats.chisquare(counts, expect).pvalue > 1e-3
    # a different step or block re-keys the draws
    st2 = oracle.stats(np.tile(z, (n, 1)), T, 123, 0, 4, np.arange(n))
    assert (st2["y"] != st["y"]).mean() > 0.5


def test_gumbel_sample_follows_softmax_across_groups():
    """40 entries span two whole groups of 16 and a partial one: the sample still follows softmax."""
    V, n, T = 40, 24000, 0.9
    z = np.random.default_rng(8).uniform(-1.5, 1.5, V)
    st = oracle.stats(np.tile(z, (n, 1)), T, 77, 1, 5, np.arange(n))
    counts = np.bincount(st["y"], minlength=V)
    assert scipy.stats.chisquare(counts, scipy.special.softmax(z / T) * n).pvalue > 1e-3


def _exp_variates(n, V, seed=11, block=0, step=2):
    return np.stack([oracle.exp_variates(seed, block, step, p, V) for p in range(n)])


def test_exp_variates_marginals_are_exponential():
    """Every entry's E_v is Exp(1) (Kolmogorov-Smirnov over 3000 positions), including the entries
    of a partial last group (V = 40)."""
    E = _exp_variates(3000, 40)
    pvals = [scipy.stats.kstest(E[:, v], "expon").pvalue for v in range(40)]
    assert min(pvals) > 1e-4, min(pvals)
    assert abs(E.mean() - 1.0) < 0.02


def test_exp_variates_group_minimum_slot_and_independence():
    """Renyi's representation: the minimum of a group of 16 is Exp(16), the slot holding it is
    uniform over the 16, and the entries of a group are uncorrelated."""
    n = 4000
    E = _exp_variates(n, 32, seed=3, block=1, step=7)
    for g in range(2):
        grp = E[:, 16 * g:16 * g + 16]
        assert scipy.stats.kstest(16.0 * grp.min(axis=1), "expon").pvalue > 1e-3
        assert scipy.stats.chisquare(np.bincount(grp.argmin(axis=1), minlength=16)).pvalue > 1e-3
        c = np.corrcoef(grp.T)
        assert np.max(np.abs(c - np.eye(16))) < 5.0 / math.sqrt(n)
    # the two groups draw independently
    assert abs(np.corrcoef(E[:, :16].min(axis=1), E[:, 16:].min(axis=1))[0, 1]) < 5.0 / math.sqrt(n)


def test_exp_variates_sorted_spacings_are_exponential():
    """For i.i.d. Exp(1) variates, the k-th spacing of the sorted sixteen, scaled by 16 - k, is Exp(1)
    and independent of the others (Renyi, 1953): checked for the first, a middle and the last
    spacing of each group over 4000 positions."""
    n = 4000
    E = np.sort(_exp_variates(n, 32, seed=21, block=3, step=9).reshape(n, 2, 16), axis=2)
    gaps = np.diff(np.concatenate([np.zeros((n, 2, 1)), E], axis=2), axis=2) * (16 - np.arange(16))
    for k in (0, 1, 7, 15):
        for g in range(2):
            assert scipy.stats.kstest(gaps[:, g, k], "expon").pvalue > 1e-3, (k, g)
    assert abs(np.corrcoef(gaps[:, 0, 1], gaps[:, 0, 2])[0, 1]) < 5.0 / math.sqrt(n)


def test_exp_variates_rekey_with_position_step_block_and_seed():
    base = oracle.exp_variates(5, 0, 0, 0, 64)
    for args in ((6, 0, 0, 0), (5, 1, 0, 0), (5, 0, 1, 0), (5, 0, 0, 1)):
        assert np.mean(oracle.exp_variates(*args, 64) != base) > 0.9


def test_gumbel_sample_is_argmax_of_perturbed_logits():
    """The sample stats() reports is argmax_v (z_v/T - ln E_v) of the oracle's own variates."""
    V, T = 50, 0.6
    rng = np.random.default_rng(4)
    z = rng.standard_normal((20, V))
    st = oracle.stats(z, T, 9, 2, 3, np.arange(20))
    for p in range(20):
        s = z[p] / T - np.log(oracle.exp_variates(9, 2, 3, p, V))
        assert st["y"][p] == int(np.argmax(s))
        assert abs(st["gbest"][p] - s.max()) < 1e-12


def test_gumbel_sample_of_dominant_token_is_argmax():
    V = 4096
    z = np.random.default_rng(5).standard_normal(V)
    z[1234] = 80.0  # a 70-nat margin exceeds any Gumbel spread a 32-bit uniform can produce (< 24 nats)
    st = oracle.stats(np.tile(z, (50, 1)), 1.0, 1, 0, 0, np.arange(50))
    assert np.all(st["y"] == 1234) and np.all(st["amax"] == 1234)


def test_gumbel_sample_uniform_when_logits_equal():
    V, n = 64, 12800
    st = oracle.stats(np.zeros((n, V)), 0.5, 42, 2, 7, np.arange(n))
    assert scipy.stats.chisquare(np.bincount(st["y"], minlength=V)).pvalue > 1e-3


# ------------------------------------------------------- self-conditioning input
def test_expected_embedding_uniform_logits_is_mean_embedding():
    """Equal logits: P is uniform, so P W is the mean of the W rows."""
    W = synth.wvocab(1, 300, 24, sigma_w=0.3)
    e, a = oracle.expected_embedding(np.full((3, 300), 0.7), 0.5, W)
    mean = np.array([[np.mean([float(oracle.bf16_value(W[v, k])) for v in range(300)]) for k in range(24)]])
    np.testing.assert_allclose(e, np.repeat(mean, 3, axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(a, np.repeat(np.abs(oracle.bf16_value(W)).mean(axis=0, keepdims=True), 3, 0),
                               atol=1e-14)


def test_expected_embedding_of_a_dominant_token_is_its_row():
    W = synth.wvocab(2, 512, 16, sigma_w=0.3)
    z = np.random.default_rng(3).standard_normal((2, 512))
    z[0, 77] = 60.0  # a 40-nat margin at T = 1: every other weight is below e^-40
    z[1, 500] = 60.0
    e, _ = oracle.expected_embedding(z, 1.0, W)
    np.testing.assert_allclose(e[0], oracle.bf16_value(W[77]), atol=1e-12)
    np.testing.assert_allclose(e[1], oracle.bf16_value(W[500]), atol=1e-12)


def test_expected_embedding_two_point_closed_form():
    """Two finite logits: e = s W_a + (1 - s) W_b with s = sigmoid((z_a - z_b) / T)."""
    W = synth.wvocab(4, 64, 8, sigma_w=0.3)
    z = np.full((1, 64), -np.inf)
    z[0, 5], z[0, 40] = 0.9, -0.3
    e, _ = oracle.expected_embedding(z, 0.6, W)
    s_ = 1.0 / (1.0 + math.exp(-(0.9 + 0.3) / 0.6))
    np.testing.assert_allclose(e[0], s_ * oracle.bf16_value(W[5]) + (1 - s_) * oracle.bf16_value(W[40]), atol=1e-15)


def test_expected_embedding_is_a_convex_combination_and_temperature_sharpens_it():
    W = synth.wvocab(5, 1000, 32, sigma_w=0.3)
    Wv = oracle.bf16_value(W)
    z = np.random.default_rng(6).standard_normal((4, 1000))
    for T in (0.3, 1.0, 3.0):
        e, a = oracle.expected_embedding(z, T, W)
        assert np.all(e >= Wv.min(axis=0) - 1e-15) and np.all(e <= Wv.max(axis=0) + 1e-15)
        assert np.all(np.abs(e) <= a + 1e-15)
    # as T -> 0 the distribution collapses onto the argmax token
    e0, _ = oracle.expected_embedding(z, 1e-3, W)
    np.testing.assert_allclose(e0, Wv[np.argmax(z, axis=1)], atol=1e-12)


# ------------------------------------------------- top-K self-conditioning input
def test_topk_embedding_keeping_every_token_is_the_dense_one():
    """k >= V keeps the whole distribution: the dense expected embedding (itself pinned above)."""
    W = synth.wvocab(7, 300, 24, sigma_w=0.3)
    z = np.random.default_rng(8).standard_normal((5, 300))
    dense, da = oracle.expected_embedding(z, 0.7, W)
    for k in (300, 1000):
        e, a, gap, sel = oracle.expected_embedding_topk(z, 0.7, W, k)
        np.testing.assert_allclose(e, dense, rtol=0, atol=1e-14)
        np.testing.assert_allclose(a, da, rtol=0, atol=1e-14)
        assert np.all(np.isinf(gap)) and sel.shape == (5, 300)


def test_topk_embedding_of_one_token_is_the_argmax_row_with_ties_to_the_lower_index():
    W = synth.wvocab(9, 128, 16, sigma_w=0.3)
    z = np.random.default_rng(10).standard_normal((3, 128))
    z[0, 17] = 9.0
    z[1, 90] = z[1, 33] = 9.0  # a tie: the lower index is kept
    z[2, 127] = 9.0
    e, _, gap, sel = oracle.expected_embedding_topk(z, 0.5, W, 1)
    assert list(sel[:, 0]) == [17, 33, 127]
    np.testing.assert_array_equal(e, oracle.bf16_value(W[[17, 33, 127]]))
    assert gap[1] == 0.0 and gap[0] > 0 and gap[2] > 0


def test_topk_embedding_of_equal_logits_is_the_mean_of_the_first_k_rows():
    """Every token equally likely: ties go to the lower index, so the first k rows are kept with
    equal weights."""
    W = synth.wvocab(11, 200, 12, sigma_w=0.3)
    for k in (1, 7, 32):
        e, _, gap, sel = oracle.expected_embedding_topk(np.full((2, 200), -1.25), 0.9, W, k)
        assert np.all(sel == np.arange(k)) and np.all(gap == 0.0)
        mean = [sum(float(oracle.bf16_value(W[v, j])) for v in range(k)) / k for j in range(12)]
        np.testing.assert_allclose(e, np.array([mean, mean]), rtol=0, atol=1e-15)


def test_topk_embedding_two_kept_tokens_closed_form():
    """k = 2 of many tokens: the two largest logits are renormalised between themselves,
    e = s W_a + (1 - s) W_b with s = sigmoid((z_a - z_b) / T), whatever the other logits are."""
    W = synth.wvocab(12, 64, 8, sigma_w=0.3)
    z = np.random.default_rng(13).uniform(-3.0, 0.0, (1, 64))
    z[0, 50], z[0, 9] = 2.0, 1.4
    e, _, gap, sel = oracle.expected_embedding_topk(z, 0.8, W, 2)
    s_ = 1.0 / (1.0 + math.exp(-(2.0 - 1.4) / 0.8))
    np.testing.assert_allclose(e[0], s_ * oracle.bf16_value(W[50]) + (1 - s_) * oracle.bf16_value(W[9]), atol=1e-15)
    assert list(sel[0]) == [50, 9]
    assert abs(gap[0] - (1.4 - np.sort(z[0])[-3]) / 0.8) < 1e-15


def test_topk_embedding_matches_brute_force_over_subsets():
    """The kept set maximises the sum of the kept logits over all k-subsets (unique for distinct
    logits), and the weights are the softmax restricted to it: the coordinate of W that is 1 for
    every token gives 1 exactly, and adding a constant to every logit changes nothing."""
    rng = np.random.default_rng(14)
    V, d = 9, 6
    W = synth.wvocab(15, V, d, sigma_w=0.3)
    Wv = oracle.bf16_value(W)
    W1 = W.copy()
    W1[:, 0] = 0x3F80  # bf16 1.0
    for k in (1, 2, 4, 8):
        z = rng.standard_normal((3, V))
        e, _, _, sel = oracle.expected_embedding_topk(z, 0.6, W, k)
        for p in range(3):
            best = max(itertools.combinations(range(V), k), key=lambda s: sum(z[p, list(s)]))
            assert set(sel[p]) == set(best)
            q = np.exp(z[p, list(best)] / 0.6)
            q /= q.sum()
            np.testing.assert_allclose(e[p], q @ Wv[list(best)], rtol=0, atol=1e-14)
        e1, _, _, _ = oracle.expected_embedding_topk(z, 0.6, W1, k)
        np.testing.assert_allclose(e1[:, 0], 1.0, rtol=0, atol=1e-15)
        e2, _, _, _ = oracle.expected_embedding_topk(z + 3.5, 0.6, W, k)
        np.testing.assert_allclose(e2, e, rtol=0, atol=1e-14)


# ----------------------------------------------------------------- commit rule
def test_acceptance_matches_pages_prefix_expression():
    """The pages' acceptance: sort H, accept where cumsum(sH) - sH <= bound ("Denoise, stage,
    commit, and generate").  Evaluated here with numpy's stable sort and cumulative sum."""
    rng = np.random.default_rng(6)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        H = rng.exponential(rng.choice([0.001, 0.03, 0.3, 3.0]), n)
        bound = float(rng.choice([0.0, 0.01, 0.1, 1.0]))
        order, excl, k = entropy_bounded_accept(H, range(n), bound)
        idx = np.argsort(H, kind="stable")
        sH = H[idx]
        ok = (np.cumsum(sH) - sH) <= bound
        assert set(order[:k]) == set(idx[ok].tolist())


def test_acceptance_brute_force_and_properties():
    rng = np.random.default_rng(7)
    for trial in range(200):
        n = int(rng.integers(1, 9))
        H = np.round(rng.exponential(0.05, n), 3)  # rounding creates exact ties
        bound = float(rng.choice([0.0, 0.02, 0.1, 0.5]))
        order, excl, k = entropy_bounded_accept(H, range(n), bound)
        acc = set(order[:k])
        # brute force: the accepted set is the unique subset A that is a lowest-(H,p) prefix,
        # whose own exclusive sums all fit in the bound, and that cannot be extended
        keyed = sorted(range(n), key=lambda p: (H[p], p))
        cands = []
        for m in range(1, n + 1):
            for A in itertools.combinations(range(n), m):
                if set(A) != set(keyed[:m]):
                    continue
                fits = all(sum(H[q] for q in keyed[:j]) <= bound for j in range(m))
                extends = m < n and sum(H[q] for q in keyed[:m]) <= bound
                if fits and not extends:
                    cands.append(set(A))
        assert cands == [acc]
        assert k >= 1
        if np.all(H > bound):
            assert k == 1
        k_big = entropy_bounded_accept(H, range(n), bound + 0.3)[2]
        assert k_big >= k


def test_acceptance_regime_one_per_step_when_all_entropies_exceed_bound():
    H = np.array([7.5, 7.49, 7.52, 7.48])
    order, excl, k = entropy_bounded_accept(H, [0, 1, 2, 3], 0.1)
    assert k == 1 and order[0] == 3


# ------------------------------------------------------------------- schedule
def test_schedule_closed_form_and_defaults(golden):
    d = {k: v for k, v in golden("sampler_defaults.txt")}
    N, tmin, tmax = int(d["num_inference_steps"]), float(d["t_min"]), float(d["t_max"])
    for s, T in golden("schedule.txt"):
        assert abs(temperature(int(s), N, tmin, tmax) - float(T)) < 1e-15
    for s in range(N):
        t = (N - s) / N  # the node page's schedule position, decreasing 1 -> 1/N
        assert abs(temperature(s, N, tmin, tmax) - (tmin + (tmax - tmin) * t)) < 1e-15
    assert temperature(N - 1, N, tmin, tmax) > tmin  # t_min is never applied


# ------------------------------------------------------------------- the loop
def _cfg0(**kw):
    base = dict(vocab=2048, hidden=128, canvas_len=16, num_inference_steps=8, seeds=[0])
    base.update(kw)
    return oracle.OracleConfig(**base)


def _run(cfg, W, sigma, on_tick=None):
    s = oracle.OracleSampler(cfg, W)
    fn = oracle.sampler.synth_resid_fn(cfg, W, sigma)
    s.run(fn, on_tick=on_tick)
    return s


def test_loop_invariants_tiny_config():
    cfg = _cfg0()
    W = synth.wvocab(0, cfg.vocab, cfg.hidden)
    seen = {}
    frozen = np.zeros((1, cfg.canvas_len), bool)
    tokens = {}

    def on_tick(rec):
        st = rec.step[0]
        n_new = rec.n_accepted[0]
        assert n_new >= 1
        if st < cfg.num_inference_steps - 1:
            assert n_new == 1  # every entropy ~7.5 nats >> bound: exactly one commit per step
        seen[st] = n_new

    s = oracle.OracleSampler(cfg, W)
    fn = oracle.sampler.synth_resid_fn(cfg, W, 0.5)
    while not s.done():
        before = s.x.copy(), s.committed.copy()
        rec = s.tick(fn)
        on_tick(rec)
        # committed tokens never change
        assert np.array_equal(s.x[before[1]], before[0][before[1]]) or s.done()
        assert np.all(s.committed >= before[1]) or s.done()
    out = s.tokens_out[0, 0]
    assert np.all((out >= 0) & (out < cfg.vocab))
    assert s.steps_used[0] == cfg.num_inference_steps and s.converged_blocks[0] == 0
    assert sorted(seen) == list(range(cfg.num_inference_steps))
    assert sum(seen.values()) == cfg.canvas_len
    assert np.array_equal(np.sort(np.bincount(s.commit_step[0].astype(np.int64), minlength=8))[:1], [1])


def test_early_stop_returns_argmax_canvas():
    """Peaked distributions (H ~ 0) whose argmax does not move: the canvas stops at the first step
    where the test runs (s = 1) and every position holds its argmax."""
    V, d, L = 64, 128, 16
    cfg = oracle.OracleConfig(vocab=V, hidden=d, canvas_len=L, num_inference_steps=48, seeds=[3])
    W = synth.wvocab(5, V, d, sigma_w=1.0)
    Wf = synth.bf16_to_f32(W)
    fn = lambda canv, blocks, steps, tok: np.concatenate([Wf[:L] for _ in canv])  # r_p = W[p]
    s = oracle.OracleSampler(cfg, W)
    recs = []
    s.run(fn, on_tick=recs.append)
    assert len(recs) == 2 and recs[1].converged[0] and not recs[0].converged[0]
    assert recs[0].n_accepted[0] == L  # all entropies ~0: the whole canvas fits the bound at step 0
    assert np.array_equal(s.tokens_out[0, 0], np.arange(L))
    assert s.steps_used[0] == 2 and s.converged_blocks[0] == 1


def test_no_early_stop_when_argmax_moves():
    V, d, L, N = 64, 128, 8, 6
    cfg = oracle.OracleConfig(vocab=V, hidden=d, canvas_len=L, num_inference_steps=N, seeds=[3])
    W = synth.wvocab(5, V, d, sigma_w=1.0)
    Wf = synth.bf16_to_f32(W)
    fn = lambda canv, blocks, steps, tok: np.concatenate([Wf[(np.arange(L) + steps[0]) % V] for _ in canv])
    s = oracle.OracleSampler(cfg, W)
    s.run(fn)
    assert s.steps_used[0] == N and s.converged_blocks[0] == 0


def test_batch_and_admission_invariance():
    """A canvas's result depends on its own seed only, not on which canvases share its ticks or
    when it was admitted (TensorSharp doc, "7. Test coverage": batched decode is the per-sequence decode)."""
    base = dict(vocab=512, hidden=64, canvas_len=8, num_inference_steps=6)
    W = synth.wvocab(1, 512, 64)
    alone = [_run(oracle.OracleConfig(**base, seeds=[sd]), W, 0.5).tokens_out[0] for sd in (10, 11, 12)]
    both = _run(oracle.OracleConfig(**base, n_canvases=3, seeds=[10, 11, 12], admit_tick=[0, 3, 5]), W, 0.5)
    for c in range(3):
        assert np.array_equal(both.tokens_out[c], alone[c])
    assert both.tick_no == 5 + 6


def test_blocks_run_one_after_another():
    cfg = oracle.OracleConfig(vocab=512, hidden=64, canvas_len=8, num_inference_steps=5, gen_blocks=3, seeds=[4])
    W = synth.wvocab(1, 512, 64)
    s = _run(cfg, W, 0.5)
    assert s.steps_used[0] == 15 and s.tick_no == 15
    assert not np.array_equal(s.tokens_out[0, 0], s.tokens_out[0, 1])
    assert np.all(s.tokens_out >= 0)


def test_multi_commit_regime_low_noise():
    """Low hidden noise makes distributions peaked, several positions fit the bound in one step,
    and the run can stop early; the invariants must still hold."""
    V, d, L = 512, 256, 32
    cfg = oracle.OracleConfig(vocab=V, hidden=d, canvas_len=L, num_inference_steps=24, t_max=0.8, t_min=0.4,
                              entropy_bound=1.0, seeds=[9])
    W = synth.wvocab(2, V, d, sigma_w=0.1)
    recs = []
    s = _run(cfg, W, 0.1, on_tick=recs.append)
    assert max(r.n_accepted[0] for r in recs[:-1]) > 1
    assert int(s.committed[0].sum()) in (0, L)  # block finished: a fresh canvas or all committed
    assert np.all(s.tokens_out[0, 0] >= 0)


def test_committed_token_is_a_sample_not_the_argmax():
    """Accepted positions take a draw from the categorical distribution with logits z/T ("Denoise,
    stage, commit, and generate"), not the argmax: over near-uniform distributions on V=2048 the two
    almost never agree."""
    cfg = _cfg0(n_canvases=4, seeds=[0, 1, 2, 3])
    W = synth.wvocab(0, cfg.vocab, cfg.hidden)
    hits, total = 0, 0
    s = oracle.OracleSampler(cfg, W)
    fn = oracle.sampler.synth_resid_fn(cfg, W, 0.5)
    while not s.done():
        rec = s.tick(fn)
        L = cfg.canvas_len
        for i, c in enumerate(rec.canvases):
            acc = np.nonzero(rec.accepted[i])[0]
            amax = rec.stats["amax"][i * L:(i + 1) * L]
            committed_tok = s.tokens_out[c, 0] if rec.final[i] else s.x[c]
            hits += int(np.sum(committed_tok[acc] == amax[acc]))
            total += acc.size
    assert total == 4 * cfg.canvas_len and hits <= total // 8


# ------------------------------------------------------------ re-accepting commit mode
def _pages_next_canvas(H, y, seed, block, step, bound, V):
    """The next canvas as the Annotated page's denoise code builds it ("Denoise, stage, commit, and
    generate"): sort all entropies, accepted = scatter(cumsum(sH) - sH <= bound), then
    where(accepted, sample, uniform token) over the whole canvas.  numpy's stable sort gives the
    (H, p) tie order; the uniform tokens come from the pinned Philox re-noise draw."""
    idx = np.argsort(H, kind="stable")
    sH = H[idx]
    accepted = np.zeros(H.size, bool)
    accepted[idx] = (np.cumsum(sH) - sH) <= bound
    noise = np.array([oracle.uniform_token(oracle.draw_u32(seed, oracle.PURPOSE_RENOISE, block, step, p), V)
                      for p in range(H.size)])
    return accepted, np.where(accepted, y, noise)


def test_reaccept_rebuilds_the_canvas_as_the_pages_code_does():
    """Moderate hidden noise: several positions fit the bound per step and the accepted set changes
    from step to step, so positions accepted earlier are re-noised; every tick must equal the page's
    expression evaluated on that tick's entropies and samples, and the last step takes every sample."""
    V, d, L = 512, 256, 32
    cfg = oracle.OracleConfig(vocab=V, hidden=d, canvas_len=L, num_inference_steps=12, entropy_bound=1.0,
                              seeds=[9], mode="reaccept", confidence=0.0)
    W = synth.wvocab(2, V, d, sigma_w=0.1)
    s = oracle.OracleSampler(cfg, W)
    fn = oracle.sampler.synth_resid_fn(cfg, W, 0.3)
    remasked = 0
    while not s.done():
        rec = s.tick(fn)
        st = rec.stats
        H, y = st["H"], st["y"]
        if rec.final[0]:
            assert np.array_equal(s.tokens_out[0, 0], y)
            continue
        accepted, x_next = _pages_next_canvas(H, y, 9, int(rec.block[0]), int(rec.step[0]), cfg.entropy_bound, V)
        assert np.array_equal(s.committed[0], accepted)
        assert np.array_equal(s.x[0], x_next)
        assert rec.n_accepted[0] == accepted.sum() == s.committed[0].sum()
        remasked += int(rec.n_remasked[0])
    assert remasked > 0  # the run did re-noise positions accepted at an earlier step


def test_reaccept_remasks_a_position_whose_entropy_rank_rises():
    """Hand-made entropies: position 0 is accepted at step 0; at step 1 two other positions have
    lower entropy and use up the budget, so position 0 is re-noised (and counted), while under the
    freezing mode it would keep its token."""
    V, L = 64, 4
    for mode in ("reaccept", "freeze"):
        cfg = oracle.OracleConfig(vocab=V, hidden=8, canvas_len=L, num_inference_steps=4, entropy_bound=0.1,
                                  confidence=0.0, seeds=[1], mode=mode)
        s = oracle.OracleSampler(cfg, np.zeros((V, 8), np.uint16))
        outs = []
        for step, (H, y) in enumerate((([0.05, 2.0, 3.0, 4.0], [5, 6, 7, 8]),
                                       ([3.0, 0.02, 0.07, 4.0], [9, 10, 11, 12]))):
            st = np.zeros(L, oracle.POS_DTYPE)
            st["H"], st["y"], st["amax"] = H, y, step
            rec = oracle.sampler.TickRecord(
                tick=step, canvases=np.array([0]), block=np.array([0]), step=np.array([step]), T=np.ones(1),
                stats=st, mean_H=np.zeros(1), converged=np.zeros(1, bool), final=np.zeros(1, bool),
                accepted=np.zeros((1, L), bool), n_accepted=np.zeros(1, np.int32),
                flag_y=np.zeros(L, bool), flag_amax=np.zeros(L, bool), flag_commit=np.zeros((1, L), bool),
                flag_canvas=np.zeros(1, bool), n_remasked=np.zeros(1, np.int32))
            s._commit(0, st, rec, 0, oracle.draw_u32, oracle.uniform_token, oracle.PURPOSE_RENOISE)
            s.step_no[0] = step + 1
            outs.append((s.x[0].copy(), s.committed[0].copy(), int(rec.n_remasked[0]), int(rec.n_accepted[0])))
        noise = lambda p, stp: oracle.uniform_token(oracle.draw_u32(1, oracle.PURPOSE_RENOISE, 0, stp, p), V)
        # step 0 (both modes): sorted H 0.05, 2, ...; exclusive sums 0, 0.05, 2.05 -> positions 0 and 1
        x0, c0, r0, k0 = outs[0]
        assert k0 == 2 and list(c0) == [True, True, False, False] and r0 == 0
        assert list(x0) == [5, 6, noise(2, 0), noise(3, 0)]
        x1, c1, r1, k1 = outs[1]
        if mode == "reaccept":
            # all four open: sorted 0.02 (p1), 0.07 (p2), 3 (p0); sums 0, 0.02, 0.09 -> p1, p2, p0 accepted
            assert k1 == 3 and list(c1) == [True, True, True, False] and r1 == 0
            assert list(x1) == [9, 10, 11, noise(3, 1)]
        else:
            # p0, p1 frozen; open p2 (0.07), p3 (4): sums 0, 0.07 -> both accepted
            assert k1 == 2 and list(c1) == [True, True, True, True]
            assert list(x1) == [5, 6, 11, 12]


def test_reaccept_remask_count_matches_mask_difference():
    """n_remasked = |accepted(s-1) minus accepted(s)|, and at high entropy exactly one position is accepted
    per step, so the canvas never keeps more than one accepted position before the last step."""
    cfg = _cfg0(mode="reaccept")
    W = synth.wvocab(0, cfg.vocab, cfg.hidden)
    s = oracle.OracleSampler(cfg, W)
    fn = oracle.sampler.synth_resid_fn(cfg, W, 0.5)
    prev = np.zeros(cfg.canvas_len, bool)
    while not s.done():
        rec = s.tick(fn)
        if rec.final[0]:
            break
        cur = s.committed[0].copy()
        assert rec.n_accepted[0] == 1 and cur.sum() == 1
        assert rec.n_remasked[0] == int(np.sum(prev & ~cur))
        prev = cur


# ------------------------------------------------------------------ logit softcap
def test_softcap_limits_and_shape():
    """"Logit Softcapping": c tanh(z/c) leaves |z| << c essentially unchanged (z - z^3/(3c^2) to
    third order), tends to +-c as z -> +-inf, is odd, monotone and bounded by c, and c -> inf
    (here c = 0 meaning off, and a huge c) gives back the logits."""
    z = np.linspace(-5.0, 5.0, 1001)
    c = 30.0
    zc = oracle.softcap(z, c)
    small = np.abs(z) < 0.5
    assert np.max(np.abs(zc[small] - (z[small] - z[small] ** 3 / (3 * c * c)))) < 1e-7
    assert np.allclose(oracle.softcap(np.array([1e6, -1e6, 1e3]), c), [c, -c, c], rtol=0, atol=1e-12)
    assert np.array_equal(oracle.softcap(-z, c), -zc)
    assert np.all(np.diff(zc) > 0) and np.all(np.abs(zc) < c)
    assert np.array_equal(oracle.softcap(z, 0.0), z)
    assert np.max(np.abs(oracle.softcap(z, 1e9) - z)) < 1e-15 * 1e3


def test_softcap_bounds_the_entropy_of_a_two_point_distribution():
    """Two tokens with logits +-a: after the cap their gap is 2c tanh(a/c), so H is the binary
    entropy of sigmoid(-gap/T), however large a grows (the stats routine on capped logits)."""
    c, T = 2.0, 0.5
    for a in (0.3, 3.0, 300.0):
        z = oracle.softcap(np.array([[a, -a]]), c)
        st = oracle.stats(z, T, 1, 0, 0, np.array([0]))
        gap = 2 * c * math.tanh(a / c) / T
        p = 1.0 / (1.0 + math.exp(gap))
        assert abs(st["H"][0] - (-(p * math.log(p) + (1 - p) * math.log(1 - p)))) < 1e-12


def test_commit_heatmap_of_finished_blocks():
    """The heatmap of a finished block records when each position took its final token.  At high
    entropy (one commit per step, freezing mode) steps 0..N-2 appear exactly once and the last step
    holds every remaining position; under re-acceptance the whole block takes the last step."""
    for mode in ("freeze", "reaccept"):
        cfg = _cfg0(gen_blocks=2, mode=mode)
        W = synth.wvocab(0, cfg.vocab, cfg.hidden)
        s = _run(cfg, W, 0.5)
        N, L = cfg.num_inference_steps, cfg.canvas_len
        for b in range(2):
            hm = s.commit_steps_out[0, b].astype(np.int64)
            if mode == "freeze":
                assert np.array_equal(np.bincount(hm, minlength=N), [1] * (N - 1) + [L - N + 1])
            else:
                assert np.all(hm == N - 1)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_early_stop_needs_k_unchanged_argmax_canvases(k):
    """"the argmax canvas has remained unchanged for stability_threshold previous canvases"
    ("Check for early stopping"): with a constant argmax and entropies ~0 the block stops at the
    first step s with s >= k, i.e. after k + 1 equal argmax canvases."""
    V, d, L = 64, 128, 16
    cfg = oracle.OracleConfig(vocab=V, hidden=d, canvas_len=L, num_inference_steps=48, seeds=[3], stability=k)
    W = synth.wvocab(5, V, d, sigma_w=1.0)
    Wf = synth.bf16_to_f32(W)
    fn = lambda canv, blocks, steps, tok: np.concatenate([Wf[:L] for _ in canv])  # r_p = W[p]
    s = oracle.OracleSampler(cfg, W)
    recs = []
    s.run(fn, on_tick=recs.append)
    assert len(recs) == k + 1 and recs[-1].converged[0] and not any(r.converged[0] for r in recs[:-1])
    assert s.steps_used[0] == k + 1 and s.converged_blocks[0] == 1


def test_early_stop_run_restarts_when_the_argmax_moves():
    """Stability 2: the argmax canvas moves at step 2, so the run of unchanged canvases restarts and
    the block stops at step 4 (canvases 2, 3, 4 equal) instead of step 2."""
    V, d, L = 64, 128, 8
    cfg = oracle.OracleConfig(vocab=V, hidden=d, canvas_len=L, num_inference_steps=48, seeds=[3], stability=2)
    W = synth.wvocab(5, V, d, sigma_w=1.0)
    Wf = synth.bf16_to_f32(W)
    fn = lambda canv, blocks, steps, tok: np.concatenate([Wf[np.arange(L) + (8 if steps[0] >= 2 else 0)]
                                                          for _ in canv])
    s = oracle.OracleSampler(cfg, W)
    recs = []
    s.run(fn, on_tick=recs.append)
    assert [int(r.converged[0]) for r in recs] == [0, 0, 0, 0, 1]
