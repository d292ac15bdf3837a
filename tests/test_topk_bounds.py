"""The facts the top-K self-conditioning kernels rely on to narrow a row down to a few candidates,
checked on the CPU over rows of many shapes (no GPU, no library):

- the K-th largest of the maxima of disjoint subsets of a row (each thread's strided share of its
  16-byte groups, or each 256-wide vocabulary chunk) is at most the row's K-th largest value, so
  every entry of the top K reaches it;
- rounding to bf16 (round to nearest even) keeps order, so an entry whose rounded probability lies
  below the bound's rounded value lies below every entry of the top K;
- the margin the candidate bound is lowered by, 2^-12 (|u| + 1), is positive and below the spacing
  of the largest values of a smooth row, so it admits few extra candidates."""
import numpy as np
import pytest


def kth_largest(x, k):
    return np.sort(x)[::-1][k - 1]


def thread_maxima(row, threads=256, group=8):
    """Each thread's maximum over the 8-entry groups i, i + threads, i + 2 threads, ... (padded with -inf)."""
    n = -(-row.size // group) * group
    padded = np.full(n, -np.inf)
    padded[:row.size] = row
    g = padded.reshape(-1, group).max(axis=1)
    return np.array([g[t::threads].max() if g[t::threads].size else -np.inf for t in range(threads)])


def chunk_maxima(row, tiles_per_chunk, tile=256):
    w = tiles_per_chunk * tile
    return np.array([row[c:c + w].max() for c in range(0, row.size, w)])


def rows():
    rng = np.random.default_rng(1)
    for V in (200, 2048, 32768, 262144):
        yield rng.standard_normal(V)                      # smooth
        yield np.full(V, 0.25)                            # a plateau: every value equal
        r = rng.standard_normal(V) * 0.01
        r[rng.integers(0, V, 5)] = 40.0                   # a few dominant entries
        yield r
        yield np.sort(rng.standard_normal(V))             # the largest values all in the last chunk


@pytest.mark.parametrize("K", [1, 8, 32, 74, 256])
def test_kth_largest_subset_maximum_bounds_the_kth_largest_entry(K):
    for row in rows():
        kk = min(K, row.size)
        t = kth_largest(row, kk)
        assert kth_largest(thread_maxima(row), kk) <= t
        V = row.size
        n_vt = -(-V // 256)
        tpc = -(-n_vt // 76)  # at most 76 chunks of equal tile counts, as the library lays them out
        cm = chunk_maxima(row, tpc)
        if kk <= cm.size:
            b = kth_largest(cm, kk)
            assert b <= t
            # every entry of the top K reaches the bound, and at least K entries do
            top = np.sort(row)[::-1][:kk]
            assert np.all(top >= b) and np.sum(row >= b) >= kk


def bf16_rne(x):
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32)


def test_bf16_rounding_keeps_order_of_nonnegative_values():
    rng = np.random.default_rng(2)
    x = np.sort(np.concatenate([rng.random(200000).astype(np.float32) * 10.0 ** rng.integers(-30, 1, 200000),
                                np.float32([0.0, 1e-38, 1.0])]))
    k = bf16_rne(x)
    assert np.all(np.diff(k.astype(np.int64)) >= 0)  # a larger value never rounds to a smaller pattern


def test_candidate_margin_is_small_and_positive():
    u = np.array([-300.0, -20.0, -1.0, 0.0, 1.0, 30.0, 300.0])
    margin = 2.0 ** -12 * (np.abs(u) + 1.0)
    assert np.all(margin > 0) and np.all(margin <= 0.08)
    # below the median spacing of the 32 largest of 2^18 normal logits in the kernel's units
    # (z log2(e) / T), so lowering the bound by it admits about one more candidate a row
    rng = np.random.default_rng(3)
    for T in (0.4, 0.1):
        u = rng.standard_normal(262144) / T * 1.4426950408889634
        top = np.sort(u)[::-1][:33]
        m = 2.0 ** -12 * (abs(top[0]) + 1.0)
        assert np.median(-np.diff(top)) > 5 * m
        assert np.sum((u < top[31]) & (u >= top[31] - m)) <= 3
