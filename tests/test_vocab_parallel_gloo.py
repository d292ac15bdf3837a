"""The vocabulary-parallel split on the CPU: two ranks over gloo.

Each rank holds the W rows of its vocabulary chunks only (dg_vocab_slice) and forms, for every
position, one record per chunk of its range -- max, sum of exponentials, sum of exponentials times
the shifted logit, best perturbed score and the two indices -- from the oracle's logits of its
slice and the oracle's Gumbel variates at global vocabulary indices.  The records are exchanged
with the package's ``all_gather_partials`` (pack, all-gather, unpack into the [rows, chunks]
layout), and every rank then merges all chunks of a position: log Z, the entropy, the sample and
the argmax must be those the oracle computes over the whole vocabulary.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

V, D, ROWS, T, SEED = 1024 + 300, 64, 6, 0.7, 5  # 6 tiles of 256 -> 6 chunks, the last one ragged


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    import oracle
    import synth
    W = synth.wvocab(3, V, D, sigma_w=0.2)
    r = np.random.default_rng(1).standard_normal((ROWS, D)).astype(np.float32)
    return W, oracle.rmsnorm_bf16(r, 1e-6)


def _records(z, E, v0, chunk_ranges_v):
    """Per-chunk records (m, S, A, g, amax, gidx) of logits z [rows, v1 - v0] in natural units."""
    rows = z.shape[0]
    out = np.zeros((rows, len(chunk_ranges_v), 6))
    for k, (a, b) in enumerate(chunk_ranges_v):
        zz = z[:, a - v0:b - v0] / T
        m = zz.max(axis=1)
        e = np.exp(zz - m[:, None])
        sc = zz - np.log(E[:, a:b])
        out[:, k] = np.stack([m, e.sum(1), (e * (zz - m[:, None])).sum(1), sc.max(1), a + zz.argmax(1),
                              a + sc.argmax(1)], axis=1)
    return out


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import oracle
    import uniform_state_discrete_gb300 as dg
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    W, h = _inputs()
    tiles = math.ceil(V / 256)
    n_chunks = tiles  # fewer than 76 tiles: one tile per chunk
    v0, v1 = dg.vocab_slice(V, world, rank)
    z = oracle.logits(h, W[v0:v1])  # this rank's W rows only
    E = np.stack([oracle.exp_variates(SEED, 0, 0, p, V) for p in range(ROWS)])
    slices = [dg.vocab_slice(V, world, q) for q in range(world)]
    chunk_ranges = [(a // 256, math.ceil(b / 256)) for a, b in slices]
    records = torch.zeros((ROWS, n_chunks, 6), dtype=torch.float64)
    c0, c1 = chunk_ranges[rank]
    records[:, c0:c1] = torch.from_numpy(
        _records(z, E, v0, [(256 * c, min(256 * c + 256, V)) for c in range(c0, c1)]))
    dg.all_gather_partials(records, chunk_ranges, rank)
    rec = records.numpy()
    m = rec[:, :, 0].max(axis=1)
    f = np.exp(rec[:, :, 0] - m[:, None])
    S = (f * rec[:, :, 1]).sum(1)
    A = (f * (rec[:, :, 2] + (rec[:, :, 0] - m[:, None]) * rec[:, :, 1])).sum(1)
    y = rec[np.arange(ROWS), rec[:, :, 3].argmax(1), 5].astype(int)
    am = rec[np.arange(ROWS), rec[:, :, 0].argmax(1), 4].astype(int)
    out.put((rank, (v0, v1), chunk_ranges, m + np.log(S), np.log(S) - A / S, y, am))
    dist.barrier()
    dist.destroy_process_group()


def test_vocab_split_over_two_gloo_ranks_matches_whole_vocabulary():
    import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    W, h = _inputs()
    want = oracle.stats(oracle.logits(h, W), T, SEED, 0, 0, np.arange(ROWS, dtype=np.int32))
    # the two slices tile the vocabulary at chunk boundaries
    assert res[0][1][0] == 0 and res[0][1][1] == res[1][1][0] and res[1][1][1] == V and res[0][1][1] % 256 == 0
    for rank, _, _, logz, H, y, am in res:
        np.testing.assert_allclose(logz, want["logZ"], rtol=1e-12)
        np.testing.assert_allclose(H, want["H"], rtol=1e-9, atol=1e-12)
        assert np.array_equal(y, want["y"]) and np.array_equal(am, want["amax"])
