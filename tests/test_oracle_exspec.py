"""Pins of the oracle's ragged-pool functions (EXSPEC) -- CPU only.

"Correctness Forensics for Batch Speculative Decoding", §3.2: EXSPEC keeps
sequences ragged and batches same-length sequences so realignment is
bypassed; when grouping fails it falls back to unpad-append-repad.  §2: a
variable-length layout still rolls back rejected tokens.  Checked here:
repad gives rectangular alignment (I1) and position/KV correspondence (I2);
unpad after repad is the identity on the pool's valid rows; the commit is a
length update with its errors; and EXSPEC decoding of the toy pair, mixing
grouped rounds and unpad-append-repad fallbacks, reproduces batch-size-1
greedy token for token (App. B's equivalence).  The scheduling policy itself
is this project's construction (the appendix has no body): UNPINNED.
"""
import numpy as np
import pytest

import oracle
from oracle import DT_F32
from oracle.toy import ToyPair, run_exspec
from specgen import kv_row_values


def test_commit_ragged():
    pl = np.array([5, 9, 3, 7], np.int32)
    assert oracle.commit_ragged(pl, [2, 0], [4, 1], 16) == 0
    assert list(pl) == [6, 9, 7, 7]
    before = pl.copy()
    assert oracle.commit_ragged(pl, [1, 1], [1, 1], 16) == 2  # repeated index
    assert oracle.commit_ragged(pl, [4], [1], 16) == 2  # outside the pool
    assert oracle.commit_ragged(pl, [0], [-1], 16) == 2
    assert oracle.commit_ragged(pl, [1, 3], [1, 10], 16) == 1  # 7 + 10 > 16: nothing changes
    assert np.array_equal(pl, before)


def make_pool(lens, S, L=1, H=2, D=3, seed=0):
    rng = np.random.default_rng(seed)
    N = len(lens)
    pool = rng.standard_normal((L, 2, N, H, S, D)).astype(np.float32)  # junk everywhere
    toks = [list(rng.integers(0, 50, size=n)) for n in lens]
    for n in range(N):
        for p in range(lens[n] - 1):
            pool[:, :, n, :, p, :] = kv_row_values(n, toks[n][p], p, L, H, D)
    return pool, np.array(lens, np.int32), toks


def test_repad_gives_rectangular_alignment_and_correspondence():
    pool, pl, toks = make_pool([5, 12, 2, 9, 12, 7], 24)
    L, _, N, H, S, D = pool.shape
    idx = [3, 0, 4, 2]
    batch = np.full((L, 2, len(idx), H, S, D), 3.5, np.float32)
    st, ln, pad, W = oracle.repad_gather(pool, batch, idx, pl)
    assert st == 0 and W == 12
    assert (pad + ln == W).all() and pad.min() == 0  # I1
    for b, n in enumerate(idx):
        for p in range(pl[n] - 1):  # I2
            assert np.array_equal(batch[:, :, b, :, pad[b] + p, :], kv_row_values(n, toks[n][p], p, L, H, D))
        untouched = [s for s in range(S) if not pad[b] <= s < pad[b] + ln[b] - 1]
        assert (batch[:, :, b, :, untouched, :] == 3.5).all()
    # unpad right back: the pool's valid rows are unchanged, its lengths too
    pool2, pl2 = pool.copy(), pl.copy()
    assert oracle.unpad_scatter(batch, pool2, idx, ln, pad, pl2) == 0
    assert np.array_equal(pool2, pool) and np.array_equal(pl2, pl)


def test_repad_unpad_errors():
    pool, pl, _ = make_pool([4, 6], 8)
    L, _, N, H, S, D = pool.shape
    batch = np.zeros((L, 2, 2, H, S, D), np.float32)
    assert oracle.repad_gather(pool, batch, [0, 0], pl)[0] == 2
    assert oracle.repad_gather(pool, batch, [0, 2], pl)[0] == 2
    assert not batch.any()
    assert oracle.unpad_scatter(batch, pool, [0, 1], [4, 10], [0, 0], pl.copy()) == 2  # 9 rows past S = 8


CASES = [
    # N, B, window, k, alpha, n_new, eos, prompt lengths
    (8, 2, 4, 2, 0.7, 12, -1, [3, 3, 5, 2, 5, 3, 4, 6]),
    (10, 3, 6, 3, 0.5, 14, -1, [4, 4, 4, 2, 7, 7, 1, 5, 5, 3]),
    (6, 2, 2, 2, 0.9, 10, 4, [2, 5, 5, 3, 2, 6]),
    (9, 4, 9, 1, 0.3, 9, -1, [3, 1, 2, 3, 3, 2, 1, 3, 2]),
]


def oracle_ops():
    return dict(
        group=lambda lens, B: oracle.group_by_length(lens, B),
        verify=lambda x, d, rem, eos: oracle.verify_greedy(x, DT_F32, d, None, eos, rem),
        commit=oracle.commit_ragged,
        repad=oracle.repad_gather,
        realign=oracle.realign_kv,
        unpad=lambda b, p, i, ln, pad, pl, ne=None: oracle.unpad_scatter(
            b, p, i, ln if ne is None else np.asarray(ln, np.int32) + ne, pad, pl),
    )


@pytest.mark.parametrize("N,B,window,k,alpha,n_new,eos,lens", CASES)
def test_exspec_decoding_equals_single_sequence_greedy(N, B, window, k, alpha, n_new, eos, lens):
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=alpha, seed=N * 7 + B)
    rng = np.random.default_rng(N + B)
    prompts = [list(rng.integers(0, 11, size=n)) for n in lens]
    S = max(lens) + n_new + 2 * (k + 1) + 8
    gen, rounds, grouped = run_exspec(pair, prompts, n_new, k, S, B, window, oracle_ops(), eos_id=eos)
    for n in range(N):
        assert gen[n] == pair.ref_generate(n, prompts[n], n_new, eos_id=eos), n
    assert rounds > 0 and 0 <= grouped <= rounds


def test_both_round_kinds_occur_and_planted_mistakes_diverge():
    N, B, window, k = 10, 3, 6, 3
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=0.5, seed=77)
    rng = np.random.default_rng(3)
    prompts = [list(rng.integers(0, 11, size=n)) for n in [4, 4, 4, 2, 7, 7, 1, 5, 5, 3]]
    S = 60
    gen, rounds, grouped = run_exspec(pair, prompts, 14, k, S, B, window, oracle_ops())
    assert 0 < grouped < rounds  # grouped rounds and unpad-append-repad fallbacks both ran
    ops = oracle_ops()
    ops["commit"] = lambda pl, idx, ne, S: oracle.commit_ragged(pl, idx, np.maximum(ne - 1, 0), S)
    bad, _, _ = run_exspec(pair, prompts, 14, k, S, B, window, ops)
    assert any(bad[n] != pair.ref_generate(n, prompts[n], 14) for n in range(N))


@pytest.mark.parametrize("N,B,window,k,alpha,n_new,eos,lens", CASES)
def test_fallback_without_realignment_leaves_the_same_pool(N, B, window, k, alpha, n_new, eos, lens):
    """A fallback round unpadded straight from the extended batch (lengths
    len + n_emit at the old paddings) leaves the pool byte for byte as
    realign-then-unpad does, round after round."""
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=alpha, seed=N * 7 + B)
    rng = np.random.default_rng(N + B)
    prompts = [list(rng.integers(0, 11, size=n)) for n in lens]
    S = max(lens) + n_new + 2 * (k + 1) + 8
    a, b = {}, {}
    r1 = run_exspec(pair, prompts, n_new, k, S, B, window, oracle_ops(), eos_id=eos, result=a)
    r2 = run_exspec(pair, prompts, n_new, k, S, B, window, oracle_ops(), eos_id=eos, fallback_realign=False, result=b)
    assert r1 == r2
    assert np.array_equal(a["pool_len"], b["pool_len"])
    assert np.array_equal(a["pool"].view(np.uint32), b["pool"].view(np.uint32))
