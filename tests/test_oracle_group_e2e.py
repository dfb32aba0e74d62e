"""Pins of the oracle's grouping policy and the end-to-end equivalence test.

Grouping: the pages describe EXSPEC's same-length scheduling but print no
algorithm, so the policy (largest length bucket, ties to the smaller length,
members by index, fill by nearest length) is this project's construction and
its parity is UNPINNED by the pages.  It is checked here against an
independent restatement by sorting, on every small case.

End to end: "Correctness Forensics for Batch Speculative Decoding", App. B --
with I1 and I2 maintained every round and the bonus from the target, batched
speculative greedy decoding reproduces per-sequence decoding under exact
arithmetic.  The toy pair makes every step exact, so the check is bit for bit;
planted mistakes in the realignment or the position rebuild must diverge.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import DT_F32
from oracle.toy import ToyPair, run_batch_spec


def group_by_sorting(lens, B, active=None):
    act = [i for i in range(len(lens)) if active is None or active[i]]
    if not act:
        return [-1] * B, 0, -1
    counts = {}
    for i in act:
        counts[lens[i]] = counts.get(lens[i], 0) + 1
    Lstar = sorted(counts.items(), key=lambda kv: (-kv[1], kv[0]))[0][0]
    members = sorted(i for i in act if lens[i] == Lstar)[:B]
    rest = sorted((i for i in act if i not in members), key=lambda i: (abs(lens[i] - Lstar), i))
    idx = (members + rest)[:B]
    return idx + [-1] * (B - len(idx)), len(members), Lstar


def test_grouping_matches_restatement():
    rng = np.random.default_rng(0)
    for N in range(0, 11):
        for trial in range(30):
            lens = rng.integers(1, 5, size=N).astype(np.int32)
            active = rng.random(N) < 0.8 if trial % 2 else None
            for B in (1, 3, 8, 12):
                idx, ce, gl = oracle.group_by_length(lens, B, None if active is None else active.astype(np.uint8))
                r_idx, r_ce, r_gl = group_by_sorting(list(lens), B, active)
                assert list(idx) == r_idx and ce == r_ce and gl == r_gl


def test_grouping_degenerate_cases():
    idx, ce, gl = oracle.group_by_length(np.full(10, 7, np.int32), 4)
    assert list(idx) == [0, 1, 2, 3] and ce == 4 and gl == 7
    idx, ce, gl = oracle.group_by_length(np.array([5, 3], np.int32), 4)
    assert list(idx) == [1, 0, -1, -1] and ce == 1 and gl == 3  # tie -> smaller length
    idx, ce, gl = oracle.group_by_length(np.array([5, 3], np.int32), 2, np.zeros(2, np.uint8))
    assert list(idx) == [-1, -1] and ce == 0 and gl == -1
    idx, ce, gl = oracle.group_by_length(np.zeros(0, np.int32), 3)
    assert list(idx) == [-1, -1, -1] and ce == 0 and gl == -1


# -- end-to-end ----------------------------------------------------------------

def oracle_verify(logits, draft, remaining, eos):
    return oracle.verify_greedy(logits, DT_F32, draft, None, eos, remaining)


def oracle_realign(kv, ln, pad, ne):
    return oracle.realign_kv(kv, ln, pad, ne)


def oracle_posmask(S, pad_new, pad_old, pos, mask):
    oracle.rebuild_pos_mask(S, pad_new, pos, mask)


CASES = [
    # B, k, alpha, n_new, eos
    (3, 2, 0.7, 14, -1),
    (5, 4, 0.5, 16, -1),
    (4, 3, 0.9, 18, 5),
    (1, 3, 0.6, 12, -1),
    (6, 1, 0.3, 10, 3),
]


@pytest.mark.parametrize("B,k,alpha,n_new,eos", CASES)
def test_batch_speculative_equals_single_sequence_greedy(B, k, alpha, n_new, eos):
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=alpha, seed=B * 10 + k)
    rng = np.random.default_rng(B + k)
    prompts = [list(rng.integers(0, 11, size=int(rng.integers(1, 9)))) for _ in range(B)]
    S = 9 + n_new + 2 * (k + 1) + 8
    gen = run_batch_spec(pair, prompts, n_new, k, S, oracle_verify, oracle_realign, oracle_posmask, eos_id=eos)
    for b in range(B):
        ref = pair.ref_generate(b, prompts[b], n_new, eos_id=eos)
        assert gen[b] == ref, (b, gen[b], ref)


@pytest.mark.parametrize("name", ["skip_kv_shift", "stale_positions", "shift_one_short", "bonus_always",
                                  "row_shift"])
def test_planted_mistakes_diverge(name):
    B, k = 4, 3
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=0.6, seed=3)
    rng = np.random.default_rng(42)
    prompts = [list(rng.integers(0, 11, size=int(rng.integers(1, 9)))) for _ in range(B)]
    n_new, S = 16, 48
    with oracle.mutant(name):
        gen = run_batch_spec(pair, prompts, n_new, k, S, oracle_verify, oracle_realign, oracle_posmask)
    refs = [pair.ref_generate(b, prompts[b], n_new) for b in range(B)]
    assert any(g != r for g, r in zip(gen, refs))
