"""Pins of the oracle's realignment and position/mask rebuild (CPU only).

Checked from first principles, independently of the oracle's own code:
  I1 rectangular alignment -- pad'_b + len'_b is the same for every b and
     some sequence has no padding;
  I2 position-ID/KV correspondence -- slot pad'_b + p holds the synthetic KV
     f(b, token_p, p) for every p < len'_b - 1, and the position IDs of the
     non-pad slots are 0, 1, 2, ... ("Correctness Forensics for Batch
     Speculative Decoding", §3.1 and App. B);
  only the destination runs change; B = 1 and uniform acceptance change
  nothing (App. B); brute force over every commit vector for B <= 3, k <= 2.
"""
import itertools

import numpy as np
import pytest

import oracle
from specgen import kv_row_values


def make_state(lens, k, S, L=1, H=2, D=3, seed=0, dtype=np.float32):
    """Left-padded cache after a verification forward: prefix KV for
    positions < len_b - 1, the k+1 query slots W-1 .. W+k-1 holding the last
    token and k proposals, every other slot a 'never valid' pattern."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    lens = np.array(lens, np.int32)
    W = int(lens.max())
    pad = (W - lens).astype(np.int32)
    kv = np.zeros((L, 2, B, H, S, D), dtype)
    toks = [list(rng.integers(0, 50, size=lens[b])) for b in range(B)]
    props = rng.integers(0, 50, size=(B, k))
    for b in range(B):
        for s in range(S):
            kv[:, :, b, :, s, :] = kv_row_values(b, 999_000 + s, 0, L, H, D)  # junk pattern
        for p in range(lens[b] - 1):
            kv[:, :, b, :, pad[b] + p, :] = kv_row_values(b, toks[b][p], p, L, H, D)
        q = [toks[b][-1]] + list(props[b])
        for j, t in enumerate(q):
            kv[:, :, b, :, W - 1 + j, :] = kv_row_values(b, int(t), lens[b] - 1 + j, L, H, D)
    return kv, lens, pad, toks, props


def expected_tokens(toks, props, n):
    """History after committing n tokens: accepted proposals are the first
    n - 1 committed tokens (the last one is a correction/bonus whose value does
    not matter for the KV, which it does not have yet)."""
    return [list(toks[b]) + list(props[b][: max(n[b] - 1, 0)]) + ([-1] if n[b] > 0 else [])
            for b in range(len(toks))]


def check_invariants(kv0, kv, lens, pad, n, len_new, pad_new, W_new, hist):
    L, _, B, H, S, D = kv.shape
    # I1
    assert (pad_new + len_new == W_new).all() and pad_new.min() == 0
    assert (len_new == lens + n).all()
    for b in range(B):
        # I2: every position below len'_b - 1 holds f(b, token, position)
        for p in range(len_new[b] - 1):
            want = kv_row_values(b, int(hist[b][p]), p, L, H, D)
            assert np.array_equal(kv[:, :, b, :, pad_new[b] + p, :], want), (b, p)
        # nothing outside the destination run changed
        run = set(range(pad_new[b], pad_new[b] + len_new[b] - 1))
        for s in range(S):
            if s not in run:
                assert np.array_equal(kv[:, :, b, :, s, :], kv0[:, :, b, :, s, :]), (b, s)


@pytest.mark.parametrize("B,k", [(1, 1), (1, 2), (2, 1), (2, 2), (3, 1), (3, 2)])
def test_brute_force_all_commit_vectors(B, k):
    S = 24
    for lens in itertools.product([1, 3, 6], repeat=B):
        kv0, ln, pad, toks, props = make_state(lens, k, S, seed=sum(lens))
        for n in itertools.product(range(k + 2), repeat=B):
            n = np.array(n, np.int32)
            kv = kv0.copy()
            st, len_new, pad_new, W_new = oracle.realign_kv(kv, ln, pad, n)
            assert st == 0
            check_invariants(kv0, kv, ln, pad, n, len_new, pad_new, W_new, expected_tokens(toks, props, n))


def test_planted_mistakes_break_the_invariants():
    kv0, ln, pad, toks, props = make_state([2, 6, 4], 3, 24, seed=4)
    n = np.array([4, 1, 2], np.int32)
    for name in ("skip_kv_shift", "shift_one_short"):
        kv = kv0.copy()
        with oracle.mutant(name):
            st, len_new, pad_new, W_new = oracle.realign_kv(kv, ln, pad, n)
        with pytest.raises(AssertionError):
            check_invariants(kv0, kv, ln, pad, n, len_new, pad_new, W_new, expected_tokens(toks, props, n))


def test_no_change_for_batch_of_one_and_uniform_acceptance():
    """"No padding adjustment is needed for batch size 1 or when every sequence
    accepts the same number of tokens" (App. B): zero bytes change."""
    kv0, ln, pad, _, _ = make_state([7], 4, 32, seed=1)
    for n in range(6):
        kv = kv0.copy()
        st, len_new, pad_new, W_new = oracle.realign_kv(kv, ln, pad, np.array([n], np.int32))
        assert st == 0 and pad_new[0] == 0 and np.array_equal(kv, kv0)
    kv0, ln, pad, _, _ = make_state([3, 9, 5, 1], 4, 32, seed=2)
    for n in range(6):
        kv = kv0.copy()
        st, len_new, pad_new, W_new = oracle.realign_kv(kv, ln, pad, np.full(4, n, np.int32))
        assert st == 0 and (pad_new == pad).all() and np.array_equal(kv, kv0)


def test_plan_errors_leave_everything_untouched():
    kv0, ln, pad, _, _ = make_state([3, 5], 2, 8, seed=3)
    W = 5
    # capacity: len' = [4, 9], W' = 9 > S = 8
    kv = kv0.copy()
    st, _, _, _ = oracle.realign_kv(kv, ln, pad, np.array([1, 4], np.int32))
    assert st == 1 and np.array_equal(kv, kv0)
    # a run that would start past the buffer: W + 5 - 1 = 9 > S
    st, _, _, _ = oracle.realign_kv(kv, ln, pad, np.array([1, 5], np.int32))
    assert st == 3 and np.array_equal(kv, kv0)
    st, _, _, _ = oracle.realign_plan(8, ln, pad, np.array([3, 3], np.int32))
    assert st == 0
    st, _, _, _ = oracle.realign_plan(7, ln, pad, np.array([3, 3], np.int32))
    assert st == 1  # W' = 8 > 7
    # I1 violated on input
    st, _, _, _ = oracle.realign_plan(8, ln, np.array([2, 1], np.int32), np.array([1, 1], np.int32))
    assert st == 2
    st, _, _, _ = oracle.realign_plan(8, np.array([3, 4]), np.array([0, 0]), np.array([1, 1]))
    assert st == 2  # pad + len not constant
    st, _, _, _ = oracle.realign_plan(8, np.array([4, 4]), np.array([1, 1]), np.array([1, 1]))
    assert st == 2  # no sequence without padding
    st, _, _, _ = oracle.realign_plan(8, ln, pad, np.array([-1, 1], np.int32))
    assert st == 3
    assert W == int((ln + pad)[0])


def test_shift_directions_and_width():
    """Repad to the new maximum length: a sequence that commits more than the
    others moves left into its padding, the others move right."""
    ln = np.array([5, 3, 4], np.int32)
    pad = np.array([0, 2, 1], np.int32)
    n = np.array([1, 4, 2], np.int32)
    st, len_new, pad_new, W_new = oracle.realign_plan(64, ln, pad, n)
    assert st == 0 and W_new == 7
    assert list(len_new) == [6, 7, 6] and list(pad_new) == [1, 0, 1]
    assert list(pad_new - pad) == [1, -2, 0]


def test_positions_and_mask():
    """Positions recomputed from the mask: non-pad slots of row b carry
    0, 1, 2, ... from slot pad'_b on (continuing past the width); pad slots are
    masked out and carry 0."""
    rng = np.random.default_rng(0)
    S = 40
    pad_new = rng.integers(0, 12, size=9).astype(np.int32)
    pos, mask = oracle.rebuild_pos_mask(S, pad_new)
    for b, pd in enumerate(pad_new):
        assert (mask[b, :pd] == 0).all() and (mask[b, pd:] == 1).all()
        assert list(pos[b, pd:]) == list(range(S - pd))
        assert (pos[b, :pd] == 0).all()
    pos0 = np.full((9, S), 77, np.int32)
    mask0 = np.full((9, S), 7, np.uint8)
    with oracle.mutant("stale_positions"):
        pos1, mask1 = oracle.rebuild_pos_mask(S, pad_new, pos0.copy(), mask0.copy())
    assert not np.array_equal(pos1, pos)


def test_realign_on_bf16_and_fp16_buffers():
    """The shift moves bytes: a 2-byte cache behaves like a 4-byte one."""
    kv32, ln, pad, toks, props = make_state([2, 7, 4], 2, 20, D=4, seed=6)
    n = np.array([3, 0, 1], np.int32)
    for dt in (np.float16, np.uint16):
        kv = kv32.astype(np.float16).view(dt).copy()
        ref = kv32.copy()
        st, ln2, pd2, w2 = oracle.realign_kv(kv, ln, pad, n)
        st2, _, _, _ = oracle.realign_kv(ref, ln, pad, n)
        assert st == st2 == 0
        assert np.array_equal(kv.view(np.float16).astype(np.float32), ref)
