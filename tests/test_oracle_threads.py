"""The oracle's loops over sequences and cache slabs may run on several
threads (OpenMP): every sequence and slab is computed exactly as on one
thread, so the results must be identical for any thread count."""
import numpy as np
import pytest

import oracle
from specgen import greedy_round_inputs, sample_round_inputs


def _both(fn):
    with oracle.threads(1):
        one = fn()
    with oracle.threads(4):
        four = fn()
    return one, four


def test_greedy_independent_of_threads():
    x, d = greedy_round_inputs(16, 5, 3000, 0.6, 1.0, seed=71, dtype="bf16")
    one, four = _both(lambda: oracle.verify_greedy(x, oracle.DT_BF16, d))
    for a, b in zip(one, four):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("filt", [{}, {"top_k": 20, "top_p": 0.9}])
def test_sample_independent_of_threads(filt):
    x, q, d, u = sample_round_inputs(12, 4, 2000, 0.5, seed=72)
    one, four = _both(lambda: oracle.verify_sample(x, oracle.DT_F32, q, d, u, want_residual=True, **filt))
    for a, b in zip(one, four):
        if a is None:
            assert b is None
        else:
            assert np.array_equal(a, b)


def test_realign_independent_of_threads():
    rng = np.random.default_rng(73)
    L, B, H, S, D = 2, 6, 3, 96, 8
    kv = rng.standard_normal((L, 2, B, H, S, D)).astype(np.float32)
    ln = rng.integers(5, 60, B).astype(np.int32)
    pad = (ln.max() - ln).astype(np.int32)
    ne = rng.integers(0, 6, B).astype(np.int32)
    outs = []
    for n in (1, 4):
        kv2 = kv.copy()
        with oracle.threads(n):
            outs.append((oracle.realign_kv(kv2, ln, pad, ne), kv2))
    (r1, k1), (r4, k4) = outs
    assert r1[0] == r4[0] == 0
    for a, b in zip(r1[1:], r4[1:]):
        assert np.array_equal(a, b)
    assert np.array_equal(k1, k4)
