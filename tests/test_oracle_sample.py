"""Pins of the oracle's stochastic verification (CPU only).

The pages fix: the acceptance rule min(1, p/q), the normalised positive
residual, the bonus from the target, the two worked toys (two and three
symbols), "p = q never rejects", and acceptance mass alpha = sum min(p, q).
Exact output distributions are obtained by sweeping the uniforms over a
midpoint grid (each cell of [0,1) is hit once), and chi-square tests on 10^6
random draws check that the target distribution is preserved.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle
from conftest import golden
from oracle import DT_F32


def _grid(n):
    return ((np.arange(n) + 0.5) / n).astype(np.float32)


def exact_first_token_distribution(p, q, n=1000):
    """Distribution of the first committed token for k = 1, proposal y ~ q:
    sum over y of q(y) times the grid frequency of each committed token.
    Returns (dist, acceptance probability per y, residual used on rejection)."""
    V = len(p)
    logit = np.log(np.asarray(p, np.float64)).astype(np.float32)
    ug = _grid(n)
    u0, u1 = np.meshgrid(ug, ug, indexing="ij")
    Bn = n * n
    x = np.broadcast_to(np.stack([logit, logit]), (Bn, 2, V)).copy()
    qq = np.broadcast_to(np.asarray(q, np.float32), (Bn, 1, V)).copy()
    u = np.stack([u0.ravel(), u1.ravel()], axis=1)
    dist = np.zeros(V)
    acc = np.zeros(V)
    residual = None
    for y in range(V):
        if q[y] == 0:
            continue
        d = np.full((Bn, 1), y, np.int32)
        out, na, ne, fl, res = oracle.verify_sample(x, DT_F32, qq, d, u, want_residual=True)
        first = out[:, 0]
        dist += q[y] * np.bincount(first, minlength=V) / Bn
        acc[y] = na.mean()
        rej = np.nonzero(na == 0)[0]
        if len(rej):
            residual = res[rej[0]]
    return dist, acc, residual


def test_two_symbol_toy():
    g = golden("sample_toy_two_symbol.txt")
    dist, acc, res = exact_first_token_distribution(g["p"], g["q"])
    assert np.allclose(acc, g["accept_prob"], atol=2e-3)
    assert np.argmax(res) == g["correction"][0] and res[1 - g["correction"][0]] == 0
    assert np.allclose(dist, g["final"], atol=2e-3)
    # Exercise 3: resampling from p after rejection changes the result to
    # P(0) = 0.8*0.5 + (0.8*0.5)*0.4 = 0.56.
    with oracle.mutant("resample_from_p"):
        bad, _, _ = exact_first_token_distribution(g["p"], g["q"])
    assert bad[0] == pytest.approx(0.8 * 0.5 + 0.8 * 0.5 * 0.4, abs=2e-3)


def test_three_symbol_toy():
    g = golden("sample_toy_three_symbol.txt")
    p, q = np.array(g["p"]), np.array(g["q"])
    dist, acc, res = exact_first_token_distribution(p, q)
    assert np.allclose(acc, g["accept_prob"], atol=2e-3)
    assert np.allclose(acc * q, g["accepted_mass"], atol=2e-3)
    assert (acc * q).sum() == pytest.approx(g["alpha"][0], abs=2e-3)
    assert 1 - (acc * q).sum() == pytest.approx(g["rejected_mass"][0], abs=2e-3)
    assert np.allclose(res, g["residual"], atol=1e-6)
    assert np.allclose(dist, g["final"], atol=2e-3)
    with oracle.mutant("no_clamp"):
        _, _, bad_res = exact_first_token_distribution(p, q)
    assert not np.allclose(bad_res, g["residual"], atol=1e-3)


def _random_case(V, rng, B, k):
    """Target rows with random logits; draft distributions = softmax of
    perturbed logits; proposals drawn from q; uniforms."""
    x = rng.standard_normal((1, k + 1, V)).astype(np.float32)
    x = np.broadcast_to(x, (B, k + 1, V)).copy()
    q = special.softmax(x[:, :k].astype(np.float64) + rng.standard_normal((1, k, V)) * 0.8, axis=-1)
    q = np.broadcast_to(q.astype(np.float32), (B, k, V)).copy()
    c = np.cumsum(q[0].astype(np.float64), axis=-1)
    d = np.stack([np.minimum(np.searchsorted(c[j], rng.random(B) * c[j, -1], side="right"), V - 1)
                  for j in range(k)], axis=1).astype(np.int32)
    u = rng.random((B, k + 1), dtype=np.float32)
    return x, q, d, u


@pytest.mark.parametrize("V", [2, 3, 8])
def test_chi_square_target_preserved(V):
    """10^6 draws: the first committed token follows p_0, and the bonus after
    full acceptance follows p_1 -- chi-square at the 1e-3 level."""
    rng = np.random.default_rng(1000 + V)
    B = 1_000_000
    x, q, d, u = _random_case(V, rng, B, 1)
    p0, _ = oracle.softmax_row(x[0], DT_F32, 0)
    p1, _ = oracle.softmax_row(x[0], DT_F32, 1)

    def pvals():
        out, na, ne, fl, _ = oracle.verify_sample(x, DT_F32, q, d, u)
        first = np.bincount(out[:, 0], minlength=V)
        bonus = np.bincount(out[na == 1, 1], minlength=V)
        return (stats.chisquare(first, first.sum() * p0).pvalue,
                stats.chisquare(bonus, bonus.sum() * p1).pvalue)

    a, b = pvals()
    assert a > 1e-3 and b > 1e-3
    with oracle.mutant("resample_from_p"):
        a, _ = pvals()
    assert a < 1e-3
    with oracle.mutant("bonus_from_draft"):
        _, b = pvals()
    assert b < 1e-3


def test_acceptance_rate_is_alpha():
    """Acceptance mass alpha = sum_x min(p(x), q(x)) ("Acceptance and rejection
    correction" of the Atlas lesson)."""
    rng = np.random.default_rng(5)
    B, V = 200_000, 8
    x, q, d, u = _random_case(V, rng, B, 1)
    p0, _ = oracle.softmax_row(x[0], DT_F32, 0)
    alpha = np.minimum(p0, q[0, 0].astype(np.float64)).sum()
    _, na, _, _, _ = oracle.verify_sample(x, DT_F32, q, d, u)
    rate = na.mean()
    assert abs(rate - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / B)


def test_p_equal_q_never_rejects():
    """"If p = q no rejection occurs" (Atlas lesson, "Assumptions"): with q the
    fp32 rounding of p, p/q is 1 to within 1e-7, so uniforms below 1 - 1e-6
    are always accepted, at every position of a k = 4 round."""
    rng = np.random.default_rng(9)
    B, V, k = 20_000, 50, 4
    x = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    q = np.empty((B, k, V), np.float32)
    for j in range(k):
        q[:, j] = special.softmax(x[:, j].astype(np.float64), axis=-1).astype(np.float32)
    c = np.cumsum(q.astype(np.float64), axis=-1)
    d = np.minimum((c < rng.random((B, k, 1)) * c[..., -1:]).sum(-1), V - 1).astype(np.int32)
    u = np.minimum(rng.random((B, k + 1), dtype=np.float32), np.float32(1 - 1e-6))
    _, na, ne, _, _ = oracle.verify_sample(x, DT_F32, q, d, u)
    assert (na == k).all() and (ne == k + 1).all()


def test_zero_weight_never_chosen():
    """The inverse CDF takes the first index whose prefix sum EXCEEDS u*sum, so
    u = 0 cannot select a leading zero-weight token."""
    p = np.array([0.2, 0.8])
    q = np.array([0.5, 0.5], np.float32)
    x = np.log(p).astype(np.float32)[None, None].repeat(2, axis=1)
    d = np.array([[0]], np.int32)
    u = np.array([[0.99, 0.0]], np.float32)  # reject proposal 0, draw at u = 0
    out, na, ne, fl, res = oracle.verify_sample(x, DT_F32, q[None, None], d, u, want_residual=True)
    assert na[0] == 0 and out[0, 0] == 1 and res[0, 0] == 0.0
    with oracle.mutant("cdf_ge"):
        out, _, _, _, _ = oracle.verify_sample(x, DT_F32, q[None, None], d, u)
    assert out[0, 0] == 0


def test_flags_and_degenerate_rows():
    V = 4
    p = np.array([0.1, 0.2, 0.3, 0.4])
    x = np.log(p).astype(np.float32)[None, None].repeat(2, axis=1)
    # q(y) = 0 for the proposal: flag 1, ratio +inf -> accepted
    q = np.array([0.0, 0.5, 0.25, 0.25], np.float32)[None, None]
    out, na, ne, fl, _ = oracle.verify_sample(x, DT_F32, q, np.array([[0]], np.int32),
                                              np.array([[0.5, 0.5]], np.float32))
    assert fl[0] & 1 and na[0] == 1
    # q > p everywhere (q not normalised): rejection leaves no positive residual;
    # flag 2 and the draw comes from p
    q = (p * 1.5).astype(np.float32)[None, None]
    out, na, ne, fl, res = oracle.verify_sample(x, DT_F32, q, np.array([[3]], np.int32),
                                                np.array([[0.9, 0.5]], np.float32), want_residual=True)
    assert na[0] == 0 and fl[0] & 2
    assert np.allclose(res[0], p, atol=1e-7) and out[0, 0] == 2  # cdf 0.1,0.3,0.6 > 0.5 at 2
    # a non-finite logit in a used row: flag 4
    xb = x.copy()
    xb[0, 0, 1] = np.inf
    _, _, _, fl, _ = oracle.verify_sample(xb, DT_F32, q, np.array([[3]], np.int32),
                                          np.array([[0.9, 0.5]], np.float32))
    assert fl[0] & 4


def test_temperature_is_softmax_of_scaled_logits():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((3, 1000)) * 4).astype(np.float32)
    for T in (0.5, 1.0, 2.0, 7.0):
        for r in range(3):
            p, bad = oracle.softmax_row(x, DT_F32, r, T)
            assert not bad
            assert np.allclose(p, special.softmax(x[r].astype(np.float64) / T), rtol=1e-12, atol=1e-300)


def test_stop_rules_match_greedy_commitment():
    """EOS and the output budget stop a stochastic round exactly as they stop
    greedy commitment; remaining = 0 commits nothing."""
    V, k = 6, 3
    p = np.full(V, 1.0 / V)
    x = np.log(p).astype(np.float32)[None, None].repeat(k + 1, axis=1)
    q = np.broadcast_to(p.astype(np.float32), (1, k, V)).copy()
    d = np.array([[1, 2, 3]], np.int32)
    u = np.array([[0.1, 0.1, 0.1, 0.55]], np.float32)  # p = q: all accepted
    out, na, ne, _, _ = oracle.verify_sample(x, DT_F32, q, d, u)
    assert list(out[0, :ne[0]]) == [1, 2, 3, 3] and na[0] == 3  # bonus: cdf 3/6 <= 0.55 < 4/6
    out, na, ne, _, _ = oracle.verify_sample(x, DT_F32, q, d, u, eos_id=2)
    assert list(out[0, :ne[0]]) == [1, 2] and na[0] == 2
    out, na, ne, _, _ = oracle.verify_sample(x, DT_F32, q, d, u, remaining=np.array([1], np.int32))
    assert list(out[0, :ne[0]]) == [1]
    out, na, ne, _, _ = oracle.verify_sample(x, DT_F32, q, d, u, remaining=np.array([0], np.int32))
    assert ne[0] == 0 and (out[0] == -1).all()
    out, na, ne, _, _ = oracle.verify_sample(x, DT_F32, q, d, u, draft_len=np.array([1], np.int32))
    assert list(out[0, :ne[0]]) == [1, 3] and na[0] == 1


def test_out_of_vocabulary_proposal_is_rejected_and_flagged():
    V = 4
    p = np.array([0.1, 0.2, 0.3, 0.4])
    x = np.log(p).astype(np.float32)[None, None].repeat(2, axis=1)
    q = np.full((1, 1, V), 0.25, np.float32)
    for y in (-1, V, 10**6):
        out, na, ne, fl, res = oracle.verify_sample(x, DT_F32, q, np.array([[y]], np.int32),
                                                    np.array([[0.0, 0.5]], np.float32), want_residual=True)
        assert fl[0] & 8 and na[0] == 0 and ne[0] == 1
        # drawn from the residual max(0, p - q) = [0, 0, 0.05, 0.15]
        assert np.allclose(res[0], [0, 0, 0.25, 0.75], atol=1e-6)


def test_negative_infinity_is_a_masked_token():
    """-inf logits (masked tokens, e.g. after top-k filtering) get probability
    0 and do not make the distribution undefined; NaN, +inf or an all -inf
    row do (flag 4)."""
    V = 5
    x = np.zeros((1, 2, V), np.float32)
    x[0, :, 1] = -np.inf
    x[0, :, 3] = -np.inf
    q = np.full((1, 1, V), 0.2, np.float32)
    out, na, ne, fl, res = oracle.verify_sample(x, DT_F32, q, np.array([[1]], np.int32),
                                                np.array([[0.0, 0.5]], np.float32), want_residual=True)
    assert fl[0] == 0 and na[0] == 0  # p(1) = 0: the masked proposal is rejected
    assert res[0, 1] == 0 and res[0, 3] == 0 and out[0, 0] in (0, 2, 4)
    p, bad = oracle.softmax_row(x[0], DT_F32, 0)
    assert not bad and p[1] == 0 and np.isclose(p.sum(), 1.0)
    x[0, 0, :] = -np.inf
    _, bad = oracle.softmax_row(x[0], DT_F32, 0)
    assert bad


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_sixteen_bit_nan_of_either_sign_is_undefined(dt):
    """In 16-bit storage a NaN of either sign, or +inf, makes the row's
    distribution undefined, filtered or not; -inf alone does not."""
    code = {"bf16": oracle.DT_BF16, "f16": oracle.DT_F16}[dt]
    pats = {"bf16": dict(pnan=0x7FC1, nnan=0xFFC1, pinf=0x7F80, ninf=0xFF80, one=0x3F80),
            "f16": dict(pnan=0x7E01, nnan=0xFE01, pinf=0x7C00, ninf=0xFC00, one=0x3C00)}[dt]
    for kind, expect_bad in (("pnan", True), ("nnan", True), ("pinf", True), ("ninf", False)):
        row = np.full((1, 8), pats["one"], np.uint16)
        row[0, 3] = 0  # a smaller logit, so filters have something to cut
        row[0, 5] = pats[kind]
        xs = row if dt == "bf16" else row.view(np.float16)
        for top_k, top_p in ((0, 1.0), (2, 1.0), (0, 0.5), (3, 0.9)):
            _, bad = oracle.softmax_row(xs, code, 0, 1.0, top_k, top_p)
            assert bad == expect_bad, (kind, top_k, top_p)
