"""Pins of the oracle's sampling transforms (top-k, top-p, temperature) on
the target distribution of stochastic verification (CPU only).

The pages require the ratio test, the residual and the bonus to use the
processed distribution ("Chapter 10 Speculative Decoding (Code Walkthrough)",
§5.1; "Speculative decoding: proposals and verified output", "The mechanism"
step 1) without defining the transforms.  The oracle takes the plain
definitions and decides the top-p boundary on the masses e^((x - x_max)/T)
in fp64 with a stated error band.  Pinned here:
  - a hand-worked example with power-of-two weights (tests/golden);
  - brute force on tiny inputs, from the definitions restated independently
    (top-k: fewer than k tokens strictly larger; top-p: the smallest upper
    set of mass >= top_p): exact rationals on integer logits, and
    50-digit arithmetic on real-valued logits at several temperatures;
  - on rows of 128256 N(0,1) logits (fp32 and bf16), the kept set is the
    smallest top set reaching top_p, checked with correctly rounded sums;
  - top_k = 1 (and top_p -> 0) turns stochastic verification into greedy
    verification, checked against the greedy oracle;
  - top_k >= V, top_p = 1 leave every output unchanged;
  - the committed token's distribution equals the processed distribution
    (midpoint grid over the uniforms), and acceptance = sum min(p', q);
  - -0 and +0 are one value at the cut, in every storage type;
  - six planted mistakes each fail at least one of these.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import golden
from oracle import DT_F32

# fp32(log2 e) as the temperature: masses e^(x/T) = 2^(x (1 + d)) with
# d = 1.3e-8, so integer logits give (almost exactly) powers of two; where an
# upper set's mass equals top_p times the total exactly in powers of two,
# d > 0 moves it above that bound, as the strict test of the definition does
# at an exact tie (the set's mean logit exceeds the row's)
T_UNIT = float(np.float32(np.log2(np.e)))


def _case_table():
    g = golden("filter_worked_example.txt")
    cases = {"none": (0, 1.0), "k1": (1, 1.0), "k2": (2, 1.0), "k3": (3, 1.0), "k4": (4, 1.0),
             "p0500": (0, 0.5), "p0625": (0, 0.625), "p0875": (0, 0.875), "p09375": (0, 0.9375),
             "k3p05625": (3, 0.5625)}
    return g, cases


def test_worked_example():
    g, cases = _case_table()
    x = np.array(g["x"], np.float32)[None]
    for name, (tk, tp) in cases.items():
        p, bad = oracle.softmax_row(x, DT_F32, 0, T_UNIT, tk, tp)
        assert not bad
        assert np.allclose(p, g[name], atol=1e-7), (name, p)
        cut = oracle.filter_cut(x, DT_F32, 0, T_UNIT, tk, tp)
        want = x[0][np.array(g[name]) > 0].min()
        assert cut == (-np.inf if name == "none" else want) or (cut == want), (name, cut)


def test_temperature_enters_the_nucleus():
    """Doubling the logits and the temperature leaves the processed
    distribution unchanged; doubling the logits alone sharpens it and top-p
    keeps fewer tokens."""
    g, _ = _case_table()
    x = np.array(g["x"], np.float32)[None]
    T2 = float(np.float32(2 * T_UNIT))
    p1, _ = oracle.softmax_row(x, DT_F32, 0, T_UNIT, 0, 0.875)
    p2, _ = oracle.softmax_row(2 * x, DT_F32, 0, T2, 0, 0.875)
    assert np.allclose(p1, p2, atol=1e-7)
    p3, _ = oracle.softmax_row(2 * x, DT_F32, 0, T_UNIT, 0, 0.875)
    assert np.count_nonzero(p3) == 2 and np.count_nonzero(p1) == 3


def _brute_kept(x, top_k, top_p):
    """Kept set from the definitions, exact rationals; weights 2^x (integer x,
    scale exactly 1)."""
    V = len(x)
    w = [Fraction(2) ** int(v) for v in x]
    keep = [True] * V
    if 0 < top_k < V:
        keep = [sum(1 for u in x if u > x[v]) < top_k for v in range(V)]
    if top_p < 1.0:
        tot = sum(w[v] for v in range(V) if keep[v])
        bound = Fraction(float(np.float32(top_p))) * tot
        for t in sorted({x[v] for v in range(V) if keep[v]}, reverse=True):
            upper = [v for v in range(V) if keep[v] and x[v] >= t]
            if sum(w[v] for v in upper) >= bound:
                keep = [v in upper for v in range(V)]
                break
    return keep


def test_brute_force_tiny_rows():
    rng = np.random.default_rng(7)
    for _ in range(3000):
        V = int(rng.integers(1, 8))
        x = rng.integers(-6, 1, size=V).astype(np.float32)
        top_k = int(rng.integers(0, V + 2))
        top_p = float(np.float32(rng.choice([rng.random(), 1.0, 0.0, rng.integers(1, 16) / 16])))
        p, bad = oracle.softmax_row(x[None], DT_F32, 0, T_UNIT, top_k, top_p)
        keep = _brute_kept(list(x), top_k, top_p)
        assert not bad
        assert list(p > 0) == keep, (x, top_k, top_p, p)
        w = np.where(keep, 2.0 ** x.astype(np.float64), 0.0)
        assert np.allclose(p, w / w.sum(), atol=1e-7)


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_signed_zeros_are_one_value(dt):
    """-0 and +0 are one logit value: neither is strictly larger than the
    other, so top-k and top-p keep both or neither (brute force on tiny rows
    drawn from {-2, -1, -0, +0, 1}, in each storage type)."""
    rng = np.random.default_rng(19)
    vals = np.array([-2.0, -1.0, -0.0, 0.0, 1.0], np.float32)
    code = {"f32": DT_F32, "bf16": oracle.DT_BF16, "f16": oracle.DT_F16}[dt]
    both = 0
    for _ in range(1500):
        V = int(rng.integers(2, 8))
        x = vals[rng.integers(0, 5, size=V)]
        top_k = int(rng.integers(0, V + 1))
        top_p = float(np.float32(rng.choice([1.0, 0.0, rng.integers(1, 16) / 16, rng.random()])))
        if dt == "bf16":
            xs = (x.view(np.uint32) >> 16).astype(np.uint16)
        elif dt == "f16":
            xs = x.astype(np.float16)
        else:
            xs = x
        p, bad = oracle.softmax_row(xs[None], code, 0, T_UNIT, top_k, top_p)
        keep = _brute_kept(list(x), top_k, top_p)
        assert not bad
        assert list(p > 0) == keep, (x, top_k, top_p, p)
        zs = np.flatnonzero(x == 0)
        if np.signbit(x[zs]).any() and not np.signbit(x[zs]).all():
            both += 1
            assert len(set((p[zs] > 0).tolist())) == 1
    assert both > 300  # rows holding both zeros were drawn


def _round_inputs(rng, B, k, V, sigma=2.0):
    x = (rng.standard_normal((B, k + 1, V)) * sigma).astype(np.float32)
    dl = x[:, :k] + rng.standard_normal((B, k, V)).astype(np.float32)
    q = np.exp(dl - dl.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    d = np.array([[rng.choice(V, p=q[b, j] / q[b, j].sum()) for j in range(k)] for b in range(B)], np.int32)
    u = rng.random((B, k + 1)).astype(np.float32)
    return x, q, d, u


def test_top_k_one_is_greedy():
    """With top_k = 1 (or top_p = 0) the processed p is one-hot at the argmax:
    a proposal is accepted iff it is the argmax and the correction or bonus is
    the argmax, so the round equals greedy verification."""
    rng = np.random.default_rng(11)
    x, q, d, u = _round_inputs(rng, 64, 4, 50)
    # make half of the proposals the argmax so that rounds run long
    am = x[:, :4].argmax(-1).astype(np.int32)
    d = np.where(rng.random(d.shape) < 0.7, am, d).astype(np.int32)
    g_out, g_na, g_ne = oracle.verify_greedy(x, DT_F32, d)
    for kw in (dict(top_k=1), dict(top_p=0.0), dict(top_k=1, top_p=0.3)):
        out, na, ne, fl, _ = oracle.verify_sample(x, DT_F32, q, d, u, **kw)
        assert np.array_equal(out, g_out) and np.array_equal(na, g_na) and np.array_equal(ne, g_ne), kw


def test_off_values_change_nothing():
    rng = np.random.default_rng(12)
    x, q, d, u = _round_inputs(rng, 32, 3, 40)
    ref = oracle.verify_sample(x, DT_F32, q, d, u, want_residual=True)
    for kw in (dict(top_k=0, top_p=1.0), dict(top_k=40, top_p=1.0), dict(top_k=1000), dict(top_p=np.nan),
               dict(top_k=-3, top_p=1.5)):
        got = oracle.verify_sample(x, DT_F32, q, d, u, want_residual=True, **kw)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b), kw


def exact_first_token_distribution(x, q, top_k, top_p, n=600):
    """Distribution of the first committed token for k = 1 and proposal y ~ q,
    the uniforms swept over an n x n midpoint grid (target rows 0 and 1 equal)."""
    V = len(x)
    ug = ((np.arange(n) + 0.5) / n).astype(np.float32)
    u0, u1 = np.meshgrid(ug, ug, indexing="ij")
    Bn = n * n
    xx = np.broadcast_to(np.stack([x, x]).astype(np.float32), (Bn, 2, V)).copy()
    qq = np.broadcast_to(np.asarray(q, np.float32), (Bn, 1, V)).copy()
    u = np.stack([u0.ravel(), u1.ravel()], axis=1)
    dist, acc = np.zeros(V), 0.0
    for y in range(V):
        if q[y] == 0:
            continue
        out, na, _, _, _ = oracle.verify_sample(xx, DT_F32, qq, np.full((Bn, 1), y, np.int32), u,
                                                temperature=T_UNIT, top_k=top_k, top_p=top_p)
        dist += q[y] * np.bincount(out[:, 0], minlength=V) / Bn
        acc += q[y] * na.mean()
    return dist, acc


@pytest.mark.parametrize("name", ["k2", "k3", "p0625", "p0875", "k3p05625"])
def test_output_distribution_is_the_processed_target(name):
    g, cases = _case_table()
    tk, tp = cases[name]
    x = np.array(g["x"], np.float32)
    q = np.array([0.3, 0.1, 0.25, 0.15, 0.2])
    dist, acc = exact_first_token_distribution(x, q, tk, tp)
    pp = np.array(g[name])
    assert np.allclose(dist, pp, atol=4e-3), (name, dist)
    assert abs(acc - np.minimum(pp, q).sum()) < 4e-3


def _exact_kept(x, T, top_k, top_p, dps=50):
    """Kept set from the definitions with 50-digit masses e^((x - x_max)/T)."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = dps
    V = len(x)
    keep = [True] * V
    if 0 < top_k < V:
        keep = [sum(1 for u in x if u > x[v]) < top_k for v in range(V)]
    margin = mp.inf
    if top_p < 1.0:
        xm = max(float(x[v]) for v in range(V) if keep[v])
        w = [mp.e ** ((mp.mpf(float(x[v])) - xm) / mp.mpf(T)) if keep[v] else mp.mpf(0) for v in range(V)]
        tot = sum(w)
        bound = mp.mpf(float(np.float32(top_p))) * tot
        vals = sorted({float(x[v]) for v in range(V) if keep[v]}, reverse=True)
        for i, t in enumerate(vals):
            above = sum(w[v] for v in range(V) if keep[v] and x[v] > t)
            if i > 0:
                margin = min(margin, abs(above - bound) / tot)
            if i > 0 and not above < bound:
                keep = [keep[v] and x[v] > t for v in range(V)]
                break
    return keep, margin


def test_exact_arithmetic_on_tiny_real_rows():
    """Real-valued logits at temperatures 0.37 .. 3: the kept set equals the
    one computed with 50-digit masses (no decision here lies within 1e-12 of
    its bound, far outside the oracle's fp64 band)."""
    rng = np.random.default_rng(23)
    n = 0
    for _ in range(1500):
        V = int(rng.integers(1, 9))
        x = (rng.standard_normal(V) * rng.choice([0.5, 1.0, 3.0])).astype(np.float32)
        if rng.random() < 0.3:  # some repeated values
            x[rng.integers(0, V, size=V // 2)] = x[0]
        T = float(np.float32(rng.choice([0.37, 1.0, 1.7, 3.0])))
        top_k = int(rng.integers(0, V + 2))
        top_p = float(np.float32(rng.choice([rng.random(), 0.0, 0.5, 0.9, 0.95, 1.0])))
        keep, margin = _exact_kept(list(x), T, top_k, top_p)
        if margin < 1e-12:
            continue
        p, bad = oracle.softmax_row(x[None], DT_F32, 0, T, top_k, top_p)
        assert not bad
        assert list(p > 0) == keep, (x, T, top_k, top_p, p)
        n += 1
    assert n > 1400


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("top_p", [0.5, 0.9, 0.95])
def test_nucleus_is_the_smallest_top_set_on_full_size_rows(dt, top_p):
    """Rows of V = 128256 N(0,1) logits (the vocabulary of the stochastic
    workloads): with masses e^(x - x_max) summed by math.fsum (correctly
    rounded), the mass strictly above the cut is below top_p times the total
    and the mass at or above it reaches it -- the kept set is the smallest
    top set reaching top_p.  The oracle's reported margin is the distance of
    those two sums to the bound, and no decision falls in its error band."""
    import math

    from specgen import bf16_bits_to_f32, f32_to_bf16_bits

    rng = np.random.default_rng(int(top_p * 100) + (dt == "bf16"))
    V = 128256
    tp = float(np.float32(top_p))
    for _ in range(6):
        x = rng.standard_normal(V).astype(np.float32)
        if dt == "bf16":
            xs = f32_to_bf16_bits(x)
            xv, code = bf16_bits_to_f32(xs).astype(np.float64), oracle.DT_BF16
        else:
            xs, xv, code = x, x.astype(np.float64), DT_F32
        cut, margin, total, undecided = oracle.filter_info(xs[None], code, 0, 1.0, 0, tp)
        assert not undecided
        w = np.exp(xv - xv.max())
        M = math.fsum(w)
        above = math.fsum(w[xv > cut])
        upto = math.fsum(w[xv >= cut])
        assert above < tp * M <= upto, (above / M, upto / M)
        assert abs(total - M) <= 1e-12 * M
        assert abs(min(tp * M - above, upto - tp * M) - margin) <= 1e-9 * M
        assert cut in xv


@pytest.mark.parametrize("mut", ["topk_strict", "topp_below", "ratio_unfiltered", "resid_unfiltered",
                                 "topp_first", "zero_sign_order"])
def test_planted_mistakes_fail_a_pin(mut):
    checks = [test_worked_example, test_top_k_one_is_greedy, test_brute_force_tiny_rows,
              test_exact_arithmetic_on_tiny_real_rows,
              lambda: test_signed_zeros_are_one_value("bf16"),
              lambda: [test_output_distribution_is_the_processed_target(n)
                       for n in ("k2", "k3", "p0625", "p0875", "k3p05625")]]
    failed = 0
    with oracle.mutant(mut):
        for c in checks:
            try:
                c()
            except AssertionError:
                failed += 1
    assert failed >= 1, mut
