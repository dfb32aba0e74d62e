"""Pins of the oracle's greedy verification (CPU only).

Each test checks the oracle against something other than itself: values the
pages print, the closed form of the iid output count, exact enumeration, the
numpy/scipy definitions of the storage types, and planted mistakes that must
be caught.
"""
import itertools

import numpy as np
import pytest

import oracle
from conftest import golden
from oracle import DT_BF16, DT_F16, DT_F32
from specgen import f32_to_bf16_bits, greedy_round_inputs


def rows_with_choice(choices, V):
    """Logit rows whose unique argmax is choices[j]."""
    x = np.zeros((len(choices), V), np.float32)
    for j, c in enumerate(choices):
        x[j, c] = 1.0
    return x


def run(choices, proposals, V=10, **kw):
    x = rows_with_choice(choices, V)[None]
    d = np.array(proposals, np.int32)[None]
    out, na, ne = oracle.verify_greedy(x, DT_F32, d, **{
        key: (np.array([v], np.int32) if key in ("remaining", "draft_len") and v is not None else v)
        for key, v in kw.items()})
    return [int(t) for t in out[0, : ne[0]]], int(na[0]), int(ne[0]), out[0]


def test_worked_rejection():
    g = golden("greedy_worked_example.txt")
    choices = g["target_row_choices"] + [0, 0]  # later rows are never looked at
    got, na, ne, out = run(choices, g["proposals"], V=3)
    assert got == g["committed"]
    assert na == 1 and ne == 2
    assert list(out[ne:]) == [-1] * (4 - ne)


def test_row_alignment_exercise():
    """A full-prefix target computes one row per input position (row i predicts
    token i+1); the slice starting at row L-1 is what verification consumes.
    Proposals equal to the target's own next-token choices must all be accepted
    and the bonus must be the choice of row L+k-1."""
    g = golden("row_alignment.txt")
    L, k = g["L"][0], g["k"][0]
    V = 17
    rng = np.random.default_rng(3)
    prefix_choice = rng.integers(0, V, size=L + k)  # target's choice at each row
    full = rows_with_choice(prefix_choice, V)  # [L+k, V], row i predicts token i+1
    verification = full[L - 1:]
    assert verification.shape[0] == k + 1
    assert [L - 1 + j for j in range(k)] == g["verify_rows"]
    assert L + k - 1 == g["bonus_row"][0]
    proposals = [int(prefix_choice[r]) for r in g["verify_rows"]]
    out, na, ne = oracle.verify_greedy(verification[None], DT_F32, np.array([proposals], np.int32))
    assert na[0] == k and ne[0] == k + 1
    assert out[0, k] == prefix_choice[g["bonus_row"][0]]
    with oracle.mutant("row_shift"):
        out2, na2, _ = oracle.verify_greedy(verification[None], DT_F32, np.array([proposals], np.int32))
    assert (na2[0], out2[0, -1]) != (k, prefix_choice[g["bonus_row"][0]])


# Stopping rules of greedy_commit ("Chapter 10 Speculative Decoding (Code
# Walkthrough)", §4.1): commit the row's choice; stop after EOS, after the
# budget is reached, or after a mismatch; bonus after full acceptance if the
# budget allows.  Exercise 4 of §6.2: a rejected proposed EOS commits the
# correction and generation goes on.
EOS = 9


@pytest.mark.parametrize(
    "choices, proposals, kw, committed, n_accept",
    [
        ([5, 6, 7, 8], [5, 6, 7], {}, [5, 6, 7, 8], 3),  # full acceptance + bonus
        ([5, 6, 7, 8], [1, 6, 7], {}, [5], 0),  # first proposal rejected
        ([5, 6, 7, 8], [5, 6, 7], dict(remaining=0), [], 0),  # no budget
        ([5, EOS, 7, 8], [5, EOS, 7], dict(eos_id=EOS), [5, EOS], 2),  # accepted EOS ends it
        ([5, EOS, 7, 8], [5, 6, 7], dict(eos_id=EOS), [5, EOS], 1),  # EOS as the correction
        ([3, 6, 7, 8], [EOS, 6, 7], dict(eos_id=EOS), [3], 0),  # rejected proposed EOS
        ([5, 6, 7, 8], [5, 6, 7], dict(remaining=2), [5, 6], 2),  # budget inside the prefix
        ([5, 6, 7, 8], [5, 6, 7], dict(remaining=3), [5, 6, 7], 3),  # budget eats the bonus
        ([5, 6, 7, 8], [5, 6, 7], dict(remaining=4), [5, 6, 7, 8], 3),
        ([5, 9, 7, 8], [5, 6, 7], dict(draft_len=1), [5, 9], 1),  # bonus from row k_b
        ([4, 9, 7, 8], [5, 6, 7], dict(draft_len=0), [4], 0),  # no proposals: row 0
        ([5, 6, 7, 8], [5, 6, 7], dict(eos_id=-1), [5, 6, 7, 8], 3),  # -1: no EOS
    ],
)
def test_stopping_rules(choices, proposals, kw, committed, n_accept):
    got, na, ne, out = run(choices, proposals, **kw)
    assert got == committed
    assert na == n_accept and ne == len(committed)
    assert all(t == -1 for t in out[ne:])


def test_ties_take_lowest_index():
    V = 8
    x = np.zeros((1, 2, V), np.float32)
    x[0, 0, [2, 5]] = 3.0  # tie between 2 and 5
    x[0, 1, :] = -1.0
    x[0, 1, [1, 6]] = 0.0  # tie between 1 and 6
    out, na, ne = oracle.verify_greedy(x, DT_F32, np.array([[2]], np.int32))
    assert (na[0], ne[0], out[0, 1]) == (1, 2, 1)
    # -0.0 and +0.0 are equal: the lower index wins
    x[0, 1, 1] = -0.0
    out, _, _ = oracle.verify_greedy(x, DT_F32, np.array([[2]], np.int32))
    assert out[0, 1] == 1
    with oracle.mutant("tie_highest"):
        out, na, _ = oracle.verify_greedy(x, DT_F32, np.array([[2]], np.int32))
    assert na[0] == 0 and out[0, 0] == 5


def test_nan_counts_as_largest():
    x = np.zeros((1, 1, 6), np.float32)
    x[0, 0, 1] = np.inf
    x[0, 0, 3] = np.nan
    x[0, 0, 4] = np.nan
    out, _, _ = oracle.verify_greedy(x, DT_F32, np.zeros((1, 0), np.int32))
    assert out[0, 0] == 3


def test_storage_types_decode_like_numpy():
    """bf16 is the upper half of an fp32 bit pattern and fp16 is IEEE binary16:
    the oracle's decoders must agree with numpy's on every pattern class
    (normals, subnormals, zeros, infinities)."""
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(500).astype(np.float32) * 30,
                           np.array([0.0, -0.0, 1e-7, -3e-6, 6e-8, 65504.0, -65504.0], np.float32)])
    h = vals.astype(np.float16)
    for i in range(len(h)):
        row = np.zeros((1, 2), np.float16)
        row[0, 0] = h[i]
        p, _ = oracle.softmax_row(row, DT_F16, 0)
        z = np.array([float(h[i]), 0.0])
        e = np.exp(z - z.max())
        assert np.allclose(p, e / e.sum(), rtol=1e-14, atol=0), (i, h[i])
    bits = f32_to_bf16_bits(vals)
    as_f32 = (bits.astype(np.uint32) << 16).view(np.float32)
    for i in range(0, len(bits), 7):
        row = np.zeros((1, 2), np.uint16)  # bf16 bits of 0.0 in column 1
        row[0, 0] = bits[i]
        p, _ = oracle.softmax_row(row, DT_BF16, 0)
        z = np.array([float(as_f32[i]), 0.0])
        e = np.exp(z - z.max())
        assert np.allclose(p, e / e.sum(), rtol=1e-14, atol=0)
    # argmax on the storage types picks what numpy's argmax picks on the decoded values
    x, d = greedy_round_inputs(16, 3, 257, 0.5, 2.0, seed=11, dtype="bf16")
    out, na, ne = oracle.verify_greedy(x, DT_BF16, d)
    dec = (x.astype(np.uint32) << 16).view(np.float32)
    am = dec.argmax(-1)  # numpy: first occurrence of the maximum
    for b in range(16):
        n = int(ne[b])
        assert list(out[b, :n]) == [int(am[b, j]) for j in range(n)]
    xh, d = greedy_round_inputs(16, 3, 257, 0.5, 1.0, seed=12, dtype="f16")
    out, na, ne = oracle.verify_greedy(xh, DT_F16, d)
    am = xh.astype(np.float32).argmax(-1)
    for b in range(16):
        assert list(out[b, : ne[b]]) == [int(am[b, j]) for j in range(int(ne[b]))]


def _emission_distribution(alpha, gamma, V=5):
    """Exact distribution of the committed count under iid acceptance, by
    enumerating every acceptance pattern through the oracle."""
    dist = {}
    for pattern in itertools.product([0, 1], repeat=gamma):
        prob = 1.0
        choices, props = [], []
        for j, a in enumerate(pattern):
            prob *= alpha if a else (1.0 - alpha)
            choices.append(j % V)
            props.append(j % V if a else (j + 1) % V)
        choices.append(V - 1)
        _, _, ne, _ = run(choices, props, V=V)
        dist[ne] = dist.get(ne, 0.0) + prob
    return dist


def test_expected_count_worked_example():
    g = golden("ek_worked_example.txt")
    dist = _emission_distribution(g["alpha"][0], g["gamma"][0])
    for c, p in zip(g["counts"], g["probs"]):
        assert dist[c] == pytest.approx(p, abs=1e-12)
    ek = sum(c * p for c, p in dist.items())
    assert ek == pytest.approx(g["expected_count"][0], abs=1e-12)
    with oracle.mutant("bonus_always"):
        bad = _emission_distribution(g["alpha"][0], g["gamma"][0])
    assert sum(c * p for c, p in bad.items()) != pytest.approx(g["expected_count"][0], abs=1e-3)


@pytest.mark.parametrize("alpha,gamma", [(0.3, 8), (0.5, 5), (0.7, 4), (0.8, 5), (0.9, 8), (0.6, 3)])
def test_expected_count_closed_form(alpha, gamma):
    dist = _emission_distribution(alpha, gamma)
    ek = sum(c * p for c, p in dist.items())
    assert ek == pytest.approx((1 - alpha ** (gamma + 1)) / (1 - alpha), rel=1e-12)


@pytest.mark.parametrize("alpha,k", [(0.7, 4), (0.5, 5), (0.3, 8)])
def test_mean_emission_on_generated_rounds(alpha, k):
    """The generator's iid acceptance structure gives E[K] on average."""
    B = 3000
    x, d = greedy_round_inputs(B, k, 64, alpha, 1.0, seed=100 + k, dtype="f32")
    _, na, ne = oracle.verify_greedy(x, DT_F32, d)
    ek = (1 - alpha ** (k + 1)) / (1 - alpha)
    sd = ne.std()
    assert abs(ne.mean() - ek) < 5 * sd / np.sqrt(B)
    assert (ne == na + 1).all()
