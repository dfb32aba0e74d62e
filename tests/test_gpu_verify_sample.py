"""Stochastic verification: CUDA path (fp32 arithmetic) vs the CPU oracle
(fp64 probabilities).

Acceptance criteria: tokens, accepted and committed counts equal the oracle's
except where the oracle's own decision sits on a boundary --
  * a ratio test with |u - p/q| <= 1e-5 * p/q, or
  * a draw whose uniform lies within 1e-5 * u of every oracle CDF boundary
    C_i / sum(w) between the two chosen indices;
such cases are counted and their rate must stay below 1e-4 of all decisions.
Normalised residual / draw distributions must match within 1e-6 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import DT_OF, dev, logits_to_dev, storage_of, to_dev
from specgen import CONFIGS, sample_round_inputs
from specgen import torch_gen

pytestmark = pytest.mark.gpu

TOL = 1e-5
RES_TOL = 1e-6
STATS = {"decisions": 0, "boundary": 0, "residual_rows": 0, "widened_rows": 0}


def _per_seq(v, b):
    if v is None:
        return None
    a = np.asarray(v)
    return a.item() if a.ndim == 0 else a[b].item()


def residual_tolerance(x, dt, q, T, b, k, row, bonus, r_o, top_k=None, top_p=None):
    """Per-element tolerance of the normalised draw distribution.

    1e-6 absolute, widened only where fp32 arithmetic cannot reach it:
    r_v = w_v / W with w_v = max(0, p_v - q_v) inherits p_v's fp32 relative
    error (expf <= 2 ulp, the division and the row sum: ~5 * 2^-24 ~ 3e-7)
    amplified by p_v / W, and the error of W itself.  The bound used,
    1e-6 * (1 + (p_v + r_v * sum_{w>0} p) / W), is that estimate with a 3x
    margin; with large vocabularies (p_v << W) it is the plain 1e-6."""
    p, _ = oracle.softmax_row(x.reshape(-1, x.shape[-1]), dt, b * (k + 1) + row, T, *_filt(top_k, top_p, b))
    w = p if bonus else np.maximum(p - q[b, row].astype(np.float64), 0.0)
    if not bonus and not (w.sum() > 0):
        w = p
    W = w.sum()
    ppos = p[w > 0].sum()
    return RES_TOL * (1.0 + (p + r_o * ppos) / W)


def _filt(top_k, top_p, b):
    tk, tp = _per_seq(top_k, b), _per_seq(top_p, b)
    return (0 if tk is None else int(tk)), (1.0 if tp is None else float(tp))


def _boundary_explains(x, dt, q, d, u, T, b, o_out, o_na, o_ne, o_res, g_out, g_na, g_ne, kb, top_k=None,
                       top_p=None):
    """True when the first difference between the two results of sequence b
    is a decision on a boundary of the oracle's arithmetic."""
    k = d.shape[1]
    # first ratio test where the two sides decided differently
    j = 0
    while j < kb and j < min(o_na, g_na) + 1:
        if j >= o_ne or j >= g_ne:
            break
        if (j < o_na) != (j < g_na):
            p, _ = oracle.softmax_row(x.reshape(-1, x.shape[-1]), dt, b * (k + 1) + j, T, *_filt(top_k, top_p, b))
            y = int(d[b, j])
            r = p[y] / float(q[b, j, y])
            return abs(float(u[b, j]) - r) <= TOL * r
        j += 1
    if o_na != g_na:
        return False
    # same accepted prefix: the draw differs
    if o_res is None:
        return False
    g_tok, o_tok = int(g_out[b, o_na]), int(o_out[b, o_na])
    if g_tok == o_tok:
        return False
    c = np.cumsum(o_res[b])
    uu = float(u[b, k])
    lo, hi = min(g_tok, o_tok), max(g_tok, o_tok)
    return bool(np.all(np.abs(c[lo:hi] - uu) <= TOL * uu))


# The kernel's top-p decision weights are within ~2e-9 relative of the real
# masses (plus the floor of each fixed-point weight, 2^-40 of the top mass),
# so its kept set can differ from the oracle's only where the oracle's margin
# |A - top_p M| (in units of the top mass) is below this bound.
def kernel_topp_bound(total, V):
    return 1e-8 * total + V * 2.0 ** -39


def _kept_set_boundary(x, dt, T, b, rows, top_k, top_p):
    """True when a top-p decision of one of the sequence's rows lies within
    the kernel's arithmetic bound of the oracle's (counted, not a failure)."""
    if top_p is None:
        return False
    k1, V = x.shape[1], x.shape[-1]
    for j in rows:
        if j >= k1:
            continue
        _, margin, total, _ = oracle.filter_info(x.reshape(-1, V), dt, b * k1 + j, T, *_filt(top_k, top_p, b))
        if margin <= kernel_topp_bound(total, V):
            STATS["kept_set_boundary"] = STATS.get("kept_set_boundary", 0) + 1
            return True
    return False


def check(x, dt, q, d, u, T=1.0, draft_len=None, eos=-1, remaining=None, residual=True, top_k=None, top_p=None):
    """top_k / top_p: None, or per-sequence numpy arrays (int32 / fp32): the
    filtered entry point runs and the oracle applies the same transforms.
    Where filtering is on, the support of every drawn bonus distribution
    (the kept set itself) must equal the oracle's, except where the oracle's
    top-p margin lies within the kernel's arithmetic bound (a counted
    boundary case)."""
    kw = dict(temperature=T, draft_len=None if draft_len is None else to_dev(draft_len), eos_id=eos,
              remaining=None if remaining is None else to_dev(remaining), want_residual=residual)
    if top_k is None and top_p is None:
        g = sv.spec_verify_sample(logits_to_dev(x, dt), to_dev(q), to_dev(d), to_dev(u), **kw)
    else:
        g = sv.spec_verify_sample_filtered(logits_to_dev(x, dt), to_dev(q), to_dev(d), to_dev(u),
                                           top_k=None if top_k is None else to_dev(np.asarray(top_k, np.int32)),
                                           top_p=None if top_p is None else to_dev(np.asarray(top_p, np.float32)),
                                           **kw)
    g_out, g_na, g_ne, g_fl = (t.cpu().numpy() for t in g[:4])
    g_res = g[4].cpu().numpy() if residual else None
    o_out, o_na, o_ne, o_fl, o_res = oracle.verify_sample(x, dt, q, d, u, T, draft_len, eos, remaining,
                                                          want_residual=True, top_k=top_k, top_p=top_p)
    B, k1 = o_out.shape
    kbs = np.full(B, k1 - 1) if draft_len is None else draft_len
    for b in range(B):
        STATS["decisions"] += int(o_ne[b]) + 1
        if o_fl[b] & 4:  # non-finite rows: only the flag is specified
            assert int(g_fl[b]) & 4
            continue
        same = (np.array_equal(g_out[b], o_out[b]) and g_na[b] == o_na[b] and g_ne[b] == o_ne[b])
        used = range(int(max(o_ne[b], g_ne[b])) + 1)
        if not same:
            if not _kept_set_boundary(x, dt, T, b, used, top_k, top_p):
                assert _boundary_explains(x, dt, q, d, u, T, b, o_out, o_na[b], o_ne[b], o_res, g_out, g_na[b],
                                          g_ne[b], int(kbs[b]), top_k, top_p), (b, g_out[b], o_out[b], g_na[b],
                                                                                 o_na[b])
            STATS["boundary"] += 1
            continue
        assert (int(g_fl[b]) & ~4) == (int(o_fl[b]) & ~4), (b, g_fl[b], o_fl[b])
        if residual and not np.isnan(o_res[b]).all():
            err = np.abs(g_res[b].astype(np.float64) - o_res[b])
            STATS["residual_rows"] += 1
            row = int(o_na[b])
            kb = int(kbs[b])
            if (top_k is not None or top_p is not None) and (row == kb or int(o_fl[b]) & 2):
                if not np.array_equal(g_res[b] > 0, o_res[b] > 0):
                    assert _kept_set_boundary(x, dt, T, b, [row], top_k, top_p), (
                        b, np.flatnonzero(g_res[b] > 0)[:20], np.flatnonzero(o_res[b] > 0)[:20])
                    STATS["boundary"] += 1
                    continue
                STATS["kept_sets"] = STATS.get("kept_sets", 0) + 1
            if err.max() > RES_TOL and _kept_set_boundary(x, dt, T, b, [row], top_k, top_p):
                STATS["boundary"] += 1  # the processed distribution itself differs by a boundary group
                continue
            if err.max() > RES_TOL:
                tol = residual_tolerance(x, dt, q, T, b, k1 - 1, row, row == kb, o_res[b], top_k, top_p)
                assert (err <= tol).all(), (b, err.max(), tol[np.argmax(err - tol)])
                STATS["widened_rows"] += 1
    return g, (o_out, o_na, o_ne, o_fl, o_res)


def test_config3_rounds():
    """B=32, k=4, V=128256 fp32 target, draft = target + N(0, 0.5), 20 rounds."""
    c = CONFIGS["c3"]
    g = torch.Generator(device=dev()).manual_seed(1003)
    acc = tested = 0
    widened = STATS["widened_rows"]
    for r in range(c["rounds"]):
        xt, qt, dt_, ut = torch_gen.sample_round_inputs(c["B"], c["k"], c["V"], c["noise"], g, torch.float32, dev())
        _, o = check(xt.cpu().numpy(), oracle.DT_F32, qt.cpu().numpy(), dt_.cpu().numpy(), ut.cpu().numpy())
        acc += o[1].sum()
        tested += o[1].sum() + (o[1] < c["k"]).sum()  # ratio tests actually performed
    # acceptance rate per ratio test ~ sum min(p, q) (about 0.8 for this construction)
    assert 0.7 < acc / tested < 0.9
    assert STATS["widened_rows"] == widened  # large vocabulary: the plain 1e-6 holds


def test_config5_stochastic_full_size():
    """B=256, k=8, V=128256 bf16 target; 1 GB of draft probabilities."""
    c = CONFIGS["c5"]
    g = torch.Generator(device=dev()).manual_seed(1005)
    for r in range(2):
        xt, qt, dt_, ut = torch_gen.sample_round_inputs(c["B"], c["k"], c["V"], c["noise"], g, torch.bfloat16,
                                                        dev())
        widened = STATS["widened_rows"]
        check(storage_of(xt), oracle.DT_BF16, qt.cpu().numpy(), dt_.cpu().numpy(), ut.cpu().numpy(),
              residual=(r == 0))
        assert STATS["widened_rows"] == widened


@pytest.mark.parametrize("V", [2, 3, 8, 100, 8193, 20000])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_small_vocabularies_many_draws(V, dtype):
    B = 4096 if V <= 100 else 64
    x, q, d, u = sample_round_inputs(B, 3, V, 0.8, seed=V, dtype=dtype)
    check(x, DT_OF[dtype], q, d, u)


@pytest.mark.parametrize("V,dtype", [(262144, "bf16"), (300007, "f32"), (600000, "bf16")])
def test_large_vocabularies(V, dtype):
    """Rows longer than 256 segments of 1024 (the draw's pick walks its
    segment sums in several blocks), one of them with a ragged tail."""
    x, q, d, u = sample_round_inputs(6, 2, V, 0.5, seed=V % 1000, dtype=dtype)
    check(x, DT_OF[dtype], q, d, u)


@pytest.mark.parametrize("V,dtype", [(70001, "bf16"), (40003, "f32"), (65536, "f16")])
def test_long_chunks(V, dtype):
    """1500 target rows of two chunks each, every chunk 4096 or more 16-byte
    vectors (several full batches per thread of the 256-thread statistics
    form); rows of odd length start unaligned, so chunks have scalar heads
    and tails."""
    x, q, d, u = sample_round_inputs(300, 4, V, 0.5, seed=V % 997, dtype=dtype)
    check(x, DT_OF[dtype], q, d, u)


@pytest.mark.parametrize("T", [0.5, 0.7, 1.5, 3.0])
def test_temperature(T):
    x, q, d, u = sample_round_inputs(256, 4, 5000, 0.5, seed=int(T * 10), dtype="f32")
    check(x, oracle.DT_F32, q, d, u, T=T)


def test_stop_rules_and_per_sequence_arguments():
    rng = np.random.default_rng(11)
    B, k, V = 512, 6, 50
    for trial in range(6):
        x, q, d, u = sample_round_inputs(B, k, V, 0.3, seed=trial, dtype="bf16")
        dl = rng.integers(0, k + 1, size=B).astype(np.int32)
        rem = rng.integers(-1, k + 3, size=B).astype(np.int32)
        eos = int(rng.integers(0, V))
        check(x, oracle.DT_BF16, q, d, u, draft_len=dl, eos=eos, remaining=rem)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_stop_rules_with_chunked_rows(dtype):
    """The per-sequence arguments on rows split over several work units
    (B=128, k=6: 896 rows of 40000 logits, three chunks each), so that a
    row's stop, budget and draft length meet the chunk counters."""
    rng = np.random.default_rng(13)
    B, k, V = 128, 6, 40000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=60 + len(dtype), dtype=dtype)
    dl = rng.integers(0, k + 1, size=B).astype(np.int32)
    rem = rng.integers(-1, k + 3, size=B).astype(np.int32)
    eos = int(rng.integers(0, V))
    d[::7, 0] = eos
    check(x, DT_OF[dtype], q, d, u, draft_len=dl, eos=eos, remaining=rem)


def test_flags_and_degenerate_rows():
    V, k, B = 16, 2, 6
    rng = np.random.default_rng(3)
    x = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    q = np.full((B, k, V), 1.0 / V, np.float32)
    d = rng.integers(0, V, size=(B, k)).astype(np.int32)
    u = rng.random((B, k + 1), dtype=np.float32)
    q[0, 0, d[0, 0]] = 0.0  # flag 1
    q[1, 0] = 1.5 * np.exp(x[1, 0]) / np.exp(x[1, 0]).sum()  # q > p everywhere: zero residual
    u[1, 0] = 0.9
    x[2, 0, 3] = np.inf  # flag 4
    x[3, 0, 5] = np.nan  # flag 4
    d[4, 0] = -3  # flag 8
    d[5, 1] = V + 2
    check(x, oracle.DT_F32, q, d, u)


def test_workspace_reuse_across_kinds():
    """Greedy and stochastic calls alternate on one workspace."""
    B = 64
    ws = sv.Workspace(B, sv.MAX_K, 20000, dev())
    for trial in range(4):
        x, q, d, u = sample_round_inputs(B, 4, 20000, 0.5, seed=100 + trial, dtype="f32")
        g = sv.spec_verify_sample(to_dev(x), to_dev(q), to_dev(d), to_dev(u), workspace=ws)
        o = oracle.verify_sample(x, oracle.DT_F32, q, d, u)
        assert np.array_equal(g[2].cpu().numpy(), o[2])
        gg = sv.spec_verify_greedy(to_dev(x), to_dev(d), workspace=ws)
        og = oracle.verify_greedy(x, oracle.DT_F32, d)
        assert np.array_equal(gg[0].cpu().numpy(), og[0])


def test_masked_vocabulary_rows():
    """Rows with -inf logits (masked tokens, e.g. after top-k filtering) are
    ordinary distributions: masked tokens have probability 0."""
    rng = np.random.default_rng(21)
    B, k, V = 256, 3, 3000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=21, dtype="f32")
    keep = rng.random((B, k + 1, V)) < 0.2
    keep[np.arange(B)[:, None], np.arange(k)[None, :], d] = True  # proposals stay unmasked
    x = np.where(keep, x, -np.inf).astype(np.float32)
    x[::17] = -np.inf  # a few sequences with every logit masked: undefined, flagged
    check(x, oracle.DT_F32, q, d, u)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # -inf survives bf16 truncation
    check(xb, oracle.DT_BF16, q, d, u)


def test_zz_boundary_rate():
    """All files above: boundary cases stay below 1e-4 of the decisions."""
    assert STATS["decisions"] > 50_000
    assert STATS["boundary"] < 1e-4 * STATS["decisions"], STATS
    print("sampling parity statistics:", STATS)
