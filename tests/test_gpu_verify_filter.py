"""Stochastic verification with top-k / top-p on the target distribution:
the CUDA path (spec_verify_sample_filtered) vs the CPU oracle.

Same bar as the unfiltered stochastic tests (tokens and counts equal except
counted boundary decisions of the ratio test or the draw; normalised draw
distributions within 1e-6), plus: the kept set itself -- wherever a sequence
draws its bonus from the processed target distribution, the support of that
distribution equals the oracle's.  The oracle decides the top-p boundary on
the real masses (fp64 with an error band); the kernel on fixed-point weights
within ~2e-9 of them.  A kept set may differ only where the oracle's margin
lies inside the kernel's bound; such rows count as boundary cases, under the
same bar (fewer than 1e-4 of the decisions).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import DT_OF, dev, storage_of, to_dev
from specgen import CONFIGS, sample_round_inputs
from specgen import torch_gen
from test_gpu_verify_sample import STATS, check

pytestmark = pytest.mark.gpu


def _params(rng, B, V):
    """Per-sequence top_k / top_p covering off values, the extremes and
    typical settings."""
    tk = rng.choice([0, 1, 2, 5, 50, V - 1, V, V + 7, -1, int(rng.integers(1, V + 1))], size=B).astype(np.int32)
    tp = rng.choice([1.0, 0.0, 1e-6, 0.3, 0.5, 0.8, 0.9, 0.95, 0.999, np.nan, float(rng.random())],
                    size=B).astype(np.float32)
    return tk, tp


@pytest.mark.parametrize("V", [2, 3, 8, 100, 8193, 20000])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_small_vocabularies(V, dtype):
    B = 1024 if V <= 100 else 64
    rng = np.random.default_rng(V + 7)
    x, q, d, u = sample_round_inputs(B, 3, V, 0.8, seed=V + 1, dtype=dtype)
    tk, tp = _params(rng, B, V)
    check(x, DT_OF[dtype], q, d, u, top_k=tk, top_p=tp)


@pytest.mark.parametrize("only", ["k", "p"])
def test_one_transform_at_a_time(only):
    rng = np.random.default_rng(3 if only == "k" else 4)
    B, k, V = 128, 4, 30000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=33, dtype="bf16")
    tk, tp = _params(rng, B, V)
    check(x, oracle.DT_BF16, q, d, u, top_k=tk if only == "k" else None, top_p=tp if only == "p" else None)


def test_ties_at_the_cut():
    """Coarsely quantised logits: many tokens share each value, so the k-th
    value and the top-p boundary fall inside groups of equal logits."""
    rng = np.random.default_rng(5)
    B, k, V = 256, 3, 4000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=55, dtype="f32")
    x = (np.round(x * 4) / 4).astype(np.float32)
    tk, tp = _params(rng, B, V)
    check(x, oracle.DT_F32, q, d, u, top_k=tk, top_p=tp)
    check(x, oracle.DT_F32, q, d, u, top_k=np.full(B, 37, np.int32), top_p=np.full(B, 0.9, np.float32))


@pytest.mark.parametrize("T", [0.6, 1.0, 2.5])
def test_temperature_with_transforms(T):
    rng = np.random.default_rng(int(T * 10))
    B, k, V = 96, 4, 12000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=int(T * 100), dtype="f32")
    tk, tp = _params(rng, B, V)
    check(x, oracle.DT_F32, q, d, u, T=T, top_k=tk, top_p=tp)


def test_masked_tokens_and_stop_rules():
    rng = np.random.default_rng(9)
    B, k, V = 256, 5, 2000
    x, q, d, u = sample_round_inputs(B, k, V, 0.4, seed=99, dtype="bf16")
    xf = x.astype(np.uint32) << 16
    mask = rng.random(x.shape) < 0.7
    mask[np.arange(B)[:, None], np.arange(k)[None, :], d] = False  # proposals stay finite
    xf[mask] = np.uint32(0xFF800000)  # -inf
    xm = (xf >> 16).astype(np.uint16)
    tk, tp = _params(rng, B, V)
    dl = rng.integers(0, k + 1, size=B).astype(np.int32)
    rem = rng.integers(0, k + 3, size=B).astype(np.int32)
    check(xm, oracle.DT_BF16, q, d, u, draft_len=dl, eos=int(rng.integers(0, V)), remaining=rem, top_k=tk, top_p=tp)


def test_top_k_one_equals_greedy_on_device():
    """top_k = 1 turns stochastic verification into greedy verification where
    every row's maximum is unique (fp32 logits; tied maxima are all kept by
    top-k and then sampled, while greedy takes the lowest index)."""
    B, k, V = 128, 4, 50000
    x, q, d, u = sample_round_inputs(B, k, V, 0.3, seed=7, dtype="f32")
    top2 = np.sort(x, axis=-1)[..., -2:]
    assert (top2[..., 1] > top2[..., 0]).all()
    best = x[:, :k].argmax(-1).astype(np.int32)
    d = np.where(np.random.default_rng(1).random((B, k)) < 0.8, best, d).astype(np.int32)
    xt = to_dev(x)
    g = sv.spec_verify_sample_filtered(xt, to_dev(q), to_dev(d), to_dev(u), top_k=1)
    gg = sv.spec_verify_greedy(xt, to_dev(d))
    assert np.array_equal(g[0].cpu().numpy(), gg[0].cpu().numpy())
    assert np.array_equal(g[2].cpu().numpy(), gg[2].cpu().numpy())


def test_config3_shape_typical_settings():
    """B=32, k=4, V=128256 fp32 with top_k=50 / top_p=0.9 and mixed settings."""
    c = CONFIGS["c3"]
    g = torch.Generator(device=dev()).manual_seed(2003)
    rng = np.random.default_rng(2003)
    for r in range(3):
        xt, qt, dt_, ut = torch_gen.sample_round_inputs(c["B"], c["k"], c["V"], c["noise"], g, torch.float32, dev())
        if r == 0:
            tk, tp = np.full(c["B"], 50, np.int32), np.full(c["B"], 0.9, np.float32)
        else:
            tk, tp = _params(rng, c["B"], c["V"])
        check(xt.cpu().numpy(), oracle.DT_F32, qt.cpu().numpy(), dt_.cpu().numpy(), ut.cpu().numpy(),
              top_k=tk, top_p=tp)


@pytest.mark.parametrize("B,dtype", [(32, "f32"), (40, "bf16")])
def test_top_p_alone_between_one_and_two_rows_per_sm(B, dtype):
    """Top-p without a top-k array on 160 / 200 rows: the filter's 512-thread
    form (every row in the first wave)."""
    c = CONFIGS["c3"]
    k, V = c["k"], c["V"] if dtype == "f32" else 30000
    rng = np.random.default_rng(B)
    x, q, d, u = sample_round_inputs(B, k, V, c["noise"], seed=B + 11, dtype=dtype)
    tp = rng.choice([0.5, 0.8, 0.9, 0.95, 1.0], size=B).astype(np.float32)
    check(x, DT_OF[dtype], q, d, u, top_k=None, top_p=tp)


def test_config5_shape_bf16():
    """B=64 of config 5's rows (k=8, V=128256 bf16), top_p = 0.95."""
    c = CONFIGS["c5"]
    g = torch.Generator(device=dev()).manual_seed(2005)
    xt, qt, dt_, ut = torch_gen.sample_round_inputs(64, c["k"], c["V"], c["noise"], g, torch.bfloat16, dev())
    check(storage_of(xt), oracle.DT_BF16, qt.cpu().numpy(), dt_.cpu().numpy(), ut.cpu().numpy(),
          top_k=None, top_p=np.full(64, 0.95, np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("top_p", [0.5, 0.9, 0.95])
def test_kept_set_of_every_row(dtype, top_p):
    """k = 0: every row is its sequence's bonus row, so the support of every
    drawn distribution is the kernel's kept set for that row; 128 rows of
    128256 N(0,1) logits (the stochastic workloads' vocabulary) against the
    oracle's top-p on the real masses."""
    B, V = 128, 128256
    x, q, d, u = sample_round_inputs(B, 0, V, 0.5, seed=int(top_p * 1000) + (dtype == "bf16"), dtype=dtype)
    before = STATS.get("kept_sets", 0) + STATS["boundary"]
    check(x, DT_OF[dtype], q, d, u, top_k=None, top_p=np.full(B, top_p, np.float32))
    # every row either had its kept set compared or was a counted boundary
    # case (a top-p decision inside the kernel's bound, or a draw boundary)
    assert STATS.get("kept_sets", 0) + STATS["boundary"] - before == B


@pytest.mark.parametrize("V,dtype", [(32768, "bf16"), (50001, "f16"), (128256, "bf16"), (262144, "f16")])
def test_table_form_16bit(V, dtype):
    """16-bit rows of at least 32768 logits: the cut from the table of value
    counts (mixed per-sequence settings, off values and extremes)."""
    B = 48 if V <= 50001 else 16
    rng = np.random.default_rng(V + 3)
    x, q, d, u = sample_round_inputs(B, 3, V, 0.5, seed=V % 991, dtype=dtype)
    tk, tp = _params(rng, B, V)
    check(x, DT_OF[dtype], q, d, u, top_k=tk, top_p=tp)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_table_form_stop_rules_and_per_sequence_arguments(dtype):
    """The table form (16-bit rows of 40000 logits) with draft lengths, output
    budgets (including none) and an EOS that some proposals carry, over 160
    sequences -- more rows than SMs, so rows are skipped once a stop is known."""
    rng = np.random.default_rng(21 + len(dtype))
    B, k, V = 160, 5, 40000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=210 + len(dtype), dtype=dtype)
    tk, tp = _params(rng, B, V)
    dl = rng.integers(0, k + 1, size=B).astype(np.int32)
    rem = rng.integers(-1, k + 3, size=B).astype(np.int32)
    eos = int(rng.integers(0, V))
    d[::6, 0] = eos
    check(x, DT_OF[dtype], q, d, u, draft_len=dl, eos=eos, remaining=rem, top_k=tk, top_p=tp)


@pytest.mark.parametrize("T", [0.6, 2.5])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_table_form_temperature(T, dtype):
    """The table form with T != 1: its decision weights take log2(e) / T as
    a float pair, and the kept probabilities the scaled softmax."""
    rng = np.random.default_rng(int(T * 10) + len(dtype))
    B, k, V = 48, 3, 40000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=int(T * 100) + len(dtype), dtype=dtype)
    tk, tp = _params(rng, B, V)
    check(x, DT_OF[dtype], q, d, u, T=T, top_k=tk, top_p=tp)


def _bits16(x):
    return x.view(np.uint16) if x.dtype == np.float16 else x


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("step", [64, 4])
def test_table_form_ties_and_signed_zeros(dtype, step):
    """Logits quantised to 1/step (many tokens per value, -0 and +0 both
    present and equal): the k-th value and the top-p boundary fall inside
    groups of equal logits, some at zero; at 1/64 a value holds a few
    hundred tokens, at 1/4 several thousand."""
    rng = np.random.default_rng(61 + step)
    B, k, V = 64, 3, 40000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=62, dtype=dtype)
    xf = np.round(rng.standard_normal(x.shape).astype(np.float32) * step) / step
    xf[xf == 0] = np.where(rng.random(np.count_nonzero(xf == 0)) < 0.5, -0.0, 0.0)
    if dtype == "bf16":
        xs = (xf.view(np.uint32) >> 16).astype(np.uint16)
    else:
        xs = xf.astype(np.float16)
    assert (_bits16(xs) == 0x8000).any() and (_bits16(xs) == 0).any()
    counts = np.unique(_bits16(xs)[0, 0], return_counts=True)[1]
    assert (counts.max() < 1023) == (step == 64)
    tk, tp = _params(rng, B, V)
    check(xs, DT_OF[dtype], q, d, u, top_k=tk, top_p=tp)
    check(xs, DT_OF[dtype], q, d, u, top_k=np.full(B, 5000, np.int32), top_p=np.full(B, 0.6, np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_table_form_counter_wrap_and_bad_rows(dtype):
    """Rows where more than 65535 logits share one value (a 16-bit counter
    wraps, or would when -0 joins +0): the row takes the radix selection and
    matches all the same.  Rows with 50000 masked (-inf) logits stay in the
    table.  Rows with a NaN (either sign) or +inf are flagged."""
    rng = np.random.default_rng(71)
    B, k, V = 12, 2, 140000
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=72, dtype=dtype)
    xb = _bits16(x)
    one = 0x3F80 if dtype == "bf16" else 0x3C00
    pinf = 0x7F80 if dtype == "bf16" else 0x7C00
    for b in range(0, B, 3):  # 70000 logits equal to 1.0 in every row of these sequences
        for j in range(k + 1):
            xb[b, j, rng.choice(V, 70000, replace=False)] = one
    for b in range(1, B, 3):  # 40000 +0 and 30000 -0
        for j in range(k + 1):
            idx = rng.choice(V, 70000, replace=False)
            xb[b, j, idx[:40000]] = 0x0000
            xb[b, j, idx[40000:]] = 0x8000
    ninf = 0xFF80 if dtype == "bf16" else 0xFC00
    for b in range(2, B, 3):  # 50000 masked tokens (-inf), the proposals kept unmasked
        for j in range(k + 1):
            idx = rng.choice(V, 50000, replace=False)
            idx = idx[~np.isin(idx, d[b])]
            xb[b, j, idx] = ninf
    xb[2, 0, 17] = 0xFFC1 if dtype == "bf16" else 0xFE01   # negative NaN
    xb[5, 1, 99] = pinf                                     # +inf
    xb[8, 0, 1234] = 0x7FC1 if dtype == "bf16" else 0x7E01  # positive NaN
    d[2, 0] = d[2, 0] if d[2, 0] != 17 else 18
    tk = rng.choice([0, 3, 80000, V - 1], size=B).astype(np.int32)
    tp = rng.choice([0.5, 0.9, 0.99, 1.0], size=B).astype(np.float32)
    check(x, DT_OF[dtype], q, d, u, top_k=tk, top_p=tp)


def test_zz_filter_statistics():
    """Every file above that shares the counters: kept sets compared, and
    boundary cases (ratio test, draw, or a top-p decision inside the
    kernel's bound) below 1e-4 of the decisions."""
    assert STATS.get("kept_sets", 0) > 500, STATS
    assert STATS["decisions"] > 20_000, STATS  # one boundary case would then be below 1e-4 of them
    assert STATS["boundary"] < 1e-4 * STATS["decisions"], STATS
    print("filtered sampling statistics:", STATS)
