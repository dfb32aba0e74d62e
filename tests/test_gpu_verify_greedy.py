"""Greedy verification: CUDA path vs the CPU oracle, bit-exact on tokens,
accepted and committed counts (tokens are integers decided by an argmax in the
storage type's exact values on both sides)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import DT_OF, TORCH_DT, dev, logits_to_dev, storage_of, to_dev
from specgen import CONFIGS, greedy_round_inputs
from specgen import torch_gen

pytestmark = pytest.mark.gpu


def run_both(x, dt, d, draft_len=None, eos=-1, remaining=None, repeat=1):
    xt = logits_to_dev(x, dt)
    dt_ = to_dev(d)
    dl = None if draft_len is None else to_dev(draft_len)
    rem = None if remaining is None else to_dev(remaining)
    outs = []
    for _ in range(repeat):  # later calls reuse the workspace the first left
        o, na, ne = sv.spec_verify_greedy(xt, dt_, draft_len=dl, eos_id=eos, remaining=rem)
        outs.append((o.cpu().numpy(), na.cpu().numpy(), ne.cpu().numpy()))
    ref = oracle.verify_greedy(x, dt, d, draft_len, eos, remaining)
    for got in outs:
        for g, r, name in zip(got, ref, ("out_tokens", "n_accept", "n_emit")):
            assert np.array_equal(g, r), (name, np.nonzero(g != r))
    return ref


@pytest.mark.parametrize("name,alpha", [("c1", 0.7), ("c2", 0.5), ("c2", 0.8)])
def test_config_rounds(name, alpha):
    c = CONFIGS[name]
    dt = DT_OF[c["logit_dtype"]]
    total = 0
    for r in range(20):
        x, d = greedy_round_inputs(c["B"], c["k"], c["V"], alpha, c["sigma"], seed=1000 + r, dtype=c["logit_dtype"])
        _, _, ne = run_both(x, dt, d)
        total += ne.sum()
    ek = (1 - alpha ** (c["k"] + 1)) / (1 - alpha)
    assert abs(total / (20 * c["B"]) - ek) < 1.2  # sanity of the workload, not a parity criterion


@pytest.mark.parametrize("k", [4, 6, 8])
def test_config4_shapes(k):
    c = CONFIGS["c4"]
    x, d = greedy_round_inputs(c["B"], k, c["V"], 0.7, c["sigma"], seed=1004 + k, dtype="bf16")
    run_both(x, oracle.DT_BF16, d)


@pytest.mark.parametrize("alpha", [0.3, 0.6, 0.9])
def test_config5_full_size(alpha):
    """B=256, k=8, V=128256 bf16: 591 MB of logits, generated on the device."""
    c = CONFIGS["c5"]
    g = torch.Generator(device=dev()).manual_seed(1005 + int(alpha * 10))
    xt, dt_ = torch_gen.greedy_round_inputs(c["B"], c["k"], c["V"], alpha, c["sigma"], g, torch.bfloat16, dev())
    o, na, ne = sv.spec_verify_greedy(xt, dt_)
    ref = oracle.verify_greedy(storage_of(xt), oracle.DT_BF16, dt_.cpu().numpy())
    assert np.array_equal(o.cpu().numpy(), ref[0])
    assert np.array_equal(na.cpu().numpy(), ref[1]) and np.array_equal(ne.cpu().numpy(), ref[2])


@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 255, 8191, 8192, 8193, 3 * 8192 + 5, 40000])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_ragged_vocab_sizes(V, dtype):
    """Rows that are not 16-byte multiples start unaligned; chunk tails ragged."""
    x, d = greedy_round_inputs(6, 3, V, 0.6, 1.0, seed=V, dtype=dtype)
    run_both(x, DT_OF[dtype], d, repeat=2)


def test_stop_rules_and_per_sequence_arguments():
    rng = np.random.default_rng(7)
    B, k, V = 64, 6, 300
    for trial in range(10):
        x, d = greedy_round_inputs(B, k, V, 0.8, 1.0, seed=50 + trial, dtype="bf16")
        dl = rng.integers(0, k + 1, size=B).astype(np.int32)
        rem = rng.integers(-1, k + 3, size=B).astype(np.int32)
        eos = int(rng.integers(0, V))
        # make EOS appear as an accepted proposal in some sequences
        d[::5, 1] = eos
        run_both(x, oracle.DT_BF16, d, draft_len=dl, eos=eos, remaining=rem)


@pytest.mark.parametrize("k", [0, 1, 31])
def test_extreme_k(k):
    x, d = greedy_round_inputs(3, k, 5000, 0.95, 1.0, seed=k, dtype="f32")
    run_both(x, oracle.DT_F32, d)


def test_ties_nan_inf_and_signed_zero():
    B, k, V = 6, 3, 3 * 8192 + 100
    x = np.zeros((B, k + 1, V), np.float32)
    x[0, :, :] = 1.0  # every index ties: lowest index 0
    x[1, :, [5, 8192 + 3, 2 * 8192 + 7]] = 2.0  # ties in three different chunks
    x[2, :, 9000] = np.inf
    x[2, :, 100] = np.inf  # +inf tie: lowest index
    x[3, :, 20000] = np.nan
    x[3, :, 30] = 5.0
    x[3, 1, 10] = np.nan  # first NaN wins
    x[4, :, :] = -np.inf
    x[4, 2, 77] = -1.0
    x[5, :, :] = -0.0
    x[5, :, 4] = 0.0  # -0 and +0 equal: index 0 wins
    d = np.array([[0, 0, 0], [5, 5, 1], [100, 9000, 100], [20000, 10, 20000], [0, 0, 77], [0, 4, 0]], np.int32)
    run_both(x, oracle.DT_F32, d, repeat=2)


def test_early_rejection_declines_when_unsure():
    """A row's rejection is posted early only when a finite element lies
    strictly above the proposal's logit.  These rows must reach the oracle's
    answer through the full argmax instead: a NaN proposal logit (the only
    NaN: the proposal is the argmax), a proposal outside [0, V), a proposal
    tied with the maximum at a lower index (rejected by the tie rule), a +inf
    proposal (accepted), a -inf proposal (rejected early), a NaN elsewhere in
    the row (the NaN is the argmax), and a row where the proposal is beaten
    only in its last chunk."""
    rng = np.random.default_rng(91)
    B, k, V = 8, 4, 5 * 8192 + 37
    x = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    # make every proposal the argmax of its row first (accepted), then break some
    for b in range(B):
        for j in range(k):
            x[b, j, d[b, j]] = 10.0
    x[0, 0, d[0, 0]] = np.nan                      # the only NaN: accepted
    d[1, 0] = V + 3                                # outside the vocabulary: rejected
    x[2, 1, 7] = 10.0                              # tie with the maximum at a lower index
    d[2, 1] = max(int(d[2, 1]), 8)
    x[2, 1, d[2, 1]] = 10.0
    x[3, 0, d[3, 0]] = np.inf                      # +inf: accepted
    x[4, 0, d[4, 0]] = -np.inf                     # -inf: rejected
    x[5, 0, (d[5, 0] + 100) % V] = np.nan          # a NaN elsewhere is the argmax
    x[6, 0, :] = -5.0                              # beaten only near the row's end
    x[6, 0, d[6, 0]] = 1.0
    x[6, 0, V - 2] = 2.0
    run_both(x, oracle.DT_F32, d, repeat=2)


# Larger batches (512 to 1152 target rows, several chunks per row): the cases
# above at such sizes -- ragged chunks, stop rules, ties and NaN across chunk
# boundaries, early rejection, acceptance 0 and 1, and one workspace shared
# by calls of different k and V.
BIG_B, BIG_K = 128, 4  # 640 rows


@pytest.mark.parametrize("V", [1, 7, 16383, 16384, 16385, 2 * 16384 + 5, 40000])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_large_batch_ragged_vocab_sizes(V, dtype):
    x, d = greedy_round_inputs(BIG_B, BIG_K, V, 0.6, 1.0, seed=300 + V, dtype=dtype)
    run_both(x, DT_OF[dtype], d, repeat=2)


@pytest.mark.parametrize("alpha", [0.0, 0.5, 1.0])
def test_large_batch_acceptance_extremes(alpha):
    """alpha 0: only row 0 of every sequence is needed; alpha 1: every row."""
    x, d = greedy_round_inputs(64, 8, 50000, alpha, 1.0, seed=int(alpha * 10) + 310, dtype="bf16")
    ref = run_both(x, oracle.DT_BF16, d, repeat=2)
    if alpha == 1.0:
        assert (ref[2] == 9).all()
    if alpha == 0.0:
        assert (ref[2] == 1).all()


def test_large_batch_stop_rules_and_per_sequence_arguments():
    rng = np.random.default_rng(17)
    B, k, V = 128, 6, 20000
    for trial in range(6):
        x, d = greedy_round_inputs(B, k, V, 0.8, 1.0, seed=350 + trial, dtype="bf16")
        dl = rng.integers(0, k + 1, size=B).astype(np.int32)
        rem = rng.integers(-1, k + 3, size=B).astype(np.int32)
        eos = int(rng.integers(0, V))
        d[::5, 1] = eos
        run_both(x, oracle.DT_BF16, d, draft_len=dl, eos=eos, remaining=rem)


def test_large_batch_ties_nan_inf_and_signed_zero():
    """The special rows of the small case, placed among 128 sequences, with
    ties 16384 elements apart."""
    B, k, V = BIG_B, 3, 3 * 16384 + 100
    x, d = greedy_round_inputs(B, k, V, 0.5, 1.0, seed=360, dtype="f32")
    x[0, :, :] = 1.0
    x[1, :, [5, 16384 + 3, 2 * 16384 + 7]] = 20.0
    x[2, :, 30000] = np.inf
    x[2, :, 100] = np.inf
    x[3, :, 40000] = np.nan
    x[3, :, 30] = 25.0
    x[3, 1, 10] = np.nan
    x[4, :, :] = -np.inf
    x[4, 2, 77] = -1.0
    x[5, :, :] = -0.0
    x[5, :, 4] = 0.0
    d[:6] = np.array([[0, 0, 0], [5, 5, 1], [100, 30000, 100], [40000, 10, 40000], [0, 0, 77], [0, 4, 0]],
                     np.int32)
    run_both(x, oracle.DT_F32, d, repeat=2)


def test_large_batch_early_rejection_declines_when_unsure():
    rng = np.random.default_rng(93)
    B, k, V = BIG_B, 4, 3 * 16384 + 37
    x = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    d = rng.integers(0, V, (B, k)).astype(np.int32)
    for b in range(B):
        for j in range(k):
            x[b, j, d[b, j]] = 10.0
    x[0, 0, d[0, 0]] = np.nan
    d[1, 0] = V + 3
    x[2, 1, 7] = 10.0
    d[2, 1] = max(int(d[2, 1]), 8)
    x[2, 1, d[2, 1]] = 10.0
    x[3, 0, d[3, 0]] = np.inf
    x[4, 0, d[4, 0]] = -np.inf
    x[5, 0, (d[5, 0] + 100) % V] = np.nan
    x[6, 0, :] = -5.0
    x[6, 0, d[6, 0]] = 1.0
    x[6, 0, V - 2] = 2.0
    run_both(x, oracle.DT_F32, d, repeat=2)


def test_large_batch_calls_share_one_workspace():
    """Every counter is returned to zero by every call: calls of different k
    and V on one workspace stay exact."""
    B = BIG_B
    ws = sv.Workspace(B, sv.MAX_K, 40000, dev())
    for trial, (k, V) in enumerate([(8, 40000), (2, 40000), (3, 1000), (1, 20000), (31, 700), (8, 40000)]):
        x, d = greedy_round_inputs(B, k, V, 0.7, 2.0, seed=370 + trial, dtype="bf16")
        o, na, ne = sv.spec_verify_greedy(logits_to_dev(x, oracle.DT_BF16), to_dev(d), workspace=ws)
        ref = oracle.verify_greedy(x, oracle.DT_BF16, d)
        assert np.array_equal(o.cpu().numpy(), ref[0]) and np.array_equal(ne.cpu().numpy(), ref[2])
        assert np.array_equal(na.cpu().numpy(), ref[1])


def test_empty_batch_is_a_noop():
    x = torch.zeros((0, 3, 100), dtype=torch.float32, device=dev())
    d = torch.zeros((0, 2), dtype=torch.int32, device=dev())
    o, na, ne = sv.spec_verify_greedy(x, d)
    assert o.shape == (0, 3)


def test_interleaved_sizes_share_one_workspace():
    """Counters are returned to zero by every call, so calls with different k
    and V on one workspace (same batch size) stay correct."""
    B = 16
    ws = sv.Workspace(B, sv.MAX_K, 64000, dev())
    for trial, (k, V) in enumerate([(5, 32000), (2, 64000), (8, 1000), (31, 50), (5, 32000)]):
        x, d = greedy_round_inputs(B, k, V, 0.7, 2.0, seed=trial, dtype="bf16")
        o, na, ne = sv.spec_verify_greedy(logits_to_dev(x, oracle.DT_BF16), to_dev(d), workspace=ws)
        ref = oracle.verify_greedy(x, oracle.DT_BF16, d)
        assert np.array_equal(o.cpu().numpy(), ref[0]) and np.array_equal(ne.cpu().numpy(), ref[2])
    assert int(ws.buf.cpu().numpy()[:4096].sum()) >= 0  # buffer still readable


def test_torch_dtypes_roundtrip():
    for name in ("f32", "bf16", "f16"):
        x = torch.randn((4, 3, 999), device=dev()).to(TORCH_DT[name])
        d = torch.randint(0, 999, (4, 2), device=dev(), dtype=torch.int32)
        o, na, ne = sv.spec_verify_greedy(x, d)
        ref = oracle.verify_greedy(storage_of(x), DT_OF[name], d.cpu().numpy())
        assert np.array_equal(o.cpu().numpy(), ref[0])
