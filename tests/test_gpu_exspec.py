"""Ragged pool (EXSPEC) on the device vs the oracle, bit-exact: the commit
(length update = rollback of rejected tokens), repad (pool -> left-padded
batch) and unpad (batch -> pool), and EXSPEC decoding of the toy pair with
grouped rounds and unpad-append-repad fallbacks running on the device."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import dev, to_dev
from oracle import DT_F32
from oracle.toy import ToyPair, run_exspec

pytestmark = pytest.mark.gpu


def test_commit_matches_oracle_and_refuses_bad_input():
    rng = np.random.default_rng(1)
    N, S = 300, 2048
    for trial in range(20):
        pl = rng.integers(1, 1500, size=N).astype(np.int32)
        B = int(rng.integers(1, 65))
        idx = rng.choice(N, size=B, replace=False).astype(np.int32)
        ne = rng.integers(0, 10, size=B).astype(np.int32)
        g = to_dev(pl.copy())
        err = sv.spec_commit_ragged(g, to_dev(idx), to_dev(ne), S)
        ref = pl.copy()
        assert oracle.commit_ragged(ref, idx, ne, S) == 0 and int(err.item()) == 0
        assert np.array_equal(g.cpu().numpy(), ref)
    pl = np.full(8, 10, np.int32)
    for idx, ne, want in (([1, 1], [1, 1], sv.REALIGN_LAYOUT), ([9], [1], sv.REALIGN_LAYOUT),
                          ([2], [-1], sv.REALIGN_LAYOUT), ([3, 4], [0, 7], sv.REALIGN_CAPACITY)):
        g = to_dev(pl.copy())
        err = sv.spec_commit_ragged(g, to_dev(np.array(idx, np.int32)), to_dev(np.array(ne, np.int32)), 16)
        assert int(err.item()) == want and np.array_equal(g.cpu().numpy(), pl)


@pytest.mark.parametrize("dtype,D", [(np.float16, 128), (np.float32, 64), (np.float32, 3), (np.float16, 5)])
def test_repad_and_unpad_match_oracle(dtype, D):
    rng = np.random.default_rng(D)
    L, N, H, S, B = 2, 40, 3, 300, 12
    pool = rng.standard_normal((L, 2, N, H, S, D)).astype(dtype)
    pl = rng.integers(1, 280, size=N).astype(np.int32)
    idx = rng.choice(N, size=B, replace=False).astype(np.int32)
    batch = rng.standard_normal((L, 2, B, H, S, D)).astype(dtype)
    pool_t, batch_t = torch.from_numpy(pool.copy()).to(dev()), torch.from_numpy(batch.copy()).to(dev())
    ln, pd, w, err = sv.spec_repad_gather(pool_t, batch_t, to_dev(idx), to_dev(pl))
    st, o_ln, o_pd, o_w = oracle.repad_gather(pool, batch, idx, pl)
    assert st == 0 and int(err.item()) == 0 and int(w.item()) == o_w
    assert np.array_equal(ln.cpu().numpy(), o_ln) and np.array_equal(pd.cpu().numpy(), o_pd)
    assert np.array_equal(batch_t.cpu().numpy(), batch)
    # a round changes the batch lengths; unpad sends them back
    new_len = (o_ln + rng.integers(0, 4, size=B)).astype(np.int32)
    new_pad = (int(new_len.max()) - new_len).astype(np.int32)
    batch2 = rng.standard_normal((L, 2, B, H, S, D)).astype(dtype)
    batch2_t = torch.from_numpy(batch2.copy()).to(dev())
    pl_t = to_dev(pl.copy())
    err = sv.spec_unpad_scatter(batch2_t, pool_t, to_dev(idx), to_dev(new_len), to_dev(new_pad), pl_t)
    pl_ref = pl.copy()
    assert oracle.unpad_scatter(batch2, pool, idx, new_len, new_pad, pl_ref) == 0 and int(err.item()) == 0
    assert np.array_equal(pool_t.cpu().numpy(), pool) and np.array_equal(pl_t.cpu().numpy(), pl_ref)


def test_repad_unpad_refuse_bad_input_and_write_nothing():
    L, N, H, S, D, B = 1, 6, 2, 16, 8, 2
    pool = np.arange(L * 2 * N * H * S * D, dtype=np.float32).reshape(L, 2, N, H, S, D)
    batch = np.zeros((L, 2, B, H, S, D), np.float32)
    pool_t, batch_t = torch.from_numpy(pool.copy()).to(dev()), torch.from_numpy(batch.copy()).to(dev())
    pl = np.array([4, 6, 0, 9, 16, 17], np.int32)
    for idx in ([0, 0], [0, 6], [0, 2], [5, 1]):  # repeated, outside, length 0, length past S
        _, _, _, err = sv.spec_repad_gather(pool_t, batch_t, to_dev(np.array(idx, np.int32)), to_dev(pl))
        assert int(err.item()) == sv.REALIGN_LAYOUT
    assert not batch_t.any()
    pl_t = to_dev(pl.copy())
    err = sv.spec_unpad_scatter(batch_t, pool_t, to_dev(np.array([0, 1], np.int32)),
                                to_dev(np.array([4, 10], np.int32)), to_dev(np.array([0, 8], np.int32)), pl_t)
    assert int(err.item()) == sv.REALIGN_LAYOUT  # 8 + 10 - 1 > 16
    assert np.array_equal(pool_t.cpu().numpy(), pool) and np.array_equal(pl_t.cpu().numpy(), pl)


def test_config4_shaped_pool_round_trip():
    """A c4-shaped pool (512 sequences, lengths U[128,1024], GQA heads,
    D=128 bf16; 2 of the 28 layers): repad 64 sequences, unpad them back
    unchanged, bit-exact against the oracle on the whole pool."""
    rng = np.random.default_rng(1004)
    L, N, H, S, D, B = 2, 512, 4, 2048, 128, 64
    pool = rng.integers(0, 65535, size=(L, 2, N, H, S, D), dtype=np.uint16)
    pl = rng.integers(128, 1025, size=N).astype(np.int32)
    idx = rng.choice(N, size=B, replace=False).astype(np.int32)
    pool_t = torch.from_numpy(pool.view(np.int16)).to(dev()).view(torch.bfloat16)
    batch_t = torch.zeros((L, 2, B, H, S, D), dtype=torch.bfloat16, device=dev())
    ln, pd, w, err = sv.spec_repad_gather(pool_t, batch_t, to_dev(idx), to_dev(pl))
    batch = np.zeros((L, 2, B, H, S, D), np.uint16)
    st, o_ln, o_pd, o_w = oracle.repad_gather(pool, batch, idx, pl)
    assert st == 0 and int(err.item()) == 0
    assert np.array_equal(batch_t.view(torch.int16).cpu().numpy().view(np.uint16), batch)
    pool_t.view(torch.int16).zero_()  # unpad must rebuild the chosen sequences' valid rows
    pl_t = to_dev(pl.copy())
    err = sv.spec_unpad_scatter(batch_t, pool_t, to_dev(idx), ln, pd, pl_t)
    got = pool_t.view(torch.int16).cpu().numpy().view(np.uint16)
    for b, n in enumerate(idx):
        assert np.array_equal(got[:, :, n, :, : pl[n] - 1], pool[:, :, n, :, : pl[n] - 1])
    assert int(err.item()) == 0 and np.array_equal(pl_t.cpu().numpy(), pl)


# -- toy EXSPEC decoding on the device ------------------------------------------------

def device_ops():
    def group(lens, B):
        idx, ce, gl = sv.spec_group_by_length(to_dev(lens), B)
        return idx.cpu().numpy(), int(ce.item()), int(gl.item())

    def verify(x, d, rem, eos):
        o, na, ne = sv.spec_verify_greedy(to_dev(x), to_dev(d), eos_id=eos, remaining=to_dev(rem))
        return o.cpu().numpy(), na.cpu().numpy(), ne.cpu().numpy()

    def commit(pl, idx, ne, S):
        g = to_dev(pl.copy())
        err = sv.spec_commit_ragged(g, to_dev(np.asarray(idx, np.int32)), to_dev(np.asarray(ne, np.int32)), S)
        pl[...] = g.cpu().numpy()
        return int(err.item())

    def repad(pool, batch, idx, pl):
        p_t, b_t = torch.from_numpy(pool).to(dev()), torch.from_numpy(batch).to(dev())
        ln, pd, w, err = sv.spec_repad_gather(p_t, b_t, to_dev(np.asarray(idx, np.int32)), to_dev(pl))
        batch[...] = b_t.cpu().numpy()
        return int(err.item()), ln.cpu().numpy(), pd.cpu().numpy(), int(w.item())

    def realign(kv, ln, pad, ne):
        kv_t = torch.from_numpy(kv).to(dev())
        l2, p2, w2, err = sv.spec_realign_kv(kv_t, to_dev(ln), to_dev(pad), to_dev(ne))
        kv[...] = kv_t.cpu().numpy()
        return int(err.item()), l2.cpu().numpy(), p2.cpu().numpy(), int(w2.item())

    def unpad(batch, pool, idx, ln, pad, pl, ne=None):
        p_t, b_t = torch.from_numpy(pool).to(dev()), torch.from_numpy(batch).to(dev())
        g = to_dev(pl.copy())
        err = sv.spec_unpad_scatter(b_t, p_t, to_dev(np.asarray(idx, np.int32)), to_dev(ln), to_dev(pad), g,
                                    n_emit=None if ne is None else to_dev(np.asarray(ne, np.int32)))
        pool[...] = p_t.cpu().numpy()
        pl[...] = g.cpu().numpy()
        return int(err.item())

    return dict(group=group, verify=verify, commit=commit, repad=repad, realign=realign, unpad=unpad)


def oracle_ops():
    return dict(group=lambda lens, B: oracle.group_by_length(lens, B),
                verify=lambda x, d, rem, eos: oracle.verify_greedy(x, DT_F32, d, None, eos, rem),
                commit=oracle.commit_ragged, repad=oracle.repad_gather, realign=oracle.realign_kv,
                unpad=lambda b, p, i, ln, pad, pl, ne=None: oracle.unpad_scatter(
                    b, p, i, ln if ne is None else np.asarray(ln, np.int32) + ne, pad, pl))


@pytest.mark.parametrize("N,B,window,k,alpha,n_new,eos,lens", [
    (8, 2, 4, 2, 0.7, 12, -1, [3, 3, 5, 2, 5, 3, 4, 6]),
    (10, 3, 6, 3, 0.5, 14, -1, [4, 4, 4, 2, 7, 7, 1, 5, 5, 3]),
    (6, 2, 2, 2, 0.9, 10, 4, [2, 5, 5, 3, 2, 6]),
])
@pytest.mark.parametrize("fallback_realign", [True, False])
def test_exspec_on_device_equals_single_sequence_greedy(N, B, window, k, alpha, n_new, eos, lens, fallback_realign):
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=alpha, seed=N * 7 + B)
    rng = np.random.default_rng(N + B)
    prompts = [list(rng.integers(0, 11, size=n)) for n in lens]
    S = max(lens) + n_new + 2 * (k + 1) + 8
    a, b = {}, {}
    gen, rounds, grouped = run_exspec(pair, prompts, n_new, k, S, B, window, device_ops(), eos_id=eos,
                                      fallback_realign=fallback_realign, result=a)
    for n in range(N):
        assert gen[n] == pair.ref_generate(n, prompts[n], n_new, eos_id=eos), n
    # and the same rounds and the same final pool as the oracle's run (which realigns)
    _, r2, g2 = run_exspec(pair, prompts, n_new, k, S, B, window, oracle_ops(), eos_id=eos, result=b)
    assert (rounds, grouped) == (r2, g2)
    assert np.array_equal(a["pool"].view(np.uint32), b["pool"].view(np.uint32))
    assert np.array_equal(a["pool_len"], b["pool_len"])


def test_unpad_with_commits_matches_oracle_and_refuses_negative_counts():
    rng = np.random.default_rng(41)
    L, N, H, S, D, B = 2, 30, 2, 200, 16, 7
    pool = rng.standard_normal((L, 2, N, H, S, D)).astype(np.float32)
    batch = rng.standard_normal((L, 2, B, H, S, D)).astype(np.float32)
    idx = rng.choice(N, size=B, replace=False).astype(np.int32)
    ln = rng.integers(1, 120, size=B).astype(np.int32)
    pad = (int(ln.max()) - ln).astype(np.int32)
    ne = rng.integers(0, 6, size=B).astype(np.int32)
    pl = rng.integers(1, 150, size=N).astype(np.int32)
    pool_t, pl_t = torch.from_numpy(pool.copy()).to(dev()), to_dev(pl.copy())
    err = sv.spec_unpad_scatter(torch.from_numpy(batch).to(dev()), pool_t, to_dev(idx), to_dev(ln), to_dev(pad),
                                pl_t, n_emit=to_dev(ne))
    ref_pl = pl.copy()
    assert oracle.unpad_scatter(batch, pool, idx, ln + ne, pad, ref_pl) == 0 and int(err.item()) == 0
    assert np.array_equal(pool_t.cpu().numpy(), pool) and np.array_equal(pl_t.cpu().numpy(), ref_pl)
    bad = ne.copy()
    bad[3] = -1
    err = sv.spec_unpad_scatter(torch.from_numpy(batch).to(dev()), pool_t, to_dev(idx), to_dev(ln), to_dev(pad),
                                pl_t, n_emit=to_dev(bad))
    assert int(err.item()) == sv.REALIGN_LAYOUT and np.array_equal(pool_t.cpu().numpy(), pool)


@pytest.mark.parametrize("N,B,window,vals", [(512, 64, 512, 8), (512, 64, 96, 8), (300, 16, 40, 900),
                                            (50, 64, 50, 4), (20, 4, 1, 3)])
def test_scheduler_selection_matches_oracle_policy(N, B, window, vals):
    """ExspecScheduler (window mask + spec_group_by_length over the pool)
    picks the same sequences, in the same order, as the oracle's policy
    (group over the window's lengths, mapped back to pool indices)."""
    from oracle.toy import exspec_select
    from speculative_decoding_verification_28_gb300.exspec import ExspecScheduler

    rng = np.random.default_rng(N + window)
    for trial in range(6):
        lens = (128 * rng.integers(1, vals + 1, size=N)).astype(np.int32)
        active = rng.random(N) < (0.9 if trial % 2 else 0.5)
        pl = to_dev(lens)
        sched = ExspecScheduler(pl, B, window)
        sched.select_async(active)
        torch.cuda.synchronize()
        picks, full, _ = sched.selection()
        want, want_full = exspec_select(lens, active, window, B, lambda ln, b: oracle.group_by_length(ln, b))
        assert list(picks) == list(want) and full == want_full
