"""Realignment, position IDs and masks: CUDA path vs the CPU oracle.

Bit-exact over the WHOLE cache buffer for the small and medium cases (both
sides write exactly the destination runs; every other byte, including stale
and padding slots, must be unchanged).  At full size the oracle checks a
random sample of slabs bit for bit (the shift of a slab depends only on its
sequence), and the invariant checker runs over every slab on the device.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import dev, to_dev
from specgen import CONFIGS, prompt_lengths
from specgen import torch_gen

pytestmark = pytest.mark.gpu


def run_round(kv_t, ln, pad, n, **kw):
    ln2, pd2, w2, err = sv.spec_realign_kv(kv_t, to_dev(ln), to_dev(pad), to_dev(n), **kw)
    return ln2.cpu().numpy(), pd2.cpu().numpy(), int(w2.item()), int(err.item())


def random_state(B, S, k, lo, hi, seed):
    ln = prompt_lengths(B, lo, hi, seed)
    W = int(ln.max())
    assert W + k <= S
    return ln, (W - ln).astype(np.int32)


@pytest.mark.parametrize("dtype,D", [(np.float32, 64), (np.float32, 3), (np.float16, 5), (np.float16, 8),
                                     (np.float32, 4)])
def test_whole_buffer_rounds(dtype, D):
    """Several chained rounds on a small cache (bulk path for 16-byte rows,
    plain path otherwise), commit counts spanning both shift directions."""
    rng = np.random.default_rng(D)
    L, B, H, S, k = 2, 7, 3, 160, 5
    kv = rng.standard_normal((L, 2, B, H, S, D)).astype(dtype)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln, pad = random_state(B, S, k, 1, 40, seed=D)
    for r in range(12):
        W = int(ln[0] + pad[0])
        n = rng.integers(0, k + 2, size=B).astype(np.int32)
        if W + int(n.max()) > S or W + k + 1 > S:
            break
        g_ln, g_pd, g_w, g_err = run_round(kv_t, ln, pad, n)
        st, o_ln, o_pd, o_w = oracle.realign_kv(kv, ln, pad, n)
        assert st == 0 and g_err == 0
        assert np.array_equal(g_ln, o_ln) and np.array_equal(g_pd, o_pd) and g_w == o_w
        assert np.array_equal(kv_t.cpu().numpy(), kv), f"round {r}"
        ln, pad = o_ln, o_pd


def test_config1_full():
    c = CONFIGS["c1"]
    rng = np.random.default_rng(1001)
    kv = rng.standard_normal((c["L"], 2, c["B"], c["H"], c["S"], c["D"])).astype(np.float32)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln, pad = random_state(c["B"], c["S"], c["k"], *c["prompt"], seed=1001)
    for r in range(c["rounds"]):
        n = rng.integers(1, c["k"] + 2, size=c["B"]).astype(np.int32)
        if int(ln[0] + pad[0]) + c["k"] + 1 > c["S"]:
            break
        g = run_round(kv_t, ln, pad, n)
        st, o_ln, o_pd, o_w = oracle.realign_kv(kv, ln, pad, n)
        assert st == 0 and g[3] == 0 and np.array_equal(g[1], o_pd)
        assert np.array_equal(kv_t.cpu().numpy(), kv)
        ln, pad = o_ln, o_pd


def test_long_runs_small_shifts():
    """Runs of many bulk tiles moved by one row either way: every tile's
    destination overlaps the neighbouring tile's source."""
    L, B, H, S, D = 1, 3, 2, 4096, 128
    rng = np.random.default_rng(3)
    kv = rng.integers(0, 65535, size=(L, 2, B, H, S, D), dtype=np.uint16).view(np.float16)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln = np.array([3000, 2999, 2998], np.int32)
    pad = np.array([0, 1, 2], np.int32)
    for n in ([1, 3, 5], [5, 2, 1], [2, 2, 2], [0, 1, 3]):
        n = np.array(n, np.int32)
        g = run_round(kv_t, ln, pad, n)
        st, o_ln, o_pd, o_w = oracle.realign_kv(kv, ln, pad, n)
        assert st == 0 and g[3] == 0
        assert np.array_equal(kv_t.cpu().numpy().view(np.uint16), kv.view(np.uint16))
        ln, pad = o_ln, o_pd


def test_noop_cases_write_nothing():
    L, B, H, S, D = 2, 5, 2, 64, 16
    rng = np.random.default_rng(4)
    kv = rng.standard_normal((L, 2, B, H, S, D)).astype(np.float32)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln, pad = random_state(B, S, 4, 3, 20, seed=4)
    g = run_round(kv_t, ln, pad, np.full(B, 3, np.int32))  # uniform acceptance
    assert g[3] == 0 and np.array_equal(g[1], pad)
    assert np.array_equal(kv_t.cpu().numpy(), kv)
    kv1 = rng.standard_normal((L, 2, 1, H, S, D)).astype(np.float32)
    kv1_t = torch.from_numpy(kv1.copy()).to(dev())
    g = run_round(kv1_t, np.array([9], np.int32), np.array([0], np.int32), np.array([4], np.int32))
    assert g[3] == 0 and g[1][0] == 0 and np.array_equal(kv1_t.cpu().numpy(), kv1)


def test_errors_leave_state_untouched():
    L, B, H, S, D = 1, 3, 2, 32, 8
    kv = np.arange(L * 2 * B * H * S * D, dtype=np.float32).reshape(L, 2, B, H, S, D)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln = np.array([10, 7, 9], np.int32)
    pad = np.array([0, 3, 1], np.int32)
    sentinel = torch.full((B,), -7, dtype=torch.int32, device=dev())
    cases = [
        (ln, pad, [1, 30, 1], sv.REALIGN_EMIT),       # run would pass S: W + 30 - 1 > 32
        (ln, pad, [-1, 1, 1], sv.REALIGN_EMIT),
        (ln, np.array([0, 2, 1], np.int32), [1, 1, 1], sv.REALIGN_LAYOUT),  # pad + len not constant
        (ln - 1, pad + 1, [1, 1, 1], sv.REALIGN_LAYOUT),  # no sequence without padding
        (np.array([20, 17, 19], np.int32), pad, [13, 9, 9], sv.REALIGN_CAPACITY),  # W' = 33 > 32
    ]
    for l_, p_, n_, want in cases:
        ln_new, pd_new = sentinel.clone(), sentinel.clone()
        w = torch.full((1,), -7, dtype=torch.int32, device=dev())
        _, _, _, err = sv.spec_realign_kv(kv_t, to_dev(l_), to_dev(p_), to_dev(np.array(n_, np.int32)),
                                          len_new=ln_new, pad_new=pd_new, width_new=w)
        assert int(err.item()) == want
        assert (ln_new == -7).all() and (pd_new == -7).all() and int(w.item()) == -7
        assert np.array_equal(kv_t.cpu().numpy(), kv)


def test_outputs_may_alias_inputs():
    L, B, H, S, D = 1, 4, 2, 64, 8
    rng = np.random.default_rng(5)
    kv = rng.standard_normal((L, 2, B, H, S, D)).astype(np.float32)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln = np.array([10, 7, 9, 4], np.int32)
    pad = (10 - ln).astype(np.int32)
    n = np.array([1, 5, 2, 3], np.int32)
    ln_t, pad_t = to_dev(ln), to_dev(pad)
    sv.spec_realign_kv(kv_t, ln_t, pad_t, to_dev(n), len_new=ln_t, pad_new=pad_t)
    st, o_ln, o_pd, o_w = oracle.realign_kv(kv, ln, pad, n)
    assert np.array_equal(ln_t.cpu().numpy(), o_ln) and np.array_equal(pad_t.cpu().numpy(), o_pd)
    assert np.array_equal(kv_t.cpu().numpy(), kv)


def _full_size_rounds(name, alpha, rounds, sample_slabs):
    """Full-size cache on the device: the synthetic forward writes the query
    slots, greedy verification decides the commits, realignment runs; after
    every round the invariant checker scans the whole cache and the oracle
    checks sampled slabs bit for bit."""
    c = CONFIGS[name]
    L, B, H, S, D, V = c["L"], c["B"], c["H"], c["S"], c["D"], c["V"]
    k = c["k"] if "k" in c else max(c["ks"])
    g = torch.Generator(device=dev()).manual_seed(2000 + int(alpha * 10))
    rng = np.random.default_rng(2000)
    ln = prompt_lengths(B, *(c["prompt"] if "prompt" in c else c["pool_len"]), seed=2000 + B)
    W = int(ln.max())
    pad = (W - ln).astype(np.int32)
    kv = torch.empty((L, 2, B, H, S, D), dtype=torch.bfloat16, device=dev())
    tokens = torch.randint(0, V, (B, S), device=dev(), dtype=torch.int32, generator=g)
    ln_t, pad_t = to_dev(ln), to_dev(pad)
    torch_gen.kv_fill(kv, tokens, pad_t, ln_t - 1, junk=True)
    pos = torch.empty((B, S), dtype=torch.int32, device=dev())
    mask = torch.empty((B, S), dtype=torch.uint8, device=dev())
    sv.spec_rebuild_pos_mask(pad_t, pos, mask)
    for r in range(rounds):
        W = int(ln[0] + pad[0])
        if W + k + 1 > S:
            break
        x, d = torch_gen.greedy_round_inputs(B, k, V, alpha, c["sigma"], g, torch.bfloat16, dev())
        qtok = torch.cat([tokens[torch.arange(B, device=dev()), ln_t.long() - 1].unsqueeze(1), d], dim=1)
        torch_gen.kv_write_query(kv, qtok.contiguous(), pos, W)
        out, na, ne = sv.spec_verify_greedy(x, d)
        # sampled slabs before the shift
        slabs = [(int(rng.integers(L)), int(rng.integers(2)), int(rng.integers(B)), int(rng.integers(H)))
                 for _ in range(sample_slabs)]
        before = [kv[l_, c_, b_, h_].view(torch.int16).cpu().numpy().view(np.uint8).copy()
                  for l_, c_, b_, h_ in slabs]
        ln_new, pad_new, w_new, err = sv.spec_realign_kv(kv, ln_t, pad_t, ne)
        assert int(err.item()) == 0
        ne_h = ne.cpu().numpy()
        st, o_ln, o_pd, o_w = oracle.realign_plan(S, ln, pad, ne_h)
        assert st == 0 and np.array_equal(ln_new.cpu().numpy(), o_ln) and np.array_equal(pad_new.cpu().numpy(), o_pd)
        for (l_, c_, b_, h_), slab in zip(slabs, before):
            oracle.shift_slab(slab, D * 2, int(pad[b_]), int(o_pd[b_]), int(o_ln[b_]) - 1)
            got = kv[l_, c_, b_, h_].view(torch.int16).cpu().numpy().view(np.uint8)
            assert np.array_equal(got, slab), (r, l_, c_, b_, h_)
        # token history: the committed tokens follow the old length
        out_h = out.cpu().numpy()
        tok_h = tokens.cpu().numpy()
        for b in range(B):
            tok_h[b, ln[b]: ln[b] + ne_h[b]] = out_h[b, : ne_h[b]]
        tokens = to_dev(tok_h)
        sv.spec_rebuild_pos_mask(pad_new, pos, mask, pad_old=pad_t)
        assert torch_gen.kv_check(kv, tokens, pad_new, ln_new) == 0
        ln, pad = o_ln, o_pd
        ln_t, pad_t = ln_new, pad_new
    p_o, m_o = oracle.rebuild_pos_mask(S, pad)
    assert np.array_equal(pos.cpu().numpy(), p_o) and np.array_equal(mask.cpu().numpy(), m_o)


@pytest.mark.parametrize("alpha", [0.5, 0.8])
def test_config2_full_size(alpha):
    _full_size_rounds("c2", alpha, rounds=6, sample_slabs=24)


def test_config3_full_size():
    """8 GiB cache (32 x 2 x 32 x 8 x 2048 x 128 bf16); the commits come from
    greedy verification at alpha 0.8 (the realignment does not depend on how
    n_emit was decided)."""
    _full_size_rounds("c3", 0.8, rounds=5, sample_slabs=24)


def test_config4_full_size_batch():
    """A 64-sequence batch of config 4's cache (28 x 2 x 64 x 4 x 2048 x 128
    bf16, 7 GiB), k = 8, lengths U[128, 1024]."""
    _full_size_rounds("c4", 0.7, rounds=5, sample_slabs=24)


def test_config5_full_size():
    """128 GiB cache (32 x 2 x 256 x 8 x 4096 x 128 bf16); skipped when the
    device cannot hold it."""
    free, _ = torch.cuda.mem_get_info()
    if free < 150 * 2**30:
        pytest.skip("needs ~140 GB of free device memory")
    _full_size_rounds("c5", 0.6, rounds=3, sample_slabs=16)


@pytest.mark.parametrize("S,offset", [(4096, 0), (1000, 0), (37, 0), (256, 1)])
def test_pos_mask(S, offset):
    rng = np.random.default_rng(S)
    B = 33
    pad_old = rng.integers(0, min(S, 50), size=B).astype(np.int32)
    pad_new = pad_old.copy()
    pad_new[::3] = rng.integers(0, min(S, 50), size=len(pad_new[::3]))
    p0, m0 = oracle.rebuild_pos_mask(S, pad_old)
    pos_buf = torch.zeros(B * S + offset, dtype=torch.int32, device=dev())
    pos = pos_buf[offset:].view(B, S)  # offset 1: unaligned rows take the plain path
    pos.copy_(torch.from_numpy(p0))
    mask = to_dev(m0.copy())
    sv.spec_rebuild_pos_mask(to_dev(pad_new), pos, mask, pad_old=to_dev(pad_old))
    p1, m1 = oracle.rebuild_pos_mask(S, pad_new)
    assert np.array_equal(pos.cpu().numpy(), p1) and np.array_equal(mask.cpu().numpy(), m1)
    # without pad_old every row is rewritten, from garbage
    pos.fill_(-5)
    mask.fill_(9)
    sv.spec_rebuild_pos_mask(to_dev(pad_new), pos, mask)
    assert np.array_equal(pos.cpu().numpy(), p1) and np.array_equal(mask.cpu().numpy(), m1)


# -- several caches by one plan (target + draft) ----------------------------------

def test_multi_cache_matches_oracle_per_cache():
    """Target (bf16, 16-byte rows: bulk path), draft (fp16, 128-byte rows) and an
    odd cache (fp32, 12-byte rows: plain path) moved by one plan, several
    chained rounds; each buffer bit-exact against the oracle's realignment."""
    rng = np.random.default_rng(31)
    B, S, k = 6, 200, 5
    shapes = [(2, 4, 128, np.float16), (1, 3, 64, np.float16), (2, 2, 3, np.float32)]
    host = [rng.standard_normal((L, 2, B, H, S, D)).astype(dt) for L, H, D, dt in shapes]
    dev_t = [torch.from_numpy(h.copy()).to(dev()) for h in host]
    dev_t[0] = dev_t[0].view(torch.bfloat16)  # bf16 storage of the same bytes
    ln, pad = random_state(B, S, k, 1, 60, seed=31)
    for r in range(10):
        W = int(ln[0] + pad[0])
        if W + k + 2 > S:
            break
        n = rng.integers(0, k + 2, size=B).astype(np.int32)
        ln2, pd2, w2, err = sv.spec_realign_kv_multi(dev_t, to_dev(ln), to_dev(pad), to_dev(n))
        assert int(err.item()) == 0
        for h in host:
            st, o_ln, o_pd, o_w = oracle.realign_kv(h.view(np.uint16) if h.dtype == np.float16 else h, ln, pad, n)
            assert st == 0
        assert np.array_equal(ln2.cpu().numpy(), o_ln) and np.array_equal(pd2.cpu().numpy(), o_pd)
        assert int(w2.item()) == o_w
        assert np.array_equal(dev_t[0].view(torch.int16).cpu().numpy().view(np.float16), host[0])
        assert np.array_equal(dev_t[1].cpu().numpy(), host[1])
        assert np.array_equal(dev_t[2].cpu().numpy(), host[2])
        ln, pad = o_ln, o_pd


def test_draft_cache_follows_the_accepted_prefix():
    """The draft cache holds KV for the last token and proposals 0..k-2 (what
    the drafter consumed); after the shared realignment every position below
    len' - 1 holds the draft's entry for the committed history, except the
    row of proposal k-1 when all k proposals were accepted, which the drafter
    never computed."""
    from specgen import kv_row_values

    rng = np.random.default_rng(5)
    B, S, k, L, H, D = 5, 64, 4, 1, 2, 8
    lens = np.array([9, 4, 12, 7, 12], np.int32)
    W = int(lens.max())
    pad = (W - lens).astype(np.int32)
    toks = [list(rng.integers(0, 99, size=lens[b])) for b in range(B)]
    props = rng.integers(0, 99, size=(B, k))
    DRAFT = 1000  # the draft's KV values: f of a shifted sequence id
    kv_t = np.zeros((L, 2, B, H, S, D), np.float32)
    kv_d = np.full((L, 2, B, H, S, D), 7.0, np.float32)  # 7.0: never written by the drafter
    for b in range(B):
        for p in range(lens[b] - 1):
            kv_t[:, :, b, :, pad[b] + p, :] = kv_row_values(b, toks[b][p], p, L, H, D)
            kv_d[:, :, b, :, pad[b] + p, :] = kv_row_values(DRAFT + b, toks[b][p], p, L, H, D)
        q = [toks[b][-1]] + list(props[b])
        for j, t in enumerate(q):
            kv_t[:, :, b, :, W - 1 + j, :] = kv_row_values(b, int(t), lens[b] - 1 + j, L, H, D)
            if j < k:  # the drafter consumed the last token and proposals 0..k-2
                kv_d[:, :, b, :, W - 1 + j, :] = kv_row_values(DRAFT + b, int(t), lens[b] - 1 + j, L, H, D)
    n = np.array([k + 1, 1, 3, k + 1, 0], np.int32)
    t_dev, d_dev = torch.from_numpy(kv_t).to(dev()), torch.from_numpy(kv_d).to(dev())
    ln2, pd2, w2, err = sv.spec_realign_kv_multi([t_dev, d_dev], to_dev(lens), to_dev(pad), to_dev(n))
    assert int(err.item()) == 0
    ln2, pd2 = ln2.cpu().numpy(), pd2.cpu().numpy()
    got_d = d_dev.cpu().numpy()
    for b in range(B):
        hist = list(toks[b]) + list(props[b][: max(n[b] - 1, 0)])
        for p in range(ln2[b] - 1):
            row = got_d[:, :, b, :, pd2[b] + p, :]
            if n[b] == k + 1 and p == lens[b] - 1 + k:
                assert (row == 7.0).all()  # proposal k-1: no draft KV yet
            else:
                assert np.array_equal(row, kv_row_values(DRAFT + b, int(hist[p]), p, L, H, D)), (b, p)
    # and the target cache satisfies I2 everywhere
    got_t = t_dev.cpu().numpy()
    for b in range(B):
        hist = list(toks[b]) + list(props[b][: max(n[b] - 1, 0)])
        for p in range(ln2[b] - 1):
            assert np.array_equal(got_t[:, :, b, :, pd2[b] + p, :], kv_row_values(b, int(hist[p]), p, L, H, D))
