"""One whole round per call (spec_round_greedy / spec_round_sample): the
fused entry points against the oracle (greedy: verification, the
realignment of every cache byte for byte, positions and mask) and against
the separate entry points (stochastic, which are themselves checked against
the oracle in test_gpu_verify_sample.py / test_gpu_verify_filter.py)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import dev, logits_to_dev, to_dev
from specgen import greedy_round_inputs, prompt_lengths, sample_round_inputs

pytestmark = pytest.mark.gpu


def _state(B, S, k, seed):
    ln = prompt_lengths(B, 4, 60, seed)
    W = int(ln.max())
    assert W + k + 1 <= S
    return ln, (W - ln).astype(np.int32)


@pytest.mark.parametrize("two_caches", [False, True])
def test_greedy_round_equals_oracle_over_chained_rounds(two_caches):
    rng = np.random.default_rng(7 + two_caches)
    B, k, V, S = 9, 4, 3000, 128
    kv = rng.integers(0, 65535, size=(2, 2, B, 3, S, 16), dtype=np.uint16).view(np.float16)
    dkv = rng.standard_normal((1, 2, B, 2, S, 8)).astype(np.float32)
    kv_t, dkv_t = torch.from_numpy(kv.copy()).to(dev()), torch.from_numpy(dkv.copy()).to(dev())
    caches = [kv_t, dkv_t] if two_caches else [kv_t]
    ln, pad = _state(B, S, k, seed=11)
    pos = torch.zeros((B, S), dtype=torch.int32, device=dev())
    mask = torch.zeros((B, S), dtype=torch.uint8, device=dev())
    opos, omask = oracle.rebuild_pos_mask(S, pad)
    pos.copy_(torch.from_numpy(opos))
    mask.copy_(torch.from_numpy(omask))
    for r in range(10):
        if int(ln[0] + pad[0]) + k + 1 > S:
            break
        x, d = greedy_round_inputs(B, k, V, 0.6, 1.0, seed=100 + r, dtype="f32")
        o_out, o_na, o_ne = oracle.verify_greedy(x, oracle.DT_F32, d)
        out, na, ne, ln2, pd2, w2, err = sv.spec_round_greedy(to_dev(x), to_dev(d), caches, to_dev(ln), to_dev(pad),
                                                              pos, mask)
        st, o_ln, o_pd, o_w = oracle.realign_kv(kv, ln, pad, o_ne)
        if two_caches:
            st2, _, _, _ = oracle.realign_kv(dkv, ln, pad, o_ne)
            assert st2 == 0
        oracle.rebuild_pos_mask(S, o_pd, opos, omask)
        assert st == 0 and int(err.item()) == 0
        assert np.array_equal(out.cpu().numpy(), o_out) and np.array_equal(na.cpu().numpy(), o_na)
        assert np.array_equal(ne.cpu().numpy(), o_ne)
        assert np.array_equal(ln2.cpu().numpy(), o_ln) and np.array_equal(pd2.cpu().numpy(), o_pd)
        assert int(w2.item()) == o_w
        assert np.array_equal(kv_t.cpu().numpy().view(np.uint16), kv.view(np.uint16)), r
        if two_caches:
            assert np.array_equal(dkv_t.cpu().numpy(), dkv), r
        assert np.array_equal(pos.cpu().numpy(), opos) and np.array_equal(mask.cpu().numpy(), omask)
        ln, pad = o_ln, o_pd


@pytest.mark.parametrize("filtered", [False, True])
def test_sample_round_equals_separate_calls(filtered):
    rng = np.random.default_rng(3 + filtered)
    B, k, V, S = 12, 3, 5000, 96
    kv = rng.standard_normal((2, 2, B, 2, S, 8)).astype(np.float32)
    kv_a, kv_b = torch.from_numpy(kv.copy()).to(dev()), torch.from_numpy(kv.copy()).to(dev())
    ln, pad = _state(B, S, k, seed=5)
    x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=9, dtype="bf16")
    xt, qt, dt_, ut = logits_to_dev(x, oracle.DT_BF16), to_dev(q), to_dev(d), to_dev(u)
    tk = to_dev(rng.integers(0, 60, size=B).astype(np.int32)) if filtered else None
    tp = to_dev(rng.choice([0.5, 0.9, 1.0], size=B).astype(np.float32)) if filtered else None
    pos_a = torch.zeros((B, S), dtype=torch.int32, device=dev())
    mask_a = torch.zeros((B, S), dtype=torch.uint8, device=dev())
    pos_b, mask_b = pos_a.clone(), mask_a.clone()
    res = torch.empty((B, V), dtype=torch.float32, device=dev())
    g = sv.spec_round_sample(xt, qt, dt_, ut, [kv_a], to_dev(ln), to_dev(pad), pos_a, mask_a, top_k=tk, top_p=tp,
                             out_residual=res)
    if filtered:
        s = sv.spec_verify_sample_filtered(xt, qt, dt_, ut, top_k=tk, top_p=tp, want_residual=True)
    else:
        s = sv.spec_verify_sample(xt, qt, dt_, ut, want_residual=True)
    ln2, pd2, w2, err = sv.spec_realign_kv(kv_b, to_dev(ln), to_dev(pad), s[2])
    sv.spec_rebuild_pos_mask(pd2, pos_b, mask_b, pad_old=to_dev(pad))
    for a, b in zip(g[:3], s[:3]):
        assert torch.equal(a, b)
    assert torch.equal(g[7], s[3]) and torch.equal(g[8], s[4])
    assert torch.equal(g[3], ln2) and torch.equal(g[4], pd2) and torch.equal(g[5], w2) and int(g[6].item()) == 0
    assert torch.equal(kv_a, kv_b) and torch.equal(pos_a, pos_b) and torch.equal(mask_a, mask_b)


def test_round_rejects_aliased_padding_and_launches_nothing():
    B, k, V, S = 4, 2, 100, 32
    x, d = greedy_round_inputs(B, k, V, 0.5, 1.0, seed=1, dtype="f32")
    kv = torch.zeros((1, 2, B, 1, S, 8), dtype=torch.float32, device=dev())
    ln = to_dev(np.full(B, 5, np.int32))
    pad = to_dev(np.zeros(B, np.int32))
    pos = torch.zeros((B, S), dtype=torch.int32, device=dev())
    mask = torch.zeros((B, S), dtype=torch.uint8, device=dev())
    out = torch.full((B, k + 1), -9, dtype=torch.int32, device=dev())
    with pytest.raises(sv.SpecError):
        sv.spec_round_greedy(to_dev(x), to_dev(d), [kv], ln, pad, pos, mask, out_tokens=out, pad_new=pad)
    torch.cuda.synchronize()
    assert (out == -9).all()


def test_round_replayed_from_a_cuda_graph_equals_oracle():
    """spec_round_greedy captured once per buffer parity (RoundGraph) and
    replayed over chained rounds: same results as the oracle, byte for byte."""
    rng = np.random.default_rng(17)
    B, k, V, S = 8, 3, 2000, 96
    kv = rng.standard_normal((2, 2, B, 2, S, 16)).astype(np.float32)
    kv_t = torch.from_numpy(kv.copy()).to(dev())
    ln, pad = _state(B, S, k, seed=21)
    pos = torch.from_numpy(oracle.rebuild_pos_mask(S, pad)[0]).to(dev())
    mask = torch.from_numpy(oracle.rebuild_pos_mask(S, pad)[1]).to(dev())
    opos, omask = oracle.rebuild_pos_mask(S, pad)
    x_d = torch.empty((B, k + 1, V), dtype=torch.float32, device=dev())
    d_d = torch.empty((B, k), dtype=torch.int32, device=dev())
    blocks = [torch.empty(B * (k + 1) + 4 * B + 2, dtype=torch.int32, device=dev()) for _ in range(2)]
    ws = sv.Workspace(B, k, V, dev())

    def views(blk):
        o = B * (k + 1)
        return (blk[:o].view(B, k + 1), blk[o:o + B], blk[o + B:o + 2 * B], blk[o + 2 * B:o + 3 * B],
                blk[o + 3 * B:o + 4 * B], blk[o + 4 * B:o + 4 * B + 1], blk[o + 4 * B + 1:])

    def enqueue(par):
        out, na, ne, _, _, w, err = views(blocks[1 - par])
        _, _, _, ln_in, pad_in, _, _ = views(blocks[par])
        _, _, _, ln_out, pad_out, _, _ = views(blocks[1 - par])
        sv.spec_round_greedy(x_d, d_d, [kv_t], ln_in, pad_in, pos, mask, out_tokens=out, n_accept=na, n_emit=ne,
                             len_new=ln_out, pad_new=pad_out, width_new=w, err=err, workspace=ws)

    graphs = [sv.RoundGraph(lambda p=p: enqueue(p), dev()) for p in (0, 1)]
    views(blocks[0])[3].copy_(to_dev(ln))
    views(blocks[0])[4].copy_(to_dev(pad))
    cur = 0
    for r in range(8):
        if int(ln[0] + pad[0]) + k + 1 > S:
            break
        x, d = greedy_round_inputs(B, k, V, 0.6, 1.0, seed=300 + r, dtype="f32")
        x_d.copy_(torch.from_numpy(x))
        d_d.copy_(torch.from_numpy(d))
        graphs[cur].replay()
        torch.cuda.synchronize()
        out, na, ne, ln2, pd2, w2, err = (t.cpu().numpy() for t in views(blocks[1 - cur]))
        o_out, o_na, o_ne = oracle.verify_greedy(x, oracle.DT_F32, d)
        st, o_ln, o_pd, o_w = oracle.realign_kv(kv, ln, pad, o_ne)
        oracle.rebuild_pos_mask(S, o_pd, opos, omask)
        assert st == 0 and int(err[0]) == 0
        assert np.array_equal(out, o_out) and np.array_equal(na, o_na) and np.array_equal(ne, o_ne)
        assert np.array_equal(ln2, o_ln) and np.array_equal(pd2, o_pd) and int(w2[0]) == o_w
        assert np.array_equal(kv_t.cpu().numpy(), kv), r
        assert np.array_equal(pos.cpu().numpy(), opos) and np.array_equal(mask.cpu().numpy(), omask)
        ln, pad = o_ln, o_pd
        cur = 1 - cur


@pytest.mark.parametrize("filtered", [False, True])
def test_sample_round_replayed_from_a_cuda_graph_equals_direct_calls(filtered):
    """spec_round_sample captured once per buffer parity (RoundGraph: the
    statistics or filter kernel, the two programmatically launched draw
    kernels, the realignment and the positions / mask) and replayed over
    chained rounds gives, round after round, exactly what direct calls give
    on a twin state: tokens, counts, lengths, paddings, width, flags, cache,
    positions and mask."""
    rng = np.random.default_rng(23 + filtered)
    B, k, V, S = 8, 3, 3000, 128
    kv = rng.standard_normal((2, 2, B, 2, S, 16)).astype(np.float32)
    kv_g, kv_e = torch.from_numpy(kv.copy()).to(dev()), torch.from_numpy(kv.copy()).to(dev())
    ln, pad = _state(B, S, k, seed=29)
    p0, m0 = oracle.rebuild_pos_mask(S, pad)
    pos_g, mask_g = torch.from_numpy(p0).to(dev()), torch.from_numpy(m0).to(dev())
    pos_e, mask_e = pos_g.clone(), mask_g.clone()
    x_d = torch.empty((B, k + 1, V), dtype=torch.bfloat16, device=dev())
    q_d = torch.empty((B, k, V), dtype=torch.float32, device=dev())
    d_d = torch.empty((B, k), dtype=torch.int32, device=dev())
    u_d = torch.empty((B, k + 1), dtype=torch.float32, device=dev())
    tk = to_dev(rng.integers(0, 40, size=B).astype(np.int32)) if filtered else None
    tp = to_dev(rng.choice([0.6, 0.9, 1.0], size=B).astype(np.float32)) if filtered else None
    n = B * (k + 1) + 5 * B + 2
    blocks = [torch.zeros(n, dtype=torch.int32, device=dev()) for _ in range(2)]
    ws = sv.Workspace(B, k, V, dev())

    def views(blk):
        o = B * (k + 1)
        return (blk[:o].view(B, k + 1), blk[o:o + B], blk[o + B:o + 2 * B], blk[o + 2 * B:o + 3 * B],
                blk[o + 3 * B:o + 4 * B], blk[o + 4 * B:o + 4 * B + 1], blk[o + 4 * B + 1:o + 4 * B + 2],
                blk[o + 4 * B + 2:o + 5 * B + 2])

    def enqueue(par):
        out, na, ne, ln_out, pad_out, w, err, fl = views(blocks[1 - par])
        ln_in, pad_in = views(blocks[par])[3], views(blocks[par])[4]
        sv.spec_round_sample(x_d, q_d, d_d, u_d, [kv_g], ln_in, pad_in, pos_g, mask_g, top_k=tk, top_p=tp,
                             out_tokens=out, n_accept=na, n_emit=ne, flags=fl, len_new=ln_out, pad_new=pad_out,
                             width_new=w, err=err, workspace=ws)

    graphs = [sv.RoundGraph(lambda p=p: enqueue(p), dev()) for p in (0, 1)]
    views(blocks[0])[3].copy_(to_dev(ln))
    views(blocks[0])[4].copy_(to_dev(pad))
    ln_e, pad_e = to_dev(ln), to_dev(pad)
    cur, rounds = 0, 0
    for r in range(8):
        if int(views(blocks[cur])[3][0].item() + views(blocks[cur])[4][0].item()) + k + 1 > S:
            break
        x, q, d, u = sample_round_inputs(B, k, V, 0.5, seed=400 + r, dtype="bf16")
        x_d.copy_(logits_to_dev(x, oracle.DT_BF16))
        q_d.copy_(to_dev(q))
        d_d.copy_(to_dev(d))
        u_d.copy_(to_dev(u))
        graphs[cur].replay()
        e = sv.spec_round_sample(x_d, q_d, d_d, u_d, [kv_e], ln_e, pad_e, pos_e, mask_e, top_k=tk, top_p=tp)
        torch.cuda.synchronize()
        out, na, ne, ln2, pd2, w2, err, fl = views(blocks[1 - cur])
        assert torch.equal(out, e[0]) and torch.equal(na, e[1]) and torch.equal(ne, e[2]), r
        assert torch.equal(ln2, e[3]) and torch.equal(pd2, e[4]) and torch.equal(w2, e[5].view(1)), r
        assert int(err.item()) == 0 and int(e[6].item()) == 0
        assert torch.equal(fl, e[7].view(-1)), r
        assert torch.equal(kv_g, kv_e) and torch.equal(pos_g, pos_e) and torch.equal(mask_g, mask_e), r
        ln_e, pad_e = e[3].clone(), e[4].clone()
        cur = 1 - cur
        rounds += 1
    assert rounds >= 4


# ---------------------------------------------------------------------------
# work enqueued right after a round, with no host synchronisation
# ---------------------------------------------------------------------------
def _chain_without_host_sync(mode, via, seed):
    """Chained rounds on one stream with nothing waiting for the host.  After
    each round, at once: the committed tokens are written into the token
    table, a device kernel checks invariant I2 over the whole cache (slot
    pad'_b + p holds f(b, tok_p, p) for every p < len'_b - 1) and the round's
    error word is copied on the device; the next round's forward writes its
    query slots at the width the round left on the device.  Any of these
    running before the KV shift completed would see (or clobber) rows in
    flight.  Shapes: greedy = config 2's cache and logits (B=8, k=5,
    V=32000 bf16, alpha=0.8, KV 32x2x8x32x1024x128 bf16) with prompts
    U[64,256]; sample = config 3's (B=32, k=4, V=128256 fp32, KV
    32x2x32x8x2048x128 bf16) with prompts U[128,512], so that the width
    stays within the cache for every round of the chain."""
    from specgen import torch_gen

    d_ = dev()
    if mode == "greedy":
        B, k, V, L, H, S, D, lo, hi, ldt = 8, 5, 32000, 32, 32, 1024, 128, 64, 256, torch.bfloat16
    else:
        B, k, V, L, H, S, D, lo, hi, ldt = 32, 4, 128256, 32, 8, 2048, 128, 128, 512, torch.float32
    g = torch.Generator(device=d_).manual_seed(seed)
    kv = torch.empty((L, 2, B, H, S, D), dtype=torch.bfloat16, device=d_)
    tokens = torch.randint(0, V, (B, S), device=d_, dtype=torch.int32, generator=g)
    ln0 = prompt_lengths(B, lo, hi, seed)
    W0 = int(ln0.max())
    pad0 = (W0 - ln0).astype(np.int32)
    R = (S - W0 - (k + 1)) // (k + 1)  # the width grows by at most k + 1 per round
    lens = [to_dev(ln0), torch.empty(B, dtype=torch.int32, device=d_)]
    pads = [to_dev(pad0), torch.empty(B, dtype=torch.int32, device=d_)]
    widths = [torch.tensor([W0], dtype=torch.int32, device=d_), torch.empty(1, dtype=torch.int32, device=d_)]
    torch_gen.kv_fill(kv, tokens, pads[0], lens[0] - 1, junk=True)
    pos = torch.empty((B, S), dtype=torch.int32, device=d_)
    mask = torch.empty((B, S), dtype=torch.uint8, device=d_)
    sv.spec_rebuild_pos_mask(pads[0], pos, mask)
    x_d = torch.empty((B, k + 1, V), dtype=ldt, device=d_)
    d_d = torch.empty((B, k), dtype=torch.int32, device=d_)
    q_d = torch.empty((B, k, V), dtype=torch.float32, device=d_)
    u_d = torch.empty((B, k + 1), dtype=torch.float32, device=d_)
    out = torch.empty((B, k + 1), dtype=torch.int32, device=d_)
    na = torch.empty(B, dtype=torch.int32, device=d_)
    ne = torch.empty(B, dtype=torch.int32, device=d_)
    err = torch.empty(1, dtype=torch.int32, device=d_)
    ws = sv.Workspace(B, k, V, d_)
    bad = torch.zeros(1, dtype=torch.int64, device=d_)
    errs = torch.full((R,), -99, dtype=torch.int32, device=d_)
    ne_log = torch.zeros((R, B), dtype=torch.int32, device=d_)
    cols = torch.arange(k + 1, device=d_)

    def enqueue(par):
        ln_in, pad_in, ln_out, pad_out = lens[par], pads[par], lens[1 - par], pads[1 - par]
        w_out = widths[1 - par]
        if via == "calls":
            if mode == "greedy":
                sv.spec_verify_greedy(x_d, d_d, out_tokens=out, n_accept=na, n_emit=ne, workspace=ws)
            else:
                sv.spec_verify_sample(x_d, q_d, d_d, u_d, out_tokens=out, n_accept=na, n_emit=ne, workspace=ws)
            sv.spec_realign_kv(kv, ln_in, pad_in, ne, len_new=ln_out, pad_new=pad_out, width_new=w_out, err=err,
                               workspace=ws)
            sv.spec_rebuild_pos_mask(pad_out, pos, mask, pad_old=pad_in)
        elif mode == "greedy":
            sv.spec_round_greedy(x_d, d_d, [kv], ln_in, pad_in, pos, mask, out_tokens=out, n_accept=na, n_emit=ne,
                                 len_new=ln_out, pad_new=pad_out, width_new=w_out, err=err, workspace=ws)
        else:
            sv.spec_round_sample(x_d, q_d, d_d, u_d, [kv], ln_in, pad_in, pos, mask, out_tokens=out, n_accept=na,
                                 n_emit=ne, len_new=ln_out, pad_new=pad_out, width_new=w_out, err=err, workspace=ws)

    graphs = [sv.RoundGraph(lambda p=p: enqueue(p), d_) for p in (0, 1)] if via == "graph" else None
    torch.cuda.synchronize()
    cur = 0
    for r in range(R):
        if mode == "greedy":
            x, d = torch_gen.greedy_round_inputs(B, k, V, 0.8, 2.0, g, ldt, d_)
        else:
            x, q, d, u = torch_gen.sample_round_inputs(B, k, V, 0.5, g, ldt, d_)
            q_d.copy_(q)
            u_d.copy_(u)
        x_d.copy_(x)
        d_d.copy_(d)
        # the forward: KV of the last token and the k proposals at the width on the device
        last = torch.gather(tokens, 1, (lens[cur].long() - 1).unsqueeze(1))
        torch_gen.kv_write_query_dev(kv, torch.cat([last, d_d], 1).contiguous(), pos, widths[cur])
        if graphs is not None:
            graphs[cur].replay()
        else:
            enqueue(cur)
        # straight after the round, on the same stream: the token table, the I2 check, the error word
        at = (lens[cur].long().unsqueeze(1) + cols).clamp(max=S - 1)
        keep = cols.unsqueeze(0) < ne.unsqueeze(1)
        tokens.scatter_(1, at, torch.where(keep, out, torch.gather(tokens, 1, at)))
        torch_gen.kv_check_async(kv, tokens, pads[1 - cur], lens[1 - cur], bad)
        errs[r:r + 1].copy_(err)
        ne_log[r].copy_(ne)
        cur = 1 - cur
    torch.cuda.synchronize()
    assert R >= 100
    assert int(bad.item()) == 0
    assert (errs == 0).all(), errs
    # the metadata the device ended with, replayed on the host from the commits
    ln_h, pad_h = ln0.astype(np.int64), pad0.astype(np.int64)
    moved = 0
    for n in ne_log.cpu().numpy():
        ln_n = ln_h + n
        pad_n = ln_n.max() - ln_n
        moved += int((pad_n != pad_h).sum())
        ln_h, pad_h = ln_n, pad_n
    assert np.array_equal(lens[cur].cpu().numpy(), ln_h) and np.array_equal(pads[cur].cpu().numpy(), pad_h)
    opos, omask = oracle.rebuild_pos_mask(S, pad_h.astype(np.int32))
    assert np.array_equal(pos.cpu().numpy(), opos) and np.array_equal(mask.cpu().numpy(), omask)
    assert moved > R  # sequences moved in most rounds


@pytest.mark.parametrize("via", ["round", "graph", "calls"])
def test_greedy_work_after_a_round_needs_no_host_sync(via):
    _chain_without_host_sync("greedy", via, seed=61)


@pytest.mark.parametrize("via", ["round", "calls"])
def test_sample_work_after_a_round_needs_no_host_sync(via):
    _chain_without_host_sync("sample", via, seed=67)
