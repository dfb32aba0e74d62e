"""Toy table-driven target/draft pair for the end-to-end equivalence test.

TEST INFRASTRUCTURE ONLY.

The summary of "Correctness Forensics for Batch Speculative Decoding" (App. B)
states that with rectangular alignment (I1) and position-ID/KV correspondence
(I2) maintained every round, and the bonus token drawn from the target,
deterministic decoding yields the same tokens as per-sequence decoding under
exact arithmetic.  This toy makes that checkable bit for bit:

* the target's "forward" at a query slot folds, in slot order, the position ID
  and the KV-cache contents of every visible slot (mask = 1, slot <= query)
  into a 64-bit digest, and turns the digest into integer-valued logits with a
  unique maximum -- so a KV row in the wrong slot, a kept rejected row or a
  stale position ID changes the logits;
* the reference decodes one sequence alone (batch size 1, no padding, no
  speculation), computing the same digest straight from its token history;
* the draft proposes the target's own choice with an iid hash coin of
  probability alpha, and a different token otherwise.

KV rows are the synthetic values f(seq, token, pos, ...) of ``specgen``, and
the query slots' KV is written by the harness at the slot's position ID, as a
real forward would do through its rotary embedding.
"""
from __future__ import annotations

import numpy as np

from specgen import kv_row_values, splitmix64

_M = (1 << 64) - 1


def _mix(x: int) -> int:
    """splitmix64 output function (Vigna) on a Python int, used as the toy's
    digest mixer."""
    z = (x + 0x9E3779B97F4A7C15) & _M
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M
    return z ^ (z >> 31)


def _pack(vals) -> int:
    """Pack up to eight multiples of 1/128 in [-1, 1) into a 64-bit word."""
    w = 0
    for i, v in enumerate(np.asarray(vals, dtype=np.float64)[:8]):
        w |= (int(round(v * 128.0)) & 0xFF) << (8 * i)
    return w


class ToyPair:
    def __init__(self, V: int, L: int, H: int, D: int, alpha: float, seed: int = 7):
        assert D <= 8 and V >= 2
        self.V, self.L, self.H, self.D = V, L, H, D
        self.alpha, self.seed = alpha, seed
        self._row_cache = {}

    # -- KV contents -----------------------------------------------------
    def kv_rows(self, seq, tok, pos):
        key = (seq, tok, pos)
        r = self._row_cache.get(key)
        if r is None:
            r = kv_row_values(seq, tok, pos, self.L, self.H, self.D)
            self._row_cache[key] = r
        return r

    # -- target ------------------------------------------------------------
    def fold(self, digest: int, pos: int, krow, vrow) -> int:
        """One visible slot: its position ID, the K row of (layer 0, head 0)
        and the V row of (last layer, last head)."""
        digest = _mix(digest ^ _pack(krow))
        digest = _mix(digest ^ _pack(vrow))
        return _mix(digest ^ (pos & 0xFFFFFFFF) ^ (0xABCD << 40))

    def logits(self, digest: int) -> np.ndarray:
        v = np.arange(self.V, dtype=np.uint64)
        with np.errstate(over="ignore"):
            h = splitmix64(np.uint64(digest) ^ (v * np.uint64(0x9E3779B97F4A7C15)))
        x = (h >> np.uint64(54)).astype(np.float32)  # 0 .. 1023
        x[digest % self.V] = 2048.0  # unique maximum
        return x

    def ref_digest(self, seq: int, tokens) -> int:
        """Digest after the last token of a history decoded alone."""
        d = 0
        for p, t in enumerate(tokens):
            r = self.kv_rows(seq, int(t), p)
            d = self.fold(d, p, r[0, 0, 0], r[self.L - 1, 1, self.H - 1])
        return d

    def ref_next(self, seq: int, tokens) -> int:
        return int(np.argmax(self.logits(self.ref_digest(seq, tokens))))

    def ref_generate(self, seq, prompt, n_new, eos_id=-1):
        """Batch-size-1, non-speculative greedy decoding."""
        toks = list(prompt)
        d = self.ref_digest(seq, toks)
        out = []
        for _ in range(n_new):
            t = int(np.argmax(self.logits(d)))
            out.append(t)
            if t == eos_id:
                break
            r = self.kv_rows(seq, t, len(toks))
            d = self.fold(d, len(toks), r[0, 0, 0], r[self.L - 1, 1, self.H - 1])
            toks.append(t)
        return out

    # -- draft ---------------------------------------------------------------
    def propose(self, seq: int, history, k: int):
        """k proposals; each equals the target's own choice with probability
        alpha (a hash coin of (seed, seq, position)), else another token."""
        hist = list(history)
        props = []
        for _ in range(k):
            want = self.ref_next(seq, hist)
            pos = len(hist)
            h = _mix((self.seed << 48) ^ (seq << 24) ^ pos)
            if (h >> 11) / float(1 << 53) < self.alpha:
                t = want
            else:
                t = (want + 1 + (h % (self.V - 1))) % self.V
            props.append(t)
            hist.append(t)
        return props

    # -- batched forward on a left-padded cache ----------------------------------
    def write_query_kv(self, kv, pos, b, slot, tok):
        """The forward's KV write for one query slot at that slot's position ID."""
        kv[:, :, b, :, slot, :] = self.kv_rows(b, int(tok), int(pos[b, slot]))

    def write_query_kv_seq(self, kv, pos, b, seq, slot, tok):
        """As write_query_kv for batch row b holding pool sequence `seq`."""
        kv[:, :, b, :, slot, :] = self.kv_rows(seq, int(tok), int(pos[b, slot]))

    def batched_logits(self, kv, pos, mask, b, q_slot0, n_rows):
        """Logits of query slots q_slot0 .. q_slot0 + n_rows - 1 of sequence b,
        folding every visible slot of the cache in slot order."""
        out = np.empty((n_rows, self.V), np.float32)
        d = 0
        s_end = q_slot0 + n_rows
        r = 0
        for s in range(s_end):
            if mask[b, s]:
                d = self.fold(d, int(pos[b, s]), kv[0, 0, b, 0, s], kv[self.L - 1, 1, b, self.H - 1, s])
            if s >= q_slot0:
                out[r] = self.logits(d)
                r += 1
        return out


def run_batch_spec(pair: ToyPair, prompts, n_new, k, S, verify, realign, posmask, eos_id=-1,
                   kv_dtype=np.float32, max_rounds=1000):
    """Batch speculative greedy decoding of the toy pair on a contiguous
    left-padded cache, one verification round at a time.

    verify(logits [B,k+1,V] f32, draft [B,k], remaining [B], eos) ->
        (out_tokens, n_accept, n_emit)
    realign(kv, len, pad, n_emit) -> (status, len_new, pad_new, width_new)
    posmask(S, pad_new, pad_old, pos, mask) -> None (in place)
    Returns the generated tokens of every sequence.
    """
    B = len(prompts)
    L, H, D = pair.L, pair.H, pair.D
    ln = np.array([len(p) for p in prompts], np.int32)
    W = int(ln.max())
    pad = (W - ln).astype(np.int32)
    kv = np.zeros((L, 2, B, H, S, D), kv_dtype)
    pos = np.zeros((B, S), np.int32)
    mask = np.zeros((B, S), np.uint8)
    posmask(S, pad, None, pos, mask)
    hist = [list(p) for p in prompts]
    # prefill: KV of every prompt token but the last
    for b in range(B):
        for p in range(len(prompts[b]) - 1):
            kv[:, :, b, :, pad[b] + p, :] = pair.kv_rows(b, prompts[b][p], p)
    gen = [[] for _ in range(B)]
    done = np.zeros(B, bool)
    for _ in range(max_rounds):
        if done.all():
            break
        W = int(pad[0] + ln[0])
        assert W + k <= S, "toy cache too small"
        draft = np.zeros((B, k), np.int32)
        logits = np.zeros((B, k + 1, pair.V), np.float32)
        for b in range(B):
            props = pair.propose(b, hist[b], k) if not done[b] else [0] * k
            draft[b] = props
            q_toks = [hist[b][-1]] + props
            for j, t in enumerate(q_toks):
                pair.write_query_kv(kv, pos, b, W - 1 + j, t)
            logits[b] = pair.batched_logits(kv, pos, mask, b, W - 1, k + 1)
        remaining = np.array([0 if done[b] else n_new - len(gen[b]) for b in range(B)], np.int32)
        out, _, ne = verify(logits, draft, remaining, eos_id)
        for b in range(B):
            toks = [int(t) for t in out[b, : ne[b]]]
            gen[b] += toks
            hist[b] += toks
            if len(gen[b]) >= n_new or (eos_id >= 0 and eos_id in toks):
                done[b] = True
        st, ln2, pad2, _ = realign(kv, ln, pad, ne)
        assert st == 0, f"realign status {st}"
        posmask(S, pad2, pad, pos, mask)
        ln, pad = ln2.astype(np.int32), pad2.astype(np.int32)
    return gen


def exspec_select(lens, active, window, B, group):
    """The cross-batch selection: the first `window` active sequences in pool
    order form the window; `group(window_lens, B)` returns (idx into the
    window, count_equal, L*).  Returns pool indices (-1 dropped) and whether a
    full same-length group formed.  (The pages give no algorithm for EXSPEC's
    scheduler; this policy is this project's construction.)"""
    win = [n for n in range(len(lens)) if active[n]][:window]
    if not win:
        return [], False
    idx, ce, _ = group(np.array([lens[n] for n in win], np.int32), B)
    picks = [win[i] for i in idx if i >= 0]
    return picks, ce == B and len(picks) == B


def run_exspec(pair: ToyPair, prompts, n_new, k, S, B, window, ops, eos_id=-1, max_rounds=2000,
               fallback_realign=True, result=None):
    """EXSPEC-style decoding of the toy pair over a ragged pool: each round the
    window's largest same-length group is verified in place (grouped round, no
    realignment: the commit is a length update); when no full group forms the
    chosen sequences are repadded into a batch, verified and realigned there,
    and unpadded back (fallback round).

    ops: dict of callables
      group(lens, B) -> (idx, count_equal, L*)
      verify(logits, draft, remaining, eos) -> (out_tokens, n_accept, n_emit)
      commit(pool_len, idx, n_emit, S) -> status            (pool_len in place)
      repad(pool, batch, idx, pool_len) -> (status, len, pad, width)
      realign(kv, len, pad, n_emit) -> (status, len_new, pad_new, width)
      unpad(batch, pool, idx, len, pad, pool_len, n_emit=None) -> status
                                                   (pool_len in place; with n_emit the
                                                    lengths written back are len + n_emit)
    fallback_realign=False unpads a fallback round straight from the extended
    batch (lengths len + n_emit at the old paddings) instead of realigning
    the batch first: the rows pad .. pad + len + n_emit - 2 already hold
    positions 0 .. len + n_emit - 2, so the pool must end byte for byte the
    same.  result (a dict, optional) receives the final pool and lengths.
    Returns (generated tokens per sequence, rounds, grouped rounds)."""
    N = len(prompts)
    L, H, D = pair.L, pair.H, pair.D
    pool = np.zeros((L, 2, N, H, S, D), np.float32)
    pool_len = np.array([len(p) for p in prompts], np.int32)
    hist = [list(p) for p in prompts]
    for n in range(N):
        for p in range(len(prompts[n]) - 1):
            pool[:, :, n, :, p, :] = pair.kv_rows(n, prompts[n][p], p)
    pool_pos = np.broadcast_to(np.arange(S, dtype=np.int32), (N, S)).copy()
    pool_mask = np.ones((N, S), np.uint8)
    gen = [[] for _ in range(N)]
    active = np.ones(N, bool)
    rounds = grouped = 0
    for _ in range(max_rounds):
        if not active.any():
            break
        picks, full = exspec_select(pool_len, active, window, B, ops["group"])
        Bb = len(picks)
        rounds += 1
        draft = np.zeros((Bb, k), np.int32)
        logits = np.zeros((Bb, k + 1, pair.V), np.float32)
        remaining = np.array([n_new - len(gen[n]) for n in picks], np.int32)
        if full:
            grouped += 1
            for i, n in enumerate(picks):  # forward on the pool: position = slot
                props = pair.propose(n, hist[n], k)
                draft[i] = props
                q0 = int(pool_len[n]) - 1
                assert q0 + k < S, "toy pool too small"
                for j, t in enumerate([hist[n][-1]] + props):
                    pair.write_query_kv(pool, pool_pos, n, q0 + j, t)
                logits[i] = pair.batched_logits(pool, pool_pos, pool_mask, n, q0, k + 1)
            out, _, ne = ops["verify"](logits, draft, remaining, eos_id)
            assert ops["commit"](pool_len, np.array(picks, np.int32), ne, S) == 0
        else:
            batch = np.zeros((L, 2, Bb, H, S, D), np.float32)
            st, ln, pad, W = ops["repad"](pool, batch, np.array(picks, np.int32), pool_len)
            assert st == 0 and W + k < S
            pos = np.zeros((Bb, S), np.int32)
            mask = np.zeros((Bb, S), np.uint8)
            for i in range(Bb):
                mask[i, pad[i]:] = 1
                pos[i, pad[i]:] = np.arange(S - pad[i])
            for i, n in enumerate(picks):
                props = pair.propose(n, hist[n], k)
                draft[i] = props
                for j, t in enumerate([hist[n][-1]] + props):
                    pair.write_query_kv_seq(batch, pos, i, n, W - 1 + j, t)
                logits[i] = pair.batched_logits(batch, pos, mask, i, W - 1, k + 1)
            out, _, ne = ops["verify"](logits, draft, remaining, eos_id)
            if fallback_realign:
                st, ln2, pad2, _ = ops["realign"](batch, ln, pad, ne)
                assert st == 0
                assert ops["unpad"](batch, pool, np.array(picks, np.int32), ln2, pad2, pool_len) == 0
            else:
                assert ops["unpad"](batch, pool, np.array(picks, np.int32), ln, pad, pool_len,
                                    np.asarray(ne, np.int32)) == 0
        for i, n in enumerate(picks):
            toks = [int(t) for t in out[i, : ne[i]]]
            gen[n] += toks
            hist[n] += toks
            if len(gen[n]) >= n_new or (eos_id >= 0 and eos_id in toks):
                active[n] = False
    if result is not None:
        result["pool"], result["pool_len"] = pool, pool_len
    return gen, rounds, grouped
