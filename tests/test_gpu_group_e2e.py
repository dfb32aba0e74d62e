"""Same-length grouping vs the oracle (bit-exact), and the toy end-to-end
equivalence run through the CUDA path: greedy verification, realignment and
the position/mask rebuild all on the device, the toy target on the host."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_28_gb300 as sv
from gpu_util import dev, to_dev
from oracle.toy import ToyPair, run_batch_spec
from specgen import CONFIGS

pytestmark = pytest.mark.gpu


def group_both(lens, B, active=None):
    idx, ce, gl = sv.spec_group_by_length(to_dev(lens), B, active=None if active is None else to_dev(active))
    r_idx, r_ce, r_gl = oracle.group_by_length(lens, B, active)
    assert np.array_equal(idx.cpu().numpy(), r_idx), (idx.cpu().numpy(), r_idx)
    assert int(ce.item()) == r_ce and int(gl.item()) == r_gl
    return r_ce


@pytest.mark.parametrize("variant", ["a", "b"])
def test_config4_pools(variant):
    c = CONFIGS["c4"]
    rng = np.random.default_rng(1004)
    full = 0
    for r in range(20):
        if variant == "a":
            lens = rng.integers(c["pool_len"][0], c["pool_len"][1] + 1, size=c["N"]).astype(np.int32)
        else:
            lens = (rng.integers(1, 9, size=c["N"]) * 128).astype(np.int32)
        act = (rng.random(c["N"]) < 0.9).astype(np.uint8) if r % 2 else None
        full += group_both(lens, c["B"], act) == c["B"]
    if variant == "b":
        assert full >= 16  # 8 length buckets of ~60 sequences: a full group of 64 most rounds


def test_small_pools_and_degenerate_cases():
    rng = np.random.default_rng(0)
    for N in list(range(0, 12)) + [1000, 1024, 1025, 4096]:
        for trial in range(5):
            lens = rng.integers(-3, 6, size=N).astype(np.int32)
            act = (rng.random(N) < 0.7).astype(np.uint8)
            for B in (0, 1, 5, 64):
                group_both(lens, B, act if trial % 2 else None)
    group_both(np.zeros(0, np.int32), 3)
    group_both(np.array([5, 5], np.int32), 3, np.zeros(2, np.uint8))


# -- toy end to end through the device ---------------------------------------------

def gpu_verify(logits, draft, remaining, eos):
    out, na, ne = sv.spec_verify_greedy(to_dev(logits), to_dev(draft), eos_id=eos, remaining=to_dev(remaining))
    return out.cpu().numpy(), na.cpu().numpy(), ne.cpu().numpy()


def gpu_realign(kv, ln, pad, ne):
    kv_t = torch.from_numpy(kv).to(dev())
    ln2, pd2, w2, err = sv.spec_realign_kv(kv_t, to_dev(ln), to_dev(pad), to_dev(ne))
    kv[...] = kv_t.cpu().numpy()
    return int(err.item()), ln2.cpu().numpy(), pd2.cpu().numpy(), int(w2.item())


def gpu_posmask(S, pad_new, pad_old, pos, mask):
    p_t, m_t = to_dev(pos), to_dev(mask)
    sv.spec_rebuild_pos_mask(to_dev(pad_new), p_t, m_t, pad_old=None if pad_old is None else to_dev(pad_old))
    pos[...] = p_t.cpu().numpy()
    mask[...] = m_t.cpu().numpy()


@pytest.mark.parametrize("B,k,alpha,n_new,eos,kvdt", [
    (3, 2, 0.7, 14, -1, np.float32),
    (5, 4, 0.5, 16, -1, np.float16),
    (4, 3, 0.9, 18, 5, np.float32),
    (6, 1, 0.3, 10, 3, np.float16),
])
def test_batch_speculative_equals_single_sequence_greedy_on_device(B, k, alpha, n_new, eos, kvdt):
    pair = ToyPair(V=11, L=2, H=2, D=4, alpha=alpha, seed=B * 10 + k)
    rng = np.random.default_rng(B + k)
    prompts = [list(rng.integers(0, 11, size=int(rng.integers(1, 9)))) for _ in range(B)]
    S = 9 + n_new + 2 * (k + 1) + 8
    gen = run_batch_spec(pair, prompts, n_new, k, S, gpu_verify, gpu_realign, gpu_posmask, eos_id=eos,
                         kv_dtype=kvdt)
    for b in range(B):
        assert gen[b] == pair.ref_generate(b, prompts[b], n_new, eos_id=eos), b
