"""The C ABI boundary, checked on the host (no GPU needed).

The library must load and export every entry point include/specverify.h
declares; argument errors must be reported before anything is launched (these
calls return before any CUDA runtime call, so they run on a CPU-only box).
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_28_gb300 import _lib
    from speculative_decoding_verification_28_gb300 import build as libbuild

    libbuild.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"spec_verify_greedy", "spec_verify_sample", "spec_realign_kv", "spec_rebuild_pos_mask",
            "spec_group_by_length", "spec_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    from speculative_decoding_verification_28_gb300._lib import SIGNATURES

    assert set(SIGNATURES) == set(names)


def test_workspace_sizes(lib):
    assert lib.spec_workspace_bytes(0, 4, 100) == 0
    a = lib.spec_workspace_bytes(8, 5, 32000)
    b = lib.spec_workspace_bytes(8, 5, 64000)
    c = lib.spec_workspace_bytes(16, 5, 32000)
    assert 0 < a < b and a < c and a % 256 == 0
    # the realignment needs only the batch-dependent part
    assert lib.spec_workspace_bytes(8, 0, 1) <= a


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below returns first
FAKE_ODD = ctypes.c_void_p(0x10001)


def greedy(lib, logits=FAKE, dt=1, B=2, k=3, V=100, draft=FAKE, out=FAKE, ws=FAKE, wsb=1 << 30):
    return lib.spec_verify_greedy(logits, dt, B, k, V, draft, None, -1, None, out, FAKE, FAKE, ws, wsb, None)


def test_greedy_argument_errors(lib):
    assert greedy(lib, B=-1) == -1
    assert greedy(lib, k=-1) == -1
    assert greedy(lib, k=32) == -1  # above SPEC_MAX_K
    assert greedy(lib, V=0) == -1
    assert greedy(lib, dt=7) == -2
    assert greedy(lib, logits=None) == -1
    assert greedy(lib, draft=None) == -1
    assert greedy(lib, out=None) == -1
    assert greedy(lib, ws=None) == -3
    assert greedy(lib, wsb=16) == -3
    assert greedy(lib, ws=FAKE_ODD) == -3
    assert greedy(lib, logits=FAKE_ODD) == -5
    assert greedy(lib, B=0) == 0  # empty batch: valid no-op, nothing launched


def test_per_sequence_arguments_must_be_aligned(lib):
    """draft_len and remaining are int32 arrays: a misaligned one is refused
    on the host (SPEC_EALIGN) by every verification entry point, before any
    launch."""
    for dl, rem in ((FAKE_ODD, None), (None, FAKE_ODD)):
        assert lib.spec_verify_greedy(FAKE, 1, 2, 3, 100, FAKE, dl, -1, rem, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                                      None) == -5
        assert lib.spec_verify_sample(FAKE, 0, 1.0, FAKE, FAKE, FAKE, 2, 2, 50, dl, -1, rem, FAKE, FAKE, FAKE, None,
                                      None, FAKE, 1 << 30, None) == -5
        assert lib.spec_verify_sample_filtered(FAKE, 0, 1.0, FAKE, None, FAKE, FAKE, FAKE, 2, 2, 50, dl, -1, rem,
                                               FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == -5
        assert lib.spec_verify_greedy_static(FAKE, 1, 2, 3, 100, FAKE, dl, -1, rem, FAKE, FAKE, FAKE, None) == -5
    # aligned ones pass the same checks (the greedy call then fails only on its
    # missing workspace)
    assert lib.spec_verify_greedy(FAKE, 1, 2, 3, 100, FAKE, FAKE, -1, FAKE, FAKE, FAKE, FAKE, None, 0, None) == -3


def test_sample_argument_errors(lib):
    def sample(temp=1.0, u=FAKE, q=FAKE, k=2):
        return lib.spec_verify_sample(FAKE, 0, temp, q, FAKE, u, 2, k, 50, None, -1, None, FAKE, FAKE, FAKE, None,
                                      None, FAKE, 1 << 30, None)

    assert sample(temp=0.0) == -1
    assert sample(temp=-1.0) == -1
    assert sample(temp=float("nan")) == -1
    assert sample(temp=float("inf")) == -1
    assert sample(u=None) == -1
    assert sample(q=None) == -1
    assert sample(u=FAKE_ODD) == -5


def test_filtered_sample_argument_errors(lib):
    def sample(temp=1.0, tk=FAKE, tp=FAKE, u=FAKE):
        return lib.spec_verify_sample_filtered(FAKE, 0, temp, tk, tp, FAKE, FAKE, u, 2, 2, 50, None, -1, None, FAKE,
                                               FAKE, FAKE, None, None, FAKE, 1 << 30, None)

    assert sample(temp=0.0) == -1
    assert sample(u=None) == -1
    assert sample(tk=FAKE_ODD) == -5
    assert sample(tp=FAKE_ODD) == -5
    assert sample(tk=FAKE, tp=None, u=FAKE_ODD) == -5


def test_realign_argument_errors(lib):
    def realign(kv=FAKE, dt=1, L=2, B=3, H=2, S=64, D=8, ws=FAKE, wsb=1 << 20, err=FAKE):
        return lib.spec_realign_kv(kv, dt, L, B, H, S, D, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, err, ws, wsb, None)

    assert realign(L=0) == -1
    assert realign(S=0) == -1
    assert realign(B=-2) == -1
    assert realign(B=0) == 0
    assert realign(dt=5) == -2
    assert realign(kv=None) == -1
    assert realign(err=None) == -1
    assert realign(ws=None) == -3
    assert realign(wsb=8) == -3
    assert realign(kv=FAKE_ODD) == -5


def test_posmask_and_group_argument_errors(lib):
    assert lib.spec_rebuild_pos_mask(-1, 8, None, FAKE, FAKE, FAKE, None) == -1
    assert lib.spec_rebuild_pos_mask(0, 8, None, FAKE, FAKE, FAKE, None) == 0
    assert lib.spec_rebuild_pos_mask(2, 0, None, FAKE, FAKE, FAKE, None) == 0
    assert lib.spec_rebuild_pos_mask(2, 8, FAKE, FAKE, FAKE, FAKE, None) == -1  # pad_old aliases pad_new
    assert lib.spec_rebuild_pos_mask(2, 8, None, None, FAKE, FAKE, None) == -1
    assert lib.spec_group_by_length(-1, FAKE, None, 4, FAKE, FAKE, FAKE, None) == -1
    assert lib.spec_group_by_length(4097, FAKE, None, 4, FAKE, FAKE, FAKE, None) == -1
    assert lib.spec_group_by_length(8, None, None, 4, FAKE, FAKE, FAKE, None) == -1
    assert lib.spec_group_by_length(8, FAKE, None, -1, FAKE, FAKE, FAKE, None) == -1


def test_status_strings(lib):
    for rc in (0, -1, -2, -3, -4, -5):
        assert lib.spec_status_str(rc)
    assert lib.spec_status_str(0) == b"ok"


def test_product_path_has_no_fallback():
    """The binding never imports the oracle and fails loudly without its library."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_28_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "oracle" not in src, fn
            assert "specgen" not in src, fn
    from speculative_decoding_verification_28_gb300 import _lib

    saved = _lib.LIB_PATH, _lib._lib
    try:
        _lib.LIB_PATH, _lib._lib = "/nonexistent/libspecverify.so", None
        with pytest.raises(ImportError):
            _lib.load()
    finally:
        _lib.LIB_PATH, _lib._lib = saved


def test_host_tensors_are_refused_not_computed():
    """Every entry point of the binding refuses CPU tensors before any call:
    there is no host path to fall back to."""
    import torch

    import speculative_decoding_verification_28_gb300 as sv

    x = torch.zeros((2, 3, 64), dtype=torch.float32)
    d = torch.zeros((2, 2), dtype=torch.int32)
    q = torch.full((2, 2, 64), 1.0 / 64)
    u = torch.zeros((2, 3))
    kv = torch.zeros((1, 2, 2, 1, 16, 8))
    ln = torch.tensor([3, 5], dtype=torch.int32)
    pad = torch.tensor([2, 0], dtype=torch.int32)
    ne = torch.tensor([1, 2], dtype=torch.int32)
    pos = torch.zeros((2, 16), dtype=torch.int32)
    mask = torch.zeros((2, 16), dtype=torch.uint8)
    pool_len = torch.tensor([3, 5, 4], dtype=torch.int32)
    idx = torch.tensor([0, 2], dtype=torch.int32)
    calls = [lambda: sv.spec_verify_greedy(x, d),
             lambda: sv.spec_verify_sample(x, q, d, u),
             lambda: sv.spec_verify_sample_filtered(x, q, d, u, top_k=5, top_p=0.9),
             lambda: sv.spec_realign_kv(kv, ln, pad, ne),
             lambda: sv.spec_rebuild_pos_mask(pad, pos, mask),
             lambda: sv.spec_group_by_length(pool_len, 2),
             lambda: sv.spec_commit_ragged(pool_len, idx, ne, 16)]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA"):
            call()


def test_static_entry_point_rejects_oversized_batches_before_any_launch(lib):
    """The allocation-free variant has a fixed scratch: sizes beyond it are a
    clear error (-6) found on the host."""
    from speculative_decoding_verification_28_gb300 import STATIC_SCRATCH_BYTES

    B, k, V = 4096, 31, 151936
    assert lib.spec_workspace_bytes(B, k, V) > STATIC_SCRATCH_BYTES
    rc = lib.spec_verify_greedy_static(FAKE, 1, B, k, V, FAKE, None, -1, None, FAKE, FAKE, FAKE, None)
    assert rc == -6 and b"SPEC_STATIC_SCRATCH_BYTES" in lib.spec_status_str(-6)
    assert lib.spec_verify_greedy_static(FAKE, 1, -1, k, V, FAKE, None, -1, None, FAKE, FAKE, FAKE, None) == -1
    assert lib.spec_verify_greedy_static(FAKE, 9, 2, k, V, FAKE, None, -1, None, FAKE, FAKE, FAKE, None) == -2
    assert lib.spec_verify_greedy_static(FAKE, 1, 0, k, V, FAKE, None, -1, None, FAKE, FAKE, FAKE, None) == 0
    # the benchmark's largest workload fits
    assert lib.spec_workspace_bytes(256, 8, 128256) <= STATIC_SCRATCH_BYTES


def test_multi_cache_argument_errors(lib):
    from speculative_decoding_verification_28_gb300._lib import KVCacheDesc

    def multi(descs, n=None, B=3, S=64, ws=FAKE):
        arr = (KVCacheDesc * max(1, len(descs)))(*descs)
        return lib.spec_realign_kv_multi(ctypes.cast(arr, ctypes.c_void_p), len(descs) if n is None else n, B, S,
                                         FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, 1 << 20, None)

    good = KVCacheDesc(0x10000, 1, 2, 4, 128)
    assert multi([good], n=0) == -1
    assert multi([good] * 5) == -1  # above SPEC_MAX_CACHES
    assert multi([good, KVCacheDesc(0x10000, 9, 2, 4, 128)]) == -2
    assert multi([good, KVCacheDesc(0x10000, 1, 0, 4, 128)]) == -1
    assert multi([good, KVCacheDesc(None, 1, 2, 4, 128)]) == -1
    assert multi([good, KVCacheDesc(0x10001, 1, 2, 4, 128)]) == -5
    assert multi([good], B=0) == 0
    assert multi([good], ws=None) == -3
    assert lib.spec_realign_kv_multi(None, 1, 3, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20,
                                     None) == -1


def test_pool_argument_errors(lib):
    assert lib.spec_commit_ragged(-1, FAKE, 2, FAKE, FAKE, 16, FAKE, None) == -1
    assert lib.spec_commit_ragged(65537, FAKE, 2, FAKE, FAKE, 16, FAKE, None) == -1
    assert lib.spec_commit_ragged(8, FAKE, 0, FAKE, FAKE, 16, FAKE, None) == 0
    assert lib.spec_commit_ragged(8, None, 2, FAKE, FAKE, 16, FAKE, None) == -1

    def repad(pool=FAKE, batch=FAKE, dt=1, L=2, N=8, B=2, H=2, S=64, D=8, ws=FAKE, pl=FAKE):
        return lib.spec_repad_gather(pool, batch, dt, L, N, B, H, S, D, FAKE, pl, FAKE, FAKE, FAKE, FAKE, ws,
                                     1 << 20, None)

    assert repad(L=0) == -1 and repad(N=70000) == -1 and repad(dt=7) == -2
    assert repad(B=0) == 0 and repad(pool=None) == -1 and repad(pl=None) == -1
    assert repad(ws=None) == -3 and repad(batch=FAKE_ODD) == -5
    assert lib.spec_unpad_scatter(FAKE, FAKE, 1, 2, 8, 2, 2, 64, 8, FAKE, None, FAKE, None, FAKE, FAKE, FAKE,
                                  1 << 20, None) == -1
    assert lib.spec_unpad_scatter(FAKE, FAKE, 1, 2, 8, 2, 2, 64, 8, FAKE, FAKE, FAKE, FAKE_ODD, FAKE, FAKE, FAKE,
                                  1 << 20, None) == -5


def test_round_entry_points_check_everything_before_launching(lib):
    from speculative_decoding_verification_28_gb300._lib import KVCacheDesc

    one = (KVCacheDesc * 1)(KVCacheDesc(0x10000, 1, 2, 2, 8))
    P = ctypes.cast(one, ctypes.c_void_p)

    def greedy(B=2, S=64, pad=FAKE, pad_new=ctypes.c_void_p(0x20000), pos=FAKE, n_caches=1, caches=P, ws=FAKE):
        return lib.spec_round_greedy(FAKE, 1, B, 3, 100, FAKE, None, -1, None, caches, n_caches, S, FAKE, pad, pos,
                                     FAKE, FAKE, FAKE, FAKE, FAKE, pad_new, FAKE, FAKE, ws, 1 << 30, None)

    assert greedy(B=-1) == -1
    assert greedy(pad_new=FAKE) == -1           # pad_new aliases pad
    assert greedy(pos=None) == -1
    assert greedy(n_caches=0) == -1
    assert greedy(caches=None) == -1
    assert greedy(pos=FAKE_ODD) == -5
    assert greedy(ws=FAKE_ODD) == -3
    assert greedy(B=0) == 0

    def sample(T=1.0, tk=None, u=FAKE):
        return lib.spec_round_sample(FAKE, 0, T, tk, None, FAKE, FAKE, u, 2, 3, 100, None, -1, None, P, 1, 64,
                                     FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE,
                                     ctypes.c_void_p(0x20000), FAKE, FAKE, FAKE, 1 << 30, None)

    assert sample(T=0.0) == -1
    assert sample(u=None) == -1
    assert sample(tk=FAKE_ODD) == -5
