"""Device-side input generators (PyTorch RNG on the GPU + specgen.cu).

Used for full-size workloads, where generating on the host would dominate.
Nothing here computes any step of verification or realignment.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "specgen.cu")
_LIB = os.path.join(_HERE, "libspecgen.so")
_NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
_ELT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
_lib = None


def build(force=False):
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([_NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.specgen_kv_fill.argtypes = [vp, i, i, i, i, i, i, vp, vp, vp, i, vp]
        lib.specgen_kv_write_query.argtypes = [vp, i, i, i, i, i, i, vp, i, vp, i, vp]
        lib.specgen_kv_check.argtypes = [vp, i, i, i, i, i, i, vp, vp, vp, vp, vp]
        lib.specgen_kv_write_query_pool.argtypes = [vp, i, i, i, i, i, i, vp, i, i, vp, vp, vp]
        lib.specgen_kv_write_query_dev.argtypes = [vp, i, i, i, i, i, i, vp, i, vp, vp, vp]
        for f in (lib.specgen_kv_fill, lib.specgen_kv_write_query, lib.specgen_kv_check,
                  lib.specgen_kv_write_query_pool, lib.specgen_kv_write_query_dev):
            f.restype = i
        _lib = lib
    return _lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def kv_fill(kv, tokens, pad, nvalid, junk=True):
    """Prefill: slot pad_b + p holds f(b, tokens[b, p], p) for p < nvalid_b;
    with junk, every other slot holds a 'never valid' pattern."""
    L, _, B, H, S, D = kv.shape
    rc = _load().specgen_kv_fill(_p(kv), _ELT[kv.dtype], L, B, H, S, D, _p(tokens), _p(pad), _p(nvalid),
                                 1 if junk else 0, _s())
    assert rc == 0, rc


def kv_write_query(kv, qtok, pos, W):
    """The verification forward's KV write: slot W-1+j of sequence b gets
    f(b, qtok[b, j], pos[b, W-1+j])."""
    L, _, B, H, S, D = kv.shape
    rc = _load().specgen_kv_write_query(_p(kv), _ELT[kv.dtype], L, B, H, S, D, _p(qtok), qtok.shape[1], _p(pos),
                                        int(W), _s())
    assert rc == 0, rc


def kv_write_query_dev(kv, qtok, pos, W):
    """kv_write_query with the width W a [1] int32 device tensor (read on the
    device: nothing waits for the host)."""
    L, _, B, H, S, D = kv.shape
    rc = _load().specgen_kv_write_query_dev(_p(kv), _ELT[kv.dtype], L, B, H, S, D, _p(qtok), qtok.shape[1], _p(pos),
                                            _p(W), _s())
    assert rc == 0, rc


def kv_check_async(kv, tokens, pad_new, len_new, bad):
    """Adds to `bad` ([1] int64 on the device) the number of KV elements that
    break I2, without waiting for the result."""
    L, _, B, H, S, D = kv.shape
    rc = _load().specgen_kv_check(_p(kv), _ELT[kv.dtype], L, B, H, S, D, _p(tokens), _p(pad_new), _p(len_new),
                                  _p(bad), _s())
    assert rc == 0, rc


def kv_write_query_pool(pool, qtok, seq, base):
    """The forward's KV write on a ragged pool: batch row b (pool sequence
    seq[b]) writes f(seq[b], qtok[b, j], base[b] + j) at slot base[b] + j."""
    L, _, N, H, S, D = pool.shape
    rc = _load().specgen_kv_write_query_pool(_p(pool), _ELT[pool.dtype], L, N, H, S, D, _p(qtok), qtok.shape[1],
                                             qtok.shape[0], _p(seq), _p(base), _s())
    assert rc == 0, rc


def kv_check(kv, tokens, pad_new, len_new):
    """Number of KV elements that break I2 (0 when every slot pad'_b + p,
    p < len'_b - 1, holds f(b, tokens[b, p], p))."""
    L, _, B, H, S, D = kv.shape
    bad = torch.zeros(1, dtype=torch.int64, device=kv.device)
    rc = _load().specgen_kv_check(_p(kv), _ELT[kv.dtype], L, B, H, S, D, _p(tokens), _p(pad_new), _p(len_new),
                                  _p(bad), _s())
    assert rc == 0, rc
    return int(bad.item())


def greedy_round_inputs(B, k, V, alpha, sigma, gen, dtype, device):
    """Device version of np_gen.greedy_round_inputs (same recipe, torch RNG)."""
    x = (torch.randn((B, k + 1, V), generator=gen, device=device, dtype=torch.float32) * sigma).to(dtype)
    d = torch.randint(0, V, (B, k), generator=gen, device=device, dtype=torch.int32)
    if k > 0 and V > 1:
        coin = torch.rand((B, k), generator=gen, device=device) < alpha
        rows = x[:, :k].float()
        val = torch.where(coin, rows.amax(-1) + 1.0, rows.amin(-1) - 1.0)
        rows.scatter_(-1, d.long().unsqueeze(-1), val.unsqueeze(-1))
        x[:, :k] = rows.to(dtype)
    return x, d


def sample_round_inputs(B, k, V, noise, gen, dtype, device, sigma=1.0):
    """Device version of np_gen.sample_round_inputs: target logits, draft
    distribution q = softmax(target + noise) in fp32, proposals drawn from q,
    uniforms [B, k+1]."""
    x = torch.randn((B, k + 1, V), generator=gen, device=device, dtype=torch.float32) * sigma
    dl = x[:, :k] + torch.randn((B, k, V), generator=gen, device=device, dtype=torch.float32) * noise
    q = torch.softmax(dl, dim=-1)
    if k > 0:
        d = torch.multinomial(q.reshape(-1, V), 1, generator=gen).reshape(B, k).to(torch.int32)
    else:
        d = torch.zeros((B, 0), dtype=torch.int32, device=device)
    u = torch.rand((B, k + 1), generator=gen, device=device, dtype=torch.float32)
    return x.to(dtype), q.contiguous(), d.contiguous(), u
