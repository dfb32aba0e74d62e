"""Thin PyTorch binding of the C ABI: argument marshalling only.

Each function has the name of its C entry point, takes CUDA tensors, passes
their device pointers and sizes, and raises on a negative return code.  All
computation happens in the library's kernels.  Outputs not supplied are
allocated with ``torch.empty`` on the input's device; workspaces not supplied
come from a per-(device, stream, batch) cache of zero-filled buffers.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

SPEC_F32, SPEC_BF16, SPEC_F16 = 0, 1, 2
_DT = {torch.float32: SPEC_F32, torch.bfloat16: SPEC_BF16, torch.float16: SPEC_F16}

REALIGN_OK, REALIGN_CAPACITY, REALIGN_LAYOUT, REALIGN_EMIT, REALIGN_TIMEOUT = 0, 1, 2, 3, 4
FLAG_Q_ZERO, FLAG_ZERO_RESIDUAL, FLAG_NONFINITE, FLAG_BAD_TOKEN = 1, 2, 4, 8
MAX_K = 31
MAX_GROUP_N = 4096


class SpecError(RuntimeError):
    pass


def _check(rc):
    if rc != 0:
        msg = _lib.load().spec_status_str(rc).decode()
        raise SpecError(f"spec call failed ({rc}): {msg}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, device=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


class Workspace:
    """Zero-filled device scratch sized by spec_workspace_bytes()."""

    def __init__(self, B, k, V, device, stream=None):
        n = int(_lib.load().spec_workspace_bytes(int(B), int(k), int(V)))
        self.B, self.nbytes = int(B), max(n, 256)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


_ws_cache = {}


def _workspace(ws, B, k, V, device, stream):
    if ws is not None:
        return ws
    key = (device.index, stream.value if stream.value else 0, int(B))
    need = int(_lib.load().spec_workspace_bytes(int(B), int(k), int(V)))
    w = _ws_cache.get(key)
    if w is None or w.nbytes < need:
        w = Workspace(B, k, V, device)
        _ws_cache[key] = w
    return w


def spec_workspace_bytes(B, k, V):
    return int(_lib.load().spec_workspace_bytes(int(B), int(k), int(V)))


def spec_verify_greedy(target_logits, draft_tokens, draft_len=None, eos_id=-1, remaining=None,
                       out_tokens=None, n_accept=None, n_emit=None, workspace=None, stream=None):
    """target_logits [B, k+1, V] (fp32/bf16/fp16), draft_tokens [B, k] int32
    -> (out_tokens [B, k+1], n_accept [B], n_emit [B]) int32."""
    lib = _lib.load()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    _need(target_logits, None, "target_logits", dev)
    if target_logits.dtype not in _DT:
        raise ValueError(f"unsupported logits dtype {target_logits.dtype}")
    _need(draft_tokens, torch.int32, "draft_tokens", dev, (B, k))
    _need(draft_len, torch.int32, "draft_len", dev, (B,))
    _need(remaining, torch.int32, "remaining", dev, (B,))
    out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev) if out_tokens is None else out_tokens
    n_accept = torch.empty(B, dtype=torch.int32, device=dev) if n_accept is None else n_accept
    n_emit = torch.empty(B, dtype=torch.int32, device=dev) if n_emit is None else n_emit
    for t, nm, shp in ((out_tokens, "out_tokens", (B, k + 1)), (n_accept, "n_accept", (B,)),
                       (n_emit, "n_emit", (B,))):
        _need(t, torch.int32, nm, dev, shp)
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, k, V, dev, st)
    _check(lib.spec_verify_greedy(_p(target_logits), _DT[target_logits.dtype], B, k, V, _p(draft_tokens),
                                  _p(draft_len), int(eos_id), _p(remaining), _p(out_tokens), _p(n_accept),
                                  _p(n_emit), ws.ptr(), ws.nbytes, st))
    return out_tokens, n_accept, n_emit


STATIC_SCRATCH_BYTES = 4 << 20


def spec_verify_greedy_static(target_logits, draft_tokens, draft_len=None, eos_id=-1, remaining=None,
                              out_tokens=None, n_accept=None, n_emit=None, stream=None):
    """spec_verify_greedy for callers that cannot allocate device memory at
    call time (a serving loop that forbids allocation after start-up, or a
    plugin given only its input and output buffers): the scratch is a device
    array built into the library (STATIC_SCRATCH_BYTES per device), so no
    workspace is passed.  Pass preallocated outputs to allocate nothing here
    either.  Calls on one device share that array: calls that overlap on the
    GPU race, so order them.  The first call on a device looks up the array's
    address; make it before any stream capture."""
    lib = _lib.load()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    _need(target_logits, None, "target_logits", dev)
    if target_logits.dtype not in _DT:
        raise ValueError(f"unsupported logits dtype {target_logits.dtype}")
    _need(draft_tokens, torch.int32, "draft_tokens", dev, (B, k))
    _need(draft_len, torch.int32, "draft_len", dev, (B,))
    _need(remaining, torch.int32, "remaining", dev, (B,))
    out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev) if out_tokens is None else out_tokens
    n_accept = torch.empty(B, dtype=torch.int32, device=dev) if n_accept is None else n_accept
    n_emit = torch.empty(B, dtype=torch.int32, device=dev) if n_emit is None else n_emit
    for t, nm, shp in ((out_tokens, "out_tokens", (B, k + 1)), (n_accept, "n_accept", (B,)),
                       (n_emit, "n_emit", (B,))):
        _need(t, torch.int32, nm, dev, shp)
    st = _stream(stream, dev)
    with torch.cuda.device(dev):  # the library uses the current device's array
        _check(lib.spec_verify_greedy_static(_p(target_logits), _DT[target_logits.dtype], B, k, V, _p(draft_tokens),
                                             _p(draft_len), int(eos_id), _p(remaining), _p(out_tokens),
                                             _p(n_accept), _p(n_emit), st))
    return out_tokens, n_accept, n_emit


def spec_verify_sample(target_logits, draft_probs, draft_tokens, uniforms, temperature=1.0, draft_len=None,
                       eos_id=-1, remaining=None, out_tokens=None, n_accept=None, n_emit=None,
                       out_residual=None, flags=None, want_residual=False, workspace=None, stream=None):
    """-> (out_tokens, n_accept, n_emit, flags [B] int32 view of the uint32
    flag words, out_residual [B, V] fp32 or None)."""
    return _verify_sample(None, None, target_logits, draft_probs, draft_tokens, uniforms, temperature, draft_len,
                          eos_id, remaining, out_tokens, n_accept, n_emit, out_residual, flags, want_residual,
                          workspace, stream)


def spec_verify_sample_filtered(target_logits, draft_probs, draft_tokens, uniforms, top_k=None, top_p=None,
                                temperature=1.0, draft_len=None, eos_id=-1, remaining=None, out_tokens=None,
                                n_accept=None, n_emit=None, out_residual=None, flags=None, want_residual=False,
                                workspace=None, stream=None):
    """spec_verify_sample on the target distribution after top-k / top-p.
    top_k: None, an int for every sequence, or [B] int32 on the device;
    top_p: None, a float for every sequence, or [B] fp32 on the device."""
    B = target_logits.shape[0]
    dev = target_logits.device
    if top_k is not None and not torch.is_tensor(top_k):
        top_k = torch.full((B,), int(top_k), dtype=torch.int32, device=dev)
    if top_p is not None and not torch.is_tensor(top_p):
        top_p = torch.full((B,), float(top_p), dtype=torch.float32, device=dev)
    _need(top_k, torch.int32, "top_k", dev, (B,))
    _need(top_p, torch.float32, "top_p", dev, (B,))
    return _verify_sample(top_k, top_p, target_logits, draft_probs, draft_tokens, uniforms, temperature, draft_len,
                          eos_id, remaining, out_tokens, n_accept, n_emit, out_residual, flags, want_residual,
                          workspace, stream)


def _verify_sample(top_k, top_p, target_logits, draft_probs, draft_tokens, uniforms, temperature, draft_len, eos_id,
                   remaining, out_tokens, n_accept, n_emit, out_residual, flags, want_residual, workspace, stream):
    lib = _lib.load()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    _need(target_logits, None, "target_logits", dev)
    if target_logits.dtype not in _DT:
        raise ValueError(f"unsupported logits dtype {target_logits.dtype}")
    _need(draft_probs, torch.float32, "draft_probs", dev, (B, k, V))
    _need(draft_tokens, torch.int32, "draft_tokens", dev, (B, k))
    _need(uniforms, torch.float32, "uniforms", dev, (B, k + 1))
    _need(draft_len, torch.int32, "draft_len", dev, (B,))
    _need(remaining, torch.int32, "remaining", dev, (B,))
    out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev) if out_tokens is None else out_tokens
    n_accept = torch.empty(B, dtype=torch.int32, device=dev) if n_accept is None else n_accept
    n_emit = torch.empty(B, dtype=torch.int32, device=dev) if n_emit is None else n_emit
    flags = torch.empty(B, dtype=torch.int32, device=dev) if flags is None else flags
    if out_residual is None and want_residual:
        out_residual = torch.empty((B, V), dtype=torch.float32, device=dev)
    _need(out_residual, torch.float32, "out_residual", dev, (B, V))
    _need(flags, torch.int32, "flags", dev, (B,))
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, k, V, dev, st)
    if top_k is None and top_p is None:
        _check(lib.spec_verify_sample(_p(target_logits), _DT[target_logits.dtype], float(temperature),
                                      _p(draft_probs), _p(draft_tokens), _p(uniforms), B, k, V, _p(draft_len),
                                      int(eos_id), _p(remaining), _p(out_tokens), _p(n_accept), _p(n_emit),
                                      _p(out_residual), _p(flags), ws.ptr(), ws.nbytes, st))
    else:
        _check(lib.spec_verify_sample_filtered(_p(target_logits), _DT[target_logits.dtype], float(temperature),
                                               _p(top_k), _p(top_p), _p(draft_probs), _p(draft_tokens),
                                               _p(uniforms), B, k, V, _p(draft_len), int(eos_id), _p(remaining),
                                               _p(out_tokens), _p(n_accept), _p(n_emit), _p(out_residual),
                                               _p(flags), ws.ptr(), ws.nbytes, st))
    return out_tokens, n_accept, n_emit, flags, out_residual


def spec_realign_kv(kv, length, pad, n_emit, len_new=None, pad_new=None, width_new=None, err=None,
                    workspace=None, stream=None):
    """kv [L, 2, B, H, S, D] (fp32/bf16/fp16) realigned in place.
    -> (len_new [B], pad_new [B], width_new [1], err [1]) int32 on the device."""
    lib = _lib.load()
    L, two, B, H, S, D = kv.shape
    if two != 2:
        raise ValueError("kv must be [L, 2, B, H, S, D]")
    dev = kv.device
    _need(kv, None, "kv", dev)
    if kv.dtype not in _DT:
        raise ValueError(f"unsupported kv dtype {kv.dtype}")
    for t, nm in ((length, "len"), (pad, "pad"), (n_emit, "n_emit")):
        _need(t, torch.int32, nm, dev, (B,))
    len_new = torch.empty(B, dtype=torch.int32, device=dev) if len_new is None else len_new
    pad_new = torch.empty(B, dtype=torch.int32, device=dev) if pad_new is None else pad_new
    width_new = torch.empty(1, dtype=torch.int32, device=dev) if width_new is None else width_new
    err = torch.empty(1, dtype=torch.int32, device=dev) if err is None else err
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, 0, 1, dev, st)
    _check(lib.spec_realign_kv(_p(kv), _DT[kv.dtype], L, B, H, S, D, _p(length), _p(pad), _p(n_emit),
                               _p(len_new), _p(pad_new), _p(width_new), _p(err), ws.ptr(), ws.nbytes, st))
    return len_new, pad_new, width_new, err


MAX_CACHES = 4


def spec_realign_kv_multi(caches, length, pad, n_emit, len_new=None, pad_new=None, width_new=None, err=None,
                          workspace=None, stream=None):
    """Realign several caches [L_c, 2, B, H_c, S, D_c] (e.g. target and draft)
    by one plan in one shift launch.
    -> (len_new [B], pad_new [B], width_new [1], err [1]) int32 on the device."""
    lib = _lib.load()
    if not 1 <= len(caches) <= MAX_CACHES:
        raise ValueError(f"1..{MAX_CACHES} caches")
    dev = caches[0].device
    B, S = caches[0].shape[2], caches[0].shape[4]
    descs = (_lib.KVCacheDesc * len(caches))()
    for i, kv in enumerate(caches):
        L, two, Bc, H, Sc, D = kv.shape
        if two != 2 or Bc != B or Sc != S:
            raise ValueError("every cache must be [L, 2, B, H, S, D] with the same B and S")
        _need(kv, None, f"caches[{i}]", dev)
        if kv.dtype not in _DT:
            raise ValueError(f"unsupported kv dtype {kv.dtype}")
        descs[i] = _lib.KVCacheDesc(kv.data_ptr(), _DT[kv.dtype], L, H, D)
    for t, nm in ((length, "len"), (pad, "pad"), (n_emit, "n_emit")):
        _need(t, torch.int32, nm, dev, (B,))
    len_new = torch.empty(B, dtype=torch.int32, device=dev) if len_new is None else len_new
    pad_new = torch.empty(B, dtype=torch.int32, device=dev) if pad_new is None else pad_new
    width_new = torch.empty(1, dtype=torch.int32, device=dev) if width_new is None else width_new
    err = torch.empty(1, dtype=torch.int32, device=dev) if err is None else err
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, 0, 1, dev, st)
    _check(lib.spec_realign_kv_multi(ctypes.cast(descs, ctypes.c_void_p), len(caches), B, S, _p(length), _p(pad),
                                     _p(n_emit), _p(len_new), _p(pad_new), _p(width_new), _p(err), ws.ptr(),
                                     ws.nbytes, st))
    return len_new, pad_new, width_new, err


def _cache_descs(caches, dev, B, S):
    if not 1 <= len(caches) <= MAX_CACHES:
        raise ValueError(f"1..{MAX_CACHES} caches")
    descs = (_lib.KVCacheDesc * len(caches))()
    for i, kv in enumerate(caches):
        L, two, Bc, H, Sc, D = kv.shape
        if two != 2 or Bc != B or Sc != S:
            raise ValueError("every cache must be [L, 2, B, H, S, D] with the same B and S")
        _need(kv, None, f"caches[{i}]", dev)
        if kv.dtype not in _DT:
            raise ValueError(f"unsupported kv dtype {kv.dtype}")
        descs[i] = _lib.KVCacheDesc(kv.data_ptr(), _DT[kv.dtype], L, H, D)
    return descs


def _round_outputs(B, k, dev, out_tokens, n_accept, n_emit, len_new, pad_new, width_new, err):
    e = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    return (e((B, k + 1)) if out_tokens is None else out_tokens, e(B) if n_accept is None else n_accept,
            e(B) if n_emit is None else n_emit, e(B) if len_new is None else len_new,
            e(B) if pad_new is None else pad_new, e(1) if width_new is None else width_new,
            e(1) if err is None else err)


def spec_round_greedy(target_logits, draft_tokens, caches, length, pad, pos, mask, draft_len=None, eos_id=-1,
                      remaining=None, out_tokens=None, n_accept=None, n_emit=None, len_new=None, pad_new=None,
                      width_new=None, err=None, workspace=None, stream=None):
    """One greedy round in one call: verify, realign every cache by one plan,
    rebuild pos / mask (pad_new must not alias pad).
    -> (out_tokens, n_accept, n_emit, len_new, pad_new, width_new, err)."""
    lib = _lib.load()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    S = caches[0].shape[4]
    _need(target_logits, None, "target_logits", dev)
    if target_logits.dtype not in _DT:
        raise ValueError(f"unsupported logits dtype {target_logits.dtype}")
    _need(draft_tokens, torch.int32, "draft_tokens", dev, (B, k))
    _need(draft_len, torch.int32, "draft_len", dev, (B,))
    _need(remaining, torch.int32, "remaining", dev, (B,))
    descs = _cache_descs(caches, dev, B, S)
    for t, nm in ((length, "len"), (pad, "pad")):
        _need(t, torch.int32, nm, dev, (B,))
    _need(pos, torch.int32, "pos", dev, (B, S))
    _need(mask, torch.uint8, "mask", dev, (B, S))
    outs = _round_outputs(B, k, dev, out_tokens, n_accept, n_emit, len_new, pad_new, width_new, err)
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, k, V, dev, st)
    o, na, ne, ln2, pd2, w2, er = outs
    _check(lib.spec_round_greedy(_p(target_logits), _DT[target_logits.dtype], B, k, V, _p(draft_tokens),
                                 _p(draft_len), int(eos_id), _p(remaining), ctypes.cast(descs, ctypes.c_void_p),
                                 len(caches), S, _p(length), _p(pad), _p(pos), _p(mask), _p(o), _p(na), _p(ne),
                                 _p(ln2), _p(pd2), _p(w2), _p(er), ws.ptr(), ws.nbytes, st))
    return outs


def spec_round_sample(target_logits, draft_probs, draft_tokens, uniforms, caches, length, pad, pos, mask,
                      temperature=1.0, top_k=None, top_p=None, draft_len=None, eos_id=-1, remaining=None,
                      out_tokens=None, n_accept=None, n_emit=None, out_residual=None, flags=None, len_new=None,
                      pad_new=None, width_new=None, err=None, workspace=None, stream=None):
    """One stochastic round in one call (top_k / top_p: None, a scalar or [B]
    device arrays, as in spec_verify_sample_filtered).
    -> (out_tokens, n_accept, n_emit, len_new, pad_new, width_new, err, flags, out_residual)."""
    lib = _lib.load()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    S = caches[0].shape[4]
    _need(target_logits, None, "target_logits", dev)
    if target_logits.dtype not in _DT:
        raise ValueError(f"unsupported logits dtype {target_logits.dtype}")
    if top_k is not None and not torch.is_tensor(top_k):
        top_k = torch.full((B,), int(top_k), dtype=torch.int32, device=dev)
    if top_p is not None and not torch.is_tensor(top_p):
        top_p = torch.full((B,), float(top_p), dtype=torch.float32, device=dev)
    _need(top_k, torch.int32, "top_k", dev, (B,))
    _need(top_p, torch.float32, "top_p", dev, (B,))
    _need(draft_probs, torch.float32, "draft_probs", dev, (B, k, V))
    _need(draft_tokens, torch.int32, "draft_tokens", dev, (B, k))
    _need(uniforms, torch.float32, "uniforms", dev, (B, k + 1))
    _need(draft_len, torch.int32, "draft_len", dev, (B,))
    _need(remaining, torch.int32, "remaining", dev, (B,))
    descs = _cache_descs(caches, dev, B, S)
    for t, nm in ((length, "len"), (pad, "pad")):
        _need(t, torch.int32, nm, dev, (B,))
    _need(pos, torch.int32, "pos", dev, (B, S))
    _need(mask, torch.uint8, "mask", dev, (B, S))
    outs = _round_outputs(B, k, dev, out_tokens, n_accept, n_emit, len_new, pad_new, width_new, err)
    flags = torch.empty(B, dtype=torch.int32, device=dev) if flags is None else flags
    _need(flags, torch.int32, "flags", dev, (B,))
    _need(out_residual, torch.float32, "out_residual", dev, (B, V))
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, k, V, dev, st)
    o, na, ne, ln2, pd2, w2, er = outs
    _check(lib.spec_round_sample(_p(target_logits), _DT[target_logits.dtype], float(temperature), _p(top_k),
                                 _p(top_p), _p(draft_probs), _p(draft_tokens), _p(uniforms), B, k, V, _p(draft_len),
                                 int(eos_id), _p(remaining), ctypes.cast(descs, ctypes.c_void_p), len(caches), S,
                                 _p(length), _p(pad), _p(pos), _p(mask), _p(o), _p(na), _p(ne), _p(out_residual),
                                 _p(flags), _p(ln2), _p(pd2), _p(w2), _p(er), ws.ptr(), ws.nbytes, st))
    return outs + (flags, out_residual)


def spec_rebuild_pos_mask(pad_new, pos, mask, pad_old=None, stream=None):
    """pos [B, S] int32 and mask [B, S] uint8 rewritten in place from pad_new."""
    lib = _lib.load()
    B, S = pos.shape
    dev = pos.device
    _need(pad_new, torch.int32, "pad_new", dev, (B,))
    _need(pad_old, torch.int32, "pad_old", dev, (B,))
    _need(pos, torch.int32, "pos", dev, (B, S))
    _need(mask, torch.uint8, "mask", dev, (B, S))
    st = _stream(stream, dev)
    _check(lib.spec_rebuild_pos_mask(B, S, _p(pad_old), _p(pad_new), _p(pos), _p(mask), st))
    return pos, mask


def spec_group_by_length(length, B, active=None, out_idx=None, out_count_equal=None, out_group_len=None,
                         stream=None):
    """length [N] int32 -> (idx [B], count_equal [1], group_len [1]) int32."""
    lib = _lib.load()
    (N,) = length.shape
    dev = length.device
    _need(length, torch.int32, "len", dev)
    _need(active, torch.uint8, "active", dev, (N,))
    out_idx = torch.empty(B, dtype=torch.int32, device=dev) if out_idx is None else out_idx
    out_count_equal = torch.empty(1, dtype=torch.int32, device=dev) if out_count_equal is None else out_count_equal
    out_group_len = torch.empty(1, dtype=torch.int32, device=dev) if out_group_len is None else out_group_len
    st = _stream(stream, dev)
    _check(lib.spec_group_by_length(N, _p(length), _p(active), int(B), _p(out_idx), _p(out_count_equal),
                                    _p(out_group_len), st))
    return out_idx, out_count_equal, out_group_len


MAX_POOL = 65536


def spec_commit_ragged(pool_len, idx, n_emit, S, err=None, stream=None):
    """pool_len [N] += n_emit at idx (in place). -> err [1] int32."""
    lib = _lib.load()
    dev = pool_len.device
    (N,) = pool_len.shape
    (B,) = idx.shape
    _need(pool_len, torch.int32, "pool_len", dev)
    _need(idx, torch.int32, "idx", dev)
    _need(n_emit, torch.int32, "n_emit", dev, (B,))
    err = torch.empty(1, dtype=torch.int32, device=dev) if err is None else err
    _check(lib.spec_commit_ragged(N, _p(pool_len), B, _p(idx), _p(n_emit), int(S), _p(err), _stream(stream, dev)))
    return err


def spec_repad_gather(pool, batch, idx, pool_len, len_out=None, pad_out=None, width_out=None, err=None,
                      workspace=None, stream=None):
    """pool [L,2,N,H,S,D] -> batch [L,2,B,H,S,D] (left-padded).
    -> (len [B], pad [B], width [1], err [1]) int32."""
    lib = _lib.load()
    L, two, N, H, S, D = pool.shape
    B = batch.shape[2]
    dev = pool.device
    if two != 2 or batch.shape != (L, 2, B, H, S, D) or batch.dtype != pool.dtype:
        raise ValueError("pool [L,2,N,H,S,D] and batch [L,2,B,H,S,D] of one dtype")
    _need(pool, None, "pool", dev)
    _need(batch, None, "batch", dev)
    _need(idx, torch.int32, "idx", dev, (B,))
    _need(pool_len, torch.int32, "pool_len", dev, (N,))
    len_out = torch.empty(B, dtype=torch.int32, device=dev) if len_out is None else len_out
    pad_out = torch.empty(B, dtype=torch.int32, device=dev) if pad_out is None else pad_out
    width_out = torch.empty(1, dtype=torch.int32, device=dev) if width_out is None else width_out
    err = torch.empty(1, dtype=torch.int32, device=dev) if err is None else err
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, 0, 1, dev, st)
    _check(lib.spec_repad_gather(_p(pool), _p(batch), _DT[pool.dtype], L, N, B, H, S, D, _p(idx), _p(pool_len),
                                 _p(len_out), _p(pad_out), _p(width_out), _p(err), ws.ptr(), ws.nbytes, st))
    return len_out, pad_out, width_out, err


def spec_unpad_scatter(batch, pool, idx, length, pad, pool_len, n_emit=None, err=None, workspace=None, stream=None):
    """batch [L,2,B,H,S,D] -> pool [L,2,N,H,S,D]; pool_len [N] updated in
    place.  n_emit [B] (optional): write back len + n_emit rows from a batch
    a round has just extended, without realigning it first.
    -> err [1] int32."""
    lib = _lib.load()
    L, two, N, H, S, D = pool.shape
    B = batch.shape[2]
    dev = pool.device
    if two != 2 or batch.shape != (L, 2, B, H, S, D) or batch.dtype != pool.dtype:
        raise ValueError("pool [L,2,N,H,S,D] and batch [L,2,B,H,S,D] of one dtype")
    _need(pool, None, "pool", dev)
    _need(batch, None, "batch", dev)
    _need(idx, torch.int32, "idx", dev, (B,))
    for t, nm in ((length, "len"), (pad, "pad")):
        _need(t, torch.int32, nm, dev, (B,))
    _need(pool_len, torch.int32, "pool_len", dev, (N,))
    _need(n_emit, torch.int32, "n_emit", dev, (B,))
    err = torch.empty(1, dtype=torch.int32, device=dev) if err is None else err
    st = _stream(stream, dev)
    ws = _workspace(workspace, B, 0, 1, dev, st)
    _check(lib.spec_unpad_scatter(_p(batch), _p(pool), _DT[pool.dtype], L, N, B, H, S, D, _p(idx), _p(length),
                                  _p(pad), _p(n_emit), _p(pool_len), _p(err), ws.ptr(), ws.nbytes, st))
    return err
