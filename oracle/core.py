"""ctypes marshalling for the C oracle (test infrastructure only).

Every function takes and returns numpy arrays; none of them computes anything
itself -- the definitions live in ``oracle.c`` with their citations.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DT_F32, DT_BF16, DT_F16 = 0, 1, 2

MUTANTS = {
    "tie_highest": 1,
    "row_shift": 2,
    "resample_from_p": 3,
    "bonus_from_draft": 4,
    "no_clamp": 5,
    "cdf_ge": 6,
    "skip_kv_shift": 7,
    "stale_positions": 8,
    "bonus_always": 9,
    "shift_one_short": 10,
    "topk_strict": 11,
    "topp_below": 12,
    "ratio_unfiltered": 13,
    "resid_unfiltered": 14,
    "topp_first": 15,
    "zero_sign_order": 16,
}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (IEEE arithmetic, no fast-math),
    with OpenMP for the loops over sequences and slabs when the compiler has it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC]
        try:
            subprocess.check_call(base + ["-fopenmp", "-lm"], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base + ["-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_set_mutant.argtypes = [i32]
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_threads_available.restype = i32
            lib.oracle_verify_greedy.argtypes = [vp, i32, i32, i32, i32, vp, vp, ctypes.c_int32, vp, vp, vp, vp]
            f32 = ctypes.c_float
            lib.oracle_verify_sample.argtypes = [
                vp, i32, f64, vp, vp, vp, i32, i32, i32, vp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp,
            ]
            lib.oracle_softmax_row.argtypes = [vp, i32, i64, i32, f64, i32, f32, vp]
            lib.oracle_softmax_row.restype = i32
            lib.oracle_filter_cut.argtypes = [vp, i32, i64, i32, f32, i32, f32, vp]
            lib.oracle_filter_cut.restype = f64
            lib.oracle_realign_plan.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_realign_plan.restype = i32
            lib.oracle_shift_slab.argtypes = [vp, i64, i32, i32, i32]
            lib.oracle_realign_kv.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_realign_kv.restype = i32
            lib.oracle_rebuild_pos_mask.argtypes = [i32, i32, vp, vp, vp]
            lib.oracle_group_by_length.argtypes = [i32, vp, vp, i32, vp, vp, vp]
            lib.oracle_commit_ragged.argtypes = [i32, vp, i32, vp, vp, i32]
            lib.oracle_commit_ragged.restype = i32
            lib.oracle_repad_gather.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
            lib.oracle_repad_gather.restype = i32
            lib.oracle_unpad_scatter.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp]
            lib.oracle_unpad_scatter.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _logits(x, dt):
    """Logits as a contiguous array of their storage type: fp32 values, or the
    uint16 bit patterns of bf16 / fp16."""
    if dt == DT_F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dt == DT_F16 and x.dtype == np.float16:
        return np.ascontiguousarray(x).view(np.uint16)
    return np.ascontiguousarray(x, dtype=np.uint16)


@contextlib.contextmanager
def mutant(name: str):
    """Plant one deliberate mistake in the oracle for the duration of a block
    (used only to show that the pins catch it)."""
    lib = _load()
    lib.oracle_set_mutant(MUTANTS[name])
    try:
        yield
    finally:
        lib.oracle_set_mutant(0)


def set_threads(n: int) -> None:
    """Threads for the oracle's loops over sequences and cache slabs (1 by
    default); results do not depend on it."""
    _load().oracle_set_threads(int(n))


def threads_available() -> int:
    """Processors OpenMP sees (1 when the oracle was built without it)."""
    return int(_load().oracle_threads_available())


@contextlib.contextmanager
def threads(n: int):
    """set_threads(n) for the duration of a block."""
    set_threads(n)
    try:
        yield
    finally:
        set_threads(1)


def verify_greedy(logits, dt, draft_tokens, draft_len=None, eos_id=-1, remaining=None):
    """logits [B,k+1,V] -> (out_tokens [B,k+1], n_accept [B], n_emit [B])."""
    lib = _load()
    x = _logits(logits, dt)
    B, k1, V = x.shape
    k = k1 - 1
    d = _c(draft_tokens, np.int32).reshape(B, k)
    dl = _c(draft_len, np.int32)
    rem = _c(remaining, np.int32)
    out = np.empty((B, k + 1), np.int32)
    na = np.empty(B, np.int32)
    ne = np.empty(B, np.int32)
    lib.oracle_verify_greedy(_ptr(x), dt, B, k, V, _ptr(d), _ptr(dl), int(eos_id), _ptr(rem),
                             _ptr(out), _ptr(na), _ptr(ne))
    return out, na, ne


def _per_seq(v, B, dtype):
    """None, a scalar for every sequence, or a [B] array."""
    if v is None:
        return None
    a = np.asarray(v, dtype=dtype)
    return np.ascontiguousarray(np.broadcast_to(a, (B,)), dtype=dtype)


def verify_sample(logits, dt, draft_probs, draft_tokens, uniforms, temperature=1.0,
                  draft_len=None, eos_id=-1, remaining=None, want_residual=False, top_k=None, top_p=None):
    """-> (out_tokens, n_accept, n_emit, flags, residual [B,V] fp64 or None).
    top_k / top_p: None (off), a scalar, or per-sequence [B] (int32 / fp32)."""
    lib = _load()
    x = _logits(logits, dt)
    B, k1, V = x.shape
    k = k1 - 1
    q = _c(draft_probs, np.float32).reshape(B, k, V)
    d = _c(draft_tokens, np.int32).reshape(B, k)
    u = _c(uniforms, np.float32).reshape(B, k + 1)
    dl = _c(draft_len, np.int32)
    rem = _c(remaining, np.int32)
    out = np.empty((B, k + 1), np.int32)
    na = np.empty(B, np.int32)
    ne = np.empty(B, np.int32)
    fl = np.empty(B, np.uint32)
    res = np.full((B, V), np.nan, np.float64) if want_residual else None
    tk, tp = _per_seq(top_k, B, np.int32), _per_seq(top_p, B, np.float32)
    lib.oracle_verify_sample(_ptr(x), dt, float(temperature), _ptr(q), _ptr(d), _ptr(u), B, k, V,
                             _ptr(dl), int(eos_id), _ptr(rem), _ptr(out), _ptr(na), _ptr(ne),
                             _ptr(res), _ptr(fl), _ptr(tk), _ptr(tp))
    return out, na, ne, fl, res


def softmax_row(logits, dt, row, temperature=1.0, top_k=0, top_p=1.0):
    """fp64 processed distribution (softmax, then top-k / top-p) of row
    ``row`` of a [rows, V] view of the logits."""
    lib = _load()
    x = _logits(logits, dt)
    V = x.shape[-1]
    p = np.empty(V, np.float64)
    bad = lib.oracle_softmax_row(_ptr(x), dt, int(row), V, float(temperature), int(top_k), float(top_p), _ptr(p))
    return p, bool(bad)


def filter_cut(logits, dt, row, temperature=1.0, top_k=0, top_p=1.0):
    """Smallest logit top-k / top-p keep in row ``row`` (-inf: no filter)."""
    return filter_info(logits, dt, row, temperature, top_k, top_p)[0]


def filter_info(logits, dt, row, temperature=1.0, top_k=0, top_p=1.0):
    """(cut, margin, total, undecided) of row ``row``: the smallest kept
    logit; min |A - top_p M| over the two top-p decisions next to the cut and
    the kept total M, both in units of the top token's mass (margin +inf
    without top-p); whether a decision fell inside the oracle's fp64 error
    band."""
    lib = _load()
    x = _logits(logits, dt)
    info = np.zeros(3, np.float64)
    cut = lib.oracle_filter_cut(_ptr(x), dt, int(row), x.shape[-1], float(temperature), int(top_k), float(top_p),
                                _ptr(info))
    return cut, float(info[0]), float(info[1]), bool(info[2])


def realign_plan(S, length, pad, n_emit):
    """-> (status, len_new, pad_new, width_new)."""
    lib = _load()
    ln, pd, ne = (_c(a, np.int32) for a in (length, pad, n_emit))
    B = ln.shape[0]
    len_new = np.zeros(B, np.int32)
    pad_new = np.zeros(B, np.int32)
    w = np.zeros(1, np.int32)
    st = lib.oracle_realign_plan(B, S, _ptr(ln), _ptr(pd), _ptr(ne), _ptr(len_new), _ptr(pad_new), _ptr(w))
    return st, len_new, pad_new, int(w[0])


def shift_slab(slab, row_bytes, pad_old, pad_new, n_rows):
    """In-place memmove of one slab (a contiguous uint8 array)."""
    lib = _load()
    assert slab.flags.c_contiguous
    lib.oracle_shift_slab(_ptr(slab), int(row_bytes), int(pad_old), int(pad_new), int(n_rows))


def realign_kv(kv, length, pad, n_emit):
    """In place on kv [L,2,B,H,S,D] (any 2- or 4-byte dtype).
    -> (status, len_new, pad_new, width_new)."""
    lib = _load()
    assert kv.flags.c_contiguous and kv.ndim == 6
    L, two, B, H, S, D = kv.shape
    assert two == 2
    ln, pd, ne = (_c(a, np.int32) for a in (length, pad, n_emit))
    len_new = np.zeros(B, np.int32)
    pad_new = np.zeros(B, np.int32)
    w = np.zeros(1, np.int32)
    st = lib.oracle_realign_kv(_ptr(kv), kv.dtype.itemsize, L, B, H, S, D, _ptr(ln), _ptr(pd), _ptr(ne),
                               _ptr(len_new), _ptr(pad_new), _ptr(w))
    return st, len_new, pad_new, int(w[0])


def rebuild_pos_mask(S, pad_new, pos=None, mask=None):
    """-> (pos [B,S] int32, mask [B,S] uint8), written in place when given."""
    lib = _load()
    pn = _c(pad_new, np.int32)
    B = pn.shape[0]
    if pos is None:
        pos = np.zeros((B, S), np.int32)
    if mask is None:
        mask = np.zeros((B, S), np.uint8)
    lib.oracle_rebuild_pos_mask(B, S, _ptr(pn), _ptr(pos), _ptr(mask))
    return pos, mask


def group_by_length(length, B, active=None):
    """-> (idx [B], count_equal, group_len)."""
    lib = _load()
    ln = _c(length, np.int32)
    act = _c(active, np.uint8)
    idx = np.zeros(B, np.int32)
    ce = np.zeros(1, np.int32)
    gl = np.zeros(1, np.int32)
    lib.oracle_group_by_length(ln.shape[0], _ptr(ln), _ptr(act), B, _ptr(idx), _ptr(ce), _ptr(gl))
    return idx, int(ce[0]), int(gl[0])


def commit_ragged(pool_len, idx, n_emit, S):
    """In place on pool_len [N]; -> status."""
    lib = _load()
    assert pool_len.dtype == np.int32 and pool_len.flags.c_contiguous
    ix, ne = _c(idx, np.int32), _c(n_emit, np.int32)
    return lib.oracle_commit_ragged(pool_len.shape[0], _ptr(pool_len), ix.shape[0], _ptr(ix), _ptr(ne), int(S))


def repad_gather(pool, batch, idx, pool_len):
    """pool [L,2,N,H,S,D] -> batch [L,2,B,H,S,D] in place.
    -> (status, len [B], pad [B], width)."""
    lib = _load()
    L, _, N, H, S, D = pool.shape
    B = batch.shape[2]
    assert batch.dtype.itemsize == pool.dtype.itemsize and batch.flags.c_contiguous
    ix, pl = _c(idx, np.int32), _c(pool_len, np.int32)
    ln = np.zeros(B, np.int32)
    pd = np.zeros(B, np.int32)
    w = np.zeros(1, np.int32)
    st = lib.oracle_repad_gather(_ptr(pool), _ptr(batch), pool.dtype.itemsize, L, N, B, H, S, D, _ptr(ix), _ptr(pl),
                                 _ptr(ln), _ptr(pd), _ptr(w))
    return st, ln, pd, int(w[0])


def unpad_scatter(batch, pool, idx, length, pad, pool_len):
    """batch -> pool in place; pool_len [N] updated in place. -> status."""
    lib = _load()
    L, _, N, H, S, D = pool.shape
    B = batch.shape[2]
    assert pool.flags.c_contiguous and pool_len.dtype == np.int32
    ix, ln, pd = _c(idx, np.int32), _c(length, np.int32), _c(pad, np.int32)
    return lib.oracle_unpad_scatter(_ptr(batch), _ptr(pool), pool.dtype.itemsize, L, N, B, H, S, D, _ptr(ix),
                                    _ptr(ln), _ptr(pd), _ptr(pool_len))
