"""ctypes loader of libspecverify.so (the C ABI in include/specverify.h).

There is no fallback: if the library is missing or does not load, importing
the package's API raises, so no computation can silently run elsewhere.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

# Entry points declared in include/specverify.h, with their ctypes signatures.
_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "spec_workspace_bytes": ([_i32, _i32, _i32], _sz),
    "spec_workspace_init": ([_vp, _sz, _vp], _i32),
    "spec_status_str": ([_i32], ctypes.c_char_p),
    "spec_verify_greedy": ([_vp, _i32, _i32, _i32, _i32, _vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _sz,
                            _vp], _i32),
    "spec_verify_sample": ([_vp, _i32, _f32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, ctypes.c_int32, _vp, _vp, _vp,
                            _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "spec_verify_sample_filtered": ([_vp, _i32, _f32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, ctypes.c_int32,
                                     _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "spec_realign_kv": ([_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
                        _i32),
    "spec_rebuild_pos_mask": ([_i32, _i32, _vp, _vp, _vp, _vp, _vp], _i32),
    "spec_group_by_length": ([_i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp], _i32),
    "spec_verify_greedy_static": ([_vp, _i32, _i32, _i32, _i32, _vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp],
                                  _i32),
}

class KVCacheDesc(ctypes.Structure):
    """spec_kv_cache of include/specverify.h."""
    _fields_ = [("kv", ctypes.c_void_p), ("dt", ctypes.c_int), ("L", ctypes.c_int), ("H", ctypes.c_int),
                ("D", ctypes.c_int)]


SIGNATURES["spec_realign_kv_multi"] = ([_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
                                       _i32)
SIGNATURES["spec_round_greedy"] = ([_vp, _i32, _i32, _i32, _i32, _vp, _vp, ctypes.c_int32, _vp, _vp, _i32, _i32,
                                    _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32)
SIGNATURES["spec_round_sample"] = ([_vp, _i32, _f32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, ctypes.c_int32,
                                    _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _sz, _vp], _i32)

SIGNATURES["spec_commit_ragged"] = ([_i32, _vp, _i32, _vp, _vp, _i32, _vp, _vp], _i32)
SIGNATURES["spec_repad_gather"] = ([_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _sz, _vp], _i32)
SIGNATURES["spec_unpad_scatter"] = ([_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _sz, _vp], _i32)

_lib = None


def load():
    """Load the library once and attach the signatures; raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                "(nvcc for sm_103a) -- there is no CPU fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib
