"""The allocation-free entry point, spec_verify_greedy_static.

Some callers cannot allocate device memory when they call in -- a serving
loop that allows no allocation after start-up so its memory use stays fixed,
or a plugin that receives only its inputs and outputs.  For them the library
keeps its verification scratch in a device array of its own.  This file runs
last (it is collected after every other test file) and checks, through the C
ABI, that the variant returns exactly what spec_verify_greedy returns (greedy
tokens and counts are integers: the tests' tolerance is bit-exactness) on two
calls in a row, including a change of batch size between the calls.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_28_gb300 as sv
from specgen import greedy_round_inputs

pytestmark = pytest.mark.gpu


def _dev_logits(x, bf16):
    if bf16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


@pytest.mark.parametrize("shapes", [
    [(8, 5, 32000, "bf16", 0.8), (8, 5, 32000, "bf16", 0.5)],        # the same size twice
    [(256, 8, 128256, "bf16", 0.6), (4, 4, 1000, "f32", 0.7)],       # large then small batch
    [(3, 31, 8193, "f32", 0.9), (64, 8, 151936, "bf16", 0.7)],
])
def test_matches_workspace_entry_point_on_consecutive_calls(shapes):
    for i, (B, k, V, dt, alpha) in enumerate(shapes):
        x, d = greedy_round_inputs(B, k, V, alpha, 1.0, seed=40 + i, dtype=dt)
        xt = _dev_logits(x, dt == "bf16")
        dtd = torch.from_numpy(d).cuda()
        rem = torch.from_numpy(np.arange(B, dtype=np.int32) % (k + 3) - 1).cuda()
        a = sv.spec_verify_greedy_static(xt, dtd, eos_id=3, remaining=rem)
        b = sv.spec_verify_greedy(xt, dtd, eos_id=3, remaining=rem)
        for ga, gb in zip(a, b):
            assert torch.equal(ga, gb)
        assert int(a[2].sum().item()) > 0


def test_rejects_sizes_beyond_the_scratch():
    """Claimed sizes whose scratch exceeds the built-in array are refused on
    the host with SPEC_ESCRATCH (-6); nothing is launched, the outputs stay."""
    import ctypes

    from speculative_decoding_verification_28_gb300 import _lib

    lib = _lib.load()
    B, k, V = 4096, 31, 151936
    assert sv.spec_workspace_bytes(B, k, V) > sv.STATIC_SCRATCH_BYTES
    buf = torch.full((64,), 7, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    rc = lib.spec_verify_greedy_static(p, 1, B, k, V, p, None, -1, None, p, p, p, None)
    assert rc == -6
    torch.cuda.synchronize()
    assert (buf == 7).all()


def test_on_a_side_stream_of_the_current_device():
    """A caller's own stream (not the default one) on the current device is
    accepted; results as with the workspace entry point."""
    B, k, V = 16, 4, 5000
    x, d = greedy_round_inputs(B, k, V, 0.7, 1.0, seed=77, dtype="f32")
    xt, dtd = _dev_logits(x, False), torch.from_numpy(d).cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        a = sv.spec_verify_greedy_static(xt, dtd, stream=s)
    s.synchronize()
    b = sv.spec_verify_greedy(xt, dtd)
    for ga, gb in zip(a, b):
        assert torch.equal(ga, gb)


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two GPUs")
def test_tensors_on_another_device_than_the_current_one():
    """Tensors on cuda:1 while cuda:0 is current: the binding makes their
    device current, so the array of the right device is used; a raw call
    with a stream of another device is refused with SPEC_EINVAL (-1)."""
    import ctypes

    from speculative_decoding_verification_28_gb300 import _lib

    B, k, V = 8, 3, 3000
    x, d = greedy_round_inputs(B, k, V, 0.6, 1.0, seed=78, dtype="f32")
    with torch.cuda.device(0):
        xt, dtd = torch.from_numpy(x).to("cuda:1"), torch.from_numpy(d).to("cuda:1")
        a = sv.spec_verify_greedy_static(xt, dtd)
    b = sv.spec_verify_greedy(xt, dtd)
    for ga, gb in zip(a, b):
        assert torch.equal(ga, gb)
    lib = _lib.load()
    p = ctypes.c_void_p(xt.data_ptr())
    s1 = ctypes.c_void_p(torch.cuda.current_stream(1).cuda_stream)
    with torch.cuda.device(0):
        rc = lib.spec_verify_greedy_static(p, 0, B, k, V, ctypes.c_void_p(dtd.data_ptr()), None, -1, None,
                                           ctypes.c_void_p(a[0].data_ptr()), ctypes.c_void_p(a[1].data_ptr()),
                                           ctypes.c_void_p(a[2].data_ptr()), s1)
    assert rc == -1
