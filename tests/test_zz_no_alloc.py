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
