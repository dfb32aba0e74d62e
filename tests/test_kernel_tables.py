"""Constant tables compiled into the kernels, checked against the
mathematics (CPU only; the source text is read, nothing is launched).

kExp2Tab64 (verify_filter.cuh) holds 2^(k/64), k = 0..63, as float pairs for
the top-p decision weights (Tang's table-driven exponential): hi must be
2^(k/64) rounded to nearest fp32, and hi + lo within 2^-48 of it relative.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "speculative_decoding_verification_28_gb300", "csrc", "verify_filter.cuh")


def _c_float(tok):
    tok = tok.strip().rstrip("f")
    return float.fromhex(tok) if "0x" in tok else float(tok)


def test_exp2_table_is_two_to_the_k_over_64():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    text = open(SRC).read()
    body = re.search(r"kExp2Tab64\[64\]\s*=\s*\{(.*?)\};", text, re.S).group(1)
    pairs = re.findall(r"\{([^{},]+),([^{},]+)\}", body)
    assert len(pairs) == 64
    for k, (h, l) in enumerate(pairs):
        hi, lo = _c_float(h), _c_float(l)
        v = mp.mpf(2) ** (mp.mpf(k) / 64)
        assert np.float32(hi) == hi and np.float32(lo) == lo  # both exact fp32 values
        assert hi == float(np.float32(float(v))), k  # hi: nearest fp32
        assert abs((mp.mpf(hi) + mp.mpf(lo)) - v) <= v * mp.mpf(2) ** -48, k
