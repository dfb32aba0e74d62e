"""NumPy generators (CPU; small and medium sizes, and every CPU-only test).

The synthetic KV value f is a counter-based hash: Vigna's splitmix64 output
function applied to packed integers.  It is defined once here for the CPU and
restated in ``specgen/csrc/specgen.cu`` for the GPU from the same published
definition; the two are checked against each other by the GPU tests.
"""
from __future__ import annotations

import numpy as np

# Synthetic workload configurations.  Values not stated by the workload
# description are marked "reading" and recorded in the design notes.
CONFIGS = {
    # tiny greedy round
    "c1": dict(B=4, k=4, V=1000, logit_dtype="f32", sigma=1.0, alphas=(0.7,), prompt=(8, 64),
               L=2, H=4, D=64, S=256, kv_dtype="f32", rounds=20, modes=("greedy",)),
    # greedy batch-8 round, 7B-like shapes
    "c2": dict(B=8, k=5, V=32000, logit_dtype="bf16", sigma=2.0, alphas=(0.5, 0.8), prompt=(64, 512),
               L=32, H=32, D=128, S=1024, kv_dtype="bf16", rounds=20, modes=("greedy",)),
    # stochastic rejection-sampling verify; prompt range is a reading
    "c3": dict(B=32, k=4, V=128256, logit_dtype="f32", sigma=1.0, noise=0.5, alphas=(), prompt=(128, 1536),
               L=32, H=8, D=128, S=2048, kv_dtype="bf16", rounds=20, modes=("sample",)),
    # same-length grouping over a pool of 512; sigma 1 is a reading
    "c4": dict(N=512, B=64, ks=(4, 6, 8), V=151936, logit_dtype="bf16", sigma=1.0, alphas=(0.7,),
               pool_len=(128, 1024), L=28, H=4, D=128, S=2048, kv_dtype="bf16", rounds=20,
               modes=("greedy",)),
    # worst-case realignment sweep; sigma 1 is a reading
    "c5": dict(B=256, k=8, V=128256, logit_dtype="bf16", sigma=1.0, noise=0.5, alphas=(0.3, 0.6, 0.9),
               prompt=(256, 3072), L=32, H=8, D=128, S=4096, kv_dtype="bf16", rounds=50,
               modes=("greedy", "sample")),
}

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def splitmix64(x):
    """Vigna's splitmix64 output function of the state x (uint64, wrapping)."""
    with np.errstate(over="ignore"):
        z = np.asarray(x, dtype=np.uint64) + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def kv_row_values(seq, tok, pos, L, H, D):
    """f(seq, tok, pos, l, c, h, d) for all (l, c, h, d): float32 [L, 2, H, D].

    f = ((splitmix64(splitmix64(key1) ^ key2) >> 56) - 128) / 128 with
    key1 = seq << 36 | tok << 16 | pos and key2 = l << 20 | c << 19 | h << 10 | d:
    a multiple of 1/128 in [-1, 1), exact in fp32, bf16 and fp16."""
    key1 = (np.uint64(seq) << np.uint64(36)) | (np.uint64(tok) << np.uint64(16)) | np.uint64(pos)
    h1 = splitmix64(key1)
    l = np.arange(L, dtype=np.uint64)[:, None, None, None]
    c = np.arange(2, dtype=np.uint64)[None, :, None, None]
    h = np.arange(H, dtype=np.uint64)[None, None, :, None]
    d = np.arange(D, dtype=np.uint64)[None, None, None, :]
    key2 = (l << np.uint64(20)) | (c << np.uint64(19)) | (h << np.uint64(10)) | d
    top = (splitmix64(h1 ^ key2) >> np.uint64(56)).astype(np.int64)
    return ((top - 128).astype(np.float32) / np.float32(128.0)).astype(np.float32)


def f32_to_bf16_bits(x):
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rnd = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((b + rnd) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed):
    return seed if isinstance(seed, np.random.Generator) else np.random.default_rng(seed)


def prompt_lengths(B, lo, hi, seed):
    """Prompt lengths uniform in [lo, hi]."""
    return _rng(seed).integers(lo, hi + 1, size=B).astype(np.int32)


def _to_storage(x, dtype):
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16)
    raise ValueError(dtype)


def _storage_values(s, dtype):
    if dtype == "bf16":
        return bf16_bits_to_f32(s)
    return s.astype(np.float32)


def greedy_round_inputs(B, k, V, alpha, sigma, seed, dtype="f32"):
    """Target logits [B, k+1, V] ~ N(0, sigma) (sigma read as the standard
    deviation) in storage dtype, and draft tokens [B, k].

    Acceptance is iid with probability alpha per proposal: the proposal's
    logit is raised to the row maximum + 1 (so it is the unique maximum), or,
    otherwise, the proposal is a uniform token whose logit is lowered below the
    row minimum (so it cannot be a maximum).  The bonus row k is left as drawn.
    """
    rng = _rng(seed)
    x = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(sigma)
    x = _storage_values(_to_storage(x, dtype), dtype).copy()
    d = rng.integers(0, V, size=(B, k)).astype(np.int32)
    if k > 0 and V > 1:
        coin = rng.random((B, k)) < alpha
        rows = x[:, :k, :]
        bi, ji = np.meshgrid(np.arange(B), np.arange(k), indexing="ij")
        up = rows.max(axis=-1) + np.float32(1.0)
        down = rows.min(axis=-1) - np.float32(1.0)
        rows[bi, ji, d] = np.where(coin, up, down)
    return _to_storage(x, dtype), d


def sample_round_inputs(B, k, V, noise, seed, dtype="f32", sigma=1.0):
    """Stochastic-verify inputs: target logits x ~ N(0, sigma) [B, k+1, V] in
    storage dtype; draft logits x[:, :k] + N(0, noise); draft distribution
    q = softmax(draft logits) computed in fp32 [B, k, V]; draft tokens drawn
    from q with a seeded uniform; uniforms [B, k+1] in [0, 1)."""
    rng = _rng(seed)
    x = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(sigma)
    xs = _to_storage(x, dtype)
    dl = x[:, :k, :] + rng.standard_normal((B, k, V), dtype=np.float32) * np.float32(noise)
    dl = dl - dl.max(axis=-1, keepdims=True)
    e = np.exp(dl, dtype=np.float32)
    q = (e / e.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)
    c = np.cumsum(q.astype(np.float64), axis=-1)
    ud = rng.random((B, k))
    d = np.empty((B, k), np.int32)
    for b in range(B):
        for j in range(k):
            t = int(np.searchsorted(c[b, j], ud[b, j] * c[b, j, -1], side="right"))
            t = min(t, V - 1)
            while q[b, j, t] == 0.0 and t > 0:
                t -= 1
            d[b, j] = t
    u = rng.random((B, k + 1), dtype=np.float32)
    return xs, q, d, u


def round_inputs_blocked(mode, B, k, V, seed, dtype, alpha=None, sigma=1.0, noise=None, threads=8, block=32):
    """greedy_round_inputs / sample_round_inputs for large batches, made on
    host threads: sequences in blocks of `block`, block i drawn from the
    generator seeded with [seed, i].  The same recipe per sequence; the
    random stream differs from the single-generator form."""
    from concurrent.futures import ThreadPoolExecutor

    starts = list(range(0, B, block))

    def part(i):
        nb = min(block, B - starts[i])
        rng = np.random.default_rng([int(seed), i])
        if mode == "greedy":
            return greedy_round_inputs(nb, k, V, alpha, sigma, rng, dtype=dtype)
        return sample_round_inputs(nb, k, V, noise, rng, dtype=dtype, sigma=sigma)

    with ThreadPoolExecutor(max(1, int(threads))) as ex:
        parts = list(ex.map(part, range(len(starts))))
    return tuple(np.concatenate([p[j] for p in parts]) for j in range(len(parts[0])))
