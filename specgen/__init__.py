"""Seeded synthetic inputs for batch speculative-decoding verification.

This module only generates inputs -- random logits with a controlled
acceptance structure, draft distributions, uniforms, prompt lengths and the
synthetic KV contents f(seq, token, pos, layer, k/v, head, d).  It holds none
of the method's arithmetic (no argmax, ratio test, residual, realignment or
position rebuild) and serves the CUDA path and the CPU oracle alike.

Workload shapes follow the five synthetic configurations the library is
measured on (see ``CONFIGS``); they stand in for the SpecBench / Multi30k
prompts and the model pairs the pages evaluate, none of which is used.
"""
from .np_gen import (  # noqa: F401
    CONFIGS,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    greedy_round_inputs,
    kv_row_values,
    prompt_lengths,
    round_inputs_blocked,
    sample_round_inputs,
    splitmix64,
)
