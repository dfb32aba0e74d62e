"""bench.py's workload assembly (CPU only): the configured workloads and
their overrides."""
import sys

import pytest


def _params(argv):
    import bench

    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.workload_params(bench.parse())
    finally:
        sys.argv = old


def test_default_workload_is_the_worst_case_batch():
    """The default line is config 5 (B=256, k=8, V=128256 bf16, 128 GiB KV),
    greedy at the middle of its acceptance sweep."""
    c = _params([])
    assert c["mode"] == "greedy" and (c["B"], c["k"], c["V"]) == (256, 8, 128256)
    assert c["logit_dtype"] == "bf16" and c["alpha"] == 0.6
    assert (c["L"], c["H"], c["S"], c["D"]) == (32, 8, 4096, 128)
    assert _params(["--workload", "c2"])["alpha"] == 0.8  # elsewhere: the heavier realignment


def test_cpu_legs_sample_layers_of_large_caches_only():
    import bench

    c5 = _params([])
    assert bench.kv_bytes(c5) == 128 << 30 and bench.cpu_layers(c5) == 1
    assert "scaled by 32" in bench.cpu_sample_text(c5)
    c3 = _params(["--workload", "c3"])
    assert bench.cpu_layers(c3) == c3["L"]


def _args(argv):
    import bench

    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def test_reference_arm_runs_the_oracle_with_the_same_config():
    """--impl reference on a tiny workload: one JSON line whose config object
    is the one our arm prints."""
    import bench

    a = _args(["--impl", "reference", "--workload", "c1", "--steps", "2", "--warmup", "1"])
    c = bench.workload_params(a)
    line = bench.run_reference(a, c)
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "rounds/s"
    assert line["config"] == bench.bench_config(a, c, 1)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_layer_sample_scales_the_realignment():
    """A cache above the CPU limit: the oracle realigns its first layer and
    the time is scaled by the layer count (checked on a shrunken limit)."""
    import numpy as np

    import bench

    a = _args(["--impl", "reference", "--workload", "c1"])
    c = bench.workload_params(a)
    old = bench.CPU_FULL_CACHE_BYTES
    bench.CPU_FULL_CACHE_BYTES = 1 << 10
    try:
        assert bench.cpu_layers(c) == 1
        kv = bench.host_cache(c)
        assert kv.shape == (1, 2, c["B"], c["H"], c["S"], c["D"])
        t, (ln, pad) = bench.oracle_rounds(c, 3, 5, kv, lambda sd: bench.host_inputs(c, sd))
        assert t > 0 and np.all(ln + pad == (ln + pad)[0])
    finally:
        bench.CPU_FULL_CACHE_BYTES = old


def test_overrides():
    c = _params(["--workload", "c5s", "--logit-dtype", "f32", "--layers", "1", "--top-p", "0.95"])
    assert c["mode"] == "sample" and c["logit_dtype"] == "f32" and c["L"] == 1 and c["top_p"] == 0.95
    assert _params(["--workload", "c4"])["k"] == 8
    assert _params(["--workload", "c4", "--k", "4"])["k"] == 4


def test_filters_only_on_stochastic_workloads():
    with pytest.raises(SystemExit):
        _params(["--workload", "c2", "--top-k", "50"])
