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


def test_default_workload_is_the_greedy_headline():
    c = _params([])
    assert c["mode"] == "greedy" and (c["B"], c["k"], c["V"]) == (8, 5, 32000)
    assert c["logit_dtype"] == "bf16" and c["alpha"] == max(c["alphas"])


def test_overrides():
    c = _params(["--workload", "c5s", "--logit-dtype", "f32", "--layers", "1", "--top-p", "0.95"])
    assert c["mode"] == "sample" and c["logit_dtype"] == "f32" and c["L"] == 1 and c["top_p"] == 0.95
    assert _params(["--workload", "c4"])["k"] == 8
    assert _params(["--workload", "c4", "--k", "4"])["k"] == 4


def test_filters_only_on_stochastic_workloads():
    with pytest.raises(SystemExit):
        _params(["--workload", "c2", "--top-k", "50"])
