"""Host-side pieces of bench.py: the all-cores oracle baseline (no GPU)."""
import pytest

import bench


def test_all_cores_oracle_counts_every_worker():
    value, wall, n = bench.oracle_all_cores("tiny", [2, 3], warmup=1)
    assert n == 2 and wall > 0
    # each tiny sample is the whole 64-token batch: 5 samples of 64 tokens in `wall` seconds
    assert value == pytest.approx(5 * 64 / wall, rel=1e-9)


def test_all_cores_oracle_reports_a_failed_worker():
    with pytest.raises(RuntimeError, match="all-cores oracle run failed"):
        bench.oracle_all_cores("no_such_workload", [1, 1], warmup=1)


def test_reference_line_uses_the_host_cores(capsys):
    import types
    args = types.SimpleNamespace(config="tiny", steps=3, warmup=1, gpus=1)
    bench.run_reference(args, 1, 0)
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3
    assert line["cpu_baseline"]["cores"] == min(bench.host_cores(), 3)
    assert line["value"] == line["cpu_baseline"]["value"] == line["e2e"]["value"] > 0
