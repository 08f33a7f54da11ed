"""bench.py's reference arm on the CPU: the JSON line the driver reads.

`--impl reference` times the float64 oracle on one sequence of the headline
decode workload; its line carries the same metric, unit and direction as the
GPU arm, plus `impl`, `cpu_baseline` and an `e2e` object with no copies.
Ranks other than 0 print nothing.
"""

import argparse
import json

import pytest


def _args(**kw):
    a = argparse.Namespace(config=2, steps=1, warmup=1, gpus=1, impl="reference")
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_reference_line_has_the_contract_keys(capsys, monkeypatch):
    import bench

    monkeypatch.delenv("RANK", raising=False)
    assert bench.run_reference(_args()) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_other_ranks_print_nothing(capsys, monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(_args()) == 0
    assert capsys.readouterr().out == ""


def test_reference_covers_decode_configs_only():
    import bench

    with pytest.raises(SystemExit):
        bench.oracle_sample(4, 1)
