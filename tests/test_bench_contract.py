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


@pytest.mark.parametrize("cfg", [3, 5])
def test_structure_only_workloads_match_the_full_ones(cfg):
    """The bench's GQA and prefix-sharing lines run the workloads' own seeded
    structure (lengths, pool, operations, batch) with values drawn on the
    device; the structure must be the one the parity tests use."""
    import workloads

    kw = {"batch": 8} if cfg == 3 else {"groups": 2, "branches": 3, "prompt": 100, "n_long": 1,
                                        "long_ctx": 600}
    full = workloads.make(cfg, **kw)
    bare = workloads.make(cfg, values=False, **kw)
    assert bare.k_rows is None and bare.v_rows is None and bare.q is None
    assert bare.notes["value_rows"] == full.k_rows.shape[0]
    assert bare.notes["value_scale"] == 0.5
    assert (bare.free_order == full.free_order).all()
    assert bare.setup == full.setup and bare.step == full.step and bare.batch == full.batch
    assert bare.num_blocks == full.num_blocks
    assert bare.notes["context_lens"] == full.notes["context_lens"]
