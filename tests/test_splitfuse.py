"""Token-budget composition (Dynamic SplitFuse): oracle pins and the C++ composer."""

import numpy as np
import pytest

from oracle import splitfuse
from tests.conftest import read_rows


def _run_scenario(compose, budget, decodes, prompt):
    """Compose passes until the prompt is consumed; return the chunk of each pass."""
    chunks, left = [], prompt
    while left > 0:
        _, c, _ = compose(budget, decodes, [left])
        chunks.append(c[0])
        left -= c[0]
    return chunks


@pytest.mark.parametrize("row", read_rows("chunk_budget_scenarios.txt"))
def test_oracle_reproduces_pages_scenarios(row):
    budget, decodes, prompt = int(row[1]), int(row[2]), int(row[3])
    want = [int(x) for x in row[4].split()]
    got = _run_scenario(splitfuse.compose, budget, decodes, prompt)
    assert got[:len(want)] == want
    assert sum(got) == prompt


@pytest.mark.parametrize("row", read_rows("chunk_budget_scenarios.txt"))
def test_cpp_composer_reproduces_pages_scenarios(lib, row):
    budget, decodes, prompt = int(row[1]), int(row[2]), int(row[3])
    want = [int(x) for x in row[4].split()]
    got = _run_scenario(lib.pkv_splitfuse_compose, budget, decodes, prompt)
    assert got[:len(want)] == want


def test_oracle_invariants_and_fusion():
    # short prompts are fused until the budget is full; only the last one served is split
    dec, chunks, used = splitfuse.compose(2048, 512, [100, 200, 3000, 50])
    assert dec == 512 and chunks == [100, 200, 1236, 0] and used == 2048
    # more decodes than budget: the first `budget` decodes run, prompts wait
    assert splitfuse.compose(8, 20, [5]) == (8, [0], 8)
    # not enough work: everything fits
    assert splitfuse.compose(100, 3, [4, 5]) == (3, [4, 5], 12)


def test_cpp_matches_oracle_on_random_inputs(lib):
    rng = np.random.default_rng(3)
    for _ in range(500):
        budget = int(rng.integers(0, 9000))
        nd = int(rng.integers(0, 600))
        rem = [int(x) for x in rng.integers(0, 5000, size=int(rng.integers(0, 12)))]
        assert lib.pkv_splitfuse_compose(budget, nd, rem) == splitfuse.compose(budget, nd, rem)


def test_cpp_rejects_negative_input(lib):
    with pytest.raises(lib.PagedKVError):
        lib.pkv_splitfuse_compose(-1, 0, [])
    with pytest.raises(lib.PagedKVError):
        lib.pkv_splitfuse_compose(10, 0, [3, -2])


@pytest.mark.parametrize("budget,seed", [(256, 1), (97, 2), (2048, 3), (17, 4)])
def test_scheduler_steps_equal_oracle_steps(lib, budget, seed):
    """The product's multi-step scheduler (C++ composer) plans the same steps as an
    independent restatement on the oracle composer."""
    import workloads
    from paged_kv_cache_51_gb300.splitfuse import Scheduler
    from tests.test_gpu_splitfuse_steps import _oracle_steps

    tr = workloads.serving_trace(seed=seed, n_requests=7, prompt_range=(1, 900),
                                 gen_range=(1, 9), d=64, hq=8, hkv=8)
    sched = Scheduler(tr, budget)
    n = 0
    for o in _oracle_steps(tr, budget):
        r = sched.next_step()
        while r is not None and not r[1]:
            r = sched.next_step()
        assert r == o
        assert sum(q for _, q in r[1]) <= budget
        n += 1
    assert sched.next_step() is None
    # every prompt token and every generated token was scheduled exactly once
    assert sched.prompt_done == tr.prompt_len and sched.generated == tr.gen_len
    assert n >= 1
