"""Multi-step SplitFuse: a request stream through the pool, append and varlen attention.

The product side plans steps with paged_kv_cache_51_gb300.splitfuse.Scheduler
(the C++ composer); the oracle side runs its own scheduler below (oracle
composer, oracle pool, oracle cache, float64 attention).  Every step's batch
must be the same on both sides, every step's output within tolerance, and the
caches byte-identical at the end.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import attention, splitfuse  # noqa: E402
from oracle.run import OracleState  # noqa: E402
from tests.gpu_parity import TOL, cache_bytes_equal, out_f64  # noqa: E402

pytestmark = pytest.mark.gpu


def _oracle_steps(trace, budget):
    """Independent restatement of the step loop: decodes first, then prompt chunks."""
    n = len(trace.prompt_len)
    done, gen, step_no = [0] * n, [0] * n, 0
    while True:
        dec = [i for i in range(n) if done[i] == trace.prompt_len[i] and gen[i] < trace.gen_len[i]]
        wait = [i for i in range(n) if trace.arrival[i] <= step_no and done[i] < trace.prompt_len[i]]
        n_dec, chunks, _ = splitfuse.compose(budget, len(dec),
                                             [trace.prompt_len[i] - done[i] for i in wait])
        ops, batch, qrows = [], [], []
        for i in dec[:n_dec]:
            pos = trace.prompt_len[i] + gen[i]
            ops.append(("grow", i, 1, trace.row_offset[i] + pos))
            batch.append((i, 1))
            qrows.append(trace.row_offset[i] + pos)
            gen[i] += 1
        for i, c in zip(wait, chunks):
            if c:
                pos = done[i]
                ops.append(("add", i, c, trace.row_offset[i]) if pos == 0
                           else ("grow", i, c, trace.row_offset[i] + pos))
                batch.append((i, c))
                qrows += range(trace.row_offset[i] + pos, trace.row_offset[i] + pos + c)
                done[i] += c
        step_no += 1
        if not batch:
            if all(done[i] == trace.prompt_len[i] and gen[i] == trace.gen_len[i] for i in range(n)):
                return
            continue
        yield ops, batch, qrows


@pytest.mark.parametrize("budget,seed", [(256, 1), (97, 2)])
def test_multi_step_splitfuse_matches_oracle(lib, budget, seed):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import runner
    from paged_kv_cache_51_gb300.splitfuse import Scheduler

    lib.device_error(clear=True)
    tr = workloads.serving_trace(seed=seed, n_requests=6, prompt_range=(20, 700),
                                 gen_range=(1, 6))
    w = workloads.Workload("serving", tr.dtype, tr.num_q_heads, tr.num_kv_heads, tr.head_dim,
                           tr.block_size, tr.num_blocks, tr.free_order, [], [], [], tr.q_rows,
                           tr.k_rows, tr.v_rows)
    dc = runner.DeviceCache(w)
    ost = OracleState(w)
    sched = Scheduler(tr, budget)
    tmax, tmean = TOL["bf16"]
    n_steps = 0
    for o_ops, o_batch, o_qrows in _oracle_steps(tr, budget):
        r = sched.next_step()
        while r is not None and not r[1]:
            r = sched.next_step()
        assert r is not None
        ops, batch, qrows = r
        assert (ops, batch, qrows) == (o_ops, o_batch, o_qrows)
        assert sum(q for _, q in batch) <= budget
        # product
        step = runner.Step(dc, dc.plan_step(ops), batch=batch, q=tr.q_rows[qrows])
        out = step.run()
        torch.cuda.synchronize()
        # oracle
        for op in ops:
            ost._apply(op, record=True)
        seqs = [s for s, _ in batch]
        width = max(len(ost.pool.block_table(s)) for s in seqs)
        bt = np.full((len(seqs), width), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            t = ost.pool.block_table(s)
            bt[i, :len(t)] = t
        ctx = np.array([ost.pool.context_len(s) for s in seqs])
        qsl = np.concatenate([[0], np.cumsum([q for _, q in batch])])
        ref = attention.varlen(tr.q_rows[qrows], ost.k_cache, ost.v_cache, bt, qsl, ctx,
                               tr.block_size, tr.dtype)
        d = np.abs(out_f64(out) - ref)
        assert float(d.max()) <= tmax and float(d.mean()) <= tmean, (n_steps, float(d.max()))
        n_steps += 1
    assert sched.next_step() is None
    assert n_steps >= 4
    assert lib.device_error() == 0
    assert cache_bytes_equal(dc.k_cache, ost.k_cache)
    assert cache_bytes_equal(dc.v_cache, ost.v_cache)
