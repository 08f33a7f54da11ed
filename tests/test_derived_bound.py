"""The derived parity bound (tests/gpu_parity.py) on CPU: wide enough for fp32
arithmetic, narrow enough to reject the plausible mistakes of a kernel.

The GPU tests with large scores compare against this bound instead of the
stated tolerance alone.  Here the same stress inputs are run through a float32
emulation of the kernels' arithmetic (scores and weights in fp32, P rounded to
bf16 for the P.V product where the bf16 kernels round it), which must stay
inside the bound, and through the float64 definition with one planted mistake
each, which must not.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle.attention import gather_sequence  # noqa: E402
from oracle.numerics import widen  # noqa: E402
from oracle.run import execute  # noqa: E402
from tests.gpu_parity import derived_bound  # noqa: E402


def _bf16_round(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).float().numpy()


def _emulate(w, ost, mistake=None):
    """Attention of every query row in float32 (or float64 with a planted mistake)."""
    bt, ctx, qsl = ost.batch_metadata()
    D = w.head_dim
    g = w.num_q_heads // w.num_kv_heads
    scale = 1.0 / math.sqrt(D)
    ft = np.float64 if mistake else np.float32
    qf = widen(w.q, w.dtype).astype(ft)
    out = np.full(qf.shape, np.nan)
    for s in range(len(ctx)):
        r0, r1 = int(qsl[s]), int(qsl[s + 1])
        c = int(ctx[s])
        kd = widen(gather_sequence(ost.k_cache, bt[s], c, w.block_size), w.dtype).astype(ft)
        vd = widen(gather_sequence(ost.v_cache, bt[s], c, w.block_size), w.dtype).astype(ft)
        for r in range(r0, r1):
            n = c - (r1 - r) + 1
            if mistake == "causal_plus_one":
                n += 1                                  # sees the next (future) key too
            sc = ft(scale) if mistake != "scale_1_over_d" else ft(1.0 / D)
            for h in range(w.num_q_heads):
                kvh = h // g if mistake != "wrong_kv_head" else (h // g + 1) % w.num_kv_heads
                k, v = kd[:n, kvh], vd[:n, kvh]
                x = (k @ qf[r, h]) * sc
                p = np.exp(x - x.max()).astype(ft)
                l = p.sum(dtype=ft)
                pv = _bf16_round(p) if (w.dtype == "bf16" and not mistake) else p
                o = (pv @ v) / l
                if w.dtype == "bf16" and not mistake:
                    o = _bf16_round(o)
                out[r, h] = o
    return out


CASES = {
    "decode_f32_large_scores": lambda: workloads.random_decode(
        4, "f32", 8, 8, 64, 16, [300, 1200], scale=1.0, q_scale=64.0),
    "varlen_bf16_large_scores": lambda: workloads.random_varlen(
        15, "bf16", 8, 2, 128, 16, [(300, 40), (0, 64)], scale=0.5, q_scale=64.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fp32_emulation_is_inside_the_bound(case):
    w = CASES[case]()
    ost, ref = execute(w)
    live = ~np.isnan(ref[:, 0, 0])
    bound, mean_bound = derived_bound(w, ost, ref)
    got = _emulate(w, ost)
    d = np.abs(got - ref)[live]
    assert float((d - bound[live]).max()) <= 0.0
    assert float(d.mean()) <= mean_bound


@pytest.mark.parametrize("case,mistake", [
    ("decode_f32_large_scores", "scale_1_over_d"), ("decode_f32_large_scores", "wrong_kv_head"),
    ("varlen_bf16_large_scores", "scale_1_over_d"), ("varlen_bf16_large_scores", "wrong_kv_head"),
    ("varlen_bf16_large_scores", "causal_plus_one"),
])
def test_planted_mistakes_exceed_the_bound(case, mistake):
    w = CASES[case]()
    ost, ref = execute(w)
    live = ~np.isnan(ref[:, 0, 0])
    bound, mean_bound = derived_bound(w, ost, ref)
    got = _emulate(w, ost, mistake)
    d = np.abs(got - ref)[live]
    assert float((d - bound[live]).max()) > 0.0 or float(d.mean()) > mean_bound


def test_bound_reduces_to_the_stated_tolerance_for_small_scores():
    # the configurations' magnitudes: the growth terms are far below the tolerance
    w = workloads.random_decode(2, "bf16", 8, 2, 128, 16, [40, 300], scale=0.5)
    ost, ref = execute(w)
    bound, mean_bound = derived_bound(w, ost, ref)
    assert float(bound.max()) < 2e-2 + 2 * 2.0 ** -9 * 3
    assert mean_bound < 2e-3 + 2e-3
