"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

A mutant is built by editing the source text of one oracle function and
executing it in a copy of that module's namespace; the pins then run against
the mutant and must fail.  This shows the pins are strong enough that a dropped
term, a wrong index or a transposed operand in the oracle would not go unseen.
"""

import inspect
import textwrap
import types

import numpy as np
import pytest

import workloads
from oracle import attention, block_pool
from tests import bruteforce


def _mutant(module, func_name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(module, func_name)))
    assert old in src, f"mutation anchor {old!r} not found in {func_name}"
    ns = dict(vars(module))
    exec(compile(src.replace(old, new, 1), f"<mutant {func_name}>", "exec"), ns)
    return ns[func_name], ns


def _attention_with(func_name, old, new):
    fn, ns = _mutant(attention, func_name, old, new)
    mod = types.SimpleNamespace(**{k: ns[k] for k in ("decode", "varlen", "gather_sequence",
                                                      "softmax_attention")})
    setattr(mod, func_name, fn)
    # rebind globals of the other functions so they call the mutant
    for name in ("decode", "varlen"):
        if name != func_name:
            f = getattr(attention, name)
            g = dict(f.__globals__)
            g[func_name] = fn
            setattr(mod, name, types.FunctionType(f.__code__, g, name))
    return mod


def _bruteforce_err(mod, w):
    from oracle.run import OracleState

    st = OracleState(w)
    st.run_setup()
    st.run_step()
    bt, ctx, qsl = st.batch_metadata()
    if all(q == 1 for _, q in w.batch):
        out = mod.decode(w.q, st.k_cache, st.v_cache, bt, ctx, w.block_size, w.dtype)
    else:
        out = mod.varlen(w.q, st.k_cache, st.v_cache, bt, qsl, ctx, w.block_size, w.dtype)
    ref = bruteforce.run(w)
    return max(float(np.max(np.abs(out[r, h] - np.array(v))))
               for r, heads in enumerate(ref) for h, v in enumerate(heads))


ATTENTION_MUTANTS = [
    ("decode", "kvh = h // g", "kvh = h % Hkv"),                        # wrong GQA map
    ("decode", "scale = 1.0 / math.sqrt(D)", "scale = 1.0 / D"),         # wrong scale
    ("gather_sequence", "np.swapaxes(cache[b], 0, 1)",
     "cache[b].reshape(cache.shape[2], cache.shape[1], cache.shape[3])"),  # layout mixed up
    ("gather_sequence", "return dense[:ctx]", "return dense"),           # tail not truncated
    ("softmax_attention", "(p @ v) / p.sum(axis=1, keepdims=True)", "p @ v"),  # no normaliser
    ("varlen", "n_visible = ctx - qlen + 1 + np.arange(qlen)",
     "n_visible = ctx - qlen + 2 + np.minimum(np.arange(qlen), qlen - 2)"),  # off-by-one causal
]


@pytest.mark.parametrize("func,old,new", ATTENTION_MUTANTS)
def test_attention_mutants_are_caught(func, old, new):
    mod = _attention_with(func, old, new)
    decode_w = workloads.random_decode(3, "bf16", 8, 2, 32, 16, [1, 16, 17, 33], scale=0.5)
    varlen_w = workloads.random_varlen(5, "bf16", 4, 2, 16, 4, [(7, 3), (0, 5), (3, 13)], 0.7)
    errs = []
    for w in (decode_w, varlen_w):
        try:
            errs.append(_bruteforce_err(mod, w))
        except Exception:            # a mutant that crashes is caught too
            errs.append(np.inf)
    assert max(errs) > 1e-6


def test_unmutated_oracle_passes_same_harness():
    decode_w = workloads.random_decode(3, "bf16", 8, 2, 32, 16, [1, 16, 17, 33], scale=0.5)
    assert _bruteforce_err(attention, decode_w) <= 1e-13


POOL_MUTANTS = [
    ("if self.ref[last] == 1:", "if self.ref[last] >= 1:"),              # never copy-on-write
    ("if pos % self.block_size == 0:", "if pos % self.block_size == 1:"),  # new block too late
    ("self._drop(last)", "pass"),                                        # leak old reference
    ("self.ref[b] += 1", "pass"),                                        # fork without ref++
]


@pytest.mark.parametrize("old,new", POOL_MUTANTS)
def test_pool_mutants_are_caught(old, new):
    src = textwrap.dedent(inspect.getsource(block_pool.BlockPoolModel))
    assert old in src
    ns = dict(vars(block_pool))
    exec(compile(src.replace(old, new, 1), "<mutant pool>", "exec"), ns)
    Mut = ns["BlockPoolModel"]
    from tests import test_oracle_pool as pins

    orig = pins.BlockPoolModel
    pins.BlockPoolModel = Mut
    try:
        failed = False
        for t in (pins.test_fork_and_copy_on_write_of_shared_tail,
                  pins.test_random_operation_invariants,
                  pins.test_paging_example_block_size_4):
            try:
                t()
            except Exception:
                failed = True
        assert failed
    finally:
        pins.BlockPoolModel = orig
