"""A pipeline wait that runs out ends the kernel with an error code and leaves
the CUDA context usable.

Every mbarrier wait in the kernels gives up after a time limit, records
PKV_DEV_WAIT_TIMEOUT in the device error word and lets the kernel finish (its
producers still wait, bounded, for the copies they issued).  To see that path
run without faulting anything, this test builds a separate copy of the library
(never the product build) with a 1 ms limit and a decode producer that never
copies its CTA's fourth tile nor marks that stage full: no copy is in flight
for it, so the consumer that waits on it runs out of time.  The product
library's next call on the same context must then give the same bits as
before.
"""

import ctypes
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle.run import execute  # noqa: E402
from tests.gpu_parity import TOL, errors  # noqa: E402

pytestmark = pytest.mark.gpu

WAIT_TEST_DEFINES = {"PKV_WAIT_LIMIT_NS": "1000000ull", "PKV_TEST_SKIP_TILE": "3"}


def _test_library(lib):
    from paged_kv_cache_51_gb300 import _build

    T = ctypes.CDLL(_build.build_variant("waittest", WAIT_TEST_DEFINES))
    i32, p, sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    T.paged_attention_decode.restype = ctypes.c_int
    T.paged_attention_decode.argtypes = [p, p, p, p, ctypes.POINTER(lib.CacheDesc), p, i32, p,
                                         i32, i32, ctypes.c_float, p, sz, p]
    T.pkv_device_error.restype = ctypes.c_int
    T.pkv_device_error.argtypes = [ctypes.POINTER(i32), i32]
    return T


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import paged_attention_decode, runner, workspace

    T = _test_library(lib)
    # group size 1 (the CUDA-core split kernel), one 300-token split per KV head:
    # every unit has 19 tiles, so each CTA that takes one skips its tile 3
    w = workloads.random_decode(51, "bf16", 8, 8, 128, 16, [300, 290], scale=0.5)
    _, ref = execute(w)
    dc, step = runner.prepare(w)
    step.write_kv()
    lib.device_error(clear=True)
    step.attend()
    torch.cuda.synchronize()
    good = step.out.clone()
    assert lib.device_error() == 0

    code = ctypes.c_int32()
    assert T.pkv_device_error(ctypes.byref(code), 1) == 0         # clear the test copy's word
    bad = torch.empty_like(step.q)
    ws = workspace(step.ws.numel())
    st = T.paged_attention_decode(
        ctypes.c_void_p(bad.data_ptr()), ctypes.c_void_p(step.q.data_ptr()),
        ctypes.c_void_p(dc.k_cache.data_ptr()), ctypes.c_void_p(dc.v_cache.data_ptr()),
        ctypes.byref(dc.desc), ctypes.c_void_p(step.tables.data_ptr()), step.tables.shape[1],
        ctypes.c_void_p(step.ctx.data_ptr()), step.q.shape[0], step.max_ctx,
        1.0 / math.sqrt(w.head_dim), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert T.pkv_device_error(ctypes.byref(code), 1) == 0          # synchronizes the device
    assert code.value == 6                                         # PKV_DEV_WAIT_TIMEOUT

    # the context is usable: the product library's word is clear, and the same
    # call gives the same bits as before the timed-out one
    assert lib.device_error() == 0
    again = torch.empty_like(step.q)
    paged_attention_decode(again, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables, step.ctx,
                           step.max_ctx)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert torch.equal(again, good)
    mx, mean = errors(again, ref)
    assert mx <= TOL["bf16"][0] and mean <= TOL["bf16"][1]
    assert np.isfinite(again.float().cpu().numpy()).all()
