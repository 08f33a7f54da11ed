"""paged_attention_decode_noalloc: decode attention for callers that cannot allocate.

Some users of this library cannot hand it a workspace: a plugin inside an
engine that owns all device memory and offers no scratch allocator, or a
server whose KV pool already took the rest of HBM.  For them the library keeps
a fixed scratch array per device.  This file checks, through the C ABI, that
the no-allocation entry point gives what the workspace entry point gives, on
two calls in a row (the second call finds the first call's leftovers in the
shared array), and that a batch too large for the array is refused up front.

The file name sorts last so a run that stops at the first failure has already
run every other test.
"""

import ctypes

import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from tests.gpu_parity import TOL  # noqa: E402


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import runner

    lib.device_error(clear=True)
    # two different batches, so the second call runs over the first call's leftovers
    batches = [workloads.config2(seed=3, batch=16),
               workloads.random_decode(4, "bf16", 32, 8, 128, 16, [1, 513, 1800, 4096, 77],
                                       scale=0.5)]
    tmax, tmean = TOL["bf16"]
    for w in batches:
        dc, step = runner.prepare(w)
        need = lib.decode_workspace_bytes(dc.desc, step.q.shape[0], step.max_ctx)
        assert need <= lib.NOALLOC_SCRATCH_BYTES
        ref = step.run().clone()        # the entry point that takes a workspace
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            lib.paged_attention_decode_noalloc(out, step.q, dc.k_cache, dc.v_cache, dc.desc,
                                               step.tables, step.ctx, step.max_ctx)
            torch.cuda.synchronize()
            d = (out.double() - ref.double()).abs()
            assert float(d.max()) <= tmax and float(d.mean()) <= tmean
            assert torch.equal(out, ref)  # same kernels, same order: same bits
        assert lib.device_error() == 0


def test_noalloc_refuses_batches_larger_than_its_scratch(lib):
    """Checked on the host before anything touches a device (runs without a GPU)."""
    L = lib.lib()
    desc = lib.CacheDesc(lib.PKV_BF16, 1 << 20, 16, 8, 64, 128)
    assert lib.decode_workspace_bytes(desc, 256, 32768) > lib.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    st = L.paged_attention_decode_noalloc(fake, fake, fake, fake, ctypes.byref(desc), fake, 2048,
                                          fake, 256, 32768, 0.1, None)
    assert st == lib.PKV_ERR_WORKSPACE
