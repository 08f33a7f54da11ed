"""Shared helpers for GPU parity tests: run one workload on both sides and compare."""

import numpy as np
import torch

from oracle.run import execute

# Tolerances against the float64 oracle.  bf16: max-abs 2e-2, mean-abs 2e-3 (the
# stated bar, with fp32 accumulation on the GPU).  fp32 inputs: max-abs 1e-5,
# mean-abs 1e-6 (the pages' own tiled-vs-standard fp32 check asserts 1e-5).
TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-5, 1e-6)}


def cache_bytes_equal(dev_cache, ora_cache):
    host = dev_cache.cpu()
    if host.dtype == torch.bfloat16:
        host = host.view(torch.int16).numpy().view(np.uint16)
    else:
        host = host.numpy()
    return host.shape == ora_cache.shape and np.array_equal(host.view(np.uint8),
                                                            ora_cache.view(np.uint8))


def out_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def errors(dev_out, ref):
    d = np.abs(out_f64(dev_out) - ref)
    return float(d.max()), float(d.mean())


def run_both(w, runner_mod):
    """Returns (oracle_state, oracle_out, device_cache, step, device_out)."""
    ost, oout = execute(w)
    dc, step = runner_mod.prepare(w)
    out = step.run()
    torch.cuda.synchronize()
    return ost, oout, dc, step, out
