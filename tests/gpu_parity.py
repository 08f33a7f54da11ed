"""Shared helpers for GPU parity tests: run one workload on both sides and compare."""

import math

import numpy as np
import torch

from oracle.attention import gather_sequence
from oracle.numerics import widen
from oracle.run import execute

# Tolerances against the float64 oracle.  bf16: max-abs 2e-2, mean-abs 2e-3 (the
# stated bar, with fp32 accumulation on the GPU).  fp32 inputs: max-abs 1e-5,
# mean-abs 1e-6 (the pages' own tiled-vs-standard fp32 check asserts 1e-5).
TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-5, 1e-6)}

# Constants of the derived bound (derived_bound below).
U32 = 2.0 ** -24          # unit roundoff of fp32
BF16_ROUND = 2.0 ** -9    # |rn_bf16(x) - x| <= 2^-9 |x|: 8 significant bits, nearest even
EXP2_REL = 2.0 ** -21     # relative error allowed for the hardware exp2 (a few fp32 ulps)


def gamma(n):
    """Higham's gamma_n = n u / (1 - n u): the relative error bound of a sum of n
    fp32 products, whatever the order of the additions."""
    return n * U32 / (1.0 - n * U32)


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


def sensitivity(w, ost, scale=None, q=None):
    """Float64 sensitivities of each output to rounding inside the GPU's softmax.

    For every query row r and head h over the keys j the row attends (weights
    p_j = exp(s_j - max s), exact):
      S[r, h]    = scale * max_j sum_d |q_d| |k_jd|   (bounds |score| and its rounding)
      W[r, h, d] = sum_j p_j |v_jd - o_d| / sum_j p_j (output change per unit of
                   relative weight error, to first order)
      A[r, h, d] = sum_j p_j |v_jd| / sum_j p_j       (output change per unit of
                   relative error in the weights of the P.V product alone)
    ``q`` overrides the workload's query rows (storage dtype)."""
    q = w.q if q is None else q
    bt, ctx, qsl = ost.batch_metadata()
    D = w.head_dim
    g = w.num_q_heads // w.num_kv_heads
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    qf = widen(q, w.dtype)
    Tq = qf.shape[0]
    S = np.zeros((Tq, w.num_q_heads))
    W = np.zeros((Tq, w.num_q_heads, D))
    A = np.zeros((Tq, w.num_q_heads, D))
    for s in range(len(ctx)):
        r0, r1 = int(qsl[s]), int(qsl[s + 1])
        if r1 == r0:
            continue
        c = int(ctx[s])
        kd = widen(gather_sequence(ost.k_cache, bt[s], c, w.block_size), w.dtype)
        vd = widen(gather_sequence(ost.v_cache, bt[s], c, w.block_size), w.dtype)
        for r in range(r0, r1):
            n = c - (r1 - r) + 1                       # keys row r attends (causal)
            for h in range(w.num_q_heads):
                k, v = kd[:n, h // g], vd[:n, h // g]
                sc = (k @ qf[r, h]) * scale
                p = np.exp(sc - sc.max())
                p /= p.sum()
                o = p @ v
                S[r, h] = scale * float((np.abs(k) @ np.abs(qf[r, h])).max())
                W[r, h] = p @ np.abs(v - o)
                A[r, h] = p @ np.abs(v)
    return S, W, A


def derived_bound(w, ost, ref, scale=None, q=None):
    """(per-element max-abs bound, mean-abs bound) for inputs whose scores or
    outputs are larger than the configurations' (values N(0,1) for fp32 and
    N(0,1)*0.5 for bf16), derived from the arithmetic.  On top of the stated
    tolerance, which covers the configurations' magnitudes, two terms grow with
    the inputs, to first order:
      * output rounding: 2^-9 |o| for a bf16 output, u |o| for fp32;
      * relative error of each softmax weight: the score is a D-term fp32 dot
        product (gamma_D sum_d |q_d k_d|, any summation order), then scaled,
        offset by the running max and exponentiated (three more roundings of at
        most |score| each, plus the exp2 error), so eps = gamma_{D+4} S + 2^-21,
        which moves the output by at most eps W; a bf16 kernel also rounds P to
        bf16 for the P.V product while its row sum keeps fp32 weights, which
        moves the output by at most 2^-9 A.
    Each term is in units of the output, so the bound is per element."""
    S, W, A = sensitivity(w, ost, scale, q)
    tmax, tmean = TOL[w.dtype]
    eps = gamma(w.head_dim + 4) * S[..., None] + EXP2_REL
    extra = eps * W
    if w.dtype == "bf16":
        extra = extra + BF16_ROUND * np.abs(ref) + BF16_ROUND * A
    else:
        extra = extra + U32 * np.abs(ref)
    return tmax + extra, tmean + float(extra.mean())


def assert_within_derived_bound(w, ost, ref, got, scale=None, q=None):
    """Element-wise max-abs and mean-abs checks of ``got`` (float64, rows that
    belong to a sequence) against derived_bound."""
    bound, mean_bound = derived_bound(w, ost, ref, scale, q)
    d = np.abs(got - ref)
    worst = float((d - bound).max())
    assert worst <= 0.0, f"max-abs bound exceeded by {worst:.3e} (max err {d.max():.3e})"
    assert float(d.mean()) <= mean_bound, (float(d.mean()), mean_bound)
    return float(d.max()), float(d.mean()), float(bound.max())
