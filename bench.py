#!/usr/bin/env python
"""Decode paged-attention benchmark on GB300 (one JSON line on stdout).

A step is one pass of the hot path over one batch: copy-on-write block copies
(if any), the slot-mapped append of the step's new K/V, and paged decode
attention (planner, split kernel, merge) over the whole batch.  The default
workload is the Llama-2-7B-shaped single-layer decode: bf16, 32 query heads =
32 KV heads, head_dim 128, block_size 16, batch 64, context ~ U[512, 4096],
values N(0,1) x 0.5, block tables from a seeded permutation of a pool 10%
larger than needed.

value    = algorithmic bytes of the step / device time of the step (inputs resident)
e2e      = the same bytes / time of a step that also copies its inputs from pinned
           host memory and reads the output back, the copies on two copy streams
           overlapping the neighbouring steps (e2e.serial: the same in series)
roofline = the decode attention call (planner + split + merge) against the
           measured HBM copy bandwidth
--impl reference runs the float64 CPU oracle on a bounded sample instead.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode paged-attn KV GB/s and % of GB300 HBM peak; mixed-batch tokens/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------
# algorithmic bytes (per step)
# ----------------------------------------------------------------------------
def attention_bytes(w, ctx):
    """K and V bytes of every attended key + q in + out + block tables + lengths."""
    es = w.elem_bytes
    kv = sum(int(c) for c in ctx) * w.num_kv_heads * w.head_dim * es * 2
    qo = len(ctx) * w.num_q_heads * w.head_dim * es * 2
    tables = sum(math.ceil(int(c) / w.block_size) for c in ctx) * 4 + 4 * len(ctx)
    return kv + qo + tables


def append_bytes(w, n_tokens, n_pairs):
    es = w.elem_bytes
    row = w.num_kv_heads * w.head_dim * es
    blk = row * w.block_size
    return n_tokens * row * 2 * 2 + 8 * n_tokens + n_pairs * blk * 2 * 2 + 8 * n_pairs


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


DECODE_SOURCES = ("decode.cu", "decode_common.cuh", "pkv_device.cuh")
INT8_SOURCES = ("kv_int8.cu", "decode_common.cuh", "pkv_device.cuh")


def source_hash(sources):
    """sha256 over the kernel's source files (csrc/), in the order given."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_51_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()


def ncu_traffic(profile, sources):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel is unchanged since."""
    try:
        h = source_hash(sources)
        vals = {}
        with open(os.path.join(ROOT, "profiles", profile)) as f:
            for line in f:
                if ":" in line and line.strip().startswith("- "):
                    k, v = line.strip()[2:].split(":", 1)
                    vals[k.strip()] = v.strip().strip("`")
        if vals.get("kernel_source_sha256") == h:
            return int(vals["dram_bytes_per_call"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.rows = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def summary(self, t0, t1):
        if not self.rows:
            return None

        def ts(r):
            try:
                return time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except Exception:
                return None

        during = [r for r in self.rows if ts(r) is not None and t0 - 1 <= ts(r) <= t1 + 1]
        rows = during if len(during) >= 3 else self.rows
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "window": "timed" if rows is during else "run"}


# ----------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------
def oracle_sample(config, n_seqs, seed=0):
    """A bounded sample of the workload (its first sequences) ready for the oracle."""
    import workloads
    from oracle.run import OracleState

    if config == 2:
        w = workloads.config2(seed=seed, batch=n_seqs)
    elif config == 3:
        w = workloads.config3(seed=seed, batch=n_seqs)
    else:
        raise SystemExit("the CPU baseline covers decode configs 2 and 3")
    st = OracleState(w)
    st.run_setup()
    st.run_step()
    bt, ctx, _ = st.batch_metadata()
    return w, st, bt, ctx


def oracle_attention_once(w, st, bt, ctx):
    from oracle import attention

    return attention.decode(w.q, st.k_cache, st.v_cache, bt, ctx, w.block_size, w.dtype)


def cpu_worker(config, n_seqs, seconds):
    w, st, bt, ctx = oracle_sample(config, n_seqs)
    nbytes = attention_bytes(w, ctx)
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle_attention_once(w, st, bt, ctx)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    print(json.dumps({"value": nbytes * passes / el / 1e9, "unit": "GB/s", "seconds": el,
                      "passes": passes, "seqs": n_seqs}))


def cpu_baseline(config, seconds=10.0, n_seqs=4, all_cores_seconds=5.0):
    """The oracle timed on the host: once on one core (BLAS threads pinned to 1),
    then once more with the host's default threading (all cores available)."""
    def run(env, secs):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker",
                            "--config", str(config), "--cpu-seqs", str(n_seqs),
                            "--cpu-seconds", str(secs)],
                           capture_output=True, text=True, env=env, cwd=ROOT)
        if r.returncode != 0:
            return None, r.stderr.strip()[-200:]
        return json.loads(r.stdout.strip().splitlines()[-1]), None

    one = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    d, err = run(one, seconds)
    if d is None:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"failed: {err}"}
    out = {"value": d["value"], "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": (f"first {n_seqs} sequences of the same workload (same generator), float64 "
                      f"NumPy oracle attention repeated {d['passes']}x over {d['seconds']:.1f} s "
                      f"on one host core")}
    full = {k: v for k, v in os.environ.items()
            if k not in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    d2, _ = run(full, all_cores_seconds)
    if d2 is not None:
        out["all_cores"] = {"value": d2["value"], "cores": os.cpu_count(),
                            "note": "same sample, default NumPy/BLAS threading"}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    n_seqs = 1
    w, st, bt, ctx = oracle_sample(args.config, n_seqs)
    nbytes = attention_bytes(w, ctx)
    for _ in range(args.warmup):
        oracle_attention_once(w, st, bt, ctx)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_attention_once(w, st, bt, ctx)
    el = time.perf_counter() - t0
    cores = 1 if os.environ.get("OPENBLAS_NUM_THREADS") == "1" else os.cpu_count()
    value = nbytes * args.steps / el / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample_seqs": n_seqs},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_seqs} sequence(s) of {w.name} per step, float64 oracle"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def accounting(w, step):
    """Algorithmic bytes and flops of one step of a prepared workload."""
    ctx = [int(c) for c in step.ctx.cpu().tolist()]
    qlens = [q for _, q in w.batch]
    es, hkv, hq, d, bs = w.elem_bytes, w.num_kv_heads, w.num_q_heads, w.head_dim, w.block_size
    kv = sum(c for c, q in zip(ctx, qlens) if q > 0) * hkv * d * es * 2
    qo = sum(qlens) * hq * d * es * 2
    tables = sum(math.ceil(c / bs) for c in ctx) * 4 + 4 * len(ctx)
    if max(qlens) > 1:
        tables += 4 * (len(ctx) + 1)
    pre_flops = sum(4 * d * hq * sum(c - q + i + 1 for i in range(q))
                    for c, q in zip(ctx, qlens) if q >= 2)
    dec_flops = sum(4 * d * hq * c for c, q in zip(ctx, qlens) if q == 1)
    pre_kv = sum(c for c, q in zip(ctx, qlens) if q >= 2) * hkv * d * es * 2
    return {"attn_bytes": kv + qo + tables, "append_bytes": append_bytes(
        w, step.slot_mapping.numel(), step.pairs.shape[0]), "prefill_flops": pre_flops,
        "decode_flops": dec_flops, "prefill_kv_bytes": pre_kv, "query_tokens": sum(qlens),
        "context_tokens": sum(ctx)}


def max_over_ranks(ms, dist=None, device=None):
    """The slowest rank's time: the whole job finishes when its last replica does."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(config, rank, batch=0, prefill_chunks=False):
    """Each rank runs its own replica of the workload, drawn with seed = rank.
    Sequences are independent, so replicas need no exchange on the data path."""
    import workloads

    if prefill_chunks:
        return workloads.random_varlen(rank, "bf16", 32, 8, 128, 16,
                                       [(0, 512), (1024, 512), (3072, 512)], scale=0.5)
    kw = {"batch": batch} if batch and config in (2, 3) else {}
    return workloads.make(config, seed=rank, **kw)


def job_throughput(bytes_per_rank, world, ms):
    """Whole-job GB/s: every replica moved `bytes_per_rank` in the slowest rank's time."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def time_steps(step, steps, warmup):
    """Device time of `steps` steps (one event pair around the whole loop), then
    the mean time of the attention call alone: the same number of attention
    calls back to back between one event pair.  (The step's tokens are already
    in the cache, so the calls repeat the step's attention exactly; every input
    is larger than L2, so a call gains nothing from the one before.  An event
    pair around each call would break the calls' launch chain and cost a few
    microseconds of each.)"""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step.run()
    ev1.record(stream)
    torch.cuda.synchronize()
    step_ms = ev0.elapsed_time(ev1) / steps
    ev0.record(stream)
    for _ in range(steps):
        step.attend()
    ev1.record(stream)
    torch.cuda.synchronize()
    return step_ms, ev0.elapsed_time(ev1) / steps


def peaks():
    bw, kind = measured_peak()
    tc, tc_kind = 1900.0, "fallback"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tc, tc_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        pass
    return bw, kind, tc, tc_kind


def mixed_batch_summary(steps, warmup):
    """The SplitFuse 2048-token step (config 4) and its prefill chunks alone."""
    import torch

    import paged_kv_cache_51_gb300 as pkv
    import workloads
    from paged_kv_cache_51_gb300 import runner

    bw, _, tc, _ = peaks()
    w = workloads.config4()
    dc, step = runner.prepare(w)
    acc = accounting(w, step)
    ms, attn_ms = time_steps(step, steps, warmup)
    if pkv.device_error() != 0:
        raise SystemExit("device error in the mixed batch")
    total_bytes = acc["attn_bytes"] + acc["append_bytes"]
    t_roof = max(total_bytes / (bw * 1e9), acc["prefill_flops"] / (tc * 1e12))
    del dc, step
    torch.cuda.empty_cache()
    # prefill chunks alone: tensor-core throughput of the tcgen05 kernel
    spans = [(p, 512) for p in w.notes["prefixes"]]
    wp = workloads.random_varlen(1, "bf16", 32, 8, 128, 16, spans, scale=0.5)
    dcp, stp = runner.prepare(wp)
    accp = accounting(wp, stp)
    _, pre_ms = time_steps(stp, steps, warmup)
    del dcp, stp
    torch.cuda.empty_cache()
    return {
        "workload": w.name, "query_tokens": acc["query_tokens"], "ms_per_step": ms,
        "tokens_per_s": acc["query_tokens"] / (ms * 1e-3),
        "attention_ms": attn_ms, "bytes_per_step": total_bytes,
        "prefill_gflop": acc["prefill_flops"] / 1e9,
        "roofline_ms": t_roof * 1e3, "roofline_frac": t_roof / (ms * 1e-3),
        "roofline_note": "max(bytes / HBM peak, prefill flops / bf16 peak) over the step time",
        "prefill_chunks_alone": {
            "spans": spans, "ms": pre_ms, "tflops": accp["prefill_flops"] / (pre_ms * 1e-3) / 1e12,
            "tensor_frac": accp["prefill_flops"] / (pre_ms * 1e-3) / (tc * 1e12),
            "note": "attention call on the three 512-token chunks only (planner + tcgen05 kernel)"},
    }


GQA_SOURCES = ("decode.cu", "decode_mma.cu", "decode_common.cuh", "pkv_device.cuh")


def configs_summary(steps, warmup, with_int8=True):
    """The other decode workloads, each timed as a whole step and as its parts.

    Config 3 (Llama-3-8B-shaped GQA decode, 256 sequences, 32/8 heads, contexts
    log-uniform in [1024, 8192], plus the append of its 256 new tokens) and
    config 5 (8 groups x 8 branches sharing a 3000-token prompt's blocks, with
    copy-on-write of the shared tail, plus 4 sequences at 32768 tokens; 64/8
    heads).  Lengths, pool, block tables, forks and copies are the workloads'
    own seeded draws; the K/V and q values are drawn on the device from the
    same distribution (N(0,1) x 0.5, bf16), since the kernels' speed does not
    depend on them (full-size parity of both workloads is in the GPU tests).
    Every input is larger than L2 (config 5: about 0.7 GB of unique KV)."""
    import torch

    import paged_kv_cache_51_gb300 as pkv
    import workloads
    from paged_kv_cache_51_gb300 import runner

    bw, kind, _, _ = peaks()
    stream = torch.cuda.current_stream()
    res = {}
    for cfg in (3, 5):
        w = workloads.make(cfg, values=False)
        dc, step = runner.prepare(w)
        acc = accounting(w, step)
        ms, attn_ms = time_steps(step, steps, warmup)
        if pkv.device_error() != 0:
            raise SystemExit(f"device error in config {cfg}")
        # the step's copy-on-write + append alone
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(steps):
            step.write_kv()
        a1.record(stream)
        torch.cuda.synchronize()
        app_ms = a0.elapsed_time(a1) / steps
        step_bytes = acc["attn_bytes"] + acc["append_bytes"]
        attn_gbs = acc["attn_bytes"] / (attn_ms * 1e-3) / 1e9
        r = {
            "workload": w.name, "batch": len(w.batch), "heads": [w.num_q_heads, w.num_kv_heads],
            "context_tokens": acc["context_tokens"], "ms_per_step": ms,
            "step_gbs": step_bytes / (ms * 1e-3) / 1e9,
            "attention": {"ms": attn_ms, "bytes": acc["attn_bytes"], "achieved_gbs": attn_gbs,
                          "frac": attn_gbs / bw,
                          "kernel": "planner + decode_split_mma_kernel + merge"},
            "append": {"tokens": int(step.slot_mapping.numel()),
                       "copy_pairs": int(step.pairs.shape[0]), "ms": app_ms,
                       "bytes": acc["append_bytes"],
                       "achieved_gbs": acc["append_bytes"] / (app_ms * 1e-3) / 1e9,
                       "note": "copy-on-write + append of the step's tokens, launch-bound "
                               "at this size"},
            "peak": bw, "peak_kind": f"{kind} hbm_gbs (burst copy)",
            "values": "drawn on the device, N(0,1) x 0.5 in bf16",
        }
        if cfg == 5:
            dram = ncu_traffic("decode_prefix_sharing_g8.md", GQA_SOURCES)
            r["attention"]["bytes_note"] = (
                "logical bytes: every branch's reads of its shared prompt blocks count")
            r["attention"]["dram_bytes_ncu"] = dram
            r["attention"]["dram_gbs"] = (dram / (attn_ms * 1e-3) / 1e9) if dram else None
            # the bar for this batch is stated on DRAM bytes (ncu), not logical ones
            r["attention"]["dram_frac"] = (dram / (attn_ms * 1e-3) / 1e9 / bw) if dram else None
        if with_int8:
            step.run()
            r["int8"] = int8_decode_summary(w, dc, step, steps, warmup, attn_ms, False)
        res[f"config{cfg}"] = r
        del dc, step
        torch.cuda.empty_cache()
    return res


def next_rows_summary(reps=20, warmup=3):
    """The widened rows beside the hot path, each with its own figure.

    rope_append: the fused rotary embedding + append over 16384 new tokens
    (32 query / 8 KV heads, D 128, bf16, slots scattered over the pool): bytes
    = k, v, q read + K/V rows and rotated q written + slots and positions +
    the cos/sin rows touched, against the HBM copy peak, with the plain append
    of the same K/V rows beside it.  Inputs are larger than L2.  The cos/sin
    table holds random values (the kernel's time does not depend on them).
    compose: the SplitFuse token-budget composer (host, C++ through the
    binding), 2048-token budget, 512 decodes, 64 waiting prompts.
    prefix_pool: the prefix-caching block pool (host): a 3000-token prompt per
    sequence, 8 sequences per shared prompt, then one token appended per
    sequence."""
    import numpy as np
    import torch

    import paged_kv_cache_51_gb300 as pkv

    bw, _, _, _ = peaks()
    dev = torch.device("cuda")
    g = torch.Generator(device="cpu").manual_seed(7)
    T, hq, hkv, d, bs, maxpos, sets = 16384, 32, 8, 128, 16, 4096, 4
    nb = sets * (T // bs)          # each input set writes its own quarter of the pool

    def rows(h):
        return (torch.randn((T, h, d), generator=g) * 0.5).to(torch.bfloat16).to(dev)

    ks = [rows(hkv) for _ in range(sets)]
    vs = [rows(hkv) for _ in range(sets)]
    qs = [rows(hq) for _ in range(sets)]
    q_outs = [torch.empty_like(qs[0]) for _ in range(sets)]
    slot_sets = [(torch.randperm(T, generator=g) + j * T).to(torch.int64).to(dev)
                 for j in range(sets)]
    pos = (torch.arange(T, dtype=torch.int32) % maxpos).to(dev)
    cos_sin = (torch.rand((maxpos, d), generator=g) * 2 - 1).to(dev)
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    desc = pkv.cache_desc(kc, hq)
    stream = torch.cuda.current_stream()

    def timed(fn):
        """(ms per call with `reps` calls back to back between one event pair,
        median ms of one call between its own event pair).  Calls rotate over
        the input sets, so a call's inputs and cache rows were last touched
        three calls (about 0.4 GB of traffic) earlier: not in L2."""
        for j in range(max(warmup, sets)):
            fn(j % sets)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            fn(i % sets)
            b.record(stream)
        torch.cuda.synchronize()
        single = statistics.median(a.elapsed_time(b) for a, b in ev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            fn(i % sets)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps, single

    rope_ms, rope_single = timed(lambda j: pkv.paged_kv_append_rope(
        ks[j], vs[j], slot_sets[j], pos, cos_sin, kc, vc, desc, q=qs[j], q_out=q_outs[j]))
    plain_ms, plain_single = timed(lambda j: pkv.paged_kv_append(ks[j], vs[j], slot_sets[j], kc,
                                                                 vc, desc))
    if pkv.device_error() != 0:
        raise SystemExit("device error in the append measurements")
    kv_bytes = T * hkv * d * 2 * 2
    q_bytes = T * hq * d * 2
    rope_bytes = 2 * kv_bytes + 2 * q_bytes + T * (8 + 4) + min(T, maxpos) * d * 4
    plain_bytes = 2 * kv_bytes + T * 8
    del ks, vs, qs, q_outs, kc, vc
    torch.cuda.empty_cache()

    # SplitFuse composer (host)
    rng = np.random.default_rng(3)
    prompts = [max(1, int(x)) for x in rng.normal(1200, 360, 64)]
    n_calls = 2000
    t0 = time.perf_counter()
    for _ in range(n_calls):
        pkv.pkv_splitfuse_compose(2048, 512, prompts)
    compose_us = (time.perf_counter() - t0) / n_calls * 1e6

    # prefix-caching pool (host)
    pool = pkv.BlockPool(65536, bs, 0, prefix_caching=True)
    groups, per = 8, 8
    shared = [[int(x) for x in rng.integers(0, 32000, 3000)] for _ in range(groups)]
    t0 = time.perf_counter()
    n_add = 0
    for gi in range(groups):
        for b in range(per):
            st, _, _ = pool.add_tokens(gi * per + b, shared[gi])
            if st != 0:
                raise SystemExit("prefix pool: add_tokens failed")
            n_add += 1
    add_us = (time.perf_counter() - t0) / n_add * 1e6
    t0 = time.perf_counter()
    n_app = 0
    for r in range(16):
        for sid in range(groups * per):
            st, _, _ = pool.append_token(sid, 1000 + r)
            if st != 0:
                raise SystemExit("prefix pool: append_token failed")
            n_app += 1
    append_us = (time.perf_counter() - t0) / n_app * 1e6
    pool.close()
    return {
        "rope_append": {
            "tokens": T, "heads": [hq, hkv], "head_dim": d, "ms": rope_ms,
            "bytes": rope_bytes, "achieved_gbs": rope_bytes / (rope_ms * 1e-3) / 1e9,
            "frac": rope_bytes / (rope_ms * 1e-3) / 1e9 / bw,
            "plain_append_ms": plain_ms,
            "plain_append_frac": plain_bytes / (plain_ms * 1e-3) / 1e9 / bw,
            "timing": "calls back to back over 4 input sets and 4 disjoint quarters of the "
                      "pool (nothing in L2); *_single_ms: one call between its own events",
            "ms_single": rope_single, "plain_append_ms_single": plain_single},
        "compose": {"us_per_step": compose_us, "budget": 2048, "decodes": 512,
                    "waiting_prompts": len(prompts)},
        "prefix_pool": {"us_per_add_tokens_3000": add_us, "us_per_append_token": append_us,
                        "note": "host, through the ctypes binding (marshalling included)"},
    }


def int8_decode_summary(w, dc, step, steps, warmup, bf16_attn_ms, full_size):
    """The same decode batch over an 8-bit copy of the cache: every slot of the
    bf16 pools quantised by the int8 append, then the int8 attention call timed
    alone (inputs larger than L2)."""
    import torch

    import paged_kv_cache_51_gb300 as pkv

    nb, hkv, bs, d = dc.k_cache.shape
    ic = pkv.Int8Cache(nb, hkv, bs, d, w.num_q_heads)

    def rows(c):
        return c.transpose(1, 2).reshape(nb * bs, hkv, d).contiguous()

    slots = torch.arange(nb * bs, dtype=torch.int64, device="cuda")
    pkv.paged_kv_append_int8(rows(dc.k_cache), rows(dc.v_cache), slots, ic)
    S = step.q.shape[0]
    out = torch.empty_like(step.q)
    ws = pkv.workspace(pkv.decode_workspace_bytes(ic.desc, S, step.max_ctx))
    stream = torch.cuda.current_stream()

    def call():
        pkv.paged_attention_decode_int8(out, step.q, ic, step.tables, step.ctx, step.max_ctx,
                                        ws=ws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()                      # back to back, as the bf16 call is timed
    e1.record(stream)
    torch.cuda.synchronize()
    if pkv.device_error() != 0:
        raise SystemExit("device error in the int8 decode")
    ms = e0.elapsed_time(e1) / steps
    # the step's own tokens through the quantising append
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(steps):
        pkv.paged_kv_append_int8(step.k_new, step.v_new, step.slot_mapping, ic)
    a1.record(stream)
    torch.cuda.synchronize()
    app_ms = a0.elapsed_time(a1) / steps
    ctx = [int(c) for c in step.ctx.cpu().tolist()]
    kv = sum(ctx) * hkv * 2 * (d + 4)
    qo = S * w.num_q_heads * d * 2 * 2
    tables = sum(math.ceil(c / bs) for c in ctx) * 4 + 4 * S
    nbytes = kv + qo + tables
    bw, kind, _, _ = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    diff = float((out.float() - step.out.float()).abs().max())
    del ic, ws
    torch.cuda.empty_cache()
    return {
        "kernel": "paged_attention_decode_int8 (planner + int8 split + merge)",
        "ms_per_launch": ms, "bytes_per_launch": nbytes, "achieved_gbs": gbs,
        "frac": gbs / bw, "peak": bw, "peak_kind": f"{kind} hbm_gbs (burst copy)",
        "speedup_vs_bf16_attention": bf16_attn_ms / ms,
        "context_tokens_per_s": sum(ctx) / (ms * 1e-3),
        "append_ms_per_step": app_ms,
        "max_abs_diff_vs_bf16_cache": diff,
        "traffic": ncu_traffic("decode_int8_llama2_7b.md", INT8_SOURCES) if full_size else None,
        "note": "same sequences, contexts and q as the headline; bytes = codes + fp32 scales "
                "of every attended key + q/out + tables",
    }


def run_gpu(args):
    import torch

    import workloads
    from paged_kv_cache_51_gb300 import _build

    _build.build()
    import paged_kv_cache_51_gb300 as pkv
    from paged_kv_cache_51_gb300 import runner

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")

    w = replica_workload(args.config, rank, args.batch, args.prefill_chunks)
    dc, step = runner.prepare(w)
    acc = accounting(w, step)
    attn_b = acc["attn_bytes"]
    step_bytes = attn_b + acc["append_bytes"]
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if pkv.device_error() != 0:
        raise SystemExit("device error during warm-up")

    sampler = ClockSampler(local)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms_per_step, attn_ms = time_steps(step, args.steps, 0)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    sampler.stop()
    ms_per_step = max_over_ranks(ms_per_step, dist, "cuda")
    if pkv.device_error() != 0:
        raise SystemExit("device error during the timed region")

    # ---- end to end through host buffers ----
    # Every input of a step (q, the new K/V rows, slot mapping, copy pairs, block
    # tables, lengths) sits in one pinned host buffer and goes to the device in
    # one copy; the step's device tensors are views into the device copy, and
    # its output is read back into pinned host memory.  As a serving loop does,
    # the uploads run on one copy stream and the read-backs on another, with two
    # device input buffers and two outputs, so step i + 1's inputs arrive while
    # step i computes.  Every step's own copies are inside the timed region.
    names = ("q", "k_new", "v_new", "slot_mapping", "tables", "ctx", "qsl", "pairs")
    host_in = {name: getattr(step, name).cpu() for name in names}
    offs, total = {}, 0
    for name, t in host_in.items():
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(max(total, 256), dtype=torch.uint8).pin_memory()
    for name, t in host_in.items():
        n = t.numel() * t.element_size()
        if n:
            host_buf[offs[name]:offs[name] + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    dev_bufs = [torch.empty(max(total, 256), dtype=torch.uint8, device="cuda") for _ in range(2)]
    views = [{name: b[offs[name]:offs[name] + t.numel() * t.element_size()]
              .view(t.dtype).view(t.shape) for name, t in host_in.items()} for b in dev_bufs]
    outs = [step.out, torch.empty_like(step.out)]
    host_outs = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    k_e2e = max(3, min(args.steps, 200))
    up_stream, down_stream = torch.cuda.Stream(), torch.cuda.Stream()
    uploaded = [torch.cuda.Event() for _ in range(2)]
    ran = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]
    n_done = [0]

    def e2e_step():
        b = n_done[0] & 1
        n_done[0] += 1
        up_stream.wait_event(ran[b])              # the last step on dev_bufs[b] is done
        with torch.cuda.stream(up_stream):
            dev_bufs[b].copy_(host_buf, non_blocking=True)
        uploaded[b].record(up_stream)
        stream.wait_event(uploaded[b])
        stream.wait_event(read_back[b])           # outs[b] has been read back
        for name, t in views[b].items():
            setattr(step, name, t)
        step.out = outs[b]
        step.run()
        ran[b].record(stream)
        down_stream.wait_event(ran[b])
        with torch.cuda.stream(down_stream):
            host_outs[b].copy_(outs[b], non_blocking=True)
        read_back[b].record(down_stream)

    def drain():
        for ev in read_back + uploaded:
            stream.wait_event(ev)

    for _ in range(3):
        e2e_step()
    drain()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up_stream.wait_event(e0)
    for _ in range(k_e2e):
        e2e_step()
    drain()                                       # the last read-back is inside the region
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / k_e2e
    if pkv.device_error() != 0:
        raise SystemExit("device error in the end-to-end steps")
    if not torch.equal(host_outs[(n_done[0] - 1) & 1], outs[(n_done[0] - 1) & 1].cpu()):
        raise SystemExit("end-to-end read-back differs from the device output")

    # the same steps with upload, step and read-back in series on one stream
    def serial_step():
        dev_bufs[0].copy_(host_buf, non_blocking=True)
        for name, t in views[0].items():
            setattr(step, name, t)
        step.out = outs[0]
        step.run()
        host_outs[0].copy_(outs[0], non_blocking=True)

    for _ in range(3):
        serial_step()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(k_e2e):
        serial_step()
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = e0.elapsed_time(e1) / k_e2e

    value = job_throughput(step_bytes, world, ms_per_step)
    peak, peak_kind, tc_peak, _ = peaks()
    achieved = attn_b / (attn_ms * 1e-3) / 1e9
    launches_per_step = ((1 if step.pairs.shape[0] else 0) + 1 + 2
                         + (1 if math.ceil(step.max_ctx / 512) > 1 else 0)
                         + (1 if step.max_qlen > 1 else 0))
    clocks = sampler.summary(t_wall0, t_wall1)
    int8 = None
    if world == 1 and step.decode_only and w.dtype == "bf16" and not args.no_int8:
        step.run()   # step.out holds the bf16 result for the comparison
        int8 = int8_decode_summary(w, dc, step, min(args.steps, 200), args.warmup, attn_ms,
                                   args.config == 2 and not args.batch)
    del dc, step
    torch.cuda.empty_cache()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    mixed = None
    if world == 1 and args.config == 2 and not args.no_mixed and not args.prefill_chunks:
        mixed = mixed_batch_summary(min(args.steps, 200), args.warmup)
    cpu = cpu_baseline(args.config if args.config in (2, 3) else 2) if (
        world == 1 and not args.no_cpu) else None
    nxt = None
    if world == 1 and args.config == 2 and not args.no_next and not args.prefill_chunks:
        nxt = next_rows_summary()
    others = None
    if world == 1 and args.config == 2 and not args.no_configs and not args.prefill_chunks:
        others = configs_summary(min(args.steps, 100), args.warmup, not args.no_int8)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {
            "workload": w.name, "batch": len(w.batch), "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "context_tokens": acc["context_tokens"], "query_tokens": acc["query_tokens"],
            "step": "copy-on-write + append of the step's tokens + paged attention",
            "l2": f"inputs larger than L2 (KV {attn_b / 1e9:.2f} GB read per step vs 129 MB L2)",
            "parallelism": f"replicas x{world}",
        },
        "pct_hbm_peak": achieved / peak,
        "tokens_per_s": acc["query_tokens"] * world / (ms_per_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": ncu_traffic("decode_attention_llama2_7b.md", DECODE_SOURCES)
                     if args.config == 2 and not args.batch else None,
                     "kernel": "paged attention call (planner + split + merge"
                               + (" + tcgen05 prefill)" if acc["prefill_flops"] else ")"),
                     "bytes_per_launch": attn_b, "ms_per_launch": attn_ms,
                     "peak_kind": f"{peak_kind} hbm_gbs (burst copy)"},
        "mixed_batch": mixed,
        "configs": others,
        "int8_kv_decode": int8,
        "next_rows": nxt,
        "cpu_baseline": cpu,
        "e2e": {"value": step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "uploads and read-backs on two copy streams, double-buffered, "
                          "overlapping the neighbouring steps",
                "serial": {"value": step_bytes / (serial_ms * 1e-3) / 1e9,
                           "ms_per_step": serial_ms,
                           "copies": "upload, step, read-back in series on one stream"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if acc["prefill_flops"]:
        line["prefill_gflop_per_step"] = acc["prefill_flops"] / 1e9
        t_roof = max((attn_b + acc["append_bytes"]) / (peak * 1e9),
                     acc["prefill_flops"] / (tc_peak * 1e12))
        line["step_roofline_frac"] = t_roof / (ms_per_step * 1e-3)
        line["prefill_tflops"] = acc["prefill_flops"] / (attn_ms * 1e-3) / 1e12
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences in the batch (decode workloads; 0 = the workload's own)")
    ap.add_argument("--prefill-chunks", action="store_true",
                    help="time only the SplitFuse batch's three 512-token prefill chunks")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-mixed", action="store_true",
                    help="skip the mixed-batch (SplitFuse) sub-measurement")
    ap.add_argument("--no-int8", action="store_true",
                    help="skip the 8-bit KV cache decode sub-measurement")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the widened rows (fused RoPE append, composer, prefix pool)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the GQA (config 3) and prefix-sharing (config 5) workloads")
    ap.add_argument("--cpu-worker", action="store_true")
    ap.add_argument("--cpu-seqs", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3 and not args.cpu_worker:
        args.warmup = 3
    if args.cpu_worker:
        cpu_worker(args.config, args.cpu_seqs, args.cpu_seconds)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
