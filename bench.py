"""Benchmark of the paged KV-cache decode step on GB300.

One step = the whole hot path over one batch: append each sequence's new
key/value through its block table (Eq. 21.6 of "KV cache: Generation state,
latency, and allocation"), then paged decode attention over every cached
position.  Default workload: the Llama-3.1-8B-style GQA layer (32 query heads,
8 KV heads, d_h 128, bf16 KV, 16-token blocks), B = 32 sequences of 8 192
cached tokens, blocks randomly permuted across the pool.

Metric: effective KV GB/s = algorithmic bytes of a step / step time (KV bytes
of every valid position read once, block-table entries, q, the appended rows,
out and lse), and decode tokens/s = B / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own pool and batch (sequences shard with no
collective, weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402

METRIC = "decode-attention effective KV GB/s and fraction of GB300 HBM roofline; tokens/s"
UNIT = "GB/s"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- bytes
def step_bytes(w) -> dict:
    """Algorithmic bytes of one step of workload w (one layer): the decode step
    and, when the workload carries a prefill chunk, the chunk's attention (its
    row's keys and values read once, its queries in, its outputs out)."""
    s = w.elem_bytes
    lens = w.lens_post.astype(np.int64)
    kv = int(lens.sum()) * 2 * w.H_KV * w.d_h * w.elem_bits // 8
    table = int(((lens + w.bs - 1) // w.bs).sum()) * 4
    q = w.B * w.H_Q * w.d_h * 2
    out = w.B * w.H_Q * w.d_h * 4 + w.B * w.H_Q * 4
    append = int(2 * w.B * w.H_KV * w.d_h * (2 + s))
    lens_b = w.B * 4 * 2
    r = {"kv": kv, "table": table, "q": q, "out": out, "append": append, "lens": lens_b}
    if w.prefill is not None:
        p = w.prefill
        r["prefill_kv"] = p.total * 2 * w.H_KV * w.d_h * w.elem_bits // 8
        r["prefill_table"] = -(-p.total // w.bs) * 4
        r["prefill_q"] = p.n_q * w.H_Q * w.d_h * 2
        r["prefill_out"] = p.n_q * w.H_Q * (w.d_h + 1) * 4
    r["total"] = sum(r.values())
    return r


def prefill_flops(w) -> int:
    """Scores and value mixture of the chunk: 4 d_h flops per (query head, visible position)."""
    p = w.prefill
    if p is None:
        return 0
    visible = p.n_q * p.q_start + p.n_q * (p.n_q + 1) // 2
    return 4 * w.d_h * w.H_Q * visible


# the sources a step's kernel is compiled from (its ncu counters go stale when one changes):
# the decode step's kernel, and the mixed step's (decode + prefill chunk) kernel
KERNEL_SOURCES = {
    "decode": ["kvc_decode.cuh", "kvc_ptx.cuh", "kvc_internal.h", "kvc_attn.cu"],
    "mixed": ["kvc_decode.cuh", "kvc_prefill.cuh", "kvc_ptx.cuh", "kvc_internal.h", "kvc_attn.cu"],
    "decode_tc": ["kvc_decode_tc.cuh", "kvc_tc.cuh", "kvc_decode.cuh", "kvc_ptx.cuh", "kvc_internal.h", "kvc_attn.cu"],
    "decode_tc8": ["kvc_decode_tc8.cuh", "kvc_decode_tc.cuh", "kvc_tc.cuh", "kvc_decode.cuh", "kvc_ptx.cuh",
                   "kvc_internal.h", "kvc_attn.cu"],
    "prefill_tc": ["kvc_prefill_tc.cuh", "kvc_decode_tc.cuh", "kvc_tc.cuh", "kvc_decode.cuh", "kvc_ptx.cuh",
                   "kvc_internal.h", "kvc_attn.cu"],
}


def step_kernel(w) -> str:
    """The kernels the library picks for this workload's step (the same rule as its dispatch)."""
    tc_on = os.environ.get("KVC_TC", "1")[:1] != "0" and w.bs == 16
    tc = tc_on and w.dtype == "bf16"
    if w.prefill is not None:
        if tc:
            return ("kvc_mixed_step: decode_kernel with fused append, then prefill_tc_kernel (tcgen05) as its "
                    "programmatic dependent launch")
        return "mixed_kernel: decode step with fused append and the prefill chunk in one launch (kvc_mixed_step)"
    if tc and w.H_Q == 32 * w.H_KV and w.d_h == 128:
        return "decode_tc_kernel (tcgen05, TMEM) with fused append, then merge_kernel (kvc_decode_step)"
    if tc_on and w.dtype == "fp8" and w.H_Q == 32 * w.H_KV and w.d_h == 128:
        return ("decode_tc8_kernel (tcgen05, TMEM; e4m3 codes widened to f16 in shared memory) with fused append, "
                "then merge_kernel (kvc_decode_step)")
    return "decode_kernel with fused append (kvc_decode_step)"


def source_digest(kind: str = "decode", read=None) -> str:
    """sha256 prefix of the kernel family's sources (read(name) -> bytes; default: the tree)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_kvc_gb300", "csrc")
    read = read or (lambda f: open(os.path.join(csrc, f), "rb").read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        h.update(read(f))
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """Per-launch DRAM bytes of the step's kernel from the committed ncu summary
    (profiles/*_<workload>.md), if it was taken on the current kernel sources; else None."""
    import glob
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", f"*_step_{workload}.md")))
    if not paths:
        return None
    path = paths[0]
    fields = {}
    for line in open(path):
        if line.startswith("<!-- ") and ":" in line:
            k, v = line[5:].split("-->")[0].split(":", 1)
            fields[k.strip()] = v.strip()
    kind = fields.get("kernel_family", "decode")
    if kind not in KERNEL_SOURCES or fields.get("source_sha") != source_digest(kind) or fields.get("workload") != workload:
        return None
    try:
        return int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 10:
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        num = lambda x: x.replace(".", "").isdigit()
        busy = [r for r in rows if num(r[9]) and float(r[9]) >= 50]   # samples while the GPU was busy
        load = busy or rows
        sm = [float(r[1]) for r in load if num(r[1])]
        mx = [float(r[2]) for r in rows if num(r[2])]
        pw = [float(r[3]) for r in load if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in load for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(busy),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- oracle (CPU) side
def oracle_sample(w, ld, budget_s: float, units_max=None):
    """Time the oracle (append into its pool image + decode) on a bounded sample
    of (sequence, KV head) units of the workload, batched into one call so every
    host thread works.  Returns (bytes/s, seconds, units, description, threads)."""
    import oracle
    from harness import logical_lists
    K, V, cu = logical_lists(w, ld, ld.k_ctx, ld.v_ctx, ld.k_new, ld.v_new)
    g = w.g
    units = [(b, h) for b in range(w.B) for h in range(w.H_KV)]

    def prepare(sel):
        qs, ks, vs, cus, ns = [], [], [], [0], []
        for (b, h) in sel:
            n = int(w.lens_post[b])
            rows = slice(int(cu[b]), int(cu[b]) + n)
            qs.append(ld.q[b, h * g:(h + 1) * g])
            ks.append(K[rows, h:h + 1])
            vs.append(V[rows, h:h + 1])
            cus.append(cus[-1] + n)
            ns.append(n)
        return (np.ascontiguousarray(np.stack(qs)), np.ascontiguousarray(np.concatenate(ks)),
                np.ascontiguousarray(np.concatenate(vs)), np.array(cus, np.int64), np.array(ns, np.int64))

    def run(sel):
        qb, kb, vb, cub, nb = prepare(sel)
        t0 = time.perf_counter()
        for i, (b, h) in enumerate(sel):     # the append of each unit's new row (Eq. 21.6) into a pool image
            img = oracle.PoolImage(1, int(nb[i]), 1, 1, w.d_h, 2)
            img.write_tokens(0, np.zeros((1, 1), np.int32), np.array([nb[i] - 1], np.int32),
                             np.array([0, 1], np.int64), ld.k_new[b:b + 1, h:h + 1], ld.v_new[b:b + 1, h:h + 1])
        oracle.decode(qb, kb, vb, cub, nb, 1, scale=w.scale)
        return int(nb.sum()) * 2 * w.d_h * w.elem_bits // 8, time.perf_counter() - t0

    _, t1 = run(units[:1])
    k = max(1, min(len(units), int(budget_s / max(t1, 1e-6))))
    if units_max:
        k = min(k, units_max)
    nbytes, dt, passes = 0, 0.0, 0
    while passes == 0 or (units_max is None and dt < budget_s and passes < 1000):
        b_, t_ = run(units[:k])        # whole passes over the sample until the budget is spent
        nbytes, dt, passes = nbytes + b_, dt + t_, passes + 1
    threads = min(oracle.num_threads(), k * g)
    desc = (f"{passes} pass(es) over {k} of {len(units)} (sequence, KV head) units of {w.name} "
            f"(each {int(w.lens_post[0])} positions, {g} query heads): oracle append + fp64 decode")
    return nbytes / dt, dt, k, desc, threads


def run_reference(args, w, ld, rank):
    """The oracle arm: each step a bounded sample of the same workload on host cores."""
    per_step = max(0.01, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    rate, dt, k, desc, cores = oracle_sample(w, ld, per_step)
    samples = []
    for i in range(args.warmup + args.steps):
        r, t, _, _, _ = oracle_sample(w, ld, per_step, units_max=k)
        if i >= args.warmup:
            samples.append((r, t))
    value = float(np.mean([r for r, _ in samples])) / 1e9
    ms = float(np.mean([t for _, t in samples])) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc + " per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w):
    c = {"workload": w.name, "B": w.B, "H_Q": w.H_Q, "H_KV": w.H_KV, "d_h": w.d_h, "block_size": w.bs,
         "layers": w.L, "context": int(w.lens_pre.max()), "attended": int(w.lens_post.max()),
         "kv_dtype": w.dtype, "num_blocks": w.num_blocks,
         "l2": f"inputs larger than L2: {step_bytes(w)['kv'] * w.L / 1e9:.2f} GB of KV per step vs "
               f"{L2_BYTES / 2**20:.0f} MiB L2"}
    if w.shared_prefix:
        c["shared_prefix"] = w.shared_prefix
    if w.prefill is not None:
        c["prefill_chunk"] = {"queries": w.prefill.n_q, "q_start": w.prefill.q_start}
    return c


# ---------------------------------------------------------------- multi-rank aggregation
def max_over_ranks(values, dist, device="cpu"):
    """Element-wise MAX of per-rank timings (every rank gets the result)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def weak_scaling_value(bytes_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return bytes_per_rank * world / (max_ms * 1e-3) / 1e9


def step_stats(ms, steps=None):
    """Mean, median and 90th percentile of per-step times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"mean": float(a.mean()), "median": float(np.median(a)), "p90": float(np.percentile(a, 90)),
            "steps": int(a.size) if steps is None else int(steps)}


STEP_GROUPS = 100   # events bracket groups of steps, never single steps


def time_steps(run, K: int, stream):
    """Time K back-to-back calls of run() on `stream`.

    Events are recorded only between groups of ceil(K / STEP_GROUPS) calls: an
    event between two steps would hold the next step's launch until the step
    before it has drained, which the library's programmatic dependent launches
    otherwise overlap (as in an untimed decode loop).  Returns (mean ms per step
    over all K steps, step_stats over the groups' per-step times)."""
    import torch
    chunk = max(1, -(-K // STEP_GROUPS))
    bounds = list(range(0, K, chunk)) + [K]
    ev = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    for j in range(len(bounds) - 1):
        ev[j].record(stream)
        for _ in range(bounds[j + 1] - bounds[j]):
            run()
    ev[-1].record(stream)
    ev[-1].synchronize()
    per = [ev[j].elapsed_time(ev[j + 1]) / (bounds[j + 1] - bounds[j]) for j in range(len(bounds) - 1)]
    mean = ev[0].elapsed_time(ev[-1]) / K
    st = step_stats(per, K)
    st["mean"] = mean
    return mean, st


# ---------------------------------------------------------------- the other target workloads
# The configurations beside the headline one, each timed in its own region: the
# 32 GiB pool (32 layers, one CUDA graph per step), the e4m3 and bf16 GQA sweep
# points, and MQA.  Their pools are filled on the device from a seeded
# generator (N(0,1) rounded to bf16, then stored as each pool stores it), so a
# 32 GiB pool is ready in seconds; the block tables and lengths are the
# workload's own.
EXTRA_WORKLOADS = "full_pool,sweep_hkv8_fp8,sweep_hkv8_bf16,sweep_hkv1_bf16,sweep_hkv1_fp8,prefill_chunk"
EXTRA_SECONDS = 1.5


def fill_on_device(kvc, g, w, layer, gen):
    """Write layer `layer`'s context through kvc_write_tokens from N(0,1) bf16 values drawn on the device."""
    import torch
    from harness import dev_i32
    units = ([(0, 0, w.shared_prefix)] if w.shared_prefix else []) + \
        [(b, w.shared_prefix, int(w.lens_pre[b])) for b in range(w.B)]
    units = [u for u in units if u[2] > u[1]]
    if not units:
        return
    rows = np.array([u[0] for u in units], np.int32)
    start = np.array([u[1] for u in units], np.int32)
    n = np.array([u[2] - u[1] for u in units], np.int64)
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    shape = (int(cu[-1]), w.H_KV, w.d_h)
    k = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    if w.dtype != "bf16":
        kvc.kvc_calibrate_scales(g.pool, layer, k, v)
    kvc.kvc_write_tokens(g.pool, layer, dev_i32(w.block_tables[rows]), dev_i32(start), dev_i32(cu), k, v,
                         max_tokens=int(n.max()))
    del k, v


def bench_prefill_chunk(kvc, seed, local, seconds=EXTRA_SECONDS):
    """The ragged workload's prefill chunk alone: 600 queries (positions 1 200 .. 1 799)
    attending causally over the row's 1 200-token shared prefix and themselves
    (kvc_prefill_attn), as TFLOP/s of scores and value mixture against the bf16 peak."""
    import torch
    import synth
    from harness import GpuCase, dev_i32
    w = synth.make_workload("ragged_prefix", seed=seed)
    pf = w.prefill
    g = GpuCase(kvc, w, fill_byte=0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    try:
        row = dev_i32(w.block_tables[pf.seq])
        shape = (pf.total, w.H_KV, w.d_h)
        k = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
        v = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
        kvc.kvc_write_tokens(g.pool, 0, row[None], dev_i32([0]), dev_i32([0, pf.total]), k, v)
        q = torch.randn((pf.n_q, w.H_Q, w.d_h), generator=gen, device="cuda").to(torch.bfloat16)
        out = torch.empty((pf.n_q, w.H_Q, w.d_h), device="cuda")
        lse = torch.empty((pf.n_q, w.H_Q), device="cuda")
        stream = torch.cuda.current_stream()
        run = lambda: kvc.kvc_prefill_attn(g.pool, 0, q, row, pf.q_start, out, lse, scale=w.scale)
        for _ in range(5):
            run()
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(5):
            run()
        t1.record(stream)
        torch.cuda.synchronize()
        n = int(min(20000, max(20, seconds / (t0.elapsed_time(t1) / 5 * 1e-3))))
        with ClockSampler(local) as clk:
            torch.cuda.synchronize()
            _, st = time_steps(run, n, stream)
            torch.cuda.synchronize()
        flops = prefill_flops(w)
        tf = flops / (st["mean"] * 1e-3) / 1e12
        peak = tensor_peak()
        return {"queries": pf.n_q, "q_start": pf.q_start, "H_Q": w.H_Q, "H_KV": w.H_KV, "d_h": w.d_h,
                "flops": flops, "ms": st["mean"], "ms_median": st["median"], "ms_p90": st["p90"], "launches": st["steps"],
                "tflops": tf, "peak_tflops": peak[0], "peak_source": peak[1], "tensor_frac": tf / peak[0],
                "clocks": clk.summary(),
                "data": "synthetic: N(0,1) bf16 drawn on the device (seeded)"}
    finally:
        g.close()


def tensor_peak():
    """bf16 dense tensor peak (burst: the chunk is timed on its own), TFLOP/s."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["bf16_tflops"]), "measured bf16_tflops (burst)"
    except Exception:
        return 1900.0, "fallback"


def bench_extra(kvc, name, seed, hbm, local, seconds=EXTRA_SECONDS):
    """Time one more workload's step (fused decode step per layer; a CUDA graph when multi-layer)."""
    import torch
    import synth
    from harness import GpuCase
    w = synth.make_workload(name, seed=seed)
    g = GpuCase(kvc, w, fill_byte=0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    try:
        ins = []
        for layer in range(w.L):
            fill_on_device(kvc, g, w, layer, gen)
            mk = lambda *shape: torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
            ins.append((mk(w.B, w.H_Q, w.d_h), mk(w.B, w.H_KV, w.d_h), mk(w.B, w.H_KV, w.d_h),
                        torch.empty((w.B, w.H_Q, w.d_h), device="cuda"), torch.empty((w.B, w.H_Q), device="cuda")))
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()

        def step():
            for layer in range(w.L):
                q, kn, vn, o, l_ = ins[layer]
                kvc.kvc_decode_step(g.pool, layer, q, g.bt_dec, g.lens_pre, kn, vn, o, l_, scale=w.scale)

        for _ in range(5):
            step()
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        run = step
        if w.L > 1:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            graph.replay()
            torch.cuda.synchronize()
            run = graph.replay
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(3):
            run()
        t1.record(stream)
        torch.cuda.synchronize()
        n = int(min(20000, max(20, seconds / (t0.elapsed_time(t1) / 3 * 1e-3))))
        with ClockSampler(local) as clk:
            torch.cuda.synchronize()
            _, st = time_steps(run, n, stream)
            torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        sb = step_bytes(w)
        launch_ms = st["mean"] / w.L
        achieved = sb["total"] / (launch_ms * 1e-3) / 1e9
        return {"kv_dtype": w.dtype, "B": w.B, "H_Q": w.H_Q, "H_KV": w.H_KV, "d_h": w.d_h, "layers": w.L,
                "attended": int(w.lens_post.max()), "ms_per_step": st["mean"], "ms_per_step_median": st["median"],
                "ms_per_step_p90": st["p90"], "steps": st["steps"], "GB_per_s": sb["total"] * w.L / (st["mean"] * 1e-3) / 1e9,
                "tokens_per_s": w.B / (st["mean"] * 1e-3), "launch_ms": launch_ms, "roofline_frac": achieved / hbm,
                "algorithmic_bytes_per_launch": sb["total"], "clocks": clk.summary(),
                "data": "synthetic: N(0,1) bf16 drawn on the device (seeded), stored as the pool stores it"}
    finally:
        g.close()


# ---------------------------------------------------------------- GPU side
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="kvc", choices=["kvc", "reference"])
    ap.add_argument("--workload", default="llama_gqa")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", default=EXTRA_WORKLOADS,
                    help="comma-separated workloads timed after the headline one (their own regions); '' for none")
    args = ap.parse_args()

    import synth
    from harness import layer_data

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        w = synth.make_workload(args.workload, seed=args.seed)
        run_reference(args, w, layer_data(w, 0), rank)
        return

    import torch
    import paged_kv_cache_kvc_gb300 as kvc
    from harness import GpuCase, dev_bits, dev_i32

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    kvc.load()

    w = synth.make_workload(args.workload, seed=args.seed + rank)     # each rank: its own batch
    L = w.L
    g = GpuCase(kvc, w, fill_byte=0)
    q, k_new, v_new, outs, lses = [], [], [], [], []
    ld = None
    for layer in range(L):          # every layer's context into the pool; keep only the step's inputs
        ld_l = layer_data(w, layer)
        g.load_context(layer, ld_l)
        a, b_, c = g.step_inputs(ld_l)
        q.append(a)
        k_new.append(b_)
        v_new.append(c)
        outs.append(torch.empty((w.B, w.H_Q, w.d_h), dtype=torch.float32, device="cuda"))
        lses.append(torch.empty((w.B, w.H_Q), dtype=torch.float32, device="cuda"))
        if layer == 0:
            ld = ld_l               # the CPU baseline samples layer 0
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sb1 = step_bytes(w)
    sb = {k: v * L for k, v in sb1.items()}
    pf = w.prefill
    if pf is not None:   # the chunk's keys and values go in once; every step attends over them
        row = dev_i32(w.block_tables[pf.seq])
        pq, p_out, p_lse = [], [], []
        for layer in range(L):
            kc = w.ctx_tokens(layer, 0, pf.seq, pf.q_start, pf.total)
            vc = w.ctx_tokens(layer, 1, pf.seq, pf.q_start, pf.total)
            kvc.kvc_write_tokens(g.pool, layer, row[None], dev_i32([pf.q_start]), dev_i32([0, pf.n_q]),
                                 dev_bits(kc), dev_bits(vc))
            pq.append(dev_bits(w.prefill_q(layer)))
            p_out.append(torch.empty((pf.n_q, w.H_Q, w.d_h), dtype=torch.float32, device="cuda"))
            p_lse.append(torch.empty((pf.n_q, w.H_Q), dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()

    def launch(layer, q_, bt_, lp_, k_, v_, o_, l_, pq_=None, po_=None, pl_=None, strm=None):
        """One layer of the step: the fused decode step, with the prefill chunk in the same launch."""
        if pf is None:
            kvc.kvc_decode_step(g.pool, layer, q_, bt_, lp_, k_, v_, o_, l_, scale=w.scale, stream=strm)
        else:
            kvc.kvc_mixed_step(g.pool, layer, q_, bt_, lp_, k_, v_, o_, l_, pq_, row, pf.q_start, po_, pl_,
                               scale=w.scale, stream=strm)

    def step():     # each layer: append + paged decode attention (+ the chunk), one launch
        for layer in range(L):
            launch(layer, q[layer], g.bt_dec, g.lens_pre, k_new[layer], v_new[layer], outs[layer], lses[layer],
                   *((pq[layer], p_out[layer], p_lse[layer]) if pf is not None else ()))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK

    run = step
    graph = None
    if L > 1:       # a multi-layer step replays as one CUDA graph of L launches
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        barrier()
        run = graph.replay

    # ---- device-resident timed region; events on the launching stream bracket the
    # region and groups of steps (per-step median / p90 over the groups)
    K = args.steps
    launches0 = kvc.kvc_launch_count()
    with ClockSampler(local) as clk:
        barrier()
        ms, per_step = time_steps(run, K, stream)
        barrier()
    launches = kvc.kvc_launch_count() - launches0 if graph is None else K * L
    attn_ms = ms / L    # per launch
    clocks = clk.summary()
    assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK

    # ---- end to end through the public API: every step copies its inputs from
    # pinned host memory and its results back.  Copies run on their own streams,
    # double-buffered, so step i's inputs arrive while step i-1 computes and its
    # results leave while step i+1 computes (a serving loop's overlap).
    # per-layer inputs and results of the step (the chunk's queries and outputs too, if any); each side
    # lives in one buffer (256-byte aligned views), so a step is one host-to-device copy and one back
    ins = {"q": q, "k": k_new, "v": v_new}
    res = {"out": outs, "lse": lses}
    if pf is not None:
        ins["pq"] = pq
        res.update(p_out=p_out, p_lse=p_lse)
    in_list = [t for ts in ins.values() for t in ts] + [g.bt_dec, g.lens_pre]
    res_list = [t for ts in res.values() for t in ts]

    def layout(ts):
        offs, n = [], 0
        for t in ts:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, n

    def views(buf, ts, offs):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(ts, offs)]

    in_offs, in_bytes = layout(in_list)
    res_offs, res_bytes = layout(res_list)
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for hv, t in zip(views(host_in, in_list, in_offs), in_list):
        hv.copy_(t.cpu())
    sets = []          # two device buffer sets: inputs and results of alternate steps
    for _ in range(2):
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device="cuda")
        d_res = torch.empty(res_bytes, dtype=torch.uint8, device="cuda")
        h_res = torch.empty(res_bytes, dtype=torch.uint8).pin_memory()
        iv, rv = views(d_in, in_list, in_offs), views(d_res, res_list, res_offs)
        d = {"in": d_in, "res": d_res, "res_h": h_res, "res_views": rv, "res_h_views": views(h_res, res_list, res_offs)}
        k_ = 0
        for n, ts in ins.items():
            d[n] = iv[k_:k_ + len(ts)]
            k_ += len(ts)
        d["bt"], d["lp"] = iv[k_], iv[k_ + 1]
        k_ = 0
        for n, ts in res.items():
            d[n] = rv[k_:k_ + len(ts)]
            k_ += len(ts)
        sets.append(d)
    h2d = sum(t.numel() * t.element_size() for t in in_list)
    d2h = sum(t.numel() * t.element_size() for t in res_list)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    computed, drained, loaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in computed + drained:
        e.record(stream)

    def e2e_step(i):
        b = sets[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(computed[i % 2])          # step i-2 has finished reading this set's inputs
            b["in"].copy_(host_in, non_blocking=True)
            loaded[i % 2].record(s_in)
        stream.wait_event(loaded[i % 2])
        stream.wait_event(drained[i % 2])             # step i-2's results have left this set
        for layer in range(L):
            launch(layer, b["q"][layer], b["bt"], b["lp"], b["k"][layer], b["v"][layer], b["out"][layer],
                   b["lse"][layer], *((b["pq"][layer], b["p_out"][layer], b["p_lse"][layer]) if pf else ()),
                   strm=stream)
        computed[i % 2].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[i % 2])
            b["res_h"].copy_(b["res"], non_blocking=True)
            drained[i % 2].record(s_out)

    for i in range(min(4, K)):                        # warm the copy path
        e2e_step(i)
    barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    s_in.wait_event(e_start)
    for i in range(K):
        e2e_step(i)
    stream.wait_event(drained[(K - 1) % 2])           # the last results are on the host
    e_end.record(stream)
    barrier()
    e2e_ms = e_start.elapsed_time(e_end) / K
    torch.cuda.synchronize()
    last = sets[(K - 1) % 2]                          # the copied-back results are the kernel's
    for hv, dv in zip(last["res_h_views"], last["res_views"]):
        assert torch.equal(hv, dv.cpu())

    # ---- max over ranks
    ms, e2e_ms, attn_ms = max_over_ranks([ms, e2e_ms, attn_ms], dist, "cuda")
    value = weak_scaling_value(sb["total"], world, ms)
    e2e_value = weak_scaling_value(sb["total"], world, e2e_ms)
    hbm, peak_kind = peaks()
    achieved = sb1["total"] / (attn_ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, dt, k, desc, cores = oracle_sample(w, ld, args.cpu_budget)
        cpu = {"value": rate / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{desc}; {dt:.1f} s"}
    extra = {}
    if rank == 0 and args.extra:
        g.close()                    # the headline pool's memory goes back before the next pools
        for name in [x for x in args.extra.split(",") if x and x != w.name]:
            extra[name] = (bench_prefill_chunk(kvc, args.seed + rank, local) if name == "prefill_chunk"
                           else bench_extra(kvc, name, args.seed + rank, hbm, local))
    if rank == 0:
        splits_note = (f"{L} launches per step (one per layer)" + (", replayed as one CUDA graph" if graph else "")
                       if launches == K * L else f"{launches / K:.1f} launches per step")
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
                "ms_per_step": ms, "ms_per_step_median": per_step["median"], "ms_per_step_p90": per_step["p90"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": w.dtype, "data": "synthetic", "config": config_dict(w),
                "tokens_per_s": w.B * world / (ms * 1e-3),
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": e2e_ms, "tokens_per_s": w.B * world / (e2e_ms * 1e-3)},
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                             "frac": achieved / hbm, "traffic": profiled_traffic(w.name),
                             "kernel": step_kernel(w),
                             "peak_source": f"{peak_kind} hbm_gbs",
                             "algorithmic_bytes_per_launch": sb1["total"], "launch_ms": attn_ms,
                             "note": splits_note},
                "gpu_launches": int(launches), "clocks": clocks, "cpu_baseline": cpu,
                "step_bytes": sb, "configs": extra}
        if pf is not None:   # the chunk's causal attention rides in the same launch
            line["prefill"] = {"queries": pf.n_q, "q_start": pf.q_start, "flops_per_step": prefill_flops(w) * L,
                               "tflops_in_step": prefill_flops(w) * L / (ms * 1e-3) / 1e12}
        print(json.dumps(line), flush=True)
    g.close()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
