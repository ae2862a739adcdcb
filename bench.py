#!/usr/bin/env python
"""Benchmark of the DFlash drafter block step on GB300.

One "step" is one pass of the whole hot path: embedding of the 16-row noise
block, every drafter layer (q/k/v + head norm + rope, sliding-window attention
over the ring and the block, o, gate/up + SwiGLU, down), output norm + LM
head + greedy drafts, and the acceptance scan, replayed from a CUDA graph with
the ring already filled (inputs resident in HBM).  Default workload: the real
drafter dimensions with bf16 storage (5 layers, n_embd 6656, 32/8 heads of 128,
n_ff 19968, window 2048 full, vocab 8192) - the configuration the dflash-ops
model card measures.  As the card runs it, eager work sits between replays
(the target verifies between drafter blocks): each timed replay has its own
CUDA event pair on the replay stream, and an eager bf16 8192^3 GEMM runs on
that stream between replays (it also flushes L2).  The metric is block steps
per second (and us/step, and the HBM bandwidth that implies); one JSON line
on rank 0.  After the headline, the fp32-storage and the 32-sequence FP8
workloads are timed the same way (extra_configs; --no-extra skips them).

Per-class times come twice: from event pairs around every launch of eager
steps (eager_classes_*: the roofline's launch durations), and from the
kernels' own %globaltimer stamps inside a replayed graph (graph_classes_*:
each launch charged from the previous launch's end to its own end, so they
sum to the graph's device time).

--impl reference times the fp64 CPU oracle on the host cores instead (the
comparison arm of this tier): each step is one whole oracle block step of the
same workload with the rings prefilled (a bounded sample of the projections
only when W + K whole steps would not fit in a few minutes).

Multi-GPU (torchrun): every rank runs an independent replica (sequences are
independent; no collective in the data path); value = steps of all ranks /
max wall time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import pathlib
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "drafter block steps/s (us/step) at real dims; achieved HBM GB/s vs GB300 peak"
UNIT = "steps/s"
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="real_bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=30)
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of replays before timing")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the real_f32 and batched_fp8 lines after the headline")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (profiling captures only; not a bench line)")
    return ap.parse_args()


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak: the measured burst figure (a projection is timed
    on its own), else the fallback."""
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured bf16_tflops (burst)"
    return 1900.0, "fallback bf16 TFLOP/s"


def step_bytes(cfg, wl):
    """Algorithmic bytes of one step: GEMM weights (+FP8 scales) + ring K/V read + logits."""
    el = 2 if cfg.ring_dtype == "bf16" else 4
    ring = 2 * cfg.n_layer * cfg.n_head_kv * cfg.window * cfg.head_dim * el * cfg.n_seq
    if not cfg.inject:                       # batched: only the filled slots are keys
        ring = sum(2 * cfg.n_layer * cfg.n_head_kv * f * cfg.head_dim * el for f in wl.fills)
    logits = cfg.n_seq * 16 * cfg.n_vocab * 4
    return wl.weight_bytes() + ring + logits


def class_bytes(cfg, wl):
    """Algorithmic bytes per launch of each projection class (weights + scales)."""
    def wb(name):
        return wl.weights[name].nbytes()
    L = cfg.n_layer
    out = {
        "qkv": sum(wb(f"l{i}.{n}") for i in range(L) for n in ("wq", "wk", "wv")) / L,
        "o_proj": sum(wb(f"l{i}.wo") for i in range(L)) / L,
        "gate_up": sum(wb(f"l{i}.{n}") for i in range(L) for n in ("gate", "up")) / L,
        "down": sum(wb(f"l{i}.down") for i in range(L)) / L,
        "lm_head": wb("lm_head") + cfg.n_seq * 16 * cfg.n_vocab * 4,
    }
    # a projection chain (one launch per layer: o, gate/up, down, then the next
    # layer's q/k/v or the LM head) streams every layer's weights but layer 0's q/k/v
    out["chain"] = (L * (out["o_proj"] + out["gate_up"] + out["down"]) + (L - 1) * out["qkv"]
                    + out["lm_head"]) / L
    return out


def class_rates(cfg, wl, prof):
    """Algorithmic GB/s of every kernel class from the live per-class event times:
    bytes per launch (projection weights + scales, the LM head's logits; for
    attention one layer's ring K/V of every sequence) / mean launch time."""
    per_launch = dict(class_bytes(cfg, wl))
    per_launch["attention"] = (step_bytes(cfg, wl) - wl.weight_bytes()
                               - cfg.n_seq * 16 * cfg.n_vocab * 4) / cfg.n_layer
    out = {}
    for k, nbytes in per_launch.items():
        ms, n = prof.get(k, (0.0, 0))
        if n and ms > 0:
            out[k] = round(nbytes / (ms / n / 1e3) / 1e9, 1)
    return out


NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal

ALL_GEMM_SOURCES = ("gemm_tma.cu", "gemm_umma.cu", "gemm_fp4.cu", "gemm_common.cuh", "common.cuh",
                    "internal.h")


def gemm_source_hash(files=ALL_GEMM_SOURCES):
    """Hash of the sources a projection kernel is compiled from: a committed ncu
    traffic figure is used only while it matches."""
    h = hashlib.sha256()
    for f in files:
        h.update((ROOT / "block_diffusion_drafter_fc_gb300" / "csrc" / f).read_bytes())
    return h.hexdigest()[:16]


def committed_traffic(cfg_name, cls):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel (the entry's "sources", else every
    projection source); else None."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text())
    e = d.get(f"{cfg_name}/{cls}")
    if not e or e.get("source_sha") != gemm_source_hash(tuple(e.get("sources", ALL_GEMM_SOURCES))):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "100", "-i", str(gpu_index)], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def workload_config(cfg, wl, world):
    """The `config` object of both arms' JSON line."""
    ring = "ring full" if cfg.inject else f"rings filled {cfg.fill_lo}..{cfg.fill_hi}"
    return {"workload": f"{cfg.name}: {cfg.n_layer} layers, n_embd {cfg.n_embd}, heads "
                        f"{cfg.n_head}/{cfg.n_head_kv} x {cfg.head_dim}, n_ff {cfg.n_ff}, window "
                        f"{cfg.window} ({ring}), block 16, vocab {cfg.n_vocab}, "
                        f"{cfg.weight_dtype} weights, {cfg.ring_dtype} ring, fp32 arithmetic",
            "sequences": cfg.n_seq, "rows_per_step": 16 * cfg.n_seq,
            "l2": f"flushed between steps by the eager GEMM (400 MB of bf16 operands and result); "
                  f"the step itself streams {wl.weight_bytes() / 1e9:.2f} GB of weights",
            "timing": "CUDA-graph replays (step + accept), a CUDA event pair around each replay on "
                      "the replay stream, an eager bf16 8192^3 GEMM on the same stream between "
                      "replays (the target's verify traffic)",
            "parallelism": f"replicas x{world}"}


def replica_timing(ms_local, steps, world, device=None):
    """Max over the ranks of the timed region (ms) and the whole-job throughput of
    `world` independent replicas (steps/s: every rank's steps over the slowest
    rank's time).  Needs an initialised process group when world > 1."""
    ms = float(ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * steps / (ms / 1e3)


TRAFFIC_N = 8192      # eager bf16 GEMM between replays: [8192 x 8192] @ [8192 x 8192]


class Traffic:
    """The target model's verify work between drafter blocks, stood in for by
    one bf16 8192^3 GEMM on the replay stream (1.1 TFLOP; its 400 MB of
    operands and result also evict L2 between replays)."""

    def __init__(self, dev):
        import torch
        self.a = torch.randn(TRAFFIC_N, TRAFFIC_N, device=dev, dtype=torch.bfloat16) / 90.0
        self.b = torch.empty_like(self.a)

    def run(self):
        import torch
        torch.matmul(self.a, self.a, out=self.b)
        self.a, self.b = self.b, self.a


def timed_replays(dr, stream, traffic, steps):
    """Per-replay device times (ms) of `steps` graph replays, each bracketed by
    its own event pair on the replay stream with the eager traffic between them."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        dr.dflash_replay(stream)
        b.record(stream)
        traffic.run()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


PROJ = ("qkv", "o_proj", "gate_up", "down", "lm_head", "chain")


def graph_breakdown(dr, stream, traffic, replays):
    """Per-class time inside the replayed graph from the kernels' own
    %globaltimer stamps (a capture with timestamps on; same kernels, launch
    order and attributes as the timed graph).  Critical-path attribution: a
    launch is charged the time from the previous launch's end to its own end,
    so the classes sum to the graph's first-start-to-last-end time.  Also the
    mean time from a launch's own first CTA start to its last CTA end."""
    import numpy as np
    crit, span, n_l, total = {}, {}, {}, []
    for _ in range(replays):
        dr.dflash_replay(stream)
        st = dr.dflash_profile_stamps(stream)
        traffic.run()
        prev = 0.0
        for cls, t0, t1 in st:
            crit[cls] = crit.get(cls, 0.0) + (t1 - prev)
            span[cls] = span.get(cls, 0.0) + (t1 - t0)
            n_l[cls] = n_l.get(cls, 0) + 1
            prev = t1
        total.append(prev)
    return ({k: round(v / replays, 2) for k, v in crit.items()},
            {k: round(span[k] / n_l[k], 2) for k in span},
            {k: n_l[k] // replays for k in n_l}, round(float(np.mean(total)), 2))


def measure_config(args, name, dev, world, full=True):
    """Build the workload, prefill it, capture step + accept and time it as the
    headline is timed; returns the measurement dict (and the workload)."""
    import numpy as np
    import torch

    from block_diffusion_drafter_fc_gb300 import dflash as D
    from block_diffusion_drafter_fc_gb300.synth import BLOCK, get_config, make_targets, make_workload
    import gpu_harness as GH

    cfg = get_config(name)
    if args.layers:
        cfg = cfg.with_(n_layer=args.layers)
    wl = make_workload(cfg)
    dw, feats = GH.to_device(wl, dev)
    max_inject = max(c[2] for c in wl.inject_calls)
    dr = D.Drafter(cfg, dw, max_seq=cfg.n_seq, max_inject=max_inject, device=dev)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    GH.prefill(dr, wl, feats)                 # encode + inject of the whole context (untimed);
    torch.cuda.synchronize()                  # the second pass (same positions, same ring) is
    p0.record()                               # timed without first-launch costs
    GH.prefill(dr, wl, feats)
    p1.record()
    torch.cuda.synchronize()
    prefill_ms = p0.elapsed_time(p1)
    n = cfg.n_seq
    id_last = wl.id_last.to(dev)
    n_past = wl.n_past.to(dev)
    logits = torch.empty((n, BLOCK, cfg.n_vocab), dtype=torch.float32, device=dev)
    drafts = torch.empty((n, BLOCK - 1), dtype=torch.int32, device=dev)
    n_ok = torch.empty((n,), dtype=torch.int32, device=dev)
    dr.dflash_step(id_last, n_past, logits, drafts)
    targets = torch.from_numpy(make_targets(drafts.cpu().numpy(), wl.mismatch.numpy(),
                                            wl.tail.numpy(), cfg.n_vocab)).to(dev)
    stream = torch.cuda.current_stream()
    dr.dflash_capture(id_last, n_past, logits, drafts, targets, n_ok, stream)
    kernels, mem_nodes, _ = dr.dflash_graph_nodes()
    traffic = Traffic(dev)

    for _ in range(args.warmup):
        dr.dflash_replay(stream)
        traffic.run()
    torch.cuda.synchronize()
    sampler = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
    t_soak = time.time()                      # keep the GPU busy ~1 s before timing
    while time.time() - t_soak < args.soak:
        timed_replays(dr, stream, traffic, 10)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    per = timed_replays(dr, stream, traffic, args.steps)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.stop()
    ms, value = replica_timing(sum(per), args.steps, world, dev)
    ms_step = ms / args.steps
    per_us = np.array(per) * 1e3
    spread = {"replays": args.steps, "p10_us": round(float(np.percentile(per_us, 10)), 2),
              "median_us": round(float(np.median(per_us)), 2),
              "p90_us": round(float(np.percentile(per_us, 90)), 2)}

    # the same graph replayed back to back (no traffic between replays)
    n_b = max(10, min(args.steps, 200))
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(n_b):
        dr.dflash_replay(stream)
    b1.record(stream)
    torch.cuda.synchronize()
    b2b_us = b0.elapsed_time(b1) / n_b * 1e3
    out = {"cfg": cfg, "wl": wl, "value": value, "ms_step": ms_step, "spread": spread,
           "clocks": clocks, "prefill_ms": prefill_ms, "b2b_us": b2b_us,
           "graph_kernels": kernels, "graph_mem_nodes": mem_nodes}
    if not full:
        dr.close()
        return out

    # live per-class device times of eager steps (events on the launching stream)
    dr.dflash_profile_enable(1)
    for _ in range(args.profile_steps):
        dr.dflash_step(id_last, n_past, logits, drafts, stream)
    out["prof"] = dr.dflash_profile_read()
    # per-class times inside the replayed graph (device timestamps)
    dr.dflash_profile_enable(2)
    dr.dflash_capture(id_last, n_past, logits, drafts, targets, n_ok, stream)
    out["graph"] = graph_breakdown(dr, stream, traffic, max(10, args.profile_steps))
    dr.dflash_profile_enable(0)
    out.update(dr=dr, id_last=id_last, n_past=n_past, drafts=drafts)
    return out


def roofline_of(cfg, wl, prof, graph_span):
    """Roofline of the dominant kernel class: algorithmic bytes (or flops) per
    launch over its mean event-timed launch duration."""
    cb = class_bytes(cfg, wl)
    dom = max(cb, key=lambda k: prof.get(k, (0.0, 0))[0])
    dom_ms, dom_n = prof[dom]
    peak, peak_src = peaks()
    rows = 16 * cfg.n_seq
    span = graph_span.get(dom)
    if rows >= 128:
        # batched rows: the projections are dense contractions on the tensor
        # cores (bf16 kind::f16 MMA after exact widening of the stored weights),
        # so the roofline is the bf16 tensor peak; algorithmic flops = 2 M N K
        flops = 2.0 * rows * (cb[dom] - (cfg.n_seq * 16 * cfg.n_vocab * 4 if dom == "lm_head" else 0)) \
            / (1 if cfg.weight_dtype == "fp8" else 2 if cfg.weight_dtype == "bf16" else 4)
        t_peak, t_src = tensor_peak()
        t_ach = flops / (dom_ms / dom_n / 1e3) / 1e12 if dom_n else 0.0
        return {"bound": "tensor", "kernel": f"{dom} projection ({cfg.weight_dtype} weights, tcgen05)",
                "achieved": round(t_ach, 1), "peak": t_peak, "unit": "TFLOP/s",
                "frac": round(t_ach / t_peak, 4), "traffic": committed_traffic(cfg.name, dom),
                "peak_source": t_src, "flops_per_launch": flops,
                "avg_launch_us": round(dom_ms / dom_n * 1e3, 2) if dom_n else None,
                "graph_span_us": span}
    achieved = cb[dom] / (dom_ms / dom_n / 1e3) / 1e9 if dom_n else 0.0
    return {"bound": "hbm", "kernel": f"{dom} projection ({cfg.weight_dtype} weights)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": committed_traffic(cfg.name, dom),
            "peak_source": f"{peak_src} hbm_gbs", "bytes_per_launch": cb[dom],
            "avg_launch_us": round(dom_ms / dom_n * 1e3, 2) if dom_n else None,
            "graph_span_us": span,
            "graph_span_frac": round(cb[dom] / (span / 1e6) / 1e9 / peak, 4) if span else None}


def extra_config(args, name, dev, world):
    """A further configuration timed the same way (no CPU leg): step time,
    bandwidth or tensor fraction, per-class graph times, clocks."""
    import torch
    m = measure_config(args, name, dev, world)
    cfg, wl = m["cfg"], m["wl"]
    sbytes = step_bytes(cfg, wl)
    crit, span, _, _ = m["graph"]
    out = {"workload": workload_config(cfg, wl, world)["workload"],
           "value": round(m["value"], 3), "unit": UNIT, "us_per_step": round(m["ms_step"] * 1e3, 2),
           "replay_us": m["spread"], "back_to_back_us_per_step": round(m["b2b_us"], 2),
           "step_bytes": sbytes, "hbm_gbs": round(sbytes / m["ms_step"] / 1e6, 1),
           "roofline": roofline_of(cfg, wl, m["prof"], span),
           "graph_classes_us_per_step": crit, "clocks": m["clocks"]}
    m["dr"].close()
    del m
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    sys.path.insert(0, str(ROOT / "tests"))
    from block_diffusion_drafter_fc_gb300.synth import BLOCK
    m = measure_config(args, args.config, dev, world)
    cfg, wl, dr = m["cfg"], m["wl"], m["dr"]
    n = cfg.n_seq
    prof = m["prof"]
    crit, span, launches, graph_total = m["graph"]
    sbytes = step_bytes(cfg, wl)
    ms_step = m["ms_step"]
    peak, _ = peaks()
    cb = class_bytes(cfg, wl)
    graph_gbs = {k: round(cb[k] / (span[k] / 1e6) / 1e9, 1) for k in PROJ if span.get(k)}

    # end to end through the C ABI from host buffers (copies inside the timed region)
    hid = wl.id_last.clone().pin_memory()
    hnp = wl.n_past.clone().pin_memory()
    hdr = torch.empty((n, BLOCK - 1), dtype=torch.int32).pin_memory()
    n_e2e = 0 if args.no_e2e else max(10, min(args.steps, 200))
    e2e_s = float("nan")
    if n_e2e:
        for _ in range(3):
            dr.dflash_step_host(hid, hnp, hdr)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            dr.dflash_step_host(hid, hnp, hdr)
        e2e_s = (time.perf_counter() - t0) / n_e2e
        assert np.array_equal(hdr.numpy(), m["drafts"].cpu().numpy())

    out = {
        "metric": METRIC, "value": round(m["value"], 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2), "replay_us": m["spread"],
        "back_to_back_us_per_step": round(m["b2b_us"], 2),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 accumulate, 2xbf16-split activations",
        "data": "synthetic (seeded random weights ~N(0,1/fan_in), features ~N(0,1))",
        "config": workload_config(cfg, wl, world),
        "prefill_ms": round(m["prefill_ms"], 3),
        "step_bytes": sbytes,
        "hbm_gbs": round(sbytes / (ms_step / 1e3) / 1e9, 1),
        "hbm_frac_of_measured": round(sbytes / (ms_step / 1e3) / 1e9 / peak, 4),
        "hbm_frac_of_nominal": round(sbytes / (ms_step / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "roofline": roofline_of(cfg, wl, prof, span),
        "graph_classes_us_per_step": crit,
        "graph_first_start_to_last_end_us": graph_total,
        "graph_launch_span_us": span,
        "graph_launch_gbs": graph_gbs,
        "eager_classes_us_per_step": {k: round(v[0] / max(1, args.profile_steps) * 1e3, 2)
                                      for k, v in prof.items() if v[1]},
        "eager_classes_gbs": class_rates(cfg, wl, prof),
        "gpu_launches": m["graph_kernels"] * args.steps,
        "graph_nodes": {"kernels": m["graph_kernels"], "mem_alloc_free": m["graph_mem_nodes"]},
        "clocks": m["clocks"],
        "e2e": {"value": round(1.0 / e2e_s * world, 3) if n_e2e else None, "unit": UNIT,
                "h2d_bytes_per_step": 8 * n, "d2h_bytes_per_step": 4 * n * (BLOCK - 1)},
    }
    dr.close()
    del m, dr
    torch.cuda.empty_cache()
    if not args.no_extra and world == 1 and not args.layers:
        out["extra_configs"] = {name: extra_config(args, name, dev, world)
                                for name in ("real_f32", "batched_fp8") if name != args.config}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl)
    return out


def oracle_ring_full(wl):
    """The oracle's weights and rings after the workload's whole prefill (the
    rings the timed step reads)."""
    sys.path.insert(0, str(ROOT / "tests"))
    import oracle_bridge as OB
    w, rings, _ = OB.oracle_prefill(wl)
    return w, rings


def oracle_step_once(wl, w, rings):
    """One whole oracle block step (embedding, every layer, LM head, greedy
    drafts, acceptance against the workload's targets); returns its seconds."""
    from oracle import dflash_oracle as O
    from block_diffusion_drafter_fc_gb300.synth import make_targets
    t0 = time.perf_counter()
    _, drafts = O.step(w, rings, wl.id_last.numpy(), wl.n_past.numpy())
    O.accept(drafts, make_targets(drafts, wl.mismatch.numpy(), wl.tail.numpy(), wl.cfg.n_vocab))
    return time.perf_counter() - t0


def cpu_baseline(wl):
    """The oracle as it stands: one whole block step on the host cores with the
    rings as the timed GPU step sees them (prefilled, untimed)."""
    w, rings = oracle_ring_full(wl)
    dt = oracle_step_once(wl, w, rings)
    return {"value": round(1.0 / dt, 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"one whole fp64 oracle block step of {wl.cfg.name} ({wl.cfg.n_seq} seq, "
                      f"rings prefilled as in the GPU run), {dt:.1f} s"}


REF_BUDGET_S = 240.0   # the reference arm's whole --warmup + --steps run


def run_reference(args):
    """Oracle arm: every step is one whole fp64 oracle block step of the same
    workload (rings prefilled, untimed), so steps/s = steps / time.  Should
    W + K whole steps not fit in REF_BUDGET_S, each step is instead a bounded
    sample: the oracle's decode + linear of a row block of the step's
    projection weights on the step's activation rows, scaled to steps/s by
    the fraction of the step's weight elements it covers."""
    import numpy as np
    sys.path.insert(0, str(ROOT / "tests"))
    from oracle import dflash_oracle as O
    import oracle_bridge as OB
    from block_diffusion_drafter_fc_gb300.synth import get_config, make_workload

    cfg = get_config(args.config)
    wl = make_workload(cfg)
    w, rings = oracle_ring_full(wl)
    t_first = oracle_step_once(wl, w, rings)   # one untimed step: the size estimate
    whole = (args.steps + args.warmup) * t_first <= REF_BUDGET_S
    line = {"impl": "reference", "metric": METRIC, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, wl, args.gpus)}
    if whole:
        for _ in range(max(0, args.warmup - 1)):
            oracle_step_once(wl, w, rings)
        dt = sum(oracle_step_once(wl, w, rings) for _ in range(args.steps))
        value = args.steps / dt
        sample = (f"{args.steps} whole fp64 oracle block steps of {cfg.name} ({cfg.n_seq} seq, "
                  f"rings prefilled), {dt / args.steps:.2f} s each")
    else:
        names = [f"l{i}.{n}" for i in range(cfg.n_layer)
                 for n in ("wq", "wk", "wv", "wo", "gate", "up", "down")]
        names.append("lm_head")
        dims = {n: tuple(wl.weights[n].shape) for n in names}    # [N, K] of every matrix
        total = sum(dims[n][0] * dims[n][1] for n in names)
        rng = np.random.default_rng(0)
        x = {k: rng.standard_normal((16 * cfg.n_seq, k)) for k in {dims[n][1] for n in names}}

        def rows_of(n, r0, rows):
            raw = w.raw[n]
            if w.dtype_of(n) != "fp4":
                return raw[r0:r0 + rows]
            N, K = dims[n]
            flat = raw.reshape(-1)
            codes = flat[r0 * K // 2:(r0 + rows) * K // 2]
            scales = flat[N * K // 2 + (r0 // 16) * K:N * K // 2 + ((r0 + rows) // 16) * K]
            return np.concatenate([codes, scales])

        def sample_rows(i, rows):
            n = names[i % len(names)]
            N, K = dims[n]
            r0 = ((i * rows) % max(1, N - rows)) // 16 * 16
            rr = min(rows, N - r0) // 16 * 16 or min(rows, N - r0)
            sc = w.scales.get(n)
            W = O.decode(rows_of(n, r0, rr), w.dtype_of(n), None if sc is None else sc[r0:r0 + rr])
            O.linear(x[K], W)
            return rr * K

        per_step_s = REF_BUDGET_S / max(1, args.steps + args.warmup)
        frac = per_step_s / t_first
        avg_k = total / sum(dims[n][0] for n in names)
        rows = int(max(16, frac * total / avg_k)) // 16 * 16
        for i in range(args.warmup):
            sample_rows(i, rows)
        done = 0
        t0 = time.perf_counter()
        for i in range(args.steps):
            done += sample_rows(i + args.warmup, rows)
        dt = time.perf_counter() - t0
        value = (done / total) / dt
        sample = (f"{rows} weight rows of one projection per step (decode + linear on "
                  f"{16 * cfg.n_seq} rows), cycling all projections; a whole step takes "
                  f"{t_first:.2f} s")
    line.update({"value": round(value, 5), "ms_per_step": round(1e3 / value, 3),
                 "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": os.cpu_count(),
                                  "kind": "oracle", "sample": sample},
                 "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0}})
    return line


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    out = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
