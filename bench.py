#!/usr/bin/env python3
"""Throughput of one FAST-AR attention layer step (TempCache + AnnSA + AnnCA) on GB300.

Prints ONE JSON line (rank 0).  Workload: a Wan2.1-1.3B-shaped layer (12 heads, d=128,
chunks of 3 latent frames x 30x52 tokens, cache cap M=9360, 64 buckets, r=2, 512
prompt tokens), its cache warmed by running the step itself through 7 earlier
chunks (21 frames).  One timed step = the whole per-chunk step captured as one CUDA
graph; L2 is flushed between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fastar|reference]

Under torchrun every rank runs its own layer instance (independent head groups: the
step has no cross-rank exchange), so scaling is weak and value = all ranks' query
tokens / the slowest rank's time.  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FAST-AR layer query-tokens/s at Wan-1.3B shape; % of HBM/TC roofline"
UNIT = "query-tokens/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="fastar", choices=["fastar", "reference"])
    p.add_argument("--config", default="wan13b_layer")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-dense", action="store_true", help="skip the dense-baseline timing")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle timing")
    p.add_argument("--no-rollout", action="store_true", help="skip the long-rollout stability run")
    p.add_argument("--no-dit", action="store_true", help="skip the whole-transformer (DiT) chunk denoise run")
    p.add_argument("--dit-chunks", type=int, default=20, help="chunks of the DiT rollout (3 latent frames each)")
    p.add_argument("--no-configs", action="store_true", help="skip the other layer shapes (HunyuanVideo 720p, tiny)")
    p.add_argument("--cpu-sample", nargs=4, metavar=("CONFIG", "FLOAT", "HEADS", "SEED"), default=None,
                   help=argparse.SUPPRESS)   # internal: one timed oracle sample (run in a child process)
    return p.parse_args()


# ---------------------------------------------------------------------------------------
# process group (one process per GPU)
# ---------------------------------------------------------------------------------------

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(tokens_per_rank: int, seconds_per_rank: float, world: int):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    t = reduce_max(seconds_per_rank, world)
    return tokens_per_rank * world / t, t


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def ready(self, n: int = 2) -> bool:
        """True once n samples are in (or there is no sampler)."""
        return self.proc is None or self.proc.poll() is not None or self._lines() >= n

    def _lines(self) -> int:
        self.out.flush()
        try:
            with open(self.path) as fh:
                return sum(1 for _ in fh)
        except OSError:
            return 0

    def _wait_lines(self, n: int, timeout: float):
        t0 = time.time()
        while self._lines() < n and time.time() - t0 < timeout and self.proc.poll() is None:
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return None
        # one more sample after the timed region, so that the samples bracket it
        self._wait_lines(self._lines() + 1, 1.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "window": "every 50 ms from before the warm-up steps to just after the timed "
                                              "steps"}


# ---------------------------------------------------------------------------------------
# roofline bookkeeping (algorithmic units per launch)
# ---------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def stage_units(cfg, layer, n_in):
    """Algorithmic bytes and flops of each stage for the measured step (bf16 = 2 B).

    n_in: per-head cache length entering the step.  Bytes are the method minimum: each
    operand a stage needs is read once and each result written once; implementation
    overheads (moving surviving cache rows, the slots' partial results) are not counted.
    Flops are the contractions the method defines (2 per multiply-add); the sparse
    attention counts 4*d*sum_b |Q_b||K_b| from the step's own bucket histograms."""
    import numpy as np
    H, d, Nq, B, r, P, F, Tf, M = cfg.H, cfg.d, cfg.Nq, cfg.B, cfg.r, cfg.P, cfg.F, cfg.Tf, cfg.M
    e = 2 if cfg.dtype == "bf16" else 4
    row = d * e
    qoff = layer.qoff.cpu().numpy().astype(np.int64)
    koff = layer.koff.cpu().numpy().astype(np.int64)
    qcnt, kcnt_b = np.diff(qoff, axis=1), np.diff(koff, axis=1)
    pairs = float((qcnt * kcnt_b).sum())
    L_out = layer.caches[1 - layer.cur].len.cpu().numpy().astype(np.int64)
    kcnt = layer.kcnt.cpu().numpy().astype(np.int64)
    n_tot = float(np.sum(n_in))
    u = {}
    u["bucket_assign"] = dict(bytes=2 * H * Nq * row + 2 * H * B * row, flops=2.0 * 2 * H * Nq * B * d)
    u["tempcache_match"] = dict(bytes=H * Nq * row * 2 + n_tot * (row + 4), flops=2.0 * Nq * d * n_tot)
    # the chunk's K/V read and appended to the cache, the index map written
    u["cache_compact"] = dict(bytes=4.0 * H * Nq * row + 4.0 * H * M, flops=0.0)
    u["bucket_sort"] = dict(bytes=4.0 * float(L_out.sum()) * 2, flops=0.0)
    u["bucket_sort_q"] = dict(bytes=4.0 * H * Nq * r * 2, flops=0.0)
    if getattr(layer, "presort", False):
        # the sorted compaction's planning launch also sorts the new keys and the step's
        # (query, slot) pairs by bucket: those bytes belong to its stage
        u["cache_compact"]["bytes"] += u["bucket_sort"]["bytes"] + u["bucket_sort_q"]["bytes"]
    u["sparse_attn"] = dict(bytes=H * Nq * row * 2 + 2 * float(L_out.sum()) * row, flops=4.0 * d * pairs)
    u["annca_select"] = dict(bytes=H * Nq * row + H * P * row, flops=2.0 * H * Nq * P * d)
    u["cross_attn_subset"] = dict(bytes=H * Nq * row * 2 + 2 * float(kcnt.sum()) * row,
                                  flops=4.0 * d * Tf * float(kcnt.sum()))
    return u


def hold_gpu(torch, cycles=6_000_000):
    """Keeps the GPU busy (a spin of about 3 ms) while the host enqueues an eager step, so
    that per-stage events bracket GPU work only, not the host's launch time between calls."""
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(cycles)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic_wan13b_layer.json")


def recorded_traffic(stage, workload):
    """DRAM bytes per launch of a stage from the committed ncu record, or None when the
    record is for another workload or a source file of the stage changed since."""
    import hashlib
    try:
        rec = json.load(open(TRAFFIC_FILE))
    except (OSError, ValueError):
        return None
    if not rec.get("workload", "").startswith(workload + " "):
        return None
    e = rec.get("stages", {}).get(stage)
    if not e:
        return None
    for f, h in e.get("sources_sha256", {}).items():
        path = os.path.join(ROOT, "kv_cache_tempcache_gb300", "csrc", f)
        if not os.path.exists(path) or hashlib.sha256(open(path, "rb").read()).hexdigest() != h:
            return None
    return int(e["bytes_per_launch"])


PEAK_NOTE = ("measured burst bf16 peak: each stage is timed alone in an eager pass well under a "
             "millisecond, not inside a seconds-long loop")


def roofline_of(name, avg_ms, units, peaks):
    b, f = units["bytes"], units["flops"]
    tpk = peaks["bf16_tflops"]
    t_mem = b / (peaks["hbm_gbs"] * 1e9)
    t_tc = f / (tpk * 1e12)
    s = avg_ms * 1e-3
    if t_tc >= t_mem:
        ach = f / s / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": round(ach, 3), "peak": tpk, "unit": "TFLOP/s",
                "frac": round(ach / tpk, 5), "traffic": None, "algorithmic_flops": f, "avg_ms": round(avg_ms, 4),
                "peak_source": peaks["source"] + " burst (" + PEAK_NOTE + ")"}
    ach = b / s / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": round(ach, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 5), "traffic": None, "algorithmic_bytes": b,
            "avg_ms": round(avg_ms, 4), "peak_source": peaks["source"]}


def step_roofline(units, peaks, ms):
    """Sum over the stages of max(method-minimum bytes / HBM, flops / bf16 burst), against
    the measured step."""
    t = sum(max(u["bytes"] / (peaks["hbm_gbs"] * 1e9), u["flops"] / (peaks["bf16_tflops"] * 1e12))
            for u in units.values())
    return {"time_us": round(t * 1e6, 2), "frac": round(t * 1e3 / ms, 5),
            "note": "sum over the stages of max(method-minimum bytes / measured HBM, algorithmic flops / measured "
                    "bf16 burst), divided by the measured step (graph replay)"}


def config_of(cfg, world):
    """The workload description both arms print (identical strings)."""
    return {"workload": f"{cfg.name}: H={cfg.H} d={cfg.d} chunk={cfg.F}x{cfg.Tf} (Nq={cfg.Nq}) "
                        f"M={cfg.M} B={cfg.B} r={cfg.r} P={cfg.P} tau={cfg.tau} tau_ca={cfg.tau_ca}",
            "l2": "GPU arm: flushed between timed steps (256 MiB memset outside the events); CPU oracle arm: n/a",
            "parallelism": f"replicas x{world} (independent head groups, no exchange)"}


# ---------------------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------------------

def make_layer(cfg, tdt, dev, **kw):
    from kv_cache_tempcache_gb300.layer import FastARLayer
    args = dict(H=cfg.H, d=cfg.d, Tf=cfg.Tf, F=cfg.F, M=cfg.M, B=cfg.B, r=cfg.r, P=cfg.P, tau=cfg.tau,
                tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=tdt, device=dev)
    args.update(kw)
    return FastARLayer(**args)


def timed_graph(graph, flush, steps, torch):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def measure_layer(cfg, args, world, dev, flush, clocks=None, main=True):
    """One layer shape: the step as a replayed CUDA graph (L2 flushed before each), its
    stages one by one, the roofline, the end-to-end pipeline through the public API with
    host buffers, the dense baseline; main=True adds the variants and ablations."""
    import numpy as np
    import torch
    from kv_cache_tempcache_gb300 import synth, _lib
    from kv_cache_tempcache_gb300.layer import DenseLayer

    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(tdt)
    rank = int(os.environ.get("RANK", "0"))
    gen = synth.DriftingMixture(cfg, seed=args.seed + rank)
    layer = make_layer(cfg, tdt, dev)
    layer.set_centroids(up(gen.centroids))
    kp, vp = gen.prompt
    layer.set_prompt(up(kp), up(vp))
    hist_k, hist_v = [], []
    n_prior_chunks = cfg.prior_frames // cfg.F
    for _ in range(n_prior_chunks):             # warm the cache through the earlier chunks
        k, v, q = gen.next_chunk()
        hist_k.append(k)
        hist_v.append(v)
        layer.step(up(q), up(k), up(v))
    k, v, q = gen.next_chunk()                  # the measured chunk
    q_d, k_d, v_d = up(q), up(k), up(v)
    torch.cuda.synchronize(dev)
    n_in = layer.cache.len.cpu().numpy()
    l0 = _lib.kernel_launches()
    layer.step(q_d, k_d, v_d, advance=False)
    torch.cuda.synchronize(dev)
    launches_per_step = _lib.kernel_launches() - l0
    assert layer.status() == 0, f"device status {layer.status()}"
    graph = layer.capture(q_d, k_d, v_d)

    soak = 0
    if clocks is not None:
        # keep the GPU under load while the clock sampler comes up (at most 5 s), so that
        # its samples see the clocks of a busy GPU; then the counted warm-up steps
        t_soak = time.time()
        while not clocks.ready(2) and time.time() - t_soak < 5.0:
            for _ in range(20):
                flush.zero_()
                graph.replay()
            soak += 20
            torch.cuda.synchronize(dev)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    barrier(world)
    step_ms = timed_graph(graph, flush, args.steps, torch)
    barrier(world)
    clk = clocks.stop() if clocks is not None else None
    ms = sum(step_ms) / len(step_ms)
    # the same replays without the flush (inputs and cache may stay in L2): context only
    ev_w = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in ev_w:
        e0.record()
        graph.replay()
        e1.record()
    torch.cuda.synchronize(dev)
    warm_ms = [e0.elapsed_time(e1) for e0, e1 in ev_w]
    value, t_max = aggregate(cfg.Nq * args.steps, sum(step_ms) * 1e-3, world)

    # per-stage timing: an eager pass with every kernel on one stream, so that each
    # stage's events bracket that stage alone (in the graph the AnnCA branch overlaps)
    stage_ev = {}

    def timer(name, stream, phase):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        stage_ev.setdefault(name, []).append(e)

    for _ in range(args.steps):
        hold_gpu(torch)
        flush.zero_()
        layer.step(q_d, k_d, v_d, advance=False, timer=timer, serial=True)
    torch.cuda.synchronize(dev)
    stages = {}
    for name, es in stage_ev.items():
        d = [es[i].elapsed_time(es[i + 1]) for i in range(0, len(es), 2)]
        stages[name] = sum(d) / len(d)
    peaks = load_peaks()
    units = stage_units(cfg, layer, n_in)
    dom = max((s_ for s_ in stages if s_ in units), key=lambda s_: stages[s_])
    roof_all = {s_: roofline_of(s_, stages[s_], units[s_], peaks) for s_ in stages if s_ in units}
    for s_, r_ in roof_all.items():
        r_["traffic"] = recorded_traffic(s_, cfg.name)

    # end to end through the public API, as a streaming pipeline: every step copies its
    # inputs in from pinned host memory and its outputs back out, and step i+1's inputs
    # travel (copy-in stream) while step i computes, step i's outputs while step i+1
    # computes (copy-out stream).  Two input sets and two output pairs, one graph each (the
    # second graph writes its outputs into its own pair); the L2 flush before every step
    # stays inside the timed region.
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(tdt).pin_memory()
    q_h, k_h, v_h = pin(q), pin(k), pin(v)
    ins = [(q_d, k_d, v_d), tuple(torch.empty_like(t) for t in (q_d, k_d, v_d))]
    outs_d = [(layer.o_self, layer.o_cross), (torch.empty_like(layer.o_self), torch.empty_like(layer.o_cross))]
    layer.o_self, layer.o_cross = outs_d[1]
    graphs2 = [graph, layer.capture(*ins[1])]
    layer.o_self, layer.o_cross = outs_d[0]
    outs_h = [(torch.empty_like(layer.o_self, device="cpu").pin_memory(),
               torch.empty_like(layer.o_cross, device="cpu").pin_memory()) for _ in range(2)]
    os_h, oc_h = outs_h[0]
    mainst = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, out_ready, out_free = [ev() for _ in range(2)], [ev() for _ in range(2)], \
        [ev() for _ in range(2)], [ev() for _ in range(2)]
    for b in range(2):
        in_free[b].record(mainst)
        out_free[b].record(mainst)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(mainst)
    s_in.wait_event(e0)

    def copy_in(i):
        b = i % 2
        s_in.wait_event(in_free[b])
        with torch.cuda.stream(s_in):
            for dst, src in zip(ins[b], (q_h, k_h, v_h)):
                dst.copy_(src, non_blocking=True)
        in_ready[b].record(s_in)

    copy_in(0)
    for i in range(args.steps):
        b = i % 2
        if i + 1 < args.steps:
            copy_in(i + 1)
        mainst.wait_event(in_ready[b])
        mainst.wait_event(out_free[b])   # step i-2's outputs (this graph's pair) are out
        flush.zero_()
        graphs2[b].replay()
        in_free[b].record(mainst)
        out_ready[b].record(mainst)
        s_out.wait_event(out_ready[b])
        with torch.cuda.stream(s_out):
            outs_h[b][0].copy_(outs_d[b][0], non_blocking=True)
            outs_h[b][1].copy_(outs_d[b][1], non_blocking=True)
        out_free[b].record(s_out)
    mainst.wait_stream(s_out)
    e1.record(mainst)
    torch.cuda.synchronize(dev)
    e2e_val, _ = aggregate(cfg.Nq * args.steps, e0.elapsed_time(e1) * 1e-3, world)
    # both graphs compute the same step from the same host inputs: their outputs as read out
    e2e_agree = bool(torch.equal(outs_h[0][0], outs_h[1][0]) and torch.equal(outs_h[0][1], outs_h[1][1])) \
        if args.steps >= 2 else None
    nb = lambda t: t.numel() * t.element_size()
    del graphs2

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(t_max * 1e3 / args.steps, 4),
        "ms_per_step_median": round(statistics.median(step_ms), 4),
        "warm_l2": {"ms_per_step_median": round(statistics.median(warm_ms), 4),
                    "note": "same graph replayed back to back without the L2 flush"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded drifting Gaussian-mixture keys; no dataset, no weights)",
        "config": config_of(cfg, world),
        "notes": {"cache": f"warmed by {n_prior_chunks} earlier chunks ({cfg.prior_frames} frames); "
                           f"{int(n_in.sum())} entries in, {int(layer.caches[1 - layer.cur].len.sum())} out",
                  "warmup_extra": f"{soak} untimed replays while the clock sampler started",
                  "stages": "per-stage times from an eager pass with all kernels on one stream, enqueued behind a "
                            "GPU spin so that host launch time between calls is not counted"},
        "latent_frames_per_s": round(value / cfg.Tf, 2),
        "roofline": roof_all[dom],
        "step_roofline": step_roofline(units, peaks, ms),
        "stages_ms": {s_: round(v_, 4) for s_, v_ in stages.items()},
        "stages_roofline_frac": {s_: r_["frac"] for s_, r_ in roof_all.items()},
        "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": nb(q_h) + nb(k_h) + nb(v_h),
                "d2h_bytes_per_step": nb(os_h) + nb(oc_h),
                "outputs_agree": e2e_agree,
                "note": "one timed region over all steps: copy-in of step i+1 and copy-out of step i overlap "
                        "step i+1's compute (two input sets and two output pairs, one graph each); L2 flushed before "
                        "every step inside the region"},
        "gpu_launches": int(launches_per_step * args.steps),
        "device_bytes": layer.device_bytes(),
    }
    if clk is not None:
        out["clocks"] = clk
    if main:
        # the ANN-restricted match (a variant of the TempCache match): timed beside the exact
        # match on the measured chunk's incoming cache, with the agreement of their choices
        out["ann_match"] = time_ann_match(layer, cfg, q_d, k_d, flush, args.steps, torch, _lib)
        # the merge variant (Lemma 5.1): its own layer warmed through the same chunks, its
        # step timed as a graph beside the replace step above
        out["merge"] = time_merge_variant(cfg, args.seed + rank, up, flush, args.steps, ms, torch, dev)
        # the quantised match (product quantization of the cached keys), beside the exact match
        if hist_k and cfg.dtype == "bf16":
            out["pq_match"] = time_pq_match(layer, cfg, q_d, k_d, flush, args.steps, torch, _lib, hist_k[0],
                                            args.seed)
    del graph
    layer._graph = None
    # dense baseline from the same build: append-only cache, full attention
    dms = None
    if not args.no_dense:
        hk = np.concatenate(hist_k, axis=1)
        hv = np.concatenate(hist_v, axis=1)
        dense = DenseLayer(cfg.H, cfg.d, cfg.Nq, hk.shape[1] + cfg.Nq, cfg.P, dtype=tdt, device=dev)
        dense.load_history(up(hk), up(hv))
        dense.set_prompt(up(kp), up(vp))
        for _ in range(2):
            dense.step(q_d, k_d, v_d, advance=False)
        dts = []
        for _ in range(max(3, args.steps // 4)):
            hold_gpu(torch)
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record()
            dense.step(q_d, k_d, v_d, advance=False)
            b_.record()
            dts.append((a_, b_))
        torch.cuda.synchronize(dev)
        dms = sum(a_.elapsed_time(b_) for a_, b_ in dts) / len(dts)
        out["dense"] = {"ms_per_step": round(dms, 4), "keys": int(hk.shape[1] + cfg.Nq),
                        "speedup_fastar_vs_dense": round(dms / ms, 3)}
        del dense
    if main:
        out["tempcache_only"] = time_tempcache_only(cfg, args, dev, flush, dms)
    del layer
    torch.cuda.empty_cache()
    return out


def time_tempcache_only(cfg, args, dev, flush, dense_ms):
    """The TempCache ablation (technical summary, Key Results: TempCache alone): the exact
    match, eviction and compaction bound the cache as in the full step, but attention is
    dense over the bounded cache (one bucket per head, r = 1) and cross-attention is over
    every prompt token (tau_ca = -1 keeps all); timed as a graph like the full step."""
    import numpy as np
    import torch
    from kv_cache_tempcache_gb300 import synth
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(tdt)
    rank = int(os.environ.get("RANK", "0"))
    gen = synth.DriftingMixture(cfg, seed=args.seed + rank)
    layer = make_layer(cfg, tdt, dev, B=1, r=1, tau_ca=-1.0, topk=cfg.P)
    one = np.zeros((cfg.H, 1, cfg.d), np.float32)
    one[:, 0, 0] = 1.0                           # every key and query in the one bucket
    layer.set_centroids(up(one))
    kp, vp = gen.prompt
    layer.set_prompt(up(kp), up(vp))
    for _ in range(cfg.prior_frames // cfg.F):
        k, v, q = gen.next_chunk()
        layer.step(up(q), up(k), up(v))
    k, v, q = gen.next_chunk()
    q_d, k_d, v_d = up(q), up(k), up(v)
    graph = layer.capture(q_d, k_d, v_d)
    for _ in range(3):
        flush.zero_()
        graph.replay()
    ms = statistics.mean(timed_graph(graph, flush, args.steps, torch))
    assert layer.status() == 0
    res = {"ms_per_step": round(ms, 4), "keys_attended": int(layer.caches[1 - layer.cur].len.sum()) // cfg.H,
           "note": "exact match + eviction + compaction (cache capped at M), dense attention over the bounded "
                   "cache, cross-attention over the whole prompt; graph replay, L2 flushed before each"}
    if dense_ms:
        res["speedup_vs_dense"] = round(dense_ms / ms, 3)
    del graph, layer
    torch.cuda.empty_cache()
    return res


def measure_tiny(args, dev, flush):
    """Latency of the tiny fp32 layer step (1 head, 256 queries, a 768-entry cache) as a
    replayed graph: the launch-bound case, reported as time per step."""
    import numpy as np
    import torch
    from kv_cache_tempcache_gb300 import synth
    cfg = synth.TINY_FP32
    inp = synth.layer_step_inputs(cfg, seed=args.seed)
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    layer = make_layer(cfg, torch.float32, dev)
    layer.set_centroids(up(inp["centroids"]))
    layer.set_prompt(up(inp["kp"]), up(inp["vp"]))
    n = min(cfg.M, inp["history_k"].shape[1])
    layer.load_cache(up(inp["history_k"][:, -n:]), up(inp["history_v"][:, -n:]))
    q_d, k_d, v_d = up(inp["q"]), up(inp["k_cur"]), up(inp["v_cur"])
    graph = layer.capture(q_d, k_d, v_d)
    for _ in range(10):
        graph.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for e0, e1 in ev:
        e0.record()
        graph.replay()
        e1.record()
    torch.cuda.synchronize(dev)
    warm = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
    cold = statistics.median(timed_graph(graph, flush, 20, torch))
    assert layer.status() == 0
    res = {"workload": f"{cfg.name}: H={cfg.H} d={cfg.d} Nq={cfg.Nq} n={n} M={cfg.M} B={cfg.B} r={cfg.r} "
                       f"P={cfg.P} fp32", "latency_us_median": round(warm * 1e3, 2),
           "latency_us_median_l2_flushed": round(cold * 1e3, 2),
           "note": "the whole step as one replayed graph; launch-bound at this size"}
    del graph, layer
    return res


def run_fastar(args, rank, world, local):
    import torch
    from kv_cache_tempcache_gb300 import synth
    from kv_cache_tempcache_gb300.build_lib import build

    if rank == 0 or not os.path.exists(os.path.join(ROOT, "kv_cache_tempcache_gb300", "libfastar.so")):
        build()
    barrier(world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.CONFIGS[args.config]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(local)
    clocks.start()
    out = measure_layer(cfg, args, world, dev, flush, clocks=clocks, main=True)
    if not args.no_rollout and cfg.name == "wan13b_layer":
        out["rollout"] = measure_rollout(cfg, args.seed + rank, flush, torch, dev)
    if not args.no_configs and cfg.name == "wan13b_layer":
        # the other layer shapes: the HunyuanVideo-shaped 720p layer, measured the same way,
        # and the latency of the tiny fp32 step
        other = synth.HUNYUAN720P_LAYER
        line = measure_layer(other, args, world, dev, flush, clocks=None, main=False)
        if rank == 0 and world == 1 and not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(other, args.seed, budget_s=5.0, variants=False)
        out["configs"] = {other.name: line, "tiny_fp32": measure_tiny(args, dev, flush)}
    if not args.no_dit and cfg.name == "wan13b_layer":
        torch.cuda.empty_cache()
        try:
            out["dit"] = measure_dit(args.dit_chunks, args.seed + rank, torch, dev)
        except Exception as exc:   # the layer's line must survive a failure of the wider run
            out["dit"] = {"error": f"{type(exc).__name__}: {exc}"[:300]}
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(cfg, args.seed, budget_s=12.0)
    return out


# ---------------------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------------------

def _oracle_case(cfg, seed):
    from kv_cache_tempcache_gb300 import synth
    inp = synth.layer_step_inputs(cfg, seed=seed)
    n = min(cfg.M, inp["history_k"].shape[1])
    return inp, inp["history_k"][:, -n:], inp["history_v"][:, -n:]


def _oracle_head(cfg, inp, ck, cv, h):
    from oracle import fastar_oracle as O
    return O.head_step(inp["q"][h], inp["k_cur"][h], inp["v_cur"][h], ck[h], cv[h], inp["centroids"][h],
                       inp["kp"][h], inp["vp"][h], F=cfg.F, Tf=cfg.Tf, tau=cfg.tau, M=cfg.M, r=cfg.r,
                       tau_ca=cfg.tau_ca, topk=cfg.topk, scale=cfg.scale)


MARGIN = 1e-4   # the method spec's near-tie margin (relative; absolute for the thresholds)


def near_ties(cfg, inp, h, res):
    """Decisions of one head whose oracle scores leave them within the near-tie margin,
    where either choice is a correct answer: query top-r and key arg-max buckets, top-1
    matches, eviction and prompt-keep thresholds, the top-k edge of the kept sets."""
    import numpy as np
    from oracle import fastar_oracle as O
    C = inp["centroids"][h]

    def gap(S, k):   # rows whose k-th and (k+1)-th largest scores are within the margin
        if S.shape[1] <= k:
            return 0
        part = -np.sort(-S, axis=1)[:, :k + 1]
        return int((part[:, k - 1] - part[:, k] < MARGIN * np.abs(part[:, k - 1])).sum())

    c = {"query_buckets": gap(O.centroid_scores(inp["q"][h], C), cfg.r),
         "key_buckets": gap(O.centroid_scores(inp["k_cur"][h], C), 1)}
    s1, s2 = res["s1"], res["s2"]
    fin = np.isfinite(s2)
    c["top1"] = int((s1[fin] - s2[fin] < MARGIN * np.abs(s1[fin])).sum())
    ce = res["cos_evict"]
    c["evict_threshold"] = int((np.abs(ce[np.isfinite(ce)] - cfg.tau) < MARGIN).sum())
    sc = res["score"]
    keep_amb = int((np.abs(sc[np.isfinite(sc)] - cfg.tau_ca) < MARGIN).sum())
    k = min(cfg.topk, cfg.P)
    for f in range(sc.shape[0]):
        o = -np.sort(-sc[f])
        if 0 < k < cfg.P and np.isfinite(o[k - 1]):
            keep_amb += int((np.abs(sc[f] - o[k - 1]) <= MARGIN * abs(o[k - 1])).sum()) - 1
    c["keep"] = keep_amb
    return c


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def oracle_sample(cfg, seed, float_name, heads, budget_s):
    """Times the oracle (as it stands, in the given float type) on up to `heads` whole heads
    of one step, at least one, stopping once the budget is spent.  Returns (heads done,
    seconds, near-tie counts summed over those heads)."""
    import numpy as np
    from oracle import fastar_oracle as O
    inp, ck, cv = _oracle_case(cfg, seed)
    O.FLOAT = np.float32 if float_name == "float32" else np.float64
    t0 = time.perf_counter()
    done, ties = 0, {}
    while done < min(heads, cfg.H) and (done == 0 or time.perf_counter() - t0 < budget_s):
        res = _oracle_head(cfg, inp, ck, cv, done)
        if O.FLOAT == np.float64:
            for k_, v_ in near_ties(cfg, inp, done, res).items():
                ties[k_] = ties.get(k_, 0) + v_
        done += 1
    dt = time.perf_counter() - t0
    O.FLOAT = np.float64
    return done, dt, ties


def cpu_baseline(cfg, seed, budget_s=12.0, variants=True):
    """The oracle as it stands (float64 NumPy, every core's BLAS threads) on whole heads of
    the same step until the budget is spent, scaled to query tokens per second of the whole
    layer; beside it the same code in float32 (the precision the method spec names for a CPU
    baseline) and both with one thread (child processes with the BLAS thread pools set to
    one).  Also the number of near-tie decisions in the sampled heads."""
    heads, dt, ties = oracle_sample(cfg, seed, "float64", cfg.H, budget_s)
    per_step = dt / heads * cfg.H
    out = {"value": round(cfg.Nq / per_step, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": f"{heads} of {cfg.H} heads of one {cfg.name} step (float64 NumPy, all cores, cache of the "
                     f"{min(cfg.M, cfg.prior_frames * cfg.Tf)} most recent history entries), scaled by "
                     f"{cfg.H}/{heads}",
           "seconds": round(dt, 2),
           "near_ties": dict(ties, note=f"oracle decisions within the {MARGIN:g} margin in the sampled heads, where "
                                        "either choice is accepted")}
    if not variants:
        return out
    var = {"float64_all_cores": {"value": out["value"], "heads": heads, "seconds": round(dt, 2)}}
    h32, dt32, _ = oracle_sample(cfg, seed, "float32", cfg.H, budget_s * 0.6)
    var["float32_all_cores"] = {"value": round(cfg.Nq / (dt32 / h32 * cfg.H), 2), "heads": h32,
                                "seconds": round(dt32, 2)}
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    for fl in ("float64", "float32"):
        try:
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", cfg.name, fl, "1",
                                str(seed)], capture_output=True, text=True, env=env, timeout=300)
            h1, dt1 = json.loads(r.stdout.strip().splitlines()[-1])
            var[f"{fl}_one_thread"] = {"value": round(cfg.Nq / (dt1 / h1 * cfg.H), 2), "heads": h1,
                                       "seconds": round(dt1, 2)}
        except (OSError, subprocess.SubprocessError, ValueError, IndexError) as exc:
            var[f"{fl}_one_thread"] = {"error": f"{type(exc).__name__}"}
    out["variants"] = var
    return out


def time_ann_match(layer, cfg, q_d, k_d, flush, steps, torch, L):
    dev = q_d.device
    cin = layer.caches[layer.cur]
    H, M, B, r, nq = cfg.H, cfg.M, cfg.B, cfg.r, cfg.Nq
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32, device=dev)
    kperm, koff, status = i32(H, M), i32(H, B + 1), i32(1)
    L.fastar_bucket_sort(cin.kb, B, kperm, koff, cin.len, status)     # the incoming cache's bucket order
    ws = torch.zeros(L.workspace_bytes(L.OP_MATCH_ANN, H, nq, M, cfg.d, B, r), dtype=torch.uint8, device=dev)
    t_ann, s_ann = i32(H, nq), torch.zeros((H, nq), dtype=torch.float32, device=dev)
    e_ann = torch.zeros((H, M), dtype=torch.uint8, device=dev)
    t_ex, s_ex = i32(H, nq), torch.zeros((H, nq), dtype=torch.float32, device=dev)
    e_ex = torch.zeros((H, M), dtype=torch.uint8, device=dev)

    def ann():
        L.fastar_tempcache_match_ann(q_d, k_d, r, B, layer.qperm, layer.qoff, cin.k, cin.knorm, cin.len, kperm,
                                     koff, cfg.tau, t_ann, s_ann, e_ann, status, ws)

    def exact():
        L.fastar_tempcache_match(q_d, k_d, cin.k, cin.knorm, cin.len, cfg.tau, t_ex, s_ex, None, e_ex, status,
                                 layer.ws_match)

    def timed(fn):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(steps):
            hold_gpu(torch)
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return sum(ms) / len(ms)

    ann_ms, ex_ms = timed(ann), timed(exact)
    torch.cuda.synchronize()
    agree = float((t_ann == t_ex).float().mean().item())
    return {"ms": round(ann_ms, 4), "exact_ms": round(ex_ms, 4), "speedup_vs_exact": round(ex_ms / ann_ms, 3),
            "top1_agree_with_exact": round(agree, 4),
            "evicted": {"ann": int(e_ann.sum().item()), "exact": int(e_ex.sum().item())},
            "status": int(status.item()),
            "note": "each query compared only with the incoming cache's keys in its own r buckets; "
                    "one call incl. the bucket-order copy and the slot merge, L2 flushed before each"}


ROLLOUT_REPLAYS = 3


def measure_rollout(cfg, seed, flush, torch, dev):
    """The layer stepped through a 200-frame rollout from an empty cache (67 chunks of 3
    frames): per chunk the step's time (its CUDA graph for the cache half it reads, L2
    flushed before), the cache length, evictions and FIFO drops, and the device bytes;
    beside it the dense path from the same build, whose append-only cache grows."""
    import numpy as np
    from kv_cache_tempcache_gb300 import synth
    from kv_cache_tempcache_gb300.layer import FastARLayer, DenseLayer
    chunks = synth.WAN13B_ROLLOUT_CHUNKS
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    gen = synth.DriftingMixture(cfg, seed=seed)
    layer = FastARLayer(H=cfg.H, d=cfg.d, Tf=cfg.Tf, F=cfg.F, M=cfg.M, B=cfg.B, r=cfg.r, P=cfg.P, tau=cfg.tau,
                        tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=tdt, device=dev)
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(tdt).pin_memory()
    layer.set_centroids(up(gen.centroids).to(dev))
    kp, vp = gen.prompt
    layer.set_prompt(up(kp).to(dev), up(vp).to(dev))
    dense = DenseLayer(cfg.H, cfg.d, cfg.Nq, chunks * cfg.Nq, cfg.P, dtype=tdt, device=dev)
    dense.set_prompt(up(kp).to(dev), up(vp).to(dev))
    q_d, k_d, v_d = (torch.zeros((cfg.H, cfg.Nq, cfg.d), dtype=tdt, device=dev) for _ in range(3))
    # one graph per direction of the double-buffered cache, then start from empty
    graphs = [layer.capture(q_d, k_d, v_d)]
    layer.cur = 1
    graphs.append(layer.capture(q_d, k_d, v_d))
    layer.reset()
    torch.cuda.synchronize(dev)
    ms, dense_ms, lens, lens_in, evicted, dropped, dev_bytes, alloc = [], [], [], [], [], [], [], []
    for t in range(chunks):
        k, v, q = gen.next_chunk()
        q_d.copy_(up(q))
        k_d.copy_(up(k))
        v_d.copy_(up(v))
        n_in = int(layer.cache.len.sum().item())
        # the step reads one cache half and writes the other, so replaying its graph before
        # the flip repeats exactly the same work: the chunk's time is the median of three
        reps = []
        for _ in range(ROLLOUT_REPLAYS):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graphs[layer.cur].replay()
            b.record()
            reps.append((a, b))
        layer.cur = 1 - layer.cur
        flush.zero_()
        c, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c.record()
        dense.step(q_d, k_d, v_d)
        e.record()
        torch.cuda.synchronize(dev)
        ms.append(statistics.median(x.elapsed_time(y) for x, y in reps))
        dense_ms.append(c.elapsed_time(e))
        n_out = int(layer.cache.len.sum().item())
        ev = int(layer.evict.sum().item())
        lens_in.append(n_in)
        lens.append(n_out)
        evicted.append(ev)
        dropped.append(n_in - ev + cfg.H * cfg.Nq - n_out)
        dev_bytes.append(layer.device_bytes())
        alloc.append(torch.cuda.memory_allocated(dev))
    assert layer.status() == 0
    # steady state: the chunks whose INCOMING cache is full (the step's shape no longer changes)
    full = [i for i in range(chunks) if lens_in[i] == cfg.H * cfg.M]
    first = full[0] if full else chunks
    steady = ms[first:] if full else ms
    med = statistics.median(steady)
    dense_kv = 2 * dense.n * cfg.H * cfg.d * (2 if cfg.dtype == "bf16" else 4)
    out = {"chunks": chunks, "frames": chunks * cfg.F, "first_full_chunk": first,
           "ms_median_full": round(med, 4), "ms_max_dev_frac_full": round(max(abs(x - med) / med for x in steady), 4),
           "ms_per_chunk": [round(x, 4) for x in ms],
           "cache_entries_per_chunk": lens, "evicted_per_chunk": evicted, "fifo_dropped_per_chunk": dropped,
           "device_bytes": sorted(set(dev_bytes)), "memory_allocated": [min(alloc), max(alloc)],
           "dense_ms_per_chunk": [round(x, 3) for x in dense_ms], "dense_keys_last": int(dense.n),
           "dense_kv_bytes_last": dense_kv,
           "note": f"per chunk: the median of {ROLLOUT_REPLAYS} replays of the step's graph on the same incoming "
                   "cache (after the chunk's upload and a synchronize), the L2 flushed before each; the dense path "
                   "appends, so it is timed once per chunk; flat = max deviation from the median over the chunks "
                   "that start from a full cache"}
    del layer, dense, graphs
    torch.cuda.empty_cache()
    return out


def time_pq_match(layer, cfg, q_d, k_d, flush, steps, torch, L, first_chunk_keys, seed, m=32, Kc=16):
    from kv_cache_tempcache_gb300 import synth
    dev = q_d.device
    tdt = q_d.dtype
    cin = layer.caches[layer.cur]
    H, M, nq = cfg.H, cfg.M, cfg.Nq
    cb = torch.from_numpy(synth.pq_codebooks(first_chunk_keys[:, :cfg.Tf], m, Kc, seed=seed)).to(dev).to(tdt)
    codes = torch.zeros((H, M, m), dtype=torch.uint8, device=dev)
    codes_cur = torch.zeros((H, nq, m), dtype=torch.uint8, device=dev)
    L.fastar_pq_encode(cin.k, cb, codes)                    # the incoming (full) cache, once
    ws = torch.zeros(L.workspace_bytes(L.OP_MATCH_PQ, H, nq, M, cfg.d), dtype=torch.uint8, device=dev)
    i32 = lambda *s_: torch.zeros(s_, dtype=torch.int32, device=dev)
    status = i32(1)
    t_pq, s_pq = i32(H, nq), torch.zeros((H, nq), dtype=torch.float32, device=dev)
    e_pq = torch.zeros((H, M), dtype=torch.uint8, device=dev)
    t_ex, s_ex = i32(H, nq), torch.zeros((H, nq), dtype=torch.float32, device=dev)
    e_ex = torch.zeros((H, M), dtype=torch.uint8, device=dev)

    def pq():
        L.fastar_tempcache_match_pq(q_d, k_d, cin.k, cin.knorm, codes, cin.len, cb, cfg.tau, t_pq, s_pq, e_pq, status,
                                    ws)

    def encode():
        L.fastar_pq_encode(k_d, cb, codes_cur)

    def exact():
        L.fastar_tempcache_match(q_d, k_d, cin.k, cin.knorm, cin.len, cfg.tau, t_ex, s_ex, None, e_ex, status,
                                 layer.ws_match)

    def timed(fn):
        for _ in range(3):
            fn()
        res = []
        for _ in range(steps):
            hold_gpu(torch)
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            res.append(a.elapsed_time(b))
        return sum(res) / len(res)

    pq_ms, enc_ms, ex_ms = timed(pq), timed(encode), timed(exact)
    torch.cuda.synchronize()
    agree = float((t_pq == t_ex).float().mean().item())
    return {"ms": round(pq_ms, 4), "encode_chunk_ms": round(enc_ms, 4), "exact_ms": round(ex_ms, 4),
            "m": m, "Kc": Kc, "code_bytes_per_key": m, "top1_agree_with_exact": round(agree, 4),
            "evicted": {"pq": int(e_pq.sum().item()), "exact": int(e_ex.sum().item())},
            "status": int(status.item()),
            "note": "cached keys product-quantized (m sub-spaces of d/m dims, Kc codewords drawn from the first "
                    "frame's keys); the match ranks the decoded keys on the tensor cores (decode + match + "
                    "finaliser, eviction on the true keys); encode = the chunk's current keys"}


def measure_dit(chunks, seed, torch, dev):
    """The Wan-1.3B-shaped DiT (random weights) denoising a rollout of `chunks` chunks of 3
    latent frames (4 Euler steps each, every block's attention FAST-AR or dense), timed
    per chunk over the replayed step graphs; plus the tensor-core GEMM alone at the
    feed-forward shape."""
    from kv_cache_tempcache_gb300 import _lib as L
    from kv_cache_tempcache_gb300.dit import WAN13B_DIT, DiT
    cfg = WAN13B_DIT
    N = cfg.tokens
    g = torch.Generator(device=dev).manual_seed(seed)
    text = torch.randn(cfg.text_len, cfg.text_dim, generator=g, device=dev).to(torch.bfloat16)
    noises = [torch.randn(N, cfg.patch_ch, generator=g, device=dev).to(torch.bfloat16) for _ in range(chunks)]
    res = {"config": f"{cfg.name}: {cfg.layers} blocks, dim {cfg.dim}, {cfg.heads} heads, FFN {cfg.ffn}, "
                     f"chunk {cfg.frames}x{cfg.grid_h}x{cfg.grid_w} = {N} tokens, {cfg.steps} steps, text "
                     f"{cfg.text_len}x{cfg.text_dim}, random weights",
           "chunks": chunks, "frames": chunks * cfg.frames}
    # the GEMM alone: the feed-forward up-projection, L2 flushed before each
    A = torch.randn(N, cfg.dim, generator=g, device=dev).to(torch.bfloat16)
    W = (torch.randn(cfg.ffn, cfg.dim, generator=g, device=dev) / cfg.dim ** 0.5).to(torch.bfloat16)
    C = torch.empty(N, cfg.ffn, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        L.fastar_gemm(A, W, C, act=L.ACT_GELU_TANH)
    ms = []
    for _ in range(10):
        hold_gpu(torch)
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        L.fastar_gemm(A, W, C, act=L.ACT_GELU_TANH)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    gms = statistics.median(ms)
    peaks = load_peaks()
    tf = 2.0 * N * cfg.ffn * cfg.dim / (gms * 1e-3) / 1e12
    res["gemm_ffn_up"] = {"shape": [N, cfg.ffn, cfg.dim], "ms": round(gms, 4), "tflops": round(tf, 1),
                          "frac_of_bf16_burst": round(tf / peaks["bf16_tflops"], 3) if peaks.get("bf16_tflops") else None}
    del A, W, C
    for attention in ("fastar", "dense"):
        model = DiT(cfg, attention, seed=seed, device=dev, dense_capacity=chunks * N)
        model.set_text(text)
        per_chunk = []
        for c in range(chunks):
            ev = []
            model.denoise_chunk(noises[c], use_graph=True,
                                timer=lambda ph: ev.append(torch.cuda.Event(enable_timing=True)) or ev[-1].record())
            torch.cuda.synchronize(dev)
            per_chunk.append(sum(ev[i].elapsed_time(ev[i + 1]) for i in range(0, len(ev), 2)))
        assert model.status_word() == 0
        total = sum(per_chunk)
        res[attention] = {"ms_per_chunk": [round(x, 2) for x in per_chunk], "total_ms": round(total, 1),
                          "latent_frames_per_s": round(chunks * cfg.frames / (total * 1e-3), 2),
                          "peak_bytes": int(torch.cuda.max_memory_allocated(dev))}
        del model
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
    res["speedup_fastar_vs_dense"] = round(res["dense"]["total_ms"] / res["fastar"]["total_ms"], 3)
    res["note"] = ("per chunk: the 4 replayed denoising-step graphs (graph capture excluded); FAST-AR caches "
                   "capped at M per block, the dense caches append every chunk")
    return res


def time_merge_variant(cfg, seed, up, flush, steps, replace_ms, torch, dev):
    from kv_cache_tempcache_gb300 import synth
    from kv_cache_tempcache_gb300.layer import FastARLayer
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    gen = synth.DriftingMixture(cfg, seed=seed)
    layer = FastARLayer(H=cfg.H, d=cfg.d, Tf=cfg.Tf, F=cfg.F, M=cfg.M, B=cfg.B, r=cfg.r, P=cfg.P, tau=cfg.tau,
                        tau_ca=cfg.tau_ca, topk=cfg.topk, dtype=tdt, device=dev, merge=True)
    layer.set_centroids(up(gen.centroids))
    kp, vp = gen.prompt
    layer.set_prompt(up(kp), up(vp))
    for _ in range(cfg.prior_frames // cfg.F):
        k, v, q = gen.next_chunk()
        layer.step(up(q), up(k), up(v))
    k, v, q = gen.next_chunk()
    q_d, k_d, v_d = up(q), up(k), up(v)
    graph = layer.capture(q_d, k_d, v_d)
    for _ in range(3):
        flush.zero_()
        graph.replay()
    ev = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    stage_ev = {}

    def timer(name, stream, phase):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        stage_ev.setdefault(name, []).append(e)

    for _ in range(steps):
        hold_gpu(torch)
        flush.zero_()
        layer.step(q_d, k_d, v_d, advance=False, timer=timer, serial=True)
    torch.cuda.synchronize(dev)
    stages = {}
    for name in ("cache_compact", "sparse_attn"):
        es = stage_ev[name]
        stages[name] = round(sum(es[i].elapsed_time(es[i + 1]) for i in range(0, len(es), 2)) / (len(es) // 2), 4)
    cin, cout = layer.caches[layer.cur], layer.caches[1 - layer.cur]
    n_in = cin.len.long()
    g_in = sum(int(cin.g[h, :int(n_in[h])].sum().item()) for h in range(cfg.H))
    out = {"ms_per_step": round(ms, 4), "replace_ms_per_step": round(replace_ms, 4),
           "ratio_to_replace": round(ms / replace_ms, 3), "stages_ms": stages,
           "entries_in": int(n_in.sum().item()), "keys_represented_in": g_in,
           "merged_this_step": int((layer.owner >= 0).sum().item()), "status": layer.status(),
           "note": "Lemma 5.1 merge variant: evicted entries fold into their owner (mean value, summed count), "
                   "AnnSA with a ln g logit shift; same chunks and graph protocol as the main step"}
    del layer, graph
    return out


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is one head of the layer step (a
    bounded sample); value counts the layer's query tokens that step covers (Nq / H)
    over its measured time, and ms_per_step is that measured time."""
    if rank != 0:
        return None
    from kv_cache_tempcache_gb300 import synth
    cfg = synth.CONFIGS[args.config]
    inp, ck, cv = _oracle_case(cfg, args.seed)
    W = max(args.warmup, 3)
    # warm-up steps are capped at one so that the run stays within minutes
    for i in range(min(W, 1)):
        _oracle_head(cfg, inp, ck, cv, 0)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        _oracle_head(cfg, inp, ck, cv, i % cfg.H)
        times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    value = (cfg.Nq / cfg.H) / per_step
    sample = (f"each step: one of the {cfg.H} heads of one {cfg.name} step (Nq/H = {cfg.Nq / cfg.H:g} layer query "
              f"tokens), float64 NumPy, all cores")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": W, "ms_per_step": round(per_step * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(cfg, world),
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.cpu_sample:
        from kv_cache_tempcache_gb300 import synth
        name, fl, heads, seed = args.cpu_sample
        h, dt, _ = oracle_sample(synth.CONFIGS[name], int(seed), fl, int(heads), 0.0)
        print(json.dumps([h, dt]))
        return
    rank, world, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_fastar(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
