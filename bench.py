#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify step on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
tree visibility (spec_tree_prepare), split-K verify attention (partials +
log-sum-exp combine) and the acceptance sampler.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

Timing: inputs resident in HBM; the step is captured once in a CUDA graph
(attention on the launching stream, the sampler on a second stream forked and
joined inside the graph: the two share no inputs) and replayed; L2 is flushed
before every timed step, outside the timed events: a 2 x L2-size write, then a
2 x L2-size read of another buffer so that the flush leaves no dirty lines whose
write-back would land inside the step; each step is timed with CUDA events on
its stream; K steps are bracketed by a barrier + synchronize; the max over ranks
is reported.  The partial pass and the sampler are timed with their own events
inside the captured step.  The other configurations are timed the same way and
reported under "per_workload".
"""
import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")   # the oracle legs: one core per thread
os.environ.setdefault("OMP_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_verification_76_gb300 import workloads as wl  # noqa: E402

METRIC = "verified positions/sec and achieved HBM GB/s (fraction of roofline), 1×GB300"
UNIT = "positions/s"
DEFAULT_WORKLOAD = "batched_serving_a75"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 2 * 129 * 1024 * 1024


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device="cpu") -> float:
    """Largest value of x over all ranks (x itself when running alone)."""
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int, device="cpu") -> float:
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm"):
            if k in d and isinstance(d[k], (int, float)):
                return float(d[k]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (MEASURED_PEAKS.json absent)"


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured burst (MEASURED_PEAKS.json bf16_tflops)"
    except (OSError, ValueError, KeyError):
        return 1900.0, "fallback 1.9 PFLOP/s"


def source_hash(files) -> str:
    """Hash of the named kernel sources (a traffic record holds for them only)."""
    h = hashlib.sha256()
    for f in files:
        p = os.path.join(ROOT, "speculative_decoding_verification_76_gb300", "csrc", f)
        if os.path.exists(p):
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the partial kernel from an ncu capture, if the
    capture was taken on the current source of the kernel it names."""
    path = os.path.join(ROOT, "profiles", "attn_partial_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == source_hash(e.get("sources", [])):
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def pct(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.idx)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ the step on the GPU
def step_splits(spec: wl.Spec, device, overlap: bool, max_pages: int) -> int:
    """The attention's split count in the step.  The library's own plan fills
    one wave of SMs; when the sampler runs beside it as a few clusters (few
    rows: one cluster of min(8, ceil(V / 16384)) CTAs per row) the attention
    of a short block (at most 64 query rows per KV head: one row tile) is cut
    into fewer splits, so that both fit on the SMs at once (the library rounds
    an explicit count to its chunk granularity: the largest request whose
    plan fits is taken)."""
    if spec.num_splits or not overlap:
        return spec.num_splits
    import speculative_decoding_verification_76_gb300 as sv
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    samp_ctas = spec.B * spec.R * min(8, -(-spec.V // 16384))
    units = spec.B * spec.Hkv
    if samp_ctas > 2 * sms or spec.R * spec.Hq // spec.Hkv > 64 or units >= sms - samp_ctas:
        return 0
    for req in range((sms - samp_ctas) // units, 0, -1):
        got = sv.attn_num_splits(spec.B, spec.R, spec.Hq, spec.Hkv, spec.D, spec.page_size,
                                 max_pages, req)
        if 0 < got * units <= sms - samp_ctas:
            return req
    return 0


class GpuStep:
    """All buffers of one verify step, resident on the device."""

    def __init__(self, spec: wl.Spec, device, seed=None, overlap=True):
        import speculative_decoding_verification_76_gb300 as sv
        self.sv = sv
        self.spec = spec
        self.dev = device
        w = wl.make_workload(spec, seed=seed, device=device)
        self.w = w
        B, R = spec.B, spec.R
        # a chain needs no ancestor masks: the attention takes none (row i sees
        # block rows 0 .. i) and no tree_prepare launch is made
        self.anc = torch.empty((B, R), dtype=torch.int64, device=device) if spec.is_tree \
            else None
        self.pos = torch.empty((B, R), dtype=torch.int32, device=device)
        self.tst = torch.empty((B,), dtype=torch.int32, device=device)
        self.splits = step_splits(spec, device, overlap, w.block_table.shape[1])
        self.attn = sv.AttnCall(w.q, w.k_cache, w.v_cache, w.block_table, w.ctx_len, self.anc,
                                num_splits=self.splits)
        self.cfg = sv.SamplerConfig(temperature=spec.temperature, top_k=spec.top_k,
                                    top_p=spec.top_p, greedy=spec.greedy)
        self.sws = sv.new_workspace(sv.sample_workspace_size(B, R, spec.V), device)
        self.sout = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=device),
                         emitted=torch.empty((B, R), dtype=torch.int32, device=device),
                         status=torch.empty(B, dtype=torch.int32, device=device))
        if spec.is_tree:
            self.sout["path"] = torch.empty((B, R), dtype=torch.int32, device=device)
        self.overlap = overlap
        self.side = torch.cuda.Stream(device=device)
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()
        self.launches_per_step = 4 if spec.is_tree else 3

    def sample(self):
        sv, w = self.sv, self.w
        if self.spec.is_tree:
            sv.accept_sample_tree(w.logits, w.draft_probs, w.draft_tokens, w.parent, w.uniforms,
                                  self.cfg, workspace=self.sws, out=self.sout)
        else:
            sv.accept_sample(w.logits, None if self.spec.greedy else w.draft_probs,
                             w.draft_tokens, w.uniforms, self.cfg, workspace=self.sws,
                             out=self.sout)

    def run(self, ev=None):
        """One step.  ev: 4 events (partial start/end, sampler start/end) or None."""
        sv, w = self.sv, self.w
        main = torch.cuda.current_stream()
        if self.overlap:            # the sampler on a second stream, joined below
            self.fork.record(main)
            self.side.wait_event(self.fork)
            with torch.cuda.stream(self.side):
                if ev is not None:
                    ev[2].record(self.side)
                self.sample()
                if ev is not None:
                    ev[3].record(self.side)
            self.join.record(self.side)
        if self.spec.is_tree:
            sv.tree_prepare(w.parent, w.ctx_len, anc_mask=self.anc, pos_ids=self.pos,
                            status=self.tst)
        if ev is not None:
            ev[0].record(main)
        self.attn.partials()
        if ev is not None:
            ev[1].record(main)
        self.attn.combine()
        if self.overlap:
            main.wait_event(self.join)
        else:
            if ev is not None:
                ev[2].record(main)
            self.sample()
            if ev is not None:
                ev[3].record(main)


def make_flusher(dev):
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def flush_l2():
        flush.zero_()           # evict the inputs: write more than L2 holds
        clean.sum()             # then read more than L2 holds: write-backs finish here
    return flush_l2


def time_step(step: GpuStep, steps: int, warmup: int, flush_l2, ws: int, gpu_index=None):
    """Capture the step in a graph and time `steps` replays (L2 flushed before each)."""
    stream = torch.cuda.current_stream()
    for _ in range(3):                     # eager warm-up: attributes, descriptors
        step.run()
    torch.cuda.synchronize()
    # the timed graph holds the step's kernels only; a second graph of the same
    # step with event-record nodes (which lengthen a replay by ~10 us) gives the
    # partial pass's and the sampler's spans inside the step, after the timed region
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    try:
        ev_in = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    except TypeError:
        ev_in = None
    graph_ev = None
    if ev_in is not None:
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev):
            step.run(ev_in)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms, part_ms, samp_ms = [], [], []
    clk = ClockSampler(gpu_index) if gpu_index is not None else None
    if clk:
        clk.__enter__()
    try:
        for _ in range(warmup):
            flush_l2()
            graph.replay()
        barrier(ws)
        torch.cuda.synchronize()
        for _ in range(steps):
            flush_l2()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
        torch.cuda.synchronize()
        barrier(ws)
    finally:
        if clk:
            clk.__exit__()
    if graph_ev is not None:
        for i in range(min(steps, 200) + 3):
            flush_l2()
            graph_ev.replay()
            ev_in[3].synchronize()
            torch.cuda.synchronize()
            if i >= 3:
                part_ms.append(ev_in[0].elapsed_time(ev_in[1]))
                samp_ms.append(ev_in[2].elapsed_time(ev_in[3]))
    else:   # no graph event nodes: time the partial pass eagerly
        for _ in range(min(steps, 200)):
            flush_l2()
            e0.record(stream)
            step.attn.partials()
            e1.record(stream)
            e1.synchronize()
            part_ms.append(e0.elapsed_time(e1))
    # the partial pass alone (nothing running beside it), right after the timed
    # region: inside the step the sampler's CTAs share its SMs and stretch it
    iso_ms = []
    for _ in range(min(steps, 50)):
        flush_l2()
        e0.record(stream)
        step.attn.partials()
        e1.record(stream)
        e1.synchronize()
        iso_ms.append(e0.elapsed_time(e1))
    err = step.sv.workspace_error(step.attn.workspace) | step.sv.workspace_error(step.sws)
    if err:
        raise RuntimeError(f"device wait timed out (error word {err:#x})")
    return {"step_ms": step_ms, "part_ms": part_ms, "samp_ms": samp_ms, "iso_part_ms": iso_ms,
            "clocks": clk.summary() if clk else None}


def acceptance_stats(spec, acc: np.ndarray):
    """Accepted-length histogram over all sequences and the empirical acceptance
    rate of each draft position (accepted / reached)."""
    acc = np.asarray(acc)
    hist = np.bincount(np.clip(acc, 0, None), minlength=spec.R).tolist()
    out = {"accepted_len_hist": hist, "mean_accepted": float(acc.mean()),
           "mean_emitted": float(acc.mean() + 1)}
    if not spec.is_tree:
        alpha = []
        for i in range(1, spec.R):
            reached = int((acc >= i - 1).sum())
            alpha.append(float((acc >= i).sum()) / reached if reached else None)
        out["alpha_per_position"] = alpha
    return out


def step_record(spec, step, t, nbytes, peak, ws, dev):
    """Throughput, fractions and timing statistics of one timed workload."""
    ms = t["step_ms"]
    mean_ms = statistics.fmean(ms)
    mean_all = max_over_ranks(mean_ms, ws, device=dev)
    med = statistics.median(ms)
    part = statistics.fmean(t["part_ms"])
    rec = {
        "ms_mean": mean_all, "ms_median": med, "ms_p10": pct(ms, 10), "ms_p90": pct(ms, 90),
        "positions_per_s": sum_over_ranks(spec.B * spec.R, ws, device=dev) / (mean_all * 1e-3),
        "sequences_per_s": sum_over_ranks(spec.B, ws, device=dev) / (mean_all * 1e-3),
        "step_bytes": nbytes["step"], "step_bytes_all_q_rows": nbytes["step_all_q"],
        "step_hbm_frac": nbytes["step"] / (med * 1e-3) / 1e9 / peak,
        "step_hbm_frac_all_q_rows": nbytes["step_all_q"] / (med * 1e-3) / 1e9 / peak,
        "attn_partial_us": part * 1e3,
        "attn_partial_frac": nbytes["attn"] / (part * 1e-3) / 1e9 / peak,
        "attn_partial_alone_us": (statistics.median(t["iso_part_ms"]) * 1e3
                                  if t.get("iso_part_ms") else None),
        "sampler_us": statistics.fmean(t["samp_ms"]) * 1e3 if t["samp_ms"] else None,
        "attn_num_splits": step.sv.attn_num_splits(
            spec.B, spec.R, spec.Hq, spec.Hkv, spec.D, spec.page_size,
            step.w.block_table.shape[1], step.splits),
    }
    if spec.is_tree or spec.R * spec.Hq // spec.Hkv >= 128:
        # a contraction-heavy shape: also against the bf16 tensor peak
        ctx = step.w.ctx_len.cpu().numpy().astype(np.float64)
        flop = 4.0 * spec.D * spec.Hq * spec.R * float(np.sum(ctx + spec.R))
        tpk, _ = bf16_peak()
        rec["attn_partial_tflops"] = flop / (part * 1e-3) / 1e12
        rec["attn_partial_tensor_frac"] = rec["attn_partial_tflops"] / tpk
        if rec["attn_partial_alone_us"]:
            rec["attn_partial_alone_tflops"] = flop / (rec["attn_partial_alone_us"] * 1e-6) / 1e12
            rec["attn_partial_alone_tensor_frac"] = rec["attn_partial_alone_tflops"] / tpk
    return rec


def bench_gpu(args, spec, ws, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import speculative_decoding_verification_76_gb300 as sv
    sv.load()
    flush_l2 = make_flusher(dev)
    step = GpuStep(spec, dev, overlap=not args.serial)
    ctx = step.w.ctx_len.cpu().numpy()
    nbytes = wl.algorithmic_bytes(spec, ctx)
    peak, peak_src = hbm_peak()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    t = time_step(step, args.steps, args.warmup, flush_l2, ws, gpu_index)
    rec = step_record(spec, step, t, nbytes, peak, ws, dev)
    part_mean = rec["attn_partial_us"] * 1e-6
    attn_gbs = nbytes["attn"] / part_mean / 1e9
    traffic = recorded_traffic(spec.name)
    acc = step.sout["accepted_len"].cpu().numpy()
    e2e = bench_e2e(step, spec, max(3, min(args.steps, 50)), ws, dev)
    out = {
        "metric": METRIC, "value": rec["positions_per_s"], "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_mean"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": arm_config(spec, int(ctx.max()), ws),
        "ms_median": rec["ms_median"], "ms_p10": rec["ms_p10"], "ms_p90": rec["ms_p90"],
        "sequences_per_s": rec["sequences_per_s"],
        "step_hbm_gbs": nbytes["step"] / (rec["ms_median"] * 1e-3) / 1e9,
        "step_hbm_frac": rec["step_hbm_frac"], "step_algorithmic_bytes": nbytes["step"],
        "step_hbm_frac_all_q_rows": rec["step_hbm_frac_all_q_rows"],
        "step_algorithmic_bytes_all_q_rows": nbytes["step_all_q"],
        "attn_num_splits": rec["attn_num_splits"], "sampler_us": rec["sampler_us"],
        "roofline": {"bound": "hbm", "kernel": partial_kernel_name(spec),
                     "achieved": attn_gbs, "peak": peak, "unit": "GB/s",
                     "frac": attn_gbs / peak, "traffic": traffic,
                     "algorithmic_bytes": nbytes["attn"], "mean_launch_us": part_mean * 1e6,
                     "peak_source": peak_src,
                     "alone": alone_roofline(t["iso_part_ms"], nbytes["attn"], peak)},
        **acceptance_stats(spec, acc),
        "e2e": e2e,
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": t["clocks"],
    }
    if not args.no_per_workload:
        del step
        torch.cuda.empty_cache()
        out["per_workload"] = per_workload(args, spec, ws, dev, flush_l2, peak)
    return out


def alone_roofline(iso_ms, nbytes, peak):
    """The partial pass timed alone (L2 flushed, CUDA events), after the timed
    region: its rate without the sampler's CTAs on the same SMs."""
    if not iso_ms:
        return None
    us = statistics.median(iso_ms) * 1e3
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"median_launch_us": us, "achieved": gbs, "frac": gbs / peak,
            "launches": len(iso_ms)}


def partial_kernel_name(spec) -> str:
    """The partial-pass kernel the library's plan runs for this shape."""
    rows = spec.R * spec.Hq // spec.Hkv
    if spec.kv_dtype == "f32":
        return "attn_partial_f32 (CUDA cores)"
    if rows > 128:
        return "attn_partial_tc2 (tcgen05, two 128-row tiles per CTA)"
    if rows > 64:
        return "attn_partial_tc1 (tcgen05, one 128-row tile per CTA)"
    return "attn_partial_bf16 (warp-level mma.sync)"


def per_workload(args, headline, ws, dev, flush_l2, peak):
    """The other configurations (the tiny one is a parity case only), each in its
    own graph, timed like the headline."""
    res = {}
    for name, spec in wl.SPECS.items():
        if name in (headline.name, "tiny_chain"):
            continue
        step = GpuStep(spec, dev, overlap=not args.serial)
        ctx = step.w.ctx_len.cpu().numpy()
        nbytes = wl.algorithmic_bytes(spec, ctx)
        t = time_step(step, args.per_workload_steps, args.warmup, flush_l2, ws)
        rec = step_record(spec, step, t, nbytes, peak, ws, dev)
        rec["attn_partial_kernel"] = partial_kernel_name(spec)
        rec.update(acceptance_stats(spec, step.sout["accepted_len"].cpu().numpy()))
        res[name] = rec
        del step
        torch.cuda.empty_cache()
    return res


def arm_config(spec, seq_len, ws):
    """The workload description both arms print (identical keys and values)."""
    return {
        "workload": spec.name, "global_batch": spec.B * ws, "seq_len": seq_len,
        "rows_per_seq": spec.R, "tree": spec.is_tree, "q_heads": spec.Hq,
        "kv_heads": spec.Hkv, "head_dim": spec.D, "vocab": spec.V, "page_size": spec.page_size,
        "temperature": spec.temperature, "top_k": spec.top_k, "top_p": spec.top_p,
        "greedy": spec.greedy, "draft_noise": spec.draft_noise, "parallelism": f"replicas{ws}",
        "l2": "flushed before every timed step (2 x L2 write, then 2 x L2 read of a second "
              "buffer; outside the timed events)",
        "timing": ("CUDA-graph replay of the step's kernels, CUDA events per step; the phase "
                   "spans from a second graph with event-record nodes")}


def bench_e2e(step: GpuStep, spec, n, ws, dev):
    """Same metric through the public API with host buffers: every step
    copies its inputs from pinned host memory, runs the calls and reads the
    accepted lengths and emitted tokens back.  The attention's inputs (a few
    MB) go first on the launching stream and its call runs under the sampler's
    copies (the target and draft rows: hundreds of MB), which a copy stream
    makes in four batch slices; a third stream samples each slice as soon as
    it has landed, while the next one is copied.  Steps with less than 64 MB
    of inputs (where the extra streams' launch latency outweighs the copies)
    run everything in order on one stream."""
    sv, w = step.sv, step.w
    small = ["q", "block_table", "ctx_len", "parent"]
    big = ["logits", "draft_probs", "draft_tokens", "uniforms"]
    host = {k: getattr(w, k).cpu().pin_memory() for k in small + big}
    dst = {k: torch.empty_like(getattr(w, k)) for k in small + big}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    out = {k: torch.empty_like(v) for k, v in step.sout.items()}
    res_host = {k: torch.empty_like(v, device="cpu").pin_memory()
                for k, v in out.items() if k in ("accepted_len", "emitted")}
    d2h = sum(t.numel() * t.element_size() for t in res_host.values())
    cfg = step.cfg
    overlap = h2d >= (64 << 20) and spec.B % 4 == 0
    nch = 4 if overlap else 1
    cb = spec.B // nch
    cs, ss = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    fork, small_in, join = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    landed = [torch.cuda.Event() for _ in range(nch)]

    def serial():
        for k in small + big:
            dst[k].copy_(host[k], non_blocking=True)
        anc = sv.tree_prepare(dst["parent"], dst["ctx_len"])[0] if spec.is_tree else None
        sv.verify_attn(dst["q"], w.k_cache, w.v_cache, dst["block_table"], dst["ctx_len"], anc,
                       num_splits=step.splits, workspace=step.attn.workspace)
        if spec.is_tree:
            sv.accept_sample_tree(dst["logits"], dst["draft_probs"], dst["draft_tokens"],
                                  dst["parent"], dst["uniforms"], cfg, workspace=step.sws, out=out)
        else:
            sv.accept_sample(dst["logits"], None if spec.greedy else dst["draft_probs"],
                             dst["draft_tokens"], dst["uniforms"], cfg, workspace=step.sws,
                             out=out)
        for k in res_host:
            res_host[k].copy_(out[k], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def one():
        if not overlap:
            serial()
            return
        main = torch.cuda.current_stream()
        fork.record(main)
        cs.wait_event(fork)
        for k in small:
            dst[k].copy_(host[k], non_blocking=True)
        small_in.record(main)
        ss.wait_event(small_in)   # a tree's sampling reads the parent array
        with torch.cuda.stream(cs):
            for c in range(nch):
                sl = slice(c * cb, (c + 1) * cb)
                for k in big:
                    dst[k][sl].copy_(host[k][sl], non_blocking=True)
                landed[c].record(cs)
        with torch.cuda.stream(ss):
            for c in range(nch):
                sl = slice(c * cb, (c + 1) * cb)
                ss.wait_event(landed[c])
                o = {k: v[sl] for k, v in out.items()}
                if spec.is_tree:
                    sv.accept_sample_tree(dst["logits"][sl], dst["draft_probs"][sl],
                                          dst["draft_tokens"][sl], dst["parent"][sl],
                                          dst["uniforms"][sl], cfg, workspace=step.sws, out=o)
                else:
                    sv.accept_sample(dst["logits"][sl],
                                     None if spec.greedy else dst["draft_probs"][sl],
                                     dst["draft_tokens"][sl], dst["uniforms"][sl], cfg,
                                     workspace=step.sws, out=o)
            join.record(ss)
        anc = sv.tree_prepare(dst["parent"], dst["ctx_len"])[0] if spec.is_tree else None
        sv.verify_attn(dst["q"], w.k_cache, w.v_cache, dst["block_table"], dst["ctx_len"], anc,
                       num_splits=step.splits, workspace=step.attn.workspace)
        main.wait_event(join)
        for k in res_host:
            res_host[k].copy_(out[k], non_blocking=True)
        main.synchronize()

    for _ in range(3):
        one()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(n):
        one()
    dt = (time.perf_counter() - t0) / n
    dt = max_over_ranks(dt, ws, device=dev)
    # the same inputs and uniforms: the host copies of the results equal the
    # device-resident step's (the graph replays above left them in step.sout)
    same = all(torch.equal(res_host[k], step.sout[k].cpu()) for k in res_host)
    return {"value": sum_over_ranks(spec.B * spec.R, ws, device=dev) / dt, "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": dt * 1e3, "steps": n, "results_match_step": bool(same),
            "note": ("KV cache resident in HBM; per-step inputs copied from pinned host "
                     + ("memory (the sampler's in 4 batch slices on a copy stream, each "
                        "sampled on a third stream once it has landed; the attention under "
                        "the copies)" if overlap else "memory, in order on one stream"))}


# ------------------------------------------------------------------ the oracle on the host
def cpu_inputs(spec, device=None):
    """The workload's inputs on the host (generated where the GPU run makes them)."""
    dev = device if device is not None else ("cuda" if torch.cuda.is_available() else "cpu")
    w = wl.make_workload(spec, device=dev)
    return w.to("cpu")


def oracle_sample_plan(spec):
    """A bounded sample of one step: every sampler row, and attention for a
    subset of query heads (the step time is scaled up by Hq / heads)."""
    heads = max(1, min(spec.Hq, 4 if spec.Hq >= 4 else spec.Hq))
    batches = list(range(min(spec.B, 2)))
    return heads, batches


def oracle_step(spec, w, heads, batches):
    """Time one bounded oracle step; returns estimated full-step seconds."""
    import oracle
    from oracle.sampler import SamplerCfg
    from tests.util import oracle_attention   # plumbing: one sequence at a time
    t0 = time.perf_counter()
    anc, _, _ = oracle.tree.tree_prepare(w.parent.numpy(), w.ctx_len.numpy())
    oracle_attention(w, anc, batches=batches, heads=list(range(heads)))
    t_attn = time.perf_counter() - t0
    cfg = SamplerCfg(temperature=spec.temperature, top_k=spec.top_k, top_p=spec.top_p,
                     greedy=spec.greedy)
    t1 = time.perf_counter()
    sl = slice(0, len(batches))
    if spec.is_tree:
        oracle.sampler.accept_tree_batch(w.logits[sl].numpy(), w.draft_probs[sl].numpy(),
                                         w.draft_tokens[sl].numpy(), w.parent[sl].numpy(),
                                         w.uniforms[sl].numpy(), cfg)
    else:
        oracle.sampler.accept_chain_batch(w.logits[sl].numpy(), w.draft_probs[sl].numpy(),
                                          w.draft_tokens[sl].numpy(), w.uniforms[sl].numpy(), cfg)
    t_samp = time.perf_counter() - t1
    scale_b = spec.B / len(batches)
    return (t_attn * spec.Hq / heads + t_samp) * scale_b


def cpu_baseline(spec, w, budget_s=15.0):
    heads, batches = oracle_sample_plan(spec)
    est, n, t0 = [], 0, time.perf_counter()
    while n == 0 or (time.perf_counter() - t0 < budget_s and n < 20):
        est.append(oracle_step(spec, w, heads, batches))
        n += 1
    step_s = statistics.fmean(est)
    return {"value": spec.B * spec.R / step_s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{n} oracle step(s) of {spec.name}: sampler rows of {len(batches)} "
                       f"sequence(s) and attention for {heads} of {spec.Hq} query heads, "
                       f"scaled to the full step (B={spec.B}); numpy float64, one thread")}


def cpu_baseline_all_cores(spec, w):
    """The oracle across every host core: one thread per (sequence, KV head)
    attention task and per sequence's sampler rows, over enough sequences to
    give every core a task; wall time scaled to the full batch."""
    import oracle
    from oracle.sampler import SamplerCfg
    from tests.util import sub_sequence
    n = os.cpu_count() or 1
    G = spec.Hq // spec.Hkv
    seqs = list(range(min(spec.B, max(1, -(-n // spec.Hkv)))))
    anc, _, _ = oracle.tree.tree_prepare(w.parent.numpy(), w.ctx_len.numpy())
    subs = {b: sub_sequence(w, b) for b in seqs}
    cfg = SamplerCfg(temperature=spec.temperature, top_k=spec.top_k, top_p=spec.top_p,
                     greedy=spec.greedy)

    def attn_task(b, kvh):
        q, k, v, table, ctx = subs[b]
        hs = slice(kvh * G, (kvh + 1) * G)
        oracle.attention.verify_attention(q[:, :, hs], k[:, :, kvh:kvh + 1], v[:, :, kvh:kvh + 1],
                                          table, ctx, anc[b:b + 1])

    def samp_task(b):
        sl = slice(b, b + 1)
        if spec.is_tree:
            oracle.sampler.accept_tree_batch(w.logits[sl].numpy(), w.draft_probs[sl].numpy(),
                                             w.draft_tokens[sl].numpy(), w.parent[sl].numpy(),
                                             w.uniforms[sl].numpy(), cfg)
        else:
            oracle.sampler.accept_chain_batch(w.logits[sl].numpy(), w.draft_probs[sl].numpy(),
                                              w.draft_tokens[sl].numpy(),
                                              w.uniforms[sl].numpy(), cfg)

    tasks = [(attn_task, (b, k)) for b in seqs for k in range(spec.Hkv)] + \
        [(samp_task, (b,)) for b in seqs]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(lambda t: t[0](*t[1]), tasks))
    wall = time.perf_counter() - t0
    step_s = wall * spec.B / len(seqs)
    return {"value": spec.B * spec.R / step_s, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": (f"{len(seqs)} of {spec.B} sequences of {spec.name} (every row and head), "
                       f"{len(tasks)} tasks on {n} threads (numpy float64; parts that hold the "
                       f"interpreter lock serialise), wall time scaled to the full batch")}


def parity_sample(spec, step, w, max_seqs=16):
    """The GPU step's outputs against the oracle on the same inputs: sampler
    decisions of up to max_seqs sequences (bit-exact except flagged draws) and
    attention of two sequences (every row, one query head per KV head)."""
    import oracle
    from tests.util import cfg_of, oracle_attention
    B = spec.B
    seqs = list(range(min(B, max_seqs)))
    sl = slice(0, len(seqs))
    cfg = cfg_of(spec)
    if spec.is_tree:
        ref = oracle.sampler.accept_tree_batch(w.logits[sl].numpy(), w.draft_probs[sl].numpy(),
                                               w.draft_tokens[sl].numpy(), w.parent[sl].numpy(),
                                               w.uniforms[sl].numpy(), cfg)
    else:
        ref = oracle.sampler.accept_chain_batch(w.logits[sl].numpy(), w.draft_probs[sl].numpy(),
                                                w.draft_tokens[sl].numpy(),
                                                w.uniforms[sl].numpy(), cfg)
    g_acc = step.sout["accepted_len"].cpu().numpy()[sl]
    g_emit = step.sout["emitted"].cpu().numpy()[sl]
    ok = ~ref["flagged"]
    mism = int(((g_acc != ref["accepted_len"]) | (g_emit != ref["emitted"]).any(1))[ok].sum())
    anc, _, _ = oracle.tree.tree_prepare(w.parent.numpy(), w.ctx_len.numpy())
    G = spec.Hq // spec.Hkv
    heads = [k * G + k % G for k in range(spec.Hkv)]
    bs = list(range(min(B, 2)))
    out, _ = oracle_attention(w, anc, batches=bs, heads=heads)
    g_out = step.attn.out.float().cpu().numpy()
    err = max(float(np.abs(g_out[b][:, heads] - out[b][:, heads]).max()) for b in bs)
    return {"sampler_sequences": len(seqs), "flagged": int(ref["flagged"].sum()),
            "mismatched_unflagged": mism, "attn_sequences": len(bs),
            "attn_max_abs_err": err, "attn_tolerance": 2e-2}


def bench_reference(args, spec):
    w = cpu_inputs(spec)
    heads, batches = oracle_sample_plan(spec)
    for _ in range(args.warmup):
        oracle_step(spec, w, heads, batches)
    est = [oracle_step(spec, w, heads, batches) for _ in range(args.steps)]
    step_s = statistics.fmean(est)
    value = spec.B * spec.R / step_s
    cb = {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
          "sample": (f"each step: sampler rows of {len(batches)} sequence(s) and attention for "
                     f"{heads} of {spec.Hq} query heads of {spec.name}, scaled to the full step")}
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": arm_config(spec, int(np.asarray(w.ctx_len).max()), 1),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.SPECS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--per-workload-steps", type=int, default=200)
    ap.add_argument("--serial", action="store_true",
                    help="run the sampler after the attention on one stream")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    spec = wl.SPECS[args.workload]
    ws, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args, spec)), flush=True)
        return 0

    init_dist(ws, "nccl")
    out = bench_gpu(args, spec, ws, rank, local)
    if rank == 0 and not args.no_cpu_baseline:
        dev = torch.device("cuda", local)
        step = GpuStep(spec, dev, overlap=not args.serial)   # the headline's inputs again
        step.run()
        torch.cuda.synchronize()
        w = step.w.to("cpu")
        out["parity_sample"] = parity_sample(spec, step, w)
        out["cpu_baseline"] = cpu_baseline(spec, w)
        out["cpu_baseline_all_cores"] = cpu_baseline_all_cores(spec, w)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
