#!/usr/bin/env python3
"""Benchmark of the routed-expert FP8 MoE FFN on GB300.

One step = the whole hot path over one batch: 1x128 quant -> permute -> GEMM1
-> SwiGLU+quant -> GEMM2 -> combine (moe_ffn), on the DeepSeek-V3-shaped
EP72-like decode workload: 4 local experts, hidden 7168, intermediate 2048,
masked layout (max_m 1024), routing of 72x256 tokens with top-8 over 288
experts at Zipf(1.1) popularity.  Units: "tokens" are the routed
(token, local expert) rows the rank's FFN processes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c2] [--no-cpu-baseline]

Under torchrun each rank runs an independent replica (the path has no
exchange step on one GPU's experts); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

import synth  # noqa: E402

METRIC = "MoE FFN tokens/s; FP8 TFLOPS & HBM GB/s as % of GB300 roofline (1 GPU)"
UNIT = "tokens/s"
FP8_PER_BF16 = 2.0          # nominal dense FP8 : BF16 tensor rate on GB300 (4.5 : 2.25 PF)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- workload
def build_workload(cfg_name: str, device="cuda", quantise_on_gpu=True):
    """Seeded inputs of one config resident on `device`; expert weights quantised
    to E4M3 128x128 blocks by the library's weight-quant kernel."""
    import torch
    import fp8_grouped_expert_x128_gb300 as moe
    cfg = synth.get_config(cfg_name)
    r = synth.make_routing(cfg)
    T, k = r["T"], r["k"]
    x = synth.make_activations(cfg, T, device=device)
    ids = torch.from_numpy(r["topk_ids"].astype(np.int32)).to(device)
    w = torch.from_numpy(r["topk_w"].astype(np.float32)).to(device)
    E, H, I = cfg.E, cfg.H, cfg.I
    w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
    w13_s = torch.empty((E, 2 * I // 128, H // 128), dtype=torch.float32, device=device)
    w2 = torch.empty((E, H, I), dtype=torch.uint8, device=device)
    w2_s = torch.empty((E, H // 128, I // 128), dtype=torch.float32, device=device)
    for e in range(E):
        b13 = synth.make_expert_weights(cfg, "w13", e, device=device)
        moe.moe_quant_weight_fp8(b13[None], w13[e:e + 1], w13_s[e:e + 1])
        b2 = synth.make_expert_weights(cfg, "w2", e, device=device)
        moe.moe_quant_weight_fp8(b2[None], w2[e:e + 1], w2_s[e:e + 1])
        del b13, b2
    torch.cuda.synchronize()
    layout = moe.MOE_LAYOUT_MASKED if cfg.layout == "masked" else moe.MOE_LAYOUT_CONTIG
    local = (r["topk_ids"] >= r["expert_begin"]) & (r["topk_ids"] < r["expert_begin"] + E)
    rows_raw = int(local.sum())
    counts = np.array([(r["topk_ids"] == r["expert_begin"] + e).sum() for e in range(E)])
    rows = int(np.minimum(counts, cfg.max_m).sum()) if cfg.layout == "masked" else rows_raw
    expected_m = int(math.ceil(rows / max(1, int((counts > 0).sum()))))
    return dict(cfg=cfg, routing=r, T=T, k=k, x=x, topk_ids=ids, topk_w=w, w13=w13, w13_s=w13_s,
                w2=w2, w2_s=w2_s, layout=layout, rows=rows, counts=counts,
                active_experts=int((counts > 0).sum()), expected_m=expected_m)


def make_desc(wl, out, err=None, stage_events=None, x=None, ids=None, w=None):
    import fp8_grouped_expert_x128_gb300 as moe
    cfg = wl["cfg"]
    return moe.make_ffn_desc(x if x is not None else wl["x"], ids if ids is not None else wl["topk_ids"],
                             w if w is not None else wl["topk_w"], wl["w13"], wl["w13_s"], wl["w2"],
                             wl["w2_s"], out, wl["routing"]["expert_begin"], cfg.E, wl["layout"],
                             max_m=cfg.max_m, expected_m=wl["expected_m"],
                             gemm_flags=wl.get("gemm_flags", 0), err=err, stage_events=stage_events)


def gemm1_variant(wl):
    """The GEMM1 kernel moe_ffn runs for this workload."""
    import fp8_grouped_expert_x128_gb300 as moe
    if wl["layout"] == moe.MOE_LAYOUT_MASKED:
        v = moe.moe_gemm_fp8_masked_variant(wl["cfg"].max_m, wl["expected_m"], wl.get("gemm_flags", 0))
        if v != 0:
            return f"gemm_fp8_weights_m_kernel<{v}>"
    if wl.get("gemm_flags", 0) & moe.MOE_FFN_FUSE_SWIGLU:
        return "gemm_fp8_tokens_m_kernel<swiglu>"
    return "gemm_fp8_tokens_m_kernel"


def gemm1_fused(wl):
    return gemm1_variant(wl).endswith("<swiglu>")


def algorithmic_counts(wl):
    """Algorithmic FLOPs and bytes per step and per GEMM1 launch."""
    cfg = wl["cfg"]
    H, I = cfg.H, cfg.I
    rows, act = wl["rows"], wl["active_experts"]
    fused = gemm1_fused(wl)
    flops_g1 = 2.0 * rows * H * 2 * I
    flops_g2 = 2.0 * rows * I * H
    w13_bytes = act * (2 * I * H + 4 * (2 * I // 128) * (H // 128))
    w2_bytes = act * (H * I + 4 * (H // 128) * (I // 128))
    g1_out = rows * (I + 4 * I / 128) if fused else rows * 2 * I * 2   # FP8 h + scales, or bf16 Y1
    g1_bytes = w13_bytes + rows * (H + 4 * H / 128) + g1_out
    return dict(flops=flops_g1 + flops_g2, flops_g1=flops_g1, g1_bytes=g1_bytes,
                weight_bytes=w13_bytes + w2_bytes)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [p.strip() for p in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle leg
def _oracle_token_rows(wl, oracle_w, tokens):
    """The oracle chain restricted to `tokens` (rows are independent): quant,
    each local assignment's GEMM1 -> SwiGLU+quant -> GEMM2, combine.  Returns
    the number of routed rows processed."""
    import oracle
    cfg = wl["cfg"]
    r = wl["routing"]
    x = wl["x_host_bits"][tokens]
    q, s = oracle.quant_1x128(oracle.bf16_decode(x).astype(np.float32))
    n_rows = 0
    for i, t in enumerate(tokens):
        y2_rows, ws = [], []
        for j in range(r["k"]):
            e = int(r["topk_ids"][t, j]) - r["expert_begin"]
            if not 0 <= e < cfg.E:
                continue
            w13q, w13s, w2q, w2s = oracle_w[e]
            y1 = oracle.bf16_encode(oracle.gemm_block_scaled(q[i:i + 1], s[:, i:i + 1], w13q, w13s))
            q2, s2 = oracle.swiglu_quant(y1)
            y2_rows.append(oracle.bf16_encode(oracle.gemm_block_scaled(q2, s2, w2q, w2s))[0])
            ws.append(float(r["topk_w"][t, j]))
            n_rows += 1
        if y2_rows:
            oracle.combine(np.stack(y2_rows), np.arange(len(ws)), np.array([ws], np.float32))
    return n_rows


class OracleWeights:
    """Oracle-quantised expert weights, prepared on demand (set-up, never timed)."""

    def __init__(self, wl, device_for_gen):
        self.wl, self.dev, self.cache = wl, device_for_gen, {}

    def _one(self, e):
        import oracle
        import torch
        cfg = self.wl["cfg"]
        f = lambda t: oracle.bf16_decode(
            t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)).astype(np.float32)
        q13, s13 = oracle.quant_128x128(f(synth.make_expert_weights(cfg, "w13", e, device=self.dev)))
        q2, s2 = oracle.quant_128x128(f(synth.make_expert_weights(cfg, "w2", e, device=self.dev)))
        return q13, s13, q2, s2

    def prepare(self, experts):
        from concurrent.futures import ThreadPoolExecutor
        todo = sorted(set(int(e) for e in experts) - set(self.cache))
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
            for e, w in zip(todo, ex.map(self._one, todo)):
                self.cache[e] = w

    def __getitem__(self, e):
        return self.cache[e]


def _local_experts(wl, tokens):
    r = wl["routing"]
    ids = r["topk_ids"][tokens].reshape(-1) - r["expert_begin"]
    return [int(e) for e in ids if 0 <= e < wl["cfg"].E]


def time_oracle(wl, oracle_w, budget_s=15.0, start=0):
    """Time the oracle on a bounded sample of whole local tokens taken in order
    from `start`: one token first to estimate the cost, then as many as fit in
    about `budget_s`.  Weight preparation happens before each timed region.
    Returns (rows/s, seconds timed, tokens, rows)."""
    T = wl["T"]
    first = [start % T]
    oracle_w.prepare(_local_experts(wl, first))
    t0 = time.perf_counter()
    rows = _oracle_token_rows(wl, oracle_w, first)
    dt = time.perf_counter() - t0
    n_more = int(max(0.0, budget_s - dt) / max(dt, 1e-3))
    more = [(start + 1 + i) % T for i in range(min(n_more, T - 1))]
    if more:
        oracle_w.prepare(_local_experts(wl, more))
        t1 = time.perf_counter()
        rows += _oracle_token_rows(wl, oracle_w, more)
        dt += time.perf_counter() - t1
    return rows / dt, dt, 1 + len(more), rows


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(world, v):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(world, v):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def recorded_traffic(kernel_label: str, workload: str):
    """DRAM bytes (read + write) per launch of this kernel on this workload from
    the ncu capture recorded in profiles/traffic.json, or None when there is no
    capture or gemm.cu has changed since it was taken."""
    import hashlib
    path = os.path.join(HERE, "profiles", "traffic.json")
    src = os.path.join(HERE, "fp8_grouped_expert_x128_gb300", "csrc", "gemm.cu")
    if not os.path.exists(path):
        return None
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    with open(path) as f:
        rec = json.load(f)
    r = rec.get(f"{kernel_label}@{workload}")
    if not r or r.get("gemm_cu_sha256") != sha:
        return None
    return r["dram_read_bytes"] + r["dram_write_bytes"]


def load_peaks():
    p = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample per step."""
    if rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = reference_workload(args.workload, dev)
    oracle_w = OracleWeights(wl, dev)
    per_step = []
    for i in range(args.warmup + args.steps):
        rate, dt, ntok, nrows = time_oracle(wl, oracle_w, budget_s=args.ref_step_s, start=i)
        if i >= args.warmup:
            per_step.append((rate, dt, ntok, nrows))
    rows = sum(p[3] for p in per_step)
    secs = sum(p[1] for p in per_step)
    value = rows / secs
    cfg = wl["cfg"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, len(per_step)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": {"workload": f"{cfg.name}: {cfg.description}", "tokens": "routed (token, local expert) rows",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: whole local tokens in order, ~{args.ref_step_s:.0f}s "
                                   f"of CPU work (~{per_step[0][2]} tokens, {per_step[0][3]} rows); "
                                   "numpy float64, BLAS threads = all affinity cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reference_workload(cfg_name, dev):
    import torch
    cfg = synth.get_config(cfg_name)
    r = synth.make_routing(cfg)
    x = synth.make_activations(cfg, r["T"], device=dev)
    counts = np.array([(r["topk_ids"] == r["expert_begin"] + e).sum() for e in range(cfg.E)])
    return dict(cfg=cfg, routing=r, T=r["T"], counts=counts,
                x_host_bits=x.cpu().view(torch.int16).numpy().view(np.uint16))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager moe_ffn calls instead of a CUDA graph")
    ap.add_argument("--expected-m", type=int, default=None,
                    help="override the per-expert count hint given to the masked GEMMs (tuning)")
    ap.add_argument("--gemm-flags", type=int, default=0, help="MOE_GEMM_* flags for both GEMMs (tuning)")
    args = ap.parse_args()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import fp8_grouped_expert_x128_gb300 as moe

    dev = torch.device("cuda", local if world > 1 else 0)
    wl = build_workload(args.workload, dev)
    if args.expected_m is not None:
        wl["expected_m"] = args.expected_m
    wl["gemm_flags"] = args.gemm_flags
    cfg = wl["cfg"]
    T, H = wl["T"], cfg.H
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    err = moe.new_error_word(dev)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    desc = make_desc(wl, out, err=err)                           # the timed step
    desc_ev = make_desc(wl, out, err=err, stage_events=events)   # the per-stage split
    ws = moe.alloc_workspace(desc, dev)
    l2_flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        moe.moe_ffn(desc, ws)
    torch.cuda.synchronize(dev)
    status, bits = moe.moe_read_device_status(err)
    if status not in (moe.MOE_OK, moe.MOE_ERR_OVERFLOW):
        raise SystemExit(f"device status {moe.moe_status_string(status)} during warm-up")

    # One step = one moe_ffn.  By default it is captured once in a CUDA graph
    # (as the decode path runs in serving) and replayed.  The timed step is
    # bracketed by two events on the stream around the replay; the per-stage
    # split comes from a second graph of the same call with the stage events
    # as event-record nodes (they sit between the kernels, so that graph is
    # used for the split only).
    step = lambda: moe.moe_ffn(desc, ws)
    step_ev = lambda: moe.moe_ffn(desc_ev, ws)
    graph = None
    if not args.eager:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            moe.moe_ffn(desc, ws)
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            moe.moe_ffn(desc, ws)
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev):
            moe.moe_ffn(desc_ev, ws)
        for _ in range(args.warmup):
            graph.replay()
            graph_ev.replay()
        torch.cuda.synchronize(dev)
        try:                                       # the graph's stage events must be timeable
            events[0].elapsed_time(events[6])
            step, step_ev = graph.replay, graph_ev.replay
        except RuntimeError as exc:
            print(f"graph stage events not timeable ({exc}); timing eager calls", file=sys.stderr)
            graph = None

    step_ms = []
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            l2_flush.fill_(1)                       # evict the previous step from L2
            t0.record(stream)
            step()
            t1.record(stream)
            torch.cuda.synchronize(dev)
            step_ms.append(t0.elapsed_time(t1))
        t_wall = time.perf_counter() - t_wall
    _barrier(world)
    torch.cuda.synchronize(dev)
    status, bits = moe.moe_read_device_status(err)
    if status not in (moe.MOE_OK, moe.MOE_ERR_OVERFLOW):
        raise SystemExit(f"device status {moe.moe_status_string(status)} in the timed region")
    stage_ms = [0.0] * 6
    g1_ms = []
    # instrumented passes for the per-stage split and the GEMM1 launch time
    # (not part of the value)
    n_split = max(3, min(args.steps, 10))
    for _ in range(n_split):
        l2_flush.fill_(1)
        step_ev()
        torch.cuda.synchronize(dev)
        for i in range(6):
            stage_ms[i] += events[i].elapsed_time(events[i + 1]) / n_split
        g1_ms.append(events[2].elapsed_time(events[3]))

    total_s = sum(step_ms) / 1e3
    total_s = _max_over_ranks(world, total_s)
    rows_all = _sum_over_ranks(world, wl["rows"] * args.steps)
    value = rows_all / total_s
    ms_per_step = 1e3 * total_s / args.steps

    # ------------------------------------------------------------------ e2e (host buffers)
    e2e = None
    if not args.no_e2e:
        x_h = wl["x"].cpu().pin_memory()
        ids_h = wl["topk_ids"].cpu().pin_memory()
        w_h = wl["topk_w"].cpu().pin_memory()
        out_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        x_d = torch.empty_like(wl["x"])
        ids_d = torch.empty_like(wl["topk_ids"])
        w_d = torch.empty_like(wl["topk_w"])
        d2 = make_desc(wl, out, err=err, x=x_d, ids=ids_d, w=w_d)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def host_step():
            x_d.copy_(x_h, non_blocking=True); ids_d.copy_(ids_h, non_blocking=True)
            w_d.copy_(w_h, non_blocking=True)
            moe.moe_ffn(d2, ws)
            out_h.copy_(out, non_blocking=True)

        def time_e2e(run):
            for _ in range(3):
                run()
            torch.cuda.synchronize(dev)
            ms = []
            for _ in range(args.steps):
                l2_flush.fill_(1)
                e0.record(stream)
                run()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms.append(e0.elapsed_time(e1))
            return _max_over_ranks(world, sum(ms) / 1e3)

        def graphed(fn):
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream(dev).wait_stream(side)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                fn()
            return gr

        # Three ways from host buffers, every byte crossing the host link inside
        # the timed region of each step:
        #  host I/O  moe_ffn given the pinned host x / routing / out directly:
        #            the kernels read and write them in place, overlapped with
        #            the compute (the library's host-buffer path; the value);
        #  copies    explicit copies in, moe_ffn, copy out;
        #  eager     the copies path with eager calls instead of a graph.
        # The graph variants are captured once and replayed (as the decode
        # path runs in serving); without graphs (--eager) all are eager.
        eager_s = time_e2e(host_step)
        copies_s = time_e2e(graphed(host_step).replay) if graph is not None else eager_s
        d_host = make_desc(wl, out_h, err=err, x=x_h, ids=ids_h, w=w_h)
        host_io = lambda: moe.moe_ffn(d_host, ws)
        try:
            host_io()
            torch.cuda.synchronize(dev)
            host_s = time_e2e(graphed(host_io).replay if graph is not None else host_io)
        except moe.MoeError as exc:
            print(f"host-buffer moe_ffn refused ({exc}); e2e = the copies path", file=sys.stderr)
            host_s = None
        e2e_s = host_s if host_s is not None else copies_s
        h2d = x_h.numel() * 2 + ids_h.numel() * 4 + w_h.numel() * 4
        e2e = {"value": rows_all / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(out_h.numel() * 2),
               "ms_per_step": 1e3 * e2e_s / args.steps,
               "copies": {"value": rows_all / copies_s, "ms_per_step": 1e3 * copies_s / args.steps},
               "eager": {"value": rows_all / eager_s, "ms_per_step": 1e3 * eager_s / args.steps},
               "how": ("moe_ffn on pinned host x, topk_ids, topk_w and out (read and written in place "
                       "by the kernels across the host link)" if host_s is not None else
                       "pinned-host x, topk_ids, topk_w -> device, moe_ffn, out -> pinned host")
                      + ("; one CUDA graph replay per step" if graph is not None else "; eager calls")
                      + "; 'copies' = explicit copies in and out around moe_ffn; 'eager' = copies, eager calls"}

    # ------------------------------------------------------------------ roofline (GEMM1)
    peaks, peak_src = load_peaks()
    alg = algorithmic_counts(wl)
    g1_s = statistics.mean(g1_ms) / 1e3
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    fp8_peak = FP8_PER_BF16 * peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    t_mem = alg["g1_bytes"] / (hbm_peak * 1e9)
    t_cmp = alg["flops_g1"] / (fp8_peak * 1e12)
    if t_mem >= t_cmp:
        achieved = alg["g1_bytes"] / g1_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak}
    else:
        achieved = alg["flops_g1"] / g1_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak}
    kname = gemm1_variant(wl)
    what = "GEMM1 (W13) + SwiGLU + FP8 requant" if gemm1_fused(wl) else "GEMM1 (W13)"
    roof.update({"traffic": recorded_traffic(kname, args.workload), "kernel": f"{kname} ({what})",
                 "launch_ms": 1e3 * g1_s, "peak_source": f"{peak_src}" +
                 ("" if roof["bound"] == "hbm" else " bf16 burst x2 (nominal FP8:BF16)"),
                 "algorithmic": {"bytes": alg["g1_bytes"], "flops": alg["flops_g1"]}})

    # ------------------------------------------------------------------ CPU oracle baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref_wl = dict(wl, x_host_bits=wl["x"].cpu().view(torch.int16).numpy().view(np.uint16))
        oracle_w = OracleWeights(ref_wl, dev)
        rate, dt, ntok, nrows = time_oracle(ref_wl, oracle_w, budget_s=args.cpu_budget_s)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"first {ntok} local tokens ({nrows} routed rows) through the whole "
                         f"chain, {dt:.1f}s; numpy float64, BLAS threads = all affinity cores"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded)",
            "config": {"workload": f"{cfg.name}: {cfg.description}",
                       "tokens": "routed (token, local expert) rows", "rows_per_step": wl["rows"],
                       "local_tokens": T, "counts": [int(c) for c in wl["counts"]],
                       "max_m": cfg.max_m, "active_experts": wl["active_experts"],
                       "expected_m_hint": wl["expected_m"], "gemm_flags": args.gemm_flags,
                       "l2": "flushed (256 MiB write) before every timed step",
                       "launch": "eager moe_ffn" if graph is None else "moe_ffn captured once in a CUDA graph, replayed per step",
                       "timing": "CUDA events on the launching stream around each step; stage split from a separate instrumented replay",
                       "parallelism": f"replicas x{world}"},
            "stage_ms": {n: round(v, 4) for n, v in zip(
                ["quant (fused into permute)", "quant+permute", "gemm1", "swiglu_quant (fused into gemm1 when 0)", "gemm2", "combine (fused into gemm2 when 0)"], stage_ms)},
            "tflops": alg["flops"] / (ms_per_step / 1e3) / 1e12,
            "weight_gbs": alg["weight_bytes"] / (ms_per_step / 1e3) / 1e9,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": moe.moe_ffn_kernel_count(desc) * args.steps,
            "clocks": clk.summary(),
            "device_status": moe.moe_status_string(status),
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
