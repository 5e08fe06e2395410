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
def build_workload(cfg_name: str, device="cuda", gen_device=None, ue8m0=False, local_experts=None):
    """Seeded inputs of one config resident on `device`; expert weights quantised
    to E4M3 128x128 blocks by the library's weight-quant kernel (with `ue8m0`:
    power-of-two tile scales, also packed for the block-scaled GEMMs, and the
    FFN run with MOE_FFN_UE8M0).  The inputs are drawn on `gen_device`
    (default: `device`) and copied over; the generator is device independent,
    so the values are the same either way.  `local_experts` keeps the routing
    and keeps only the first that many local experts resident (the others act
    as another rank's: their routing slots are skipped) -- a cut-down case of
    the same workload for profiling."""
    import dataclasses
    import torch
    import fp8_grouped_expert_x128_gb300 as moe
    gen = device if gen_device is None else gen_device
    cfg = synth.get_config(cfg_name)
    r = synth.make_routing(cfg)
    cut = local_experts is not None and local_experts < cfg.E
    if cut:
        cfg = dataclasses.replace(cfg, E=local_experts,
                                  description=cfg.description + f" [cut down to the first {local_experts} "
                                                                "local experts, for profiling]")
        r = dict(r, E=cfg.E)
    T, k = r["T"], r["k"]
    x = synth.make_activations(cfg, T, device=gen).to(device)
    ids = torch.from_numpy(r["topk_ids"].astype(np.int32)).to(device)
    w = torch.from_numpy(r["topk_w"].astype(np.float32)).to(device)
    E, H, I = cfg.E, cfg.H, cfg.I
    w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
    w13_s = torch.empty((E, 2 * I // 128, H // 128), dtype=torch.float32, device=device)
    w2 = torch.empty((E, H, I), dtype=torch.uint8, device=device)
    w2_s = torch.empty((E, H // 128, I // 128), dtype=torch.float32, device=device)
    wquant = moe.moe_quant_weight_fp8_ue8m0 if ue8m0 else moe.moe_quant_weight_fp8
    for e in range(E):
        b13 = synth.make_expert_weights(cfg, "w13", e, device=gen).to(device)
        wquant(b13[None], w13[e:e + 1], w13_s[e:e + 1])
        b2 = synth.make_expert_weights(cfg, "w2", e, device=gen).to(device)
        wquant(b2[None], w2[e:e + 1], w2_s[e:e + 1])
        del b13, b2
    extra = {}
    if ue8m0:
        w13_sf = torch.empty(moe.moe_ue8m0_weight_words(E, 2 * I, H), dtype=torch.int32, device=device)
        w2_sf = torch.empty(moe.moe_ue8m0_weight_words(E, H, I), dtype=torch.int32, device=device)
        moe.moe_pack_ue8m0_weight(w13_s, w13_sf, H)
        moe.moe_pack_ue8m0_weight(w2_s, w2_sf, I)
        extra = dict(w13_sf=w13_sf, w2_sf=w2_sf, gemm_flags=moe.MOE_FFN_UE8M0, ue8m0=True)
    torch.cuda.synchronize()
    layout = moe.MOE_LAYOUT_MASKED if cfg.layout == "masked" else moe.MOE_LAYOUT_CONTIG
    local = (r["topk_ids"] >= r["expert_begin"]) & (r["topk_ids"] < r["expert_begin"] + E)
    rows_raw = int(local.sum())
    counts = np.array([(r["topk_ids"] == r["expert_begin"] + e).sum() for e in range(E)])
    rows = int(np.minimum(counts, cfg.max_m).sum()) if cfg.layout == "masked" else rows_raw
    expected_m = int(math.ceil(rows / max(1, int((counts > 0).sum()))))
    return dict(cfg=cfg, routing=r, T=T, k=k, x=x, topk_ids=ids, topk_w=w, w13=w13, w13_s=w13_s,
                w2=w2, w2_s=w2_s, layout=layout, rows=rows, counts=counts,
                active_experts=int((counts > 0).sum()), expected_m=expected_m, **extra)


def make_desc(wl, out, err=None, stage_events=None, x=None, ids=None, w=None):
    import fp8_grouped_expert_x128_gb300 as moe
    cfg = wl["cfg"]
    return moe.make_ffn_desc(x if x is not None else wl["x"], ids if ids is not None else wl["topk_ids"],
                             w if w is not None else wl["topk_w"], wl["w13"], wl["w13_s"], wl["w2"],
                             wl["w2_s"], out, wl["routing"]["expert_begin"], cfg.E, wl["layout"],
                             max_m=cfg.max_m, expected_m=wl["expected_m"],
                             gemm_flags=wl.get("gemm_flags", 0), err=err, stage_events=stage_events,
                             w13_sf=wl.get("w13_sf"), w2_sf=wl.get("w2_sf"))


def is_ue8m0(wl):
    import fp8_grouped_expert_x128_gb300 as moe
    return bool(wl.get("gemm_flags", 0) & moe.MOE_FFN_UE8M0)


def _ue8m0_variant(wl):
    import fp8_grouped_expert_x128_gb300 as moe
    if wl["layout"] == moe.MOE_LAYOUT_MASKED:
        v = moe.moe_gemm_fp8_masked_variant(wl["cfg"].max_m, wl["expected_m"], wl.get("gemm_flags", 0))
        if v != 0:
            return f"gemm_fp8_ue8m0_weights_m_kernel<{min(v, 128)}>"
    return "gemm_fp8_ue8m0_kernel"


def gemm1_variant(wl):
    """The GEMM1 kernel moe_ffn runs for this workload."""
    import fp8_grouped_expert_x128_gb300 as moe
    if is_ue8m0(wl):
        return _ue8m0_variant(wl)
    if wl["layout"] == moe.MOE_LAYOUT_MASKED:
        v = moe.moe_gemm_fp8_masked_variant(wl["cfg"].max_m, wl["expected_m"], wl.get("gemm_flags", 0))
        if v != 0:
            return f"gemm_fp8_weights_m_kernel<{v}>"
    if wl.get("gemm_flags", 0) & moe.MOE_FFN_FUSE_SWIGLU:
        return "gemm_fp8_tokens_m_kernel<swiglu>"
    return "gemm_fp8_tokens_m_kernel"


def gemm1_fused(wl):
    return gemm1_variant(wl).endswith("<swiglu>")


def gemm2_variant(wl):
    """The GEMM2 kernel moe_ffn runs for this workload."""
    import fp8_grouped_expert_x128_gb300 as moe
    if is_ue8m0(wl):
        return _ue8m0_variant(wl) + ("<combine1>" if combine_fused(wl) else "")
    if wl["layout"] == moe.MOE_LAYOUT_MASKED:
        v = moe.moe_gemm_fp8_masked_variant(wl["cfg"].max_m, wl["expected_m"], wl.get("gemm_flags", 0))
        if v != 0:
            return f"gemm_fp8_weights_m_kernel<{v}>"
    if combine_fused(wl):
        return "gemm_fp8_tokens_m_kernel<combine1>"
    return "gemm_fp8_tokens_m_kernel"


def combine_fused(wl):
    """moe_ffn folds the combine into GEMM2's epilogue for one routing slot per
    token (device output; the tokens-as-M kernel serving GEMM2)."""
    import fp8_grouped_expert_x128_gb300 as moe
    if wl["k"] != 1:
        return False
    if wl["layout"] == moe.MOE_LAYOUT_MASKED:
        return moe.moe_gemm_fp8_masked_variant(wl["cfg"].max_m, wl["expected_m"], wl.get("gemm_flags", 0)) == 0
    return True


def units_per_step(wl):
    """The metric's unit per step: routed (token, local expert) rows for the
    post-dispatch workloads (EP72 decode, EP32 prefill), tokens otherwise."""
    return wl["rows"] if wl["cfg"].name.startswith(("c2", "c3")) else wl["T"]


def unit_name(wl):
    return "routed (token, local expert) rows" if wl["cfg"].name.startswith(("c2", "c3")) else "tokens"


def algorithmic_counts(wl):
    """Algorithmic FLOPs and HBM bytes per step and per GEMM launch (padding
    rows and idle experts excluded): weights once per active expert, each
    activation tensor once in and once out."""
    cfg = wl["cfg"]
    H, I = cfg.H, cfg.I
    rows, act, T, k = wl["rows"], wl["active_experts"], wl["T"], wl["k"]
    fused = gemm1_fused(wl)
    sb = 1 if is_ue8m0(wl) else 4                    # bytes per block scale: exponent byte or fp32
    flops_g1 = 2.0 * rows * H * 2 * I
    flops_g2 = 2.0 * rows * I * H
    w13_bytes = act * (2 * I * H + sb * (2 * I // 128) * (H // 128))
    w2_bytes = act * (H * I + sb * (H // 128) * (I // 128))
    a1 = rows * (H + sb * H / 128)                   # FP8 rows + their scales into GEMM1
    a2 = rows * (I + sb * I / 128)                   # FP8 h + scales into GEMM2
    y1 = rows * 2 * I * 2                            # bf16 Y1
    y2 = rows * H * 2                                # bf16 Y2
    out = T * H * 2
    g1_bytes = w13_bytes + a1 + (a2 if fused else y1)
    g2_bytes = w2_bytes + a2 + (out if combine_fused(wl) else y2)
    # the whole step: x in, the routed rows through both GEMMs, out
    step_bytes = (T * H * 2 + T * k * 4 * 2 + a1 + w13_bytes + w2_bytes + a2 +
                  (0 if fused else 2 * y1) + (out if combine_fused(wl) else 2 * y2 + out))
    return dict(flops=flops_g1 + flops_g2, flops_g1=flops_g1, flops_g2=flops_g2, g1_bytes=g1_bytes,
                g2_bytes=g2_bytes, weight_bytes=w13_bytes + w2_bytes, step_bytes=step_bytes)


def roofline(flops, nbytes, seconds, peaks):
    """Bound = whichever of bytes / HBM peak and FLOPs / FP8 peak is larger;
    achieved and frac against that peak; both fractions alongside."""
    hbm, fp8 = peaks["hbm_gbs"], peaks["fp8_tflops"]
    t_mem, t_cmp = nbytes / (hbm * 1e9), flops / (fp8 * 1e12)
    gbs, tfs = nbytes / seconds / 1e9, flops / seconds / 1e12
    if t_mem >= t_cmp:
        r = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm}
    else:
        r = {"bound": "tensor", "achieved": tfs, "peak": fp8, "unit": "TFLOP/s", "frac": tfs / fp8}
    r.update({"hbm_frac": gbs / hbm, "fp8_frac": tfs / fp8, "t_min_ms": 1e3 * max(t_mem, t_cmp),
              "algorithmic": {"bytes": nbytes, "flops": flops}})
    return r


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
def _oracle_rows(wl, oracle_w, assignments):
    """The oracle chain on a sample of routed rows (rows are independent): each
    sampled assignment (t, j) quantises token t, runs GEMM1 -> SwiGLU+quant ->
    GEMM2 against its expert, and the sampled rows of each token are combined
    with their weights.  Returns the number of routed rows processed."""
    import oracle
    cfg = wl["cfg"]
    r = wl["routing"]
    by_token = {}
    for t, j in assignments:
        by_token.setdefault(t, []).append(j)
    n_rows = 0
    for t, slots in by_token.items():
        q, s = oracle.quant_1x128(oracle.bf16_decode(wl["x_host_bits"][t:t + 1]).astype(np.float32))
        y2_rows, ws = [], []
        for j in slots:
            e = int(r["topk_ids"][t, j]) - r["expert_begin"]
            w13q, w13s, w2q, w2s = oracle_w[e]
            y1 = oracle.bf16_encode(oracle.gemm_block_scaled(q, s, w13q, w13s))
            q2, s2 = oracle.swiglu_quant(y1)
            y2_rows.append(oracle.bf16_encode(oracle.gemm_block_scaled(q2, s2, w2q, w2s))[0])
            ws.append(float(r["topk_w"][t, j]))
            n_rows += 1
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


def local_assignments(wl):
    """The routed (token, slot) pairs the FFN processes, in assignment order
    (masked layouts: the ones kept under max_m)."""
    r = wl["routing"]
    cfg = wl["cfg"]
    e = r["topk_ids"] - r["expert_begin"]
    out = []
    seen = np.zeros(cfg.E, np.int64)
    for t in range(r["T"]):
        for j in range(r["k"]):
            ee = int(e[t, j])
            if 0 <= ee < cfg.E and (cfg.layout != "masked" or seen[ee] < cfg.max_m):
                seen[ee] += 1
                out.append((t, j))
    return out


def time_oracle(wl, oracle_w, budget_s=15.0, start=0):
    """Time the oracle on a bounded sample of the workload's routed rows, taken
    in assignment order from `start`: one row first to estimate the cost, then
    as many as fit in about `budget_s`.  Weight preparation happens before each
    timed region.  Returns (value in the metric's unit per second, seconds
    timed, rows): rows/s for row-unit workloads, rows/s x tokens per routed row
    for token-unit workloads."""
    rows_all = wl.get("_assign")
    if rows_all is None:
        rows_all = wl["_assign"] = local_assignments(wl)
    n = len(rows_all)
    e_of = lambda a: int(wl["routing"]["topk_ids"][a]) - wl["routing"]["expert_begin"]
    first = [rows_all[start % n]]
    oracle_w.prepare([e_of(a) for a in first])
    t0 = time.perf_counter()
    rows = _oracle_rows(wl, oracle_w, first)
    dt = time.perf_counter() - t0
    n_more = int(max(0.0, budget_s - dt) / max(dt, 1e-3))
    more = [rows_all[(start + 1 + i) % n] for i in range(min(n_more, n - 1))]
    if more:
        oracle_w.prepare([e_of(a) for a in more])
        t1 = time.perf_counter()
        rows += _oracle_rows(wl, oracle_w, more)
        dt += time.perf_counter() - t1
    per_unit = units_per_step(wl) / wl["rows"]           # metric units per routed row
    return rows / dt * per_unit, dt, rows


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


def kernel_source(kernel_label: str) -> str:
    """The source file that holds a GEMM kernel (by its label)."""
    return "gemm_bs.cu" if "ue8m0" in kernel_label else "gemm.cu"


def recorded_traffic(kernel_label: str, workload: str, which: str = "gemm1"):
    """DRAM bytes (read + write) per launch of this kernel (as GEMM1 or GEMM2) on
    this workload from the ncu capture recorded in profiles/traffic.json, or
    None when there is no capture or the kernel's source file has changed since
    it was taken.  A record may hold a capture of a cut-down case scaled to the
    full launch (its "scaled_from" field says how)."""
    import hashlib
    path = os.path.join(HERE, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    src_name = kernel_source(kernel_label)
    with open(os.path.join(HERE, "fp8_grouped_expert_x128_gb300", "csrc", src_name), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    with open(path) as f:
        rec = json.load(f)
    r = rec.get(f"{kernel_label}@{workload}:{which}")
    if not r or r.get("src") != src_name or r.get("src_sha256") != sha:
        return None
    return r["dram_read_bytes"] + r["dram_write_bytes"]


def load_peaks():
    p = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def config_dict(wl, world):
    """The workload the line is quoted on (the same dict for both arms)."""
    cfg = wl["cfg"]
    return {"workload": f"{cfg.name}: {cfg.description}", "tokens": unit_name(wl),
            "units_per_step": units_per_step(wl), "rows_per_step": wl["rows"], "local_tokens": wl["T"],
            "counts": [int(c) for c in wl["counts"]], "max_m": cfg.max_m,
            "active_experts": wl["active_experts"], "hidden": cfg.H, "intermediate": cfg.I,
            "l2": "flushed (256 MiB write) before every timed step", "parallelism": f"replicas x{world}"}


def routing_summary(cfg_name):
    """Host-side facts of a workload (no GPU): routing, counts, rows."""
    cfg = synth.get_config(cfg_name)
    r = synth.make_routing(cfg)
    E = cfg.E
    counts = np.array([(r["topk_ids"] == r["expert_begin"] + e).sum() for e in range(E)])
    rows = int(np.minimum(counts, cfg.max_m).sum()) if cfg.layout == "masked" else int(counts.sum())
    return dict(cfg=cfg, routing=r, T=r["T"], k=r["k"], counts=counts, rows=rows,
                active_experts=int((counts > 0).sum()))


def host_workload(name):
    """The host-side facts of '<config>' or '<config>:ue8m0' that choose the
    kernels and their labels (no tensors, no GPU): what build_workload returns
    minus the device buffers."""
    import fp8_grouped_expert_x128_gb300 as moe
    cfg_name, _, variant = name.partition(":")
    wl = routing_summary(cfg_name)
    wl["layout"] = moe.MOE_LAYOUT_MASKED if wl["cfg"].layout == "masked" else moe.MOE_LAYOUT_CONTIG
    wl["expected_m"] = int(math.ceil(wl["rows"] / max(1, wl["active_experts"])))
    if variant == "ue8m0":
        wl["ue8m0"] = True
        wl["gemm_flags"] = moe.MOE_FFN_UE8M0
    return wl


def traffic_name(name):
    """The workload part of a profiles/traffic.json key ('c3:ue8m0' -> 'c3-ue8m0':
    the key itself is '<kernel>@<workload>:<gemm1|gemm2>')."""
    return name.replace(":", "-")


DEFAULT_HEADLINE = "c5"
DEFAULT_EXTRA = "c2,c3,c4,c3:ue8m0,c4:ue8m0,c2:ue8m0,c5:ue8m0"


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample per step."""
    if rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = routing_summary(args.workload)
    x = synth.make_activations(wl["cfg"], wl["T"], device=dev)
    wl["x_host_bits"] = x.cpu().view(torch.int16).numpy().view(np.uint16)
    oracle_w = OracleWeights(wl, dev)
    per_step = []
    for i in range(args.warmup + args.steps):
        rate, dt, nrows = time_oracle(wl, oracle_w, budget_s=args.ref_step_s, start=i * 7)
        if i >= args.warmup:
            per_step.append((rate, dt, nrows))
    per_unit = units_per_step(wl) / wl["rows"]
    units = sum(p[2] for p in per_step) * per_unit
    secs = sum(p[1] for p in per_step)
    value = units / secs
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, len(per_step)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": config_dict(wl, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: routed rows in assignment order, ~{args.ref_step_s:.0f}s of "
                                   f"CPU work (~{per_step[0][2]} rows), scaled to {unit_name(wl)} at "
                                   f"{per_unit:.4g} per routed row; numpy float64, BLAS threads = all "
                                   "affinity cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Step:
    """One moe_ffn step of a workload, captured once in a CUDA graph (as the
    decode path runs in serving) and replayed; a second graph of the same call
    records the seven stage events between the kernels (used for the per-stage
    split and the GEMM launch times only, never for the value)."""

    def __init__(self, wl, dev, eager=False):
        import torch
        import fp8_grouped_expert_x128_gb300 as moe
        self.moe, self.dev, self.wl = moe, dev, wl
        cfg = wl["cfg"]
        self.out = torch.empty((wl["T"], cfg.H), dtype=torch.bfloat16, device=dev)
        self.err = moe.new_error_word(dev)
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        self.desc = make_desc(wl, self.out, err=self.err)
        self.desc_ev = make_desc(wl, self.out, err=self.err, stage_events=self.events)
        self.ws = moe.alloc_workspace(self.desc, dev)
        self.run = lambda: moe.moe_ffn(self.desc, self.ws)
        self.run_ev = lambda: moe.moe_ffn(self.desc_ev, self.ws)
        self.graph = None
        self.eager = eager

    def capture(self, warmup):
        import torch
        dev = self.dev
        for _ in range(warmup):
            self.run()
        torch.cuda.synchronize(dev)
        self.check("warm-up")
        if self.eager:
            return
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        g_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ev):
            self.run_ev()
        for _ in range(warmup):
            g.replay()
            g_ev.replay()
        torch.cuda.synchronize(dev)
        try:                                       # the graph's stage events must be timeable
            self.events[0].elapsed_time(self.events[6])
            self.graph = g
            self.run, self.run_ev = g.replay, g_ev.replay
        except RuntimeError as exc:
            print(f"graph stage events not timeable ({exc}); timing eager calls", file=sys.stderr)

    def check(self, where):
        st, _ = self.moe.moe_read_device_status(self.err)
        if st not in (self.moe.MOE_OK, self.moe.MOE_ERR_OVERFLOW):
            raise SystemExit(f"device status {self.moe.moe_status_string(st)} in {where}")
        return st

    def time(self, n, l2_flush, stream):
        """Device time of n steps, each preceded by an L2-evicting write, with two
        CUDA events on the launching stream around each step."""
        import torch
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ms = []
        for _ in range(n):
            l2_flush.fill_(1)
            t0.record(stream)
            self.run()
            t1.record(stream)
            torch.cuda.synchronize(self.dev)
            ms.append(t0.elapsed_time(t1))
        return ms

    def soak(self, seconds, l2_flush):
        """Untimed steps for about `seconds` (the clock sampler sees the load)."""
        import torch
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(16):
                l2_flush.fill_(1)
                self.run()
            torch.cuda.synchronize(self.dev)

    def split(self, n, l2_flush):
        """Per-stage times (mean over n instrumented replays) and the GEMM1 and
        GEMM2 launch times of each replay."""
        import torch
        stage = [0.0] * 6
        g1, g2 = [], []
        for _ in range(n):
            l2_flush.fill_(1)
            self.run_ev()
            torch.cuda.synchronize(self.dev)
            for i in range(6):
                stage[i] += self.events[i].elapsed_time(self.events[i + 1]) / n
            g1.append(self.events[2].elapsed_time(self.events[3]))
            g2.append(self.events[4].elapsed_time(self.events[5]))
        return stage, g1, g2


STAGES = ["quant (fused into permute)", "quant+permute", "gemm1", "swiglu_quant (fused into gemm1 when 0)",
          "gemm2", "combine (fused into gemm2 when 0)"]


def kernel_rooflines(wl, name, g1_s, g2_s, peaks, peak_src):
    alg = algorithmic_counts(wl)
    out = {}
    for which, kname, sec, flops, nbytes in (
            ("gemm1", gemm1_variant(wl), g1_s, alg["flops_g1"], alg["g1_bytes"]),
            ("gemm2", gemm2_variant(wl), g2_s, alg["flops_g2"], alg["g2_bytes"])):
        r = roofline(flops, nbytes, sec, peaks)
        what = {"gemm1": "GEMM1 (W13)" + (" + SwiGLU + FP8 requant" if gemm1_fused(wl) else ""),
                "gemm2": "GEMM2 (W2)" + (" + single-slot combine" if combine_fused(wl) else "")}[which]
        r.update({"kernel": f"{kname} ({what})", "launch_ms": 1e3 * sec,
                  "traffic": recorded_traffic(kname.split(" ")[0], name, which),
                  "peak_source": peak_src + ("" if r["bound"] == "hbm" else " bf16 burst x2 (nominal FP8:BF16)")})
        out[which] = r
    return out


def measure(name, args, dev, world, l2_flush, stream, peaks, peak_src, clk_seconds=0.0):
    """Build a workload ('<config>' or '<config>:ue8m0' for the power-of-two
    reading of the scales end to end), time K steps, and report its line fields."""
    cfg_name, _, variant = name.partition(":")
    wl = build_workload(cfg_name, dev, ue8m0=variant == "ue8m0", local_experts=args.local_experts)
    if args.expected_m is not None:
        wl["expected_m"] = args.expected_m
    wl["gemm_flags"] = wl.get("gemm_flags", 0) | args.gemm_flags
    st = Step(wl, dev, eager=args.eager)
    st.capture(args.warmup)
    clk = ClockSampler(dev.index if dev.index is not None else 0) if clk_seconds > 0 else None
    _barrier(world)
    import torch
    torch.cuda.synchronize(dev)
    if clk is not None:
        clk.__enter__()
        st.soak(clk_seconds, l2_flush)
    t_wall = time.perf_counter()
    step_ms = st.time(args.steps, l2_flush, stream)
    t_wall = time.perf_counter() - t_wall
    if clk is not None:
        clk.__exit__(None, None, None)
    _barrier(world)
    status = st.check("the timed region")
    stage_ms, g1, g2 = st.split(max(3, min(args.steps, 10)), l2_flush)
    total_s = _max_over_ranks(world, sum(step_ms) / 1e3)
    units = _sum_over_ranks(world, units_per_step(wl) * args.steps)
    ms_per_step = 1e3 * total_s / args.steps
    alg = algorithmic_counts(wl)
    g1_s, g2_s = statistics.mean(g1) / 1e3, statistics.mean(g2) / 1e3
    rep = {
        "value": units / total_s, "ms_per_step": ms_per_step,
        "stage_ms": {n: round(v, 4) for n, v in zip(STAGES, stage_ms)},
        "kernels": kernel_rooflines(wl, traffic_name(name), g1_s, g2_s, peaks, peak_src),
        "step_roofline": roofline(alg["flops"], alg["step_bytes"], ms_per_step / 1e3, peaks),
        "tflops": alg["flops"] / (ms_per_step / 1e3) / 1e12,
        "weight_gbs": alg["weight_bytes"] / (ms_per_step / 1e3) / 1e9,
        "gpu_launches": moe_kernel_count(st) * args.steps,
        "device_status": st.moe.moe_status_string(status),
        "tuning": {"expected_m_hint": wl["expected_m"], "gemm_flags": wl["gemm_flags"],
                   "launch": "eager moe_ffn" if st.graph is None else
                             "moe_ffn captured once in a CUDA graph, replayed per step",
                   "gemm1": gemm1_variant(wl), "gemm2": gemm2_variant(wl)},
        "wall_s_timed": t_wall,
    }
    return wl, st, rep, clk


def moe_kernel_count(st):
    return st.moe.moe_ffn_kernel_count(st.desc)


def e2e_leg(wl, st, args, dev, world, l2_flush, stream):
    """The same metric through the public call with the step's inputs and output
    crossing the host link inside every timed step (pinned host buffers)."""
    import torch
    moe = st.moe
    T, H = wl["T"], wl["cfg"].H
    x_h = wl["x"].cpu().pin_memory()
    ids_h = wl["topk_ids"].cpu().pin_memory()
    w_h = wl["topk_w"].cpu().pin_memory()
    out_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(wl["x"])
    ids_d = torch.empty_like(wl["topk_ids"])
    w_d = torch.empty_like(wl["topk_w"])
    d2 = make_desc(wl, st.out, err=st.err, x=x_d, ids=ids_d, w=w_d)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def host_step():
        x_d.copy_(x_h, non_blocking=True); ids_d.copy_(ids_h, non_blocking=True)
        w_d.copy_(w_h, non_blocking=True)
        moe.moe_ffn(d2, st.ws)
        out_h.copy_(st.out, non_blocking=True)

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

    # Three ways from host buffers, every byte crossing the host link inside the
    # timed region of each step:
    #  host I/O  moe_ffn given the pinned host x / routing / out directly: the
    #            kernels read and write them in place, overlapped with the
    #            compute (the library's host-buffer path; the value);
    #  copies    explicit copies in, moe_ffn, copy out;
    #  eager     the copies path with eager calls instead of a graph.
    use_graph = st.graph is not None
    eager_s = time_e2e(host_step)
    copies_s = time_e2e(graphed(host_step).replay) if use_graph else eager_s
    d_host = make_desc(wl, out_h, err=st.err, x=x_h, ids=ids_h, w=w_h)
    host_io = lambda: moe.moe_ffn(d_host, st.ws)
    try:
        host_io()
        torch.cuda.synchronize(dev)
        host_s = time_e2e(graphed(host_io).replay if use_graph else host_io)
    except moe.MoeError as exc:
        print(f"host-buffer moe_ffn refused ({exc}); e2e = the copies path", file=sys.stderr)
        host_s = None
    e2e_s = host_s if host_s is not None else copies_s
    units = _sum_over_ranks(world, units_per_step(wl) * args.steps)
    h2d = x_h.numel() * 2 + ids_h.numel() * 4 + w_h.numel() * 4
    return {"value": units / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(out_h.numel() * 2),
            "ms_per_step": 1e3 * e2e_s / args.steps,
            "copies": {"value": units / copies_s, "ms_per_step": 1e3 * copies_s / args.steps},
            "eager": {"value": units / eager_s, "ms_per_step": 1e3 * eager_s / args.steps},
            "how": ("moe_ffn on pinned host x, topk_ids, topk_w and out (read and written in place "
                    "by the kernels across the host link)" if host_s is not None else
                    "pinned-host x, topk_ids, topk_w -> device, moe_ffn, out -> pinned host")
                   + ("; one CUDA graph replay per step" if use_graph else "; eager calls")
                   + "; 'copies' = explicit copies in and out around moe_ffn; 'eager' = copies, eager calls"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_HEADLINE,
                    help="the headline workload (default: the all-experts decode layer, the largest "
                         "configuration that fits one GPU)")
    ap.add_argument("--extra", default=DEFAULT_EXTRA,
                    help="comma-separated workloads also measured in the same run, reported under "
                         "'workloads' (not part of the value); '<config>:ue8m0' runs the power-of-two "
                         "reading of the scales end to end (block-scaled GEMMs); empty for none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--clock-soak-s", type=float, default=1.0,
                    help="untimed steps run under the clock sampler right before the timed region")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--local-experts", type=int, default=None,
                    help="keep only the first N local experts resident (the rest act as another rank's); "
                         "a cut-down case of the workload for profiling, not a bench line")
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
    dev = torch.device("cuda", local if world > 1 else 0)
    peaks_raw, peak_src = load_peaks()
    peaks = {"hbm_gbs": peaks_raw.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]),
             "fp8_tflops": FP8_PER_BF16 * peaks_raw.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])}
    l2_flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # other workloads first (each freed before the next), the headline last
    extra = {}
    for name in [n for n in args.extra.split(",") if n and n != args.workload]:
        wl_x, st_x, rep_x, _ = measure(name, args, dev, world, l2_flush, stream, peaks, peak_src)
        rep_x.update({"workload": f"{wl_x['cfg'].name}: {wl_x['cfg'].description}", "tokens": unit_name(wl_x),
                      "scales": "UE8M0 (power-of-two, packed; block-scaled MMA)" if is_ue8m0(wl_x)
                                else "fp32 (per-k-block promotion)"})
        extra[name] = rep_x
        del wl_x, st_x
        torch.cuda.empty_cache()

    wl, st, rep, clk = measure(args.workload, args, dev, world, l2_flush, stream, peaks, peak_src,
                               clk_seconds=args.clock_soak_s)
    e2e = None if args.no_e2e else e2e_leg(wl, st, args, dev, world, l2_flush, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref_wl = dict(wl, x_host_bits=wl["x"].cpu().view(torch.int16).numpy().view(np.uint16))
        oracle_w = OracleWeights(ref_wl, dev)
        rate, dt, nrows = time_oracle(ref_wl, oracle_w, budget_s=args.cpu_budget_s)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"the first {nrows} routed rows in assignment order through the whole chain "
                         f"(quant, GEMM1, SwiGLU+quant, GEMM2, combine), {dt:.1f}s, scaled to "
                         f"{unit_name(wl)} at {units_per_step(wl) / wl['rows']:.4g} per routed row; "
                         "numpy float64, BLAS threads = all affinity cores"}

    if rank == 0:
        k = rep["kernels"]
        dominant = max(("gemm1", "gemm2"), key=lambda w: k[w]["launch_ms"])
        roof = dict(k[dominant])
        clocks = clk.summary() if clk is not None else {"sm_mhz": None, "reasons": ["unsampled"]}
        clocks["window"] = (f"{args.clock_soak_s:.1f}s of untimed steps immediately before the timed region, "
                            "and the timed region")
        line = {
            "metric": METRIC, "value": rep["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rep["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded)",
            "config": config_dict(wl, world),
            "stage_ms": rep["stage_ms"],
            "tflops": rep["tflops"], "weight_gbs": rep["weight_gbs"],
            "roofline": roof,
            "kernels": k,
            "step_roofline": rep["step_roofline"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": rep["gpu_launches"],
            "clocks": clocks,
            "device_status": rep["device_status"],
            "tuning": rep["tuning"],
            "timing": "CUDA events on the launching stream around each step (graph replay); stage split "
                      "and GEMM launch times from a separate instrumented replay",
            "wall_s_timed": rep["wall_s_timed"],
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
