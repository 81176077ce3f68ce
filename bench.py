"""Benchmark of the LLSA hot path on GB300: one step = pool -> select ->
forward -> index transpose -> backward over one batch of synthetic inputs
already resident in HBM (256x256 pixel tokens by default), timed with CUDA
events. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl llsa|reference]

Under torchrun (N > 1) every rank runs its own independent problem of the
same size (weak scaling, no collective on the data path); the rank times are
reduced with MAX. `--impl reference` times the CPU oracle on a bounded sample
of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from hierarchical_sparse_attention_mean_gb300 import synth  # noqa: E402

METRIC = "LLSA fwd+bwd ms & effective TFLOP/s at N=65536 (1×GB300); % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
SMS, FP32_LANES_PER_SM = 152, 128


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p.get(k, FALLBACK_PEAKS[k])) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def csrc_digest() -> str:
    """Digest of the CUDA sources and the C header: a recorded ncu figure
    applies only to the build it was taken on."""
    import hashlib
    h = hashlib.sha256()
    for d in ("hierarchical_sparse_attention_mean_gb300/csrc", "include"):
        for f in sorted(os.listdir(os.path.join(ROOT, d))):
            if f.endswith((".cu", ".cuh", ".h")):
                rel = os.path.join(d, f)
                h.update(rel.encode())
                with open(os.path.join(ROOT, rel), "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    of `kernel` from the committed ncu summary of this workload, or None when
    the summary is missing or was taken on other sources."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.md")
    if not os.path.exists(path):
        return None
    digest, table = None, {}
    with open(path) as f:
        for line in f:
            if line.startswith("csrc digest:"):
                digest = line.split(":", 1)[1].strip().strip("`")
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0].startswith("`"):
                try:
                    table[cells[0].strip("`")] = float(cells[3].replace(",", ""))
                except ValueError:
                    pass
    if digest != csrc_digest():
        return None
    return table.get(kernel)


def rank_workload(w0, rank: int):
    """Each rank's problem: the same size, its own seed (weak scaling, no
    data shared between ranks)."""
    return synth.Workload(**{**w0.__dict__, "seed": w0.seed + 7919 * rank})


def max_over_ranks(x: float, ws: int, device) -> float:
    """MAX of a per-rank time over all ranks (the job ends with its slowest
    rank); the identity on one rank."""
    if ws == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(ws: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput (TFLOP/s): every rank's work over the slowest
    rank's time."""
    return ws * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------- work model

def work_model(w: synth.Workload, s) -> dict:
    """Algorithmic work of one step (useful sparse work only)."""
    bh, n, d = w.bh, w.n, w.d
    es = 2 if w.dtype == "bf16" else 4
    pairs = bh * n * s.keys_per_query                 # (query, key) pairs incl. coarse tokens
    fine_pairs = bh * n * s.topk_level[1] * w.block
    tok = bh * n * d * es                             # bytes of one token tensor
    P = s.pyr_rows
    scored = s.n_level[s.levels] ** 2 + sum(s.n_level[l] * s.topk_level[l + 1] * w.block
                                             for l in range(1, s.levels))
    return {
        "pairs": pairs,
        "fwd_flops": 4 * d * pairs,
        "bwd_flops": 10 * d * pairs,
        "step_flops": 14 * d * pairs,
        "select_flops": 2 * d * scored * bh,
        # per kernel: (bytes, flops) that the kernel's algorithm needs
        "kernels": {
            "pool_chunk": (3 * tok + 3 * bh * P * d * 4, 0),
            "fwd": (4 * tok + bh * n * 4, 4 * d * pairs),
            # reads Q, dO, o, lse and the gathered K, V (each once from HBM);
            # writes dq, the (lse, D) pairs and the pooled-level partials
            "bwd_dq": (6 * tok + bh * n * 12 + 2 * bh * s.n_blocks * s.enrich_cols * d * 4, 6 * d * pairs),
            "bwd_dkv": (6 * tok + bh * n * 8, 8 * d * fine_pairs),
            # reads the selection, writes row_idx and col_ptr (each once)
            "transpose": (4 * bh * (2 * s.n_blocks * s.topk_level[1] + s.n_blocks + 1), 0),
            "select_level": (0, 2 * d * scored * bh),
        },
    }


# Per-SM intake of scattered 2 KB copies into a ring of stages, measured by a
# TMA microbenchmark on GB300 (one 128-row box per request; bytes per SM clock).
GATHER_B_PER_CLK_SM = 23.9


def gather_intake(w, s, b, stage_ms, clocks, dev):
    """The tensor-core kernels' gathered bytes (every selected block and
    stacked query block as it is copied into shared memory) per step, their
    rate, and that rate against the per-SM copy-intake ceiling at the SM clock
    seen in the timed region. A diagnostic beside the HBM roofline: these
    kernels gather from L2, so HBM is not what binds them."""
    import torch
    if w.dtype != "bf16" or not clocks or not clocks.get("sm_mhz"):
        return None
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ceiling = GATHER_B_PER_CLK_SM * sms * clocks["sm_mhz"] * 1e6  # bytes/s
    blk = 16 * w.d * 2                                  # one 16-row block of a token tensor
    pooled = 2 * s.enrich_cols * w.d * 4                # pooled K and V rows (fp32)
    qblocks = w.bh * s.n_blocks
    k1 = s.topk_level[1]
    cnt = (b.col_ptr[:, 1:] - b.col_ptr[:, :-1]).to(torch.int64)
    items = int(((cnt + 7) // 8).sum().item())
    entries = int(cnt.sum().item())
    fwd_blocks = grouped_fwd_blocks(b, s)  # key blocks the grouped forward gathers (K and V each)
    gathered = {
        "fwd": (qblocks * blk + 2 * fwd_blocks * blk + qblocks * pooled) if fwd_blocks is not None
        else qblocks * (blk + 2 * k1 * blk + pooled),
        "bwd_dq": qblocks * (3 * blk + 2 * k1 * blk + 64 + pooled),
        "bwd_dkv": items * 2 * blk + entries * 2 * blk,
    }
    out = {}
    for k, nbytes in gathered.items():
        if k in stage_ms and stage_ms[k] > 0:
            rate = nbytes / (stage_ms[k] * 1e-3)
            out[k] = {"gathered_gb": round(nbytes / 1e9, 3), "tbs": round(rate / 1e12, 2),
                      "frac": round(rate / ceiling, 3)}
    return {"ceiling_tbs": round(ceiling / 1e12, 2),
            "ceiling_source": f"{GATHER_B_PER_CLK_SM} B per SM clock (copy-intake microbenchmark) x {sms} SMs "
                              f"x {clocks['sm_mhz']:.0f} MHz",
            "kernels": out}


def grouped_fwd_blocks(b, s, window: int = 1024):
    """Key blocks the grouped tensor-core forward gathers in one step: for
    every group of query blocks (read back from the forward's workspace), the
    size of the union of their selections. None when the forward took no
    workspace (no grouping) or the per-query-block forward took the call
    (groups of fewer than 4.5 query blocks on average, the library's rule)."""
    import numpy as np
    import torch
    T, slices = s.n_blocks, s.slices
    if b.ws_f.numel() < 8 * slices * T:
        return None
    windows = (T + window - 1) // window
    ws = b.ws_f.view(torch.int32)[:2 * slices * T + slices * windows + 128].cpu().numpy()
    a = ((4 * slices * T + 255) // 256) * 256 // 4
    order = ws[:slices * T].reshape(slices, T)
    gdesc = ws[a:a + slices * T].reshape(slices, T)
    ngroups = ws[2 * a:2 * a + slices * windows].reshape(slices, windows)
    if 2 * slices * T < 9 * int(ngroups.sum()):
        return None
    sel = b.sel_idx.cpu().numpy().astype(np.int64)
    total = 0
    for sl in range(slices):
        gid = np.empty(T, np.int64)
        g0 = 0
        for wi in range(windows):
            gd = gdesc[sl, wi * window:wi * window + ngroups[sl, wi]]
            for k, v in enumerate(gd):
                start, c = int(v) & 0xFFFF, int(v) >> 16
                gid[order[sl, start:start + c]] = g0 + k
            g0 += len(gd)
        total += np.unique(gid[:, None] * T + sel[sl]).size
    return int(total)


def spread(values):
    """Median and 10th / 90th percentiles (nearest rank) of per-step times, ms."""
    if not values:
        return None
    v = sorted(values)
    at = lambda q: v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]
    return {"p10": round(at(0.1), 4), "median": round(at(0.5), 4), "p90": round(at(0.9), 4)}


def kernel_key(name: str) -> str:
    for key in ("pool_chunk", "bwd_dq", "bwd_dkv", "select_level", "coarse_reduce"):
        if name.startswith(key):
            return key
    if name.startswith("fwd"):
        return "fwd"
    if name.startswith("transpose"):
        return "transpose"
    return name


def kernel_bound(key, avg_ms, work, peaks, tensor_path):
    """Roofline of one kernel: the resource whose ideal time is longest."""
    nbytes, flops = work["kernels"].get(key, (0, 0))
    t = avg_ms * 1e-3
    hbm_t = nbytes / (peaks["hbm_gbs"] * 1e9) if nbytes else 0.0
    if tensor_path:
        cpeak, cunit, cbound = peaks["bf16_tflops_sustained"], "TFLOP/s", "tensor"
    else:
        cpeak = SMS * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        cunit, cbound = "TFLOP/s", "alu"
    c_t = flops / (cpeak * 1e12) if flops else 0.0
    if hbm_t >= c_t:
        ach = nbytes / t / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes}
    ach = flops / t / 1e12
    return {"bound": cbound, "achieved": round(ach, 2), "peak": round(cpeak, 1), "unit": cunit,
            "frac": round(ach / cpeak, 4), "algorithmic_flops": flops}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- GPU arm

def run_llsa(args, ws, rank, local):
    import hierarchical_sparse_attention_mean_gb300 as llsa
    from hierarchical_sparse_attention_mean_gb300 import build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    w0 = synth.WORKLOADS[args.workload]
    # each rank: an independent problem of the same size (weak scaling)
    w = rank_workload(w0, rank)
    x = synth.make_inputs(w, threads=os.cpu_count() or 8)
    shape = (w.batch, w.heads, w.n, w.d)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {k: torch.from_numpy(v).to(td).reshape(shape).pin_memory() for k, v in x.items()}
    d = {k: v.to(dev) for k, v in host.items()}
    p = llsa.Params(w.batch, w.heads, w.n, w.d, block=w.block, topk=w.topk, dtype=w.dtype)
    s = llsa.get_sizes(p)
    b = llsa.Buffers(p, dev)
    dq, dk, dv = (torch.empty_like(d["q"]) for _ in range(3))
    stream = torch.cuda.current_stream(dev)

    def step():
        llsa.forward(p, d["q"], d["k"], d["v"], b)
        llsa.backward(p, d["q"], d["k"], d["v"], d["dout"], b, dq, dk, dv)

    forced = {"auto": 0, "grouped": llsa.LLSA_TEST_FORCE_GROUPED,
              "per_block": llsa.LLSA_TEST_FORCE_PER_BLOCK}[args.forward]
    if forced:
        llsa.test_set_wait_limit(0, forced)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if llsa.llsa_get_status() != 0:
        raise RuntimeError("device status set during warm-up")

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    # ---- per-kernel durations, from a profiled pass before the timed region:
    # events recorded between kernels keep each launch from overlapping the
    # drain of the one before, so the timed region brackets only the
    # dominant kernel with events
    n_prof = max(3, min(args.steps, 10))
    llsa.profile_reset()
    llsa.profile_only(None)
    llsa.profile_enable(True)
    for _ in range(n_prof):
        step()
    torch.cuda.synchronize()
    llsa.profile_enable(False)
    records = llsa.profile_read(cap=64 * n_prof + 64)
    per = {}
    for name, ms in records:
        k = kernel_key(name)
        tot, cnt = per.get(k, (0.0, 0))
        per[k] = (tot + ms, cnt + 1)
    stage_ms = {k: round(t / n_prof, 4) for k, (t, c) in per.items()}
    stage_each = {}  # stage -> per-step sums (every step launches the same kernels in order)
    if len(records) % n_prof == 0:
        per_step = len(records) // n_prof
        for k in range(n_prof):
            sums = {}
            for name, ms in records[k * per_step:(k + 1) * per_step]:
                key = kernel_key(name)
                sums[key] = sums.get(key, 0.0) + ms
            for key, v in sums.items():
                stage_each.setdefault(key, []).append(v)
    dom = max(per, key=lambda k: per[k][0])
    dom_names = sorted({name for name, _ in records if kernel_key(name) == dom})
    tensor_path = dom in llsa_tensor_kernels(records)

    # ---- timed region: K device-resident steps, events around the dominant
    # kernel's launches only
    sampler = ClockSampler(torch.cuda.current_device())
    llsa.profile_reset()
    llsa.profile_only(dom_names[0] if len(dom_names) == 1 else None)
    llsa.profile_enable(True)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    launches0 = llsa.llsa_launch_count()
    # an event at every step boundary: the first and last bracket the timed
    # region, the others give the spread of single steps
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    e0, e1 = marks[0], marks[-1]
    e0.record(stream)
    for k in range(args.steps):
        step()
        marks[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    launches = llsa.llsa_launch_count() - launches0
    llsa.profile_enable(False)
    llsa.profile_only(None)
    timed = [ms for name, ms in llsa.profile_read(cap=64 * args.steps + 64) if kernel_key(name) == dom]
    elapsed = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    ms_step = elapsed / args.steps
    step_each = [marks[k].elapsed_time(marks[k + 1]) for k in range(args.steps)]
    peaks, peak_src = load_peaks()
    work = work_model(w, s)
    # the dominant kernel's duration, live in the timed region
    avg_ms = sum(timed) / len(timed) if timed else per[dom][0] / per[dom][1]
    roof = kernel_bound(dom, avg_ms, work, peaks, tensor_path)
    traffic = args.traffic if args.traffic is not None else recorded_traffic(w.name, dom)
    roof.update({"kernel": dom, "avg_launch_ms": round(avg_ms, 4), "peak_source": peak_src,
                 "traffic": traffic, "traffic_source": "ncu dram bytes per launch, same sources" if traffic else None})

    # ---- end to end through host buffers: every step uploads its inputs from
    # pinned host memory and downloads its results (o, dq, dk, dv). Inputs and
    # outputs are double-buffered and the copies run on their own streams, so
    # step k computes while step k+1 uploads and step k-1 downloads.
    e2e_steps = max(3, min(args.steps, 50))
    hout = [{k: torch.empty(shape, dtype=td).pin_memory() for k in ("o", "dq", "dk", "dv")} for _ in range(2)]
    din = [d, {k: torch.empty_like(v) for k, v in d.items()}]
    bout = [(b, dq, dk, dv), (llsa.Buffers(p, dev),) + tuple(torch.empty_like(d["q"]) for _ in range(3))]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in hout[0].values())
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    barrier()
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(s_up)
    with torch.cuda.stream(s_up):
        for k in din[0]:
            din[0][k].copy_(host[k], non_blocking=True)
        in_ready[0].record(s_up)
    for it in range(e2e_steps):
        c = it & 1
        stream.wait_event(in_ready[c])
        if it >= 2:
            stream.wait_event(out_done[c])
        bb, gq, gk, gv = bout[c]
        x_ = din[c]
        llsa.forward(p, x_["q"], x_["k"], x_["v"], bb, stream=stream)
        llsa.backward(p, x_["q"], x_["k"], x_["v"], x_["dout"], bb, gq, gk, gv, stream=stream)
        comp_done[c].record(stream)
        if it + 1 < e2e_steps:
            n_ = (it + 1) & 1
            if it >= 1:
                s_up.wait_event(comp_done[n_])
            with torch.cuda.stream(s_up):
                for k in din[n_]:
                    din[n_][k].copy_(host[k], non_blocking=True)
                in_ready[n_].record(s_up)
        s_down.wait_event(comp_done[c])
        with torch.cuda.stream(s_down):
            hout[c]["o"].copy_(bb.o, non_blocking=True)
            hout[c]["dq"].copy_(gq, non_blocking=True)
            hout[c]["dk"].copy_(gk, non_blocking=True)
            hout[c]["dv"].copy_(gv, non_blocking=True)
            out_done[c].record(s_down)
    s_up.wait_stream(s_down)
    s_up.wait_stream(stream)
    e3.record(s_up)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e2.elapsed_time(e3) / e2e_steps, ws, dev)
    status = llsa.llsa_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    value = job_value(ws, work["step_flops"], ms_step)
    stage_gbs = {k: round(work["kernels"][k][0] / (stage_ms[k] * 1e-3) / 1e9, 1)
                 for k in ("pool_chunk", "transpose") if k in stage_ms and stage_ms[k] > 0}
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w0.name, "batch": w.batch, "heads": w.heads, "n": w.n, "d": w.d, "block": w.block,
                   "topk": w.topk, "levels": s.levels, "enrich_levels": s.enrich_levels,
                   "keys_per_query": s.keys_per_query, "inputs": f"{w.kind}, seed {w0.seed} (+7919 per rank)",
                   "l2": "no flush: the step's inputs (4 x %.0f MB) exceed the 129 MB L2" % (h2d / 4 / 1e6),
                   "parallelism": f"replicas{ws}", "step": "pool+select+fwd+transpose+bwd",
                   "forward": args.forward,
                   "flops_per_step": work["step_flops"], "flops_counted": "14*d per (query, key) pair: "
                   "fwd 4d, bwd 10d (S, dP, dV, dK, dQ); selection excluded"},
        "stage_ms": stage_ms,
        "stage_ms_from": f"{n_prof} profiled steps before the timed region (events around every launch)",
        "spread_ms": {"step": spread(step_each), **{k: spread(v) for k, v in stage_each.items()}},
        "stage_gbs": stage_gbs,
        "roofline": roof,
        "gather_intake": gather_intake(w, s, b, stage_ms, clocks, dev) if tensor_path else None,
        "e2e": {"value": round(job_value(ws, work["step_flops"], e2e_ms), 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1:
        out["reorder"] = reorder_rate(w, dev, peaks)
        out["routing_recall"] = routing_recall(p, b, w, dev)
        if not args.no_reorder:
            out["reorder_in_step"] = reorder_in_step(w, d, ms_step, dev)
    if rank == 0 and ws == 1 and not args.no_dense:
        out["dense_sdpa"] = dense_comparator(w, dev, ms_step)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, x, s)
    return out


def routing_recall(p, b, w, dev):
    """Share of the exhaustive level-1 Top-K (single-level full scoring of the
    level-1 tokens) that the hierarchical selection of the timed step keeps,
    over every query block of every slice, with the exhaustive kernel's time."""
    import hierarchical_sparse_attention_mean_gb300 as llsa
    T = llsa.get_sizes(p).n_blocks
    ex = torch.empty(w.bh, T, min(w.topk, T), dtype=torch.int32, device=dev)
    llsa.llsa_select_exhaustive(p, b.pyr, ex)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    llsa.llsa_select_exhaustive(p, b.pyr, ex)
    e1.record()
    torch.cuda.synchronize()
    return {"value": round(llsa.routing_recall(b.sel_idx, ex), 4), "exhaustive_ms": round(e0.elapsed_time(e1), 3),
            "what": "fraction of the exhaustive level-1 Top-K held by the hierarchical selection, all query blocks"}


def reorder_in_step(w, d, ms_tile_as_given, dev, steps: int = 50):
    """Index reordering inside the step (token_order "raster"): pool, the
    per-query-block forward, dQ and dK/dV read the raster tokens as 4 x 4
    patches and write o, dq, dk, dv back in raster order. Times, on the same
    tokens: the tile-order step on tokens permuted beforehand (the library's
    own choice of forward, and with the per-query-block forward, whose
    arithmetic the raster order repeats exactly), then the raster-order step,
    and reports the routing recall of the reordered step. Events around
    `steps` whole steps each."""
    import hierarchical_sparse_attention_mean_gb300 as llsa
    side = int(round(math.sqrt(w.n)))
    pr = llsa.Params(w.batch, w.heads, w.n, w.d, block=w.block, topk=w.topk, dtype=w.dtype, token_order="raster")
    try:
        llsa.get_sizes(pr)
    except llsa.LLSAError as e:
        return {"unavailable": f"raster token order: {e}"}
    pt = llsa.Params(w.batch, w.heads, w.n, w.d, block=w.block, topk=w.topk, dtype=w.dtype)
    tiled = {}
    for k, t in d.items():
        tiled[k] = torch.empty_like(t)
        llsa.llsa_reorder(pt, side, side, t, tiled[k])

    def timed(p, x, flags=0):
        b = llsa.Buffers(p, dev)
        g = [torch.empty_like(x["q"]) for _ in range(3)]

        def step():
            llsa.forward(p, x["q"], x["k"], x["v"], b)
            llsa.backward(p, x["q"], x["k"], x["v"], x["dout"], b, *g)

        llsa.test_set_wait_limit(0, flags)
        try:
            for _ in range(3):
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                step()
            e1.record()
            torch.cuda.synchronize()
        finally:
            llsa.test_set_wait_limit(0, 0)
        if llsa.llsa_get_status() != 0:
            raise RuntimeError("device status set in the reordered step")
        return e0.elapsed_time(e1) / steps, b

    ms_t, _ = timed(pt, tiled)
    ms_tp, _ = timed(pt, tiled, llsa.LLSA_TEST_FORCE_PER_BLOCK)
    ms_r, br = timed(pr, d)
    return {"ms_per_step_raster_order": round(ms_r, 4),
            "ms_per_step_prepermuted_per_block_forward": round(ms_tp, 4),
            "overhead": round(ms_r / ms_tp - 1.0, 4),
            "ms_per_step_prepermuted": round(ms_t, 4),
            "ms_per_step_as_given": round(ms_tile_as_given, 4),
            "routing_recall": routing_recall(pr, br, w, dev)["value"],
            "what": f"{steps} fwd+bwd steps each on the workload's raster tokens: raster order (reordering "
                    "inside the kernels; the per-query-block forward); the same tokens permuted beforehand, "
                    "tile order, with the per-query-block forward (identical arithmetic: overhead) and with "
                    "the library's choice of forward; as given = the headline step, blocks of 16 consecutive "
                    "raster tokens (no reordering)"}


def reorder_rate(w, dev, peaks):
    """Index reordering (hierarchical tile order) of one token tensor of the
    workload's shape, outside the step: HBM GB/s of `llsa_reorder`."""
    from hierarchical_sparse_attention_mean_gb300 import llsa_reorder, Params
    side, s = int(round(math.sqrt(w.n))), int(round(math.sqrt(w.block)))
    m = int(round(math.log(side) / math.log(s))) if side > 1 and s > 1 else 0
    if side * side != w.n or s * s != w.block or s ** m != side:
        return {"unavailable": "the tile order needs a square image of side s^m with B = s^2"}
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    p = Params(w.batch, w.heads, w.n, w.d, block=w.block, topk=w.topk, dtype=w.dtype)
    x = torch.randn(w.batch, w.heads, w.n, w.d, device=dev, dtype=td)
    y = torch.empty_like(x)
    for _ in range(3):
        llsa_reorder(p, side, side, x, y)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record()
    for i in range(reps):
        llsa_reorder(p, side, side, x, y, inverse=bool(i & 1))
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nbytes = 2 * x.numel() * x.element_size()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 3),
            "what": "one [batch, heads, N, d] tensor to the tile order and back, alternating, 20 launches"}


def dense_comparator(w, dev, llsa_ms):
    """Context, not a target: PyTorch's fused dense attention (scaled_dot_
    product_attention, flash / cuDNN / memory-efficient backends only) forward
    plus backward on the same shape and dtype, timed with CUDA events."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    import torch.nn.functional as F
    shape = (w.batch, w.heads, w.n, w.d)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev).manual_seed(11)
    q, k, v = (torch.randn(shape, device=dev, dtype=td, generator=g).requires_grad_(True) for _ in range(3))
    do = torch.randn(shape, device=dev, dtype=td, generator=g)
    backends = [SDPBackend.FLASH_ATTENTION, SDPBackend.CUDNN_ATTENTION, SDPBackend.EFFICIENT_ATTENTION]
    try:
        with sdpa_kernel(backends):
            def step():
                o = F.scaled_dot_product_attention(q, k, v)
                o.backward(do)
            for _ in range(2):
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 3
            e0.record()
            for _ in range(reps):
                step()
            e1.record()
            torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
    except RuntimeError as err:  # no fused backend for this shape / device
        return {"unavailable": str(err).splitlines()[0][:160]}
    flops = 14 * w.d * w.batch * w.heads * w.n * w.n
    return {"ms_per_step": round(ms, 3), "value": round(flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "flops_per_step": flops, "flops_counted": "14*d per (query, key) pair over all N^2 pairs",
            "llsa_speedup": round(ms / llsa_ms, 2),
            "what": "torch scaled_dot_product_attention fwd+bwd, dense, same shape and dtype, random inputs"}


# Throughput across the method's hyperparameters on the same inputs (the
# pages' ablations vary K, B, L and L_e; only the step time is measured here):
# (label, B, K, L (0: floor(log_B N - 1)), L_e (-1: all levels)[, enrichment rule])
SWEEP = [
    ("B16-K8", 16, 8, 0, -1),
    ("B16-K4", 16, 4, 0, -1),
    ("B16-K16", 16, 16, 0, -1),
    ("B16-K32", 16, 32, 0, -1),
    ("B8-K8", 8, 8, 0, -1),
    ("B32-K8", 32, 8, 0, -1),
    ("B64-K8", 64, 8, 0, -1),
    ("B16-K8-L2", 16, 8, 2, -1),
    ("B16-K8-L1", 16, 8, 1, -1),
    ("B16-K8-Le0", 16, 8, 0, 0),
    ("B16-K8-Le1", 16, 8, 0, 1),
    ("B16-K8-Le2", 16, 8, 0, 2),
    ("B16-K8-ancestor", 16, 8, 0, -1, "ancestor"),
    ("B16-K8-allk", 16, 8, 0, -1, "allk"),
]


def run_sweep(args):
    """One JSON line: ms per fwd+bwd step for each SWEEP entry on the
    workload's inputs, with the effective TFLOP/s (14 d per (query, key) pair)
    and whether the attention kernels ran on the tensor cores."""
    import dataclasses
    import hierarchical_sparse_attention_mean_gb300 as llsa
    from hierarchical_sparse_attention_mean_gb300 import build

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    w0 = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w0, threads=os.cpu_count() or 8)
    shape = (w0.batch, w0.heads, w0.n, w0.d)
    td = torch.bfloat16 if w0.dtype == "bf16" else torch.float32
    d = {k: torch.from_numpy(v).to(td).reshape(shape).to(dev) for k, v in x.items()}
    rows = []
    for label, B, K, L, Le, *rule in SWEEP:
        p = llsa.Params(w0.batch, w0.heads, w0.n, w0.d, block=B, topk=K, levels=L, enrich_levels=Le, dtype=w0.dtype,
                        enrich_rule=rule[0] if rule else "top1")
        try:
            s = llsa.get_sizes(p)
            b = llsa.Buffers(p, dev)
            dq, dk, dv = (torch.empty_like(d["q"]) for _ in range(3))

            def step():
                llsa.forward(p, d["q"], d["k"], d["v"], b)
                llsa.backward(p, d["q"], d["k"], d["v"], d["dout"], b, dq, dk, dv)

            for _ in range(3):
                step()
            torch.cuda.synchronize()
            llsa.profile_reset()
            llsa.profile_enable(True)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.sweep_steps):
                step()
            e1.record()
            torch.cuda.synchronize()
            llsa.profile_enable(False)
            records = llsa.profile_read(cap=64 * args.sweep_steps + 64)
            if llsa.llsa_get_status() != 0:
                raise RuntimeError("device status set")
        except (llsa.LLSAError, RuntimeError) as e:
            rows.append({"config": label, "unavailable": str(e)})
            continue
        ms = e0.elapsed_time(e1) / args.sweep_steps
        work = work_model(dataclasses.replace(w0, block=B, topk=K), s)
        tc = sorted(llsa_tensor_kernels(records))
        rows.append({"config": label, "block": B, "topk": K, "levels": s.levels, "enrich_levels": s.enrich_levels,
                     "enrich_rule": p.enrich_rule, "keys_per_query": s.keys_per_query, "ms_per_step": round(ms, 4),
                     "tflops": round(work["step_flops"] / (ms * 1e-3) / 1e12, 2),
                     "attention": "tensor cores (" + ", ".join(tc) + ")" if tc else "CUDA cores"})
        del b, dq, dk, dv
    return {"metric": "LLSA fwd+bwd ms per step across B, K, L and L_e", "unit": "ms", "n_gpus": 1,
            "steps": args.sweep_steps, "warmup": 3, "dtype": w0.dtype, "data": "synthetic",
            "config": {"workload": w0.name}, "sweep": rows}


def llsa_tensor_kernels(records):
    return {kernel_key(n) for n, _ in records if n.endswith("_tc") or n.startswith("fwd_grp")}


def cpu_baseline(w, x, s):
    """The oracle as it stands, the whole path on one slice per host thread."""
    import oracle
    oracle.build()
    n_sl = max(1, min(os.cpu_count() or 1, w.bh))
    t0 = time.perf_counter()
    oracle.run(x["q"][:n_sl], x["k"][:n_sl], x["v"][:n_sl], x["dout"][:n_sl], B=w.block, K=w.topk, threads=n_sl)
    wall = time.perf_counter() - t0
    flops = 14 * w.d * n_sl * w.n * s.keys_per_query
    return {"value": round(flops / wall / 1e12, 6), "unit": "TFLOP/s", "cores": n_sl, "kind": "oracle",
            "wall_s": round(wall, 2),
            "sample": f"whole path (pool, select, fwd, transpose, bwd) of {n_sl} of {w.bh} (batch, head) slices, "
                      "one oracle thread per slice, fp64"}


# --------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle timed as it stands, on a bounded sample of the same
    workload: pooling, selection and the forward of slice 0 are prepared once;
    each step then runs the oracle forward and backward (dq of R query tokens,
    dk/dv of R/B key blocks), R sized so the whole run stays within minutes."""
    import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    x = synth.make_slice(w, 0)
    B, K, d, n = w.block, w.topk, w.d, w.n
    L = oracle.num_levels(n, B)
    scale = 1.0 / math.sqrt(d)
    qp, kp, vp = (oracle.pool(x[t], B, L) for t in ("q", "k", "v"))
    sel = oracle.select_all(qp, kp, n, B, L, K)
    I1, coarse = sel["levels"][1], sel["coarse"]
    o, lse = oracle.fwd(x["q"], x["k"], x["v"], kp, vp, B, L, L, I1, coarse, scale)
    kpq = I1.shape[1] * B + L

    def one(start, R):
        rows = (np.arange(R) + start) % n
        blocks = (np.arange(R // B) + start // B) % (n // B)
        oracle.fwd(x["q"], x["k"], x["v"], kp, vp, B, L, L, I1, coarse, scale, qlist=rows)
        oracle.bwd_dq_rows(x["q"], x["k"], x["v"], kp, vp, o[rows], lse[rows], x["dout"], B, L, L, I1, coarse,
                           scale, rows)
        oracle.bwd_dkv_blocks(x["q"], x["k"], x["v"], kp, vp, o, lse, x["dout"], B, L, L, I1, coarse, scale,
                              blocks)

    budget_s = min(1.0, 100.0 / max(1, args.steps + args.warmup))
    R = 256
    t0 = time.perf_counter()
    one(0, R)
    dt = time.perf_counter() - t0
    R = int(max(B, min(n, R * budget_s / max(dt, 1e-6))) // B * B)
    for i in range(args.warmup):
        one(i * R, R)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one((args.warmup + i) * R, R)
    wall = time.perf_counter() - t0
    ms = wall / args.steps * 1e3
    value = 14 * d * R * kpq / (ms * 1e-3) / 1e12
    sample = (f"per step: oracle fwd + dq of {R} query tokens and dk/dv of {R // B} key blocks of slice 0 "
              f"(pool/select/fwd of that slice prepared before timing); 14*d FLOPs per (query, key) pair")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "n": n, "d": d, "block": B,
                       "topk": K, "levels": L},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["llsa", "reference"], default="llsa")
    ap.add_argument("--workload", default=synth.HEADLINE, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-attention comparator")
    ap.add_argument("--no-reorder", action="store_true", help="skip the index-reordering steps after the timed region")
    ap.add_argument("--forward", choices=["auto", "grouped", "per_block"], default="auto",
                    help="which tensor-core forward runs: the library's choice per call (default), or one of the "
                         "two forced (for comparing them; both compute the same outputs)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture of this build")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: one line of step times across B, K, L and L_e")
    ap.add_argument("--sweep-steps", type=int, default=10)
    args = ap.parse_args()
    if args.sweep:
        print(json.dumps(run_sweep(args)), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    try:
        out = run_llsa(args, ws, rank, local)
        if rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
