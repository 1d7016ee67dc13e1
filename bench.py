"""Benchmark of the relative-bias paged attention hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload local_decode|global_decode|chunked_prefill|decode_66_layers]
                    [--no-cpu-baseline] [--extra]

Prints ONE JSON line (rank 0).  The default workload is the local-layer decode
batch (B=64, 48/16 heads, D=128, page 64, lengths uniform in [1024, 8192],
window 512, R=512): one step = one decode call over the whole batch, inputs
resident in HBM; L2 reuse between steps is defeated by rotating through input
sets whose visible K/V together exceed the 129 MB L2.  The timed region is a
CUDA-graph replay of exactly K steps bracketed by events (and, for N > 1, a
barrier with the max over ranks); ranks are independent replicas (the path
has no exchange step), so scaling is weak.

``--impl reference`` times the CPU fp64 oracle instead (on this host's cores,
rank 0 only, each step a bounded sample of the same workload).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "rel-bias paged attn: decode KV GB/s (% of HBM peak); prefill TFLOP/s"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# environment helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str, src_paths):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(f"{kernel}:{workload}")
    if not rec or rec.get("source_hash") != source_hash(src_paths):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# decode workload accounting

def decode_bytes(inp):
    """Algorithmic bytes of one decode call: visible K+V rows, plus q, out and
    the bias entries of visible distances (each read once)."""
    L = inp.seq_lens.cpu().long()
    vis = torch.clamp(L, max=inp.window) if inp.window > 0 else L
    vis_keys = int(vis.sum())
    kv = vis_keys * inp.H_kv * inp.D * 2 * 2
    q_out = inp.B * inp.H_q * inp.D * 2 * 2
    bias = int(torch.clamp(vis, max=inp.R).sum()) * inp.H_q * 4
    lse = inp.B * inp.H_q * 4
    return kv, kv + q_out + bias + lse


# ---------------------------------------------------------------------------
# our arm

def bench_decode(args, device, rank):
    import paged_attention_relative_attn_gb300 as ira
    name = args.workload
    sets = []
    n_sets = 0
    kv_bytes = total_bytes = None
    while True:
        inp = W.make_decode_config(name, device=device, seed=n_sets, batch=args.batch)
        kvb, totb = decode_bytes(inp)
        sets.append(inp)
        n_sets += 1
        kv_bytes = kvb if kv_bytes is None else kv_bytes
        if args.sets is not None:
            if n_sets >= args.sets:
                break
        # rotate until the distinct visible K/V of one rotation exceeds 2x L2
        elif n_sets >= 3 and sum(decode_bytes(s)[0] for s in sets) > 2 * L2_BYTES:
            break
    per_set = [decode_bytes(s) for s in sets]
    B, H_q, H_kv, D = sets[0].B, sets[0].H_q, sets[0].H_kv, sets[0].D
    S = ira.choose_splits(B, H_kv, sets[0].window, sets[0].max_seq_len,
                          torch.cuda.get_device_properties(device).multi_processor_count)
    ws_bytes = ira.decode_workspace_bytes(B, H_q, H_kv, D, sets[0].window, sets[0].max_seq_len)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    outs = [torch.empty_like(s.q) for s in sets]
    lses = [torch.empty((B, H_q), dtype=torch.float32, device=device) for s in sets]

    def step(i, stream=None):
        s = sets[i % n_sets]
        ira.decode_inputs(s, out=outs[i % n_sets], lse=lses[i % n_sets], workspace=ws,
                          stream=stream)

    # warm-up (eager)
    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()

    K = args.steps
    g_len = min(K, 60 * n_sets // math.gcd(60, n_sets))  # whole rotations per graph
    g_len = max(1, min(g_len, K))
    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream())

    def make_graph(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(n):
                    step(i, stream=cap)
        return g

    g_main = make_graph(g_len)
    reps, rem = divmod(K, g_len)
    g_rem = make_graph(rem) if rem else None
    torch.cuda.synchronize()
    g_main.replay()  # one more warm-up pass through the graph
    torch.cuda.synchronize()

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(args)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(cap):
            ev0.record(cap)
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(cap)
        torch.cuda.synchronize()
    barrier(args)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(args, ms)

    # bytes of exactly the K steps that ran (rotation order i % n_sets)
    kv_total = sum(per_set[i % n_sets][0] for i in range(K))
    all_total = sum(per_set[i % n_sets][1] for i in range(K))
    launches_per_step = 1 + (1 if S > 1 else 0)

    res = dict(ms=ms, kv_total=kv_total, all_total=all_total, K=K, S=S, n_sets=n_sets,
               launches=K * launches_per_step, clocks=clk.summary(), sets=sets, outs=outs,
               lses=lses, ws=ws, kv_per_step=sum(p[0] for p in per_set) / n_sets,
               total_per_step=sum(p[1] for p in per_set) / n_sets)
    return res


def bench_decode_e2e(args, device, sets, ws):
    """Same metric through the public API with host buffers: every step copies
    its per-step inputs (q, rel_logits, page_table, seq_lens) from pinned host
    memory, runs decode and reads out + lse back.  The paged K/V cache is the
    model's resident state and stays in HBM."""
    import paged_attention_relative_attn_gb300 as ira
    host = []
    for s in sets:
        host.append(dict(q=s.q.cpu().pin_memory(), rel=s.rel_logits.cpu().pin_memory(),
                         pt=s.page_table.cpu().pin_memory(), sl=s.seq_lens.cpu().pin_memory()))
    dq = torch.empty_like(sets[0].q)
    drel = torch.empty_like(sets[0].rel_logits)
    dpt = torch.empty_like(sets[0].page_table)
    dsl = torch.empty_like(sets[0].seq_lens)
    out = torch.empty_like(sets[0].q)
    lse = torch.empty(sets[0].q.shape[:2], dtype=torch.float32, device=device)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = (host[0]["q"].numel() * 2 + host[0]["rel"].numel() * 4 + host[0]["pt"].numel() * 4 +
           host[0]["sl"].numel() * 4)
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    n = len(sets)

    def step(i):
        h = host[i % n]
        s = sets[i % n]
        dq.copy_(h["q"], non_blocking=True)
        drel.copy_(h["rel"], non_blocking=True)
        dpt.copy_(h["pt"], non_blocking=True)
        dsl.copy_(h["sl"], non_blocking=True)
        ira.decode(dq, s.k_cache, s.v_cache, dpt, dsl, drel, window=s.window, scale=s.scale,
                   max_seq_len=s.max_seq_len, out=out, lse=lse, workspace=ws)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    K = max(30, min(args.steps, 300))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record()
    for i in range(K):
        step(i)
    ev1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(ev0.elapsed_time(ev1), wall * 1e3)
    kv = sum(decode_bytes(sets[i % n])[0] for i in range(K))
    return dict(value=kv / (ms * 1e-3) / 1e9, unit="GB/s", h2d_bytes_per_step=h2d,
                d2h_bytes_per_step=d2h, steps=K)


# ---------------------------------------------------------------------------
# oracle timing

def oracle_units(inp, budget_s, max_units=None):
    """Time the oracle, as it stands, on (sequence, KV-head group) units of a
    decode batch until ~budget_s of CPU work (at least one unit).  Only the
    pages a unit uses are copied to the host.  Returns (GB/s of visible K+V,
    units done, seconds)."""
    from oracle.ref import ref_decode
    P = inp.page_size
    G = inp.H_q // inp.H_kv
    done_bytes = 0
    t_used = 0.0
    n = 0
    total = inp.B * inp.H_kv
    for u in range(total):
        b, hk = divmod(u, inp.H_kv)
        L = int(inp.seq_lens[b])
        npg = (L + P - 1) // P
        ids = inp.page_table[b, :npg].long()
        kc = inp.k_cache.index_select(0, ids)[:, :, hk:hk + 1].float().cpu().numpy().astype(np.float64)
        vc = inp.v_cache.index_select(0, ids)[:, :, hk:hk + 1].float().cpu().numpy().astype(np.float64)
        pt = np.arange(npg, dtype=np.int64)[None, :]
        q = inp.q[b:b + 1, hk * G:(hk + 1) * G].float().cpu().numpy().astype(np.float64)
        rel = inp.rel_logits[b:b + 1, hk * G:(hk + 1) * G].float().cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        ref_decode(q, kc, vc, pt, np.array([L]), rel, inp.window, inp.scale)
        t_used += time.perf_counter() - t0
        vis = min(L, inp.window) if inp.window > 0 else L
        done_bytes += vis * inp.D * 2 * 2
        n += 1
        if t_used >= budget_s or (max_units and n >= max_units):
            break
    return done_bytes / t_used / 1e9, n, t_used


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(int(x.get("num_threads", 1)) for x in info)
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# distributed helpers

def barrier(args):
    if args.world > 1:
        torch.distributed.barrier()


def max_over_ranks(args, x):
    if args.world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=f"cuda:{args.local}")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(args, x):
    if args.world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=f"cuda:{args.local}")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------

def run_reference(args):
    """The oracle arm: rank 0 only, on host cores.  Each step is a bounded
    sample of (sequence, KV-head) units of the workload, sized so the whole
    run stays within a few minutes."""
    if args.rank != 0:
        return
    n_seq = 4
    inp = W.make_decode_config(args.workload, device="cpu", seed=0, batch=n_seq)
    per_step = min(args.ref_budget, max(0.002, 150.0 / max(1, args.steps + args.warmup)))
    vals = []
    units = 0
    for i in range(args.warmup + args.steps):
        gbs, n, _ = oracle_units(inp, per_step)
        if i >= args.warmup:
            vals.append(gbs)
            units += n
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": f"per step: (sequence, KV head) units of the first "
                                       f"{n_seq} sequences of {args.workload}, ~{per_step:.3f} s "
                                       f"of fp64 oracle time; {units} units timed"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="local_decode",
                    choices=["local_decode", "global_decode"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=5.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first sequences (profiling of a smaller case)")
    ap.add_argument("--sets", type=int, default=None, help="number of rotated input sets")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    args.world, args.rank, args.local = dist_env()

    if args.impl == "reference":
        run_reference(args)
        return

    if args.world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(args.local)
    device = torch.device(f"cuda:{args.local}")

    # the C-ABI library must be built; fail loudly if not
    from paged_attention_relative_attn_gb300 import _lib
    _lib.load()

    pk = peaks()
    r = bench_decode(args, device, args.rank)
    if args.no_e2e:
        e2e = None
    else:
        e2e = bench_decode_e2e(args, device, r["sets"], r["ws"])
        e2e["value"] = sum_over_ranks(args, e2e["value"])
    ms = r["ms"]
    kv_total = sum_over_ranks(args, r["kv_total"])
    value = kv_total / (ms * 1e-3) / 1e9
    # dominant kernel: the decode kernel (one launch per step when S == 1)
    per_launch_ms = ms / r["K"]
    achieved = r["total_per_step"] / (per_launch_ms * 1e-3) / 1e9
    traffic = traffic_record("decode_kernel", args.workload,
                             ["paged_attention_relative_attn_gb300/csrc/decode.cu",
                              "paged_attention_relative_attn_gb300/csrc/ptx.cuh"])
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": r["sets"][0].B,
                   "heads": f"{r['sets'][0].H_q}/{r['sets'][0].H_kv}", "head_dim": r["sets"][0].D,
                   "page_size": r["sets"][0].page_size, "window": r["sets"][0].window,
                   "R": r["sets"][0].R, "num_splits": r["S"],
                   "l2": f"rotating {r['n_sets']} input sets, {r['kv_per_step'] * r['n_sets'] / 1e6:.0f} MB "
                         f"of visible K/V per rotation (L2 129 MB)",
                   "parallelism": f"replicas x{args.world}", "timing": "CUDA graph replay, events"},
        "clocks": r["clocks"],
        "e2e": e2e,
        "gpu_launches": r["launches"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "peak_source": f"{pk['source']} hbm_gbs",
                     "kv_frac": value / args.world / pk["hbm_gbs"]},
    }
    if args.rank == 0 and not args.no_cpu_baseline:
        gbs, n, t = oracle_units(r["sets"][0], args.cpu_budget)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"{n} (sequence, KV head) units of {args.workload} "
                                          f"(first of {r['sets'][0].B * r['sets'][0].H_kv}), "
                                          f"{t:.1f} s of fp64 oracle time"}
    if args.rank == 0:
        print(json.dumps(line), flush=True)
    if args.world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
