"""Benchmark of the relative-bias paged attention hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload local_decode|global_decode|chunked_prefill|global_prefill|
                                kv_append|kv_conv_append|mtp_decode|decode_66_layers]
                    [--no-cpu-baseline] [--no-e2e] [--no-extra] [--batch B] [--sets S]

Prints ONE JSON line (rank 0).  The default workload is the local-layer decode
batch (B=64, 48/16 heads, D=128, page 64, lengths uniform in [1024, 8192],
window 512, R=512): one step = one decode call over the whole batch, inputs
resident in HBM; L2 reuse between steps is defeated by rotating through input
sets whose visible K/V together exceed the 129 MB L2.  The timed region is a
CUDA-graph replay of exactly K steps bracketed by events (and, for N > 1, a
barrier with the max over ranks); ranks are independent replicas (the path
has no exchange step), so scaling is weak.

With the default workload the line also carries the other workloads (each
with its own roofline) under ``extra_workloads`` unless ``--no-extra``.

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
BUSY_WINDOW_S = 0.15  # untimed load before and after the timed region (clock samples)


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

    def wait_first(self, timeout_s=5.0):
        """Block until nvidia-smi has printed its first sample (it takes a
        moment to start), so that samples cover what runs next."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.01)

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


def strip_c_comments(text: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed, so
    that an edit to comments or layout alone leaves the code's hash as is.
    String and character literals are kept verbatim."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(paths):
    """Hash of the kernel's sources, comments and layout excluded."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(strip_c_comments(f.read()).encode())
        h.update(b"\0")
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

def time_steps(args, device, step, K, warmup, per_graph):
    """Warm up eagerly, capture `per_graph` consecutive steps in a CUDA graph,
    then time exactly K steps (graph replays + a remainder graph) with events
    on the capture stream while nvidia-smi samples the clocks.  Returns
    (ms for the K steps, clock summary)."""
    for i in range(max(warmup, 3)):
        step(i, None)
    torch.cuda.synchronize()
    g_len = max(1, min(K, per_graph))
    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream())

    def make_graph(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(n):
                    step(i, cap)
        return g

    g_main = make_graph(g_len)
    reps, rem = divmod(K, g_len)
    g_rem = make_graph(rem) if rem else None
    torch.cuda.synchronize()
    g_main.replay()  # one more warm-up pass through the graph
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def keep_busy(seconds):
        # untimed replays of the same graph, so that the clock samples taken
        # around a short timed region still see the GPU under this load
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            with torch.cuda.stream(cap):
                g_main.replay()
            torch.cuda.synchronize()

    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.wait_first()
        keep_busy(BUSY_WINDOW_S)
        barrier(args)
        torch.cuda.synchronize()
        with torch.cuda.stream(cap):
            ev0.record(cap)
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(cap)
        torch.cuda.synchronize()
        barrier(args)
        keep_busy(BUSY_WINDOW_S)
    ms = max_over_ranks(args, ev0.elapsed_time(ev1))
    summary = clk.summary()
    summary["window"] = (f"nvidia-smi every 50 ms over the timed region plus {BUSY_WINDOW_S:.2f} s "
                         f"of untimed replays of the same steps before and after it")
    return ms, summary


def decode_rotation(name, batch=None, n_sets=None):
    """Visible K+V bytes of each input set the decode bench rotates through:
    sets are added (seed = set index) until one rotation's visible K/V exceeds
    2 x L2, at least 3, or exactly ``n_sets``.  Only the drawn lengths matter,
    so both arms compute it without building the inputs."""
    c = W.DECODE_CONFIGS[name]
    lo, hi = c["len_range"]
    per = []
    while True:
        lens = W.draw_uniform_lengths(c["B"], lo, hi, len(per))
        if batch is not None:
            lens = lens[:batch]
        vis = [min(L, c["window"]) if c["window"] > 0 else L for L in lens]
        per.append(sum(vis) * c["H_kv"] * c["D"] * 2 * 2)
        if n_sets is not None:
            if len(per) >= n_sets:
                break
        elif len(per) >= 3 and sum(per) > 2 * L2_BYTES:
            break
    return per


def decode_workload_config(args, name):
    """The description of a decode workload, identical in both arms."""
    c = W.DECODE_CONFIGS[name]
    B = c["B"] if args.batch is None else args.batch
    lens = c.get("len_range")
    per = decode_rotation(name, args.batch, args.sets)
    return {"workload": name, "batch": B, "heads": f"{c['H_q']}/{c['H_kv']}", "head_dim": c["D"],
            "page_size": c["P"], "window": c["window"], "R": c["R"],
            "lengths": f"uniform [{lens[0]}, {lens[1]}]" if lens else "fixed",
            "l2": f"rotating {len(per)} input sets, {sum(per) / 1e6:.0f} MB of visible K/V per "
                  f"rotation (L2 129 MB)",
            "parallelism": f"replicas x{args.world}"}


def bench_decode(args, device, name, K, warmup):
    import paged_attention_relative_attn_gb300 as ira
    # rotate until the distinct visible K/V of one rotation exceeds 2x L2
    n_sets = len(decode_rotation(name, args.batch, args.sets))
    sets = [W.make_decode_config(name, device=device, seed=i, batch=args.batch)
            for i in range(n_sets)]
    per_set = [decode_bytes(x) for x in sets]
    B, H_q, H_kv, D = sets[0].B, sets[0].H_q, sets[0].H_kv, sets[0].D
    S = ira.choose_splits(B, H_kv, sets[0].window, sets[0].max_seq_len,
                          torch.cuda.get_device_properties(device).multi_processor_count)
    ws_bytes = ira.decode_workspace_bytes(B, H_q, H_kv, D, sets[0].window, sets[0].max_seq_len)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    outs = [torch.empty_like(x.q) for x in sets]
    lses = [torch.empty((B, H_q), dtype=torch.float32, device=device) for x in sets]

    def step(i, stream):
        x = sets[i % n_sets]
        ira.decode_inputs(x, out=outs[i % n_sets], lse=lses[i % n_sets], workspace=ws,
                          stream=stream)

    ms, clocks = time_steps(args, device, step, K, warmup, 60 * n_sets // math.gcd(60, n_sets))
    kv_total = sum(per_set[i % n_sets][0] for i in range(K))
    all_total = sum(per_set[i % n_sets][1] for i in range(K))
    launches = K * (1 + (1 if S > 1 else 0))
    config = decode_workload_config(args, name)
    assert config["l2"].startswith(f"rotating {n_sets} ")
    return dict(ms=ms, K=K, clocks=clocks, launches=launches, config=config, sets=sets, ws=ws,
                units_total=kv_total, bytes_total=all_total, kernel="decode_kernel",
                kernel_launches=K, unit="GB/s", launch={"num_splits": S})


def prefill_work(inp, window):
    """Algorithmic work of one prefill call: MMA flops over visible (query,
    key) pairs and bytes (the bias entries a row needs -- min(visible, R), as
    distances past the table share its last column -- q, out, K/V of the key
    range)."""
    cu = inp.cu_seqlens_q.cpu().tolist()
    sl = inp.seq_lens.cpu().tolist()
    pairs = 0
    bias_entries = 0
    kv_keys = 0
    for b in range(inp.B):
        n = cu[b + 1] - cu[b]
        L = sl[b]
        if n == 0:
            continue
        pos = torch.arange(L - n, L, dtype=torch.int64)
        vis = torch.clamp(pos + 1, max=window) if window > 0 else pos + 1
        pairs += int(vis.sum())
        bias_entries += int(torch.clamp(vis, max=inp.R).sum())
        lo = max(0, L - n - window + 1) if window > 0 else 0
        kv_keys += L - lo
    flops = 4 * inp.D * pairs * inp.H_q
    bias = bias_entries * inp.H_q * 4
    qo = inp.T * inp.H_q * inp.D * 2 * 2
    kv = kv_keys * inp.H_kv * inp.D * 2 * 2
    return flops, bias + qo + kv + inp.T * inp.H_q * 4


PREFILL_WORKLOADS = {"chunked_prefill": W.CHUNKED_PREFILL, "global_prefill": W.GLOBAL_PREFILL}


def bench_prefill(args, device, K, warmup, name="chunked_prefill"):
    """One step = the whole chunked prefill: 4 calls, each 4 sequences x 2048
    new tokens against the cached prefix (positions 2048c .. 2048c+2047).
    chunked_prefill is a local layer (window 512, R = 512; bound by the bias
    stream), global_prefill a global layer (full causal, R = 1024; bound by
    the tensor cores)."""
    import paged_attention_relative_attn_gb300 as ira
    cfg = PREFILL_WORKLOADS[name]
    chunks = []
    cache = None
    for c in range(4):
        inp, cache = W.make_chunked_prefill(c, device=device, seed=0, cache=cache,
                                            n_seqs=args.batch, cfg=cfg)
        chunks.append(inp)
    work = [prefill_work(x, x.window) for x in chunks]
    outs = [torch.empty_like(x.q) for x in chunks]
    lses = [torch.empty(x.q.shape[:2], dtype=torch.float32, device=device) for x in chunks]

    def step(i, stream):
        for c, x in enumerate(chunks):
            ira.prefill_inputs(x, out=outs[c], lse=lses[c], stream=stream)

    ms, clocks = time_steps(args, device, step, K, warmup, 10)
    flops = K * sum(w[0] for w in work)
    nbytes = K * sum(w[1] for w in work)
    x0 = chunks[0]
    config = {"workload": name, "sequences": x0.B, "seq_len": cfg["seq_len"],
              "chunk": cfg["chunk"], "tokens_per_call": x0.T, "heads": f"{x0.H_q}/{x0.H_kv}",
              "head_dim": x0.D, "window": x0.window, "R": x0.R, "page_size": x0.page_size,
              "l2": f"{x0.T * x0.H_q * x0.R * 4 / 1e6:.0f} MB of rel_logits per call (L2 129 MB)"}
    return dict(ms=ms, K=K, clocks=clocks, launches=4 * K, config=config, units_total=flops,
                bytes_total=nbytes, kernel="prefill_kernel", kernel_launches=4 * K, unit="TFLOP/s",
                bound="tensor" if name == "global_prefill" else "hbm")


MTP_DECODE = dict(B=64, q_len=4, H_q=48, H_kv=16, D=128, P=64, window=512, R=512,
                  len_range=(1024, 8192))


def bench_decode_multi(args, device, K, warmup):
    """One step = one multi-token decode call on a local layer: 64 sequences
    x 4 new tokens (3 draft tokens + 1), lengths uniform in [1024, 8192], window
    512, R = 512.  Metric: K/V bytes of each (sequence, KV head)'s visible keys
    -- the union over its 4 tokens, min(L, 512 + 3) keys, read once -- per
    second.  Input sets rotate until one rotation's visible K/V exceeds 2 x L2."""
    import paged_attention_relative_attn_gb300 as ira
    c = MTP_DECODE
    B = c["B"] if args.batch is None else args.batch
    sets = []
    while True:
        lens = W.draw_uniform_lengths(c["B"], *c["len_range"], len(sets))[:B]
        cache = W.make_prefill_cache(lens, c["H_kv"], c["D"], c["P"], device=device,
                                     seed=len(sets))
        sets.append(W.make_prefill(cache, [c["q_len"]] * B, lens, c["H_q"], c["R"], c["window"],
                                   device=device, seed=len(sets) + 1,
                                   max_seq_len=c["len_range"][1]))
        kv_rot = sum(multi_decode_bytes(x, c["q_len"])[0] for x in sets)
        if args.sets is not None:
            if len(sets) >= args.sets:
                break
        elif len(sets) >= 3 and kv_rot > 2 * L2_BYTES:
            break
    n = len(sets)
    per = [multi_decode_bytes(x, c["q_len"]) for x in sets]
    x0 = sets[0]
    ws_bytes = ira.decode_multi_workspace_bytes(B, c["q_len"], c["H_q"], c["H_kv"], c["D"],
                                                c["window"], x0.max_seq_len)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    outs = [torch.empty_like(x.q) for x in sets]
    lses = [torch.empty(x.q.shape[:2], dtype=torch.float32, device=device) for x in sets]

    def step(i, stream):
        x = sets[i % n]
        ira.decode_multi(x.q, x.k_cache, x.v_cache, x.page_table, x.seq_lens, x.rel_logits,
                         q_len=c["q_len"], window=x.window, scale=x.scale,
                         max_seq_len=x.max_seq_len, out=outs[i % n], lse=lses[i % n],
                         workspace=ws, stream=stream)

    ms, clocks = time_steps(args, device, step, K, warmup, 60 * n // math.gcd(60, n))
    config = {"workload": "mtp_decode", "batch": B, "q_len": c["q_len"],
              "heads": f"{c['H_q']}/{c['H_kv']}", "head_dim": c["D"], "page_size": c["P"],
              "window": c["window"], "R": c["R"],
              "l2": f"rotating {n} input sets, {sum(p[0] for p in per) / 1e6:.0f} MB of visible "
                    f"K/V per rotation (L2 129 MB)"}
    return dict(ms=ms, K=K, clocks=clocks, launches=K, config=config,
                units_total=sum(per[i % n][0] for i in range(K)),
                bytes_total=sum(per[i % n][1] for i in range(K)), kernel="decode_kernel",
                kernel_launches=K, unit="GB/s")


def multi_decode_bytes(inp, q_len):
    """(visible K/V bytes, all algorithmic bytes) of one multi-token decode
    call: per (sequence, KV head) the union of its tokens' visible keys (read
    once), plus q, out, lse and the bias entries of every row's visible keys."""
    L = inp.seq_lens.cpu().long()
    W_ = inp.window
    keys = torch.clamp(L, max=W_ + q_len - 1) if W_ > 0 else L
    kv = int(keys.sum()) * inp.H_kv * inp.D * 2 * 2
    T = inp.T
    q_out = T * inp.H_q * inp.D * 2 * 2
    bias = 0
    for i in range(q_len):
        vis = L - q_len + i + 1
        vis = torch.clamp(vis, max=W_) if W_ > 0 else vis
        bias += int(torch.clamp(vis, max=inp.R).sum()) * inp.H_q * 4
    return kv, kv + q_out + bias + T * inp.H_q * 4


def bench_kv_append(args, device, K, warmup):
    """One step = the KV append of one chunked-prefill call: 4 sequences x 2048
    new tokens (16 KV heads, D = 128, pages of 64) written at positions
    2048c .. 2048c + 2047, c cycling over the four calls, so consecutive steps
    write different cache slots from different inputs (4 x 134 MB per
    rotation, L2 129 MB).  Bytes: every new K and V row read once and written
    once."""
    import paged_attention_relative_attn_gb300 as ira
    cfg = W.CHUNKED_PREFILL
    n = cfg["n_seqs"] if args.batch is None else args.batch
    chunk, L = cfg["chunk"], cfg["seq_len"]
    cache = W.make_prefill_cache([L] * n, cfg["H_kv"], cfg["D"], cfg["P"], device=device, seed=0)
    g = torch.Generator(device=device).manual_seed(5)
    T = n * chunk
    cu = (torch.arange(n + 1, dtype=torch.int32) * chunk).to(device)
    calls = []
    for c in range(4):
        k_new = torch.randn((T, cfg["H_kv"], cfg["D"]), generator=g, device=device).to(torch.bfloat16)
        v_new = torch.randn((T, cfg["H_kv"], cfg["D"]), generator=g, device=device).to(torch.bfloat16)
        sl = torch.full((n,), chunk * (c + 1), dtype=torch.int32, device=device)
        calls.append((k_new, v_new, sl))
    per_call = 2 * 2 * T * cfg["H_kv"] * cfg["D"] * 2

    def step(i, stream):
        k_new, v_new, sl = calls[i % 4]
        ira.kv_append(k_new, v_new, cu, sl, cache.page_table, cache.k_cache, cache.v_cache,
                      stream=stream)

    ms, clocks = time_steps(args, device, step, K, warmup, 40)
    config = {"workload": "kv_append", "sequences": n, "tokens_per_call": T,
              "heads_kv": cfg["H_kv"], "head_dim": cfg["D"], "page_size": cfg["P"],
              "l2": f"4 calls x {per_call / 1e6:.0f} MB per rotation (L2 129 MB)"}
    return dict(ms=ms, K=K, clocks=clocks, launches=K, config=config, units_total=K * per_call,
                bytes_total=K * per_call, kernel="kv_append_kernel", kernel_launches=K,
                unit="GB/s")


def bench_kv_conv_append(args, device, K, warmup):
    """One step = the short convolutions on K and V (width 4) ahead of the
    KV append, for one chunked-prefill call: the same 4 sequences x 2048 new
    tokens as ``kv_append``, c cycling over the four calls; each sequence has
    its own state pool row.  Bytes: every new K and V row read once and every
    convolved row written once, plus the state rows read and rewritten and the
    taps."""
    import paged_attention_relative_attn_gb300 as ira
    cfg = W.CHUNKED_PREFILL
    width = 4
    n = cfg["n_seqs"] if args.batch is None else args.batch
    chunk, L = cfg["chunk"], cfg["seq_len"]
    H, D = cfg["H_kv"], cfg["D"]
    cache = W.make_prefill_cache([L] * n, H, D, cfg["P"], device=device, seed=0)
    g = torch.Generator(device=device).manual_seed(6)
    T = n * chunk
    cu = (torch.arange(n + 1, dtype=torch.int32) * chunk).to(device)
    w_k = 0.5 * torch.randn((H, D, width), generator=g, device=device)
    w_v = 0.5 * torch.randn((H, D, width), generator=g, device=device)
    s_k = torch.randn((n, width - 1, H, D), generator=g, device=device).to(torch.bfloat16)
    s_v = torch.randn((n, width - 1, H, D), generator=g, device=device).to(torch.bfloat16)
    slots = torch.arange(n, dtype=torch.int32, device=device)
    calls = []
    for c in range(4):
        k_new = torch.randn((T, H, D), generator=g, device=device).to(torch.bfloat16)
        v_new = torch.randn((T, H, D), generator=g, device=device).to(torch.bfloat16)
        sl = torch.full((n,), chunk * (c + 1), dtype=torch.int32, device=device)
        calls.append((k_new, v_new, sl))
    per_call = (2 * 2 * T * H * D * 2            # new rows read, convolved rows written
                + 2 * 2 * n * (width - 1) * H * D * 2  # state rows read and rewritten
                + 2 * H * D * width * 4)          # taps

    def step(i, stream):
        k_new, v_new, sl = calls[i % 4]
        ira.kv_conv_append(k_new, v_new, cu, sl, cache.page_table, cache.k_cache, cache.v_cache,
                           w_k, w_v, s_k, s_v, slots, max_q_len=chunk, stream=stream)

    ms, clocks = time_steps(args, device, step, K, warmup, 40)
    config = {"workload": "kv_conv_append", "sequences": n, "tokens_per_call": T, "width": width,
              "heads_kv": H, "head_dim": D, "page_size": cfg["P"],
              "l2": f"4 calls x {per_call / 1e6:.0f} MB per rotation (L2 129 MB)"}
    return dict(ms=ms, K=K, clocks=clocks, launches=K, config=config, units_total=K * per_call,
                bytes_total=K * per_call, kernel="kv_conv_append_kernel", kernel_launches=K,
                unit="GB/s")


def bench_stack(args, device, K, warmup):
    """One step = one decode step over the 66-layer stack: 55 local layers
    (16 KV heads, window 512, R=512) and 11 global layers (8 KV heads, full
    causal, R=1024), batch 128 with lognormal lengths, fresh K/V/bias per
    layer (every layer's own paged pool)."""
    import paged_attention_relative_attn_gb300 as ira
    s = W.STACK
    lens = W.draw_stack_lengths(0)
    layers = []
    for layer in range(s["n_layers"]):
        c = s["glob"] if W.is_global_layer(layer) else s["local"]
        layers.append(W.make_decode(s["B"], s["H_q"], c["H_kv"], s["D"], s["P"], lens,
                                    c["window"], c["R"], device=device, seed=1000 + layer,
                                    max_seq_len=s["max_len"]))
    ws_bytes = max(ira.decode_workspace_bytes(x.B, x.H_q, x.H_kv, x.D, x.window, x.max_seq_len)
                   for x in layers)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(layers[0].q)
    lse = torch.empty(layers[0].q.shape[:2], dtype=torch.float32, device=device)
    per_layer = [decode_bytes(x) for x in layers]
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    n_merge = sum(1 for x in layers if ira.choose_splits(x.B, x.H_kv, x.window, x.max_seq_len, sms) > 1)

    def step(i, stream):
        for x in layers:
            ira.decode_inputs(x, out=out, lse=lse, workspace=ws, stream=stream)

    ms, clocks = time_steps(args, device, step, K, warmup, 4)
    config = {"workload": "decode_66_layers", "layers": "55 local (48/16, W=512, R=512) + 11 "
              "global (48/8, causal, R=1024)", "batch": s["B"], "head_dim": s["D"],
              "page_size": s["P"], "lengths": "lognormal mean 2048, sigma 0.5, clipped [1, 8192]",
              "l2": f"{sum(p[0] for p in per_layer) / 1e9:.1f} GB of visible K/V per step"}
    return dict(ms=ms, K=K, clocks=clocks, launches=K * (len(layers) + n_merge), config=config,
                units_total=K * sum(p[0] for p in per_layer),
                bytes_total=K * sum(p[1] for p in per_layer), kernel="decode_kernel",
                kernel_launches=K * len(layers), unit="GB/s")


def _packed_views(buf, specs):
    """Views (dtype, shape) into one flat uint8 buffer at 256-byte aligned
    offsets; returns (views, bytes used)."""
    views, off = [], 0
    for dtype, shape in specs:
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        views.append(buf[off:off + n].view(dtype).view(shape))
        off += (n + 255) // 256 * 256
    return views, off


def _packed_bytes(specs):
    off = 0
    for dtype, shape in specs:
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        off += (n + 255) // 256 * 256
    return off


def bench_decode_e2e(args, device, sets, ws, nbuf=2):
    """Same metric through the public API with host buffers, the way a serving
    loop drives it: every step copies its per-step inputs (q, rel_logits,
    page_table, seq_lens) from pinned host memory, runs decode and reads out +
    lse back to pinned host memory.  A step's inputs sit packed in one pinned
    staging buffer and move in one host-to-device copy (each copy has a fixed
    cost of several microseconds); out and lse are written into one device
    buffer and move back in one copy.  Inputs and outputs are double-buffered
    on the device: step i+1's upload runs on one side stream and step i-1's
    download on another while step i's kernel runs.  The calls of a rotation
    of steps are captured once in a CUDA graph and replayed, so every timed
    step still performs its own copies.  The paged K/V cache is the model's
    resident state and stays in HBM."""
    import paged_attention_relative_attn_gb300 as ira
    n = len(sets)
    NB = nbuf  # device input / output buffers
    s0 = sets[0]
    in_specs = [(s0.q.dtype, s0.q.shape), (s0.rel_logits.dtype, s0.rel_logits.shape),
                (s0.page_table.dtype, s0.page_table.shape), (s0.seq_lens.dtype, s0.seq_lens.shape)]
    out_specs = [(s0.q.dtype, s0.q.shape), (torch.float32, s0.q.shape[:2])]
    in_bytes = _packed_bytes(in_specs)
    out_bytes = _packed_bytes(out_specs)
    host_in = []
    for s in sets:
        hb = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        views, _ = _packed_views(hb, in_specs)
        for v, t in zip(views, (s.q, s.rel_logits, s.page_table, s.seq_lens)):
            v.copy_(t.cpu())
        host_in.append(hb)
    dev_in = [torch.empty(in_bytes, dtype=torch.uint8, device=device) for _ in range(NB)]
    dev_in_v = [_packed_views(b, in_specs)[0] for b in dev_in]
    dev_out = [torch.empty(out_bytes, dtype=torch.uint8, device=device) for _ in range(NB)]
    dev_out_v = [_packed_views(b, out_specs)[0] for b in dev_out]
    host_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(NB)]
    main = torch.cuda.Stream(device)
    up = torch.cuda.Stream(device)    # host-to-device copies
    down = torch.cuda.Stream(device)  # device-to-host copies
    per = n * max(1, 32 // n)  # steps per graph replay (a whole number of rotations)

    def enqueue(steps):
        up.wait_stream(main)
        down.wait_stream(main)
        kdone, ddone = [], []
        for i in range(steps):
            b = i % NB
            s = sets[i % n]
            with torch.cuda.stream(up):
                if i >= NB:
                    up.wait_event(kdone[i - NB])  # step i-NB's kernel has read dev_in[b]
                dev_in[b].copy_(host_in[i % n], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(up)
            q, rel, pt, sl = dev_in_v[b]
            out, lse = dev_out_v[b]
            with torch.cuda.stream(main):
                main.wait_event(ready)
                if i >= NB:
                    main.wait_event(ddone[i - NB])  # step i-NB's result has left dev_out[b]
                ira.decode(q, s.k_cache, s.v_cache, pt, sl, rel, window=s.window,
                           scale=s.scale, max_seq_len=s.max_seq_len, out=out, lse=lse,
                           workspace=ws, stream=main)
                ev = torch.cuda.Event()
                ev.record(main)
                kdone.append(ev)
            with torch.cuda.stream(down):
                down.wait_event(ev)
                host_out[b].copy_(dev_out[b], non_blocking=True)
                ev2 = torch.cuda.Event()
                ev2.record(down)
                ddone.append(ev2)
        main.wait_stream(up)
        main.wait_stream(down)

    main.wait_stream(torch.cuda.current_stream())
    enqueue(per)  # eager warm-up
    torch.cuda.synchronize()
    # the packed round trip returns the same result as the direct call
    ref_out, ref_lse = ira.decode_inputs(sets[(per - 1) % n])
    torch.cuda.synchronize()
    got_out, got_lse = _packed_views(host_out[(per - 1) % NB], out_specs)[0]
    if not (torch.equal(got_out, ref_out.cpu()) and torch.equal(got_lse, ref_lse.cpu())):
        raise RuntimeError("e2e: the packed round trip differs from the direct decode call")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(main):
        with torch.cuda.graph(g, stream=main):
            enqueue(per)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 3000) // per)
    K = reps * per
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(main):
        ev0.record(main)
        for _ in range(reps):
            g.replay()
        ev1.record(main)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(ev0.elapsed_time(ev1), wall * 1e3)
    kv = sum(decode_bytes(sets[i % n])[0] for i in range(K))
    return dict(value=kv / (ms * 1e-3) / 1e9, unit="GB/s", h2d_bytes_per_step=in_bytes,
                d2h_bytes_per_step=out_bytes, steps=K,
                how="public API calls captured in a CUDA graph; per step: one H2D copy of the packed "
                    "q, rel_logits, page_table, seq_lens from pinned host memory (double-buffered, "
                    "overlapping the previous step's kernel), decode, one D2H copy of the packed "
                    "out and lse to pinned host memory on a third stream")


# ---------------------------------------------------------------------------
# oracle timing

def oracle_units(inp, budget_s, max_units=None):
    """Time the oracle, as it stands, on (sequence, KV-head group) units of a
    decode batch until ~budget_s of CPU work (at least one unit).  Only the
    pages a unit uses are gathered into fp64 host arrays; that preparation is
    timed with the oracle call.  Returns (GB/s of visible K+V, units done,
    seconds)."""
    from oracle.ref import ref_decode
    P = inp.page_size
    G = inp.H_q // inp.H_kv
    done_bytes = 0
    t_used = 0.0
    n = 0
    total = inp.B * inp.H_kv
    for u in range(total):
        t0 = time.perf_counter()
        b, hk = divmod(u, inp.H_kv)
        L = int(inp.seq_lens[b])
        npg = (L + P - 1) // P
        ids = inp.page_table[b, :npg].long()
        kc = inp.k_cache.index_select(0, ids)[:, :, hk:hk + 1].float().cpu().numpy().astype(np.float64)
        vc = inp.v_cache.index_select(0, ids)[:, :, hk:hk + 1].float().cpu().numpy().astype(np.float64)
        pt = np.arange(npg, dtype=np.int64)[None, :]
        q = inp.q[b:b + 1, hk * G:(hk + 1) * G].float().cpu().numpy().astype(np.float64)
        rel = inp.rel_logits[b:b + 1, hk * G:(hk + 1) * G].float().cpu().numpy().astype(np.float64)
        ref_decode(q, kc, vc, pt, np.array([L]), rel, inp.window, inp.scale)
        t_used += time.perf_counter() - t0
        vis = min(L, inp.window) if inp.window > 0 else L
        done_bytes += vis * inp.D * 2 * 2
        n += 1
        if t_used >= budget_s or (max_units and n >= max_units):
            break
    return done_bytes / t_used / 1e9, n, t_used


def cpu_cores():
    """(host cores, BLAS threads the oracle's NumPy uses)."""
    return os.cpu_count() or 1, blas_threads()


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


def _reduce(args, x, op):
    if args.world <= 1:
        return x
    dev = "cpu" if torch.distributed.get_backend() == "gloo" else f"cuda:{args.local}"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(args, x):
    """Slowest rank's time: the job's time."""
    return _reduce(args, x, torch.distributed.ReduceOp.MAX) if args.world > 1 else x


def sum_over_ranks(args, x):
    """Units processed by all ranks together."""
    return _reduce(args, x, torch.distributed.ReduceOp.SUM) if args.world > 1 else x


# ---------------------------------------------------------------------------

def run_reference(args):
    """The oracle arm: rank 0 only, on host cores.  Each step is a bounded
    sample of (sequence, KV-head) units of the workload -- every unit of its
    first 4 sequences, or as many as fit the per-step budget -- sized so the
    whole run stays within a few minutes.  ms_per_step is the measured time
    of a step."""
    if args.rank != 0:
        return
    n_seq = 4
    inp = W.make_decode_config(args.workload, device="cpu", seed=0, batch=n_seq)
    per_step = min(args.ref_budget, max(0.002, 150.0 / max(1, args.steps + args.warmup)))
    vals, secs = [], []
    units = 0
    for i in range(args.warmup + args.steps):
        gbs, n, t = oracle_units(inp, per_step)
        if i >= args.warmup:
            vals.append(gbs)
            secs.append(t)
            units += n
    v = statistics.median(vals)
    cores, blas = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(secs) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": decode_workload_config(args, args.workload),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "blas_threads": blas,
                             "kind": "oracle",
                             "sample": f"per step: (sequence, KV head) units of the first "
                                       f"{n_seq} sequences of {args.workload} (all "
                                       f"{n_seq * inp.H_kv}, or as many as fit "
                                       f"{per_step:.3f} s); {units} units timed over "
                                       f"{args.steps} steps, {sum(secs):.2f} s"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DEFAULT_STEPS = {"local_decode": 10000, "global_decode": 2000, "chunked_prefill": 200,
                 "global_prefill": 50, "kv_append": 2000, "kv_conv_append": 2000,
                 "mtp_decode": 5000, "decode_66_layers": 40}
KERNEL_SOURCES = {
    "kv_append_kernel": ["paged_attention_relative_attn_gb300/csrc/kv_append.cu",
                         "paged_attention_relative_attn_gb300/csrc/plan.cuh"],
    "kv_conv_append_kernel": ["paged_attention_relative_attn_gb300/csrc/kv_conv.cu",
                              "paged_attention_relative_attn_gb300/csrc/plan.cuh"],
    "decode_kernel": ["paged_attention_relative_attn_gb300/csrc/decode.cu",
                      "paged_attention_relative_attn_gb300/csrc/plan.cuh",
                      "paged_attention_relative_attn_gb300/csrc/ptx.cuh"],
    "prefill_kernel": ["paged_attention_relative_attn_gb300/csrc/prefill.cu",
                       "paged_attention_relative_attn_gb300/csrc/plan.cuh",
                       "paged_attention_relative_attn_gb300/csrc/ptx.cuh",
                       "paged_attention_relative_attn_gb300/csrc/tc.cuh"],
}


def run_workload(args, device, name, K, warmup):
    if name in ("local_decode", "global_decode"):
        return bench_decode(args, device, name, K, warmup)
    if name in PREFILL_WORKLOADS:
        return bench_prefill(args, device, K, warmup, name)
    if name == "kv_append":
        return bench_kv_append(args, device, K, warmup)
    if name == "kv_conv_append":
        return bench_kv_conv_append(args, device, K, warmup)
    if name == "mtp_decode":
        return bench_decode_multi(args, device, K, warmup)
    return bench_stack(args, device, K, warmup)


def summarize(args, r, pk):
    """Metric value, roofline and the common keys of one workload's result."""
    ms = r["ms"]
    sec = ms * 1e-3
    units = sum_over_ranks(args, r["units_total"])
    nbytes = sum_over_ranks(args, r["bytes_total"])
    per_launch_s = sec / r["kernel_launches"]
    bytes_per_launch = r["bytes_total"] / r["kernel_launches"]
    achieved = bytes_per_launch / per_launch_s / 1e9
    name = r["config"]["workload"]
    r["config"].setdefault("parallelism", f"replicas x{args.world}")
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"],
            "traffic": traffic_record(r["kernel"], name, KERNEL_SOURCES[r["kernel"]]),
            "kernel": r["kernel"], "peak_source": f"{pk['source']} hbm_gbs (of {pk['source']})",
            "bytes_per_launch": bytes_per_launch}
    out = {"value": None, "unit": r["unit"], "ms_per_step": ms / r["K"], "steps": r["K"],
           "config": r["config"], "clocks": r["clocks"], "gpu_launches": r["launches"],
           "launch": dict(r.get("launch", {}),
                          timing="CUDA graph replay of exactly K steps, CUDA events")}
    if r["unit"] == "TFLOP/s":
        tflops = units / sec / 1e12
        out["value"] = tflops
        out["metric"] = METRIC + " [prefill TFLOP/s]"
        if r.get("bound") == "tensor":
            # one kernel timed alone for a fraction of a second: the burst
            # bf16 figure applies
            peak = pk["bf16_tflops"]
            roof = {"bound": "tensor", "achieved": tflops / args.world, "peak": peak,
                    "unit": "TFLOP/s", "frac": tflops / args.world / peak,
                    "traffic": roof["traffic"], "kernel": r["kernel"],
                    "peak_source": f"{pk['source']} bf16_tflops, burst (of {pk['source']})",
                    "flops_per_launch": r["units_total"] / r["kernel_launches"],
                    "hbm_achieved_gbs": achieved, "hbm_frac": achieved / pk["hbm_gbs"]}
        else:
            roof["tflops"] = tflops / args.world
            roof["tensor_peak_tflops"] = pk["bf16_tflops"]
            roof["tensor_frac"] = tflops / args.world / pk["bf16_tflops"]
    else:
        out["value"] = units / sec / 1e9
        roof["kv_frac"] = units / args.world / sec / 1e9 / pk["hbm_gbs"]
        out["metric"] = METRIC
    out["roofline"] = roof
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="local_decode",
                    choices=["local_decode", "global_decode", "chunked_prefill",
                             "global_prefill", "kv_append", "kv_conv_append", "mtp_decode",
                             "decode_66_layers"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=5.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first sequences (profiling of a smaller case)")
    ap.add_argument("--sets", type=int, default=None, help="number of rotated input sets")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary workloads (global decode, prefill, 66-layer step)")
    args = ap.parse_args()
    args.world, args.rank, args.local = dist_env()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]
    if args.workload not in ("local_decode", "global_decode") and args.impl == "reference":
        args.workload = "local_decode"

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
    r = run_workload(args, device, args.workload, args.steps, args.warmup)
    head = summarize(args, r, pk)
    line = {"metric": head["metric"], "value": head["value"], "unit": head["unit"],
            "n_gpus": args.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": head["config"], "launch": head["launch"],
            "clocks": head["clocks"], "gpu_launches": head["gpu_launches"],
            "roofline": head["roofline"]}
    if args.workload in ("local_decode", "global_decode") and not args.no_e2e:
        e2e = bench_decode_e2e(args, device, r["sets"], r["ws"])
        e2e["value"] = sum_over_ranks(args, e2e["value"])
        line["e2e"] = e2e
    else:
        line["e2e"] = None
    if args.rank == 0 and not args.no_cpu_baseline and "sets" in r:
        gbs, n, t = oracle_units(r["sets"][0], args.cpu_budget)
        cores, blas = cpu_cores()
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores,
                                "blas_threads": blas, "kind": "oracle",
                                "sample": f"{n} (sequence, KV head) units of {args.workload} "
                                          f"(first of {r['sets'][0].B * r['sets'][0].H_kv}), "
                                          f"{t:.1f} s of fp64 oracle time"}
    del r
    torch.cuda.empty_cache()
    if not args.no_extra and args.workload == "local_decode":
        extra = {}
        for name, K in (("global_decode", 1000), ("chunked_prefill", 100),
                        ("global_prefill", 20), ("kv_append", 1000), ("kv_conv_append", 1000),
                        ("mtp_decode", 2000),
                        ("decode_66_layers", 20)):
            rr = run_workload(args, device, name, K, 5)
            extra[name] = summarize(args, rr, pk)
            del rr
            torch.cuda.empty_cache()
        line["extra_workloads"] = extra
    if args.rank == 0:
        print(json.dumps(line), flush=True)
    if args.world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
