#!/usr/bin/env python
"""Benchmark of the GB300 attention path (one JSON line on stdout).

A step is one pass of the hot path over one batch of synthetic input:
  * prefill (the headline): attn_fwd on bf16 causal prefill B=4, Hq=32,
    Hkv=8, S=2048, D=128 (tile loads, Q K^T, masks, online softmax, P V,
    normalisation and store, all in one kernel launch), inputs resident in HBM;
  * decode (reported beside it): attn_decode on bf16 B=64, Hq=32, Hkv=8,
    Sk=8192, D=128 (split-KV partials and the log-sum-exp combine);
  * paged decode (reported beside it): attn_decode_paged on the same heads
    with seeded contexts of 4096..8192 keys in 64-token blocks of a shuffled
    pool;
  * varlen prefill (reported beside it): attn_fwd_varlen on 32 packed causal
    sequences of seeded lengths 512..4096;
  * backward (reported beside it): attn_bwd on the headline shape with the
    forward's out and lse given (dQ, dK, dV; 10 D flops per admissible pair);
  * long causal prefill (reported beside it): attn_fwd on bf16 causal B=1,
    Hq=32, Hkv=8, S=8192, D=128, timed like the headline;
  * masked prefill (reported beside it): attn_fwd on bf16 B=2, Hq=Hkv=16,
    S=4096, D=64, causal with window (1024, 0), softcap 50, ALiBi and 82
    empty rows, timed like the headline.
value = causal-adjusted attention TFLOP/s (4 D flops per admissible
(query, key) pair) over all ranks.  The decode object reports HBM GB/s of its
algorithmic bytes (Q + K + V + O).  e2e = the headline through attn_fwd with
Q, K, V in pinned host memory and O copied back every step (steps pipelined
over two streams); e2e.link = pinned copies of one step's bytes, up and down
at once with no kernel, timed in the same run: the host link's own floor.

--impl reference runs the float64 CPU oracle (the only other implementation
of the method here) on a bounded row sample of the same workload.

Multi-GPU: one process per GPU (torchrun); the workload is replicated per GPU
(independent problems, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "attn fwd TFLOP/s (causal-adj) & decode HBM GB/s, % of roofline, 1×GB300"
PREFILL = "bf16_causal_b4_h32_s2048_d128"
DECODE = "bf16_decode_b64_h32_sk8192_d128"
LONG = "bf16_causal_b1_h32_s8192_d128"
MASKED = "bf16_masked_b2_h16_s4096_d64"
L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gbattn", choices=["gbattn", "reference"])
    ap.add_argument("--workload", default=PREFILL, choices=[n for n in WORKLOADS if not WORKLOADS[n].decode])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time of the CPU baseline")
    ap.add_argument("--no-paged", action="store_true")
    ap.add_argument("--no-varlen", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the S=8192 causal prefill object")
    ap.add_argument("--no-masked", action="store_true", help="skip the masked D=64 prefill object")
    ap.add_argument("--profile", choices=["prefill", "decode", "both", "paged", "varlen", "backward"], default=None,
                    help="launch warm-up + steps of one path and exit (for ncu); no timing, one input copy")
    ap.add_argument("--decode-b", type=int, default=None, help="override the decode batch (smaller ncu captures)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- environment
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
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle sampling of one GPU while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        if not shutil.which("nvidia-smi"):
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.out = open(self.path, "w")
        self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-lms", "100", "-i", str(self.gpu)], stdout=self.out,
                                     stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                     hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy), "power_w_max": max(r["power"] for r in rows)}


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    # NCCL reduces device tensors, gloo (the CPU tests) host tensors
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- ncu traffic
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel, from one ncu capture, keyed by a fingerprint of the
# kernel's source files (comments and whitespace excluded): a changed kernel
# reports null until it is captured again.  The captures and their commands
# are summarised under profiles/.
KERNEL_SOURCES = {
    # api.cu chooses the tensor-map boxes, grids and split plans of every launch
    "prefill": ("prefill_bf16.cu", "ptx.cuh", "kernels.h", "api.cu"),
    "decode": ("decode_bf16.cu", "decode_balanced.cu", "decode_common.cuh", "ptx.cuh", "kernels.h", "api.cu"),
    "backward": ("backward_bf16.cu", "ptx.cuh", "kernels.h", "api.cu"),
}
NCU_TRAFFIC = {
    # (kernel, workload, source fingerprint): bytes per launch, one-pass ncu
    # captures of the full-size workloads (values as ncu prints them)
    ("prefill", "bf16_causal_b4_h32_s2048_d128", "9c79f61dcc9de1e5"): 130435328,
    ("prefill", "bf16_causal_b1_h32_s8192_d128", "9c79f61dcc9de1e5"): 134017280,
    ("prefill", "bf16_masked_b2_h16_s4096_d64", "9c79f61dcc9de1e5"): 51230464,
    ("prefill", "bf16_varlen_causal_b32_h32_kv8_len512-4096_d128", "9c79f61dcc9de1e5"): 1779241984,
    ("decode", "bf16_decode_b64_h32_sk8192_d128", "2661c8e8b5421807"): 2154888448,
    ("decode", "bf16_paged_decode_b64_h32_kv8_ctx4096-8192_bs64_d128", "2661c8e8b5421807"): 1746260224,
    ("backward", "bf16_causal_bwd_b4_h32_kv8_s2048_d128:dkdv", "042fcd65f6122d1e"): 337790976,
    ("backward", "bf16_causal_bwd_b4_h32_kv8_s2048_d128:dq", "042fcd65f6122d1e"): 296857600,
}


def source_tokens(text):
    """C/C++ source without comments, each run of whitespace collapsed to one
    space: what the compiler sees of it, so that an edit to a comment or to
    indentation keeps a kernel's fingerprint while `a - -b` and `a--b` stay
    different programs."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_fingerprint(kind, read=None):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        if read is None:
            with open(os.path.join(ROOT, "tiled_scaled_dot_gb300", "csrc", f)) as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(source_tokens(text).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kind, workload):
    return NCU_TRAFFIC.get((kind, workload, kernel_fingerprint(kind)))


# ----------------------------------------------------------------------------- GPU arm
def prefill_call(g, w, x, out):
    return g.attn_fwd(x["q"], x["k"], x["v"], x["alibi_slopes"], softmax_scale=w.scale, causal=w.causal,
                      window_left=w.window_left, window_right=w.window_right, softcap=w.softcap,
                      row_kv_bounds=x["row_kv_bounds"], out=out)


def time_region(fn, steps, ws, stream):
    barrier(ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return e0.elapsed_time(e1)


def soak(fn, seconds):
    """Untimed back-to-back steps so that clocks settle before the timed region."""
    t0 = time.time()
    i = 0
    while time.time() - t0 < seconds:
        fn(i)
        i += 1
        if i % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def bench_prefill(g, w, args, ws, dev, pk, e2e=True):
    stream = torch.cuda.current_stream()
    base = make_inputs(w, dev)
    in_bytes = sum(t.numel() * t.element_size() for k, t in base.items() if k in ("q", "k", "v"))
    n_copies = 1 if args.profile else max(1, math.ceil(2 * L2_BYTES / in_bytes))  # rotate past L2
    sets = [base] + [{k: (None if t is None else t.clone()) for k, t in base.items()} for _ in range(n_copies - 1)]
    outs = [torch.empty_like(base["q"]) for _ in range(n_copies)]
    fn = lambda i: prefill_call(g, w, sets[i % n_copies], outs[i % n_copies])
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    if g.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")
    if args.profile:
        for i in range(args.steps):
            fn(i)
        torch.cuda.synchronize()
        return None
    soak(fn, 1.0)
    ms = time_region(fn, args.steps, ws, stream)
    ms = max_over_ranks(ms, ws)
    flops = w.flops(None if base["row_kv_bounds"] is None else base["row_kv_bounds"].cpu())
    per_launch_ms = ms / args.steps
    tflops = flops / (per_launch_ms * 1e-3) / 1e12
    res = dict(ms_per_step=per_launch_ms, tflops_per_gpu=tflops, flops=flops, dense_flops=w.dense_flops(),
               rotation=n_copies, in_bytes=in_bytes)
    res["roofline"] = {"bound": "tensor", "achieved": round(tflops, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                       "frac": round(tflops / pk["bf16"], 4), "traffic": ncu_traffic("prefill", w.name),
                       "peak_source": f"bf16_tflops ({pk['source']}, burst: the kernel is timed alone)"}
    if e2e and not args.no_e2e:
        res["e2e"] = e2e_prefill(g, w, base, args, ws, stream, flops)
    del sets, outs
    return res


def bench_prefill_object(g, name, args, ws, dev, pk, what, bound_note=None):
    """Another forward workload, timed exactly like the headline (inputs
    rotated past L2, a soak, CUDA events on the launching stream), with its
    own roofline and a bounded oracle sample as its CPU baseline."""
    w = WORKLOADS[name]
    r = bench_prefill(g, w, args, ws, dev, pk, e2e=False)
    obj = {"workload": name, "metric": what, "value": round(r["tflops_per_gpu"] * ws, 2), "unit": "TFLOP/s",
           "ms_per_step": round(r["ms_per_step"], 4), "flops_per_step": r["flops"],
           "dense_flops_per_step": r["dense_flops"], "gpu_launches": args.steps,
           "l2": f"inputs rotated over {r['rotation']} copies ({r['in_bytes'] / 2**20:.0f} MiB each)",
           "roofline": r["roofline"]}
    if bound_note:
        obj["roofline"]["limiter"] = bound_note
    if ws == 1 and not args.no_cpu_baseline:
        x_cpu = make_inputs(w, "cpu")
        tf, sample, threads = oracle_sample(w, x_cpu, min(args.cpu_seconds, 5.0))
        obj["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                               "sample": sample}
    return obj


def e2e_prefill(g, w, base, args, ws, stream, flops):
    """The headline through the public attn_fwd call with the inputs in pinned
    host memory: every step uploads its Q, K, V and downloads its output.  Steps
    are pipelined the way a serving loop runs them: step i + 1's upload (one
    stream) and step i - 1's download (another) overlap step i's kernel, with
    two device buffer sets and events ordering each buffer's reuse.  The timed
    region runs from the first upload to the last download."""
    host = {k: (None if t is None else t.cpu().pin_memory()) for k, t in base.items()}
    devs = [{k: (None if t is None else torch.empty_like(t)) for k, t in base.items()} for _ in range(2)]
    outs = [torch.empty_like(base["q"]) for _ in range(2)]
    out_h = torch.empty(outs[0].shape, dtype=outs[0].dtype, pin_memory=True)
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v"))
    d2h = out_h.numel() * out_h.element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[b])     # the kernel of step i - 2 read these inputs
            for k in ("q", "k", "v"):
                devs[b][k].copy_(host[k], non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if i >= 2:
            stream.wait_event(out_done[b])        # the download of step i - 2 read this output
        with torch.cuda.stream(stream):
            prefill_call(g, w, devs[b], outs[b])
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            out_h.copy_(outs[b], non_blocking=True)
            out_done[b].record(s_out)

    def run(n):
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(n):
            step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier(ws)
        return e0.elapsed_time(e1)

    run(max(2, args.warmup))
    ms = max_over_ranks(run(args.steps), ws)
    tf = flops / (ms / args.steps * 1e-3) / 1e12 * ws
    per = ms / args.steps
    link = host_link_bandwidth(h2d, d2h, args.steps)
    return {"value": round(tf, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(per, 4),
            "pipelining": "upload of step i + 1 and download of step i - 1 overlap step i (two buffer sets)",
            "link": dict(link, frac=round(link["concurrent_ms"] / per, 4))}


def host_link_bandwidth(h2d, d2h, reps):
    """The host link's own ceiling for one step's copies: pinned-memory copies
    of the same byte counts (h2d up on one stream while d2h comes down on
    another), timed with CUDA events, with no kernel between them.  `frac` in
    the e2e object is this time over the measured step time."""
    up_h = torch.empty(h2d, dtype=torch.uint8, pin_memory=True)
    dn_h = torch.empty(d2h, dtype=torch.uint8, pin_memory=True)
    up_d = torch.empty(h2d, dtype=torch.uint8, device="cuda")
    dn_d = torch.empty(d2h, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(up, down):
        torch.cuda.synchronize()
        e0, e1, mid = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                       torch.cuda.Event())
        e0.record(s1)
        s2.wait_event(e0)
        for _ in range(reps):
            if up:
                with torch.cuda.stream(s1):
                    up_d.copy_(up_h, non_blocking=True)
            if down:
                with torch.cuda.stream(s2):
                    dn_h.copy_(dn_d, non_blocking=True)
        mid.record(s2)
        s1.wait_event(mid)
        e1.record(s1)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    timed(True, True)
    t_up, t_dn, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_gbs": round(h2d / (t_up * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h / (t_dn * 1e-3) / 1e9, 1),
            "concurrent_ms": round(t_both, 4),
            "what": "pinned-memory copies of one step's bytes, up and down at once, no kernel"}


def bench_decode(g, args, ws, dev, pk):
    w = WORKLOADS[DECODE]
    if args.decode_b:
        from synth.workloads import scaled
        w = scaled(w, B=args.decode_b)
    stream = torch.cuda.current_stream()
    x = make_inputs(w, dev)
    out = torch.empty_like(x["q"])
    ws_bytes = g.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Sk, w.D, 0)
    wsp = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    fn = lambda i: g.attn_decode(x["q"], x["k"], x["v"], softmax_scale=w.scale, out=out, workspace=wsp)
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    if args.profile:
        for i in range(args.steps):
            fn(i)
        torch.cuda.synchronize()
        return None
    soak(fn, 0.5)
    ms = max_over_ranks(time_region(fn, args.steps, ws, stream), ws)
    per = ms / args.steps
    nbytes = w.bytes_moved()
    gbs = nbytes / (per * 1e-3) / 1e9
    splits = ws_bytes // (w.B * w.Hq * (w.D + 1) * 4) if ws_bytes else 1
    res = {"workload": DECODE, "metric": "decode HBM GB/s (Q+K+V+O bytes)", "value": round(gbs * ws, 1),
           "unit": "GB/s", "ms_per_step": round(per, 4), "bytes_per_step": nbytes,
           "launches_per_step": 2 if ws_bytes else 1, "gpu_launches": args.steps * (2 if ws_bytes else 1),
           "splits": int(splits),
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                        "frac": round(gbs / pk["hbm"], 4),
                        "traffic": None if args.decode_b else ncu_traffic("decode", w.name),
                        "peak_source": f"hbm_gbs ({pk['source']})", "frac_of_8tbs_nominal": round(gbs / 8000.0, 4)}}
    res["graph"] = decode_graph_timing(fn, args, ws, stream)
    if ws == 1 and not args.no_cpu_baseline:
        # the float64 oracle on batch 0 of the same inputs (its Q + K + V + O bytes per second)
        import oracle
        qb, kb, vb = x["q"][:1].cpu(), x["k"][:1].cpu(), x["v"][:1].cpu()
        t0 = time.time()
        oracle.decode(qb, kb, vb, scale=w.scale)
        dt = time.time() - t0
        nb = 2 * qb.numel() * 2 + kb.numel() * 2 + vb.numel() * 2
        res["cpu_baseline"] = {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.max_threads(),
                               "kind": "oracle", "sample": f"batch 0 of {w.B}: {w.Hq} query rows ({dt:.2f} s)"}
    if not args.no_e2e:
        qh = x["q"].cpu().pin_memory()
        kh = x["k"].cpu().pin_memory()
        vh = x["v"].cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

        def step(i):
            x["q"].copy_(qh, non_blocking=True)
            x["k"].copy_(kh, non_blocking=True)
            x["v"].copy_(vh, non_blocking=True)
            fn(i)
            oh.copy_(out, non_blocking=True)

        step(0)
        ms2 = max_over_ranks(time_region(step, max(3, args.steps // 4), ws, stream), ws)
        per2 = ms2 / max(3, args.steps // 4)
        res["e2e"] = {"value": round(nbytes / (per2 * 1e-3) / 1e9 * ws, 1), "unit": "GB/s",
                      "h2d_bytes_per_step": qh.numel() * 2 + kh.numel() * 2 + vh.numel() * 2,
                      "d2h_bytes_per_step": oh.numel() * 2, "ms_per_step": round(per2, 4)}
    return res


# What bounds the masked D=64 workload below the tensor roofline (the
# counters behind it are summarised under profiles/).
MASKED_LIMITER = ("softmax per key tile, not the tensor pipe: each 128-key tile costs a row tanh.approx and "
                  "ex2.approx per key on MUFU (XU pipe busy 47.9 % of cycles) and about 5 other instructions, "
                  "against 512 tensor cycles per slot at D = 64 (tensor pipe 17.4 % active; ncu full set)")


PAGED_SHAPE = dict(B=64, Hq=32, Hkv=8, D=128, block_size=64, ctx_lo=4096, ctx_hi=8192)


def paged_workload_name():
    c = PAGED_SHAPE
    return (f"bf16_paged_decode_b{c['B']}_h{c['Hq']}_kv{c['Hkv']}_ctx{c['ctx_lo']}-{c['ctx_hi']}_"
            f"bs{c['block_size']}_d{c['D']}")


def bench_decode_paged(g, args, ws, dev, pk):
    """Paged-cache decode (attn_decode_paged): seeded per-sequence contexts of
    4096..8192 keys in 64-token blocks at shuffled pool positions.  GB/s of the
    algorithmic bytes: K and V of every live context, plus Q and O."""
    import synth
    from synth.workloads import make_paged_inputs
    c = PAGED_SHAPE
    ctx = (c["ctx_lo"] + synth.randint(c["B"], c["ctx_hi"] - c["ctx_lo"] + 1, 0, 5)).tolist()
    x = make_paged_inputs(c["B"], c["Hq"], c["Hkv"], c["D"], ctx, c["block_size"], device=dev)
    out = torch.empty_like(x["q"])
    wsb = g.decode_paged_workspace_size(c["B"], c["Hq"], c["Hkv"], x["block_table"].shape[1], c["block_size"],
                                        c["D"], 0)
    wsp = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    fn = lambda i: g.attn_decode_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["context_lens"],
                                       out=out, workspace=wsp)
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    if args.profile:
        for i in range(args.steps):
            fn(i)
        torch.cuda.synchronize()
        return None
    soak(fn, 0.5)
    stream = torch.cuda.current_stream()
    ms = max_over_ranks(time_region(fn, args.steps, ws, stream), ws)
    per = ms / args.steps
    nbytes = 2 * sum(ctx) * c["Hkv"] * c["D"] * 2 + 2 * c["B"] * c["Hq"] * c["D"] * 2
    gbs = nbytes / (per * 1e-3) / 1e9
    return {"workload": paged_workload_name(), "metric": "paged decode HBM GB/s (live K+V, Q, O bytes)",
            "value": round(gbs * ws, 1), "unit": "GB/s", "ms_per_step": round(per, 4), "bytes_per_step": nbytes,
            "gpu_launches": args.steps * (2 if wsb else 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm"], 4),
                         "traffic": ncu_traffic("decode", paged_workload_name()),
                         "peak_source": f"hbm_gbs ({pk['source']})", "frac_of_8tbs_nominal": round(gbs / 8000.0, 4)},
            "graph": decode_graph_timing(fn, args, ws, stream)}


VARLEN_SHAPE = dict(B=32, Hq=32, Hkv=8, D=128, len_lo=512, len_hi=4096)


def varlen_workload_name():
    c = VARLEN_SHAPE
    return f"bf16_varlen_causal_b{c['B']}_h{c['Hq']}_kv{c['Hkv']}_len{c['len_lo']}-{c['len_hi']}_d{c['D']}"


def bench_varlen(g, args, ws, dev, pk):
    """Packed variable-length causal prefill (attn_fwd_varlen): 32 sequences
    of seeded lengths 512..4096 (queries = keys), Hq 32, Hkv 8, D 128.
    TFLOP/s of 4 D flops per admissible (query, key) pair."""
    import synth
    c = VARLEN_SHAPE
    lens = (c["len_lo"] + synth.randint(c["B"], c["len_hi"] - c["len_lo"] + 1, 0, 7)).tolist()
    cu = torch.tensor([0] + [sum(lens[:i + 1]) for i in range(len(lens))], dtype=torch.int32, device=dev)
    T = int(cu[-1])
    q = synth.normal((T, c["Hq"], c["D"]), 0, synth.STREAM_Q, torch.bfloat16, dev)
    k = synth.normal((T, c["Hkv"], c["D"]), 0, synth.STREAM_K, torch.bfloat16, dev)
    v = synth.normal((T, c["Hkv"], c["D"]), 0, synth.STREAM_V, torch.bfloat16, dev)
    out = torch.empty_like(q)
    fn = lambda i: g.attn_fwd_varlen(q, k, v, cu, cu, max(lens), causal=True, out=out)
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    if args.profile:
        for i in range(args.steps):
            fn(i)
        torch.cuda.synchronize()
        return None
    soak(fn, 0.5)
    stream = torch.cuda.current_stream()
    ms = max_over_ranks(time_region(fn, args.steps, ws, stream), ws)
    per = ms / args.steps
    flops = 4.0 * c["D"] * c["Hq"] * sum(n * (n + 1) / 2 for n in lens)
    tf = flops / (per * 1e-3) / 1e12
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        # the float64 oracle on the shortest packed sequence of the same inputs
        import oracle
        b = min(range(len(lens)), key=lambda i: lens[i])
        a0, a1 = int(cu[b]), int(cu[b + 1])
        cs = torch.tensor([0, a1 - a0], dtype=torch.int32)
        t0 = time.time()
        oracle.attn_varlen(q[a0:a1].cpu(), k[a0:a1].cpu(), v[a0:a1].cpu(), cs, cs, causal=True)
        dt = time.time() - t0
        n = a1 - a0
        cpu = {"value": round(4.0 * c["D"] * c["Hq"] * n * (n + 1) / 2 / dt / 1e12, 6), "unit": "TFLOP/s",
               "cores": torch.get_num_threads(), "kind": "oracle",
               "sample": f"sequence {b} ({n} tokens, all {c['Hq']} heads; {dt:.1f} s)"}
    return {"workload": varlen_workload_name(), "metric": "varlen causal prefill TFLOP/s (causal-adj)",
            "cpu_baseline": cpu,
            "value": round(tf * ws, 2), "unit": "TFLOP/s", "ms_per_step": round(per, 4), "flops_per_step": flops,
            "total_tokens": T, "gpu_launches": args.steps,
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                         "frac": round(tf / pk["bf16"], 4), "traffic": ncu_traffic("prefill", varlen_workload_name()),
                         "peak_source": f"bf16_tflops ({pk['source']}, burst)"}}


BWD_SHAPE = dict(B=4, Hq=32, Hkv=8, S=2048, D=128)


def bwd_workload_name():
    c = BWD_SHAPE
    return f"bf16_causal_bwd_b{c['B']}_h{c['Hq']}_kv{c['Hkv']}_s{c['S']}_d{c['D']}"


def bench_backward(g, args, ws, dev, pk):
    """Attention backward (attn_bwd with the forward's out and lse given, as
    in training) on the headline shape: bf16 causal B4 Hq32 Hkv8 S2048 D128.
    value = TFLOP/s of 10 D flops per admissible (query, key) pair (the five
    products S, dP, dV, dK, dQ); the kernels run seven (S and dP are formed
    once in each of the two main kernels).  Inputs (q, k, v, dO, out: 224 MiB)
    exceed L2."""
    import synth
    c = BWD_SHAPE
    B, Hq, Hkv, S, D = c["B"], c["Hq"], c["Hkv"], c["S"], c["D"]
    q = synth.normal((B, Hq, S, D), 0, synth.STREAM_Q, torch.bfloat16, dev)
    k = synth.normal((B, Hkv, S, D), 0, synth.STREAM_K, torch.bfloat16, dev)
    v = synth.normal((B, Hkv, S, D), 0, synth.STREAM_V, torch.bfloat16, dev)
    do = synth.normal((B, Hq, S, D), 0, synth.STREAM_DO, torch.bfloat16, dev)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    out = g.attn_fwd(q, k, v, causal=True, lse=lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = torch.empty(g.bwd_workspace_size(B, Hq, Hkv, S, S, D, recompute=False), dtype=torch.uint8, device=dev)
    fn = lambda i: g.attn_bwd(q, k, v, do, out, lse, causal=True, dq=dq, dk=dk, dv=dv, workspace=wsb)
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    if g.device_status() != 0:
        raise RuntimeError("device status word set during the backward warm-up")
    if args.profile:
        for i in range(args.steps):
            fn(i)
        torch.cuda.synchronize()
        return None
    soak(fn, 0.5)
    stream = torch.cuda.current_stream()
    ms = max_over_ranks(time_region(fn, args.steps, ws, stream), ws)
    per = ms / args.steps
    pairs = B * Hq * S * (S + 1) / 2
    flops = 10.0 * D * pairs
    tf = flops / (per * 1e-3) / 1e12
    # per-launch durations from CUDA events recorded between the launches
    *_, phases = g.attn_bwd(q, k, v, do, out, lse, causal=True, dq=dq, dk=dk, dv=dv, workspace=wsb,
                            phase_times_reps=args.steps)
    _, prep_ms, dkdv_ms, dq_ms = phases
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        # the float64 backward oracle on one (batch, kv group) slice of the same inputs
        import oracle
        G = Hq // Hkv
        t0 = time.time()
        oracle.attn_bwd(q[:1, :G].cpu(), k[:1, :1].cpu(), v[:1, :1].cpu(), do[:1, :G].cpu(), causal=True)
        dt = time.time() - t0
        cpu = {"value": round(10.0 * D * G * S * (S + 1) / 2 / dt / 1e12, 6), "unit": "TFLOP/s",
               "cores": torch.get_num_threads(), "kind": "oracle",
               "sample": f"batch 0, kv head 0 and its {G} query heads ({dt:.1f} s)"}
    tf_a = 8.0 * D * pairs / (dkdv_ms * 1e-3) / 1e12  # S, dP, dV, dK
    tf_b = 6.0 * D * pairs / (dq_ms * 1e-3) / 1e12    # S, dP, dQ
    name = bwd_workload_name()
    return {"workload": name, "metric": "attention backward TFLOP/s (causal-adj, 10 D flops per admissible pair)",
            "value": round(tf * ws, 2), "unit": "TFLOP/s", "ms_per_step": round(per, 4), "flops_per_step": flops,
            "flops_convention": "5 products x 2 D per admissible pair; the pages' cost line counts 12 D "
                                "(a 4 D forward recompute)",
            "gpu_launches": 3 * args.steps,  # row intervals, dQ (with Delta), dK / dV
            "cpu_baseline": cpu,
            "phase_ms": {"prep": round(prep_ms, 4), "dkdv": round(dkdv_ms, 4), "dq": round(dq_ms, 4)},
            "roofline": {"bound": "tensor", "kernel": "bwd_kernel dK/dV (S, dP, dV, dK: 8 D flops per pair)",
                         "achieved": round(tf_a, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                         "frac": round(tf_a / pk["bf16"], 4), "traffic": ncu_traffic("backward", name + ":dkdv"),
                         "peak_source": f"bf16_tflops ({pk['source']}, burst)"},
            "roofline_dq": {"bound": "tensor", "kernel": "bwd_kernel dQ (S, dP, dQ: 6 D flops per pair)",
                            "achieved": round(tf_b, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                            "frac": round(tf_b / pk["bf16"], 4), "traffic": ncu_traffic("backward", name + ":dq"),
                            "peak_source": f"bf16_tflops ({pk['source']}, burst)"}}


def decode_graph_timing(fn, args, ws, stream, per_graph=10):
    """The decode step replayed from a CUDA graph of `per_graph` steps (the
    same calls, so host launch overhead is the only difference from eager)."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn(0)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(per_graph):
                fn(i)
        graph.replay()
        torch.cuda.synchronize()
        reps = max(2, args.steps // per_graph)
        ms = max_over_ranks(time_region(lambda i: graph.replay(), reps, ws, stream), ws)
        return {"ms_per_step": round(ms / (reps * per_graph), 4), "steps_per_graph": per_graph, "replays": reps}
    except Exception as e:  # reported, never hidden
        torch.cuda.synchronize()
        return {"error": f"{type(e).__name__}: {e}"[:200]}


# ----------------------------------------------------------------------------- CPU oracle
def admissible_pairs(w, rows, rb):
    """Admissible (query, key) pairs of the given flat (b*Hq + h)*Sq + qi rows."""
    n = 0
    for r in rows.tolist():
        qi = r % w.Sq
        b = r // (w.Sq * w.Hq)
        a, e = 0, w.Sk - 1
        if w.causal:
            e = min(e, qi)
        if w.window_left is not None:
            a = max(a, qi - w.window_left)
        if w.window_right is not None:
            e = min(e, qi + w.window_right)
        if rb is not None:
            a, e = max(a, int(rb[b, qi, 0])), min(e, int(rb[b, qi, 1]))
        n += max(0, e - a + 1)
    return n


def oracle_kwargs(w, x_cpu):
    return dict(scale=w.scale, causal=w.causal, window_left=w.window_left, window_right=w.window_right,
                softcap=w.softcap, alibi_slopes=x_cpu["alibi_slopes"], row_kv_bounds=x_cpu["row_kv_bounds"])


def oracle_rows(w, x_cpu, seconds, seed=11):
    """A seeded row sample of the workload that takes the oracle about
    `seconds` (every row when the whole workload takes less); returns
    (rows, seconds taken)."""
    import oracle
    import synth
    total_rows = w.B * w.Hq * w.Sq
    n = 64
    while True:
        if n >= total_rows:
            rows = torch.arange(total_rows, dtype=torch.int64)
        else:
            rows = torch.unique(synth.randint(n, total_rows, seed, 12))
        t0 = time.time()
        oracle.attn(x_cpu["q"], x_cpu["k"], x_cpu["v"], rows=rows, **oracle_kwargs(w, x_cpu))
        dt = time.time() - t0
        if dt >= seconds or n >= total_rows:
            return rows, dt
        n = min(total_rows, int(n * max(1.2, min(16.0, 1.05 * seconds / max(dt, 1e-3)))))


def oracle_sample(w, x_cpu, seconds):
    """CPU baseline: oracle TFLOP/s on a bounded row sample."""
    import oracle
    rows, dt = oracle_rows(w, x_cpu, seconds)
    flops = 4.0 * w.D * admissible_pairs(w, rows, x_cpu["row_kv_bounds"])
    total = w.B * w.Hq * w.Sq
    return flops / dt / 1e12, f"{sample_text(rows, total)} ({dt:.1f} s)", oracle.max_threads()


def sample_text(rows, total):
    return f"all {total} query rows" if rows.numel() == total else \
        f"{rows.numel()} seeded random query rows of {total}"


# ----------------------------------------------------------------------------- main
def main():
    args = parse()
    ws, rank, local = dist_env()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return main_reference(args, ws, rank, w)
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import tiled_scaled_dot_gb300 as g
    g.lib()
    pk = peaks()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[dev.index]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else dev.index
    if args.profile:
        if args.profile in ("prefill", "both"):
            bench_prefill(g, w, args, ws, dev, pk)
        if args.profile in ("decode", "both"):
            bench_decode(g, args, ws, dev, pk)
        if args.profile == "paged":
            bench_decode_paged(g, args, ws, dev, pk)
        if args.profile == "varlen":
            bench_varlen(g, args, ws, dev, pk)
        if args.profile == "backward":
            bench_backward(g, args, ws, dev, pk)
        if g.device_status() != 0:
            raise RuntimeError("device status word set")
        if rank == 0:
            print(json.dumps({"profile_run": args.profile, "workload": w.name}))
        return
    sampler = ClockSampler(gpu_index)
    sampler.start()
    try:
        pre = bench_prefill(g, w, args, ws, dev, pk)
        dec = None if args.no_decode else bench_decode(g, args, ws, dev, pk)
        paged = None if args.no_paged else bench_decode_paged(g, args, ws, dev, pk)
        varl = None if args.no_varlen else bench_varlen(g, args, ws, dev, pk)
        bwd = None if args.no_backward else bench_backward(g, args, ws, dev, pk)
        long_ = None if args.no_long or w.name == LONG else bench_prefill_object(
            g, LONG, args, ws, dev, pk, "long causal prefill TFLOP/s (causal-adj)")
        masked = None if args.no_masked or w.name == MASKED else bench_prefill_object(
            g, MASKED, args, ws, dev, pk, "masked prefill TFLOP/s (admissible pairs: causal, window, row bounds)",
            MASKED_LIMITER)
    finally:
        clocks = sampler.stop()
    if g.device_status() != 0:
        raise RuntimeError("device status word set during the benchmark")
    total_tf = pre["tflops_per_gpu"] * ws
    line = {
        "metric": METRIC, "value": round(total_tf, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(pre["ms_per_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded SplitMix64 + Box-Muller N(0,1), cast to the storage dtype)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                   "causal": w.causal, "flops_per_step": pre["flops"], "dense_flops_per_step": pre["dense_flops"],
                   "l2": f"inputs rotated over {pre['rotation']} copies ({pre['in_bytes'] / 2**20:.0f} MiB each) "
                         f"so no step reads data left in L2 by the previous one",
                   "parallelism": f"replicas x{ws} (no collective)"},
        "roofline": pre["roofline"],
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if "e2e" in pre:
        line["e2e"] = pre["e2e"]
    if dec is not None:
        line["decode"] = dec
    if paged is not None:
        line["decode_paged"] = paged
    if varl is not None:
        line["varlen"] = varl
    if bwd is not None:
        line["backward"] = bwd
    if long_ is not None:
        line["long_causal"] = long_
    if masked is not None:
        line["masked"] = masked
    if rank == 0 and not args.no_cpu_baseline:
        x_cpu = make_inputs(w, "cpu")
        tf, sample, threads = oracle_sample(w, x_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main_reference(args, ws, rank, w):
    """The float64 oracle on the host cores, each step a bounded row sample."""
    if rank != 0:
        return
    import oracle
    x = make_inputs(w, "cpu")
    # one step is sized to about 3 s so that warm-up + steps end within a few minutes
    per_step = max(0.5, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    rows, _ = oracle_rows(w, x, per_step)
    kw = oracle_kwargs(w, x)
    for _ in range(args.warmup):
        oracle.attn(x["q"], x["k"], x["v"], rows=rows, **kw)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.attn(x["q"], x["k"], x["v"], rows=rows, **kw)
    dt = time.time() - t0
    flops_step = 4.0 * w.D * admissible_pairs(w, rows, x["row_kv_bounds"])
    value = flops_step * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded inputs as the GPU arm)",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                       "causal": w.causal},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{sample_text(rows, w.B * w.Hq * w.Sq)} per step"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
