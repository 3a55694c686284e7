"""Throughput benchmark of the DeltaProduct forward on GB300.

One step = one dp_forward call over the whole workload (by default the
largest single-GPU configuration: the gated B4 H16 T8192 n_h 4 D128 bf16
workload with a nonzero initial state and the final state returned): every
row of the hot path (extended sequence, gate, chunk Gram, UT transform, W/U,
state pass, masked readout, state I/O) runs inside that call. The same line
carries the other bf16 workloads (B4 H8 T2048 n_h 2; B8 H16 T4096 n_h 3 with
near-duplicate keys; B1 H16 T32768 n_h 3 as one call and as 8 carried
4096-token calls), each timed the same way, under "configs".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Arms:
  ours       the library's kernels through the C ABI. `value` is tokens/s with
             inputs resident in HBM; `e2e` is the same call fed from pinned host
             buffers with the host->device copies of the inputs and the
             device->host copy of the outputs inside the timed region.
  reference  the fp64 CPU oracle on the host cores (the only reference this
             method has), on a bounded sample of the same workload.
Under torchrun each rank runs its own copy of the workload (independent
problems, no collective; weak scaling); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from deltaproduct_householder_product_gb300 import workloads as W  # noqa: E402

WORKLOADS = {"base": W.BASE, "neardup": W.NEARDUP, "gated": W.GATED, "long": W.LONG}
# the workloads reported beside the headline one, in this order
SIDE_CONFIGS = ("base", "neardup", "long")
METRIC = "DeltaProduct fwd tokens/s on 1 GB300; % of tensor-pipe/HBM roofline"
L2_BYTES = 129 * 2 ** 20
# o is written in the input dtype (bf16), the size the algorithmic byte count
# takes; the parity tests check the fp32 o against the oracle and the bf16 o
# against the fp32 o rounded once (bit for bit)
OUT_DTYPE = torch.bfloat16


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gated", choices=list(WORKLOADS))
    ap.add_argument("--no-configs", action="store_true",
                    help="measure only --workload, not the other bf16 workloads beside it")
    ap.add_argument("--kernel", default="auto", choices=["auto", "recurrent", "chunk_tc"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    ap.add_argument("--no-varlen", action="store_true", help="skip the packed variable-length measurement")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--no-prologue", action="store_true", help="skip the fused-prologue measurement")
    ap.add_argument("--no-osdn", action="store_true", help="skip the OSDN write-key measurement")
    ap.add_argument("--only", choices=["decode", "varlen", "backward", "prologue", "osdn"],
                    help="run just this measurement (one GPU) and print its object: for profiling")
    ap.add_argument("--fused", action="store_true",
                    help="give dp_forward only the minimum workspace: the chunk path then "
                         "runs as one fused kernel instead of prep + state-pass kernels")
    ap.add_argument("--B", type=int, help="batch of the workload (default: its own); for small profiling cases")
    ap.add_argument("--H", type=int, help="heads of the workload (default: its own)")
    ap.add_argument("--T", type=int, help="tokens per sequence of the workload (default: its own)")
    ap.add_argument("--split", action="store_true",
                    help="give the forward a workspace that holds the per-chunk records but not the "
                         "cooperative flags, so it runs as prep + state-pass kernels (for profiling)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, world, device):
    """The largest of each rank's ``x`` (a time): the job is as slow as its
    slowest replica. Identity at world size 1."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput: the tokens all replicas processed over the
    slowest replica's time per step."""
    return tokens_per_rank * world / (ms * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


def make_copies(w, n_copies, device):
    """n_copies independent device copies of the inputs and outputs so that
    consecutive steps never reuse data still resident in L2."""
    x = W.make_inputs(w)
    copies = []
    for _ in range(n_copies):
        c = {k: (None if v is None else v.to(device)) for k, v in x.items()}
        c["o"] = torch.empty((w.B, w.T, w.H, w.Dv), dtype=OUT_DTYPE, device=device)
        c["hf"] = torch.empty((w.B, w.H, w.Dk, w.Dv), dtype=torch.float32, device=device)
        copies.append(c)
    return x, copies


def forward_calls(dp, L, w, copies, kernel, stream, fused=False, split=False):
    """Pre-marshalled dp_forward calls, one per input copy (keeps per-call host
    work to the ABI call itself)."""
    import ctypes
    from deltaproduct_householder_product_gb300 import _lib
    dims = _lib.make_dims(w.B, w.T, w.H, w.Dk, w.Dv, w.nh, w.torch_dtype, kernel, OUT_DTYPE)
    need = _lib.workspace_size(dims, fast=not fused)
    if split:   # records only: n_chunks x 18688 B after the 256-B status block
        ct = min(16, 32 // w.nh)
        need = 256 + (w.B * w.H * (-(-w.T // ct)) * 18688 + 255) // 256 * 256
    calls = []
    s = ctypes.c_void_p(stream.cuda_stream)
    for c in copies:
        c["ws"] = torch.zeros(need, dtype=torch.uint8, device=c["q"].device)
        args = (ctypes.byref(dims), _lib._ptr(c["q"]), _lib._ptr(c["k"]), _lib._ptr(c["v"]),
                _lib._ptr(c["beta"]), _lib._ptr(c["g"]), _lib._ptr(c["h0"]), _lib._ptr(c["o"]),
                _lib._ptr(c["hf"]), _lib._ptr(c["ws"]), ctypes.c_size_t(need), s)
        calls.append((L.dp_forward, args))
    path = _lib.forward_path(dims, need)
    return calls, dims, path


def run_calls(calls, n, start=0):
    for i in range(start, start + n):
        fn, args = calls[i % len(calls)]
        rc = fn(*args)
        if rc != 0:
            raise RuntimeError(f"dp_forward returned {rc}")


def oracle_sample(w, x, seconds, threads):
    """Time the fp64 oracle on a bounded sample of the workload: every
    (batch, head) sequence, cut to the token prefix that fits `seconds` (the
    whole workload when it fits). Returns (tokens_per_s, description, cores, s)."""
    import oracle
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    flops_tok_head = W.algorithmic_flops(w.scaled(B=1, T=1, H=1))

    def sub(T_s):
        bs = [p[0] for p in pairs]
        hs = [p[1] for p in pairs]
        def take(t, lead):
            if t is None:
                return None
            y = t[bs, :T_s, hs] if lead else t[bs, hs]
            return y.unsqueeze(2) if lead else y.unsqueeze(1)
        return dict(q=take(x["q"], True), k=take(x["k"], True), v=take(x["v"], True),
                    beta=take(x["beta"], True), g=take(x["g"], True),
                    h0=None if x["h0"] is None else take(x["h0"], False))
    # calibrate on a short prefix
    T_cal = min(w.T, 64)
    s = sub(T_cal)
    t0 = time.perf_counter()
    oracle.forward(s["q"], s["k"], s["v"], s["beta"], s["g"], s["h0"], threads=threads)
    rate = len(pairs) * T_cal * flops_tok_head / max(time.perf_counter() - t0, 1e-6)
    T_s = int(max(1, min(w.T, seconds * rate / (len(pairs) * flops_tok_head))))
    s = sub(T_s)
    t0 = time.perf_counter()
    oracle.forward(s["q"], s["k"], s["v"], s["beta"], s["g"], s["h0"], threads=threads)
    dt = time.perf_counter() - t0
    # tokens/s of the full problem = (token-heads/s) / H
    tok_per_s = len(pairs) * T_s / dt / w.H
    desc = (f"{len(pairs)} of {w.B * w.H} (batch,head) sequences x first {T_s} of {w.T} tokens, "
            f"fp64, {dt:.2f} s; tokens/s = token-heads/s / H")
    return tok_per_s, desc, min(threads, len(pairs)), dt


def reference_arm(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    x = W.make_inputs(w)
    per_step = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, x, per_step, threads)
    times, vals, desc, cores = [], [], "", 1
    for _ in range(args.steps):
        v, desc, cores, dt = oracle_sample(w, x, per_step, threads)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "nh": w.nh,
                       "Dk": w.Dk, "Dv": w.Dv},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_measure(dev, hbm_peak, n_steps=256, reps=5):
    """The decode step (one token on a carried fp32 state, in place) on the
    long workload's heads: B1 H16 n_h 3 D128 bf16. Per-step device time with
    one dp_decode_step call per step, and with n_steps calls captured once in
    a CUDA graph and replayed (no host work between steps). Roofline: the
    step must read and write every state once (2 x 64 KiB per (b,h)) plus
    its inputs and o."""
    import ctypes
    from deltaproduct_householder_product_gb300 import _lib
    w = W.LONG
    d = {k: (None if v is None else v.to(dev)) for k, v in W.make_decode_inputs(w, n_steps).items()}
    state = torch.zeros(w.B, w.H, w.Dk, w.Dv, dtype=torch.float32, device=dev)
    o = torch.empty(n_steps, w.B, w.H, w.Dv, dtype=torch.float32, device=dev)
    dims = _lib.make_dims(w.B, 1, w.H, w.Dk, w.Dv, w.nh, w.torch_dtype, "auto", torch.float32)
    L = _lib.lib()

    def run(stream):
        s = ctypes.c_void_p(stream.cuda_stream)
        for i in range(n_steps):
            rc = L.dp_decode_step(ctypes.byref(dims), _lib._ptr(d["q"][i]), _lib._ptr(d["k"][i]),
                                  _lib._ptr(d["v"][i]), _lib._ptr(d["beta"][i]), None, _lib._ptr(state),
                                  _lib._ptr(o[i]), s)
            if rc != 0:
                raise RuntimeError(f"dp_decode_step returned {rc}")

    stream = torch.cuda.current_stream()
    run(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    us_launch = 1e3 * e0.elapsed_time(e1) / n_steps
    us_graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run(torch.cuda.current_stream())
        graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us_graph = 1e3 * e0.elapsed_time(e1) / (reps * n_steps)
    except Exception as exc:   # capture not possible here: report the launched figure only
        print(f"decode graph capture failed: {exc}", file=sys.stderr)
    per_head = (w.Dk + w.nh * (w.Dk + w.Dv + 1)) * 2 + w.Dv * 4 + 2 * w.Dk * w.Dv * 4
    step_bytes = w.B * w.H * per_head
    best = us_graph if us_graph is not None else us_launch
    achieved = step_bytes / (best * 1e-6) / 1e9
    return {"workload": "b1h16-nh3-d128-bf16 decode (fp32 state, fp32 o)", "steps": n_steps,
            "us_per_step_launched": us_launch, "us_per_step_graph": us_graph,
            "steps_per_s": 1e6 / best,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "algorithmic_bytes": step_bytes}}


def backward_measure(dp, dev, hbm_peak, steps=5, warmup=2):
    """The backward pass (dp_backward) on the bench workload (B4 H8 T2048
    n_h 2 D128 bf16, fp32 d_o and dh_final, fp32 gradients): tokens/s from
    CUDA events, inputs resident. Roofline: every input and cotangent read
    once, every gradient written once, the states h0 / dh_final / dh0 once
    per (b,h); the checkpoints the kernel keeps are its own traffic."""
    w = W.BASE
    x = {k: (None if v is None else v.to(dev)) for k, v in W.make_inputs(w).items()}
    gen = torch.Generator().manual_seed(140)
    d_o = torch.randn(w.B, w.T, w.H, w.Dv, generator=gen).to(dev)
    dhf = torch.randn(w.B, w.H, w.Dk, w.Dv, generator=gen).to(dev)
    from deltaproduct_householder_product_gb300 import _lib
    dims = _lib.make_dims(w.B, w.T, w.H, w.Dk, w.Dv, w.nh, w.torch_dtype, "auto", torch.float32)
    ws = torch.zeros(_lib.backward_workspace_size(dims), dtype=torch.uint8, device=dev)

    def timed(impl):
        def call():
            return dp.backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], d_o=d_o, dh_final=dhf,
                               workspace=ws, impl=impl)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream()
        e0.record(stream)
        for _ in range(steps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    ms = timed("auto")
    ms_rec = timed("recurrent")
    # the gated recipe at the same batch, heads and length (n_h = 4): the
    # chunked form (impl="chunk_tc"; "auto" keeps the recurrent form for
    # gated problems) against the recurrent one
    wg = W.GATED.scaled(B=w.B, H=w.H, T=w.T)
    xg = {k: (None if v is None else v.to(dev)) for k, v in W.make_inputs(wg).items()}
    dims_g = _lib.make_dims(wg.B, wg.T, wg.H, wg.Dk, wg.Dv, wg.nh, wg.torch_dtype, "chunk_tc", torch.float32)
    ws_g = torch.zeros(_lib.backward_workspace_size(dims_g), dtype=torch.uint8, device=dev)

    def timed_g(impl):
        def call():
            return dp.backward(xg["q"], xg["k"], xg["v"], xg["beta"], xg["g"], xg["h0"], d_o=d_o, dh_final=dhf,
                               workspace=ws_g, impl=impl)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream()
        e0.record(stream)
        for _ in range(steps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    gated_form = {"workload": f"{wg.name} recipe at B{wg.B} H{wg.H} T{wg.T}",
                  "chunked_ms_per_call": timed_g("chunk_tc"), "recurrent_ms_per_call": timed_g("recurrent")}
    gated_form["chunked_tokens_per_s"] = wg.B * wg.T / (gated_form["chunked_ms_per_call"] * 1e-3)
    del xg, ws_g
    nh, Dk, Dv = w.nh, w.Dk, w.Dv
    gated = 1 if w.gated else 0
    per_tok = 2 * (Dk + nh * Dk + nh * Dv + nh + gated) + 4 * Dv + 4 * (Dk + nh * Dk + nh * Dv + nh + gated)
    states = (3 if w.h0_std > 0 else 2) * Dk * Dv * 4
    step_bytes = w.B * w.T * w.H * per_tok + w.B * w.H * states
    achieved = step_bytes / (ms * 1e-3) / 1e9
    return {"workload": f"{w.name} backward (fp32 d_o, dh_final and gradients)", "ms_per_call": ms,
            "tokens_per_s": w.B * w.T / (ms * 1e-3),
            "kernel": ("chunked: cb_prep, cb_chains, cb_grad_s, cb_grad_r (CUDA cores)" if not w.gated
                       else "backward_kernel (recurrent, CUDA cores)"),
            "recurrent_ms_per_call": ms_rec, "gated": gated_form,
            "workspace_bytes": int(ws.numel()),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "algorithmic_bytes": step_bytes}}


def prologue_measure(dp, dev, hbm_peak, steps=50, warmup=5):
    """The input prologue on the bench workload (B4 H8 T2048 n_h 2 D128
    bf16, fp32 o), from raw projections: fused (dims.prologue: the kernels
    map k, q, beta while loading them) against unfused (dp_prologue writes
    the mapped tensors, then dp_forward reads them). CUDA events, inputs
    resident, one workspace."""
    from deltaproduct_householder_product_gb300 import _lib
    w = W.BASE
    x = {k: (None if v is None else v.to(dev)) for k, v in W.make_raw_inputs(w).items()}
    flags = W.prologue_flags(w)
    # the fast workspace of the prologue call (its records carry the mapped K, Q rows)
    dims = _lib.make_dims(w.B, w.T, w.H, w.Dk, w.Dv, w.nh, w.torch_dtype, "auto", torch.float32,
                          prologue=flags)
    ws = torch.zeros(_lib.workspace_size(dims, fast=True), dtype=torch.uint8, device=dev)
    o = torch.empty(w.B, w.T, w.H, w.Dv, dtype=torch.float32, device=dev)
    hf = torch.empty(w.B, w.H, w.Dk, w.Dv, dtype=torch.float32, device=dev)

    def fused():
        dp.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], out=o, h_final=hf, workspace=ws,
                   prologue=flags)

    def unfused():
        q, k, b, g = dp.prologue(x["q"], x["k"], x["beta"], x["g"], flags=flags)
        dp.forward(q, k, x["v"], b, g, x["h0"], out=o, h_final=hf, workspace=ws)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    ms_f, ms_u = timed(fused), timed(unfused)
    dp.check_status(ws)
    step_bytes = W.algorithmic_bytes(w, out_bytes=4)
    el = 2
    tok = w.B * w.T * w.H
    extra = 2 * el * tok * (w.Dk + w.nh * w.Dk + w.nh + (1 if w.gated else 0))   # mapped tensors out and back in
    achieved = step_bytes / (ms_f * 1e-3) / 1e9
    return {"workload": f"{w.name} from raw projections (SiLU+L2 keys, L2 queries, "
                        f"{'2 ' if w.beta_max == 2.0 else ''}sigmoid betas)",
            "flags": flags, "path": _lib.forward_path(dims, ws.numel()),
            "ms_fused": ms_f, "ms_unfused": ms_u, "tokens_per_s_fused": w.B * w.T / (ms_f * 1e-3),
            "unfused_extra_bytes": extra,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "algorithmic_bytes": step_bytes}}


def osdn_measure(dp, dev, hbm_peak, steps=10, warmup=2):
    """OSDN write keys on the bench workload (B4 H8 T2048 n_h 2 D128 bf16,
    fp32 o): phase 1 (dp_osdn_write_keys: the preconditioner scan, one warp
    per head) and phase 2 (dp_forward_write_keys),
    each timed with CUDA events, inputs resident (phase 2 on the tensor-core
    chunk path, fast workspace). Roofline of phase 2: the
    forward's algorithmic bytes plus the write keys read."""
    w = W.BASE
    x = {k: (None if v is None else v.to(dev)) for k, v in W.make_inputs(w).items()}
    o = torch.empty(w.B, w.T, w.H, w.Dv, dtype=torch.float32, device=dev)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    kw, _ = dp.osdn_write_keys(x["k"], x["beta"])
    ms1 = timed(lambda: dp.osdn_write_keys(x["k"], x["beta"]))
    ms2 = timed(lambda: dp.forward_write_keys(x["q"], x["k"], kw, x["v"], x["beta"], x["g"], x["h0"], out=o,
                                              h_final=False))
    tok = w.B * w.T * w.H
    scan_bytes = tok * w.nh * (2 * w.Dk * 2 + 2)                 # k and beta in, k~ out
    fwd_bytes = W.algorithmic_bytes(w, out_bytes=4) + tok * w.nh * w.Dk * 2
    a2 = fwd_bytes / (ms2 * 1e-3) / 1e9
    return {"workload": f"{w.name} OSDN write keys (eta 0.003, d in [0.5, 2])",
            "ms_scan": ms1, "ms_forward_write_keys": ms2, "tokens_per_s": w.B * w.T / ((ms1 + ms2) * 1e-3),
            "kernels": "dscan_kernel (one warp per head); chunk_coop_kernel with write keys",
            "path": "chunk_coop",
            "scan_roofline": {"bound": "hbm", "achieved": scan_bytes / (ms1 * 1e-3) / 1e9, "peak": hbm_peak,
                              "unit": "GB/s", "frac": scan_bytes / (ms1 * 1e-3) / 1e9 / hbm_peak,
                              "algorithmic_bytes": scan_bytes},
            "roofline": {"bound": "hbm", "achieved": a2, "peak": hbm_peak, "unit": "GB/s",
                         "frac": a2 / hbm_peak, "algorithmic_bytes": fwd_bytes}}


VARLEN_LENGTHS = [384, 2944, 1024, 512, 1792, 256, 896, 384]   # 8 sequences, 8192 tokens


def varlen_measure(dp, dev, hbm_peak, steps=20, warmup=3):
    """Packed variable-length sequences (dp_forward_varlen) with the bench
    workload's heads and token count (H8 n_h 2 D128 bf16, fp32 o): the eight
    lengths above, drawn with the bench workload's recipe. Whole-call
    tokens/s from CUDA events (inputs resident; one workspace reused)."""
    from deltaproduct_householder_product_gb300 import _lib
    T, N = sum(VARLEN_LENGTHS), len(VARLEN_LENGTHS)
    w = W.BASE.scaled(B=1, T=T)
    x = {k: (None if v is None else v[0].to(dev).contiguous()) for k, v in W.make_inputs(w).items()
         if k in ("q", "k", "v", "beta")}
    cu = torch.tensor([0] + list(np.cumsum(VARLEN_LENGTHS)), dtype=torch.int32, device=dev)
    max_len = max(VARLEN_LENGTHS)
    dims = _lib.make_dims(N, T, w.H, w.Dk, w.Dv, w.nh, w.torch_dtype, "auto", torch.float32, max_len)
    ws = torch.zeros(_lib.workspace_size(dims, fast=True), dtype=torch.uint8, device=dev)
    o = torch.empty(T, w.H, w.Dv, dtype=torch.float32, device=dev)
    hf = torch.empty(N, w.H, w.Dk, w.Dv, dtype=torch.float32, device=dev)

    def call():
        dp.forward_varlen(x["q"], x["k"], x["v"], x["beta"], None, None, cu_seqlens=cu, max_seqlen=max_len,
                          out=o, h_final=hf, workspace=ws)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    dp.check_status(ws)
    ms = e0.elapsed_time(e1) / steps
    wbytes = W.algorithmic_bytes(w, out_bytes=4) - w.B * w.H * w.Dk * w.Dv * 4 + N * w.H * w.Dk * w.Dv * 4
    achieved = wbytes / (ms * 1e-3) / 1e9
    return {"workload": f"H{w.H} n_h {w.nh} D{w.Dk} bf16, {N} packed sequences of lengths {VARLEN_LENGTHS}",
            "path": _lib.forward_path(dims, ws.numel()), "ms_per_call": ms, "tokens_per_s": T / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "algorithmic_bytes": wbytes}}


def roofline_obj(w, ms, hbm_peak, peak_kind, path, scope, captured=True):
    """HBM roofline of one forward: algorithmic bytes (inputs, bf16 o, state
    I/O) over the measured time per call. `captured`: the measured DRAM
    traffic of one forward of this workload and path applies (not for other
    call patterns over the same tokens)."""
    wbytes = W.algorithmic_bytes(w, out_bytes=OUT_DTYPE.itemsize)
    achieved = wbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": TRAFFIC.get((w.name, path)) if captured else None,
            "peak_kind": peak_kind, "algorithmic_bytes": wbytes, "scope": scope}


def timed_forward(dp, L, w, dev, steps, warmup, kernel):
    """Time `steps` dp_forward calls over rotating device copies of the
    workload (more than 3x the L2 in total, so no call finds its inputs in
    L2), after `warmup` calls, with CUDA events on the launching stream.
    Returns (ms per call, path, launches per call, number of copies)."""
    from deltaproduct_householder_product_gb300 import _lib
    stream = torch.cuda.current_stream()
    wbytes = W.algorithmic_bytes(w, out_bytes=OUT_DTYPE.itemsize)
    n_copies = max(2, -(-3 * L2_BYTES // wbytes))
    _, copies = make_copies(w, n_copies, dev)
    calls, _, path = forward_calls(dp, L, w, copies, kernel, stream)
    run_calls(calls, warmup)
    torch.cuda.synchronize()
    for c in copies:
        dp.check_status(c["ws"])
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    run_calls(calls, steps, start=warmup)
    ev1.record(stream)
    torch.cuda.synchronize()
    for c in copies:
        dp.check_status(c["ws"])
    ms = ev0.elapsed_time(ev1) / steps
    del copies, calls
    torch.cuda.empty_cache()
    return ms, path, _lib.LAUNCHES[path], n_copies


def carried_calls_measure(dp, dev, w, n_calls, steps, warmup):
    """The long workload as `n_calls` sequential dp_forward calls of T /
    n_calls tokens each, the state carried from one call to the next (h0 and
    h_final the same buffer): time per whole sequence, CUDA events."""
    seg = w.T // n_calls
    x = W.make_inputs(w)
    parts = []
    for s in range(n_calls):
        sl = slice(s * seg, (s + 1) * seg)
        parts.append({k: x[k][:, sl].contiguous().to(dev) for k in ("q", "k", "v", "beta")})
    state = torch.zeros(w.B, w.H, w.Dk, w.Dv, dtype=torch.float32, device=dev)
    o = [torch.empty(w.B, seg, w.H, w.Dv, dtype=OUT_DTYPE, device=dev) for _ in range(n_calls)]
    ws = torch.zeros(dp.workspace_size(w.B, seg, w.H, w.Dk, w.Dv, w.nh, w.torch_dtype, fast=True),
                     dtype=torch.uint8, device=dev)

    def one():
        state.zero_()
        for s in range(n_calls):
            p = parts[s]
            dp.forward(p["q"], p["k"], p["v"], p["beta"], None, state, out=o[s], h_final=state, workspace=ws)
    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    dp.check_status(ws)
    ms = e0.elapsed_time(e1) / steps
    path = dp.forward_path(w.B, seg, w.H, w.Dk, w.Dv, w.nh, ws.numel())
    return ms, path


def side_configs(dp, L, dev, args, hbm_peak, peak_kind):
    """The other bf16 workloads, each timed like the headline one."""
    out = {}
    steps, warmup = max(3, min(args.steps, 50)), max(3, args.warmup)
    for name in SIDE_CONFIGS:
        if name == args.workload:
            continue
        w = WORKLOADS[name]
        ms, path, launches, n_copies = timed_forward(dp, L, w, dev, steps, warmup, args.kernel)
        out[w.name] = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3), "path": path,
                       "launches_per_call": launches, "steps": steps, "warmup": warmup,
                       "l2": f"{n_copies} rotating copies",
                       "roofline": roofline_obj(w, ms, hbm_peak, peak_kind, path, "one forward")}
        if name == "long":
            cms, cpath = carried_calls_measure(dp, dev, w, W.LONG_CALLS, max(3, steps // 5), 2)
            out[w.name + f" as {W.LONG_CALLS} carried calls"] = {
                "ms": cms, "tokens_per_s": w.B * w.T / (cms * 1e-3), "path": cpath,
                "calls": W.LONG_CALLS, "tokens_per_call": w.T // W.LONG_CALLS,
                "roofline": roofline_obj(w, cms, hbm_peak, peak_kind, cpath,
                                         f"{W.LONG_CALLS} carried calls over distinct inputs", captured=False)}
        torch.cuda.empty_cache()
    return out


def ours_arm(args, w):
    import deltaproduct_householder_product_gb300 as dp
    from deltaproduct_householder_product_gb300 import _lib
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = _lib.lib()
    stream = torch.cuda.current_stream()
    hbm_peak, _, peak_kind = measured_peaks()

    wbytes = W.algorithmic_bytes(w, out_bytes=OUT_DTYPE.itemsize)
    n_copies = max(2, -(-3 * L2_BYTES // wbytes))          # rotate copies: > 3x L2 in total
    x, copies = make_copies(w, n_copies, dev)
    calls, dims, path = forward_calls(dp, L, w, copies, args.kernel, stream, args.fused, args.split)
    launches = _lib.LAUNCHES[path]

    run_calls(calls, args.warmup)
    torch.cuda.synchronize()
    for c in copies:
        dp.check_status(c["ws"])

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    ev0.record(stream)
    run_calls(calls, args.steps, start=args.warmup)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall_timed = time.perf_counter() - t_wall
    barrier()
    # keep the GPU busy with the same step while the clock sampler catches up
    soak_until = time.perf_counter() + max(0.0, 1.5 - wall_timed)
    i = args.warmup + args.steps
    while time.perf_counter() < soak_until:
        run_calls(calls, 20, start=i)
        i += 20
    torch.cuda.synchronize()
    clocks = sampler.stop()
    clocks["window"] = "timed region" + (" + soak of the same step" if wall_timed < 1.5 else "")
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    for c in copies:
        dp.check_status(c["ws"])

    # e2e: pinned host inputs -> device, forward, outputs -> host, every step,
    # pipelined as a serving loop runs it: step i+1's inputs upload (copy-in
    # stream) while step i computes and step i-1's outputs download
    # (copy-out stream); two device buffer sets alternate, and events keep a
    # buffer from being overwritten before its step has finished with it.
    host = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
    bufs = copies[:2]
    o_host = [torch.empty(b["o"].shape, dtype=b["o"].dtype).pin_memory() for b in bufs]
    hf_host = [torch.empty(b["hf"].shape, dtype=torch.float32).pin_memory() for b in bufs]
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = o_host[0].numel() * o_host[0].element_size() + hf_host[0].numel() * 4
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        ev = lambda: torch.cuda.Event()
        ev_in, ev_comp, ev_out = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])        # buffer b's inputs consumed
                for kname in ("q", "k", "v", "beta", "g", "h0"):
                    if host[kname] is not None:
                        bufs[b][kname].copy_(host[kname], non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])           # buffer b's outputs downloaded
            run_calls(calls[b:b + 1], 1)
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                o_host[b].copy_(bufs[b]["o"], non_blocking=True)
                hf_host[b].copy_(bufs[b]["hf"], non_blocking=True)
                ev_out[i].record(s_out)
    e2e_run(3)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    stream.wait_stream(s_in)
    s_out.wait_stream(s_in)
    e2e_run(args.e2e_steps)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
    del copies, calls, bufs, host, o_host, hf_host
    torch.cuda.empty_cache()

    if rank != 0:
        return
    tokens = w.B * w.T
    line = {
        "metric": METRIC, "value": job_tokens_per_s(tokens, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "out_dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "nh": w.nh, "Dk": w.Dk,
                   "Dv": w.Dv, "kernel": args.kernel, "gated": w.gated, "h0": w.h0_std > 0,
                   "path": path,
                   "l2": f"{n_copies} rotating input/output copies "
                         f"({n_copies * wbytes / 1e6:.0f} MB > 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": job_tokens_per_s(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipeline": "copy-in, compute and copy-out streams over two device buffer sets"},
        "gpu_launches": args.steps * launches,
        "roofline": roofline_obj(w, ms, hbm_peak, peak_kind, path,
                                 "one forward: every launch dp_forward enqueues"),
        "clocks": clocks,
    }
    if not args.no_configs:
        line["configs"] = side_configs(dp, L, dev, args, hbm_peak, peak_kind)
    if not args.no_decode:
        line["decode"] = decode_measure(dev, hbm_peak)
    if not args.no_varlen:
        line["varlen"] = varlen_measure(dp, dev, hbm_peak)
    if not args.no_backward:
        line["backward"] = backward_measure(dp, dev, hbm_peak)
    if not args.no_prologue:
        line["prologue"] = prologue_measure(dp, dev, hbm_peak)
    if not args.no_osdn:
        line["osdn"] = osdn_measure(dp, dev, hbm_peak)
    if not args.no_cpu_baseline:
        v, desc, cores, _ = oracle_sample(w, x, 8.0, os.cpu_count() or 1)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


# DRAM bytes (read + write) per forward, summed over its launches, from a
# one-pass ncu capture of the current kernels on the full-size workload (bf16
# o; the profiles/ summaries named for each kernel and workload); keyed by
# (workload, path); absent = not captured for the kernels as they stand
TRAFFIC = {
    ("b4h16t8192-nh4-d128-bf16-gated-h0", "chunk_coop"): 1894.8e6,
    ("b4h8t2048-nh2-d128-bf16", "chunk_coop"): 107.7e6,
    ("b8h16t4096-nh3-d128-bf16-neardup", "chunk_split"): 2469.4e6,
    ("b1h16t32768-nh3-d128-bf16-long", "chunk_seg"): 3304.0e6,
}


def only_arm(args):
    """One secondary measurement alone (the object the full line carries),
    with --steps / --warmup as given: a short command to profile it with."""
    import deltaproduct_householder_product_gb300 as dp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_peak, _, _ = measured_peaks()
    steps, warmup = max(1, args.steps), max(1, args.warmup)
    if args.only == "decode":
        out = decode_measure(dev, hbm_peak, reps=steps)
    elif args.only == "varlen":
        out = varlen_measure(dp, dev, hbm_peak, steps=steps, warmup=warmup)
    elif args.only == "backward":
        out = backward_measure(dp, dev, hbm_peak, steps=steps, warmup=warmup)
    elif args.only == "prologue":
        out = prologue_measure(dp, dev, hbm_peak, steps=steps, warmup=warmup)
    else:
        out = osdn_measure(dp, dev, hbm_peak, steps=steps, warmup=warmup)
    print(json.dumps({"only": args.only, **out}))


def main():
    args = parse()
    w = WORKLOADS[args.workload]
    resize = {k: getattr(args, k) for k in ("B", "H", "T") if getattr(args, k)}
    if resize:   # the same recipe at another size (named as such)
        w = w.scaled(**resize)
        w = w.scaled(name=f"{WORKLOADS[args.workload].name} at B{w.B} H{w.H} T{w.T}")
    if args.only:
        only_arm(args)
        return
    if args.impl == "reference":
        reference_arm(args, w)
    else:
        ours_arm(args, w)


if __name__ == "__main__":
    main()
