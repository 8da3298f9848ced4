"""Bench: one layer of Gated DeltaNet prefill on GB300 through the C ABI.

Workload (default): one layer, 16 key heads x 3 = 48 value heads, d = 128,
T = 32768 tokens processed as 16 calls of 2048 tokens with the state carried
between calls, then the gated RMSNorm of all 32768 outputs to FP16.  Seeded
synthetic inputs of the prefill distributions (inputs.py); q/k/v/z are larger
than the 129 MB L2, so every step streams them from HBM.

One step = the 16 recurrence calls in the selected mode + the norm.  The other
mode is timed in the same run and reported under "modes".  Printed: one JSON
line with the metric (us per token per layer, lower is better), per-mode
kernel timings, the roofline of the dominant kernel, the end-to-end number with
host buffers, clocks during the timed region, and the FP64 oracle timed on the
host cores (cpu_baseline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--mode chunked|sequential]
  python bench.py --impl reference     # the FP64 oracle as the reference arm
Under torchrun (N > 1) every rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill recurrence µs/token/layer (48 vh, d=128) and % of roofline"
N_KH, N_VH, D = 16, 48, 128
# algorithmic work per token and layer (48 value heads, d = 128)
FLOP_SEQ = 48 * 7 * D * D                                            # 5.505 Mflop
FLOP_CHUNKED = 48 * (6 * D * D + D * D // 32 + (10 * 32 * D) / 3 + 32 * 32 / 3)  # ~5.42 Mflop
BYTES_REC = 16 * D * 4 * 2 + 48 * D * 4 + 48 * 4 * 2 + 48 * D * 4   # q,k + v + g,beta + o = 65,920 B
BYTES_NORM = 48 * D * 4 * 2 + 48 * D * 2                             # o + z + y = 61,440 B
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), float(d.get("sm_max_mhz", SM_MAX_MHZ)), "measured"
    return 6800.0, SM_MAX_MHZ, "fallback"


def _tf32_peak():
    """Dense TF32 tensor peak: the measured bf16 GEMM rate x the nominal TF32:BF16
    ratio (1.1 : 2.25 PFLOP/s dense), with its basis."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            bf16 = float(json.load(f).get("bf16_tflops", 1900.0))
        src = "measured"
    else:
        bf16, src = 1900.0, "fallback"
    return bf16 * 1.1 / 2.25, f"{src} bf16 GEMM {bf16:.0f} TFLOP/s x 1.1/2.25 (nominal TF32:BF16 dense)"


def aggregate(local_ms: float, tokens_per_rank: int, world_size: int, device=None):
    """Whole-job figures for `world_size` independent replicas: the slowest rank's
    time (max over ranks) and the tokens of all ranks.  Returns (max_ms,
    us_per_token_layer, tokens_per_s).  Needs an initialised process group when
    world_size > 1 (NCCL on the GPUs, gloo in the CPU tests)."""
    ms = float(local_ms)
    if world_size > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    tokens = tokens_per_rank * world_size
    return ms, ms * 1e3 / tokens, tokens / (ms * 1e-3)


def captured_traffic(source_file: str):
    """DRAM bytes per launch from profiles/dram_traffic.md for the unit whose kernel
    source is `source_file`, or None when that file changed since the capture."""
    import hashlib
    import re

    table = os.path.join(ROOT, "profiles", "dram_traffic.md")
    src = os.path.join(ROOT, "linear_attention_recurrence_gb300", "csrc", source_file)
    if not (os.path.exists(table) and os.path.exists(src)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(table):
        m = re.match(r"\|[^|]*\|\s*csrc/(\S+)\s*\|\s*([0-9a-f]{16})\s*\|\s*(\d+)\s*\|", line)
        if m and m.group(1) == source_file:
            return int(m.group(3)) if m.group(2) == sha else None
    return None


def captured_counts(source_file: str):
    """Instruction counts of one launch from profiles/flop_counts.md for the kernel
    whose source is `source_file` (None when that file changed since the capture):
    {"fp32_flop": FFMA x 2 + FFMA2 x 4 + FADD + FADD2 x 2 + FMUL + FMUL2 x 2 (thread
    instructions), "tensor_flop": mma.sync m16n8k8 warp instructions x 2048 + tcgen05.mma
    kind::tf32 math ops (two per multiply-add)}."""
    import hashlib
    import re

    table = os.path.join(ROOT, "profiles", "flop_counts.md")
    src = os.path.join(ROOT, "linear_attention_recurrence_gb300", "csrc", source_file)
    if not (os.path.exists(table) and os.path.exists(src)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(table):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 11 and cells[1] == "csrc/" + source_file and re.fullmatch(r"[0-9a-f]{16}", cells[2]):
            if cells[2] != sha:
                return None
            ffma, ffma2, fadd, fadd2, fmul, fmul2, hmma, umma = (int(c) for c in cells[3:11])
            return {"fp32_flop": 2 * ffma + 4 * ffma2 + fadd + 2 * fadd2 + fmul + 2 * fmul2,
                    "tensor_flop": hmma * 2048 + umma}
    return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.window = None
        self.windows = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def mark(self, t_begin: float, t_end: float):
        """Wall-clock bounds of the timed region (time.time())."""
        self.window = (t_begin, t_end)
        self.windows.append((t_begin, t_end))

    def add_window(self, t_begin: float, t_end: float):
        """Wall-clock bounds of another GPU-timed pass (per-kernel, other mode, C3, C5)."""
        self.windows.append((t_begin, t_end))

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self, all_windows: bool = False):
        """Clocks and throttle reasons in the timed region (or, with all_windows, in
        every GPU-timed pass marked)."""
        import datetime

        wins = self.windows if all_windows else ([self.window] if self.window else [])
        rows = []
        for ln in (self.out or "").splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 9:
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if not wins or any(a <= ts <= b for a, b in wins):
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def cpu_baseline(tokens_target_s: float = 10.0, seed: int = 0):
    """The FP64 oracle (unchanged) on the host cores: recurrence + norm over a
    bounded prefix of the workload, sized for ~tokens_target_s of CPU time."""
    import oracle
    from linear_attention_recurrence_gb300.inputs import make_inputs

    nt = oracle.max_threads()
    probe = 128
    x = make_inputs(probe, seed=seed)
    t0 = time.perf_counter()
    o, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], nthreads=nt)
    oracle.out_norm(o, x["z"], x["w"], 1e-6, nthreads=nt)
    per_tok = (time.perf_counter() - t0) / probe
    T = int(min(32768, max(256, tokens_target_s / max(per_tok, 1e-9))))
    T = (T // 128) * 128
    x = make_inputs(T, seed=seed)
    t0 = time.perf_counter()
    o, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], nthreads=nt)
    oracle.out_norm(o, x["z"], x["w"], 1e-6, nthreads=nt)
    dt = time.perf_counter() - t0
    return {"value": dt / T * 1e6, "unit": "µs/token/layer", "cores": nt, "kind": "oracle",
            "sample": f"first {T} tokens of the T=32768 workload, 48 value heads, FP64 recurrence + norm, "
                      f"{nt} OpenMP threads, {dt:.1f} s"}


def oracle_t8192(seed: int = 0, with_t32768: bool = True):
    """The FP64 oracle (unchanged) at the T = 8192 configuration (recurrence + norm,
    one layer): single-thread and all-core wall times; and, all cores, the whole
    T = 32768 headline workload (its 16 calls of 2048 carry the state, which the
    oracle's one pass over the 32768 tokens does likewise).  The all-core T = 8192
    run is the cpu_baseline of the headline line."""
    import oracle
    from linear_attention_recurrence_gb300.inputs import make_inputs

    T = 8192
    nt = oracle.max_threads()
    x = make_inputs(32768 if with_t32768 else T, seed=seed)

    def run(n, threads):
        t0 = time.perf_counter()
        o, _ = oracle.recurrence(x["q"][:n], x["k"][:n], x["v"][:n], x["g"][:n], x["beta"][:n], x["S0"],
                                 nthreads=threads)
        oracle.out_norm(o, x["z"][:n], x["w"], 1e-6, nthreads=threads)
        return time.perf_counter() - t0

    res = {threads: run(T, threads) for threads in (nt, 1)}
    line = {"value": res[nt] / T * 1e6, "unit": "µs/token/layer", "cores": nt, "kind": "oracle",
            "sample": f"T=8192 (the first 8192 tokens of the workload), 48 value heads, FP64 recurrence + norm, "
                      f"{nt} OpenMP threads: {res[nt]:.2f} s; 1 thread: {res[1]:.2f} s",
            "t8192_all_cores_s": res[nt], "t8192_one_thread_s": res[1],
            "one_thread_us_per_token_layer": res[1] / T * 1e6}
    if with_t32768:
        t = run(32768, nt)
        line["t32768_all_cores_s"] = t
        line["t32768_all_cores_us_per_token_layer"] = t / 32768 * 1e6
    return line


def _stack_layer_inputs(layer: int):
    from linear_attention_recurrence_gb300.inputs import make_inputs

    return make_inputs(2048, seed=0, layer=layer)


def stack_inputs_async(n_layers: int):
    """Start drawing the stack's per-layer inputs (2048 tokens each, each layer its
    own seed) on the host cores in a spawn pool; returns (pool, async result)."""
    import multiprocessing as mp

    pool = mp.get_context("spawn").Pool(processes=max(1, min(16, os.cpu_count() or 1)))
    return pool, pool.map_async(_stack_layer_inputs, range(n_layers))


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    steps = []
    cb = None
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(tokens_target_s=args.ref_seconds)
        if i >= args.warmup:
            steps.append(cb["value"])
    v = statistics.median(steps)
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "µs/token/layer", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v * args.tokens / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(args), "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "µs/token/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_sweep(args):
    """GPU time per call of each recurrence mode against T: back-to-back calls
    captured in a CUDA graph and replayed (so host-side call overhead is not
    counted), medians of 3 replays; one layer, 48 value heads."""
    import torch

    from linear_attention_recurrence_gb300 import build, gdn
    from linear_attention_recurrence_gb300.inputs import make_inputs

    build.build()
    gdn.gdn_set_option("chunk_products", args.chunk_products)
    dev = torch.device("cuda", torch.cuda.current_device())
    Ts = [1, 8, 16, 32, 64, 96, 128, 192, 256, 512, 1024, 2048, 8192, 32768]
    x = make_inputs(max(Ts), seed=0, norm=False)
    t = {k: torch.from_numpy(v).to(dev) for k, v in x.items()}
    out = torch.empty((max(Ts), N_VH, D), device=dev)
    st = torch.empty_like(t["S0"])
    res = {}
    for T in Ts:
        reps = 20 if T <= 8192 else 5
        res[T] = {}
        for mode in ("sequential", "chunked"):
            def calls():
                for _ in range(reps):
                    gdn.gdn_recurrence(t["q"][:T], t["k"][:T], t["v"][:T], t["g"][:T], t["beta"][:T], st,
                                       out=out[:T], mode=mode)
            st.copy_(t["S0"])
            calls()  # warm-up (allocates the chunked scratch once)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                calls()
            samples = []
            for _ in range(3):
                st.copy_(t["S0"])
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                graph.replay()
                e1.record()
                torch.cuda.synchronize()
                samples.append(e0.elapsed_time(e1) * 1e3 / reps)
            res[T][mode] = statistics.median(samples)
    line = {"metric": "GDN recurrence GPU time per call (µs) by mode and T", "unit": "µs", "data": "synthetic",
            "config": {"n_kh": N_KH, "n_vh": N_VH, "d": D, "state": "carried, non-zero", "timing": "CUDA graph replay",
                       "chunk_products": args.chunk_products},
            "sweep": {str(T): v for T, v in res.items()}}
    print(json.dumps(line), flush=True)
    return 0


def make_stack_step(gdn, torch, dev, layers, mode):
    """One prefill step of a stack of independent layers (2048 tokens each):
    layer i's recurrence on the main stream, its FP16 norm on a second stream
    beside layer i+1's recurrence (two output buffers alternate, and a layer's
    recurrence waits for the norm that last read its buffer).  Returns step()."""
    T = layers[0]["q"].shape[0]
    states = [torch.empty_like(x["S0"]) for x in layers]
    outs = [torch.empty((T, N_VH, D), device=dev) for _ in range(2)]
    y = torch.empty((T, N_VH, D), device=dev, dtype=torch.float16)
    main, side = torch.cuda.current_stream(), torch.cuda.Stream(dev)

    def step():
        side.wait_stream(main)
        norm_done = [None, None]
        for i, (x, st) in enumerate(zip(layers, states)):
            o = outs[i % 2]
            if norm_done[i % 2] is not None:
                main.wait_event(norm_done[i % 2])
            st.copy_(x["S0"])
            gdn.gdn_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], st, out=o, mode=mode, stream=main)
            rec_done = torch.cuda.Event()
            rec_done.record(main)
            side.wait_event(rec_done)
            gdn.gdn_out_norm(o, x["z"], x["w"], 1e-6, y=y, stream=side)
            norm_done[i % 2] = torch.cuda.Event()
            norm_done[i % 2].record(side)
        main.wait_stream(side)

    return step


def run_stack(args):
    """A stack of L independent layers, 2048 tokens each (every layer its own seeded
    q/k/v/g/beta/S0/z/w), recurrence in the selected mode then the FP16 norm per
    layer: the whole-stack prefill time of one 2048-token prompt chunk."""
    import torch

    from linear_attention_recurrence_gb300 import build, gdn

    pool, pending = stack_inputs_async(args.stack)
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    L, T = args.stack, 2048
    layers = [{k: torch.from_numpy(v).to(dev) for k, v in x.items()} for x in pending.get()]
    pool.close()
    step = make_stack_step(gdn, torch, dev, layers, args.mode)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n0 = gdn.gdn_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index) as clk:
        time.sleep(0.5)
        wall0 = time.time()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        clk.mark(wall0, time.time())
        time.sleep(0.1)
    ms = e0.elapsed_time(e1) / args.steps
    assert gdn.gdn_device_status() == gdn.GDN_OK
    line = {"metric": "GDN prefill stack time, recurrence + norm (ms per 2048-token chunk)", "value": ms, "unit": "ms",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False, "dtype": "f32",
            "data": "synthetic", "us_per_token_layer": ms * 1e3 / (T * L),
            "step_schedule": "layer i's norm on a second stream beside layer i+1's recurrence",
            "config": {"workload": f"{L} independent layers x {T} tokens, recurrence + FP16 norm", "layers": L,
                       "T": T, "mode": args.mode, "n_kh": N_KH, "n_vh": N_VH, "d": D},
            "gpu_launches": gdn.gdn_launch_count() - n0, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args):
    """Batched decode: one token for each of B independent sequences (own states),
    48 value heads.  HBM-bound: every step reads and rewrites all states once."""
    import torch

    from linear_attention_recurrence_gb300 import build, gdn
    from linear_attention_recurrence_gb300.inputs import make_inputs

    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    B = args.decode
    x = make_inputs(B, seed=0, norm=False)  # token b of the draw is sequence b's input
    t = {k: torch.from_numpy(v).to(dev) for k, v in x.items() if k != "S0"}
    states = torch.from_numpy(x["S0"]).to(dev)[None].repeat(B, 1, 1, 1).contiguous()
    out = torch.empty((B, N_VH, D), device=dev)
    step = lambda: gdn.gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], states, out=out)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n0 = gdn.gdn_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index) as clk:
        time.sleep(0.5)
        wall0 = time.time()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        clk.mark(wall0, time.time())
        time.sleep(0.1)
    ms = e0.elapsed_time(e1) / args.steps
    assert gdn.gdn_device_status() == gdn.GDN_OK
    hbm_gbs, _, peak_src = _peaks()
    # algorithmic bytes per sequence: state read + write, q, k, v, g, beta, o
    bytes_step = B * (2 * N_VH * D * D * 4 + 2 * N_KH * D * 4 + 2 * N_VH * D * 4 + 2 * N_VH * 4)
    gbs = bytes_step / (ms * 1e-3) / 1e9
    line = {"metric": "GDN decode step µs (48 vh, d=128) and % of HBM roofline", "value": ms * 1e3, "unit": "µs/step",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False, "dtype": "f32",
            "data": "synthetic", "config": {"workload": f"decode, {B} sequences x 1 token", "batch": B, "n_kh": N_KH,
                                            "n_vh": N_VH, "d": D, "l2": f"states {B * 3} MB, read and written per step"},
            "gpu_launches": gdn.gdn_launch_count() - n0,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
                         "peak_basis": f"{peak_src} copy bandwidth",
                         "traffic": captured_traffic("gdn_decode.cu") if B == 64 else None},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    return 0


def run_prestage(args):
    """The pre-stage over T tokens of one layer in one call (causal conv of the
    packed qkv rows, SiLU, q/k L2 norms, gates).  HBM-bound: reads every qkv row
    once (plus three halo rows per 64-token run, mostly from L2) and writes q, k,
    v, g, beta once."""
    import torch

    from linear_attention_recurrence_gb300 import build, gdn
    from linear_attention_recurrence_gb300.inputs import make_prestage_inputs

    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    T = args.tokens
    x = make_prestage_inputs(T, seed=0)
    t = {k: torch.from_numpy(v).to(dev) for k, v in x.items()}
    cw = t["qkv"].shape[1]
    hist_out = torch.empty((3, cw), device=dev)
    res = gdn.gdn_prestage(t["qkv"], t["conv_w"], t["a"], t["b"], t["A_log"], t["dt_bias"], N_KH, N_VH,
                           hist_in=t["conv_hist"], hist_out=hist_out)
    step = lambda: gdn.gdn_prestage(t["qkv"], t["conv_w"], t["a"], t["b"], t["A_log"], t["dt_bias"],  # noqa: E731
                                    N_KH, N_VH, hist_in=t["conv_hist"], hist_out=hist_out, out=res)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # enough steps for about a second of timed work, so the clock sampler sees it
    t0 = time.time()
    for _ in range(10):
        step()
    torch.cuda.synchronize()
    steps = max(args.steps, int(1.0 / max((time.time() - t0) / 10, 1e-6)))
    n0 = gdn.gdn_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index) as clk:
        time.sleep(0.5)
        wall0 = time.time()
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        clk.mark(wall0, time.time())
        time.sleep(0.1)
    ms = e0.elapsed_time(e1) / steps
    hbm_gbs, _, peak_src = _peaks()
    bytes_tok = 2 * cw * 4 + 4 * N_VH * 4  # qkv in, q/k/v out; a, b in, g, beta out
    gbs = bytes_tok * T / (ms * 1e-3) / 1e9
    line = {"metric": "GDN pre-stage µs/token/layer (conv + norms + gates, 48 vh, d=128) and % of HBM roofline",
            "value": ms * 1e3 / T, "unit": "µs/token/layer", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "dtype": "f32",
            "data": "synthetic", "config": {"workload": f"pre-stage, 1 layer, T={T} in one call", "T": T,
                                            "n_kh": N_KH, "n_vh": N_VH, "d": D, "activation": "silu",
                                            "l2": f"inputs {T * cw * 4 / 1e9:.2f} GB, larger than L2"},
            "gpu_launches": gdn.gdn_launch_count() - n0,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
                         "peak_basis": f"{peak_src} copy bandwidth", "bytes_per_token": bytes_tok,
                         "traffic": captured_traffic("gdn_prestage.cu") if T == 32768 else None},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    return 0


def _config(args):
    return {"workload": f"gdn-prefill 1 layer, T={args.tokens} as {args.tokens // args.call_tokens} calls of "
                        f"{args.call_tokens} with the state carried, then the FP16 norm",
            "T": args.tokens, "tokens_per_call": args.call_tokens, "n_kh": N_KH, "n_vh": N_VH, "d": D,
            "mode": args.mode, "global_batch": 1, "seq_len": args.tokens,
            "l2": "inputs larger than L2 (q/k/v/z stream from HBM every step)",
            "parallelism": "replicas" if _dist()[0] > 1 else "single"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="chunked", choices=["chunked", "sequential"])
    ap.add_argument("--tokens", type=int, default=32768)
    ap.add_argument("--call-tokens", type=int, default=2048)
    ap.add_argument("--skip-cpu", action="store_true", help="no oracle timing")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--step-api", choices=["fused", "overlap", "plain"], default="overlap",
                    help="timed step: fused = gdn_recurrence_norm per call (the norm inside the recurrence's "
                         "launch); overlap = each call's rows normed on a second stream; plain = the calls, then "
                         "one norm")
    ap.add_argument("--prestage", action="store_true",
                    help="time the pre-stage (conv + norms + gates) over --tokens tokens in one call")
    ap.add_argument("--skip-other-mode", action="store_true")
    ap.add_argument("--skip-extra", action="store_true",
                    help="skip the T=8192 (both modes) and 36-layer stack measurements")
    ap.add_argument("--chunk-products", default="tmem", choices=["mma", "fma", "tc", "tmem"],
                    help="how the chunked form computes its products (library option chunk_products)")
    ap.add_argument("--prep-ctas", type=int, default=0,
                    help="tensor-memory chunked form: CTAs running the prep beside the scan (library option "
                         "chunk_prep_ctas; 0 = the library's choice)")
    ap.add_argument("--no-fp32-out", action="store_true",
                    help="with --step-api fused: the FP32 output is not stored (the norm in the scan's epilogue: "
                         "sequential mode, and the tensor-memory chunked form)")
    ap.add_argument("--norm-in-launch", action="store_true",
                    help="with --step-api fused: the norm inside the recurrence's launch (library option "
                         "norm_in_launch; sequential mode: the scan's fused epilogue)")
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", action="store_true",
                    help="time one call of each mode for T = 1 .. 32768 (one JSON line) instead of the step")
    ap.add_argument("--stack", type=int, default=0, metavar="L",
                    help="time L independent layers x 2048 tokens (recurrence + norm per layer, one JSON line)")
    ap.add_argument("--decode", type=int, default=0, metavar="B",
                    help="time the batched decode step for B sequences (one JSON line) instead of the prefill step")
    args = ap.parse_args()
    if args.sweep:
        return run_sweep(args)
    if args.prestage:
        return run_prestage(args)
    if args.decode:
        return run_decode(args)
    if args.stack:
        return run_stack(args)
    assert args.tokens % args.call_tokens == 0
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from linear_attention_recurrence_gb300 import build, gdn
    from linear_attention_recurrence_gb300.inputs import make_inputs

    ws, rank, local = _dist()
    want_extra = ws == 1 and not args.skip_extra
    stack_pool = stack_inputs_async(36) if want_extra else None
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0 or ws == 1:
        build.build()
    if ws > 1:
        dist.barrier()
    gdn.load_library()
    gdn.gdn_set_option("chunk_products", args.chunk_products)
    gdn.gdn_set_option("chunk_prep_ctas", args.prep_ctas)
    gdn.gdn_set_option("norm_in_launch", 1 if args.norm_in_launch else 0)

    T, CT = args.tokens, args.call_tokens
    ncalls = T // CT
    x = make_inputs(T, seed=0, layer=rank)
    h = {k: torch.from_numpy(v).pin_memory() for k, v in x.items()}
    t = {k: v.to(dev, non_blocking=True) for k, v in h.items()}
    state = torch.empty_like(t["S0"])
    out = torch.empty((T, N_VH, D), device=dev)
    y = torch.empty((T, N_VH, D), device=dev, dtype=torch.float16)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    norm_stream = torch.cuda.Stream(dev)

    def overlapped_step(mode):
        """The same work as step(): each call's rows are normed on a second stream as
        soon as that call has finished, beside the next call's recurrence (the norm
        is HBM-bound, the recurrence ALU-bound)."""
        state.copy_(t["S0"])
        norm_stream.wait_stream(stream)
        for i in range(ncalls):
            a, b = i * CT, (i + 1) * CT
            gdn.gdn_recurrence(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], state,
                               out=out[a:b], mode=mode, stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            norm_stream.wait_event(done)
            gdn.gdn_out_norm(out[a:b], t["z"][a:b], t["w"], 1e-6, y=y[a:b], stream=norm_stream)
        stream.wait_stream(norm_stream)

    def fused_step(mode):
        """The same work as step(), each call through gdn_recurrence_norm: the
        recurrence and the norm of its rows in one call (in chunked mode, inside the
        one launch)."""
        state.copy_(t["S0"])
        for i in range(ncalls):
            a, b = i * CT, (i + 1) * CT
            gdn.gdn_recurrence_norm(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], state,
                                    t["z"][a:b], t["w"], 1e-6, out=out[a:b], y=y[a:b], mode=mode, stream=stream,
                                    store_out=not args.no_fp32_out)

    def step(mode, ev=None):
        if ev is None and args.step_api == "fused":
            return fused_step(mode)
        if ev is None and args.step_api == "overlap":
            return overlapped_step(mode)
        state.copy_(t["S0"])
        for i in range(ncalls):
            a, b = i * CT, (i + 1) * CT
            if ev is not None:
                ev[0].append(torch.cuda.Event(enable_timing=True))
                ev[0][-1].record(stream)
            gdn.gdn_recurrence(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], state,
                               out=out[a:b], mode=mode, stream=stream)
            if ev is not None:
                ev[1].append(torch.cuda.Event(enable_timing=True))
                ev[1][-1].record(stream)
        if ev is not None:
            ev[2].append(torch.cuda.Event(enable_timing=True))
            ev[2][-1].record(stream)
        gdn.gdn_out_norm(out, t["z"], t["w"], 1e-6, y=y, stream=stream)
        if ev is not None:
            ev[3].append(torch.cuda.Event(enable_timing=True))
            ev[3][-1].record(stream)

    def timed(mode, steps, warmup, per_kernel, clk=None):
        for _ in range(warmup):
            step(mode)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.time()
        ev = ([], [], [], []) if per_kernel else None
        n0 = gdn.gdn_launch_count()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(mode, ev)
        e1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        launches = gdn.gdn_launch_count() - n0
        if clk is not None:
            clk.mark(wall0, time.time())
        step_ms, _, _ = aggregate(e0.elapsed_time(e1) / steps, T, ws, device=dev)
        res = {"ms_per_step": step_ms, "launches": launches}
        if per_kernel:
            rec = [a.elapsed_time(b) for a, b in zip(ev[0], ev[1])]
            nrm = [a.elapsed_time(b) for a, b in zip(ev[2], ev[3])]
            res["rec_call_ms"] = statistics.mean(rec)
            res["rec_ms_per_step"] = sum(rec) / steps
            res["norm_ms"] = statistics.mean(nrm)
        return res

    def timed_alternating(modes, rounds):
        """Per-call CUDA-event times of the recurrence and of the norm for each mode,
        the modes' steps alternating (the last one of each round is modes[-1]);
        medians over the rounds."""
        for mode in modes:
            step(mode)
        torch.cuda.synchronize()
        per = {m: {"rec": [], "step": [], "norm": [], "launches": 0} for m in modes}
        for _ in range(rounds):
            for mode in modes:
                ev = ([], [], [], [])
                n0 = gdn.gdn_launch_count()
                step(mode, ev)
                torch.cuda.synchronize()
                per[mode]["launches"] += gdn.gdn_launch_count() - n0
                rec = [a.elapsed_time(b) for a, b in zip(ev[0], ev[1])]
                per[mode]["rec"] += rec
                per[mode]["step"].append(sum(rec))
                per[mode]["norm"] += [a.elapsed_time(b) for a, b in zip(ev[2], ev[3])]
        return {m: {"rec_call_ms": statistics.median(r["rec"]), "rec_ms_per_step": statistics.median(r["step"]),
                    "norm_ms": statistics.median(r["norm"]), "launches": r["launches"] / rounds * args.steps}
                for m, r in per.items()}

    def time_c3(rounds=20):
        """The T = 8192 configuration: one call per mode (then the norm of its 8192
        rows), the modes alternating, L2 flushed before every call (the 8192-token
        inputs would fit in it); medians over `rounds` after one warm-up round."""
        T3 = 8192
        flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MB, twice the L2
        st = torch.empty_like(t["S0"])
        res = {m: {"rec": [], "norm": []} for m in ("sequential", "chunked")}
        for r in range(rounds + 1):
            for mode in ("sequential", "chunked"):
                st.copy_(t["S0"])
                flush.zero_()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(stream)
                gdn.gdn_recurrence(t["q"][:T3], t["k"][:T3], t["v"][:T3], t["g"][:T3], t["beta"][:T3], st,
                                   out=out[:T3], mode=mode, stream=stream)
                e[1].record(stream)
                gdn.gdn_out_norm(out[:T3], t["z"][:T3], t["w"], 1e-6, y=y[:T3], stream=stream)
                e[2].record(stream)
                torch.cuda.synchronize()
                if r > 0:
                    res[mode]["rec"].append(e[0].elapsed_time(e[1]))
                    res[mode]["norm"].append(e[1].elapsed_time(e[2]))
        out_c3 = {}
        for mode, r in res.items():
            rec, nrm = statistics.median(r["rec"]), statistics.median(r["norm"])
            flop = FLOP_SEQ if mode == "sequential" else FLOP_CHUNKED
            out_c3[mode] = {"recurrence_ms": rec, "norm_ms": nrm, "us_per_token_layer": (rec + nrm) * 1e3 / T3,
                            "recurrence_us_per_token_layer": rec * 1e3 / T3,
                            "alu_tflops": flop * T3 / (rec * 1e-3) / 1e12}
        return out_c3

    other = "sequential" if args.mode == "chunked" else "chunked"
    clk = Clocks(dev.index).__enter__()
    time.sleep(0.5)  # nvidia-smi's first samples
    main_res = timed(args.mode, args.steps, args.warmup, per_kernel=False, clk=clk)
    time.sleep(0.1)
    y_main = y.clone()
    wall0 = time.time()
    alt = timed_alternating(([] if args.skip_other_mode else [other]) + [args.mode], args.steps)
    clk.add_window(wall0, time.time())
    kern = alt[args.mode]
    other_res = alt.get(other)
    torch.cuda.synchronize()
    assert torch.equal(y_main, y), "the overlapped step's output differs from the plain step's"
    c3 = None
    if want_extra:
        wall0 = time.time()
        c3 = time_c3()
        clk.add_window(wall0, time.time())
    assert gdn.gdn_device_status() == gdn.GDN_OK

    # end to end through the public API with host buffers: every step copies its inputs
    # from pinned host memory and reads the FP16 output and the final state back, inside
    # the timed region.  The copies are pipelined per call: a copy-in stream brings call
    # i+1's rows (q, k, v, g, beta, z) while the compute stream runs call i (recurrence,
    # then the norm of its rows) and a copy-out stream returns call i-1's y rows.  The
    # device inputs and y are double-buffered across steps, so step k+1's rows start
    # landing while step k still computes (the host link is the bound).
    e2e = None
    if not args.skip_e2e:
        hy = torch.empty((T, N_VH, D), dtype=torch.float16).pin_memory()
        hs = torch.empty_like(h["S0"]).pin_memory()
        row_names = ["q", "k", "v", "g", "beta", "z"]
        h2d = sum(h[n].numel() * h[n].element_size() for n in row_names + ["S0", "w"])
        d2h = hy.numel() * 2 + hs.numel() * 4
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        tb = [t, {n: torch.empty_like(t[n]) for n in row_names + ["S0", "w"]}]
        yb = [y, torch.empty_like(y)]
        inputs_free = [None, None]  # compute of the last step that read this input set is done
        y_free = [None, None]       # copy-out of the last step that wrote this y is done
        last_out = [None]           # the previous step's copy-outs (state included) are done

        def e2e_step(k):
            ti, yi = tb[k % 2], yb[k % 2]
            if inputs_free[k % 2] is not None:
                s_in.wait_event(inputs_free[k % 2])
            landed = []
            with torch.cuda.stream(s_in):
                ti["S0"].copy_(h["S0"], non_blocking=True)
                ti["w"].copy_(h["w"], non_blocking=True)
                for i in range(ncalls):
                    a, b = i * CT, (i + 1) * CT
                    for n in row_names:
                        ti[n][a:b].copy_(h[n][a:b], non_blocking=True)
                    landed.append(torch.cuda.Event())
                    landed[-1].record(s_in)
            stream.wait_event(landed[0])
            for ev in (last_out[0], y_free[k % 2]):
                if ev is not None:
                    stream.wait_event(ev)
            state.copy_(ti["S0"])
            for i in range(ncalls):
                a, b = i * CT, (i + 1) * CT
                stream.wait_event(landed[i])
                gdn.gdn_recurrence(ti["q"][a:b], ti["k"][a:b], ti["v"][a:b], ti["g"][a:b], ti["beta"][a:b], state,
                                   out=out[a:b], mode=args.mode, stream=stream)
                gdn.gdn_out_norm(out[a:b], ti["z"][a:b], ti["w"], 1e-6, y=yi[a:b], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    hy[a:b].copy_(yi[a:b], non_blocking=True)
            inputs_free[k % 2] = torch.cuda.Event()
            inputs_free[k % 2].record(stream)
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_out):
                hs.copy_(state, non_blocking=True)
            last_out[0] = torch.cuda.Event()
            last_out[0].record(s_out)
            y_free[k % 2] = last_out[0]

        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)  # no copy of the timed steps starts before the clock does
        for k in range(2, 2 + args.steps):
            e2e_step(k)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        ms, e2e_us, _ = aggregate(e0.elapsed_time(e1) / args.steps, T, ws, device=dev)
        e2e = {"value": e2e_us, "unit": "µs/token/layer", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms,
               "pipelining": f"per {CT}-token call: copy-in, compute (recurrence + norm of its rows), copy-out, "
                             "on separate streams; inputs and y double-buffered across steps"}
        y_last = yb[(1 + args.steps) % 2].clone()
        # the pipelined step must give the bits of the plain one
        step(args.mode)
        torch.cuda.synchronize()
        assert torch.equal(y_last, y), "pipelined end-to-end step differs from the plain step"
        assert torch.equal(hy, y.cpu()) and torch.equal(hs, state.cpu())

    # the 36-layer stack (36 independent layers x 2048 tokens, recurrence + norm per
    # layer, each layer's own seeded inputs, drawn on the host cores meanwhile)
    c5 = None
    if stack_pool is not None:
        pool, pending = stack_pool
        layers = [{k: torch.from_numpy(v).to(dev) for k, v in xl.items()} for xl in pending.get()]
        pool.close()
        stack_step = make_stack_step(gdn, torch, dev, layers, args.mode)
        for _ in range(2):
            stack_step()
        torch.cuda.synchronize()
        wall0 = time.time()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_stack = 5
        e0.record()
        for _ in range(n_stack):
            stack_step()
        e1.record()
        torch.cuda.synchronize()
        clk.add_window(wall0, time.time())
        ms5 = e0.elapsed_time(e1) / n_stack
        c5 = {"ms": ms5, "us_per_token_layer": ms5 * 1e3 / (36 * 2048), "mode": args.mode, "steps": n_stack,
              "workload": "36 independent layers x 2048 tokens, recurrence + FP16 norm per layer (each layer its "
                          "own seeded inputs; layer i's norm on a second stream beside layer i+1's recurrence)"}
        del layers
        assert gdn.gdn_device_status() == gdn.GDN_OK
    time.sleep(0.1)
    clk.__exit__(None, None, None)

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    hbm_gbs, sm_mhz_max, peak_src = _peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak_tflops = sms * FP32_LANES_PER_SM * 2 * sm_mhz_max * 1e6 / 1e12
    clocks = clk.summary()

    def mode_summary(mode, r):
        flop = FLOP_SEQ if mode == "sequential" else FLOP_CHUNKED
        achieved = flop * CT / (r["rec_call_ms"] * 1e-3) / 1e12
        return {"us_per_token_layer": r["rec_ms_per_step"] * 1e3 / T,
                "recurrence_call_ms": r["rec_call_ms"], "norm_ms": r["norm_ms"],
                "alu_tflops": achieved, "alu_frac": achieved / alu_peak_tflops,
                "launches_per_step": r["launches"] / args.steps}

    modes = {args.mode: mode_summary(args.mode, kern)}
    if other_res is not None:
        modes[other] = mode_summary(other, other_res)
    flop = FLOP_SEQ if args.mode == "sequential" else FLOP_CHUNKED
    achieved = flop * CT / (kern["rec_call_ms"] * 1e-3) / 1e12
    per_call = (kern["launches"] / args.steps - 1) / ncalls  # the norm is one launch per step
    scan_kind = args.chunk_products
    products = {"fma": "products as packed FP32 FMAs",
                "tc": "S0 products as split-TF32 tcgen05 MMAs",
                "mma": "products as split-TF32 mma.sync MMAs"}.get(
                    scan_kind, "state in tensor memory, every product a split-TF32 tcgen05 MMA")
    one_launch = per_call < 1.5
    tmem = scan_kind == "tmem" and one_launch
    if tmem:
        chunk_label = "gdn_chunk_tmem_kernel (prep and one scan CTA per value head in one launch) per 2048-token call"
    else:
        chunk_label = ("gdn_chunk_fused_kernel (prep and scan in one launch) per 2048-token call" if one_launch
                       else "gdn_chunk_prep_kernel + gdn_chunk_scan_kernel per 2048-token call")
    chunk_label += ", " + products
    # the captures in profiles/ are of the one-launch kernels (tensor-memory and warp-MMA forms)
    chunk_src = "gdn_chunk_tmem.cu" if tmem else "gdn_chunk.cu"
    chunk_traffic = captured_traffic(chunk_src) if one_launch and scan_kind in ("mma", "tmem") else None
    norm_gbs = BYTES_NORM * T / (kern["norm_ms"] * 1e-3) / 1e9
    counts = captured_counts(chunk_src if args.mode == "chunked" else "gdn_seq.cu")
    if args.mode == "chunked" and not (one_launch and scan_kind in ("mma", "tmem")):
        counts = None  # the captures are of the one-launch kernels
    counted = None
    if counts is not None:
        call_s = kern["rec_call_ms"] * 1e-3
        tf32_peak, tf32_basis = _tf32_peak()
        counted = {"fp32_flop_per_call": counts["fp32_flop"], "tensor_flop_per_call": counts["tensor_flop"],
                   "fp32_tflops": counts["fp32_flop"] / call_s / 1e12,
                   "tensor_tflops": counts["tensor_flop"] / call_s / 1e12,
                   "tensor_frac_of_tf32_peak": counts["tensor_flop"] / call_s / 1e12 / tf32_peak,
                   "tf32_peak_tflops": tf32_peak, "tf32_peak_basis": tf32_basis,
                   "source": "ncu thread-instruction counts of one 2048-token launch (profiles/flop_counts.md) "
                             "at this run's median call time"}
    value = main_res["ms_per_step"] * 1e3 / (T * ws)  # already the max over ranks
    line = {
        "metric": METRIC, "value": value, "unit": "µs/token/layer", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"], "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(args),
        "tokens_per_s": T * ws / (main_res["ms_per_step"] * 1e-3),
        "step_schedule": {"fused": "16 gdn_recurrence_norm calls (recurrence + norm of the call's rows"
                                   + (", no FP32 output)" if args.no_fp32_out else ")"),
                          "overlap": "16 recurrence calls on one stream; each call's rows normed on a second "
                                     "stream once that call is done",
                          "plain": "16 recurrence calls, then the norm"}[args.step_api],
        "gpu_launches": main_res["launches"],
        "roofline": {"bound": "alu", "achieved": achieved, "peak": alu_peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / alu_peak_tflops,
                     "traffic": chunk_traffic if args.mode == "chunked" else captured_traffic("gdn_seq.cu"),
                     "kernel": chunk_label if args.mode == "chunked" else "gdn_seq_kernel per 2048-token call",
                     "peak_basis": f"{sms} SMs x 128 FP32 lanes x 2 x {sm_mhz_max:.0f} MHz ({peak_src} max clock)",
                     "frac_at_observed_clock": (achieved / (sms * FP32_LANES_PER_SM * 2 * clocks["sm_mhz"] * 1e6
                                                            / 1e12)) if clocks.get("sm_mhz") else None,
                     "counted": counted},
        "norm_roofline": {"bound": "hbm", "achieved": norm_gbs, "peak": hbm_gbs, "unit": "GB/s",
                          "frac": norm_gbs / hbm_gbs, "peak_basis": f"{peak_src} copy bandwidth"},
        "modes": modes,
        "modes_timing": "per-call CUDA events on the launching stream, the two modes' steps alternating, medians "
                        f"over {args.steps} steps",
        "clocks": clocks,
        "clocks_all_passes": clk.summary(all_windows=True),
    }
    if c3 is not None:
        for mode, r in c3.items():
            r["alu_frac"] = r["alu_tflops"] / alu_peak_tflops
        line["c3_t8192"] = dict(c3, timing="one 8192-token call per mode then the norm of its rows, modes "
                                           "alternating, L2 flushed before each call, medians over 20 runs")
    if c5 is not None:
        line["c5_stack36"] = c5
    if e2e is not None:
        line["e2e"] = e2e
    if not args.skip_cpu and ws == 1:
        line["cpu_baseline"] = oracle_t8192()
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
