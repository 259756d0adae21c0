#!/usr/bin/env python
"""Throughput of the masked post-LN encoder stack forward on GB300.

One step = one forward of the whole stack (every layer: fused QKV, masked
attention, out-projection + residual + LayerNorm, FFN with exact GELU,
residual + LayerNorm) over one batch of synthetic inputs already resident in
HBM.  The headline workload is the 4-layer d_model=128 encoder on 4096
sequences of 64 tokens, fp16 I/O.  Prints ONE JSON line (rank 0); its
``per_workload`` object times the same forward on every one of the five
synthetic workloads (configs of the pages' task), each with its dominant
kernel's roofline fraction and the gate's envelope utilisation on a sample of
the timed output.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 is launched by torch.distributed.run, one rank per GPU; every rank runs
its own batch (sequences are independent: weak scaling, no collective on the
data path) and the step time is the max over ranks.  ``--impl reference``
times the fp64 CPU oracle on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "encoder forward tokens/s on 1 GB300 (masked); % of tensor/HBM roofline"
DEFAULT_WORKLOAD = "short_d128_L64_B4096"
WORKLOADS = ("tiny_d32_L32", "short_d128_L64_B4096", "batch1_d256_L512",
             "wide_d1024_L1024_B32", "long_d64_L100k_B8")
# Timed steps per workload in the per-workload table (the headline uses --steps).
PER_WORKLOAD_STEPS = {"tiny_d32_L32": 50, "short_d128_L64_B4096": 30, "batch1_d256_L512": 50,
                      "wide_d1024_L1024_B32": 20, "long_d64_L100k_B8": 5}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def sum_visible_keys(valid_len, L):
    """sum over sequences and query rows of min(i + 1, valid_len)."""
    tot = 0
    for v in np.asarray(valid_len, dtype=np.int64):
        v = int(v)
        tot += v * (v + 1) // 2 + (L - v) * v
    return tot


def algorithmic_counts(shape, valid_len):
    """Flops and minimal HBM bytes of one forward (what the method must do)."""
    T, d, dff, nl = shape.tokens, shape.d_model, shape.d_ff, shape.n_layers
    es = 4 if shape.dtype == "f32" else 2
    keys = sum_visible_keys(valid_len, shape.seq_len)
    per_layer = {
        "qkv": 2.0 * T * 3 * d * d,
        "attention": 4.0 * d * keys,
        "out": 2.0 * T * d * d,
        "ffn1": 2.0 * T * d * dff,
        "ffn2": 2.0 * T * dff * d,
    }
    weights = nl * ((4 * d * d + 2 * d * dff) * es + (3 * d + d + 4 * d + dff + d) * es)
    return {
        "flops_per_layer": per_layer,
        "flops": nl * sum(per_layer.values()),
        "hbm_bytes": 2 * T * d * es + weights + 4 * shape.batch,
        "visible_keys": keys,
        # transcendental evaluations: one exponential per visible score, one
        # erf per FFN hidden value
        "sfu_ops": nl * (keys * shape.n_heads + T * dff),
    }


# SFU base-2 exponentials per SM per clock on GB300: 32.  A throughput loop of
# independent ex2.approx.ftz.f32 chains (608 blocks of 512 threads) ran
# 9.48e12 per second on 152 SMs at about 2.0 GHz, 30 per SM per clock: twice
# the 4 per SM sub-partition assumed before.
SFU_PER_SM_CLK = 32


def fp32_alu_tflops(peaks, sms):
    """FP32 FMA peak derived from unit counts: SMs x 128 lanes x 2 flops x
    max SM clock."""
    return sms * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def step_fractions(counts, ms_per_step, peaks, sms, dtype):
    """The whole step's algorithmic work over the rooflines that apply to the
    path: the tensor cores (16-bit I/O; measured bf16 burst peak, fp16 dense
    runs at the same rate) or the FP32 ALUs (fp32 I/O runs on the CUDA
    cores), HBM (measured copy bandwidth) and the SFU (SMs x 32 x max
    clock).  The largest is the binding one."""
    t = ms_per_step / 1e3
    clk = peaks.get("sm_max_mhz", 2070.0) * 1e6
    f = {}
    if dtype == "f32":
        f["fp32_alu"] = counts["flops"] / t / (fp32_alu_tflops(peaks, sms) * 1e12)
    else:
        f["tensor"] = counts["flops"] / t / (peaks["bf16_tflops"] * 1e12)
    f["hbm"] = counts["hbm_bytes"] / t / (peaks["hbm_gbs"] * 1e9)
    f["sfu"] = counts["sfu_ops"] / t / (sms * SFU_PER_SM_CLK * clk)
    f["binding"] = max(f, key=f.get)
    return f


# Kernel class -> (bound, algorithmic work per launch) for the roofline line.
def kernel_work(cls, shape, counts):
    pl = counts["flops_per_layer"]
    T, d = shape.tokens, shape.d_model
    table = {
        "simt_gemm_qkv": ("alu", pl["qkv"]), "simt_attention": ("alu", pl["attention"]),
        "simt_gemm_out": ("alu", pl["out"]), "simt_gemm_ffn1": ("alu", pl["ffn1"]),
        "simt_gemm_ffn2": ("alu", pl["ffn2"]),
        "simt_layernorm": ("hbm", 2.0 * T * d * 4),
        "tc_gemm_qkv": ("tensor", pl["qkv"]), "tc_attention": ("tensor", pl["attention"]),
        "tc_gemm_out_ln": ("tensor", pl["out"]), "tc_gemm_ffn1": ("tensor", pl["ffn1"]),
        "tc_gemm_ffn2_ln": ("tensor", pl["ffn2"]),
        "megakernel": ("tensor", counts["flops"]),
        "dag": ("alu", counts["flops"]),
        "megakernel_simt": ("alu", counts["flops"]),
        # per launch, averaged over the 2 per layer: read the fp32 pre-LN rows
        # and row stats, write (hi, lo) planes (the last: the 16-bit output)
        "ln_apply": ("hbm", ((2 * shape.n_layers - 1) * (T * d * 8 + T * 8) + (T * d * 6 + T * 8))
                     / (2 * shape.n_layers)),
    }
    return table.get(cls)


def traffic_entry(cls, workload):
    """The committed ncu DRAM figures of kernel class `cls` on `workload`
    (an entry "cls@workload", else "cls"), if they were taken on the current
    kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        t = json.load(f)
    e = t.get(f"{cls}@{workload}") or t.get(cls)
    if not e or e.get("workload", workload) != workload:
        return None
    src = os.path.join(ROOT, "transformer_encoder_layer_gb300", "csrc", e["source"])
    if not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return e if sha == e["source_sha"] else None


def traffic_from_profiles(cls, workload):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch, or None."""
    e = traffic_entry(cls, workload)
    return e["dram_bytes_per_launch"] if e else None


def kernel_roofline(per_kernel, shape, counts, peaks, sms, total_ms):
    """The dominant kernel's algorithmic work per launch over its average
    event-timed launch duration, against the peak of the unit that bounds it
    (tensor: measured bf16 burst peak; HBM: measured copy bandwidth; FP32
    ALU: derived from unit counts and the max clock)."""
    if not per_kernel:
        return None
    dom = max(per_kernel, key=lambda k: per_kernel[k][0])
    ms, n = per_kernel[dom]
    bound, work = kernel_work(dom, shape, counts) or ("tensor", counts["flops"])
    avg_s = ms / n / 1e3
    if bound == "hbm":
        achieved, peak, unit, src = work / avg_s / 1e9, peaks["hbm_gbs"], "GB/s", peaks["source"]
    elif bound == "alu":
        achieved, peak, unit = work / avg_s / 1e12, fp32_alu_tflops(peaks, sms), "TFLOP/s"
        src = "derived: SMs x 128 FP32 lanes x 2 x max SM clock"
    else:
        achieved, peak, unit = work / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        src = peaks["source"] + " bf16 burst (fp16 dense runs at the bf16 rate)"
    te = traffic_entry(dom, shape.name)
    return {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": te["dram_bytes_per_launch"] if te else None,
            # output bytes the kernel leaves dirty in L2 reach DRAM after it ends
            "traffic_with_l2_writeback": te.get("dram_bytes_with_writeback") if te else None,
            "peak_source": src, "share_of_step": ms / total_ms if total_ms else None,
            "launches": n, "avg_launch_ms": ms / n}


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except (ValueError, IndexError):
                continue
            try:
                pw.append(float(f[2]))
            except (ValueError, IndexError):
                pass
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest of every rank's `value` (the job ends when its slowest
    rank does); `value` itself when not distributed."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world_size, tokens_per_rank, ms_per_step):
    """Weak scaling: every rank runs its own batch of the workload, so the job
    processes world_size x tokens_per_rank tokens per step."""
    return world_size * tokens_per_rank / (ms_per_step / 1e3)


def percentile(v, q):
    return float(np.percentile(np.asarray(v, dtype=np.float64), q))


def run_reference(args, shape):
    """The fp64 CPU oracle as the reference arm: each step is a bounded
    sample of the same workload (the first `ref_seqs` sequences)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from transformer_encoder_layer_gb300.inputs import make_inputs
    n = min(args.ref_seqs, shape.batch)
    inp = make_inputs(shape, seed=0, input_scale=1.0, batch=n)
    for _ in range(args.warmup):
        oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, shape.n_heads, check=False)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, shape.n_heads, check=False)
        times.append(time.perf_counter() - t0)
    tok = n * shape.seq_len
    value = tok * len(times) / sum(times)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name, "sample_sequences": n, "seq_len": shape.seq_len},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {shape.batch} sequences ({tok} tokens) per step, "
                                   f"numpy fp64 oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(shape, n_seqs):
    import oracle
    from transformer_encoder_layer_gb300.inputs import make_inputs
    n = min(n_seqs, shape.batch)
    inp = make_inputs(shape, seed=0, input_scale=1.0, batch=n)
    t0 = time.perf_counter()
    oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, shape.n_heads, check=False)
    dt = time.perf_counter() - t0
    tok = n * shape.seq_len
    return {"value": tok / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {n} of {shape.batch} sequences ({tok} tokens), numpy fp64 oracle, "
                      f"{dt:.1f} s"}


def envelope_on_sample(inp, out_np):
    """The gate's envelope utilisation of a timed output against the oracle,
    on a sample the oracle finishes in seconds: whole sequences where the
    workload allows (sequences are independent), else, at 100k tokens, the
    causal prefix of 2048 rows (rows < P see only tokens < P when every
    valid_len > P)."""
    import oracle
    from transformer_encoder_layer_gb300.gate import gate
    s = inp.shape
    if s.seq_len > 8192:
        P = 2048
        assert int(inp.valid_len.min()) > P
        ref = oracle.encoder_forward(inp.x[:, :P], np.full(s.batch, P), inp.layers, s.n_heads,
                                     check=False)
        ok, util, _ = gate(out_np[:, :P], ref)
        return {"utilisation": util, "passed": ok,
                "sample": f"rows < {P} of all {s.batch} sequences (causal prefix)"}
    n = max(1, min(s.batch, 16, (1 << 16) // (s.seq_len * max(1, s.d_model // 64))))
    ref = oracle.encoder_forward(inp.x[:n], inp.valid_len[:n], inp.layers, s.n_heads, check=False)
    ok, util, _ = gate(out_np[:n], ref)
    return {"utilisation": util, "passed": ok, "sample": f"first {n} of {s.batch} sequences"}


class Workload:
    """One workload's encoder, device buffers and pinned host copies."""

    def __init__(self, shape, seed, dev, path="auto", attention_split=-1, gemm_pairs=-1,
                 graphs=False, mega_assist=-1):
        import torch
        from transformer_encoder_layer_gb300 import binding
        from transformer_encoder_layer_gb300.inputs import make_inputs, to_storage
        self.shape = shape
        self.inp = make_inputs(shape, seed=seed, input_scale=1.0)
        self.counts = algorithmic_counts(shape, self.inp.valid_len)
        self.enc = binding.Encoder(self.inp.layers, shape.d_model, shape.n_heads, shape.d_ff,
                                   shape.dtype)
        if path != "auto":
            self.enc.set_path(path)
        self.enc.set_attention_split(attention_split)
        self.enc.set_gemm_pairs(gemm_pairs)
        self.enc.set_graphs(graphs)
        self.enc.set_mega_assist(mega_assist)
        self.graphs = bool(graphs)
        self.path = self.enc.plan(shape.batch, shape.seq_len)
        self.attention_split = self.enc.attention_split(shape.batch, shape.seq_len)
        xs = to_storage(self.inp.x, shape.dtype)
        if shape.dtype == "bf16":
            x_host = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16)
        else:
            x_host = torch.from_numpy(xs)
        self.x_host = x_host.contiguous().pin_memory()
        self.vl_host = torch.from_numpy(self.inp.valid_len.astype(np.int32)).pin_memory()
        self.x = self.x_host.to(dev)
        self.vl = self.vl_host.to(dev)
        self.out = torch.empty_like(self.x)
        wsz = self.enc.workspace_size(shape.batch, shape.seq_len)
        self.work = torch.empty(max(wsz, 256), dtype=torch.uint8, device=dev)

    def step(self, stream):
        self.enc.forward(self.x, self.vl, out=self.out, workspace=self.work, stream=stream, check=False)

    def out_f64(self):
        import torch
        from transformer_encoder_layer_gb300.inputs import from_storage
        o = self.out.cpu()
        if self.shape.dtype == "bf16":
            return from_storage(o.view(torch.int16).numpy().view(np.uint16), "bf16")
        return from_storage(o.numpy(), self.shape.dtype)

    def close(self):
        self.enc.close()


def time_steps(w, steps, warmup, flush, stream, dist=None, clock_index=None):
    """W warm-up steps, then K timed steps with an L2 flush (a 256 MB write)
    before each, timed by CUDA events on the launch stream, with the
    library's per-launch event timer on.  Returns per-step ms, per-kernel
    (ms, launches), the host wall time of the timed region and the clocks
    sampled during it."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        w.step(stream)
    torch.cuda.synchronize()
    if w.enc.get_status() != 0:
        raise RuntimeError(f"{w.shape.name}: device status error during warm-up")
    # (graph mode replays whole forwards; the per-launch timer would bypass it)
    if not w.graphs:
        w.enc.enable_timing(True, capacity=max(4096, 64 * steps * w.shape.n_layers))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(clock_index) if clock_index is not None else None
    if clk:
        clk.__enter__()
    t_wall0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()  # L2 flush between timed steps (outside the events)
        starts[i].record(stream)
        w.step(stream)
        stops[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if clk:
        clk.__exit__(None, None, None)
    if dist:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, stops)]
    per_kernel = {} if w.graphs else w.enc.read_timing()
    w.enc.enable_timing(False)
    if w.enc.get_status() != 0:
        raise RuntimeError(f"{w.shape.name}: device status error in the timed region")
    return step_ms, per_kernel, t_wall, (clk.summary() if clk else None)


def first_calls(workloads):
    """First-call time of each workload in a fresh process (the pages' harness
    runs every measurement in a new process): create the encoder, then the
    host wall time of its first forward up to the stream synchronisation.
    Workloads run in the given order in one child process, so the first entry
    also pays the library's module load."""
    cmd = [sys.executable, os.path.abspath(__file__), "--first-call-probe", ",".join(workloads)]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
        for ln in r.stdout.splitlines()[::-1]:
            if ln.startswith("{"):
                return json.loads(ln)
    except (subprocess.TimeoutExpired, OSError, ValueError):
        pass
    return None


def first_call_probe(names):
    import torch
    from transformer_encoder_layer_gb300.inputs import SHAPES
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    out = {}
    for name in names.split(","):
        w = Workload(SHAPES[name], 0, dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        w.step(torch.cuda.current_stream())
        torch.cuda.synchronize()
        out[name] = 1e3 * (time.perf_counter() - t0)
        w.close()
    print(json.dumps(out), flush=True)


def per_workload_entry(w, step_ms, per_kernel, peaks, sms, env, first_ms):
    s = w.shape
    med = statistics.median(step_ms)
    total = sum(step_ms)
    return {
        "path": w.path, "steps": len(step_ms),
        "ms_per_forward": {"median": med, "p10": percentile(step_ms, 10),
                           "p90": percentile(step_ms, 90), "mean": statistics.mean(step_ms)},
        "tokens_per_s": s.tokens / (med / 1e3),
        "valid_tokens_per_s": int(w.inp.valid_len.sum()) / (med / 1e3),
        "algorithmic_tflop_per_s": w.counts["flops"] / (med / 1e3) / 1e12,
        "roofline": kernel_roofline(per_kernel, s, w.counts, peaks, sms, total),
        "step_fractions": step_fractions(w.counts, med, peaks, sms, s.dtype),
        "per_kernel_ms": {k: v[0] / len(step_ms) for k, v in per_kernel.items()},
        "gpu_launches_per_forward": sum(n for _, n in per_kernel.values()) / len(step_ms),
        "envelope": env,
        "first_call_ms": first_ms,
        "config": {"n_layers": s.n_layers, "d_model": s.d_model, "n_heads": s.n_heads,
                   "d_ff": s.d_ff, "batch": s.batch, "seq_len": s.seq_len, "io_dtype": s.dtype,
                   "valid_len": f"U[{s.vl_lo},{s.vl_hi}]"},
    }


def run_ours(args, shape):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    from transformer_encoder_layer_gb300 import binding, build
    from transformer_encoder_layer_gb300.inputs import SHAPES

    if rank == 0 or not os.path.exists(binding.LIB_PATH):
        build.build()
    if dist:
        dist.barrier()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # ---- headline: the chosen workload, K timed steps
    w = Workload(shape, rank, dev, args.path, args.attention_split, args.gemm_pairs, args.graphs,
                 args.mega_assist)
    step_ms, per_kernel, t_wall, clocks = time_steps(w, args.steps, args.warmup, flush, stream,
                                                     dist, dev.index)
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tokens_per_s(ws, shape.tokens, ms_per_step)
    launches = sum(n for _, n in per_kernel.values())

    # End to end: the C-ABI host-buffer call (H2D of x and valid_len, the
    # forward, D2H of out, stream sync) timed by the host clock.
    out_host = torch.empty_like(w.x_host).pin_memory()
    hws = torch.empty(w.enc.host_workspace_size(shape.batch, shape.seq_len), dtype=torch.uint8,
                      device=dev)
    w.enc.forward_host(w.x_host, w.vl_host, out_host, workspace=hws)
    e2e_t = []
    for _ in range(max(3, min(args.steps, 10))):
        t0 = time.perf_counter()
        w.enc.forward_host(w.x_host, w.vl_host, out_host, workspace=hws)
        e2e_t.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(statistics.mean(e2e_t), dist, dev)
    if not torch.equal(out_host, w.out.cpu()):
        raise RuntimeError("host-buffer forward disagrees with the device forward")

    if rank != 0:
        w.close()
        if dist:
            dist.destroy_process_group()
        return

    head_env = envelope_on_sample(w.inp, w.out_f64())
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": shape.dtype, "data": "synthetic",
        "config": {"workload": shape.name, "n_layers": shape.n_layers, "d_model": shape.d_model,
                   "n_heads": shape.n_heads, "d_ff": shape.d_ff, "batch_per_gpu": shape.batch,
                   "global_batch": ws * shape.batch, "seq_len": shape.seq_len,
                   "io_dtype": shape.dtype, "valid_len": f"U[{shape.vl_lo},{shape.vl_hi}]",
                   "input_scale": 1.0, "path": w.path, "attention_split": w.attention_split,
                   "gemm_pairs": args.gemm_pairs, "graphs": bool(args.graphs),
                   "mega_assisted": w.enc.mega_assisted(shape.batch, shape.seq_len),
                   "parallelism": f"dp{ws}" if ws > 1 else "single",
                   "l2": "flushed between timed steps (256 MB write)"},
        "ms_per_step_p10": percentile(step_ms, 10), "ms_per_step_p90": percentile(step_ms, 90),
        "valid_tokens_per_s": ws * int(w.inp.valid_len.sum()) / (ms_per_step / 1e3),
        "algorithmic_tflop_per_s": w.counts["flops"] / (ms_per_step / 1e3) / 1e12,
        "step_fractions": step_fractions(w.counts, ms_per_step, peaks, sms, shape.dtype),
        "roofline": kernel_roofline(per_kernel, shape, w.counts, peaks, sms, total_ms),
        "per_kernel_ms": {k: v[0] / args.steps for k, v in per_kernel.items()},
        "gpu_launches": launches,
        "wall_s_timed_region": t_wall,
        "envelope": head_env,
        "e2e": {"value": whole_job_tokens_per_s(ws, shape.tokens, 1e3 * e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": int(w.x_host.numel() * w.x_host.element_size() +
                                          w.vl_host.numel() * 4),
                "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size())},
        "clocks": clocks,
    }
    w.close()
    del hws, out_host

    # ---- every workload: a short timed loop each, same method
    if ws == 1 and not args.no_per_workload:
        firsts = first_calls(WORKLOADS) or {}
        table = {}
        for name in WORKLOADS:
            s = SHAPES[name]
            wk = Workload(s, 0, dev)
            k = min(args.steps, PER_WORKLOAD_STEPS[name])
            sm, pk, _, _ = time_steps(wk, k, args.warmup, flush, stream)
            env = envelope_on_sample(wk.inp, wk.out_f64())
            table[name] = per_workload_entry(wk, sm, pk, peaks, sms, env, firsts.get(name))
            wk.close()
        line["per_workload"] = table
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, args.cpu_seqs)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "layered", "mega", "dag"])
    ap.add_argument("--cpu-seqs", type=int, default=4096,
                    help="sequences in the bounded CPU-oracle sample")
    ap.add_argument("--ref-seqs", type=int, default=64,
                    help="sequences per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time the headline workload only (profiling runs)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (small cases for profiling)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the workload's sequence length (valid lengths scaled with it)")
    ap.add_argument("--attention-split", type=int, default=-1,
                    help="split-K attention chunk in 64-key tiles (-1 per shape, 0 off)")
    ap.add_argument("--gemm-pairs", type=int, default=-1, choices=[-1, 0, 1],
                    help="layered GEMMs on CTA pairs: -1 where measured faster, 0 none, 1 all")
    ap.add_argument("--graphs", action="store_true", help="layered path in graph mode")
    ap.add_argument("--mega-assist", type=int, default=-1, choices=[-1, 0, 1],
                    help="megakernel assisting CTAs: -1 automatic, 0 off, 1 on where possible")
    ap.add_argument("--first-call-probe", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.first_call_probe:
        first_call_probe(args.first_call_probe)
        return
    if args.warmup < 3:
        args.warmup = 3
    from transformer_encoder_layer_gb300.inputs import SHAPES
    shape = SHAPES[args.workload]
    if args.batch:
        shape = shape.with_(batch=args.batch)
    if args.seq_len:
        f = args.seq_len / shape.seq_len
        shape = shape.with_(seq_len=args.seq_len, vl_lo=max(1, int(shape.vl_lo * f)),
                            vl_hi=max(1, min(args.seq_len, int(shape.vl_hi * f))))
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_ours(args, shape)


if __name__ == "__main__":
    main()
